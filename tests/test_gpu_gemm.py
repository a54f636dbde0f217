"""GPU parity of the FP8 GEMMs against the oracle's FP64 dequantize-then-GEMM.

Bar: |Y_gpu - Y_oracle| <= 2e-3 * sum_k |a b| + 1e-2 * |Y_oracle| per element,
with a = Sa * dec(Qa), b = Sw * dec(Qw). Small shapes (several tiles and a
ragged tail) are compared in full; full-size shapes on sampled outputs (tile
boundary rows plus seeded random points) and, in full, against a plain
PyTorch per-block FP32 check. All calls go through the C ABI.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from fp8_w8a8_quantized_group_gb300 import build, ops
from helpers import (assert_within_tolerance, bf16_to_f64, f32_bits, secondary_block_gemm, tile_boundary_rows,
                     to_dev_bf16)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _ready():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build.build()
    oracle.build()


def _quantize_both(x, w):
    """GPU quantization through the ABI, checked bit-exact against the oracle's."""
    qa, sa = ops.quant_act_group(to_dev_bf16(x))
    qw, sw = ops.quant_weight_block(to_dev_bf16(w))
    qao, sao = oracle.quant_act_group(x)
    qwo, swo = oracle.quant_weight_block(w)
    assert np.array_equal(qa.cpu().numpy(), qao) and np.array_equal(f32_bits(sa.cpu().numpy()), f32_bits(sao))
    assert np.array_equal(qw.cpu().numpy(), qwo) and np.array_equal(f32_bits(sw.cpu().numpy()), f32_bits(swo))
    return (qa, sa, qw, sw), (qao, sao, qwo, swo)


def _sample_points(M, N, n_random=4096, seed=0):
    rng = np.random.default_rng(seed)
    rows = tile_boundary_rows(M)
    cols = np.unique(np.concatenate([np.arange(0, N, 128), np.arange(127, N, 128), [N - 1],
                                     rng.integers(0, N, 8)]))
    ms = np.concatenate([np.repeat(rows, cols.size), rng.integers(0, M, n_random)])
    ns = np.concatenate([np.tile(cols, rows.size), rng.integers(0, N, n_random)])
    return ms.astype(np.int64), ns.astype(np.int64)


# ------------------------------------------------------------ dense block --

@pytest.mark.parametrize("M,N,K", [
    (16, 256, 256),     # tiny layer (decode kernel)
    (1, 256, 256), (4, 384, 1024), (7, 512, 512), (16, 1024, 2048), (3, 272, 384),
    (17, 256, 256),     # smallest prefill-kernel case, ragged
    (129, 384, 512), (300, 272, 1024), (256, 256, 128),
    # decode, unsplit (153 row blocks): a K range of exactly the ring depth
    # (every stage loaded before the upstream wait) and one block more (the
    # first refill after those)
    (16, 19584, 640), (5, 19584, 768),
    # decode split-K with K ranges that do not divide evenly (6, 10 and 14
    # K blocks over clusters of 4, 8 and 8)
    (5, 640, 768), (9, 1024, 1280), (11, 896, 1792),
])
def test_block_gemm_full_compare(M, N, K):
    if (M, N, K) == (16, 256, 256):
        x, w = synth.tiny_block_case()
    else:
        x, w = synth.block_case(M, N, K, seed=1)
    (qa, sa, qw, sw), (qao, sao, qwo, swo) = _quantize_both(x, w)
    y = ops.block_gemm(qa, sa, qw, sw)
    yo, ab = oracle.gemm_block(qao, sao, qwo, swo)
    assert_within_tolerance(bf16_to_f64(y), yo, ab, f"block {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", [(16, 4096, 4096), (1, 28672, 4096), (4, 4096, 14336), (16, 6144, 4096)])
def test_block_gemm_decode_full_size(M, N, K):
    x, w = synth.block_case(M, N, K, seed=0)
    (qa, sa, qw, sw), (qao, sao, qwo, swo) = _quantize_both(x, w)
    y = ops.block_gemm(qa, sa, qw, sw)
    yg = bf16_to_f64(y)
    ms, ns = _sample_points(M, N, n_random=3000)
    yo, ab = oracle.gemm_block_points(qao, sao, qwo, swo, ms, ns)
    assert_within_tolerance(yg[ms, ns], yo, ab, f"decode {M}x{N}x{K} sampled")
    ys, mags = secondary_block_gemm(qa, sa, qw, sw)
    assert_within_tolerance(yg, ys.cpu().numpy(), mags.cpu().numpy(), "decode secondary")


@pytest.mark.parametrize("M,N,K", [(2048, 4096, 4096), (8192, 4096, 14336), (2048, 28672, 4096)])
def test_block_gemm_prefill_full_size(M, N, K):
    x, w = synth.block_case(M, N, K, seed=0)
    (qa, sa, qw, sw), (qao, sao, qwo, swo) = _quantize_both(x, w)
    y = ops.block_gemm(qa, sa, qw, sw)
    yg = bf16_to_f64(y)
    ms, ns = _sample_points(M, N)
    yo, ab = oracle.gemm_block_points(qao, sao, qwo, swo, ms, ns)
    assert_within_tolerance(yg[ms, ns], yo, ab, f"prefill {M}x{N}x{K} sampled")
    r1 = min(M, 1024)
    ys, mags = secondary_block_gemm(qa, sa, qw, sw, rows=(M - r1, M))
    assert_within_tolerance(yg[M - r1:], ys.cpu().numpy(), mags.cpu().numpy(), "prefill secondary")


def test_block_gemm_repeatable():
    x, w = synth.block_case(300, 512, 1024, seed=4)
    (qa, sa, qw, sw), _ = _quantize_both(x, w)
    y1 = ops.block_gemm(qa, sa, qw, sw)
    y2 = ops.block_gemm(qa, sa, qw, sw)
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))


def test_block_gemm_integer_exact():
    """Unit scales and small-integer codes: every partial sum is an exact
    integer below 2^24, so the BF16 result must equal the rounded integer."""
    rng = np.random.default_rng(2)
    M, N, K = 200, 256, 512
    int_codes = np.array([0x00, 0x38, 0x40, 0x44, 0x48], dtype=np.uint8)  # 0, 1, 2, 3, 4
    ia = rng.integers(0, 5, size=(M, K))
    iw = rng.integers(0, 5, size=(N, K))
    neg = rng.random((M, K)) < 0.5
    qa = torch.from_numpy(int_codes[ia] | np.where(neg, 0x80, 0).astype(np.uint8)).cuda()
    qw = torch.from_numpy(int_codes[iw]).cuda()
    sa = torch.ones((K // 128, M), dtype=torch.float32, device="cuda")
    sw = torch.ones((N // 128, K // 128), dtype=torch.float32, device="cuda")
    y = ops.block_gemm(qa, sa, qw, sw)
    exact = (ia * np.where(neg, -1, 1)) @ iw.T
    expect = torch.from_numpy(exact.astype(np.float32)).to(torch.bfloat16)
    assert torch.equal(y.cpu().view(torch.int16), expect.view(torch.int16))
    for m in (1, 5):  # decode kernel
        yd = ops.block_gemm(qa[:m].contiguous(), sa[:, :m].contiguous(), qw, sw)
        assert torch.equal(yd.cpu().view(torch.int16), expect[:m].view(torch.int16))


# ---------------------------------------------------------------- grouped --

def _grouped_case(counts, N, K, seed=0):
    counts = np.asarray(counts)
    offsets = np.zeros(len(counts) + 1, dtype=np.int32)
    offsets[1:] = np.cumsum(counts)
    M = int(offsets[-1])
    x = synth.activations(M, K, seed, f"gtest/{M}")
    w = np.stack([synth.weights(N, K, seed, f"gtest/W{e}") for e in range(len(counts))])
    return x, w, offsets


def _run_grouped(x, w, offsets, extra_rows=0):
    E, N, K = w.shape
    M = x.shape[0]
    qa, sa = ops.quant_act_group(to_dev_bf16(x))
    qw = torch.empty((E, N, K), dtype=torch.uint8, device="cuda")
    sw = torch.empty((E, (N + 127) // 128, K // 128), dtype=torch.float32, device="cuda")
    for e in range(E):
        ops.fp8_quant_weight_block(to_dev_bf16(w[e]), qw[e], sw[e])
    y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    off_d = torch.from_numpy(offsets).cuda()
    ops.fp8_block_gemm(qa, sa, qw, sw, y, num_groups=E, group_offsets=off_d)
    return (qa, sa, qw, sw), bf16_to_f64(y)


def test_grouped_small_full_compare():
    x, w, offsets = _grouped_case([5, 0, 300, 129, 1, 128], N=256, K=512)
    (qa, sa, qw, sw), yg = _run_grouped(x, w, offsets)
    qao, sao = oracle.quant_act_group(x)
    qwo = np.stack([oracle.quant_weight_block(w[e])[0] for e in range(w.shape[0])])
    swo = np.stack([oracle.quant_weight_block(w[e])[1] for e in range(w.shape[0])])
    M, N = yg.shape
    ms = np.repeat(np.arange(M), N)
    ns = np.tile(np.arange(N), M)
    yo, ab = oracle.gemm_grouped_points(qao, sao, qwo, swo, offsets, ms, ns)
    assert_within_tolerance(yg.ravel(), yo, ab, "grouped small")


def test_grouped_rows_outside_experts_untouched():
    x, w, offsets = _grouped_case([40, 200], N=128, K=256)
    offsets = offsets.copy()
    offsets[0] = 10        # rows 0..9 belong to no expert
    offsets[-1] = 230      # rows 230..239 belong to no expert
    (qa, sa, qw, sw), yg = _run_grouped(x, w, offsets)
    assert np.all(np.isnan(yg[:10])) and np.all(np.isnan(yg[230:]))
    assert not np.any(np.isnan(yg[10:230]))


def test_grouped_moe_full_size():
    """Mixture-of-experts layer: 8 experts [2048, 7168], 4096 tokens routed
    top-2 by a seeded uniform router (8192 permuted rows, uneven counts)."""
    x, w, offsets = synth.moe_case()
    (qa, sa, qw, sw), yg = _run_grouped(x, w, offsets)
    qao, sao = oracle.quant_act_group(x)
    assert np.array_equal(qa.cpu().numpy(), qao)
    qwo = qw.cpu().numpy()
    swo = sw.cpu().numpy()
    for e in range(w.shape[0]):  # expert weights bit-exact too
        q_e, s_e = oracle.quant_weight_block(w[e])
        assert np.array_equal(qwo[e], q_e) and np.array_equal(f32_bits(swo[e]), f32_bits(s_e))
    M, N = yg.shape
    rng = np.random.default_rng(5)
    edge_rows = np.unique(np.concatenate([offsets[:-1], offsets[1:] - 1]).clip(0, M - 1))
    cols = np.array([0, 127, 128, 1000, N - 1])
    ms = np.concatenate([np.repeat(edge_rows, cols.size), rng.integers(0, M, 4096)])
    ns = np.concatenate([np.tile(cols, edge_rows.size), rng.integers(0, N, 4096)])
    yo, ab = oracle.gemm_grouped_points(qao, sao, qwo, swo, offsets, ms, ns)
    assert_within_tolerance(yg[ms, ns], yo, ab, "moe sampled")
    for e in (0, 7):
        r0, r1 = int(offsets[e]), int(offsets[e + 1])
        ys, mags = secondary_block_gemm(qa[r0:r1], sa[:, r0:r1].contiguous(), qw[e], sw[e])
        assert_within_tolerance(yg[r0:r1], ys.cpu().numpy(), mags.cpu().numpy(), f"moe expert {e} secondary")


# ------------------------------------------------------------- per tensor --

@pytest.mark.parametrize("M,N,K", [(1, 512, 1024), (16, 1024, 2048), (5, 256, 208), (17, 256, 256),
                                   (300, 512, 1040)])
def test_tensor_gemm_full_compare(M, N, K):
    x, w = synth.per_tensor_case(M, N, K, seed=2)
    qa, sa = ops.quant_per_tensor(to_dev_bf16(x))
    qao, sao = oracle.quant_per_tensor(x)
    _, swo = oracle.quant_per_tensor(w)
    qw, sw = ops.quant_per_tensor(to_dev_bf16(w), scale=torch.tensor([float(swo)], device="cuda"))
    qwo, _ = oracle.quant_per_tensor(w, scale=swo)
    assert np.array_equal(qa.cpu().numpy(), qao) and np.array_equal(qw.cpu().numpy(), qwo)
    y = ops.tensor_gemm(qa, sa, qw, sw)
    yo, ab = oracle.gemm_tensor(qao, sao, qwo, swo)
    assert_within_tolerance(bf16_to_f64(y), yo, ab, f"tensor {M}x{N}x{K}")


@pytest.mark.parametrize("M", [1, 16, 512, 4096])
def test_tensor_gemm_full_size(M):
    N = K = 8192
    x, w = synth.per_tensor_case(M, N, K, seed=0)
    qa, sa = ops.quant_per_tensor(to_dev_bf16(x))
    _, swo = oracle.quant_per_tensor(w)
    qw, sw = ops.quant_per_tensor(to_dev_bf16(w), scale=torch.tensor([float(swo)], device="cuda"))
    qao, sao = oracle.quant_per_tensor(x)
    qwo, _ = oracle.quant_per_tensor(w, scale=swo)
    assert f32_bits(sa.cpu().numpy())[0] == f32_bits(sao)
    y = ops.tensor_gemm(qa, sa, qw, sw)
    yg = bf16_to_f64(y)
    ms, ns = _sample_points(M, N, n_random=2000)
    yo, ab = oracle.gemm_tensor_points(qao, sao, qwo, swo, ms, ns)
    assert_within_tolerance(yg[ms, ns], yo, ab, f"tensor {M} sampled")


def test_tensor_gemm_matches_block_gemm_with_uniform_scales():
    """Per-tensor scales are block scales that happen to be equal: both GEMMs agree."""
    rng = np.random.default_rng(1)
    M, N, K = 40, 256, 512
    qa = torch.from_numpy(rng.integers(0, 0x7E, size=(M, K)).astype(np.uint8)).cuda()
    qw = torch.from_numpy(rng.integers(0, 0x7E, size=(N, K)).astype(np.uint8) | 0x80).cuda()
    sa = torch.tensor([0.013], dtype=torch.float32, device="cuda")
    sw = torch.tensor([0.0007], dtype=torch.float32, device="cuda")
    yt = bf16_to_f64(ops.tensor_gemm(qa, sa, qw, sw))
    yb = bf16_to_f64(ops.block_gemm(qa, sa.expand(K // 128, M).contiguous(), qw,
                                    sw.expand(N // 128, K // 128).contiguous()))
    qao, qwo = qa.cpu().numpy(), qw.cpu().numpy()
    yo, ab = oracle.gemm_tensor(qao, np.float32(0.013), qwo, np.float32(0.0007))
    assert_within_tolerance(yt, yo, ab, "tensor")
    assert_within_tolerance(yb, yo, ab, "block with uniform scales")


# ---------------------------------------------------------- fused linear --

@pytest.mark.parametrize("M,N,K", [(1, 256, 256), (3, 384, 1024), (16, 256, 256), (16, 4096, 4096),
                                   (7, 272, 14336), (1, 28672, 4096), (40, 512, 512)])
def test_block_linear_matches_separate_calls_and_oracle(M, N, K):
    """fp8_block_linear writes the same activation codes and scales as
    fp8_quant_act_group and the same Y, bit for bit, as fp8_block_gemm on them;
    Y is within tolerance of the oracle."""
    x, w = synth.block_case(M, N, K, seed=3)
    xd = to_dev_bf16(x)
    qw, sw = ops.quant_weight_block(to_dev_bf16(w))
    y, qa, sa = ops.block_linear(xd, qw, sw)
    qa2, sa2 = ops.quant_act_group(xd)
    y2 = ops.block_gemm(qa2, sa2, qw, sw)
    torch.cuda.synchronize()
    assert torch.equal(qa, qa2) and torch.equal(sa.view(torch.int32), sa2.view(torch.int32))
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16))
    qao, sao = oracle.quant_act_group(x)
    qwo, swo = oracle.quant_weight_block(w)
    assert np.array_equal(qa.cpu().numpy(), qao) and np.array_equal(f32_bits(sa.cpu().numpy()), f32_bits(sao))
    yg = bf16_to_f64(y)
    if M * N * K <= 64 * 2 ** 20:
        yo, ab = oracle.gemm_block(qao, sao, qwo, swo)
        assert_within_tolerance(yg, yo, ab, f"linear {M}x{N}x{K}")
    else:
        ms, ns = _sample_points(M, N, n_random=2000)
        yo, ab = oracle.gemm_block_points(qao, sao, qwo, swo, ms, ns)
        assert_within_tolerance(yg[ms, ns], yo, ab, f"linear {M}x{N}x{K} sampled")


def test_block_linear_wide_unsplit_matches_separate_calls():
    """M <= 16 with N = 19584 (more 128-row blocks than fit twice on the GPU,
    so K is not split) and K = 8320 (65 K blocks per CTA, more than the ring
    holds several times over): same codes, scales and Y as the separate calls."""
    M, N, K = 5, 19584, 8320
    xd = synth.device_normal_bf16(M, K, 11, "long-k/X", outlier_cols=[7, 4000], outlier_scale=50.0)
    wd = synth.device_normal_bf16(N, K, 11, "long-k/W", sigma=0.02)
    qw, sw = ops.quant_weight_block(wd)
    y, qa, sa = ops.block_linear(xd, qw, sw)
    qa2, sa2 = ops.quant_act_group(xd)
    y2 = ops.block_gemm(qa2, sa2, qw, sw)
    torch.cuda.synchronize()
    assert torch.equal(qa, qa2) and torch.equal(sa.view(torch.int32), sa2.view(torch.int32))
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16))


def test_block_linear_repeated_calls_stable():
    x, w = synth.block_case(16, 1024, 2048, seed=8)
    xd = to_dev_bf16(x)
    qw, sw = ops.quant_weight_block(to_dev_bf16(w))
    outs = [ops.block_linear(xd, qw, sw)[0] for _ in range(3)]
    assert all(torch.equal(o.view(torch.int16), outs[0].view(torch.int16)) for o in outs[1:])


# -------------------------------------------- per token x per channel --

@pytest.mark.parametrize("rows,cols", [(1, 4096), (16, 14336), (7, 272), (300, 1040), (2048, 4096), (5, 20480)])
def test_quant_rowwise_bit_exact(rows, cols):
    x = synth.activations(rows, cols, 6, f"rowq/{rows}x{cols}")
    q, s = ops.quant_rowwise(to_dev_bf16(x))
    qo, so = oracle.quant_rowwise(x)
    assert np.array_equal(f32_bits(s.cpu().numpy()), f32_bits(so))
    assert np.array_equal(q.cpu().numpy(), qo)


def _rowwise_case(M, N, K, seed):
    x, w = synth.block_case(M, N, K, seed=seed)
    qa, sa = ops.quant_rowwise(to_dev_bf16(x))
    qw, sw = ops.quant_rowwise(to_dev_bf16(w))
    qao, sao = oracle.quant_rowwise(x)
    qwo, swo = oracle.quant_rowwise(w)
    assert np.array_equal(qa.cpu().numpy(), qao) and np.array_equal(f32_bits(sa.cpu().numpy()), f32_bits(sao))
    assert np.array_equal(qw.cpu().numpy(), qwo) and np.array_equal(f32_bits(sw.cpu().numpy()), f32_bits(swo))
    return (qa, sa, qw, sw), (qao, sao, qwo, swo)


@pytest.mark.parametrize("M,N,K", [(1, 256, 256), (16, 1024, 2048), (5, 272, 208), (3, 19584, 768),
                                   (17, 256, 256), (300, 512, 1040), (129, 384, 512)])
def test_rowwise_gemm_full_compare(M, N, K):
    (qa, sa, qw, sw), (qao, sao, qwo, swo) = _rowwise_case(M, N, K, seed=12)
    y = ops.rowwise_gemm(qa, sa, qw, sw)
    yo, ab = oracle.gemm_rowwise(qao, sao, qwo, swo)
    assert_within_tolerance(bf16_to_f64(y), yo, ab, f"rowwise {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", [(1, 28672, 4096), (16, 4096, 14336), (2048, 4096, 4096), (4096, 6144, 4096)])
def test_rowwise_gemm_full_size(M, N, K):
    (qa, sa, qw, sw), (qao, sao, qwo, swo) = _rowwise_case(M, N, K, seed=13)
    yg = bf16_to_f64(ops.rowwise_gemm(qa, sa, qw, sw))
    ms, ns = _sample_points(M, N, n_random=3000)
    yo, ab = oracle.gemm_rowwise_points(qao, sao, qwo, swo, ms, ns)
    assert_within_tolerance(yg[ms, ns], yo, ab, f"rowwise {M}x{N}x{K} sampled")


# ------------------------------------------- the linear layer at decode --

@pytest.mark.parametrize("M,N,K", [(16, 4096, 4096), (16, 6144, 4096), (16, 4096, 14336), (9, 1024, 1280),
                                   (2, 19584, 8320), (16, 256, 128)])
def test_block_linear_decode_matches_separate_calls(M, N, K):
    """At decode sizes fp8_block_linear (the quantizer chained to the decode
    GEMM by programmatic dependent launch) writes codes, scales and Y
    bit-identical to fp8_quant_act_group followed by fp8_block_gemm, for K
    ranges of one to 65 blocks per CTA, split and unsplit, and M not a
    multiple of four."""
    xd = synth.device_normal_bf16(M, K, 21, f"fused/X/{M}x{K}", outlier_cols=[3, K // 2], outlier_scale=50.0)
    wd = synth.device_normal_bf16(N, K, 21, f"fused/W/{N}x{K}", sigma=0.02)
    qw, sw = ops.quant_weight_block(wd)
    y, qa, sa = ops.block_linear(xd, qw, sw)
    qa2, sa2 = ops.quant_act_group(xd)
    y2 = ops.block_gemm(qa2, sa2, qw, sw)
    assert ops.fp8_device_error() == (0, 0)
    assert torch.equal(qa, qa2) and torch.equal(sa.view(torch.int32), sa2.view(torch.int32))
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16))
    x = xd.view(torch.int16).cpu().numpy().view(np.uint16)
    qao, sao = oracle.quant_act_group(x)
    assert np.array_equal(qa.cpu().numpy(), qao) and np.array_equal(f32_bits(sa.cpu().numpy()), f32_bits(sao))
    # The oracle on the first and the last 128-row weight block (block
    # quantization is local to a block), all M rows of Y there.
    for n0 in sorted({0, (N - 1) // 128 * 128}):
        n1 = min(N, n0 + 128)
        w_blk = wd[n0:n1].contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
        qwo, swo = oracle.quant_weight_block(w_blk)
        yo, ab = oracle.gemm_block(qao, sao, qwo, swo)
        assert_within_tolerance(bf16_to_f64(y)[:, n0:n1], yo, ab, f"linear {M}x{N}x{K} columns {n0}..{n1}")


def test_block_linear_back_to_back_no_sync():
    """Twenty linear calls on one stream, fresh activations, one
    shared qa / sa pair (as a layer loop reuses them), no host sync: each Y
    matches the two-kernel path bit for bit."""
    M, N, K = 16, 4096, 4096
    wd = synth.device_normal_bf16(N, K, 22, "fused/seq/W", sigma=0.02)
    qw, sw = ops.quant_weight_block(wd)
    xs = [synth.device_normal_bf16(M, K, i, f"fused/seq/X/{i}") for i in range(20)]
    qa = torch.empty((M, K), dtype=torch.uint8, device="cuda")
    sa = torch.empty((K // 128, M), dtype=torch.float32, device="cuda")
    ys = [torch.empty((M, N), dtype=torch.bfloat16, device="cuda") for _ in xs]
    torch.cuda.synchronize()
    for x, y in zip(xs, ys):
        ops.fp8_block_linear(x, qa, sa, qw, sw, y)
    assert ops.fp8_device_error() == (0, 0)
    for x, y in zip(xs, ys):
        qa2, sa2 = ops.quant_act_group(x)
        assert torch.equal(y.view(torch.int16), ops.block_gemm(qa2, sa2, qw, sw).view(torch.int16))


# ------------------------------------------------------- gathered rows --

def test_quant_gather_equals_quant_of_permuted_rows():
    """Routed-row quantization reads each row through the index: codes and
    scales equal fp8_quant_act_group on the permuted copy, and the oracle."""
    rng = np.random.default_rng(3)
    tokens, K = 700, 1152
    M = 1301
    row_index = rng.integers(0, tokens, size=M).astype(np.int32)
    x = synth.activations(tokens, K, 3, "gather/X", outlier_channels=2, outlier_scale=50.0)
    xd = to_dev_bf16(x)
    ri = torch.from_numpy(row_index).cuda()
    q = torch.empty((M, K), dtype=torch.uint8, device="cuda")
    s = torch.empty((K // 128, M), dtype=torch.float32, device="cuda")
    ops.fp8_quant_act_group_gather(xd, ri, q, s)
    q2, s2 = ops.quant_act_group(xd.index_select(0, ri.long()).contiguous())
    assert ops.fp8_device_error() == (0, 0)
    assert torch.equal(q, q2) and torch.equal(s.view(torch.int32), s2.view(torch.int32))
    qo, so = oracle.quant_act_group(x[row_index])
    assert np.array_equal(q.cpu().numpy(), qo) and np.array_equal(f32_bits(s.cpu().numpy()), f32_bits(so))


def test_gathered_moe_full_size():
    """The MoE layer without a permuted copy of X: X [4096, 7168] in token
    order, top-2 routing gathered by the activation quantizer, 8 experts
    [2048, 7168] in the grouped GEMM; sampled against the oracle."""
    tokens, E, N, K = 4096, 8, 2048, 7168
    x = synth.activations(tokens, K, 0, "moe/X", outlier_channels=0)
    token_of_row, offsets = synth.route_top2(tokens, E, seed=0)
    M = token_of_row.size
    qa = torch.empty((M, K), dtype=torch.uint8, device="cuda")
    sa = torch.empty((K // 128, M), dtype=torch.float32, device="cuda")
    ops.fp8_quant_act_group_gather(to_dev_bf16(x), torch.from_numpy(token_of_row.astype(np.int32)).cuda(), qa, sa)
    qw = torch.empty((E, N, K), dtype=torch.uint8, device="cuda")
    sw = torch.empty((E, N // 128, K // 128), dtype=torch.float32, device="cuda")
    for e in range(E):
        ops.fp8_quant_weight_block(to_dev_bf16(synth.weights(N, K, 0, f"moe/W{e}", sigma=0.02)), qw[e], sw[e])
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    ops.fp8_block_gemm(qa, sa, qw, sw, y, num_groups=E, group_offsets=torch.from_numpy(offsets).cuda())
    assert ops.fp8_device_error() == (0, 0)
    qao, sao = oracle.quant_act_group(x[token_of_row])
    assert np.array_equal(qa.cpu().numpy(), qao) and np.array_equal(f32_bits(sa.cpu().numpy()), f32_bits(sao))
    yg = bf16_to_f64(y)
    rng = np.random.default_rng(6)
    edge_rows = np.unique(np.concatenate([offsets[:-1], offsets[1:] - 1]).clip(0, M - 1))
    cols = np.array([0, 127, 128, 1000, N - 1])
    ms = np.concatenate([np.repeat(edge_rows, cols.size), rng.integers(0, M, 4096)])
    ns = np.concatenate([np.tile(cols, edge_rows.size), rng.integers(0, N, 4096)])
    yo, ab = oracle.gemm_grouped_points(qao, sao, qw.cpu().numpy(), sw.cpu().numpy(), offsets, ms, ns)
    assert_within_tolerance(yg[ms, ns], yo, ab, "gathered moe sampled")


def test_quant_gather_bad_row_index_reported():
    x = synth.device_normal_bf16(64, 256, 0, "gather/bad")
    ri = torch.arange(40, dtype=torch.int32, device="cuda")
    q = torch.empty((40, 256), dtype=torch.uint8, device="cuda")
    s = torch.empty((2, 40), dtype=torch.float32, device="cuda")
    ops.fp8_quant_act_group_gather(x, ri, q, s)
    assert ops.fp8_device_error() == (0, 0)
    ri[7] = 64
    ops.fp8_quant_act_group_gather(x, ri, q, s)
    assert ops.fp8_device_error() == (5, 303)
