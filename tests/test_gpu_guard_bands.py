"""Guard bands: every output buffer sits between canary bytes, checked after
the call, at ragged sizes (M = 1, 3, 17, 129, 300; N not a multiple of 128;
an empty expert; padding KV slots).

Each kernel clips its stores to the sizes it is given; a store past the end
of an output (a tile's padding rows, a rounded-up column block, a skipped KV
row) lands in a canary and fails here even when the compared values are right.
The interiors are compared with the oracle as in the other parity tests:
codes and scales bit-exact, GEMM outputs within the tolerance.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from fp8_w8a8_quantized_group_gb300 import build, ops
from helpers import assert_within_tolerance, bf16_to_f64, f32_bits, to_dev_bf16

pytestmark = pytest.mark.gpu

CANARY = 0xA5
GUARD = 4096  # elements on each side; a multiple of 16 bytes for every dtype used


@pytest.fixture(scope="module", autouse=True)
def _ready():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build.build()
    oracle.build()


class Guarded:
    """A contiguous tensor of `shape` inside a buffer with GUARD canary
    elements before and after it."""

    def __init__(self, shape, dtype):
        n = int(np.prod(shape))
        self.buf = torch.empty(n + 2 * GUARD, dtype=dtype, device="cuda")
        self.buf.view(torch.uint8).fill_(CANARY)
        self.t = self.buf[GUARD:GUARD + n].view(shape)

    def check(self, what):
        raw = self.buf.view(torch.uint8)
        g = GUARD * self.buf.element_size()
        for part, name in ((raw[:g], "before"), (raw[raw.numel() - g:], "after")):
            bad = torch.nonzero(part != CANARY)
            assert bad.numel() == 0, f"{what}: {bad.numel()} canary bytes overwritten {name} the buffer"


def _check_all(*gs):
    torch.cuda.synchronize()
    assert ops.fp8_device_error() == (0, 0)
    for g, what in gs:
        g.check(what)


@pytest.mark.parametrize("M,N,K", [(1, 384, 512), (3, 272, 384), (17, 384, 512), (129, 272, 1024),
                                   (300, 256, 128)])
def test_block_path_guarded(M, N, K):
    x, w = synth.block_case(M, N, K, seed=M)
    qa, sa = Guarded((M, K), torch.uint8), Guarded((K // 128, M), torch.float32)
    qw, sw = Guarded((N, K), torch.uint8), Guarded(((N + 127) // 128, K // 128), torch.float32)
    y, yl = Guarded((M, N), torch.bfloat16), Guarded((M, N), torch.bfloat16)
    qal, sal = Guarded((M, K), torch.uint8), Guarded((K // 128, M), torch.float32)
    xd = to_dev_bf16(x)
    ops.fp8_quant_act_group(xd, qa.t, sa.t)
    ops.fp8_quant_weight_block(to_dev_bf16(w), qw.t, sw.t)
    ops.fp8_block_gemm(qa.t, sa.t, qw.t, sw.t, y.t)
    ops.fp8_block_linear(xd, qal.t, sal.t, qw.t, sw.t, yl.t)
    _check_all((qa, "qa"), (sa, "sa"), (qw, "qw"), (sw, "sw"), (y, "y"), (qal, "linear qa"), (sal, "linear sa"),
               (yl, "linear y"))
    qao, sao = oracle.quant_act_group(x)
    qwo, swo = oracle.quant_weight_block(w)
    for q, s, what in ((qa, sa, "act"), (qal, sal, "linear act")):
        assert np.array_equal(q.t.cpu().numpy(), qao), what
        assert np.array_equal(f32_bits(s.t.cpu().numpy()), f32_bits(sao)), what
    assert np.array_equal(qw.t.cpu().numpy(), qwo) and np.array_equal(f32_bits(sw.t.cpu().numpy()), f32_bits(swo))
    yo, ab = oracle.gemm_block(qao, sao, qwo, swo)
    assert_within_tolerance(bf16_to_f64(y.t), yo, ab, "block gemm")
    assert torch.equal(yl.t.view(torch.int16), y.t.view(torch.int16)), "fp8_block_linear differs from the two calls"


@pytest.mark.parametrize("M", [1, 17, 129])
@pytest.mark.parametrize("static", [False, True])
def test_per_tensor_path_guarded(M, static):
    N, K = 272, 512
    x, w = synth.block_case(M, N, K, seed=10 + M)
    _, sw_o = oracle.quant_per_tensor(w)
    qa, sa = Guarded((M, K), torch.uint8), Guarded((1,), torch.float32)
    qw, sw = Guarded((N, K), torch.uint8), Guarded((1,), torch.float32)
    y = Guarded((M, N), torch.bfloat16)
    ops.fp8_quant_per_tensor(to_dev_bf16(x), qa.t, sa.t, is_static=False)
    if static:
        sw.t.fill_(float(sw_o))
    ops.fp8_quant_per_tensor(to_dev_bf16(w), qw.t, sw.t, is_static=static)
    ops.fp8_tensor_gemm(qa.t, sa.t, qw.t, sw.t, y.t)
    _check_all((qa, "qa"), (sa, "sa"), (qw, "qw"), (sw, "sw"), (y, "y"))
    qao, sao = oracle.quant_per_tensor(x)
    qwo, swo = oracle.quant_per_tensor(w, scale=sw_o if static else None)
    assert np.array_equal(qa.t.cpu().numpy(), qao) and np.float32(sa.t.item()) == sao
    assert np.array_equal(qw.t.cpu().numpy(), qwo) and np.float32(sw.t.item()) == swo
    yo, ab = oracle.gemm_tensor(qao, sao, qwo, swo)
    assert_within_tolerance(bf16_to_f64(y.t), yo, ab, "tensor gemm")


@pytest.mark.parametrize("M,N,K", [(1, 272, 512), (17, 384, 1024), (129, 256, 384)])
def test_rowwise_path_guarded(M, N, K):
    x, w = synth.block_case(M, N, K, seed=20 + M)
    qa, sa = Guarded((M, K), torch.uint8), Guarded((M,), torch.float32)
    qw, sw = Guarded((N, K), torch.uint8), Guarded((N,), torch.float32)
    y = Guarded((M, N), torch.bfloat16)
    ops.fp8_quant_rowwise(to_dev_bf16(x), qa.t, sa.t)
    ops.fp8_quant_rowwise(to_dev_bf16(w), qw.t, sw.t)
    ops.fp8_rowwise_gemm(qa.t, sa.t, qw.t, sw.t, y.t)
    _check_all((qa, "qa"), (sa, "sa"), (qw, "qw"), (sw, "sw"), (y, "y"))
    qao, sao = oracle.quant_rowwise(x)
    qwo, swo = oracle.quant_rowwise(w)
    assert np.array_equal(qa.t.cpu().numpy(), qao) and np.array_equal(f32_bits(sa.t.cpu().numpy()), f32_bits(sao))
    assert np.array_equal(qw.t.cpu().numpy(), qwo) and np.array_equal(f32_bits(sw.t.cpu().numpy()), f32_bits(swo))
    yo, ab = oracle.gemm_rowwise(qao, sao, qwo, swo)
    assert_within_tolerance(bf16_to_f64(y.t), yo, ab, "rowwise gemm")


def test_moe_path_guarded():
    """Routed-row quantization and the grouped GEMM: 4 experts, one of them
    empty, ragged expert row counts."""
    tokens, E, N, K = 150, 4, 384, 512
    x = synth.activations(tokens, K, 3, "guard/moe/X")
    counts = [37, 0, 129, 21]
    token_of_row = np.concatenate([synth.pick(3, f"guard/moe/e{e}", tokens, c) for e, c in enumerate(counts)])
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    M = int(offsets[-1])
    qa, sa = Guarded((M, K), torch.uint8), Guarded((K // 128, M), torch.float32)
    qw, sw = Guarded((E, N, K), torch.uint8), Guarded((E, N // 128, K // 128), torch.float32)
    y = Guarded((M, N), torch.bfloat16)
    ops.fp8_quant_act_group_gather(to_dev_bf16(x), torch.from_numpy(token_of_row.astype(np.int32)).cuda(),
                                   qa.t, sa.t)
    ws = [synth.weights(N, K, 3, f"guard/moe/W{e}") for e in range(E)]
    for e in range(E):
        ops.fp8_quant_weight_block(to_dev_bf16(ws[e]), qw.t[e], sw.t[e])
    ops.fp8_block_gemm(qa.t, sa.t, qw.t, sw.t, y.t, num_groups=E, group_offsets=torch.from_numpy(offsets).cuda())
    _check_all((qa, "qa"), (sa, "sa"), (qw, "qw"), (sw, "sw"), (y, "y"))
    qao, sao = oracle.quant_act_group(x[token_of_row])
    assert np.array_equal(qa.t.cpu().numpy(), qao) and np.array_equal(f32_bits(sa.t.cpu().numpy()), f32_bits(sao))
    yg = bf16_to_f64(y.t)
    for e in range(E):
        r0, r1 = int(offsets[e]), int(offsets[e + 1])
        if r1 == r0:
            continue
        qwo, swo = oracle.quant_weight_block(ws[e])
        yo, ab = oracle.gemm_block(qao[r0:r1], np.ascontiguousarray(sao[:, r0:r1]), qwo, swo)
        assert_within_tolerance(yg[r0:r1], yo, ab, f"expert {e}")


def test_kv_cache_guarded():
    """Store into a cache between canaries, with padding slots (-1); load back
    into outputs between canaries. Rows of padding slots stay unwritten."""
    T, E, S = 13, 384, 40
    k = synth.activations(T, E, 4, "guard/kv/k")
    v = synth.activations(T, E, 4, "guard/kv/v")
    slots = np.array([3, -1, 0, 39, 7, -1, 12, 25, 1, 2, 38, 20, 30], dtype=np.int64)
    kc, vc = Guarded((S, E), torch.uint8), Guarded((S, E), torch.uint8)
    kc.t.zero_()
    vc.t.zero_()
    ko, vo = Guarded((T, E), torch.bfloat16), Guarded((T, E), torch.bfloat16)
    ks = torch.tensor([0.25], dtype=torch.float32, device="cuda")
    vs = torch.tensor([1.0], dtype=torch.float32, device="cuda")
    sd = torch.from_numpy(slots).cuda()
    ops.fp8_kv_cache_store(to_dev_bf16(k), to_dev_bf16(v), kc.t, vc.t, sd, ks, vs)
    ops.fp8_kv_cache_load(kc.t, vc.t, ko.t, vo.t, sd, ks, vs)
    _check_all((kc, "key cache"), (vc, "value cache"), (ko, "key out"), (vo, "value out"))
    kco = oracle.kv_store(k, slots, np.zeros((S, E), np.uint8), 0.25)
    vco = oracle.kv_store(v, slots, np.zeros((S, E), np.uint8), 1.0)
    assert np.array_equal(kc.t.cpu().numpy(), kco) and np.array_equal(vc.t.cpu().numpy(), vco)
    canary_rows = np.full((T, E), (CANARY << 8) | CANARY, np.uint16)
    koo = oracle.kv_load(kco, slots, canary_rows.copy(), 0.25)
    voo = oracle.kv_load(vco, slots, canary_rows.copy(), 1.0)
    assert np.array_equal(ko.t.view(torch.int16).cpu().numpy().view(np.uint16), koo)
    assert np.array_equal(vo.t.view(torch.int16).cpu().numpy().view(np.uint16), voo)


@pytest.mark.parametrize("N", [272, 512])
def test_grouped_output_at_expert_boundaries(N):
    """Grouped GEMM whose expert boundaries fall at many row residues mod 32,
    between canaries, with rows before the first expert and after the last
    one: a warp whose 32 output rows cross an expert's end stores them with
    guarded plain stores, every other warp by TMA boxes. Each expert's rows
    match the oracle; rows outside the experts keep their canary bytes."""
    K, lead, tail = 256, 5, 3
    counts = [1, 31, 32, 33, 0, 63, 64, 65, 127, 128, 129, 7]
    E = len(counts)
    offsets = np.concatenate([[lead], lead + np.cumsum(counts)]).astype(np.int32)
    M = int(offsets[-1]) + tail
    x = synth.activations(M, K, 6, f"guard/edges/X/{N}")
    qa_h, sa_h = oracle.quant_act_group(x)
    ws = [synth.weights(N, K, 6, f"guard/edges/W{e}/{N}") for e in range(E)]
    qw = torch.empty((E, N, K), dtype=torch.uint8, device="cuda")
    sw = torch.empty((E, (N + 127) // 128, K // 128), dtype=torch.float32, device="cuda")
    for e in range(E):
        ops.fp8_quant_weight_block(to_dev_bf16(ws[e]), qw[e], sw[e])
    y = Guarded((M, N), torch.bfloat16)
    y.t.view(torch.uint8).fill_(CANARY)
    ops.fp8_block_gemm(torch.from_numpy(qa_h).cuda(), torch.from_numpy(sa_h).cuda(), qw, sw, y.t, num_groups=E,
                       group_offsets=torch.from_numpy(offsets).cuda())
    _check_all((y, "y"))
    yb = y.t.view(torch.int16).cpu().numpy().view(np.uint16)
    outside = np.r_[0:lead, int(offsets[-1]):M]
    assert np.all(yb[outside] == (CANARY << 8) | CANARY), "rows outside the experts were written"
    yg = bf16_to_f64(y.t)
    for e in range(E):
        r0, r1 = int(offsets[e]), int(offsets[e + 1])
        if r1 == r0:
            continue
        qwo, swo = oracle.quant_weight_block(ws[e])
        yo, ab = oracle.gemm_block(qa_h[r0:r1], np.ascontiguousarray(sa_h[:, r0:r1]), qwo, swo)
        assert_within_tolerance(yg[r0:r1], yo, ab, f"expert {e}")
