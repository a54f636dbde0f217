"""Quantize-then-GEMM enqueued back to back, with no host synchronisation in
between, as a serving loop enqueues it.

The decode GEMM (M <= 16) is a programmatic dependent of the kernel before it
and streams its weights before waiting for that kernel. The weight quantizers
must therefore not let it launch before they have finished writing the codes.
Each iteration draws fresh weights into a new buffer and quantizes them into
ONE shared code buffer, whose previous contents are the last iteration's
codes, then runs the decode GEMMs at once. A GEMM that read any code before
the quantizer had written it would mix two different weight matrices and fall
far outside the tolerance. Every iteration's output is compared with the
oracle on sampled output columns (all rows of each). The host reads nothing
until every iteration is enqueued.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from fp8_w8a8_quantized_group_gb300 import build, ops
from helpers import assert_within_tolerance, bf16_to_f64, f32_bits, to_dev_bf16

pytestmark = pytest.mark.gpu

ITERS = 20


@pytest.fixture(scope="module", autouse=True)
def _ready():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build.build()
    oracle.build()


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def _sample_cols(N, n, seed):
    rng = np.random.default_rng(seed)
    cols = np.unique(np.concatenate([[0, 127, 128, N - 128, N - 1], rng.choice(N, n, replace=False)]))
    return cols.astype(np.int64)


def test_static_per_tensor_weight_then_decode_gemm_no_sync():
    """fp8_quant_per_tensor(W 8192 x 8192, static scale) -> fp8_tensor_gemm at
    M = 1 and M = 16, twenty times with fresh weights, no host sync."""
    N = K = 8192
    x1, _ = synth.per_tensor_case(1, 16, K, seed=1)
    x16, _ = synth.per_tensor_case(16, 16, K, seed=2)
    qa1, sa1 = ops.quant_per_tensor(to_dev_bf16(x1))
    qa16, sa16 = ops.quant_per_tensor(to_dev_bf16(x16))
    w0 = synth.weights(N, K, 0, "order/W0", sigma=0.015)
    _, s_static = oracle.quant_per_tensor(w0)           # a calibrated static scale
    sw = torch.tensor([float(s_static)], dtype=torch.float32, device="cuda")
    qw = torch.empty((N, K), dtype=torch.uint8, device="cuda")
    ws, y1s, y16s = [], [], []
    torch.cuda.synchronize()
    for i in range(ITERS):
        w = synth.device_normal_bf16(N, K, i, f"order/Wt/{i}", sigma=0.015)
        ws.append(w)
        ops.fp8_quant_per_tensor(w, qw, sw, True)
        y1 = torch.empty((1, N), dtype=torch.bfloat16, device="cuda")
        y16 = torch.empty((16, N), dtype=torch.bfloat16, device="cuda")
        ops.fp8_tensor_gemm(qa1, sa1, qw, sw, y1)
        ops.fp8_tensor_gemm(qa16, sa16, qw, sw, y16)
        y1s.append(y1)
        y16s.append(y16)
    assert ops.fp8_device_error() == (0, 0)   # synchronises
    qao1, sao1 = oracle.quant_per_tensor(x1)
    qao16, sao16 = oracle.quant_per_tensor(x16)
    assert f32_bits(sa1.cpu().numpy())[0] == f32_bits(sao1) and f32_bits(sa16.cpu().numpy())[0] == f32_bits(sao16)
    for i in range(ITERS):
        cols = _sample_cols(N, 768, seed=i)
        w_rows = _bits(ws[i][torch.from_numpy(cols).cuda()])
        qwo, _ = oracle.quant_per_tensor(w_rows, scale=s_static)
        if i == ITERS - 1:  # the shared buffer holds the last codes
            assert np.array_equal(qw[torch.from_numpy(cols).cuda()].cpu().numpy(), qwo)
        for qao, sao, y, what in ((qao1, sao1, y1s[i], "M=1"), (qao16, sao16, y16s[i], "M=16")):
            yo, ab = oracle.gemm_tensor(qao, sao, qwo, s_static)
            assert_within_tolerance(bf16_to_f64(y)[:, cols], yo, ab, f"iteration {i} {what}")


def test_weight_block_then_decode_gemm_no_sync():
    """fp8_quant_weight_block(W 4096 x 4096) -> fp8_block_gemm at M = 1, twenty
    times with fresh weights, no host sync."""
    N = K = 4096
    x, _ = synth.block_case(1, 16, K, seed=3)
    qa, sa = ops.quant_act_group(to_dev_bf16(x))
    qw = torch.empty((N, K), dtype=torch.uint8, device="cuda")
    sw = torch.empty((N // 128, K // 128), dtype=torch.float32, device="cuda")
    ws, ys = [], []
    torch.cuda.synchronize()
    for i in range(ITERS):
        w = synth.device_normal_bf16(N, K, i, f"order/Wb/{i}", sigma=0.02)
        ws.append(w)
        ops.fp8_quant_weight_block(w, qw, sw)
        y = torch.empty((1, N), dtype=torch.bfloat16, device="cuda")
        ops.fp8_block_gemm(qa, sa, qw, sw, y)
        ys.append(y)
    assert ops.fp8_device_error() == (0, 0)
    qao, sao = oracle.quant_act_group(x)
    rng = np.random.default_rng(7)
    for i in range(ITERS):
        # Whole 128-row blocks: block quantization is local to a block.
        blocks = np.unique(np.concatenate([[0, N // 128 - 1], rng.choice(N // 128, 6, replace=False)]))
        rows = np.concatenate([np.arange(b * 128, b * 128 + 128) for b in blocks])
        qwo, swo = oracle.quant_weight_block(_bits(ws[i][torch.from_numpy(rows).cuda()]))
        yo, ab = oracle.gemm_block(qao, sao, qwo, swo)
        assert_within_tolerance(bf16_to_f64(ys[i])[:, rows], yo, ab, f"iteration {i}")


def test_rowwise_weight_then_decode_gemm_no_sync():
    """fp8_quant_rowwise(W 4096 x 4096, per output channel) -> fp8_rowwise_gemm
    at M = 1, twenty times with fresh weights, no host sync."""
    N = K = 4096
    x, _ = synth.block_case(1, 16, K, seed=4)
    qa, sa = ops.quant_rowwise(to_dev_bf16(x))
    qw = torch.empty((N, K), dtype=torch.uint8, device="cuda")
    sw = torch.empty((N,), dtype=torch.float32, device="cuda")
    ws, ys = [], []
    torch.cuda.synchronize()
    for i in range(ITERS):
        w = synth.device_normal_bf16(N, K, i, f"order/Wr/{i}", sigma=0.02)
        ws.append(w)
        ops.fp8_quant_rowwise(w, qw, sw)
        y = torch.empty((1, N), dtype=torch.bfloat16, device="cuda")
        ops.fp8_rowwise_gemm(qa, sa, qw, sw, y)
        ys.append(y)
    assert ops.fp8_device_error() == (0, 0)
    qao, sao = oracle.quant_rowwise(x)
    for i in range(ITERS):
        rows = _sample_cols(N, 256, seed=100 + i)  # output channels: per-row quantization is local to a row
        qwo, swo = oracle.quant_rowwise(_bits(ws[i][torch.from_numpy(rows).cuda()]))
        yo, ab = oracle.gemm_rowwise(qao, sao, qwo, swo)
        assert_within_tolerance(bf16_to_f64(ys[i])[:, rows], yo, ab, f"iteration {i}")


def test_kv_store_then_load_no_sync():
    """fp8_kv_cache_store -> fp8_kv_cache_load of the same slots, twenty times
    with fresh keys and values into one cache, no host sync: every load must
    see its own store."""
    T, E, S = 512, 1024, 2048
    kc = torch.zeros((S, E), dtype=torch.uint8, device="cuda")
    vc = torch.zeros((S, E), dtype=torch.uint8, device="cuda")
    ks = torch.tensor([0.02], dtype=torch.float32, device="cuda")
    vs = torch.tensor([0.015], dtype=torch.float32, device="cuda")
    g = torch.Generator(device="cuda")
    g.manual_seed(9)
    slots = torch.randperm(S, generator=g, device="cuda")[:T].contiguous()
    keys, vals, kouts, vouts = [], [], [], []
    torch.cuda.synchronize()
    for i in range(ITERS):
        k = synth.device_normal_bf16(T, E, i, f"order/K/{i}")
        v = synth.device_normal_bf16(T, E, i, f"order/V/{i}")
        ko = torch.empty_like(k)
        vo = torch.empty_like(v)
        ops.fp8_kv_cache_store(k, v, kc, vc, slots, ks, vs)
        ops.fp8_kv_cache_load(kc, vc, ko, vo, slots, ks, vs)
        keys.append(k)
        vals.append(v)
        kouts.append(ko)
        vouts.append(vo)
    assert ops.fp8_device_error() == (0, 0)
    sl = slots.cpu().numpy()
    for i in range(ITERS):
        for x, out, s in ((keys[i], kouts[i], 0.02), (vals[i], vouts[i], 0.015)):
            cache = oracle.kv_store(_bits(x), sl, np.zeros((S, E), np.uint8), s)
            ref = oracle.kv_load(cache, sl, np.zeros((T, E), np.uint16), s)
            assert np.array_equal(_bits(out), ref), f"iteration {i}"
