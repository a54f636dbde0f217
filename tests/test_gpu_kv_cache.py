"""GPU parity of the FP8 KV cache kernels against the oracle: every code
written by the store and every BF16 value written by the load must be
bit-identical; padding slots are skipped, bad slots and scales are reported
through the device error word. Calls go through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
import synth
from fp8_w8a8_quantized_group_gb300 import build, ops
from helpers import to_dev_bf16

pytestmark = pytest.mark.gpu

FP8_ERR_ARG = 5


@pytest.fixture(scope="module", autouse=True)
def _ready():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build.build()
    oracle.build()


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def _case(T, E, S, seed):
    k = synth.activations(T, E, seed, "kvgpu/k", outlier_channels=2, outlier_scale=20.0)
    v = synth.activations(T, E, seed, "kvgpu/v", outlier_channels=0)
    rng = np.random.default_rng(seed)
    slots = rng.permutation(S)[:T].astype(np.int64)
    slots[rng.random(T) < 0.05] = -1  # padding tokens
    return k, v, slots


@pytest.mark.parametrize("T,E,S,ks,vs", [(7, 128, 16, 1.0, 1.0), (300, 1024, 4096, 0.011, 0.0093),
                                         (64, 1040, 64, 2.0 ** -12, 3.0), (2048, 1024, 8192, 1.0, 0.5)])
def test_kv_store_then_load_bit_exact(T, E, S, ks, vs):
    k, v, slots = _case(T, E, S, seed=T + E)
    kc = torch.full((S, E), 0x5A, dtype=torch.uint8, device="cuda")
    vc = torch.full((S, E), 0x5A, dtype=torch.uint8, device="cuda")
    sd = torch.from_numpy(slots).cuda()
    kst = torch.tensor([ks], dtype=torch.float32, device="cuda")
    vst = torch.tensor([vs], dtype=torch.float32, device="cuda")
    ops.fp8_kv_cache_store(to_dev_bf16(k), to_dev_bf16(v), kc, vc, sd, kst, vst)
    ko = oracle.kv_store(k, slots, np.full((S, E), 0x5A, np.uint8), ks)
    vo = oracle.kv_store(v, slots, np.full((S, E), 0x5A, np.uint8), vs)
    assert np.array_equal(kc.cpu().numpy(), ko) and np.array_equal(vc.cpu().numpy(), vo)
    # Load back in another order, including a padding row and a repeated slot.
    order = np.concatenate([slots[::-1], [-1, int(slots.max())]])
    od = torch.from_numpy(order).cuda()
    kout = torch.full((order.size, E), 7.0, dtype=torch.bfloat16, device="cuda")
    vout = torch.full((order.size, E), 7.0, dtype=torch.bfloat16, device="cuda")
    ops.fp8_kv_cache_load(kc, vc, kout, vout, od, kst, vst)
    seven = np.full((order.size, E), 0x40E0, np.uint16)  # bf16(7.0)
    assert np.array_equal(_bits(kout), oracle.kv_load(ko, order, seven.copy(), ks))
    assert np.array_equal(_bits(vout), oracle.kv_load(vo, order, seven.copy(), vs))
    assert ops.fp8_device_error() == (0, 0)


def test_kv_load_every_code():
    """All 256 codes (NaN codes included) dequantized at several scales."""
    E = 256
    cache = torch.arange(256, dtype=torch.int32).to(torch.uint8).repeat(4, 1).cuda()
    slots = np.array([0, 1, 2, 3], dtype=np.int64)
    for s in (1.0, 0.0173, 2.0 ** -100, 1e30):
        st = torch.tensor([s], dtype=torch.float32, device="cuda")
        out_k = torch.empty((4, E), dtype=torch.bfloat16, device="cuda")
        out_v = torch.empty((4, E), dtype=torch.bfloat16, device="cuda")
        ops.fp8_kv_cache_load(cache, cache, out_k, out_v, torch.from_numpy(slots).cuda(), st, st)
        got = _bits(out_k)
        ref = oracle.kv_load(cache.cpu().numpy(), slots, np.zeros((4, E), np.uint16), s)
        nan_codes = np.array([0x7F, 0xFF])
        finite = np.setdiff1d(np.arange(256), nan_codes)
        assert np.array_equal(got[:, finite], ref[:, finite]), s
        assert np.all((got[:, nan_codes] & 0x7F80) == 0x7F80) and np.all((got[:, nan_codes] & 0x7F) != 0)
        assert torch.equal(out_k.view(torch.int16), out_v.view(torch.int16))


def test_kv_bad_slot_and_scale_reported():
    T, E, S = 4, 128, 8
    k = to_dev_bf16(synth.activations(T, E, 0, "kvbad/k"))
    kc = torch.zeros((S, E), dtype=torch.uint8, device="cuda")
    vc = torch.zeros((S, E), dtype=torch.uint8, device="cuda")
    one = torch.ones(1, dtype=torch.float32, device="cuda")
    assert ops.fp8_device_error() == (0, 0)
    ops.fp8_kv_cache_store(k, k, kc, vc, torch.tensor([0, 8, 1, 2], device="cuda"), one, one)
    assert ops.fp8_device_error() == (FP8_ERR_ARG, 401)
    ops.fp8_kv_cache_store(k, k, kc, vc, torch.tensor([0, 1, 2, 3], device="cuda"), one,
                           torch.zeros(1, device="cuda"))
    assert ops.fp8_device_error() == (FP8_ERR_ARG, 402)
