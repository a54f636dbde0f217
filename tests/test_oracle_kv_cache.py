"""Pins of the oracle's FP8 KV cache (store: e4m3(fl32(x / scale)) into slot
rows; load: bf16(fl32(dec(q) * scale)) out of slot rows), the FP8 KV cache of
"[vLLM] FP8", section "KV 캐시 양자화" (one scale per tensor for keys and one
for values, 1.0 when uncalibrated).

Independent of the oracle's arithmetic: torch's IEEE float32 division, its
float8_e4m3fn and bfloat16 casts, and numpy's fancy indexing for the slots.
"""
import numpy as np
import pytest
import torch

import synth


def _torch_store(x_bits, slots, cache, scale):
    xt = torch.from_numpy(synth.bf16_bits_to_f32(x_bits))
    q = (xt / torch.tensor(scale, dtype=torch.float32)).clamp(-448, 448).to(torch.float8_e4m3fn)
    q = q.view(torch.uint8).numpy()
    out = cache.copy()
    for t, s in enumerate(slots):
        if 0 <= s < cache.shape[0]:
            out[s] = q[t]
    return out


def _torch_load(cache, slots, out, scale):
    dec = torch.from_numpy(cache).view(torch.float8_e4m3fn).to(torch.float64) * float(np.float32(scale))
    rows = dec.to(torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    out = out.copy()
    for t, s in enumerate(slots):
        if 0 <= s < cache.shape[0]:
            out[t] = rows[s]
    return out


def test_bf16_rounding_matches_torch_cast(oracle_lib):
    rng = np.random.default_rng(0)
    bits = rng.integers(0, 2 ** 32, size=200000, dtype=np.uint64).astype(np.uint32)
    special = np.array([0x00000000, 0x80000000, 0x00008000, 0x00018000, 0x3F808000, 0x3F818000, 0x3F807FFF,
                        0x7F7F8000, 0x7F7FFFFF, 0xFF7F8000, 0x7F800000, 0xFF800000, 0x00000001, 0x807FFFFF,
                        0x3F7FFFFF, 0x477FE000], dtype=np.uint32)
    x = np.concatenate([bits, special]).view(np.float32)
    x = x[~np.isnan(x)]
    got = oracle_lib.bf16_from_f32(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, ref)
    nan = oracle_lib.bf16_from_f32(np.array([np.nan, -np.nan], dtype=np.float32))
    assert all((v & 0x7F80) == 0x7F80 and (v & 0x7F) != 0 for v in nan)


@pytest.mark.parametrize("scale", [1.0, 0.0173, 3.5, 2.0 ** -20])
def test_kv_store_matches_torch(oracle_lib, scale):
    T, E, S = 9, 64, 16
    x = synth.activations(T, E, 1, f"kv/x/{scale}", outlier_channels=1, outlier_scale=50.0)
    slots = np.array([3, 0, -1, 15, 7, 16, 2, -5, 9], dtype=np.int64)  # padding and one out of range
    cache = np.full((S, E), 0xA5, dtype=np.uint8)
    ref = _torch_store(x, slots, cache, np.float32(scale))
    got = oracle_lib.kv_store(x, slots, cache.copy(), scale)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("scale", [1.0, 0.0173, 3.5, 2.0 ** -20])
def test_kv_load_matches_torch(oracle_lib, scale):
    rng = np.random.default_rng(3)
    S, E = 12, 256
    cache = rng.integers(0, 256, size=(S, E)).astype(np.uint8)
    cache[(cache & 0x7F) == 0x7F] = 0x00  # NaN codes are checked apart
    cache[0, :] = np.arange(256, dtype=np.uint16).astype(np.uint8)
    cache[0, [0x7F, 0xFF]] = [0x7E, 0xFE]
    slots = np.array([0, 11, -1, 4, 12, 4], dtype=np.int64)
    out = np.full((slots.size, E), 0x1234, dtype=np.uint16)
    ref = _torch_load(cache, slots, out, np.float32(scale))
    got = oracle_lib.kv_load(cache, slots, out.copy(), scale)
    assert np.array_equal(got, ref)


def test_kv_round_trip_error_bound(oracle_lib):
    """load(store(x)) is within half an E4M3 step of x (times the scale), plus
    the BF16 rounding of the result, for values inside the scaled range."""
    T, E = 32, 128
    x = synth.activations(T, E, 5, "kv/rt", outlier_channels=0)
    scale = np.float32(4.0 / 448)
    slots = np.arange(T, dtype=np.int64)[::-1].copy()
    cache = oracle_lib.kv_store(x, slots, np.zeros((T, E), np.uint8), scale)
    y = oracle_lib.kv_load(cache, slots, np.zeros((T, E), np.uint16), scale)
    xf = synth.bf16_bits_to_f32(x).astype(np.float64)
    yf = synth.bf16_bits_to_f32(y).astype(np.float64)
    inside = np.abs(xf) <= 448 * float(scale)
    bound = np.maximum(2.0 ** -4 * np.abs(xf), float(scale) * 2.0 ** -10) + 2.0 ** -8 * np.abs(xf) + 1e-30
    assert np.all(np.abs(yf - xf)[inside] <= bound[inside] * 1.01)
