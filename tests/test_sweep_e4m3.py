"""Every FP32 value through the device's E4M3 conversion, against the
oracle's encoder: all 2^32 bit patterns, in chunks.

The device conversion is the one the quantizers apply to their quotients
(round to nearest even, saturating to +-448); the oracle's encoder is pinned to
the pages' format and to an independent library in test_oracle_e4m3.py. Every
code must agree except on NaN inputs, where the pages say nothing about the
sign of NaN: there both sides must give a NaN code (0x7F or 0xFF) and the
device's choice is reported.

The sweep itself runs on the GPU (marked gpu; this file sorts after the other
GPU test files, so a stop at a first failure leaves them run). The CPU tests
check the sweep's own logic, with the oracle standing in for the device: it
finds no mismatch there, it finds planted ones, and it tolerates a NaN of the
other sign.
"""
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest

import oracle

CHUNK = 1 << 28
NAN_CODES = (0x7F, 0xFF)
# FP32 NaN patterns: exponent all ones, mantissa non-zero, either sign.
NAN_RANGES = ((0x7F800001, 0x80000000), (0xFF800001, 0x100000000))


def oracle_codes(first: int, n: int, out: np.ndarray, threads: int) -> None:
    """The oracle's codes of patterns first .. first + n - 1 into out, split
    over host threads (the C encoder runs without the interpreter lock)."""
    bounds = [first + n * t // threads for t in range(threads + 1)]

    def part(t):
        a, b = bounds[t], bounds[t + 1]
        oracle.e4m3_encode_bits(a, b - a, out[a - first:b - first])

    with ThreadPoolExecutor(threads) as pool:
        list(pool.map(part, range(threads)))


def sweep(encode_chunk, first: int, count: int, chunk: int = CHUNK, threads: int | None = None):
    """Compare encode_chunk(first_bits, n) -> uint8[n] with the oracle over the
    patterns first .. first + count - 1. Returns (mismatches, examples, the
    set of codes the encoder gave NaN inputs)."""
    threads = threads or min(16, os.cpu_count() or 1)
    ref = np.empty(chunk, dtype=np.uint8)
    mismatches = 0
    examples = []
    nan_seen = set()
    for c0 in range(first, first + count, chunk):
        n = min(chunk, first + count - c0)
        got = encode_chunk(c0, n)
        r = ref[:n]
        oracle_codes(c0, n, r, threads)
        bad = got != r
        for lo, hi in NAN_RANGES:
            a, b = max(lo, c0), min(hi, c0 + n)
            if a < b:
                sl = slice(a - c0, b - c0)
                nan_seen.update(int(v) for v in np.unique(got[sl]))
                bad[sl] = ~np.isin(got[sl], NAN_CODES) | (r[sl] != 0x7F)
        k = int(np.count_nonzero(bad))
        if k:
            mismatches += k
            for i in np.flatnonzero(bad)[:4]:
                examples.append((hex(c0 + int(i)), int(got[i]), int(r[i])))
    return mismatches, examples[:8], nan_seen


# ------------------------------------------------------ on the GPU -------

@pytest.mark.gpu
def test_device_conversion_matches_the_oracle_on_every_fp32_pattern():
    import torch

    from fp8_w8a8_quantized_group_gb300 import build, ops
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build.build()
    oracle.build()
    buf = torch.empty(CHUNK, dtype=torch.uint8, device="cuda")

    def device_chunk(c0, n):
        out = buf[:n]
        ops.fp8_selftest_encode_f32(c0, out)
        return out.cpu().numpy()

    mismatches, examples, nan_seen = sweep(device_chunk, 0, 1 << 32)
    print(f"\ndevice codes for NaN inputs: {sorted(hex(v) for v in nan_seen)}")
    assert mismatches == 0, f"{mismatches} patterns differ (bits, device, oracle): {examples}"
    assert nan_seen and nan_seen <= set(NAN_CODES)
    assert ops.fp8_device_error() == (0, 0)


# ------------------------------------------- the sweep's logic, on CPU ---

# Chunk-aligned windows around zero, the subnormals, +-448, +-Inf and the NaNs.
WINDOWS = [(0, 1 << 16), (0x3C000000, 1 << 16), (0x43DF0000, 1 << 17), (0x7F7F0000, 1 << 17),
           (0x80000000, 1 << 16), (0xC3DF0000, 1 << 17), (0xFF7F0000, 1 << 17), (0xFFFF0000, 1 << 16)]


@pytest.fixture(scope="module", autouse=True)
def _built():
    oracle.build()


def _oracle_as_device(c0, n):
    out = np.empty(n, dtype=np.uint8)
    oracle.e4m3_encode_bits(c0, n, out)
    return out


@pytest.mark.parametrize("first,count", WINDOWS)
def test_sweep_finds_nothing_when_the_encoders_agree(first, count):
    mismatches, examples, nan_seen = sweep(_oracle_as_device, first, count, chunk=1 << 15, threads=4)
    assert mismatches == 0, examples
    if first >= 0x7F7F0000 and first < 0x80000000 or first >= 0xFF7F0000:
        assert nan_seen == {0x7F}


def test_sweep_counts_planted_mismatches():
    """Codes changed at chosen patterns (a rounding step near 448, a sign of
    zero, a saturation) are found, counted and reported with their bits."""
    planted = {0x43DFFFFF: 0x7D, 0x80000000: 0x00, 0x7F7FFFFF: 0x7F}

    def wrong(c0, n):
        out = _oracle_as_device(c0, n)
        for bits, code in planted.items():
            if c0 <= bits < c0 + n:
                out[bits - c0] = code
        return out

    total = 0
    for bits in planted:
        first = bits - (bits % (1 << 15))
        mismatches, examples, _ = sweep(wrong, first, 1 << 15, chunk=1 << 13, threads=2)
        total += mismatches
        assert examples and examples[0][0] == hex(bits)
    assert total == len(planted)


def test_sweep_tolerates_a_nan_of_the_other_sign_but_not_a_number():
    def negative_nans(c0, n):
        out = _oracle_as_device(c0, n)
        for lo, hi in NAN_RANGES:
            a, b = max(lo, c0), min(hi, c0 + n)
            if a < b:
                out[a - c0:b - c0] = 0xFF
        return out

    m, _, seen = sweep(negative_nans, 0x7FFF0000, 1 << 16, chunk=1 << 14, threads=2)
    assert m == 0 and seen == {0xFF}

    def nan_as_max(c0, n):
        out = _oracle_as_device(c0, n)
        a = max(0x7F800001, c0)
        if a < c0 + n:
            out[a - c0] = 0x7E
        return out

    m, ex, _ = sweep(nan_as_max, 0x7F800000, 1 << 12, chunk=1 << 12, threads=2)
    assert m == 1 and ex[0][0] == hex(0x7F800001)


def test_chunks_cover_the_range_exactly():
    """The sweep asks for every pattern once, in order, with no chunk past 2^32."""
    asked = []

    def record(c0, n):
        asked.append((c0, n))
        return _oracle_as_device(c0, n)

    sweep(record, (1 << 32) - 3 * 4096 - 8, 3 * 4096 + 8, chunk=4096, threads=2)
    assert asked[0][0] == (1 << 32) - 3 * 4096 - 8
    assert all(a + n == b for (a, n), (b, _) in zip(asked, asked[1:]))
    assert asked[-1][0] + asked[-1][1] == 1 << 32
