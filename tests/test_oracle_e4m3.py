"""Pins of the oracle's E4M3 codec against facts it does not compute itself.

- The pages' format facts (tests/golden/e4m3_format.txt): bit counts, +-448,
  no infinity; E5M2 and FP16 ranges used to confirm the exponent-bias reading.
- torch.float8_e4m3fn (an independent library codec) for every code and for
  encodes inside the range where its behaviour is unambiguous (|v| <= 448).
- Exhaustive nearest-value search in exact rational arithmetic.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "e4m3_format.txt")


def _golden():
    facts = {}
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                k, v = line.split()
                facts[k] = float(v)
    return facts


def _torch_decode_all():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def _ieee_like_max(exp_bits, man_bits, has_inf):
    """Largest finite value of a binary format with bias 2^(e-1)-1.
    With infinity the top exponent field is reserved; without it (E4M3 reading)
    only the all-ones mantissa of the top exponent is NaN."""
    bias = 2 ** (exp_bits - 1) - 1
    if has_inf:
        top = 2 ** exp_bits - 2
        return 2.0 ** (top - bias) * (2 - 2.0 ** -man_bits)
    top = 2 ** exp_bits - 1
    return 2.0 ** (top - bias) * (1 + (2 ** man_bits - 2) / 2 ** man_bits)


def test_format_reading_reproduces_page_ranges(oracle_lib):
    g = _golden()
    # The IEEE-style bias reproduces the pages' E5M2 and FP16 ranges ...
    assert _ieee_like_max(g["e5m2_exponent_bits"], g["e5m2_mantissa_bits"], True) == g["e5m2_max"]
    assert _ieee_like_max(g["fp16_exponent_bits"], g["fp16_mantissa_bits"], True) == g["fp16_max"]
    # ... and with "no infinity" the same bias gives exactly +-448 for 4/3 bits.
    assert not g["e4m3_has_infinity"]
    assert _ieee_like_max(int(g["e4m3_exponent_bits"]), int(g["e4m3_mantissa_bits"]), False) == g["e4m3_max"]
    vals = np.array([oracle_lib.e4m3_decode(c) for c in range(256)])
    finite = vals[np.isfinite(vals)]
    assert finite.max() == g["e4m3_max"] and finite.min() == g["e4m3_min"]
    assert not np.isinf(vals).any()
    assert np.isnan(vals).sum() == 2  # S.1111.111
    assert 2 ** (8 * g["e4m3_bytes_per_value"]) == 256


def test_decode_all_codes_match_torch(oracle_lib):
    ours = np.array([oracle_lib.e4m3_decode(c) for c in range(256)])
    ref = _torch_decode_all()
    both_nan = np.isnan(ours) & np.isnan(ref)
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    assert np.array_equal(ours[~both_nan], ref[~both_nan])
    # signed zero: 0x80 decodes to -0.0
    assert math.copysign(1.0, ours[0x80]) == -1.0


def test_round_trip_all_codes(oracle_lib):
    for c in range(256):
        v = oracle_lib.e4m3_decode(c)
        e = oracle_lib.e4m3_encode(v)
        if math.isnan(v):
            assert e & 0x7F == 0x7F
        else:
            assert e == c, (hex(c), v, hex(e))


def test_decode_monotone(oracle_lib):
    pos = [oracle_lib.e4m3_decode(c) for c in range(0x7F)]
    assert all(a < b for a, b in zip(pos, pos[1:]))
    neg = [oracle_lib.e4m3_decode(c) for c in range(0x80, 0xFF)]
    assert all(a > b for a, b in zip(neg, neg[1:]))


def _midpoints():
    ref = _torch_decode_all()
    pos = np.sort(ref[:0x7F])  # 0 .. 448
    mids = (pos[:-1] + pos[1:]) / 2  # exact in float64; representable in float32
    return pos, mids


def test_encode_matches_torch_in_range(oracle_lib):
    pos, mids = _midpoints()
    rng = np.random.default_rng(1)
    samples = [
        mids.astype(np.float32),
        np.nextafter(mids.astype(np.float32), np.float32(np.inf)),
        np.nextafter(mids.astype(np.float32), np.float32(0)),
        pos.astype(np.float32),
        (rng.uniform(-448, 448, 4000)).astype(np.float32),
        (np.exp2(rng.uniform(-14, 9, 4000)) * rng.choice([-1, 1], 4000)).astype(np.float32),
        np.array([2.0 ** -10, 2.0 ** -9 * 0.5, 2.0 ** -9 * 1.5, 2.0 ** -6 - 2.0 ** -10], np.float32),
    ]
    v = np.concatenate(samples)
    v = np.concatenate([v, -v])
    v = v[np.abs(v) <= 448]
    ours = oracle_lib.e4m3_encode_array(v)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    bad = np.nonzero(ours != ref)[0]
    assert bad.size == 0, [(float(v[i]), hex(ours[i]), hex(ref[i])) for i in bad[:8]]


def test_midpoints_round_to_even_code(oracle_lib):
    pos, mids = _midpoints()
    codes = [oracle_lib.e4m3_encode(float(m)) for m in mids]
    # the even neighbour has the lower mantissa bit clear
    assert all(c & 1 == 0 for c in codes)
    for i, m in enumerate(mids):
        up = np.nextafter(np.float32(m), np.float32(np.inf))
        dn = np.nextafter(np.float32(m), np.float32(0))
        assert oracle_lib.e4m3_decode(oracle_lib.e4m3_encode(float(up))) == pos[i + 1]
        assert oracle_lib.e4m3_decode(oracle_lib.e4m3_encode(float(dn))) == pos[i]


def _nearest_code_exact(v: float, values: np.ndarray) -> int:
    """Brute force: nearest finite E4M3 value in exact rationals, ties -> even code,
    values beyond the largest saturate."""
    fv = Fraction(float(v))
    best, best_d = None, None
    for c in range(256):
        if not np.isfinite(values[c]):
            continue
        d = abs(Fraction(float(values[c])) - fv)
        if best is None or d < best_d or (d == best_d and (c & 1) == 0 and (best & 1) == 1):
            best, best_d = c, d
    # keep the sign of zero, and of results that round to zero
    if values[best] == 0:
        best = 0x80 if math.copysign(1.0, v) < 0 else 0x00
    return best


def test_encode_brute_force_exact(oracle_lib):
    values = _torch_decode_all()
    rng = np.random.default_rng(7)
    v = np.concatenate([
        np.exp2(rng.uniform(-12, 8.9, 300)) * rng.choice([-1, 1], 300),
        rng.uniform(-460, 460, 100),
    ]).astype(np.float32)
    for x in v:
        if abs(float(x)) >= 448:
            expect = 0xFE if x < 0 else 0x7E
        else:
            expect = _nearest_code_exact(float(x), values)
        assert oracle_lib.e4m3_encode(float(x)) == expect, (float(x), hex(expect))


@pytest.mark.parametrize("v,code", [
    (448.0, 0x7E), (448.00003, 0x7E), (463.99997, 0x7E), (464.0, 0x7E), (480.0, 0x7E),
    (1e30, 0x7E), (float("inf"), 0x7E), (-464.0, 0xFE), (-1e30, 0xFE), (float("-inf"), 0xFE),
])
def test_saturation(oracle_lib, v, code):
    assert oracle_lib.e4m3_encode(v) == code


def test_signed_zero_and_underflow(oracle_lib):
    assert oracle_lib.e4m3_encode(0.0) == 0x00
    assert oracle_lib.e4m3_encode(-0.0) == 0x80
    assert oracle_lib.e4m3_encode(-1e-30) == 0x80
    assert oracle_lib.e4m3_encode(1e-30) == 0x00
    # half the smallest subnormal ties to zero (even), just above rounds up
    assert oracle_lib.e4m3_encode(2.0 ** -10) == 0x00
    assert oracle_lib.e4m3_encode(float(np.nextafter(np.float32(2.0 ** -10), np.float32(1)))) == 0x01
    assert oracle_lib.e4m3_encode(float("nan")) & 0x7F == 0x7F


@pytest.mark.parametrize("first,n", [(0, 4096), (0x3F7FF000, 8192), (0x43DFF000, 8192), (0x7F7FFF00, 0x100),
                                     (0x7F800000 - 8, 16), (0x80000000, 4096), (0xC3E00000 - 64, 128),
                                     (0xFFFFFFFF - 15, 16)])
def test_bulk_encoder_is_the_per_value_encoder(oracle_lib, first, n):
    """The range encoder used for sweeps over all FP32 patterns gives, for every
    pattern, the code of the per-value encoder (pinned above), including the
    last pattern 0xFFFFFFFF and ranges across +-448, +-Inf and NaN."""
    bits = (np.arange(n, dtype=np.uint64) + first).astype(np.uint32)
    vals = bits.view(np.float32)
    got = oracle_lib.e4m3_encode_bits(first, n)
    assert np.array_equal(got, oracle_lib.e4m3_encode_array(vals))


def test_bulk_encoder_refuses_ranges_past_the_last_pattern(oracle_lib):
    with pytest.raises(ValueError):
        oracle_lib.e4m3_encode_bits(0xFFFFFFF0, 17)
