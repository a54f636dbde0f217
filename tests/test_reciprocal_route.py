"""The reciprocal route of the issue-bound quantizers (weight blocks, per
tensor, per row, decode-sized activation groups, KV store), checked as
mathematics on the host (the GPU tests check the kernels themselves).

For a scale s the kernels form r = RN(1/s), lo = RN(r (1 - 2^-21)) and
hi = RN(r (1 + 2^-21)) once; for each value x they accept the E4M3 code of
RN(x lo) when RN(x hi) converts to the same code, and divide otherwise (and
for every x when r is not a normal number or hi overflows). The claim: an
accepted code always equals the code of the correctly rounded quotient
RN(x/s). numpy's float32 arithmetic is IEEE round-to-nearest-even with
subnormals, so it reproduces every rounding step; the E4M3 conversion is
round-to-nearest-even with saturation, here torch's cast of the value clipped
to +-448 (the oracle's encoder is pinned to that cast within the range).
Every BF16 value is tried against scales over the whole FP32 range, subnormal
and largest included, and against scales that put x/s next to a rounding
midpoint.
"""
import numpy as np
import pytest
import torch

import synth

E4M3_MAX = np.float32(448.0)
DOWN = np.float32(1.0 - 2.0 ** -21)
UP = np.float32(1.0 + 2.0 ** -21)


def _codes(v: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.clip(v, -E4M3_MAX, E4M3_MAX))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def _all_bf16_values() -> np.ndarray:
    x = synth.bf16_bits_to_f32(np.arange(65536, dtype=np.uint32).astype(np.uint16))
    return x[~np.isnan(x)].astype(np.float32)


def _scales() -> list[float]:
    rng = np.random.default_rng(2024)
    out = list(np.exp2(rng.uniform(-149.0, 127.99, 300)).astype(np.float32))
    out += [np.float32(v) for v in (1.4e-45, 1e-40, 2.0 ** -126, 1e-10 / 448, 1.0, 3.0, 0.1, 448.0, 3e38,
                                    3.4028235e38)]
    # scales that put x/s a few ulps from the midpoint between two E4M3 codes
    vals = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    mids = (vals[:0x7E] + vals[1:0x7F]) / 2
    for _ in range(40):
        x = float(_all_bf16_values()[rng.integers(0, 65000)])
        if x == 0 or not np.isfinite(x):
            continue
        s = np.float32(abs(x) / rng.choice(mids[8:]))
        for k in (-2, -1, 0, 1, 2):
            out.append(np.float32(s + np.float32(k) * np.spacing(s)))
    return [float(v) for v in out if np.isfinite(v) and v > 0]


SCALES = _scales()


def _bracket(s, down, up):
    """(lo, hi) multipliers of scale s, or None where the kernels divide."""
    with np.errstate(over="ignore", divide="ignore", under="ignore"):
        r = np.float32(1.0) / s
        lo, hi = r * down, r * up
    if not (abs(r) >= np.float32(2.0 ** -126) and np.isfinite(hi)):
        return None
    return lo, hi


def _accepted_and_wrong(scales, down, up):
    """(accepted, accepted with a code other than the division's, an example)."""
    x = _all_bf16_values()
    accepted = wrong = 0
    example = None
    for s in scales:
        s = np.float32(s)
        b = _bracket(s, down, up)
        if b is None:
            continue  # the kernels divide for every element
        with np.errstate(over="ignore", invalid="ignore", divide="ignore", under="ignore"):
            exact = x / s
            lo, hi = x * b[0], x * b[1]
        clo = _codes(lo)
        accept = clo == _codes(hi)
        bad = accept & (clo != _codes(exact))
        accepted += int(accept.sum())
        wrong += int(bad.sum())
        if bad.any() and example is None:
            example = (s, x[bad][:4])
    return accepted, wrong, example


@pytest.mark.parametrize("chunk", range(4))
def test_accepted_codes_equal_the_divided_codes(chunk):
    accepted, wrong, example = _accepted_and_wrong(SCALES[chunk::4], DOWN, UP)
    assert wrong == 0, f"s, x = {example}: accepted with a code other than the division's"
    assert accepted > 0


def test_a_bracket_too_narrow_to_move_q_is_caught():
    """The check has teeth: with multipliers RN(r (1 -+ 2^-25)), which round
    back to r itself, lo and hi coincide, every element is accepted, and the
    same enumeration finds accepted codes that differ from the division's."""
    narrow_down, narrow_up = np.float32(1.0 - 2.0 ** -25), np.float32(1.0 + 2.0 ** -25)
    _, wrong, _ = _accepted_and_wrong(SCALES[::4], narrow_down, narrow_up)
    assert wrong > 0


def test_most_values_take_the_fast_path_at_typical_scales():
    """At scales of ordinary weights and activations nearly every element is
    accepted, so the division stays rare."""
    x = synth.bf16_bits_to_f32(synth.to_bf16(np.random.default_rng(5).normal(0.0, 1.0, 65536)))
    s = np.float32(np.abs(x).max() / 448.0)
    lo, hi = _bracket(s, DOWN, UP)
    accept = _codes((x * lo).astype(np.float32)) == _codes((x * hi).astype(np.float32))
    assert accept.mean() > 0.99


def test_scales_with_a_subnormal_reciprocal_divide():
    """Scales above 2^126 have a subnormal reciprocal, whose relative error is
    not bounded by 2^-24: the kernels divide there."""
    for s in (np.float32(3e38), np.float32(2.0 ** 126) * np.float32(1.5), np.float32(3.4028235e38)):
        assert _bracket(s, DOWN, UP) is None
    assert _bracket(np.float32(2.0 ** 125), DOWN, UP) is not None
