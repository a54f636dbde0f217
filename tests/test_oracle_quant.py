"""Pins of the oracle's quantizers (block, group, per-tensor).

Independent of the oracle's own arithmetic:
- exact rational brute force (scale and quotient rounded exactly to FP32,
  nearest E4M3 value by exhaustive search over torch-decoded codes);
- torch's IEEE FP32 division and its float8_e4m3fn cast;
- invariants that follow from "scale = amax/448" and symmetric scaling
  (vLLM page, sections "스케일링 전략 체계" and "블록 양자화"), and the outlier
  containment that section "왜 이 설계인가" (2) gives as the reason for blocks.
"""
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

import synth

E4M3_VALUES = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def _f32_exact(fr: Fraction) -> np.float32:
    """Correctly rounded FP32 value of a rational (ties to even)."""
    c = np.float32(float(fr))
    cands = [np.nextafter(c, np.float32(-np.inf)), c, np.nextafter(c, np.float32(np.inf))]
    best = None
    for v in cands:
        d = abs(Fraction(float(v)) - fr)
        if best is None or d < best[0] or (d == best[0] and (int(np.float32(v).view(np.uint32)) & 1) == 0):
            best = (d, v)
    return np.float32(best[1])


def _nearest_code(v: np.float32) -> int:
    fv = Fraction(float(v))
    if abs(fv) >= 448:
        return 0xFE if fv < 0 else 0x7E
    best = None
    for c in range(0x7F):  # non-negative finite codes 0 .. 448
        d = abs(Fraction(float(E4M3_VALUES[c])) - abs(fv))
        if best is None or d < best[0] or (d == best[0] and c % 2 == 0):
            best = (d, c)
    code = best[1]
    return code | (0x80 if math.copysign(1.0, float(v)) < 0 else 0)


def _brute_block_quant(x_bits, br, bc):
    """Exact-arithmetic reference: per block amax, s = RN32(amax/448), q = e4m3(RN32(x/s))."""
    x = synth.bf16_bits_to_f32(x_bits)
    rows, cols = x.shape
    q = np.zeros_like(x_bits, dtype=np.uint8)
    scales = {}
    for r0 in range(0, rows, br):
        for c0 in range(0, cols, bc):
            blk = x[r0:r0 + br, c0:c0 + bc]
            amax = max(Fraction(float(abs(v))) for v in blk.ravel())
            amax = max(amax, Fraction(float(np.float32(1e-10))))
            s = _f32_exact(amax / 448)
            scales[(r0 // br, c0 // bc)] = s
            for i in range(blk.shape[0]):
                for j in range(blk.shape[1]):
                    quot = _f32_exact(Fraction(float(blk[i, j])) / Fraction(float(s)))
                    if quot == 0:
                        quot = np.float32(math.copysign(0.0, float(blk[i, j])))
                    q[r0 + i, c0 + j] = _nearest_code(quot)
    return q, scales


@pytest.mark.parametrize("shape,br,bc", [((3, 48), 1, 16), ((5, 40), 2, 16), ((4, 32), 4, 32), ((7, 20), 3, 8)])
def test_block_quant_brute_force(oracle_lib, shape, br, bc):
    rng = np.random.default_rng(sum(shape) + br + bc)
    x = rng.standard_normal(shape) * np.exp2(rng.integers(-8, 8, size=shape))
    x[0, :3] = [0.0, -0.0, 1e-39]
    xb = synth.to_bf16(x)
    q, s = oracle_lib.quant_blocks(xb, br, bc, "rows_major")
    qr, sr = _brute_block_quant(xb, br, bc)
    assert np.array_equal(q, qr)
    for (rb, cb), v in sr.items():
        assert s[rb, cb] == v


def _torch_group_quant(x_bits, gk):
    """Activation groups via torch: IEEE FP32 division and the library's E4M3 cast."""
    x = torch.from_numpy(synth.bf16_bits_to_f32(x_bits).copy())
    M, K = x.shape
    g = x.view(M, K // gk, gk)
    amax = g.abs().amax(dim=2).clamp_min(1e-10)
    s = amax / 448.0
    v = (g / s[:, :, None]).clamp(-448, 448)
    q = v.to(torch.float8_e4m3fn).view(torch.uint8).reshape(M, K)
    return q.numpy(), s.t().contiguous().numpy()


def test_act_group_matches_torch_on_tiny_case(oracle_lib):
    x, _ = synth.tiny_block_case()
    q, s = oracle_lib.quant_act_group(x, 128)
    qt, st = _torch_group_quant(x, 128)
    assert s.shape == (2, 16)
    assert np.array_equal(s, st)
    assert np.array_equal(q, qt)


def test_act_group_matches_torch_wide(oracle_lib):
    x = synth.activations(33, 1024, seed=3, label="pin")
    q, s = oracle_lib.quant_act_group(x, 128)
    qt, st = _torch_group_quant(x, 128)
    assert np.array_equal(s, st) and np.array_equal(q, qt)


def test_weight_block_matches_torch(oracle_lib):
    w = synth.weights(256 + 40, 384, seed=5, label="pin", outlier_rows=3)
    q, s = oracle_lib.quant_weight_block(w, 128, 128)
    wt = torch.from_numpy(synth.bf16_bits_to_f32(w).copy())
    N, K = wt.shape
    assert s.shape == (3, 3)
    for nb in range(3):
        for kb in range(3):
            blk = wt[nb * 128:(nb + 1) * 128, kb * 128:(kb + 1) * 128]
            sc = blk.abs().amax().clamp_min(1e-10) / 448.0
            assert s[nb, kb] == sc.item()
            qt = (blk / sc).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
            assert np.array_equal(q[nb * 128:(nb + 1) * 128, kb * 128:(kb + 1) * 128], qt)


def test_every_block_reaches_448(oracle_lib):
    """amax/fl32(amax/448) rounds to 448, so each non-degenerate block holds a +-448 code."""
    x = synth.activations(40, 512, seed=11, label="pin448")
    q, s = oracle_lib.quant_act_group(x, 128)
    for m in range(40):
        for g in range(4):
            codes = q[m, g * 128:(g + 1) * 128]
            assert np.any((codes & 0x7F) == 0x7E)


def test_quantization_error_bound(oracle_lib):
    """|x - s*dec(q)| <= max(2^-4 |x|, s 2^-10)(1 + 2^-22): half an E4M3 step,
    relative 2^-4 for normals and absolute s*2^-10 in the subnormal range."""
    x = synth.activations(24, 768, seed=12, label="err")
    q, s = oracle_lib.quant_act_group(x, 128)
    xf = synth.bf16_bits_to_f32(x).astype(np.float64)
    dq = E4M3_VALUES[q] * np.repeat(s.T.astype(np.float64), 128, axis=1)
    bound = np.maximum(2.0 ** -4 * np.abs(xf), np.repeat(s.T.astype(np.float64), 128, axis=1) * 2.0 ** -10)
    assert np.all(np.abs(xf - dq) <= bound * (1 + 2.0 ** -22))


def test_symmetric(oracle_lib):
    x = synth.activations(8, 256, seed=13, label="sym")
    neg = x ^ np.uint16(0x8000)
    q1, s1 = oracle_lib.quant_act_group(x, 128)
    q2, s2 = oracle_lib.quant_act_group(neg, 128)
    assert np.array_equal(s1, s2)
    assert np.array_equal(q2, q1 ^ np.uint8(0x80))


def test_outlier_containment(oracle_lib):
    """An outlier only affects its own group: with and without the x50 channels,
    groups that do not hold them get bit-identical scales and codes, while a
    single per-tensor scale changes every code's grid."""
    x_out = synth.activations(16, 1024, seed=0, label="cont", outlier_channels=2, outlier_scale=50.0)
    x_clean = synth.activations(16, 1024, seed=0, label="cont", outlier_channels=0)
    cols = synth.pick(0, "cont/outlier-channels/1024", 1024, 2)
    hit = sorted(set(int(c) // 128 for c in cols))
    q1, s1 = oracle_lib.quant_act_group(x_out, 128)
    q0, s0 = oracle_lib.quant_act_group(x_clean, 128)
    for g in range(8):
        sl = slice(g * 128, (g + 1) * 128)
        if g in hit:
            assert np.all(s1[g] >= s0[g]) and np.median(s1[g] / s0[g]) > 4
        else:
            assert np.array_equal(s1[g], s0[g]) and np.array_equal(q1[:, sl], q0[:, sl])
    _, st1 = oracle_lib.quant_per_tensor(x_out)
    _, st0 = oracle_lib.quant_per_tensor(x_clean)
    assert st1 > 4 * st0


def test_all_zero_group(oracle_lib):
    x = np.zeros((2, 256), dtype=np.uint16)
    x[1, :128] = 0x8000  # -0.0
    q, s = oracle_lib.quant_act_group(x, 128)
    assert np.all(s == np.float32(np.float32(1e-10) / np.float32(448.0)))
    assert np.all(q[0] == 0) and np.all(q[1, :128] == 0x80) and np.all(q[1, 128:] == 0)


def test_special_cases_reduce(oracle_lib):
    """Group = whole row is per-token; block = whole tensor is per-tensor (dynamic)."""
    x = synth.activations(6, 384, seed=21, label="red")
    q_tok, s_tok = oracle_lib.quant_blocks(x, 1, 384, "rows_major")
    for m in range(6):
        q_t, s_t = oracle_lib.quant_per_tensor(x[m:m + 1])
        assert s_tok[m, 0] == s_t and np.array_equal(q_tok[m], q_t[0])
    q_all, s_all = oracle_lib.quant_blocks(x, 6, 384, "rows_major")
    q_t, s_t = oracle_lib.quant_per_tensor(x)
    assert s_all[0, 0] == s_t and np.array_equal(q_all, q_t)
    # static scale equal to the dynamic one gives the same codes
    q_s, s_s = oracle_lib.quant_per_tensor(x, scale=s_t)
    assert np.array_equal(q_s, q_t)


@pytest.mark.parametrize("where", ["first", "last", "interior"])
@pytest.mark.parametrize("sign", [1.0, -1.0])
def test_per_tensor_scale_sees_every_element(oracle_lib, where, sign):
    """The dynamic per-tensor scale is RN32(amax/448) over the whole tensor: a
    single largest element, wherever it lies and whatever its sign, sets it."""
    x = synth.weights(9, 48, seed=31, label="pt-amax", sigma=0.02)
    n = x.size
    pos = {"first": 0, "last": n - 1, "interior": n // 2 + 7}[where]
    flat = x.ravel().copy()
    big = synth.to_bf16(np.array([sign * 3.0625]))[0]  # exact in BF16, far above N(0, 0.02^2)
    flat[pos] = big
    xt = flat.reshape(x.shape)
    q, s = oracle_lib.quant_per_tensor(xt)
    assert s == _f32_exact(Fraction(3.0625) / 448)
    assert q.ravel()[pos] == (0xFE if sign < 0 else 0x7E)
    q_b, s_b = oracle_lib.quant_blocks(xt, 9, 48, "rows_major")
    assert s_b[0, 0] == s and np.array_equal(q_b, q)


def test_ragged_last_block(oracle_lib):
    w = synth.weights(130, 256, seed=2, label="rag")
    q, s = oracle_lib.quant_weight_block(w, 128, 128)
    assert s.shape == (2, 2)
    q2, s2 = oracle_lib.quant_weight_block(np.ascontiguousarray(w[128:]), 128, 128)
    assert np.array_equal(q[128:], q2) and np.array_equal(s[1], s2[0])
