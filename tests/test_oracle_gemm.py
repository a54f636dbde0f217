"""Pins of the oracle's FP64 dequantize-then-GEMM.

Independent of its arithmetic: exact rational brute force on tiny shapes, a
one-hot closed form, integer-exact cases checked with integer matmul, numpy's
float64 matmul of operands decoded by torch, and the per-tensor / grouped
special cases.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import synth

E4M3 = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def _rand_codes(rng, shape):
    c = rng.integers(0, 256, size=shape).astype(np.uint8)
    c[(c & 0x7F) == 0x7F] = 0x7E  # no NaN codes
    return c


def _dequant(q, scale_of):
    return E4M3[q] * scale_of


@pytest.mark.parametrize("M,N,K,gk,bn,bk", [(3, 5, 32, 16, 16, 16), (4, 33, 48, 16, 16, 16), (2, 8, 64, 32, 4, 32)])
def test_gemm_block_fraction_exact(oracle_lib, M, N, K, gk, bn, bk):
    rng = np.random.default_rng(M * 100 + N)
    qa = _rand_codes(rng, (M, K))
    qw = _rand_codes(rng, (N, K))
    sa = (rng.uniform(0.01, 2, size=(K // gk, M))).astype(np.float32)
    sw = (rng.uniform(0.001, 1, size=(-(-N // bn), K // bk))).astype(np.float32)
    y, ab = oracle_lib.gemm_block(qa, sa, qw, sw, gk=gk, bn=bn, bk=bk)
    for m in range(M):
        for n in range(N):
            acc = Fraction(0)
            mag = Fraction(0)
            for k in range(K):
                a = Fraction(float(sa[k // gk, m])) * Fraction(float(E4M3[qa[m, k]]))
                b = Fraction(float(sw[n // bn, k // bk])) * Fraction(float(E4M3[qw[n, k]]))
                acc += a * b
                mag += abs(a * b)
            assert abs(Fraction(y[m, n]) - acc) <= Fraction(1, 10 ** 12) * (mag + 1)
            assert abs(Fraction(ab[m, n]) - mag) <= Fraction(1, 10 ** 12) * (mag + 1)


def test_gemm_block_one_hot(oracle_lib):
    rng = np.random.default_rng(4)
    M, N, K = 4, 256, 256
    qw = _rand_codes(rng, (N, K))
    sw = rng.uniform(0.01, 1, size=(2, 2)).astype(np.float32)
    qa = np.zeros((M, K), dtype=np.uint8)
    ks = [0, 127, 128, 255]
    codes = [0x38, 0x7E, 0xC1, 0x01]  # 1.0, 448, -2.25 (0xC1: s=1 e=8 m=1), 2^-9
    for m, (k, c) in enumerate(zip(ks, codes)):
        qa[m, k] = c
    sa = rng.uniform(0.5, 2, size=(2, M)).astype(np.float32)
    y, _ = oracle_lib.gemm_block(qa, sa, qw, sw)
    for m, (k, c) in enumerate(zip(ks, codes)):
        expect = (float(sa[k // 128, m]) * E4M3[c]) * (sw[np.arange(N) // 128, k // 128].astype(np.float64) * E4M3[qw[:, k]])
        assert np.array_equal(y[m], expect)


def test_gemm_block_integer_exact(oracle_lib):
    """Scales 1 and small-integer codes: the result is an exact integer."""
    rng = np.random.default_rng(9)
    M, N, K = 8, 128, 256
    ints = np.array([0, 1, 2, 3, 4, 5, 6, 7, 8], dtype=np.int64)
    int_codes = np.array([0x00, 0x38, 0x40, 0x44, 0x48, 0x4A, 0x4C, 0x4E, 0x50], dtype=np.uint8)
    assert np.array_equal(E4M3[int_codes], ints.astype(np.float64))
    ia = rng.integers(0, 9, size=(M, K))
    iw = rng.integers(0, 9, size=(N, K))
    sign_a = rng.choice([1, -1], size=(M, K))
    qa = int_codes[ia] | np.where(sign_a < 0, 0x80, 0).astype(np.uint8)
    qw = int_codes[iw]
    sa = np.ones((K // 128, M), np.float32)
    sw = np.ones((1, K // 128), np.float32)
    y, _ = oracle_lib.gemm_block(qa, sa, qw, sw)
    expect = (ints[ia] * sign_a) @ ints[iw].T
    assert np.array_equal(y, expect.astype(np.float64))


def test_gemm_block_matches_numpy_matmul(oracle_lib):
    x, w = synth.tiny_block_case()
    qa, sa = oracle_lib.quant_act_group(x)
    qw, sw = oracle_lib.quant_weight_block(w)
    y, ab = oracle_lib.gemm_block(qa, sa, qw, sw)
    a = E4M3[qa] * np.repeat(sa.T.astype(np.float64), 128, axis=1)
    b = E4M3[qw] * np.repeat(np.repeat(sw.astype(np.float64), 128, axis=0), 128, axis=1)
    ref = a @ b.T
    mag = np.abs(a) @ np.abs(b).T
    assert np.all(np.abs(y - ref) <= 1e-12 * mag)
    assert np.allclose(ab, mag, rtol=1e-12)
    # and it is close to the unquantized product (accuracy report, not a gate)
    xf = synth.bf16_bits_to_f32(x).astype(np.float64)
    wf = synth.bf16_bits_to_f32(w).astype(np.float64)
    exact = xf @ wf.T
    rel = np.linalg.norm(y - exact) / np.linalg.norm(exact)
    assert rel < 0.1


def test_gemm_points_equal_rows(oracle_lib):
    rng = np.random.default_rng(5)
    M, N, K = 7, 256, 384
    qa = _rand_codes(rng, (M, K))
    qw = _rand_codes(rng, (N, K))
    sa = rng.uniform(0.01, 1, size=(3, M)).astype(np.float32)
    sw = rng.uniform(0.01, 1, size=(2, 3)).astype(np.float32)
    y, ab = oracle_lib.gemm_block(qa, sa, qw, sw)
    ms = rng.integers(0, M, 50)
    ns = rng.integers(0, N, 50)
    yp, abp = oracle_lib.gemm_block_points(qa, sa, qw, sw, ms, ns)
    assert np.array_equal(yp, y[ms, ns]) and np.array_equal(abp, ab[ms, ns])
    ys, _ = oracle_lib.gemm_block(qa, sa, qw, sw, rows=(2, 5))
    assert np.array_equal(ys, y[2:5])


def test_tensor_gemm_is_block_gemm_with_constant_scales(oracle_lib):
    rng = np.random.default_rng(6)
    M, N, K = 5, 256, 256
    qa = _rand_codes(rng, (M, K))
    qw = _rand_codes(rng, (N, K))
    sa, sw = np.float32(0.37), np.float32(0.0021)
    y, ab = oracle_lib.gemm_tensor(qa, sa, qw, sw)
    yb, abb = oracle_lib.gemm_block(qa, np.full((2, M), sa, np.float32), qw, np.full((2, 2), sw, np.float32))
    assert np.array_equal(y, yb) and np.array_equal(ab, abb)
    a = E4M3[qa] * float(sa)
    b = E4M3[qw] * float(sw)
    assert np.allclose(y, a @ b.T, rtol=1e-12, atol=1e-15)
    yp, _ = oracle_lib.gemm_tensor_points(qa, sa, qw, sw, np.array([0, 4]), np.array([3, 255]))
    assert np.array_equal(yp, y[[0, 4], [3, 255]])


def test_grouped_points_follow_expert_ranges(oracle_lib):
    rng = np.random.default_rng(8)
    E, N, K = 3, 128, 256
    offsets = np.array([0, 5, 5, 12], dtype=np.int32)  # expert 1 empty
    M = 14  # rows 12, 13 belong to no expert
    qa = _rand_codes(rng, (M, K))
    sa = rng.uniform(0.01, 1, size=(2, M)).astype(np.float32)
    qw = _rand_codes(rng, (E, N, K))
    sw = rng.uniform(0.01, 1, size=(E, 1, 2)).astype(np.float32)
    ms = np.repeat(np.arange(M), 3)
    ns = np.tile([0, 64, 127], M)
    y, ab = oracle_lib.gemm_grouped_points(qa, sa, qw, sw, offsets, ms, ns)
    for i, (m, n) in enumerate(zip(ms, ns)):
        e = np.searchsorted(offsets, m, side="right") - 1
        if m >= offsets[-1]:
            assert y[i] == 0 and ab[i] == 0
            continue
        yd, _ = oracle_lib.gemm_block_points(qa, sa, qw[e], sw[e], [m], [n])
        assert y[i] == yd[0]
