"""Randomised breadth for the oracle's exact pins (hypothesis): block shapes,
scale layouts and values drawn at random, with signed zeros, BF16 subnormals,
values near the BF16 maximum and all-zero blocks among them. The block
quantizer is checked against the exact-rational brute force of
test_oracle_quant.py, and the block-scaled GEMM against exact rational sums.
Neither reference shares arithmetic with the oracle.
"""
from fractions import Fraction

import numpy as np
import pytest

import synth
from test_oracle_gemm import E4M3
from test_oracle_quant import _brute_block_quant

hypothesis = pytest.importorskip("hypothesis")
st = hypothesis.strategies
settings = hypothesis.settings(max_examples=40, deadline=None, derandomize=True)

SPECIAL = [0.0, -0.0, 1e-40, -1e-40, 3.3e38, -3.3e38, 448.0, 464.0, 2.0 ** -10, 1.0]


@st.composite
def bf16_blocks(draw):
    br = draw(st.integers(1, 4))
    bc = draw(st.sampled_from([4, 8, 16]))
    rows = draw(st.integers(1, 3 * br))
    cols = bc * draw(st.integers(1, 3)) + draw(st.sampled_from([0, 0, 3]))  # sometimes a short last block
    seed = draw(st.integers(0, 2 ** 32 - 1))
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((rows, cols)) * np.exp2(rng.integers(-20, 20, size=(rows, cols)))
    for _ in range(draw(st.integers(0, 4))):
        x[rng.integers(rows), rng.integers(cols)] = SPECIAL[rng.integers(len(SPECIAL))]
    if draw(st.booleans()):
        x[:br, :bc] = 0.0  # an all-zero block
    return synth.to_bf16(x), br, bc


@settings
@hypothesis.given(bf16_blocks(), st.sampled_from(["rows_major", "cols_major"]))
def test_block_quant_matches_exact_brute_force(oracle_lib, case, layout):
    xb, br, bc = case
    q, s = oracle_lib.quant_blocks(xb, br, bc, layout)
    qr, sr = _brute_block_quant(xb, br, bc)
    assert np.array_equal(q, qr)
    for (rb, cb), v in sr.items():
        got = s[rb, cb] if layout == "rows_major" else s[cb, rb]
        assert got == v


@st.composite
def gemm_cases(draw):
    g = draw(st.sampled_from([8, 16]))
    M = draw(st.integers(1, 3))
    N = draw(st.integers(1, 9))
    K = g * draw(st.integers(1, 3))
    bn = draw(st.sampled_from([1, 4, 8]))
    seed = draw(st.integers(0, 2 ** 32 - 1))
    rng = np.random.default_rng(seed)

    def codes(shape):
        c = rng.integers(0, 256, size=shape).astype(np.uint8)
        c[(c & 0x7F) == 0x7F] = 0x7E  # no NaN codes
        return c

    qa, qw = codes((M, K)), codes((N, K))
    sa = np.exp2(rng.uniform(-30, 10, size=(K // g, M))).astype(np.float32)
    sw = np.exp2(rng.uniform(-30, 10, size=(-(-N // bn), K // g))).astype(np.float32)
    return qa, sa, qw, sw, g, bn


@settings
@hypothesis.given(gemm_cases())
def test_block_gemm_matches_exact_sums(oracle_lib, case):
    qa, sa, qw, sw, g, bn = case
    y, ab = oracle_lib.gemm_block(qa, sa, qw, sw, gk=g, bn=bn, bk=g)
    M, K = qa.shape
    N = qw.shape[0]
    for m in range(M):
        for n in range(N):
            acc = mag = Fraction(0)
            for k in range(K):
                a = Fraction(float(sa[k // g, m])) * Fraction(float(E4M3[qa[m, k]]))
                b = Fraction(float(sw[n // bn, k // g])) * Fraction(float(E4M3[qw[n, k]]))
                acc += a * b
                mag += abs(a * b)
            # FP64 accumulation of K terms: relative to the magnitude sum
            assert abs(Fraction(y[m, n]) - acc) <= Fraction(K, 2 ** 50) * mag
            assert abs(Fraction(ab[m, n]) - mag) <= Fraction(K, 2 ** 50) * mag
