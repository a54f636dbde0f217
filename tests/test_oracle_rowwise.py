"""Pins of the oracle's row-wise scaling: one scale per token for activations
and one per output channel for weights (kFp8DynamicTokenSym on "[vLLM] FP8",
section "스케일링 전략 체계"; channel-wise weight scales on "서빙을 위한 양자화
가이드 FP8, AWQ, GPTQ", section "연산까지 빨라지는 W8A8, FP8").

The oracle reaches both through its block quantizer and block GEMM with
blocks of one row by all of K; these pins check that indexing against
references that do not reuse it: exact rational brute force, torch's IEEE
division and E4M3 cast, numpy's float64 matmul of torch-decoded operands,
and the per-tensor special case.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import synth
from test_oracle_quant import _brute_block_quant

E4M3 = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()


@pytest.mark.parametrize("rows,cols", [(1, 16), (5, 48), (3, 80)])
def test_quant_rowwise_brute_force(oracle_lib, rows, cols):
    rng = np.random.default_rng(rows * 7 + cols)
    x = rng.standard_normal((rows, cols)) * np.exp2(rng.integers(-6, 6, size=(rows, cols)))
    x[0, :2] = [-0.0, 3e-39]
    if rows > 2:
        x[2, :] = 0.0  # an all-zero row takes the floor scale
    xb = synth.to_bf16(x)
    q, s = oracle_lib.quant_rowwise(xb)
    qr, sr = _brute_block_quant(xb, 1, cols)
    assert np.array_equal(q, qr)
    assert s.shape == (rows,)
    for r in range(rows):
        assert s[r] == sr[(r, 0)]


def test_quant_rowwise_matches_torch_division_and_cast(oracle_lib):
    """Per row: s = RN32(amax / 448) (IEEE float32 division in torch), codes =
    torch's float8_e4m3fn cast of the IEEE float32 quotient x / s."""
    x = synth.activations(37, 1040, 3, "rowwise/X", outlier_channels=3, outlier_scale=50.0)
    q, s = oracle_lib.quant_rowwise(x)
    xt = torch.from_numpy(synth.bf16_bits_to_f32(x))
    amax = xt.abs().amax(dim=1).clamp_min(torch.tensor(1e-10, dtype=torch.float32))
    st = amax / torch.tensor(448.0, dtype=torch.float32)
    qt = (xt / st[:, None]).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(s.view(np.uint32), st.numpy().view(np.uint32))
    assert np.array_equal(q, qt)


def test_quant_rowwise_outliers_stay_in_their_rows(oracle_lib):
    """A row's scale depends on that row only: scaling one row by 1000 leaves
    every other row's codes and scale unchanged."""
    x = synth.activations(8, 256, 4, "rowwise/contain", outlier_channels=0)
    q0, s0 = oracle_lib.quant_rowwise(x)
    xf = synth.bf16_bits_to_f32(x).astype(np.float64)
    xf[3] *= 1000.0
    q1, s1 = oracle_lib.quant_rowwise(synth.to_bf16(xf))
    others = [r for r in range(8) if r != 3]
    assert np.array_equal(q0[others], q1[others]) and np.array_equal(s0[others], s1[others])
    assert s1[3] > 500 * s0[3]


@pytest.mark.parametrize("M,N,K", [(2, 3, 16), (3, 5, 48)])
def test_gemm_rowwise_fraction_exact(oracle_lib, M, N, K):
    rng = np.random.default_rng(M + 10 * N + K)
    qa = rng.integers(0, 256, size=(M, K)).astype(np.uint8)
    qw = rng.integers(0, 256, size=(N, K)).astype(np.uint8)
    qa[(qa & 0x7F) == 0x7F] = 0x7E
    qw[(qw & 0x7F) == 0x7F] = 0x7E
    sa = rng.uniform(0.01, 2, size=M).astype(np.float32)
    sw = rng.uniform(0.001, 1, size=N).astype(np.float32)
    y, ab = oracle_lib.gemm_rowwise(qa, sa, qw, sw)
    for m in range(M):
        for n in range(N):
            dot = sum(Fraction(float(E4M3[qa[m, k]])) * Fraction(float(E4M3[qw[n, k]])) for k in range(K))
            mag = sum(abs(Fraction(float(E4M3[qa[m, k]])) * Fraction(float(E4M3[qw[n, k]]))) for k in range(K))
            exact = Fraction(float(sa[m])) * Fraction(float(sw[n])) * dot
            emag = Fraction(float(sa[m])) * Fraction(float(sw[n])) * mag
            assert abs(Fraction(y[m, n]) - exact) <= Fraction(1, 10 ** 12) * (emag + 1)
            assert abs(Fraction(ab[m, n]) - emag) <= Fraction(1, 10 ** 12) * (emag + 1)


def test_gemm_rowwise_matches_numpy_matmul(oracle_lib):
    rng = np.random.default_rng(9)
    M, N, K = 9, 40, 272
    x = synth.activations(M, K, 9, "rowwise/gx")
    w = synth.weights(N, K, 9, "rowwise/gw")
    qa, sa = oracle_lib.quant_rowwise(x)
    qw, sw = oracle_lib.quant_rowwise(w)
    y, _ = oracle_lib.gemm_rowwise(qa, sa, qw, sw)
    ref = (E4M3[qa] * sa.astype(np.float64)[:, None]) @ (E4M3[qw] * sw.astype(np.float64)[:, None]).T
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())
    ms = rng.integers(0, M, 50)
    ns = rng.integers(0, N, 50)
    yp, _ = oracle_lib.gemm_rowwise_points(qa, sa, qw, sw, ms, ns)
    assert np.array_equal(yp, y[ms, ns])


def test_gemm_rowwise_uniform_scales_is_per_tensor(oracle_lib):
    rng = np.random.default_rng(2)
    M, N, K = 4, 24, 96
    qa = rng.integers(0, 0x7E, size=(M, K)).astype(np.uint8)
    qw = rng.integers(0, 0x7E, size=(N, K)).astype(np.uint8) | 0x80
    y, ab = oracle_lib.gemm_rowwise(qa, np.full(M, 0.25, np.float32), qw, np.full(N, 0.5, np.float32))
    yt, abt = oracle_lib.gemm_tensor(qa, np.float32(0.25), qw, np.float32(0.5))
    assert np.allclose(y, yt, rtol=1e-14, atol=0) and np.allclose(ab, abt, rtol=1e-14, atol=0)
