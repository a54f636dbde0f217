"""Accuracy of W8A8 against the unquantized layer, per workload: a report,
not a gate. The measure is the relative Frobenius error
||Y_q - X W^T|| / ||X W^T|| of the oracle's quantized GEMM (which the GPU
matches within the stated tolerance) against the FP64 product of the same
BF16 operands.

Quantization is local to an activation row (1 x 128 groups) and to a 128 x 128
weight block, so whole rows and whole 128-row blocks are sampled instead of
full matrices. For the per-tensor workload the sampled weight rows include an
outlier row, so that the sample's amax is that of the full matrix's
(channel outliers are in every activation row). The asserted bound is only a
sanity check; the printed figures are the report.
"""
import numpy as np
import pytest

import oracle
import synth

ROWS_S = 64   # activation rows sampled from the prefill-shaped and per-tensor workloads
COLS_S = 256  # weight rows sampled: two whole 128-row blocks


def _rel(y: np.ndarray, x_bits: np.ndarray, w_bits: np.ndarray) -> float:
    x = synth.bf16_bits_to_f32(x_bits).astype(np.float64)
    w = synth.bf16_bits_to_f32(w_bits).astype(np.float64)
    exact = x @ w.T
    return float(np.linalg.norm(y - exact) / np.linalg.norm(exact))


def _block(x_bits, w_bits) -> float:
    qa, sa = oracle.quant_act_group(x_bits)
    qw, sw = oracle.quant_weight_block(w_bits)
    y, _ = oracle.gemm_block(qa, sa, qw, sw)
    return _rel(y, x_bits, w_bits)


def _tensor(x_bits, w_bits) -> float:
    qa, sa = oracle.quant_per_tensor(x_bits)
    qw, sw = oracle.quant_per_tensor(w_bits)
    y, _ = oracle.gemm_tensor(qa, sa, qw, sw)
    return _rel(y, x_bits, w_bits)


SHAPES = synth.LLAMA8B_SHAPES


def _cases():
    yield "tiny 16x256x256", lambda: _block(*synth.tiny_block_case())
    for N, K in SHAPES:
        w = lambda N=N, K=K: synth.weights(COLS_S, K, 0, f"acc/W/{N}x{K}", sigma=0.02)  # noqa: E731
        yield f"decode M=16 (N,K)=({N},{K})", lambda w=w, K=K: _block(
            synth.activations(16, K, 0, f"acc/X/{K}"), w())
        yield f"prefill rows (N,K)=({N},{K})", lambda w=w, K=K: _block(
            synth.activations(ROWS_S, K, 1, f"acc/Xp/{K}"), w())
    yield "per-tensor N=K=8192", lambda: _tensor(
        synth.activations(ROWS_S, 8192, 0, "acc/Xt", outlier_scale=100.0),
        synth.weights(COLS_S, 8192, 0, "acc/Wt", sigma=0.015, outlier_rows=1, outlier_scale=20.0))
    yield "MoE expert (N,K)=(2048,7168)", lambda: _block(
        synth.activations(ROWS_S, 7168, 0, "acc/Xm", outlier_channels=0),
        synth.weights(COLS_S, 7168, 0, "acc/Wm", sigma=0.02))


CASES = list(_cases())


@pytest.fixture(scope="module", autouse=True)
def _built():
    oracle.build()


@pytest.mark.parametrize("name,run", CASES, ids=[c[0] for c in CASES])
def test_accuracy_vs_unquantized(name, run):
    rel = run()
    print(f"\n{name}: relative Frobenius error vs unquantized BF16 = {rel:.4f}")
    assert 0.0 < rel < 0.15
