"""The figures the pages print about storage, decode intensity and the FP8/BF16
peak ratio (tests/golden/page_figures.txt, each with its source), reproduced
from the oracle's quantized layout and from the byte and FLOP model the
benchmark divides by."""
import os

import pytest

import bench
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "page_figures.txt")
DECODE_SHAPES = synth.LLAMA8B_SHAPES


def _figures():
    out = {}
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                k, v = line.split()
                out[k] = float(v)
    return out


F = _figures()


def test_fp8_weights_take_half_the_bf16_bytes(oracle_lib):
    """Codes are one byte per weight and the 128x128 block scales add 4 bytes
    per 16384 weights, so a 70B-parameter model's quantized weights come to the
    page's ~70 GB, against ~140 GB in BF16."""
    w = synth.weights(256, 512, seed=41, label="golden/storage")
    q, s = oracle_lib.quant_weight_block(w)
    n = w.size
    assert w.nbytes / n == F["bf16_weight_bytes_per_param"]
    assert q.nbytes / n == F["fp8_weight_bytes_per_param"]
    per_param = (q.nbytes + s.nbytes) / n
    assert per_param == pytest.approx(1 + 4 / 128 ** 2)
    fp8_gb = per_param * F["dense_model_params"] / 1e9
    bf16_gb = F["bf16_weight_bytes_per_param"] * F["dense_model_params"] / 1e9
    assert fp8_gb == pytest.approx(F["fp8_weights_gb_approx"], rel=0.01)
    assert bf16_gb == pytest.approx(F["bf16_weights_gb_approx"], rel=0.01)


@pytest.mark.parametrize("N,K", DECODE_SHAPES)
def test_batch1_decode_intensity(N, K):
    """At M = 1 a BF16 GEMM moves about 2 bytes per multiply-add (the page's
    ~1 FLOP/byte); the FP8 GEMM's algorithmic bytes, as the benchmark counts
    them, halve that, so its intensity is twice the page's figure."""
    flop = 2 * 1 * N * K
    bf16_bytes = 2 * N * K + 2 * K + 2 * N  # W, x and y in BF16
    assert flop / bf16_bytes == pytest.approx(F["bf16_batch1_decode_flop_per_byte_approx"], rel=0.01)
    fp8 = flop / bench.gemm_bytes(1, N, K)
    assert fp8 == pytest.approx(2 * F["bf16_batch1_decode_flop_per_byte_approx"], rel=0.01)
    assert fp8 < 2.0  # the scales and the activation codes are counted too


def test_fp8_peak_is_twice_bf16():
    """The benchmark's FP8 peak is its measured BF16 peak times the nominal
    dense ratio, which the page's H100 figures give as 2."""
    assert bench.FP8_OVER_BF16 == F["fp8_over_bf16_ratio"]
    assert F["h100_fp8_dense_tflops"] / F["h100_bf16_dense_tflops"] == pytest.approx(F["fp8_over_bf16_ratio"],
                                                                                      rel=0.001)
