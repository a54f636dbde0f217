"""Failure detection on the GPU without a fault: the bounded-wait self-test
drives a real mbarrier wait to its limit. The expiry must be reported through
the device error word (FP8_ERR_TIMEOUT with the waiting site), the CTA's
other waiter must stop at the abort flag instead of waiting out its own
limit, and the context must stay usable afterwards."""
import time

import numpy as np
import pytest
import torch

import oracle
import synth
from fp8_w8a8_quantized_group_gb300 import build, ops
from helpers import f32_bits, to_dev_bf16

pytestmark = pytest.mark.gpu

FP8_ERR_TIMEOUT = 8
SITE_FIRST, SITE_LATE = 901, 902


@pytest.fixture(scope="module", autouse=True)
def _ready():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build.build()
    oracle.build()


def test_expired_wait_is_reported_and_stops_the_cta():
    code, _ = ops.fp8_device_error()  # nothing pending before the test
    assert code == 0
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    ops.fp8_selftest_bounded_wait()
    code, site = ops.fp8_device_error()  # synchronises, reads and clears
    elapsed = time.perf_counter() - t0
    assert code == FP8_ERR_TIMEOUT, code
    assert site == SITE_FIRST, site  # 902 would mean the late waiter ran out its own limit
    # One wait limit (about 1 s), not the late waiter's 1.5 s: it returned at
    # the abort flag.
    assert 0.9 < elapsed < 1.4, elapsed
    code, site = ops.fp8_device_error()  # the word was cleared by the read
    assert (code, site) == (0, 0)


def test_context_usable_after_an_expired_wait():
    ops.fp8_selftest_bounded_wait()
    assert ops.fp8_device_error()[0] == FP8_ERR_TIMEOUT
    x = synth.activations(16, 512, 0, "failure/X")
    q, s = ops.quant_act_group(to_dev_bf16(x))
    qo, so = oracle.quant_act_group(x)
    assert np.array_equal(q.cpu().numpy(), qo)
    assert np.array_equal(f32_bits(s.cpu().numpy()), f32_bits(so))
    assert ops.fp8_device_error() == (0, 0)


FP8_ERR_ARG = 5


@pytest.mark.parametrize("bad", [0.0, -0.5, float("nan"), float("inf")])
@pytest.mark.parametrize("rows,site", [(8, 302), (2048, 301)])  # small-tensor (one cluster) and multi-kernel paths
def test_bad_static_scale_is_reported(bad, rows, site):
    """A static per-tensor scale must be positive and finite; only the device
    can read it, so a bad one is recorded in the error word."""
    x = synth.device_normal_bf16(rows, 256, 0, "failure/static")
    q = torch.empty((rows, 256), dtype=torch.uint8, device="cuda")
    s = torch.tensor([bad], dtype=torch.float32, device="cuda")
    assert ops.fp8_device_error() == (0, 0)
    ops.fp8_quant_per_tensor(x, q, s, True)
    assert ops.fp8_device_error() == (FP8_ERR_ARG, site)
    ops.fp8_quant_per_tensor(x, q, torch.tensor([0.01], device="cuda"), True)
    assert ops.fp8_device_error() == (0, 0)


@pytest.mark.parametrize("offsets", [[0, 40, 30, 64], [-1, 20, 40, 64], [0, 20, 40, 65], [10, 5, 40, 64]])
def test_bad_group_offsets_are_reported(offsets):
    """Grouped offsets must be non-decreasing within [0, M]; the kernel clamps
    them (no access leaves the buffers) and records FP8_ERR_ARG, site 106."""
    M, N, K, E = 64, 128, 256, 3
    qa = torch.zeros((M, K), dtype=torch.uint8, device="cuda")
    sa = torch.ones((K // 128, M), dtype=torch.float32, device="cuda")
    qw = torch.zeros((E, N, K), dtype=torch.uint8, device="cuda")
    sw = torch.ones((E, N // 128, K // 128), dtype=torch.float32, device="cuda")
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    good = torch.tensor([0, 20, 40, 64], dtype=torch.int32, device="cuda")
    ops.fp8_block_gemm(qa, sa, qw, sw, y, num_groups=E, group_offsets=good)
    assert ops.fp8_device_error() == (0, 0)
    bad = torch.tensor(offsets, dtype=torch.int32, device="cuda")
    ops.fp8_block_gemm(qa, sa, qw, sw, y, num_groups=E, group_offsets=bad)
    assert ops.fp8_device_error() == (FP8_ERR_ARG, 106)
