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
