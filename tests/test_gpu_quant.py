"""GPU parity of the quantizers against the oracle: codes and scales must be
bit-identical. Calls go through the C ABI (the package's ctypes binding)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from fp8_w8a8_quantized_group_gb300 import build, ops
from helpers import f32_bits, to_dev_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _ready():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build.build()
    oracle.build()


def _act_case(M, K, seed=0):
    return synth.activations(M, K, seed, f"qtest/{M}x{K}")


@pytest.mark.parametrize("M,K", [(16, 256), (1, 4096), (4, 4096), (16, 14336), (17, 384), (129, 1024),
                                 (300, 4096), (2048, 14336), (8192, 4096)])
def test_act_group_bit_exact(M, K):
    x = synth.tiny_block_case()[0] if (M, K) == (16, 256) else _act_case(M, K)
    q, s = ops.quant_act_group(to_dev_bf16(x))
    qo, so = oracle.quant_act_group(x)
    torch.cuda.synchronize()
    assert np.array_equal(f32_bits(s.cpu().numpy()), f32_bits(so))
    assert np.array_equal(q.cpu().numpy(), qo)


@pytest.mark.parametrize("M", [24, 6])  # the general and the decode-sized kernel
def test_act_group_special_values(M):
    rng = np.random.default_rng(3)
    K = 512
    x = synth.to_bf16(rng.standard_normal((M, K)))
    x[0, :] = 0                       # all-zero row: floor scale, +0 codes
    x[1, :128] = 0x8000               # -0.0 group
    x[2, :] = synth.to_bf16(np.full(K, 3.3e38))[0]  # near the BF16 maximum
    x[3, 5] = synth.to_bf16(np.array([1e-40]))[0]   # BF16 subnormal
    x[4, :] = synth.to_bf16(rng.standard_normal(K) * 1e-30)
    x[5, 7] = synth.to_bf16(np.array([-6e4]))[0]
    q, s = ops.quant_act_group(to_dev_bf16(x))
    qo, so = oracle.quant_act_group(x)
    assert np.array_equal(f32_bits(s.cpu().numpy()), f32_bits(so))
    assert np.array_equal(q.cpu().numpy(), qo)


def test_act_group_writes_only_its_outputs():
    M, K = 37, 640
    x = _act_case(M, K, 5)
    q = torch.full((M + 3, K), 0xA5, dtype=torch.uint8, device="cuda")
    s = torch.full((K // 128 * M + 64,), -7.0, dtype=torch.float32, device="cuda")
    ops.fp8_quant_act_group(to_dev_bf16(x), q[:M], s[: K // 128 * M].view(K // 128, M))
    qo, so = oracle.quant_act_group(x)
    assert np.array_equal(q[:M].cpu().numpy(), qo)
    assert torch.all(q[M:] == 0xA5) and torch.all(s[K // 128 * M:] == -7.0)
    assert np.array_equal(f32_bits(s[: K // 128 * M].cpu().numpy()), f32_bits(so.ravel()))


@pytest.mark.parametrize("N,K", [(256, 256), (130, 256), (300, 1024), (4096, 4096), (28672, 4096), (4096, 14336)])
def test_weight_block_bit_exact(N, K):
    w = synth.tiny_block_case()[1] if (N, K) == (256, 256) else synth.weights(N, K, 0, f"qtest/W/{N}x{K}",
                                                                               outlier_rows=3)
    q, s = ops.quant_weight_block(to_dev_bf16(w))
    qo, so = oracle.quant_weight_block(w)
    assert np.array_equal(f32_bits(s.cpu().numpy()), f32_bits(so))
    assert np.array_equal(q.cpu().numpy(), qo)


@pytest.mark.parametrize("rows,cols", [(1, 8192), (16, 8192), (3, 48), (512, 8192), (4096, 8192)])
def test_per_tensor_dynamic_bit_exact(rows, cols):
    x = synth.activations(rows, cols, 0, f"qtest/T/{rows}", outlier_frac=0.001, outlier_scale=100.0)
    q, s = ops.quant_per_tensor(to_dev_bf16(x))
    qo, so = oracle.quant_per_tensor(x)
    assert f32_bits(s.cpu().numpy())[0] == f32_bits(so)
    assert np.array_equal(q.cpu().numpy(), qo)


def test_per_tensor_static_weights():
    w = synth.weights(8192, 8192, 0, "tensor/W", sigma=0.015, outlier_rows=8, outlier_scale=20.0)
    _, so = oracle.quant_per_tensor(w)
    scale = torch.tensor([float(so)], dtype=torch.float32, device="cuda")
    q, s = ops.quant_per_tensor(to_dev_bf16(w), scale=scale)
    qo, _ = oracle.quant_per_tensor(w, scale=so)
    assert np.array_equal(q.cpu().numpy(), qo)
    assert s.item() == float(so)  # a static scale is left unchanged


@pytest.mark.parametrize("scale", [1.0, 3.0, 0.1, 2.0 ** -20, 1e-30, 7.0e10, 1e-40, 3e38])
def test_every_bf16_pattern_through_static_quantization(scale):
    """All 65536 BF16 bit patterns through the static per-tensor quantizer:
    pins the device division and E4M3 conversion (rounding, saturation,
    subnormals, signed zero, infinities) to the oracle's codec. 1e-40 is a
    subnormal scale (its reciprocal overflows: the exact-division fallback),
    3e38 one whose reciprocal is subnormal."""
    x = np.arange(65536, dtype=np.uint32).astype(np.uint16).reshape(4096, 16)
    sc = np.float32(scale)
    q, _ = ops.quant_per_tensor(to_dev_bf16(x), scale=torch.tensor([sc], device="cuda"))
    qo, _ = oracle.quant_per_tensor(x, scale=sc)
    qg = q.cpu().numpy()
    xf = synth.bf16_bits_to_f32(x)
    nan = np.isnan(xf)
    assert np.array_equal(qg[~nan], qo[~nan])
    assert np.all((qg[nan] & 0x7F) == 0x7F)


def _boundary_scales():
    """Scales that put x/s within a few FP32 ulps of E4M3 rounding midpoints for
    many BF16 x (x = a BF16 value, m = an E4M3 midpoint, s = x/m nudged by
    k ulps), plus seeded random scales over many binades."""
    import torch as _t
    vals = _t.arange(256, dtype=_t.int32).to(_t.uint8).view(_t.float8_e4m3fn).to(_t.float64).numpy()[:0x7F]
    mids = (vals[:-1] + vals[1:]) / 2
    rng = np.random.default_rng(11)
    out = []
    for _ in range(12):
        x = float(synth.bf16_bits_to_f32(synth.to_bf16(rng.uniform(0.1, 100.0, 1)))[0])
        m = float(rng.choice(mids[8:]))
        s = np.float32(x / m)
        for k in (-3, -1, 0, 1, 3):
            out.append(float(np.float32(s) + np.float32(k) * np.spacing(np.float32(s))))
    out += [float(v) for v in np.exp2(rng.uniform(-40, 40, 12)).astype(np.float32)]
    return out


@pytest.mark.parametrize("scale", _boundary_scales())
def test_rounding_boundaries_bit_exact(scale):
    """Codes equal the oracle's (correctly rounded division, then E4M3) also when
    x/s falls next to a rounding midpoint."""
    x = np.arange(65536, dtype=np.uint32).astype(np.uint16).reshape(4096, 16)
    keep = ~np.isnan(synth.bf16_bits_to_f32(x))
    sc = np.float32(scale)
    q, _ = ops.quant_per_tensor(to_dev_bf16(x), scale=torch.tensor([sc], device="cuda"))
    qo, _ = oracle.quant_per_tensor(x, scale=sc)
    assert np.array_equal(q.cpu().numpy()[keep], qo[keep])
