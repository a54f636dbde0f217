"""The exact fallback of the reciprocal route, driven on purpose through every
kernel that takes the route: the weight-block, per-tensor (small-tensor and
multi-CTA paths), per-row and decode-sized activation quantizers; the same
near-midpoint inputs also go through the KV cache store (which divides).

The route accepts the code of RN(x lo) when RN(x hi) converts to the same
code (lo, hi = RN(RN(1/s) (1 -+ 2^-21))), and otherwise re-quantizes the
8-value chunk by division. Random data reach that fallback about once per
10^5 values, too rarely to pin it. Here the host repeats the route's float32
arithmetic (numpy rounds to nearest even, like the device) to find BF16 values
x that the bracket leaves undecided for a scale s, and builds inputs full of
them; each test asserts its input holds undecided chunks and that every code
and scale still equals the oracle's (correctly rounded division, then E4M3).
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from fp8_w8a8_quantized_group_gb300 import build, ops
from helpers import f32_bits, to_dev_bf16

pytestmark = pytest.mark.gpu

DOWN = np.float32(1.0 - 2.0 ** -21)
UP = np.float32(1.0 + 2.0 ** -21)


@pytest.fixture(scope="module", autouse=True)
def _ready():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build.build()
    oracle.build()


def _codes(v: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.clip(v, -448.0, 448.0).astype(np.float32))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def _undecided(x: np.ndarray, s: np.float32) -> np.ndarray:
    """Elementwise: the bracket cannot decide x under scale s."""
    with np.errstate(over="ignore", divide="ignore", under="ignore", invalid="ignore"):
        r = np.float32(1.0) / s
        lo, hi = r * DOWN, r * UP
        if not (abs(r) >= np.float32(2.0 ** -126) and np.isfinite(hi)):
            return np.ones(x.shape, dtype=bool)
        return _codes((x * lo).astype(np.float32)) != _codes((x * hi).astype(np.float32))


def _chunks_undecided(x: np.ndarray, s: np.float32) -> int:
    """8-value chunks (along the last axis) with an undecided value."""
    u = _undecided(x.astype(np.float32), s)
    return int(u.reshape(*u.shape[:-1], -1, 8).any(axis=-1).sum())


ALL = synth.bf16_bits_to_f32(np.arange(65536, dtype=np.uint32).astype(np.uint16))
FINITE = np.isfinite(ALL)


def _undecided_values(amax_bits: int) -> np.ndarray:
    """BF16 bit patterns x with |x| <= amax that the bracket leaves undecided
    under the scale a quantizer derives from amax: fl32(amax / 448)."""
    amax = ALL[amax_bits]
    s = np.float32(np.float32(amax) / np.float32(448.0))
    ok = FINITE & (np.abs(ALL) <= amax)
    hit = ok & _undecided(np.where(ok, ALL, 0.0).astype(np.float32), s)
    return np.flatnonzero(hit).astype(np.uint16)


def _amax_with_undecided(rng, count: int, need: int = 16):
    """`count` BF16 amax values, each with at least `need` undecided values
    below it, and those values. amax = 448 c 2^e (c odd) gives the scale
    s = c 2^e exactly, so BF16 values x = m s (m an E4M3 rounding midpoint)
    put x/s exactly on a midpoint, where the bracket must give way."""
    out = []
    while len(out) < count:
        c, e = int(rng.choice(np.arange(1, 36, 2))), int(rng.integers(-12, 3))
        amax = np.float32(448.0 * c * 2.0 ** e)
        bits = int(synth.to_bf16(np.array([amax], dtype=np.float32))[0])
        if ALL[bits] != amax:
            continue
        vals = _undecided_values(bits)
        if vals.size >= need:
            out.append((bits, vals))
    return out


def _fill(amax_bits: int, vals: np.ndarray, n: int, rng) -> np.ndarray:
    """n BF16 patterns: amax first, undecided values at random positions over
    the rest (about a quarter of them), zeros elsewhere."""
    out = np.zeros(n, dtype=np.uint16)
    out[0] = amax_bits
    k = min(n - 1, max(1, n // 4))
    pos = rng.choice(n - 1, size=k, replace=False) + 1
    out[pos] = vals[rng.integers(0, vals.size, k)]
    return out


def _boundary_static_scales(rng, count):
    """Static scales c 2^e (c odd) and one FP32 ulp either side: all BF16
    patterns then put x/s on or next to E4M3 rounding midpoints."""
    out = []
    for _ in range(count):
        s = np.float32(int(rng.choice(np.arange(1, 36, 2))) * 2.0 ** int(rng.integers(-10, 3)))
        out += [s, np.float32(s - np.spacing(s)), np.float32(s + np.spacing(s))]
    return out


def test_static_per_tensor_multi_cta_boundaries():
    """All BF16 patterns, tiled past the small-tensor size, through the
    multi-CTA static quantizer at scales on and next to rounding midpoints."""
    x = np.tile(np.arange(65536, dtype=np.uint32).astype(np.uint16), 4).reshape(4096, 64)
    xf = synth.bf16_bits_to_f32(x)
    keep = ~np.isnan(xf)
    rng = np.random.default_rng(21)
    total = 0
    for s in _boundary_static_scales(rng, 4):
        total += _chunks_undecided(np.where(keep, xf, 0.0), s)
        q, _ = ops.quant_per_tensor(to_dev_bf16(x), scale=torch.tensor([s], device="cuda"))
        qo, _ = oracle.quant_per_tensor(x, scale=s)
        assert np.array_equal(q.cpu().numpy()[keep], qo[keep]), f"scale {s!r}"
    assert total > 0, "no undecided chunk: the fallback was not exercised"


def test_kv_store_boundaries():
    """KV store of all BF16 patterns with per-tensor scales on and next to
    rounding midpoints."""
    T, E = 4096, 16
    key = np.arange(65536, dtype=np.uint32).astype(np.uint16).reshape(T, E)
    value = key[::-1].copy()
    kf, vf = synth.bf16_bits_to_f32(key), synth.bf16_bits_to_f32(value)
    keep_k, keep_v = ~np.isnan(kf), ~np.isnan(vf)
    slots = np.arange(T, dtype=np.int64)[::-1].copy()  # token t -> slot T-1-t
    rng = np.random.default_rng(26)
    scales = _boundary_static_scales(rng, 2)
    total = 0
    for ks, vs in zip(scales, scales[::-1]):
        total += _chunks_undecided(np.where(keep_k, kf, 0.0), ks) + _chunks_undecided(np.where(keep_v, vf, 0.0), vs)
        kc = torch.zeros((T, E), dtype=torch.uint8, device="cuda")
        vc = torch.zeros((T, E), dtype=torch.uint8, device="cuda")
        ops.fp8_kv_cache_store(to_dev_bf16(key), to_dev_bf16(value), kc, vc, torch.from_numpy(slots).cuda(),
                               torch.tensor([ks], device="cuda"), torch.tensor([vs], device="cuda"))
        assert ops.fp8_device_error() == (0, 0)
        kco = oracle.kv_store(key, slots, np.zeros((T, E), np.uint8), ks)
        vco = oracle.kv_store(value, slots, np.zeros((T, E), np.uint8), vs)
        rows_k, rows_v = keep_k[::-1], keep_v[::-1]  # cache row r holds token T-1-r
        assert np.array_equal(kc.cpu().numpy()[rows_k], kco[rows_k]), f"k scale {ks!r}"
        assert np.array_equal(vc.cpu().numpy()[rows_v], vco[rows_v]), f"v scale {vs!r}"
    assert total > 0, "no undecided chunk: the fallback was not exercised"


def test_weight_blocks_undecided():
    """Weight blocks whose amax gives a scale under which a quarter of the
    other values are undecided."""
    rng = np.random.default_rng(22)
    N, K = 384, 512
    picks = _amax_with_undecided(rng, (N // 128) * (K // 128))
    w = np.zeros((N, K), dtype=np.uint16)
    total = 0
    for i, (bits, vals) in enumerate(picks):
        nb, kb = divmod(i, K // 128)
        blk = _fill(bits, vals, 128 * 128, rng).reshape(128, 128)
        w[nb * 128:(nb + 1) * 128, kb * 128:(kb + 1) * 128] = blk
        s = np.float32(np.float32(ALL[bits]) / np.float32(448.0))
        total += _chunks_undecided(synth.bf16_bits_to_f32(blk), s)
    q, sc = ops.quant_weight_block(to_dev_bf16(w))
    qo, so = oracle.quant_weight_block(w)
    assert np.array_equal(f32_bits(sc.cpu().numpy()), f32_bits(so))
    assert np.array_equal(q.cpu().numpy(), qo)
    assert total > 0


@pytest.mark.parametrize("rows,cols", [(24, 1024), (3, 20480)])
def test_rows_undecided(rows, cols):
    """Per-row quantization, rows held in registers (1024) and rows longer
    than the held part (20480, the streaming loop)."""
    rng = np.random.default_rng(23)
    picks = _amax_with_undecided(rng, rows)
    x = np.stack([_fill(b, v, cols, rng) for b, v in picks])
    total = sum(_chunks_undecided(synth.bf16_bits_to_f32(x[r]), np.float32(np.float32(ALL[b]) / np.float32(448.0)))
                for r, (b, _) in enumerate(picks))
    q, s = ops.quant_rowwise(to_dev_bf16(x))
    qo, so = oracle.quant_rowwise(x)
    assert np.array_equal(f32_bits(s.cpu().numpy()), f32_bits(so)) and np.array_equal(q.cpu().numpy(), qo)
    assert total > 0


def test_act_groups_decode_sized_undecided():
    """1 x 128 groups at M <= 16 (the decode-sized kernel): every group's
    amax gives a scale under which a quarter of its values are undecided."""
    rng = np.random.default_rng(24)
    M, K = 16, 1024
    picks = _amax_with_undecided(rng, M * (K // 128))
    x = np.zeros((M, K), dtype=np.uint16)
    total = 0
    for i, (bits, vals) in enumerate(picks):
        m, g = divmod(i, K // 128)
        grp = _fill(bits, vals, 128, rng)
        x[m, g * 128:(g + 1) * 128] = grp
        total += _chunks_undecided(synth.bf16_bits_to_f32(grp), np.float32(np.float32(ALL[bits]) / np.float32(448.0)))
    q, s = ops.quant_act_group(to_dev_bf16(x))
    qo, so = oracle.quant_act_group(x)
    assert np.array_equal(f32_bits(s.cpu().numpy()), f32_bits(so)) and np.array_equal(q.cpu().numpy(), qo)
    assert total > 0


def test_dynamic_per_tensor_multi_cta_undecided():
    """Dynamic per-tensor quantization past the small-tensor size: the tensor's
    amax gives a scale under which a quarter of the values are undecided."""
    rng = np.random.default_rng(25)
    (bits, vals), = _amax_with_undecided(rng, 1, need=64)
    x = _fill(bits, vals, 1 << 18, rng).reshape(1024, 256)
    s = np.float32(np.float32(ALL[bits]) / np.float32(448.0))
    assert _chunks_undecided(synth.bf16_bits_to_f32(x), s) > 0
    q, sc = ops.quant_per_tensor(to_dev_bf16(x))
    qo, so = oracle.quant_per_tensor(x)
    assert np.float32(sc.item()) == so and np.array_equal(q.cpu().numpy(), qo)
