"""Seeded synthetic inputs for the FP8 W8A8 linear-layer workloads.

This module is shared by the tests, the benchmark and the oracle's callers. It
holds no quantization or GEMM arithmetic: only random-number generation, the
rounding of the generated values to the BF16 input format, and the shapes and
value distributions of the workloads (normal activations with a few outlier
channels, normal weights with a few outlier rows, a uniform top-2 router).

Generator: SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014; the 64-bit finaliser as published by Vigna).
Output i of a stream with seed s is mix(s + (i + 1) * 0x9E3779B97F4A7C15).
Uniforms in (0, 1) are ((z >> 11) + 0.5) * 2^-53; normals use Box-Muller
(both the cosine and the sine branch of each pair). Each named stream gets its
seed from an FNV-1a hash of its label and the workload seed, so that adding a
stream never shifts another.

Rounding to BF16: FP64 -> FP32 (numpy, round to nearest even) -> BF16 (round
to nearest even on the bit pattern). BF16 values travel as uint16 bit patterns.
"""
from __future__ import annotations

import numpy as np

GOLDEN_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22


def _mix(z: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        return z ^ (z >> np.uint64(31))


def splitmix64(seed: int, n: int, start: int = 0) -> np.ndarray:
    """Outputs start .. start+n-1 of the SplitMix64 stream with the given seed."""
    idx = np.arange(start + 1, start + n + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        state = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + idx * GOLDEN_GAMMA
    return _mix(state)


def stream_seed(seed: int, label: str) -> int:
    """64-bit seed of a named stream: FNV-1a over the label, mixed with the workload seed."""
    h = 0xCBF29CE484222325
    for byte in f"{seed}:{label}".encode():
        h ^= byte
        h = (h * 0x100000001B3) & 0xFFFFFFFFFFFFFFFF
    return h


def uniform01(seed: int, n: int, start: int = 0) -> np.ndarray:
    z = splitmix64(seed, n, start)
    return ((z >> np.uint64(11)).astype(np.float64) + 0.5) * (2.0 ** -53)


def normal(seed: int, n: int) -> np.ndarray:
    """n standard normals (Box-Muller over consecutive uniform pairs), chunked."""
    out = np.empty(n, dtype=np.float64)
    pairs = (n + 1) // 2
    done = 0
    while done < pairs:
        c = min(_CHUNK, pairs - done)
        u = uniform01(seed, 2 * c, 2 * done)
        r = np.sqrt(-2.0 * np.log(u[0::2]))
        t = 2.0 * np.pi * u[1::2]
        blk = np.empty(2 * c, dtype=np.float64)
        blk[0::2] = r * np.cos(t)
        blk[1::2] = r * np.sin(t)
        lo = 2 * done
        hi = min(n, lo + 2 * c)
        out[lo:hi] = blk[: hi - lo]
        done += c
    return out


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """FP32 -> BF16 bit patterns, round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    rounding = np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    with np.errstate(over="ignore"):
        return ((u + rounding) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def to_bf16(a: np.ndarray) -> np.ndarray:
    return f32_to_bf16_bits(np.asarray(a, dtype=np.float64).astype(np.float32))


def pick(seed: int, label: str, population: int, count: int) -> np.ndarray:
    """`count` distinct indices of range(population), chosen by the stream `label`."""
    if count <= 0:
        return np.zeros(0, dtype=np.int64)
    u = uniform01(stream_seed(seed, label), population)
    return np.sort(np.argsort(u, kind="stable")[:count]).astype(np.int64)


def activations(M: int, K: int, seed: int = 0, label: str = "X", outlier_channels: int | None = None,
                outlier_frac: float = 0.001, outlier_scale: float = 50.0) -> np.ndarray:
    """BF16 activations [M, K] ~ N(0, 1); `outlier_channels` columns (default
    round(outlier_frac * K)) chosen by the seed are multiplied by `outlier_scale`
    before rounding. The same columns are outliers in every row (channel outliers)."""
    n_out = int(round(outlier_frac * K)) if outlier_channels is None else int(outlier_channels)
    x = normal(stream_seed(seed, f"{label}/values/{M}x{K}"), M * K).reshape(M, K)
    cols = pick(seed, f"{label}/outlier-channels/{K}", K, n_out)
    if cols.size:
        x[:, cols] *= outlier_scale
    return to_bf16(x)


def weights(N: int, K: int, seed: int = 0, label: str = "W", sigma: float = 0.02,
            outlier_rows: int = 0, outlier_scale: float = 20.0) -> np.ndarray:
    """BF16 weights [N, K] ~ N(0, sigma^2); `outlier_rows` rows chosen by the seed
    are multiplied by `outlier_scale` before rounding."""
    w = normal(stream_seed(seed, f"{label}/values/{N}x{K}"), N * K).reshape(N, K) * sigma
    rows = pick(seed, f"{label}/outlier-rows/{N}", N, outlier_rows)
    if rows.size:
        w[rows, :] *= outlier_scale
    return to_bf16(w)


def route_top2(tokens: int, experts: int, seed: int = 0, label: str = "router"):
    """Seeded uniform top-2 router: each token picks 2 distinct experts uniformly.

    Returns (token_of_row int64 [2*tokens], offsets int32 [experts+1]): the
    (token, choice) pairs sorted stably by expert, and where each expert's rows
    start. Row r of the permuted activations is token token_of_row[r].
    """
    u = uniform01(stream_seed(seed, f"{label}/{tokens}x{experts}"), 2 * tokens).reshape(tokens, 2)
    first = np.minimum((u[:, 0] * experts).astype(np.int64), experts - 1)
    second = np.minimum((u[:, 1] * (experts - 1)).astype(np.int64), experts - 2)
    second = second + (second >= first)
    expert_of_pair = np.stack([first, second], axis=1).ravel()
    token_of_pair = np.repeat(np.arange(tokens, dtype=np.int64), 2)
    order = np.argsort(expert_of_pair, kind="stable")
    counts = np.bincount(expert_of_pair, minlength=experts)
    offsets = np.zeros(experts + 1, dtype=np.int32)
    offsets[1:] = np.cumsum(counts)
    return token_of_pair[order], offsets


# ------------------------------------------------------------ workloads ---

LLAMA8B_SHAPES = [(4096, 4096), (6144, 4096), (28672, 4096), (4096, 14336)]
DECODE_M = [1, 4, 16]
PREFILL_M = [2048, 8192]
PER_TENSOR_M = [1, 16, 512, 4096]


def tiny_block_case(seed: int = 0):
    """Tiny block-scaled layer: X [16, 256] ~ N(0,1) with 2 channels x50, W [256, 256] ~ N(0, 0.02^2)."""
    x = activations(16, 256, seed, "tiny/X", outlier_channels=2, outlier_scale=50.0)
    w = weights(256, 256, seed, "tiny/W", sigma=0.02)
    return x, w


def block_case(M: int, N: int, K: int, seed: int = 0):
    """Decode- and prefill-shaped block-scaled layer: X ~ N(0,1) with 0.1% channels x50, W ~ N(0, 0.02^2)."""
    x = activations(M, K, seed, f"block/X/{N}", outlier_frac=0.001, outlier_scale=50.0)
    w = weights(N, K, seed, "block/W", sigma=0.02)
    return x, w


def per_tensor_case(M: int, N: int = 8192, K: int = 8192, seed: int = 0):
    """Per-tensor layer: X ~ N(0,1) with 0.1% channels x100, W ~ N(0, 0.015^2) with 8 rows x20."""
    x = activations(M, K, seed, "tensor/X", outlier_frac=0.001, outlier_scale=100.0)
    w = weights(N, K, seed, "tensor/W", sigma=0.015, outlier_rows=8, outlier_scale=20.0)
    return x, w


def moe_case(tokens: int = 4096, experts: int = 8, N: int = 2048, K: int = 7168, seed: int = 0):
    """MoE layer: X [tokens, K] ~ N(0,1), expert weights [E, N, K] ~ N(0, 0.02^2), top-2 uniform routing.

    Returns (x_perm [2*tokens, K] bf16 rows grouped by expert, w [E, N, K], offsets int32 [E+1])."""
    x = activations(tokens, K, seed, "moe/X", outlier_channels=0)
    token_of_row, offsets = route_top2(tokens, experts, seed)
    w = np.stack([weights(N, K, seed, f"moe/W{e}", sigma=0.02) for e in range(experts)])
    return np.ascontiguousarray(x[token_of_row]), w, offsets


# ------------------------------------------------ device-side generation ---

def device_normal_bf16(rows: int, cols: int, seed: int, label: str, sigma: float = 1.0,
                       outlier_cols=None, outlier_rows=None, outlier_scale: float = 1.0, device="cuda"):
    """Same distributions as `activations` / `weights`, drawn on the GPU with
    torch's seeded Philox generator (for the large benchmark inputs, which no
    oracle reads): N(0, sigma^2) rounded to BF16, the given columns or rows
    multiplied by `outlier_scale` before rounding."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(stream_seed(seed, label) & 0x7FFFFFFFFFFFFFFF)
    x = torch.randn((rows, cols), generator=g, device=device, dtype=torch.float32)
    if sigma != 1.0:
        x.mul_(sigma)
    if outlier_cols is not None and len(outlier_cols):
        x[:, torch.as_tensor(outlier_cols, device=device)] *= outlier_scale
    if outlier_rows is not None and len(outlier_rows):
        x[torch.as_tensor(outlier_rows, device=device), :] *= outlier_scale
    return x.to(torch.bfloat16)
