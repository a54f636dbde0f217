"""Helpers shared by the GPU parity tests (conversions, tolerance, a second
full-coverage GEMM check in plain PyTorch)."""
from __future__ import annotations

import numpy as np
import torch


def to_dev_bf16(bits: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def f32_bits(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float32)).view(np.uint32)


def assert_within_tolerance(y_gpu: np.ndarray, y_ref: np.ndarray, absdot: np.ndarray, what: str = ""):
    """|gpu - oracle| <= 2e-3 * sum_k |a b| + 1e-2 * |oracle|, element by element."""
    err = np.abs(y_gpu - y_ref)
    tol = 2e-3 * absdot + 1e-2 * np.abs(y_ref)
    bad = err > tol
    if bad.any():
        idx = np.argwhere(bad)[:5]
        flat = [tuple(int(v) for v in i) for i in idx]
        detail = [(i, float(y_gpu[i]), float(y_ref[i]), float(tol[i])) for i in flat]
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} outside tolerance, e.g. {detail}")
    return float((err / np.maximum(tol, 1e-300)).max()) if err.size else 0.0


def decode_e4m3(q: torch.Tensor) -> torch.Tensor:
    return q.view(torch.float8_e4m3fn).float()


@torch.no_grad()
def secondary_block_gemm(qa, sa, qw, sw, rows=None):
    """Plain-PyTorch check of the block-scaled GEMM on the GPU: per 128-wide K
    block an FP32 matmul of decoded codes (products of two E4M3 values are
    exact in FP32; TF32 is off), scaled and summed in FP64.
    Returns (Y, sum |a b|) as float64 tensors for rows [r0, r1)."""
    prev = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = False
    try:
        M, K = qa.shape
        N = qw.shape[0]
        r0, r1 = (0, M) if rows is None else rows
        a = decode_e4m3(qa[r0:r1])
        b = decode_e4m3(qw)
        y = torch.zeros((r1 - r0, N), dtype=torch.float64, device=qa.device)
        mag = torch.zeros_like(y)
        nb_of_col = torch.arange(N, device=qa.device) // 128
        for g in range(K // 128):
            ks = slice(g * 128, (g + 1) * 128)
            part = (a[:, ks] @ b[:, ks].T).double()
            pabs = (a[:, ks].abs() @ b[:, ks].abs().T).double()
            scale = sa[g, r0:r1].double()[:, None] * sw[nb_of_col, g].double()[None, :]
            y += part * scale
            mag += pabs * scale
        return y, mag
    finally:
        torch.backends.cuda.matmul.allow_tf32 = prev


def tile_boundary_rows(M: int, tile: int = 128, limit: int = 48) -> np.ndarray:
    rows = set()
    for m0 in range(0, M, tile):
        rows.update([m0, min(M - 1, m0 + tile - 1)])
    rows = sorted(rows)
    if len(rows) > limit:
        step = len(rows) / limit
        rows = [rows[int(i * step)] for i in range(limit)] + [rows[-1]]
    return np.array(sorted(set(rows)), dtype=np.int64)
