"""Python binding of the C ABI: the same names as include/fp8w8a8.h.

Argument marshalling only. Each ``fp8_*`` function takes torch CUDA tensors
(used as device memory), passes their pointers, sizes and the current torch
stream to the library, and raises ``Fp8Error`` on a non-zero status. Every
step of the computation runs in the library's kernels; nothing here computes.

The helpers without the ``fp8_`` prefix allocate the outputs with torch and
call the entry point.
"""
from __future__ import annotations

import ctypes

import torch

from . import _lib

GROUP = 128


class Fp8Error(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        name = _lib.STATUS.get(status, str(status))
        try:
            msg = _lib.load().fp8_status_string(status).decode()
        except Exception:  # pragma: no cover - library missing
            msg = ""
        super().__init__(f"{where}: {name} ({msg})")


def _check(status: int, where: str):
    if status != 0:
        raise Fp8Error(status, where)


def _ptr(t: torch.Tensor | None, dtype: torch.dtype | None = None, what: str = "tensor"):
    if t is None:
        return None
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{what}: expected {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{what}: must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{what}: must be contiguous")
    return t.data_ptr() if t.numel() else None


def _stream(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if isinstance(stream, torch.cuda.Stream) else int(stream)


# ---------------------------------------------------------- C ABI mirror ---

def fp8_quant_act_group(x, q, scales, group_k: int = GROUP, stream=None) -> None:
    M, K = x.shape
    _check(_lib.load().fp8_quant_act_group(_ptr(x, torch.bfloat16, "x"), _ptr(q, torch.uint8, "q"),
                                           _ptr(scales, torch.float32, "scales"), M, K, group_k,
                                           _stream(stream)), "fp8_quant_act_group")


def fp8_quant_weight_block(w, q, scales, block_n: int = GROUP, block_k: int = GROUP, stream=None) -> None:
    N, K = w.shape
    _check(_lib.load().fp8_quant_weight_block(_ptr(w, torch.bfloat16, "w"), _ptr(q, torch.uint8, "q"),
                                              _ptr(scales, torch.float32, "scales"), N, K, block_n, block_k,
                                              _stream(stream)), "fp8_quant_weight_block")


def fp8_quant_per_tensor(x, q, scale, is_static: bool, stream=None) -> None:
    rows, cols = x.shape
    _check(_lib.load().fp8_quant_per_tensor(_ptr(x, torch.bfloat16, "x"), _ptr(q, torch.uint8, "q"),
                                            _ptr(scale, torch.float32, "scale"), rows, cols,
                                            1 if is_static else 0, _stream(stream)), "fp8_quant_per_tensor")


def fp8_block_gemm(qa, sa, qw, sw, y, block_n: int = GROUP, block_k: int = GROUP, group_k: int = GROUP,
                   num_groups: int = 1, group_offsets=None, stream=None) -> None:
    M, K = qa.shape
    N = y.shape[1]
    _check(_lib.load().fp8_block_gemm(_ptr(qa, torch.uint8, "qa"), _ptr(sa, torch.float32, "sa"),
                                      _ptr(qw, torch.uint8, "qw"), _ptr(sw, torch.float32, "sw"),
                                      _ptr(y, torch.bfloat16, "y"), M, N, K, block_n, block_k, group_k,
                                      num_groups, _ptr(group_offsets, torch.int32, "group_offsets"),
                                      _stream(stream)), "fp8_block_gemm")


def fp8_tensor_gemm(qa, sa, qw, sw, y, stream=None) -> None:
    M, K = qa.shape
    N = y.shape[1]
    _check(_lib.load().fp8_tensor_gemm(_ptr(qa, torch.uint8, "qa"), _ptr(sa, torch.float32, "sa"),
                                       _ptr(qw, torch.uint8, "qw"), _ptr(sw, torch.float32, "sw"),
                                       _ptr(y, torch.bfloat16, "y"), M, N, K, _stream(stream)),
           "fp8_tensor_gemm")


def fp8_block_linear(x, qa, sa, qw, sw, y, stream=None) -> None:
    M, K = x.shape
    N = y.shape[1]
    _check(_lib.load().fp8_block_linear(_ptr(x, torch.bfloat16, "x"), _ptr(qa, torch.uint8, "qa"),
                                        _ptr(sa, torch.float32, "sa"), _ptr(qw, torch.uint8, "qw"),
                                        _ptr(sw, torch.float32, "sw"), _ptr(y, torch.bfloat16, "y"), M, N, K,
                                        _stream(stream)), "fp8_block_linear")


def fp8_status_string(status: int) -> str:
    return _lib.load().fp8_status_string(status).decode()


def fp8_selftest_bounded_wait(stream=None) -> None:
    """Launch the bounded-wait self-test kernel (about one second on the device)."""
    _check(_lib.load().fp8_selftest_bounded_wait(_stream(stream)), "fp8_selftest_bounded_wait")


def fp8_device_error(stream=None) -> tuple[int, int]:
    """Synchronise the stream and read-and-clear the device error word: (status, site)."""
    code = ctypes.c_int(0)
    site = ctypes.c_int(0)
    _check(_lib.load().fp8_device_error(_stream(stream), ctypes.byref(code), ctypes.byref(site)),
           "fp8_device_error")
    return code.value, site.value


# ------------------------------------------------------------ helpers ---

def quant_act_group(x: torch.Tensor, stream=None):
    """BF16 [M, K] -> (E4M3 codes uint8 [M, K], scales float32 [K/128, M])."""
    M, K = x.shape
    q = torch.empty((M, K), dtype=torch.uint8, device=x.device)
    s = torch.empty((K // GROUP, M), dtype=torch.float32, device=x.device)
    fp8_quant_act_group(x, q, s, stream=stream)
    return q, s


def quant_weight_block(w: torch.Tensor, stream=None):
    """BF16 [N, K] -> (E4M3 codes uint8 [N, K], scales float32 [ceil(N/128), K/128])."""
    N, K = w.shape
    q = torch.empty((N, K), dtype=torch.uint8, device=w.device)
    s = torch.empty(((N + GROUP - 1) // GROUP, K // GROUP), dtype=torch.float32, device=w.device)
    fp8_quant_weight_block(w, q, s, stream=stream)
    return q, s


def quant_per_tensor(x: torch.Tensor, scale: torch.Tensor | None = None, stream=None):
    """BF16 [R, C] -> (codes, scale float32 [1]); dynamic when scale is None."""
    q = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    if scale is None:
        s = torch.empty(1, dtype=torch.float32, device=x.device)
        fp8_quant_per_tensor(x, q, s, False, stream=stream)
        return q, s
    fp8_quant_per_tensor(x, q, scale, True, stream=stream)
    return q, scale


def block_gemm(qa, sa, qw, sw, group_offsets=None, stream=None) -> torch.Tensor:
    """Block-scaled GEMM -> BF16 [M, N]. Grouped when qw is [E, N, K] with offsets."""
    M = qa.shape[0]
    N = qw.shape[-2]
    y = torch.empty((M, N), dtype=torch.bfloat16, device=qa.device)
    groups = qw.shape[0] if qw.dim() == 3 else 1
    fp8_block_gemm(qa, sa, qw, sw, y, num_groups=groups, group_offsets=group_offsets, stream=stream)
    return y


def block_linear(x, qw, sw, stream=None):
    """BF16 [M, K] x quantized weights -> (Y BF16 [M, N], activation codes, scales)."""
    M, K = x.shape
    N = qw.shape[0]
    qa = torch.empty((M, K), dtype=torch.uint8, device=x.device)
    sa = torch.empty((K // GROUP, M), dtype=torch.float32, device=x.device)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    fp8_block_linear(x, qa, sa, qw, sw, y, stream=stream)
    return y, qa, sa


def tensor_gemm(qa, sa, qw, sw, stream=None) -> torch.Tensor:
    y = torch.empty((qa.shape[0], qw.shape[0]), dtype=torch.bfloat16, device=qa.device)
    fp8_tensor_gemm(qa, sa, qw, sw, y, stream=stream)
    return y
