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


CODES = (torch.uint8, torch.float8_e4m3fn)  # E4M3 codes: either dtype, the same bytes


def _need(t: torch.Tensor | None, n: int, what: str) -> None:
    """The entry point reads or writes n elements of t: refuse a smaller buffer
    (the C ABI sees only a pointer and could not tell)."""
    if t is not None and t.numel() < n:
        raise ValueError(f"{what}: has {t.numel()} elements, the call uses {n}")


def _cdiv(a: int, b: int) -> int:
    return -(-a // b) if b > 0 else 0


def _dtype(t: torch.Tensor | None, dtype, what: str) -> None:
    dtypes = dtype if isinstance(dtype, tuple) else (dtype,)
    if t is not None and t.dtype not in dtypes:
        raise TypeError(f"{what}: expected {' or '.join(map(str, dtypes))}, got {t.dtype}")


def _ptr(t: torch.Tensor | None, what: str, device: int | None):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{what}: must be a CUDA tensor")
    if t.device.index != device:
        raise ValueError(f"{what}: on {t.device}, but the current device is cuda:{device}")
    if not t.is_contiguous():
        raise ValueError(f"{what}: must be contiguous")
    return t.data_ptr() if t.numel() else None


def _ptrs(*specs):
    """Pointers of (tensor, dtype, name) triples: dtypes checked first, then
    that each tensor is contiguous on the current CUDA device."""
    for t, dtype, what in specs:
        _dtype(t, dtype, what)
    device = None
    if any(t is not None and t.is_cuda for t, _, _ in specs):
        device = torch.cuda.current_device()
    return [_ptr(t, what, device) for t, _, what in specs]


def _stream(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if isinstance(stream, torch.cuda.Stream) else int(stream)


# ---------------------------------------------------------- C ABI mirror ---
#
# Each function first checks that every buffer holds at least the elements the
# entry point touches for the sizes it is given (M, K from the input's shape,
# N from the output's), then passes the pointers.

def fp8_quant_act_group(x, q, scales, group_k: int = GROUP, stream=None) -> None:
    M, K = x.shape
    _need(q, M * K, "q")
    _need(scales, (K // group_k if group_k > 0 else 0) * M, "scales")
    args = _ptrs((x, torch.bfloat16, "x"), (q, CODES, "q"), (scales, torch.float32, "scales"))
    _check(_lib.load().fp8_quant_act_group(*args, M, K, group_k, _stream(stream)), "fp8_quant_act_group")


def fp8_quant_act_group_gather(x, row_index, q, scales, group_k: int = GROUP, stream=None) -> None:
    """Routed rows: q[m] (and its scales) = the quantization of x[row_index[m]]."""
    M_src, K = x.shape
    M = row_index.shape[0]
    _need(q, M * K, "q")
    _need(scales, (K // group_k if group_k > 0 else 0) * M, "scales")
    xp, ri, qp, sp = _ptrs((x, torch.bfloat16, "x"), (row_index, torch.int32, "row_index"), (q, CODES, "q"),
                           (scales, torch.float32, "scales"))
    _check(_lib.load().fp8_quant_act_group_gather(xp, ri, qp, sp, M, M_src, K, group_k, _stream(stream)),
           "fp8_quant_act_group_gather")


def fp8_quant_weight_block(w, q, scales, block_n: int = GROUP, block_k: int = GROUP, stream=None) -> None:
    N, K = w.shape
    _need(q, N * K, "q")
    _need(scales, _cdiv(N, block_n) * (K // block_k if block_k > 0 else 0), "scales")
    args = _ptrs((w, torch.bfloat16, "w"), (q, CODES, "q"), (scales, torch.float32, "scales"))
    _check(_lib.load().fp8_quant_weight_block(*args, N, K, block_n, block_k, _stream(stream)),
           "fp8_quant_weight_block")


def fp8_quant_per_tensor(x, q, scale, is_static: bool, stream=None) -> None:
    rows, cols = x.shape
    _need(q, rows * cols, "q")
    _need(scale, 1, "scale")
    args = _ptrs((x, torch.bfloat16, "x"), (q, CODES, "q"), (scale, torch.float32, "scale"))
    _check(_lib.load().fp8_quant_per_tensor(*args, rows, cols, 1 if is_static else 0, _stream(stream)),
           "fp8_quant_per_tensor")


def fp8_block_gemm(qa, sa, qw, sw, y, block_n: int = GROUP, block_k: int = GROUP, group_k: int = GROUP,
                   num_groups: int = 1, group_offsets=None, stream=None) -> None:
    M, K = qa.shape
    N = y.shape[1]
    G = max(num_groups, 1)
    _need(sa, _cdiv(K, group_k) * M, "sa")
    _need(qw, G * N * K, "qw")
    _need(sw, G * _cdiv(N, block_n) * _cdiv(K, block_k), "sw")
    _need(y, M * N, "y")
    _need(group_offsets, G + 1, "group_offsets")
    *args, offsets = _ptrs((qa, CODES, "qa"), (sa, torch.float32, "sa"), (qw, CODES, "qw"),
                           (sw, torch.float32, "sw"), (y, torch.bfloat16, "y"),
                           (group_offsets, torch.int32, "group_offsets"))
    _check(_lib.load().fp8_block_gemm(*args, M, N, K, block_n, block_k, group_k, num_groups, offsets,
                                      _stream(stream)), "fp8_block_gemm")


def fp8_tensor_gemm(qa, sa, qw, sw, y, stream=None) -> None:
    M, K = qa.shape
    N = y.shape[1]
    _need(sa, 1, "sa")
    _need(qw, N * K, "qw")
    _need(sw, 1, "sw")
    _need(y, M * N, "y")
    args = _ptrs((qa, CODES, "qa"), (sa, torch.float32, "sa"), (qw, CODES, "qw"), (sw, torch.float32, "sw"),
                 (y, torch.bfloat16, "y"))
    _check(_lib.load().fp8_tensor_gemm(*args, M, N, K, _stream(stream)), "fp8_tensor_gemm")


def fp8_block_linear(x, qa, sa, qw, sw, y, stream=None) -> None:
    M, K = x.shape
    N = y.shape[1]
    _need(qa, M * K, "qa")
    _need(sa, _cdiv(K, GROUP) * M, "sa")
    _need(qw, N * K, "qw")
    _need(sw, _cdiv(N, GROUP) * _cdiv(K, GROUP), "sw")
    _need(y, M * N, "y")
    args = _ptrs((x, torch.bfloat16, "x"), (qa, CODES, "qa"), (sa, torch.float32, "sa"), (qw, CODES, "qw"),
                 (sw, torch.float32, "sw"), (y, torch.bfloat16, "y"))
    _check(_lib.load().fp8_block_linear(*args, M, N, K, _stream(stream)), "fp8_block_linear")


def fp8_quant_rowwise(x, q, scales, stream=None) -> None:
    rows, cols = x.shape
    _need(q, rows * cols, "q")
    _need(scales, rows, "scales")
    args = _ptrs((x, torch.bfloat16, "x"), (q, CODES, "q"), (scales, torch.float32, "scales"))
    _check(_lib.load().fp8_quant_rowwise(*args, rows, cols, _stream(stream)), "fp8_quant_rowwise")


def fp8_rowwise_gemm(qa, sa, qw, sw, y, stream=None) -> None:
    M, K = qa.shape
    N = y.shape[1]
    _need(sa, M, "sa")
    _need(qw, N * K, "qw")
    _need(sw, N, "sw")
    _need(y, M * N, "y")
    args = _ptrs((qa, CODES, "qa"), (sa, torch.float32, "sa"), (qw, CODES, "qw"), (sw, torch.float32, "sw"),
                 (y, torch.bfloat16, "y"))
    _check(_lib.load().fp8_rowwise_gemm(*args, M, N, K, _stream(stream)), "fp8_rowwise_gemm")


def _kv_args(rows_a, rows_b, cache_a, cache_b, slot_mapping, k_scale, v_scale, rows_dtype):
    T, E = rows_a.shape
    S = cache_a.shape[0]
    for t, n, what in ((rows_b, T * E, "value rows"), (cache_b, S * E, "value cache"), (cache_a, S * E, "key cache"),
                       (slot_mapping, T, "slot_mapping"), (k_scale, 1, "k_scale"), (v_scale, 1, "v_scale")):
        _need(t, n, what)
    return T, E, S


def fp8_kv_cache_store(key, value, key_cache, value_cache, slot_mapping, k_scale, v_scale, stream=None) -> None:
    """key, value: BF16 [T, E]; caches: E4M3 [S, E]; slot_mapping: int64 [T]; scales: float32 [1]."""
    T, E, S = _kv_args(key, value, key_cache, value_cache, slot_mapping, k_scale, v_scale, torch.bfloat16)
    args = _ptrs((key, torch.bfloat16, "key"), (value, torch.bfloat16, "value"), (key_cache, CODES, "key_cache"),
                 (value_cache, CODES, "value_cache"), (slot_mapping, torch.int64, "slot_mapping"),
                 (k_scale, torch.float32, "k_scale"), (v_scale, torch.float32, "v_scale"))
    _check(_lib.load().fp8_kv_cache_store(*args, T, E, S, _stream(stream)), "fp8_kv_cache_store")


def fp8_kv_cache_load(key_cache, value_cache, key, value, slot_mapping, k_scale, v_scale, stream=None) -> None:
    """Gather-and-dequantize: key, value (outputs) BF16 [T, E] from the caches' slots."""
    T, E, S = _kv_args(key, value, key_cache, value_cache, slot_mapping, k_scale, v_scale, torch.bfloat16)
    args = _ptrs((key_cache, CODES, "key_cache"), (value_cache, CODES, "value_cache"), (key, torch.bfloat16, "key"),
                 (value, torch.bfloat16, "value"), (slot_mapping, torch.int64, "slot_mapping"),
                 (k_scale, torch.float32, "k_scale"), (v_scale, torch.float32, "v_scale"))
    _check(_lib.load().fp8_kv_cache_load(*args, T, E, S, _stream(stream)), "fp8_kv_cache_load")


def fp8_status_string(status: int) -> str:
    return _lib.load().fp8_status_string(status).decode()


def fp8_selftest_bounded_wait(stream=None) -> None:
    """Launch the bounded-wait self-test kernel (about one second on the device)."""
    _check(_lib.load().fp8_selftest_bounded_wait(_stream(stream)), "fp8_selftest_bounded_wait")


def fp8_selftest_encode_f32(first_bits: int, out, stream=None) -> None:
    """Hardware E4M3 codes of the FP32 values with bit patterns first_bits,
    first_bits + 1, ... into out (one per element; numel a multiple of 8)."""
    (ptr,) = _ptrs((out, CODES, "out"))
    _check(_lib.load().fp8_selftest_encode_f32(first_bits, out.numel(), ptr, _stream(stream)),
           "fp8_selftest_encode_f32")


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


def quant_rowwise(x: torch.Tensor, stream=None):
    """BF16 [R, C] -> (E4M3 codes uint8 [R, C], one scale per row float32 [R])."""
    q = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    s = torch.empty((x.shape[0],), dtype=torch.float32, device=x.device)
    fp8_quant_rowwise(x, q, s, stream=stream)
    return q, s


def rowwise_gemm(qa, sa, qw, sw, stream=None) -> torch.Tensor:
    """Per-token x per-channel scaled GEMM -> BF16 [M, N]."""
    y = torch.empty((qa.shape[0], qw.shape[0]), dtype=torch.bfloat16, device=qa.device)
    fp8_rowwise_gemm(qa, sa, qw, sw, y, stream=stream)
    return y


def tensor_gemm(qa, sa, qw, sw, stream=None) -> torch.Tensor:
    y = torch.empty((qa.shape[0], qw.shape[0]), dtype=torch.bfloat16, device=qa.device)
    fp8_tensor_gemm(qa, sa, qw, sw, y, stream=stream)
    return y
