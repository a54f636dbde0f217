"""CPU oracle for FP8 W8A8 block-scaled linear layers (test infrastructure).

Only the tests, the package smoke check and the benchmark's CPU-baseline leg
import this package. The product path (the CUDA library and its Python binding)
never does; the two share no code. The arithmetic lives in ``fp8_oracle.c``
(plain C, no vector intrinsics, no FMA contraction); this module compiles it
with gcc and wraps it with ctypes, converting numpy arrays to pointers.

What the oracle computes is stated, with the passages it follows, at the top of
``fp8_oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fp8_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

E4M3_MAX = 448.0
AMAX_FLOOR = np.float32(1e-10)


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/liboracle.so`` (gcc, -O2, no fast-math)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
           "-fno-fast-math", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I = ctypes.c_int64
        F = ctypes.c_float
        lib.ora_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.ora_e4m3_decode.restype = ctypes.c_double
        lib.ora_e4m3_encode.argtypes = [F]
        lib.ora_e4m3_encode.restype = ctypes.c_uint8
        lib.ora_e4m3_encode_bits.argtypes = [ctypes.c_uint32, I, P]
        lib.ora_e4m3_encode_bits.restype = None
        lib.ora_quant_blocks.argtypes = [P, I, I, I, I, P, P, I, I]
        lib.ora_quant_blocks.restype = None
        lib.ora_quant_static.argtypes = [P, I, F, P]
        lib.ora_quant_static.restype = None
        lib.ora_tensor_scale.argtypes = [P, I]
        lib.ora_tensor_scale.restype = F
        lib.ora_gemm_block_rows.argtypes = [P, P, I, P, P, I, I, I, I, I, I, I, P, P]
        lib.ora_gemm_block_rows.restype = None
        lib.ora_gemm_block_points.argtypes = [P, P, I, P, P, I, I, I, I, P, P, I, P, P]
        lib.ora_gemm_block_points.restype = None
        lib.ora_gemm_grouped_points.argtypes = [P, P, I, P, P, P, I, I, I, I, I, I, P, P, I, P, P]
        lib.ora_gemm_grouped_points.restype = None
        lib.ora_gemm_tensor_rows.argtypes = [P, F, P, F, I, I, I, I, P, P]
        lib.ora_gemm_tensor_rows.restype = None
        lib.ora_gemm_tensor_points.argtypes = [P, F, P, F, I, P, P, I, P, P]
        lib.ora_gemm_tensor_points.restype = None
        lib.ora_kv_store.argtypes = [P, I, I, P, I, F, P]
        lib.ora_kv_store.restype = None
        lib.ora_kv_load.argtypes = [P, I, I, P, I, F, P]
        lib.ora_kv_load.restype = None
        lib.ora_bf16_from_f32.argtypes = [P, I, P]
        lib.ora_bf16_from_f32.restype = None
        _lib = lib
        return lib


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def _bits16(x: np.ndarray) -> np.ndarray:
    """BF16 input as its uint16 bit patterns (accepts uint16 arrays only)."""
    x = np.ascontiguousarray(x)
    if x.dtype != np.uint16:
        raise TypeError("BF16 inputs are passed as uint16 bit patterns")
    return x


# ------------------------------------------------------------------ E4M3 ---

def e4m3_decode(code: int) -> float:
    """Exact value of one E4M3 code (NaN for 0x7F / 0xFF)."""
    return _load().ora_e4m3_decode(int(code) & 0xFF)


def e4m3_encode(v: float) -> int:
    """E4M3 code of an FP32 value: RNE, saturating to +-448, signed zero kept."""
    return int(_load().ora_e4m3_encode(float(np.float32(v))))


def e4m3_encode_bits(first: int, n: int, out: np.ndarray | None = None) -> np.ndarray:
    """Codes of the n FP32 values with bit patterns first, first + 1, ...
    (first + n <= 2**32), written into out (uint8, contiguous) if given."""
    if not (0 <= first and n >= 0 and first + n <= 1 << 32):
        raise ValueError("bit range outside the 32-bit patterns")
    if out is None:
        out = np.empty(n, dtype=np.uint8)
    if out.dtype != np.uint8 or out.size != n or not out.flags["C_CONTIGUOUS"]:
        raise ValueError("out must be a contiguous uint8 array of n elements")
    if n:
        _load().ora_e4m3_encode_bits(first, n, _ptr(out))
    return out


def e4m3_decode_array(codes: np.ndarray) -> np.ndarray:
    """Decode an array of codes (uses the 256-entry decode of the C oracle)."""
    table = np.array([e4m3_decode(c) for c in range(256)], dtype=np.float64)
    return table[np.asarray(codes, dtype=np.uint8)]


def e4m3_encode_array(v: np.ndarray) -> np.ndarray:
    lib = _load()
    flat = np.asarray(v, dtype=np.float32).ravel()
    out = np.fromiter((lib.ora_e4m3_encode(float(x)) for x in flat), dtype=np.uint8, count=flat.size)
    return out.reshape(np.shape(v))


# ------------------------------------------------------------ quantizers ---

def quant_blocks(x_bf16: np.ndarray, br: int, bc: int, scale_layout: str):
    """Block quantization of a BF16 matrix [rows, cols].

    scale_layout "cols_major" stores the scale of block (rb, cb) at [cb][rb]
    (activation groups: [K/128][M]); "rows_major" at [rb][cb] (weights:
    [N/128][K/128]). Returns (codes uint8 [rows, cols], scales float32 2-D).
    """
    x = _bits16(x_bf16)
    rows, cols = x.shape
    nrb = -(-rows // br)
    ncb = -(-cols // bc)
    q = np.empty((rows, cols), dtype=np.uint8)
    if scale_layout == "cols_major":
        s = np.empty((ncb, nrb), dtype=np.float32)
        strides = (1, nrb)
    elif scale_layout == "rows_major":
        s = np.empty((nrb, ncb), dtype=np.float32)
        strides = (ncb, 1)
    else:
        raise ValueError(scale_layout)
    if rows and cols:
        _load().ora_quant_blocks(_ptr(x), rows, cols, br, bc, _ptr(q), _ptr(s), *strides)
    return q, s


def quant_act_group(x_bf16: np.ndarray, group_k: int = 128):
    """1 x group_k per-token groups; scales [K/group_k][M]."""
    return quant_blocks(x_bf16, 1, group_k, "cols_major")


def quant_weight_block(w_bf16: np.ndarray, block_n: int = 128, block_k: int = 128):
    """block_n x block_k weight blocks; scales [ceil(N/block_n)][K/block_k]."""
    return quant_blocks(w_bf16, block_n, block_k, "rows_major")


def quant_rowwise(x_bf16: np.ndarray):
    """One scale per row (per-token activations, per-channel weights): the
    block quantizer with blocks of 1 x cols. Returns (codes [rows, cols],
    scales float32 [rows])."""
    x = _bits16(x_bf16)
    q, s = quant_blocks(x, 1, max(x.shape[1], 1), "cols_major")
    return q, s.reshape(-1)


def quant_per_tensor(x_bf16: np.ndarray, scale: float | None = None):
    """Per-tensor quantization; dynamic (scale from amax) when scale is None."""
    x = _bits16(x_bf16)
    lib = _load()
    if scale is None:
        scale = np.float32(lib.ora_tensor_scale(_ptr(x), x.size)) if x.size else np.float32(
            float(np.float32(AMAX_FLOOR)) / E4M3_MAX)
    scale = np.float32(scale)
    q = np.empty(x.shape, dtype=np.uint8)
    if x.size:
        lib.ora_quant_static(_ptr(x), x.size, float(scale), _ptr(q))
    return q, scale


# ------------------------------------------------------------------ GEMM ---

def gemm_block(qa, sa, qw, sw, gk=128, bn=128, bk=128, rows=None, with_absdot=True):
    """FP64 dequantize-then-GEMM, block scales. Returns (Y [m1-m0, N], |a||b| sums)."""
    qa = np.ascontiguousarray(qa, dtype=np.uint8)
    qw = np.ascontiguousarray(qw, dtype=np.uint8)
    sa = np.ascontiguousarray(sa, dtype=np.float32)
    sw = np.ascontiguousarray(sw, dtype=np.float32)
    M, K = qa.shape
    N = qw.shape[0]
    m0, m1 = (0, M) if rows is None else rows
    y = np.zeros((m1 - m0, N), dtype=np.float64)
    ab = np.zeros((m1 - m0, N), dtype=np.float64) if with_absdot else None
    if m1 > m0 and N and K:
        _load().ora_gemm_block_rows(_ptr(qa), _ptr(sa), M, _ptr(qw), _ptr(sw), m0, m1, N, K,
                                    gk, bn, bk, _ptr(y), _ptr(ab))
    return y, ab


def gemm_block_points(qa, sa, qw, sw, ms, ns, gk=128, bn=128, bk=128):
    qa = np.ascontiguousarray(qa, dtype=np.uint8)
    qw = np.ascontiguousarray(qw, dtype=np.uint8)
    sa = np.ascontiguousarray(sa, dtype=np.float32)
    sw = np.ascontiguousarray(sw, dtype=np.float32)
    ms = np.ascontiguousarray(ms, dtype=np.int64)
    ns = np.ascontiguousarray(ns, dtype=np.int64)
    M, K = qa.shape
    y = np.zeros(ms.size, dtype=np.float64)
    ab = np.zeros(ms.size, dtype=np.float64)
    if ms.size:
        _load().ora_gemm_block_points(_ptr(qa), _ptr(sa), M, _ptr(qw), _ptr(sw), K, gk, bn, bk,
                                      _ptr(ms), _ptr(ns), ms.size, _ptr(y), _ptr(ab))
    return y, ab


def gemm_grouped_points(qa, sa, qw, sw, offsets, ms, ns, gk=128, bn=128, bk=128):
    """qw [E, N, K], sw [E, ceil(N/bn), K/bk], offsets int32 [E+1]."""
    qa = np.ascontiguousarray(qa, dtype=np.uint8)
    qw = np.ascontiguousarray(qw, dtype=np.uint8)
    sa = np.ascontiguousarray(sa, dtype=np.float32)
    sw = np.ascontiguousarray(sw, dtype=np.float32)
    offsets = np.ascontiguousarray(offsets, dtype=np.int32)
    ms = np.ascontiguousarray(ms, dtype=np.int64)
    ns = np.ascontiguousarray(ns, dtype=np.int64)
    M, K = qa.shape
    E, N, _ = qw.shape
    y = np.zeros(ms.size, dtype=np.float64)
    ab = np.zeros(ms.size, dtype=np.float64)
    if ms.size:
        _load().ora_gemm_grouped_points(_ptr(qa), _ptr(sa), M, _ptr(qw), _ptr(sw), _ptr(offsets),
                                        E, N, K, gk, bn, bk, _ptr(ms), _ptr(ns), ms.size,
                                        _ptr(y), _ptr(ab))
    return y, ab


def gemm_rowwise(qa, sa, qw, sw, rows=None):
    """Per-token activation scales sa [M] and per-channel weight scales sw [N]:
    the block-scaled GEMM with one activation group of all K per row and
    weight blocks of 1 x K. Returns (Y [m1-m0, N], |a||b| sums)."""
    M, K = np.shape(qa)
    N = np.shape(qw)[0]
    sa = np.asarray(sa, dtype=np.float32).reshape(1, M)
    sw = np.asarray(sw, dtype=np.float32).reshape(N, 1)
    return gemm_block(qa, sa, qw, sw, gk=K, bn=1, bk=K, rows=rows)


def gemm_rowwise_points(qa, sa, qw, sw, ms, ns):
    M, K = np.shape(qa)
    N = np.shape(qw)[0]
    sa = np.asarray(sa, dtype=np.float32).reshape(1, M)
    sw = np.asarray(sw, dtype=np.float32).reshape(N, 1)
    return gemm_block_points(qa, sa, qw, sw, ms, ns, gk=K, bn=1, bk=K)


def gemm_tensor(qa, sa, qw, sw, rows=None):
    qa = np.ascontiguousarray(qa, dtype=np.uint8)
    qw = np.ascontiguousarray(qw, dtype=np.uint8)
    M, K = qa.shape
    N = qw.shape[0]
    m0, m1 = (0, M) if rows is None else rows
    y = np.zeros((m1 - m0, N), dtype=np.float64)
    ab = np.zeros((m1 - m0, N), dtype=np.float64)
    if m1 > m0 and N and K:
        _load().ora_gemm_tensor_rows(_ptr(qa), float(np.float32(sa)), _ptr(qw), float(np.float32(sw)),
                                     m0, m1, N, K, _ptr(y), _ptr(ab))
    return y, ab


def gemm_tensor_points(qa, sa, qw, sw, ms, ns):
    qa = np.ascontiguousarray(qa, dtype=np.uint8)
    qw = np.ascontiguousarray(qw, dtype=np.uint8)
    ms = np.ascontiguousarray(ms, dtype=np.int64)
    ns = np.ascontiguousarray(ns, dtype=np.int64)
    K = qa.shape[1]
    y = np.zeros(ms.size, dtype=np.float64)
    ab = np.zeros(ms.size, dtype=np.float64)
    if ms.size:
        _load().ora_gemm_tensor_points(_ptr(qa), float(np.float32(sa)), _ptr(qw), float(np.float32(sw)),
                                       K, _ptr(ms), _ptr(ns), ms.size, _ptr(y), _ptr(ab))
    return y, ab


def tolerance(y_ref: np.ndarray, absdot: np.ndarray) -> np.ndarray:
    """Allowed |gpu - oracle|: 2e-3 * sum_k |a b| + 1e-2 * |oracle|."""
    return 2e-3 * absdot + 1e-2 * np.abs(y_ref)


# -------------------------------------------------------------- KV cache ---

def kv_store(x_bf16: np.ndarray, slots: np.ndarray, cache: np.ndarray, scale: float) -> np.ndarray:
    """Store rows of x [T, E] (BF16 bits) into cache [S, E] (uint8, updated in
    place and returned) at slots [T]; negative or out-of-range slots skipped."""
    x = _bits16(x_bf16)
    slots = np.ascontiguousarray(slots, dtype=np.int64)
    assert cache.dtype == np.uint8 and cache.flags["C_CONTIGUOUS"] and cache.shape[1] == x.shape[1]
    if x.shape[0]:
        _load().ora_kv_store(_ptr(x), x.shape[0], x.shape[1], _ptr(slots), cache.shape[0], float(np.float32(scale)),
                             _ptr(cache))
    return cache


def kv_load(cache: np.ndarray, slots: np.ndarray, out_bf16: np.ndarray, scale: float) -> np.ndarray:
    """Rows of out [T, E] (BF16 bit patterns, uint16, updated in place and
    returned) = cache rows slots[t] dequantized; skipped rows untouched."""
    cache = np.ascontiguousarray(cache, dtype=np.uint8)
    slots = np.ascontiguousarray(slots, dtype=np.int64)
    assert out_bf16.dtype == np.uint16 and out_bf16.flags["C_CONTIGUOUS"] and out_bf16.shape[1] == cache.shape[1]
    if out_bf16.shape[0]:
        _load().ora_kv_load(_ptr(cache), out_bf16.shape[0], out_bf16.shape[1], _ptr(slots), cache.shape[0],
                            float(np.float32(scale)), _ptr(out_bf16))
    return out_bf16


def bf16_from_f32(x: np.ndarray) -> np.ndarray:
    """BF16 bit patterns of FP32 values (round to nearest even)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    if x.size:
        _load().ora_bf16_from_f32(_ptr(x), x.size, _ptr(out))
    return out
