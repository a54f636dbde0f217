"""ctypes loader for the in-tree CUDA library ``_build/libfp8w8a8.so``.

There is no fallback: if the library has not been built, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "libfp8w8a8.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "fp8w8a8.h")

_lock = threading.Lock()
_lib = None

P = ctypes.c_void_p
I64 = ctypes.c_int64
I32 = ctypes.c_int

SIGNATURES = {
    "fp8_quant_act_group": ([P, P, P, I64, I64, I32, P], I32),
    "fp8_quant_act_group_gather": ([P, P, P, P, I64, I64, I64, I32, P], I32),
    "fp8_quant_weight_block": ([P, P, P, I64, I64, I32, I32, P], I32),
    "fp8_quant_per_tensor": ([P, P, P, I64, I64, I32, P], I32),
    "fp8_block_gemm": ([P, P, P, P, P, I64, I64, I64, I32, I32, I32, I32, P, P], I32),
    "fp8_tensor_gemm": ([P, P, P, P, P, I64, I64, I64, P], I32),
    "fp8_block_linear": ([P, P, P, P, P, P, I64, I64, I64, P], I32),
    "fp8_quant_rowwise": ([P, P, P, I64, I64, P], I32),
    "fp8_rowwise_gemm": ([P, P, P, P, P, I64, I64, I64, P], I32),
    "fp8_kv_cache_store": ([P, P, P, P, P, P, P, I64, I64, I64, P], I32),
    "fp8_kv_cache_load": ([P, P, P, P, P, P, P, I64, I64, I64, P], I32),
    "fp8_status_string": ([I32], ctypes.c_char_p),
    "fp8_device_error": ([P, ctypes.POINTER(I32), ctypes.POINTER(I32)], I32),
    "fp8_selftest_bounded_wait": ([P], I32),
    "fp8_selftest_encode_f32": ([ctypes.c_uint32, I64, P, P], I32),
}

STATUS = {0: "FP8_OK", 1: "FP8_ERR_NULL", 2: "FP8_ERR_SHAPE", 3: "FP8_ERR_ALIGN", 4: "FP8_ERR_UNSUPPORTED",
          5: "FP8_ERR_ARG", 6: "FP8_ERR_DEVICE", 7: "FP8_ERR_CUDA", 8: "FP8_ERR_TIMEOUT"}


def header_functions() -> list[str]:
    """Names of the functions declared in include/fp8w8a8.h."""
    text = open(HEADER).read()
    return re.findall(r"^(?:int|const char \*)\s*(fp8_\w+)\s*\(", text, flags=re.M)


def load() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"the FP8 CUDA library is not built ({LIB_PATH} missing); "
                "build it with fp8_w8a8_quantized_group_gb300.build.build()")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (args, res) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
        return lib
