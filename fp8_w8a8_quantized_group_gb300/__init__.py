"""GB300-native (sm_103a) FP8 W8A8 linear layers.

The computation lives in the CUDA library behind the C ABI of
``include/fp8w8a8.h``; this package is its Python binding (``ops``) and its
in-tree build (``build``). Importing the package does not load the library;
the first call does, and raises if the library is missing.
"""
from .ops import (  # noqa: F401
    Fp8Error,
    block_gemm,
    block_linear,
    fp8_block_gemm,
    fp8_block_linear,
    fp8_device_error,
    fp8_kv_cache_load,
    fp8_kv_cache_store,
    fp8_selftest_bounded_wait,
    fp8_selftest_encode_f32,
    fp8_quant_act_group,
    fp8_quant_act_group_gather,
    fp8_quant_per_tensor,
    fp8_quant_rowwise,
    fp8_quant_weight_block,
    fp8_rowwise_gemm,
    fp8_status_string,
    fp8_tensor_gemm,
    quant_act_group,
    quant_per_tensor,
    quant_rowwise,
    quant_weight_block,
    rowwise_gemm,
    tensor_gemm,
)

GROUP = 128
