// Internal launchers (C++ linkage) behind the C ABI in include/fp8w8a8.h.
// Arguments have been validated by the caller; each launcher enqueues work on
// `stream` and returns the cudaError_t of its launches.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace fp8k {

struct DeviceInfo {
    int sm_count;
    int cc_major, cc_minor;
    int max_smem_optin;
    unsigned *err;  // device error word of this device: [0] status, [1] site
};

// Encoder for tiled TMA descriptors (driver entry point, resolved once).
CUresult encode_tma_2d_u8(CUtensorMap *map, const void *base, uint64_t inner, uint64_t rows,
                          uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_rows);

cudaError_t launch_quant_act_group(const void *x, void *q, float *s, int64_t M, int64_t K,
                                   const DeviceInfo &dev, cudaStream_t stream);
cudaError_t launch_quant_weight_block(const void *w, void *q, float *s, int64_t N, int64_t K,
                                      const DeviceInfo &dev, cudaStream_t stream);
cudaError_t launch_quant_per_tensor(const void *x, void *q, float *scale, int64_t n, bool is_static,
                                    const DeviceInfo &dev, cudaStream_t stream);

// Tile-persistent tcgen05 GEMM (M > 16, or grouped). per_tensor: sa, sw point
// to one float each and no per-block promotion is done.
cudaError_t launch_gemm_prefill(const void *qa, const float *sa, const void *qw, const float *sw, void *y,
                                int64_t M, int64_t N, int64_t K, int num_groups, const int32_t *offsets,
                                bool per_tensor, const DeviceInfo &dev, cudaStream_t stream);

// Weight-streaming tcgen05 GEMM for M <= 16 (weights as the MMA's M side).
cudaError_t launch_gemm_decode(const void *qa, const float *sa, const void *qw, const float *sw, void *y,
                               int64_t M, int64_t N, int64_t K, bool per_tensor, const DeviceInfo &dev,
                               cudaStream_t stream);

// One CTA whose waits never complete: the first gives up after the wait limit
// and records FP8_ERR_TIMEOUT (site 901); the second returns at the abort flag.
cudaError_t launch_selftest_wait(const DeviceInfo &dev, cudaStream_t stream);

// The hardware E4M3 conversion of the n FP32 values with bit patterns first,
// first + 1, ... into out (n a multiple of 8, first + n <= 2^32).
cudaError_t launch_selftest_encode(uint32_t first, int64_t n, void *out, const DeviceInfo &dev,
                                   cudaStream_t stream);

}  // namespace fp8k
