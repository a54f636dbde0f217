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
// BF16 [rows][cols] (row stride cols * 2 bytes), boxes of box_cols x box_rows
// with 64-byte swizzling (box_cols = 32): the prefill GEMM's output stores.
CUresult encode_tma_2d_bf16_sw64(CUtensorMap *map, void *base, uint64_t cols, uint64_t rows, uint32_t box_cols,
                                 uint32_t box_rows);

// 1x128 activation groups. row_index (device int32 [M], or nullptr): row m of
// q / s is quantized from row row_index[m] of x [M_src][K] (M_src = M without).
cudaError_t launch_quant_act_group(const void *x, void *q, float *s, int64_t M, int64_t K,
                                   const DeviceInfo &dev, cudaStream_t stream,
                                   const int32_t *row_index = nullptr, int64_t M_src = 0);
cudaError_t launch_quant_weight_block(const void *w, void *q, float *s, int64_t N, int64_t K,
                                      const DeviceInfo &dev, cudaStream_t stream);
// One scale per row of x [rows][cols] (per-token activations, per-channel weights).
cudaError_t launch_quant_rows(const void *x, void *q, float *s, int64_t rows, int64_t cols, const DeviceInfo &dev,
                              cudaStream_t stream);
cudaError_t launch_quant_per_tensor(const void *x, void *q, float *scale, int64_t n, bool is_static,
                                    const DeviceInfo &dev, cudaStream_t stream);

// How a GEMM applies the scales:
//  kScaleBlock   sa [K/128][M], sw [ceil(N/128)][K/128]: promoted per 128-wide K block;
//  kScaleTensor  sa, sw one float each: all of K accumulated, one product at the end;
//  kScaleRowCol  sa [M] (per token), sw [N] (per output channel): all of K
//                accumulated, Y[m,n] scaled by sa[m] * sw[n] at the end.
enum ScaleMode : int { kScaleBlock = 0, kScaleTensor = 1, kScaleRowCol = 2 };

// FP8 KV cache: quantize rows of key/value [tokens][elems] into cache slots
// (store) or dequantize cache slots into rows (load), per-tensor scales.
cudaError_t launch_kv_store(const void *key, const void *value, void *kc, void *vc, const int64_t *slots,
                            const float *k_scale, const float *v_scale, int64_t tokens, int64_t elems,
                            int64_t num_slots, const DeviceInfo &dev, cudaStream_t stream);
cudaError_t launch_kv_load(const void *kc, const void *vc, void *key, void *value, const int64_t *slots,
                           const float *k_scale, const float *v_scale, int64_t tokens, int64_t elems,
                           int64_t num_slots, const DeviceInfo &dev, cudaStream_t stream);

// Tile-persistent tcgen05 GEMM (M > 16, or grouped; grouped only with kScaleBlock).
cudaError_t launch_gemm_prefill(const void *qa, const float *sa, const void *qw, const float *sw, void *y,
                                int64_t M, int64_t N, int64_t K, int num_groups, const int32_t *offsets,
                                ScaleMode mode, const DeviceInfo &dev, cudaStream_t stream);

// Weight-streaming tcgen05 GEMM for M <= 16 (weights as the MMA's M side).
cudaError_t launch_gemm_decode(const void *qa, const float *sa, const void *qw, const float *sw, void *y,
                               int64_t M, int64_t N, int64_t K, ScaleMode mode, const DeviceInfo &dev,
                               cudaStream_t stream);

// One CTA whose waits never complete: the first gives up after the wait limit
// and records FP8_ERR_TIMEOUT (site 901); the second returns at the abort flag.
cudaError_t launch_selftest_wait(const DeviceInfo &dev, cudaStream_t stream);

// The hardware E4M3 conversion of the n FP32 values with bit patterns first,
// first + 1, ... into out (n a multiple of 8, first + n <= 2^32).
cudaError_t launch_selftest_encode(uint32_t first, int64_t n, void *out, const DeviceInfo &dev,
                                   cudaStream_t stream);

}  // namespace fp8k
