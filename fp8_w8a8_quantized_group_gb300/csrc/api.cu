// C ABI entry points (include/fp8w8a8.h): argument checks, device checks,
// TMA descriptor encoding and dispatch to the kernels. Nothing here allocates
// device memory or synchronises, except fp8_device_error, whose job is to.
#include <cudaTypedefs.h>

#include <climits>
#include <mutex>

#include "fp8w8a8.h"
#include "launch.h"

namespace fp8k {

// Error word of each device: [0] first status recorded by a kernel, [1] site.
__device__ unsigned g_error_word[2];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
DeviceInfo g_info[kMaxDevices];
int g_state[kMaxDevices];  // 0 = unknown, 1 = usable, otherwise the status to return

bool misaligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) != 0; }

int to_status(cudaError_t e) { return e == cudaSuccess ? FP8_OK : FP8_ERR_CUDA; }

// Device record of the current device; sm_103 only.
int current_device(const DeviceInfo **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return FP8_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return FP8_ERR_DEVICE;
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_state[dev] == 0) {
        int major = 0, minor = 0, sms = 0, smem = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) {
            return FP8_ERR_CUDA;
        }
        if (major != 10 || minor != 3) {
            g_state[dev] = FP8_ERR_DEVICE;
        } else {
            void *err = nullptr;
            if (cudaGetSymbolAddress(&err, g_error_word) != cudaSuccess) return FP8_ERR_CUDA;
            g_info[dev].sm_count = sms;
            g_info[dev].cc_major = major;
            g_info[dev].cc_minor = minor;
            g_info[dev].max_smem_optin = smem;
            g_info[dev].err = static_cast<unsigned *>(err);
            g_state[dev] = 1;
        }
    }
    if (g_state[dev] != 1) return g_state[dev];
    *out = &g_info[dev];
    return FP8_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

// The driver's tensor-map encoder, resolved once.
PFN_cuTensorMapEncodeTiled_v12000 encoder() {
    std::call_once(g_encode_once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess) {
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        }
    });
    return g_encode;
}

}  // namespace

CUresult encode_tma_2d_u8(CUtensorMap *map, const void *base, uint64_t inner, uint64_t rows,
                          uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_rows) {
    if (encoder() == nullptr) return CUDA_ERROR_NOT_SUPPORTED;
    cuuint64_t dims[2] = {inner, rows};
    cuuint64_t strides[1] = {row_stride_bytes};
    cuuint32_t box[2] = {box_inner, box_rows};
    cuuint32_t elem[2] = {1, 1};
    return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, elem,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

CUresult encode_tma_2d_bf16_sw64(CUtensorMap *map, void *base, uint64_t cols, uint64_t rows, uint32_t box_cols,
                                 uint32_t box_rows) {
    if (encoder() == nullptr) return CUDA_ERROR_NOT_SUPPORTED;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 2};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t elem[2] = {1, 1};
    return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, elem,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

}  // namespace fp8k

using fp8k::misaligned;

extern "C" {

int fp8_quant_act_group(const void *x_bf16, void *q_e4m3, float *scales, int64_t M, int64_t K, int group_k,
                        void *stream) {
    if (M < 0 || K < 0) return FP8_ERR_SHAPE;
    if (group_k != FP8_GROUP) return FP8_ERR_UNSUPPORTED;
    if (K == 0 || K % FP8_GROUP != 0 || M > INT_MAX || K > FP8_ACT_GROUP_MAX_K) return FP8_ERR_SHAPE;
    if (M == 0) return FP8_OK;
    if (!x_bf16 || !q_e4m3 || !scales) return FP8_ERR_NULL;
    if (misaligned(x_bf16, 16) || misaligned(q_e4m3, 16) || misaligned(scales, 4)) return FP8_ERR_ALIGN;
    const fp8k::DeviceInfo *dev = nullptr;
    if (int st = fp8k::current_device(&dev)) return st;
    return fp8k::to_status(fp8k::launch_quant_act_group(x_bf16, q_e4m3, scales, M, K, *dev,
                                                        static_cast<cudaStream_t>(stream)));
}

int fp8_quant_act_group_gather(const void *x_bf16, const int32_t *row_index, void *q_e4m3, float *scales, int64_t M,
                               int64_t M_src, int64_t K, int group_k, void *stream) {
    if (M < 0 || K < 0 || M_src < 0) return FP8_ERR_SHAPE;
    if (group_k != FP8_GROUP) return FP8_ERR_UNSUPPORTED;
    if (K == 0 || K % FP8_GROUP != 0 || M > INT_MAX || K > FP8_ACT_GROUP_MAX_K || M_src > INT_MAX)
        return FP8_ERR_SHAPE;
    if (M == 0) return FP8_OK;
    if (M_src == 0) return FP8_ERR_SHAPE;
    if (!x_bf16 || !row_index || !q_e4m3 || !scales) return FP8_ERR_NULL;
    if (misaligned(x_bf16, 16) || misaligned(q_e4m3, 16) || misaligned(scales, 4) || misaligned(row_index, 4))
        return FP8_ERR_ALIGN;
    const fp8k::DeviceInfo *dev = nullptr;
    if (int st = fp8k::current_device(&dev)) return st;
    return fp8k::to_status(fp8k::launch_quant_act_group(x_bf16, q_e4m3, scales, M, K, *dev,
                                                        static_cast<cudaStream_t>(stream), row_index, M_src));
}

int fp8_quant_weight_block(const void *w_bf16, void *q_e4m3, float *scales, int64_t N, int64_t K, int block_n,
                           int block_k, void *stream) {
    if (N < 0 || K < 0) return FP8_ERR_SHAPE;
    if (block_n != FP8_GROUP || block_k != FP8_GROUP) return FP8_ERR_UNSUPPORTED;
    if (K == 0 || K % FP8_GROUP != 0 || N > FP8_WEIGHT_BLOCK_MAX_N || K > INT_MAX) return FP8_ERR_SHAPE;
    if (N == 0) return FP8_OK;
    if (!w_bf16 || !q_e4m3 || !scales) return FP8_ERR_NULL;
    if (misaligned(w_bf16, 16) || misaligned(q_e4m3, 16) || misaligned(scales, 4)) return FP8_ERR_ALIGN;
    const fp8k::DeviceInfo *dev = nullptr;
    if (int st = fp8k::current_device(&dev)) return st;
    return fp8k::to_status(fp8k::launch_quant_weight_block(w_bf16, q_e4m3, scales, N, K, *dev,
                                                           static_cast<cudaStream_t>(stream)));
}

int fp8_quant_per_tensor(const void *x_bf16, void *q_e4m3, float *scale, int64_t rows, int64_t cols,
                         int is_static, void *stream) {
    if (rows < 0 || cols < 0) return FP8_ERR_SHAPE;
    if (cols == 0 || cols % 16 != 0) return FP8_ERR_SHAPE;
    if (rows > (INT64_MAX / 2) / cols) return FP8_ERR_SHAPE;
    if (!scale) return FP8_ERR_NULL;
    if (rows > 0 && (!x_bf16 || !q_e4m3)) return FP8_ERR_NULL;
    if (misaligned(x_bf16, 16) || misaligned(q_e4m3, 16) || misaligned(scale, 4)) return FP8_ERR_ALIGN;
    if (rows == 0 && is_static) return FP8_OK;
    const fp8k::DeviceInfo *dev = nullptr;
    if (int st = fp8k::current_device(&dev)) return st;
    return fp8k::to_status(fp8k::launch_quant_per_tensor(x_bf16, q_e4m3, scale, rows * cols, is_static != 0,
                                                         *dev, static_cast<cudaStream_t>(stream)));
}

int fp8_block_gemm(const void *qa, const float *sa, const void *qw, const float *sw, void *y_bf16, int64_t M,
                   int64_t N, int64_t K, int block_n, int block_k, int group_k, int num_groups,
                   const int32_t *group_offsets, void *stream) {
    if (M < 0 || N < 0 || K < 0) return FP8_ERR_SHAPE;
    if (block_n != FP8_GROUP || block_k != FP8_GROUP || group_k != FP8_GROUP) return FP8_ERR_UNSUPPORTED;
    if (num_groups < 1) return FP8_ERR_ARG;
    if (num_groups > FP8_MAX_GROUPS) return FP8_ERR_UNSUPPORTED;
    if (num_groups > 1 && group_offsets == nullptr) return FP8_ERR_ARG;
    if (K == 0 || K % FP8_GROUP != 0 || N == 0 || N % 16 != 0) return FP8_ERR_SHAPE;
    if (M > INT_MAX || K > INT_MAX || N * static_cast<int64_t>(num_groups) > INT_MAX) return FP8_ERR_SHAPE;
    if (M == 0) return FP8_OK;
    if (!qa || !sa || !qw || !sw || !y_bf16) return FP8_ERR_NULL;
    if (misaligned(qa, 16) || misaligned(qw, 16) || misaligned(y_bf16, 16) || misaligned(sa, 4) ||
        misaligned(sw, 4) || misaligned(group_offsets, 4))
        return FP8_ERR_ALIGN;
    const fp8k::DeviceInfo *dev = nullptr;
    if (int st = fp8k::current_device(&dev)) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (group_offsets == nullptr && M <= 16)
        return fp8k::to_status(fp8k::launch_gemm_decode(qa, sa, qw, sw, y_bf16, M, N, K, fp8k::kScaleBlock, *dev, s));
    return fp8k::to_status(fp8k::launch_gemm_prefill(qa, sa, qw, sw, y_bf16, M, N, K, num_groups, group_offsets,
                                                     fp8k::kScaleBlock, *dev, s));
}

int fp8_tensor_gemm(const void *qa, const float *sa, const void *qw, const float *sw, void *y_bf16, int64_t M,
                    int64_t N, int64_t K, void *stream) {
    if (M < 0 || N < 0 || K < 0) return FP8_ERR_SHAPE;
    if (K == 0 || K % 16 != 0 || N == 0 || N % 16 != 0) return FP8_ERR_SHAPE;
    if (M > INT_MAX || N > INT_MAX || K > INT_MAX) return FP8_ERR_SHAPE;
    if (M == 0) return FP8_OK;
    if (!qa || !sa || !qw || !sw || !y_bf16) return FP8_ERR_NULL;
    if (misaligned(qa, 16) || misaligned(qw, 16) || misaligned(y_bf16, 16) || misaligned(sa, 4) ||
        misaligned(sw, 4))
        return FP8_ERR_ALIGN;
    const fp8k::DeviceInfo *dev = nullptr;
    if (int st = fp8k::current_device(&dev)) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (M <= 16) return fp8k::to_status(fp8k::launch_gemm_decode(qa, sa, qw, sw, y_bf16, M, N, K, fp8k::kScaleTensor, *dev, s));
    return fp8k::to_status(
        fp8k::launch_gemm_prefill(qa, sa, qw, sw, y_bf16, M, N, K, 1, nullptr, fp8k::kScaleTensor, *dev, s));
}

int fp8_block_linear(const void *x_bf16, void *qa, float *sa, const void *qw, const float *sw, void *y_bf16,
                     int64_t M, int64_t N, int64_t K, void *stream) {
    if (M < 0 || N < 0 || K < 0) return FP8_ERR_SHAPE;
    if (K == 0 || K % FP8_GROUP != 0 || N == 0 || N % 16 != 0) return FP8_ERR_SHAPE;
    if (M > INT_MAX || N > INT_MAX || K > FP8_ACT_GROUP_MAX_K) return FP8_ERR_SHAPE;
    if (M == 0) return FP8_OK;
    if (!x_bf16 || !qa || !sa || !qw || !sw || !y_bf16) return FP8_ERR_NULL;
    if (misaligned(x_bf16, 16) || misaligned(qa, 16) || misaligned(qw, 16) || misaligned(y_bf16, 16) ||
        misaligned(sa, 4) || misaligned(sw, 4))
        return FP8_ERR_ALIGN;
    const fp8k::DeviceInfo *dev = nullptr;
    if (int st = fp8k::current_device(&dev)) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = fp8k::launch_quant_act_group(x_bf16, qa, sa, M, K, *dev, s);
    if (e != cudaSuccess) return FP8_ERR_CUDA;
    if (M <= 16) return fp8k::to_status(fp8k::launch_gemm_decode(qa, sa, qw, sw, y_bf16, M, N, K, fp8k::kScaleBlock, *dev, s));
    return fp8k::to_status(fp8k::launch_gemm_prefill(qa, sa, qw, sw, y_bf16, M, N, K, 1, nullptr, fp8k::kScaleBlock, *dev, s));
}

int fp8_quant_rowwise(const void *x_bf16, void *q_e4m3, float *scales, int64_t rows, int64_t cols, void *stream) {
    if (rows < 0 || cols < 0) return FP8_ERR_SHAPE;
    if (cols == 0 || cols % 16 != 0 || rows > INT_MAX || cols > INT_MAX) return FP8_ERR_SHAPE;
    if (rows == 0) return FP8_OK;
    if (!x_bf16 || !q_e4m3 || !scales) return FP8_ERR_NULL;
    if (misaligned(x_bf16, 16) || misaligned(q_e4m3, 16) || misaligned(scales, 4)) return FP8_ERR_ALIGN;
    const fp8k::DeviceInfo *dev = nullptr;
    if (int st = fp8k::current_device(&dev)) return st;
    return fp8k::to_status(
        fp8k::launch_quant_rows(x_bf16, q_e4m3, scales, rows, cols, *dev, static_cast<cudaStream_t>(stream)));
}

int fp8_rowwise_gemm(const void *qa, const float *sa, const void *qw, const float *sw, void *y_bf16, int64_t M,
                     int64_t N, int64_t K, void *stream) {
    if (M < 0 || N < 0 || K < 0) return FP8_ERR_SHAPE;
    if (K == 0 || K % 16 != 0 || N == 0 || N % 16 != 0) return FP8_ERR_SHAPE;
    if (M > INT_MAX || N > INT_MAX || K > INT_MAX) return FP8_ERR_SHAPE;
    if (M == 0) return FP8_OK;
    if (!qa || !sa || !qw || !sw || !y_bf16) return FP8_ERR_NULL;
    if (misaligned(qa, 16) || misaligned(qw, 16) || misaligned(y_bf16, 16) || misaligned(sa, 4) ||
        misaligned(sw, 16))
        return FP8_ERR_ALIGN;
    const fp8k::DeviceInfo *dev = nullptr;
    if (int st = fp8k::current_device(&dev)) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (M <= 16)
        return fp8k::to_status(fp8k::launch_gemm_decode(qa, sa, qw, sw, y_bf16, M, N, K, fp8k::kScaleRowCol, *dev, s));
    return fp8k::to_status(
        fp8k::launch_gemm_prefill(qa, sa, qw, sw, y_bf16, M, N, K, 1, nullptr, fp8k::kScaleRowCol, *dev, s));
}

static int kv_check(const void *a, const void *b, const void *c, const void *d, const int64_t *slots,
                    const float *ks, const float *vs, int64_t tokens, int64_t elems, int64_t num_slots) {
    if (tokens < 0 || elems < 0 || num_slots < 0) return FP8_ERR_SHAPE;
    if (elems == 0 || elems % 16 != 0 || tokens > INT_MAX || elems > INT_MAX) return FP8_ERR_SHAPE;
    if (num_slots > INT64_MAX / elems) return FP8_ERR_SHAPE;
    if (tokens == 0) return FP8_OK;
    if (!a || !b || !c || !d || !slots || !ks || !vs) return FP8_ERR_NULL;
    if (misaligned(a, 16) || misaligned(b, 16) || misaligned(c, 16) || misaligned(d, 16) || misaligned(slots, 8) ||
        misaligned(ks, 4) || misaligned(vs, 4))
        return FP8_ERR_ALIGN;
    return FP8_OK;
}

int fp8_kv_cache_store(const void *key_bf16, const void *value_bf16, void *key_cache, void *value_cache,
                       const int64_t *slot_mapping, const float *k_scale, const float *v_scale, int64_t num_tokens,
                       int64_t token_elems, int64_t num_slots, void *stream) {
    if (int st = kv_check(key_bf16, value_bf16, key_cache, value_cache, slot_mapping, k_scale, v_scale, num_tokens,
                          token_elems, num_slots))
        return st;
    if (num_tokens == 0) return FP8_OK;
    const fp8k::DeviceInfo *dev = nullptr;
    if (int st = fp8k::current_device(&dev)) return st;
    return fp8k::to_status(fp8k::launch_kv_store(key_bf16, value_bf16, key_cache, value_cache, slot_mapping, k_scale,
                                                 v_scale, num_tokens, token_elems, num_slots, *dev,
                                                 static_cast<cudaStream_t>(stream)));
}

int fp8_kv_cache_load(const void *key_cache, const void *value_cache, void *key_bf16, void *value_bf16,
                      const int64_t *slot_mapping, const float *k_scale, const float *v_scale, int64_t num_tokens,
                      int64_t token_elems, int64_t num_slots, void *stream) {
    if (int st = kv_check(key_cache, value_cache, key_bf16, value_bf16, slot_mapping, k_scale, v_scale, num_tokens,
                          token_elems, num_slots))
        return st;
    if (num_tokens == 0) return FP8_OK;
    const fp8k::DeviceInfo *dev = nullptr;
    if (int st = fp8k::current_device(&dev)) return st;
    return fp8k::to_status(fp8k::launch_kv_load(key_cache, value_cache, key_bf16, value_bf16, slot_mapping, k_scale,
                                                v_scale, num_tokens, token_elems, num_slots, *dev,
                                                static_cast<cudaStream_t>(stream)));
}

const char *fp8_status_string(int status) {
    switch (status) {
        case FP8_OK: return "ok";
        case FP8_ERR_NULL: return "a required pointer is NULL";
        case FP8_ERR_SHAPE: return "invalid shape (negative, zero K, or not a required multiple)";
        case FP8_ERR_ALIGN: return "misaligned pointer (data needs 16 bytes, scales 4 bytes)";
        case FP8_ERR_UNSUPPORTED: return "unsupported group/block size or group count";
        case FP8_ERR_ARG: return "invalid argument (num_groups / group_offsets)";
        case FP8_ERR_DEVICE: return "current device is not compute capability 10.3 (sm_103a)";
        case FP8_ERR_CUDA: return "CUDA runtime error";
        case FP8_ERR_TIMEOUT: return "a bounded device-side wait expired";
        default: return "unknown status";
    }
}

int fp8_selftest_bounded_wait(void *stream) {
    const fp8k::DeviceInfo *dev = nullptr;
    if (int st = fp8k::current_device(&dev)) return st;
    return fp8k::to_status(fp8k::launch_selftest_wait(*dev, static_cast<cudaStream_t>(stream)));
}

int fp8_selftest_encode_f32(uint32_t first_bits, int64_t n, void *out_e4m3, void *stream) {
    if (n < 0 || n % 8 != 0) return FP8_ERR_SHAPE;
    if (static_cast<uint64_t>(first_bits) + static_cast<uint64_t>(n) > (uint64_t(1) << 32)) return FP8_ERR_SHAPE;
    if (n == 0) return FP8_OK;
    if (!out_e4m3) return FP8_ERR_NULL;
    if (misaligned(out_e4m3, 16)) return FP8_ERR_ALIGN;
    const fp8k::DeviceInfo *dev = nullptr;
    if (int st = fp8k::current_device(&dev)) return st;
    return fp8k::to_status(
        fp8k::launch_selftest_encode(first_bits, n, out_e4m3, *dev, static_cast<cudaStream_t>(stream)));
}

int fp8_device_error(void *stream, int *out_code, int *out_site) {
    if (!out_code) return FP8_ERR_NULL;
    const fp8k::DeviceInfo *dev = nullptr;
    if (int st = fp8k::current_device(&dev)) return st;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return FP8_ERR_CUDA;
    unsigned word[2] = {0u, 0u};
    const unsigned zero[2] = {0u, 0u};
    if (cudaMemcpyFromSymbol(word, fp8k::g_error_word, sizeof(word)) != cudaSuccess) return FP8_ERR_CUDA;
    if (cudaMemcpyToSymbol(fp8k::g_error_word, zero, sizeof(zero)) != cudaSuccess) return FP8_ERR_CUDA;
    *out_code = static_cast<int>(word[0]);
    if (out_site) *out_site = static_cast<int>(word[1]);
    return FP8_OK;
}

}  // extern "C"
