// FP8 KV cache: store new keys and values into a slot-addressed E4M3 cache
// with per-tensor scales, and gather-and-dequantize cached slots back to BF16.
//
// "[vLLM] FP8" (section "KV 캐시 양자화") keeps the KV cache in FP8 with a
// per-tensor scale for keys and one for values (1.0 when no calibrated scale
// is given); "서빙을 위한 양자화 가이드 FP8, AWQ, GPTQ" (FP8 KV cache) and
// "FP8 Quantization" (section D) give the memory reason. The cache layout is
// this library's reading: slot-major [num_slots][elems] E4M3, where a slot is
// one token's keys (or values) of all KV heads, elems = heads * head_dim, and a
// paged cache addresses slot = block * block_size + offset.
//
// Both kernels are HBM-bound (2 B read + 1 B written per element to store,
// 1 B read + 2 B written to load): a grid-stride loop of CTAs over groups of
// kKvTok token rows, 16-byte BF16 loads and 8-byte code stores (store), 8-byte
// code loads and 16-byte BF16 stores (load). A CTA issues the loads of all
// kKvTok rows before it stores any (the store's loads do not wait for the
// slot; the load's wait only for the kKvTok slot reads, issued together), so
// a thread has 2 kKvTok loads in flight instead of a chain of dependent
// reads per row. Codes are e4m3(fl32(x / scale)) by correctly rounded
// division (quant8; measured faster here than the reciprocal route of the
// other quantizers: 13.9 against 15.4 us for 8192 tokens of 8 x 128 keys and
// values); dequantized values are bf16(fl32(dec(q) * scale)).
#include "quantize.cuh"
#include "launch.h"

namespace fp8k {
namespace {

enum : unsigned { kSiteKvSlot = 401, kSiteKvScale = 402 };

__device__ __forceinline__ bool scale_ok(float s) { return s > 0.0f && s <= 3.402823466e38f; }

constexpr int kKvTok = 4;  // token rows per CTA iteration

// Tokens t0 .. t0 + kKvTok - 1 (t0 = kKvTok * blockIdx.x, grid-stride) of key
// and value [tokens][elems] into slots slots[t] of the caches; slots < 0 are
// padding and skipped, slots at or beyond num_slots are recorded as
// FP8_ERR_ARG and skipped.
__global__ void __launch_bounds__(256, 4) kv_store_kernel(const uint16_t *__restrict__ key, const uint16_t *__restrict__ value,
                                uint8_t *__restrict__ kc, uint8_t *__restrict__ vc,
                                const int64_t *__restrict__ slots, const float *__restrict__ k_scale,
                                const float *__restrict__ v_scale, int64_t tokens, int64_t elems,
                                int64_t num_slots, unsigned *err) {
    grid_dep_wait();
    const float ks = *k_scale, vs = *v_scale;
    if (blockIdx.x == 0 && threadIdx.x == 0 && !(scale_ok(ks) && scale_ok(vs))) record_error(err, kErrArg, kSiteKvScale);
    const int64_t e8 = elems / 8;
    for (int64_t t0 = static_cast<int64_t>(blockIdx.x) * kKvTok; t0 < tokens;
         t0 += static_cast<int64_t>(gridDim.x) * kKvTok) {
        int64_t slot[kKvTok];
#pragma unroll
        for (int u = 0; u < kKvTok; ++u) slot[u] = t0 + u < tokens ? __ldg(slots + t0 + u) : -1;
        for (int64_t j = threadIdx.x; j < e8; j += blockDim.x) {
            uint4 a[kKvTok], b[kKvTok];
#pragma unroll
            for (int u = 0; u < kKvTok; ++u) {
                a[u] = b[u] = make_uint4(0u, 0u, 0u, 0u);
                if (t0 + u < tokens) {
                    a[u] = ld_stream_v4(key + (t0 + u) * elems + j * 8);
                    b[u] = ld_stream_v4(value + (t0 + u) * elems + j * 8);
                }
            }
#pragma unroll
            for (int u = 0; u < kKvTok; ++u) {
                if (slot[u] < 0 || slot[u] >= num_slots) continue;
                *reinterpret_cast<uint2 *>(kc + slot[u] * elems + j * 8) = quant8(a[u], ks);
                *reinterpret_cast<uint2 *>(vc + slot[u] * elems + j * 8) = quant8(b[u], vs);
            }
        }
        if (threadIdx.x == 0) {
#pragma unroll
            for (int u = 0; u < kKvTok; ++u)
                if (slot[u] >= num_slots) record_error(err, kErrArg, kSiteKvSlot);
        }
    }
}

// Four E4M3 codes (memory order) -> their exact values, by the hardware
// conversion to half precision (every E4M3 value is a half value).
__device__ __forceinline__ void dec4(uint32_t w, float (&f)[4]) {
    const __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w & 0xFFFFu), __NV_E4M3);
    const __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w >> 16), __NV_E4M3);
    const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(&lo));
    const float2 b = __half22float2(*reinterpret_cast<const __half2 *>(&hi));
    f[0] = a.x;
    f[1] = a.y;
    f[2] = b.x;
    f[3] = b.y;
}

// Eight codes under scale s -> eight BF16 values bf16(fl32(dec(q) * s)).
__device__ __forceinline__ uint4 dequant8(uint2 c, float s) {
    float a[4], b[4];
    dec4(c.x, a);
    dec4(c.y, b);
    uint4 r;
    r.x = pack_bf16x2(__fmul_rn(a[0], s), __fmul_rn(a[1], s));
    r.y = pack_bf16x2(__fmul_rn(a[2], s), __fmul_rn(a[3], s));
    r.z = pack_bf16x2(__fmul_rn(b[0], s), __fmul_rn(b[1], s));
    r.w = pack_bf16x2(__fmul_rn(b[2], s), __fmul_rn(b[3], s));
    return r;
}

// Row t of the outputs = the dequantized cache slot slots[t] (same skipping
// rules and token grouping as the store; skipped rows are not written).
__global__ void kv_load_kernel(const uint8_t *__restrict__ kc, const uint8_t *__restrict__ vc,
                               uint16_t *__restrict__ key, uint16_t *__restrict__ value,
                               const int64_t *__restrict__ slots, const float *__restrict__ k_scale,
                               const float *__restrict__ v_scale, int64_t tokens, int64_t elems,
                               int64_t num_slots, unsigned *err) {
    grid_dep_wait();
    const float ks = *k_scale, vs = *v_scale;
    if (blockIdx.x == 0 && threadIdx.x == 0 && !(scale_ok(ks) && scale_ok(vs))) record_error(err, kErrArg, kSiteKvScale);
    const int64_t e8 = elems / 8;
    for (int64_t t0 = static_cast<int64_t>(blockIdx.x) * kKvTok; t0 < tokens;
         t0 += static_cast<int64_t>(gridDim.x) * kKvTok) {
        int64_t slot[kKvTok];
#pragma unroll
        for (int u = 0; u < kKvTok; ++u) slot[u] = t0 + u < tokens ? __ldg(slots + t0 + u) : -1;
        for (int64_t j = threadIdx.x; j < e8; j += blockDim.x) {
            uint2 a[kKvTok], b[kKvTok];
#pragma unroll
            for (int u = 0; u < kKvTok; ++u) {
                a[u] = b[u] = make_uint2(0u, 0u);
                if (slot[u] >= 0 && slot[u] < num_slots) {
                    a[u] = __ldg(reinterpret_cast<const uint2 *>(kc + slot[u] * elems + j * 8));
                    b[u] = __ldg(reinterpret_cast<const uint2 *>(vc + slot[u] * elems + j * 8));
                }
            }
#pragma unroll
            for (int u = 0; u < kKvTok; ++u) {
                if (slot[u] < 0 || slot[u] >= num_slots) continue;
                *reinterpret_cast<uint4 *>(key + (t0 + u) * elems + j * 8) = dequant8(a[u], ks);
                *reinterpret_cast<uint4 *>(value + (t0 + u) * elems + j * 8) = dequant8(b[u], vs);
            }
        }
        if (threadIdx.x == 0) {
#pragma unroll
            for (int u = 0; u < kKvTok; ++u)
                if (slot[u] >= num_slots) record_error(err, kErrArg, kSiteKvSlot);
        }
    }
}

// Threads per CTA: one 8-element chunk per thread of a token row, rounded up
// to whole warps, at most 256.
unsigned kv_threads(int64_t elems) {
    const int64_t e8 = elems / 8;
    const int64_t t = ((e8 + 31) / 32) * 32;
    return static_cast<unsigned>(t < 256 ? t : 256);
}

cudaError_t launch_kv(const void *fn, int64_t tokens, int64_t elems, void **args, const DeviceInfo &dev,
                      cudaStream_t stream) {
    const unsigned threads = kv_threads(elems);
    const int64_t cap = static_cast<int64_t>(dev.sm_count) * (2048 / threads);
    const int64_t groups = (tokens + kKvTok - 1) / kKvTok;
    const int64_t grid = groups < cap ? groups : cap;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(threads);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace

cudaError_t launch_kv_store(const void *key, const void *value, void *kc, void *vc, const int64_t *slots,
                            const float *k_scale, const float *v_scale, int64_t tokens, int64_t elems,
                            int64_t num_slots, const DeviceInfo &dev, cudaStream_t stream) {
    if (tokens == 0) return cudaSuccess;
    unsigned *err = dev.err;
    void *args[] = {&key, &value, &kc, &vc, &slots, &k_scale, &v_scale, &tokens, &elems, &num_slots, &err};
    return launch_kv(reinterpret_cast<const void *>(kv_store_kernel), tokens, elems, args, dev, stream);
}

cudaError_t launch_kv_load(const void *kc, const void *vc, void *key, void *value, const int64_t *slots,
                           const float *k_scale, const float *v_scale, int64_t tokens, int64_t elems,
                           int64_t num_slots, const DeviceInfo &dev, cudaStream_t stream) {
    if (tokens == 0) return cudaSuccess;
    unsigned *err = dev.err;
    void *args[] = {&kc, &vc, &key, &value, &slots, &k_scale, &v_scale, &tokens, &elems, &num_slots, &err};
    return launch_kv(reinterpret_cast<const void *>(kv_load_kernel), tokens, elems, args, dev, stream);
}

}  // namespace fp8k
