// The numeric steps every quantizer uses (scales, packed amax, E4M3 codes by
// division or by the reciprocal bracket, 16-byte streaming loads, and the
// lane-quad 1 x 128 group), shared by quant.cu and kv_cache.cu. sm_103a only.
#pragma once

#include "common.cuh"

namespace fp8k {

// --------------------------------------------------------------- numerics --

// Smallest amax that forms a scale, so an all-zero group still gets a finite
// scale (the pages do not say what an all-zero block does; this is the reading).
constexpr float kAmaxFloor = 1e-10f;
// Largest finite E4M3 magnitude (format table: range +-448).
constexpr float kE4M3Max = 448.0f;

// Scale of a block from its amax: fl32(max(amax, floor) / 448), IEEE division.
__device__ __forceinline__ float block_scale(float amax) {
    return __fdiv_rn(fmaxf(amax, kAmaxFloor), kE4M3Max);
}

// Two E4M3 codes (low byte = a, high byte = b) of a/s and b/s: correctly
// rounded FP32 quotients, then the hardware's round-to-nearest-even,
// saturating conversion.
__device__ __forceinline__ uint16_t quant_pair(float a, float b, float s) {
    float2 v = make_float2(__fdiv_rn(a, s), __fdiv_rn(b, s));
    return static_cast<uint16_t>(__nv_cvt_float2_to_fp8x2(v, __NV_SATFINITE, __NV_E4M3));
}

// BF16 pair packed in a 32-bit word -> the two FP32 values (exact).
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Packed BF16 maximum (maxNum: a NaN operand is ignored, as by fmaxf; exact).
__device__ __forceinline__ uint32_t bf16x2_max(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// Running packed amax: m (two BF16 lanes, start at 0) takes the magnitudes
// of the 8 BF16 values in v; amax_of(m) is the amax so far as a float.
__device__ __forceinline__ void amax8_acc(uint32_t &m, const uint4 &v) {
    constexpr uint32_t kAbs = 0x7FFF7FFFu;
    m = bf16x2_max(m, bf16x2_max(bf16x2_max(v.x & kAbs, v.y & kAbs), bf16x2_max(v.z & kAbs, v.w & kAbs)));
}

__device__ __forceinline__ float amax_of(uint32_t m) { return fmaxf(bf16lo(m), bf16hi(m)); }

// 8 E4M3 codes of the 8 BF16 values in v under scale s, in memory order.
__device__ __forceinline__ uint2 quant8(const uint4 &v, float s) {
    uint2 r;
    r.x = static_cast<uint32_t>(quant_pair(bf16lo(v.x), bf16hi(v.x), s)) |
          (static_cast<uint32_t>(quant_pair(bf16lo(v.y), bf16hi(v.y), s)) << 16);
    r.y = static_cast<uint32_t>(quant_pair(bf16lo(v.z), bf16hi(v.z), s)) |
          (static_cast<uint32_t>(quant_pair(bf16lo(v.w), bf16hi(v.w), s)) << 16);
    return r;
}

// The E4M3 code pair of two FP32 values (low byte = a): the hardware's
// round-to-nearest-even, saturating conversion.
__device__ __forceinline__ uint32_t e4m3_pair(float a, float b) {
    return static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3));
}

// The reciprocal route to the codes of the correctly rounded quotients
// RN(x/s), for kernels bound by instruction issue. Once per scale:
// r = RN(1/s), lo = RN(r (1 - 2^-21)), hi = RN(r (1 + 2^-21)). For each x,
// RN(x lo) and RN(x hi) lie strictly on the two sides of x/s (three roundings
// of relative size at most 2^-24 each cannot undo the 2^-21 offset; a product
// small enough to lose that precision gives the code of zero either way), so
// they bracket RN(x/s). Rounding to E4M3 (nearest even, saturating) is
// monotonic: when both give the same code, so does RN(x/s). Otherwise (x/s
// within about 2^-20 of a rounding boundary of the conversion) the chunk takes
// correctly rounded divisions. When r is not a normal number, or hi
// overflows, lo = 0 and hi = +Inf: every non-NaN x then disagrees and takes
// the division.
struct RecipBracket {
    float lo, hi;
};

__device__ __forceinline__ RecipBracket recip_bracket(float s) {
    const float r = __frcp_rn(s);
    RecipBracket b{__fmul_rn(r, 1.0f - 0x1p-21f), __fmul_rn(r, 1.0f + 0x1p-21f)};  // both factors exact
    if (!(fabsf(r) >= 0x1p-126f && fabsf(b.hi) <= 3.402823466e38f)) {
        b.lo = 0.0f;
        b.hi = INFINITY;
    }
    return b;
}

// The 8 codes of quant8(v, s), in memory order, by the route above (packed
// FP32 products, two conversions per pair of values).
__device__ __forceinline__ uint2 quant8_recip(const uint4 &v, float s, RecipBracket b) {
    const float2 x[4] = {make_float2(bf16lo(v.x), bf16hi(v.x)), make_float2(bf16lo(v.y), bf16hi(v.y)),
                         make_float2(bf16lo(v.z), bf16hi(v.z)), make_float2(bf16lo(v.w), bf16hi(v.w))};
    const float2 lo2 = make_float2(b.lo, b.lo), hi2 = make_float2(b.hi, b.hi);
    float2 p[4], q[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        p[i] = __fmul2_rn(x[i], lo2);
        q[i] = __fmul2_rn(x[i], hi2);
    }
    uint2 lo, hi;
    lo.x = e4m3_pair(p[0].x, p[0].y) | (e4m3_pair(p[1].x, p[1].y) << 16);
    lo.y = e4m3_pair(p[2].x, p[2].y) | (e4m3_pair(p[3].x, p[3].y) << 16);
    hi.x = e4m3_pair(q[0].x, q[0].y) | (e4m3_pair(q[1].x, q[1].y) << 16);
    hi.y = e4m3_pair(q[2].x, q[2].y) | (e4m3_pair(q[3].x, q[3].y) << 16);
    if ((lo.x != hi.x) | (lo.y != hi.y)) {
#pragma unroll
        for (int i = 0; i < 4; ++i) p[i] = make_float2(__fdiv_rn(x[i].x, s), __fdiv_rn(x[i].y, s));
        lo.x = e4m3_pair(p[0].x, p[0].y) | (e4m3_pair(p[1].x, p[1].y) << 16);
        lo.y = e4m3_pair(p[2].x, p[2].y) | (e4m3_pair(p[3].x, p[3].y) << 16);
    }
    return lo;
}

__device__ __forceinline__ uint4 ld_stream_v4(const void *p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
    return r;
}

// One 1 x 128 activation group quantized by a lane quad: group g of row
// src_row of x [.][K] into row m of q [M][K] and s [K/128][M]. Lane c (0..3) of
// the quad holds the 16-byte chunks c, c+4, c+8, c+12 of the group's 256
// bytes, the quad's amax is reduced with two shuffles, and each lane stores
// its 4 x 8 codes; lane 0 of the quad stores the scale at s[g * M + m]. Every
// lane of the warp must call it (ok = false where the group does not exist,
// which loads, stores and contributes nothing). `ld` loads 16 bytes of x.
template <typename Load>
__device__ __forceinline__ void quant_group_by_quad(const uint16_t *x, uint8_t *q, float *s, int64_t M, int64_t K,
                                                    int64_t m, int64_t src_row, int64_t g, int c, bool ok, Load ld) {
    const int64_t base = m * K + g * 128 + c * 8;
    const int64_t src = src_row * K + g * 128 + c * 8;
    uint4 v[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        v[i] = make_uint4(0u, 0u, 0u, 0u);
        if (ok) v[i] = ld(x + src + 32 * i);
    }
    uint32_t m2 = 0;  // packed BF16 maxima of |x| (bit patterns, sign masked)
#pragma unroll
    for (int i = 0; i < 4; ++i) amax8_acc(m2, v[i]);
    float a = amax_of(m2);
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
    if (ok) {
        const float sc = block_scale(a);
#pragma unroll
        for (int i = 0; i < 4; ++i) *reinterpret_cast<uint2 *>(q + base + 32 * i) = quant8(v[i], sc);
        if (c == 0) s[g * M + m] = sc;
    }
}

}  // namespace fp8k
