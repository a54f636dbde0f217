// Quantizer kernels: BF16 -> E4M3 codes + FP32 scales.
//
//  - 1 x 128 activation groups (dynamic, per token): four lanes per group,
//    each with four 16-byte loads of 8 BF16 in flight, a packed BF16 amax
//    of its 32 values and a two-step shuffle amax over the four lanes, one
//    scale per lane and 8-byte stores of 8 packed codes (by division); launched as a programmatic dependent so that, in a decode
//    step, its launch overlaps the previous GEMM and the next GEMM's prologue
//    overlaps it. Four lanes per group (rather than sixteen) spread the
//    per-group work - the shuffle amax and the scale division - over 32
//    elements per lane. At decode sizes (M <= 16) a kernel with sixteen lanes
//    per group takes over, and warms its x in L2 before the upstream wait.
//  - 128 x 128 weight blocks: one CTA per block, the block held in registers
//    between the amax pass and the quantize pass (read once).
//  - Per tensor: grid-wide amax (atomicMax on the bit pattern of the
//    non-negative amax, kept in the output scale slot), then quantize, each
//    pass one resident wave of CTAs over equal contiguous slices; one
//    cluster of 8 CTAs does both for small tensors (amax through distributed
//    shared memory).
//  - One scale per row (per token or per output channel): one CTA per row.
//
// The weight-block, per-tensor, row-wise and decode-sized activation
// quantizers are bound by instruction issue; they reach the correctly rounded
// quotient's code through one reciprocal bracket per block, row or tensor
// (recip_bracket / quant8_recip in quantize.cuh), with a division only near
// rounding boundaries, and take amaxes with packed BF16 maxima. Codes are
// identical to quant8's either way.
//
// Every scale is fl32(max(amax, 1e-10) / 448) and every code
// e4m3(fl32(x / scale)); "[vLLM] FP8" page, sections "스케일링 전략 체계"
// and "블록 양자화", with the rounding readings stated in fp8w8a8.h.
#include "quantize.cuh"
#include "launch.h"

namespace fp8k {
namespace {

// Error-word sites of the device-side argument checks.
enum : unsigned { kSiteStaticScale = 301, kSiteStaticScaleSmall = 302, kSiteRowIndex = 303 };

// ------------------------------------------------ 1 x 128 activation groups --

constexpr int kActThreads = 256;
constexpr int kActRows = kActThreads / 32;  // rows per CTA: one warp each
constexpr int kActGroups = 8;               // groups per CTA: one lane quad each

// Bounded to six resident CTAs per SM (at most 40 registers): at the default
// 55 registers only four fit and the kernel is latency-bound (8192 x 14336:
// 62.5 us at six, 68.7 us at four). With the packed amax it fits in 40
// registers without spilling (61.7 us; 65.7 us with the float amax, which
// spilled 24 bytes); the reciprocal route on top measured slower here (63.9).
//
// CTA (blockIdx.x, blockIdx.y) covers rows 8*blockIdx.x .. +7 (warp w takes
// row 8*blockIdx.x + w) and groups 8*blockIdx.y .. +7 (lanes 4j..4j+3 take
// group 8*blockIdx.y + j). Lane c of a quad holds the 16-byte chunks
// c, c+4, c+8, c+12 of the group's 256 bytes, so each warp-wide load covers
// 64 contiguous bytes of every group and each store 32.
template <bool GATHER>
__global__ void __launch_bounds__(kActThreads, 6) quant_act_group_kernel(const uint16_t *__restrict__ x,
                                                                      uint8_t *__restrict__ q,
                                                                      float *__restrict__ s, int64_t M,
                                                                      int64_t K,
                                                                      const int32_t *__restrict__ row_index,
                                                                      int64_t M_src, unsigned *err) {
    const int64_t Kg = K / 128;
    const int lane = threadIdx.x & 31;
    const int c = lane & 3;
    const int64_t m = static_cast<int64_t>(blockIdx.x) * kActRows + (threadIdx.x >> 5);
    // Launched as a programmatic dependent: let the next kernel start its
    // prologue, then wait for the kernel that produced x. (A dependent that
    // reads q or s before its own griddepcontrol.wait could see them half
    // written; the GEMMs of this library read them only after it.)
    grid_dep_launch();
    grid_dep_wait();

    const int64_t g = static_cast<int64_t>(blockIdx.y) * kActGroups + (lane >> 2);
    int64_t src = m;
    if (GATHER && m < M) {
        // Routed row m reads source row row_index[m]; one outside [0, M_src)
        // is recorded and reads row 0 instead.
        const int r = __ldg(row_index + m);
        const bool bad = r < 0 || static_cast<int64_t>(r) >= M_src;
        if (bad && lane == 0 && blockIdx.y == 0) record_error(err, kErrArg, kSiteRowIndex);
        src = bad ? 0 : r;
    }
    quant_group_by_quad(x, q, s, M, K, m, src, g, c, m < M && g < Kg,
                        [](const uint16_t *p) { return ld_stream_v4(p); });
}

// Decode-sized inputs (few rows): the kernel above gives each lane 32
// elements and puts only a few CTAs on the GPU, so a call is bound by one
// lane's dependent chain. Here each lane takes one 16-byte chunk (8 elements)
// and a group is spread over 16 lanes (two groups per warp, 16 per CTA), and
// the codes take the reciprocal route (quant8_recip, the same codes as the
// division). CTA b covers groups 16b .. 16b+15 in (row, group) order.
constexpr int kActSmallThreads = 256;
constexpr int64_t kActSmallMaxRows = 16;  // the decode sizes; larger M takes the kernel above
constexpr int kActSmallGroups = kActSmallThreads / 16;


__global__ void __launch_bounds__(kActSmallThreads) quant_act_group_small_kernel(const uint16_t *__restrict__ x,
                                                                                uint8_t *__restrict__ q,
                                                                                float *__restrict__ s, int M,
                                                                                int Kg) {
    const int lane = threadIdx.x & 31;
    const int c = lane & 15;
    const int gi = blockIdx.x * kActSmallGroups + (threadIdx.x >> 4);
    const bool ok = gi < M * Kg;
    const int m = ok ? gi / Kg : 0;
    const int g = ok ? gi - m * Kg : 0;
    grid_dep_launch();
    const int64_t off = static_cast<int64_t>(m) * Kg * 128 + g * 128 + c * 8;
    // Warm this chunk of x in L2 while the upstream kernel finishes. The load
    // itself waits: x may be that kernel's output. An L2 prefetch brings no
    // data into the SM and L2 holds the latest value of every line, so it
    // cannot make the load below see a stale x.
    if (ok) asm volatile("prefetch.global.L2 [%0];" ::"l"(x + off));
    grid_dep_wait();
    const uint4 v = ok ? ld_stream_v4(x + off) : make_uint4(0u, 0u, 0u, 0u);
    uint32_t m2 = 0;
    amax8_acc(m2, v);
    float a = amax_of(m2);
#pragma unroll
    for (int o = 1; o < 16; o <<= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
    if (ok) {
        const float sc = block_scale(a);
        *reinterpret_cast<uint2 *>(q + off) = quant8_recip(v, sc, recip_bracket(sc));
        if (c == 0) s[static_cast<int64_t>(g) * M + m] = sc;
    }
}

// --------------------------------------------------- 128 x 128 weight blocks --

constexpr int kWThreads = 256;
constexpr int kWChunks = 128 * 16 / kWThreads;  // 16-byte chunks per thread (8)
constexpr int kWRowsPerPass = kWThreads / 16;

// Block (nb, kb) = (blockIdx.y, blockIdx.x). Chunk c = t + 256 j covers row
// c / 16 of the block and bytes 16 (c % 16) .. of the row's 256-byte span.
// Bounded to four resident CTAs per SM (at most 64 registers): the kernel is
// bound by the latency of its load / reduce / store phases, and a fourth CTA
// per SM hides more of it (28672 x 4096: 67.6 us against 72.2 at three).
__global__ void __launch_bounds__(kWThreads, 4) quant_weight_block_kernel(const uint16_t *__restrict__ w,
                                                                       uint8_t *__restrict__ q,
                                                                       float *__restrict__ s, int64_t N,
                                                                       int64_t K) {
    __shared__ float warp_amax[kWThreads / 32];
    const int t = threadIdx.x;
    const int64_t kb = blockIdx.x, nb = blockIdx.y, Kg = K / 128;
    const int col = (t & 15) * 8;
    uint4 v[kWChunks];
    uint32_t m2 = 0;
#pragma unroll
    for (int j = 0; j < kWChunks; ++j) {
        const int64_t row = nb * 128 + (t >> 4) + kWRowsPerPass * j;
        v[j] = make_uint4(0u, 0u, 0u, 0u);
        if (row < N) v[j] = ld_stream_v4(w + row * K + kb * 128 + col);
    }
#pragma unroll
    for (int j = 0; j < kWChunks; ++j) amax8_acc(m2, v[j]);
    float a = amax_of(m2);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
    if ((t & 31) == 0) warp_amax[t >> 5] = a;
    __syncthreads();
    a = warp_amax[0];
#pragma unroll
    for (int i = 1; i < kWThreads / 32; ++i) a = fmaxf(a, warp_amax[i]);
    const float sc = block_scale(a);
    const RecipBracket rc = recip_bracket(sc);
#pragma unroll
    for (int j = 0; j < kWChunks; ++j) {
        const int64_t row = nb * 128 + (t >> 4) + kWRowsPerPass * j;
        if (row < N) *reinterpret_cast<uint2 *>(q + row * K + kb * 128 + col) = quant8_recip(v[j], sc, rc);
    }
    if (t == 0) s[nb * Kg + kb] = sc;
}

// ------------------------------------------------------------- per tensor --

constexpr int kTThreads = 256;
constexpr int kTUnroll = 4;
// Tensors up to this many elements take the single-CTA path.
constexpr int64_t kSmallTensor = 1 << 17;

__device__ __forceinline__ float block_reduce_max(float a, float *scratch) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
    if ((threadIdx.x & 31) == 0) scratch[threadIdx.x >> 5] = a;
    __syncthreads();
    a = scratch[0];
    for (int i = 1; i < static_cast<int>(blockDim.x >> 5); ++i) a = fmaxf(a, scratch[i]);
    return a;
}

// Bounds [c0, c1) of CTA b's share of n items split over g CTAs in equal
// contiguous slices (the first n % g get one more), without forming n * b.
__device__ __forceinline__ void slice_of(int64_t n, int64_t b, int64_t g, int64_t &c0, int64_t &c1) {
    const int64_t q = n / g, r = n % g;
    c0 = b * q + (b < r ? b : r);
    c1 = c0 + q + (b < r ? 1 : 0);
}

// Device-side check of a caller's static scale: it must be positive and
// finite. A bad one is recorded as FP8_ERR_ARG with `site` in the error word
// (the quantization still runs, with that scale).
__device__ __forceinline__ void check_static_scale(float sc, unsigned *err, unsigned site) {
    if (!(sc > 0.0f && sc <= 3.402823466e38f)) record_error(err, kErrArg, site);
}

// amax of the whole tensor into *amax_bits (zeroed before): the bit pattern of
// a non-negative float orders like the float, so atomicMax on it is a max.
__global__ void __launch_bounds__(kTThreads) tensor_amax_kernel(const uint16_t *__restrict__ x, int64_t n8,
                                                                unsigned *__restrict__ amax_bits) {
    __shared__ float scratch[kTThreads / 32];
    grid_dep_launch();  // the quantize pass may be scheduled; it waits for this grid
    uint32_t m2 = 0;
    int64_t c0, c1;
    slice_of(n8, blockIdx.x, gridDim.x, c0, c1);
    for (int64_t i = c0 + threadIdx.x; i < c1; i += kTThreads * kTUnroll) {
        uint4 v[kTUnroll];
#pragma unroll
        for (int u = 0; u < kTUnroll; ++u) {
            const int64_t j = i + u * kTThreads;
            v[u] = j < c1 ? ld_stream_v4(x + j * 8) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < kTUnroll; ++u) amax8_acc(m2, v[u]);
    }
    const float a = block_reduce_max(amax_of(m2), scratch);
    if (threadIdx.x == 0) atomicMax(amax_bits, __float_as_uint(a));
}

// Quantize with the scale from the amax in *amax_bits (dynamic) or the scale
// in *scale (static).
//
// Only the dynamic pass lets its dependent launch early: that dependent is the
// finalize kernel, which waits for this grid before it touches anything. A
// static call ends with this kernel, and what follows it on the stream may be
// a decode GEMM that streams its weights before its own griddepcontrol.wait;
// q may be those weights (a per-tensor weight quantized at load time), so the
// static pass triggers only by completing.
__global__ void __launch_bounds__(kTThreads) tensor_quant_kernel(const uint16_t *__restrict__ x,
                                                                 uint8_t *__restrict__ q, int64_t n8,
                                                                 const float *scale, int from_amax,
                                                                 unsigned *err) {
    // Launched as a programmatic dependent of the amax pass (or of whatever
    // precedes a static call): wait for it before reading the scale or x.
    if (from_amax) grid_dep_launch();
    grid_dep_wait();
    const float stored = *scale;
    const float sc = from_amax ? block_scale(stored) : stored;
    if (!from_amax && blockIdx.x == 0 && threadIdx.x == 0) check_static_scale(sc, err, kSiteStaticScale);
    const RecipBracket rc = recip_bracket(sc);
    int64_t c0, c1;
    slice_of(n8, blockIdx.x, gridDim.x, c0, c1);
    for (int64_t i = c0 + threadIdx.x; i < c1; i += kTThreads * kTUnroll) {
        uint4 v[kTUnroll];
#pragma unroll
        for (int u = 0; u < kTUnroll; ++u) {
            const int64_t j = i + u * kTThreads;
            v[u] = j < c1 ? ld_stream_v4(x + j * 8) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < kTUnroll; ++u) {
            const int64_t j = i + u * kTThreads;
            if (j < c1) *reinterpret_cast<uint2 *>(q + j * 8) = quant8_recip(v[u], sc, rc);
        }
    }
}

// *scale: amax bit pattern -> scale, once every CTA of the quantize pass
// (a programmatic predecessor) has read it.
__global__ void tensor_scale_finalize_kernel(float *scale) {
    grid_dep_wait();
    *scale = block_scale(*scale);
}

// Grid of one resident wave for `kernel` at kTThreads threads.
template <typename Kernel>
int64_t tensor_grid(Kernel kernel, int64_t want, const DeviceInfo &dev) {
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kTThreads, 0) != cudaSuccess || per_sm < 1)
        per_sm = 1;
    const int64_t cap = static_cast<int64_t>(dev.sm_count) * per_sm;
    return want < cap ? want : cap;
}

cudaError_t launch_pdl(const void *fn, unsigned grid, unsigned block, void **args, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelExC(&cfg, fn, args);
}

// Whole per-tensor quantization of a small tensor (up to kSmallTensor
// elements) in one cluster of kTcCtas CTAs: each CTA holds its share of x in
// registers, the CTAs' partial amaxes meet through distributed shared memory,
// and every CTA quantizes its share with the common scale. One launch, x read
// once. Launched as a programmatic dependent; it warms its share of x in L2
// before the upstream wait and lets nothing launch before it completes (its
// codes may be the weights of a following decode GEMM).
constexpr int kTcCtas = 8;
constexpr int kTcThreads = 256;
constexpr int kTcHeld = 8;  // 16-byte chunks per thread
static_assert(int64_t(kTcCtas) * kTcThreads * kTcHeld * 8 >= kSmallTensor, "the cluster must cover a small tensor");

__device__ __forceinline__ void cluster_arrive_release() { asm volatile("barrier.cluster.arrive.release;" ::: "memory"); }

__device__ __forceinline__ float ld_cluster_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

// Chunk k of thread t in cluster rank r: (k * kTcCtas + r) * kTcThreads + t, so
// each CTA reads 4 KB contiguous per k.
__global__ void __launch_bounds__(kTcThreads) tensor_quant_cluster_kernel(const uint16_t *__restrict__ x,
                                                                         uint8_t *__restrict__ q, int64_t n8,
                                                                         float *scale, int is_static,
                                                                         unsigned *err) {
    __shared__ float scratch[kTcThreads / 32];
    __shared__ float cta_amax;
    const uint32_t rank = cluster_ctarank();
    const int t = threadIdx.x;
    auto chunk = [&](int k) { return (static_cast<int64_t>(k) * kTcCtas + rank) * kTcThreads + t; };
#pragma unroll
    for (int k = 0; k < kTcHeld; ++k)
        if (chunk(k) < n8) asm volatile("prefetch.global.L2 [%0];" ::"l"(x + chunk(k) * 8));
    grid_dep_wait();
    uint4 v[kTcHeld];
#pragma unroll
    for (int k = 0; k < kTcHeld; ++k) v[k] = chunk(k) < n8 ? ld_stream_v4(x + chunk(k) * 8) : make_uint4(0u, 0u, 0u, 0u);
    float sc;
    if (is_static) {
        sc = *scale;
        if (rank == 0 && t == 0) check_static_scale(sc, err, kSiteStaticScaleSmall);
    } else {
        uint32_t m2 = 0;
#pragma unroll
        for (int k = 0; k < kTcHeld; ++k) amax8_acc(m2, v[k]);
        const float a = block_reduce_max(amax_of(m2), scratch);
        if (t == 0) cta_amax = a;
        cluster_arrive_release();  // every CTA's partial is written ...
        cluster_wait_acquire();    // ... and visible to every CTA of the cluster
        float g = 0.0f;
#pragma unroll
        for (int r = 0; r < kTcCtas; ++r) g = fmaxf(g, ld_cluster_f32(map_shared_rank(smem_u32(&cta_amax), r)));
        sc = block_scale(g);
        cluster_arrive_release();  // this CTA is done reading its peers' shared memory
    }
    const RecipBracket rc = recip_bracket(sc);
#pragma unroll
    for (int k = 0; k < kTcHeld; ++k)
        if (chunk(k) < n8) *reinterpret_cast<uint2 *>(q + chunk(k) * 8) = quant8_recip(v[k], sc, rc);
    if (!is_static && rank == 0 && t == 0) *scale = sc;
    if (!is_static) cluster_wait_acquire();  // no CTA exits while a peer may still read its shared memory
}

// ---------------------------------------------------- one scale per row --

constexpr int kRThreads = 256;
constexpr int kRHeld = 8;  // 16-byte chunks of the row held in registers per thread

// Row r of x [rows][cols] gets one scale from its own amax: per-token scales
// for activations, per-channel scales for weights (rows = output channels).
// One CTA per row (grid-stride); the first kRHeld * 256 chunks of the row stay
// in registers between the amax and the quantize pass, any rest is read
// again. Launched as a programmatic dependent, but lets nothing launch before
// it completes: its codes may be the weights of a following decode GEMM.
__global__ void __launch_bounds__(kRThreads) quant_rows_kernel(const uint16_t *__restrict__ x,
                                                               uint8_t *__restrict__ q, float *__restrict__ s,
                                                               int64_t rows, int64_t cols) {
    __shared__ float scratch[kRThreads / 32];
    const int64_t c8 = cols / 8;
    if (blockIdx.x < rows) {  // warm this CTA's first row in L2 while the upstream kernel finishes
        const uint16_t *xr = x + static_cast<int64_t>(blockIdx.x) * cols;
#pragma unroll
        for (int j = 0; j < kRHeld; ++j) {
            const int64_t i = threadIdx.x + static_cast<int64_t>(j) * kRThreads;
            if (i < c8 && (i & 7) == 0) asm volatile("prefetch.global.L2 [%0];" ::"l"(xr + i * 8));
        }
    }
    grid_dep_wait();
    for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
        const uint16_t *xr = x + r * cols;
        uint8_t *qr = q + r * cols;
        uint4 v[kRHeld];
        uint32_t m2 = 0;
#pragma unroll
        for (int j = 0; j < kRHeld; ++j) {
            const int64_t i = threadIdx.x + static_cast<int64_t>(j) * kRThreads;
            v[j] = i < c8 ? ld_stream_v4(xr + i * 8) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int j = 0; j < kRHeld; ++j) amax8_acc(m2, v[j]);
        for (int64_t i = threadIdx.x + kRHeld * kRThreads; i < c8; i += kRThreads) amax8_acc(m2, ld_stream_v4(xr + i * 8));
        const float a = block_reduce_max(amax_of(m2), scratch);
        const float sc = block_scale(a);
        const RecipBracket rc = recip_bracket(sc);
#pragma unroll
        for (int j = 0; j < kRHeld; ++j) {
            const int64_t i = threadIdx.x + static_cast<int64_t>(j) * kRThreads;
            if (i < c8) *reinterpret_cast<uint2 *>(qr + i * 8) = quant8_recip(v[j], sc, rc);
        }
        for (int64_t i = threadIdx.x + kRHeld * kRThreads; i < c8; i += kRThreads)
            *reinterpret_cast<uint2 *>(qr + i * 8) = quant8_recip(ld_stream_v4(xr + i * 8), sc, rc);
        if (threadIdx.x == 0) s[r] = sc;
        __syncthreads();  // scratch is rewritten by the next row
    }
}

}  // namespace

cudaError_t launch_quant_rows(const void *x, void *q, float *s, int64_t rows, int64_t cols, const DeviceInfo &dev,
                              cudaStream_t stream) {
    (void)dev;
    if (rows == 0 || cols == 0) return cudaSuccess;
    const int64_t grid = rows < 0x7FFFFFFF ? rows : 0x7FFFFFFF;
    const uint16_t *xp = static_cast<const uint16_t *>(x);
    uint8_t *qp = static_cast<uint8_t *>(q);
    void *args[] = {&xp, &qp, &s, &rows, &cols};
    return launch_pdl(reinterpret_cast<const void *>(quant_rows_kernel), static_cast<unsigned>(grid), kRThreads,
                      args, stream);
}

cudaError_t launch_quant_act_group(const void *x, void *q, float *s, int64_t M, int64_t K,
                                   const DeviceInfo &dev, cudaStream_t stream, const int32_t *row_index,
                                   int64_t M_src) {
    const int64_t groups = M * (K / 128);
    if (row_index == nullptr && M <= kActSmallMaxRows && groups > 0) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>((groups + kActSmallGroups - 1) / kActSmallGroups));
        cfg.blockDim = dim3(kActSmallThreads);
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        return cudaLaunchKernelEx(&cfg, quant_act_group_small_kernel, static_cast<const uint16_t *>(x),
                                  static_cast<uint8_t *>(q), s, static_cast<int>(M), static_cast<int>(K / 128));
    }
    const int64_t rows = (M + kActRows - 1) / kActRows;
    const int64_t cols = (K / 128 + kActGroups - 1) / kActGroups;
    if (rows == 0 || cols == 0) return cudaSuccess;
    if (rows > 0x7FFFFFFF || cols > 65535) return cudaErrorInvalidValue;  // the entry point checks K first
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(rows), static_cast<unsigned>(cols));
    cfg.blockDim = dim3(kActThreads);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (row_index != nullptr)
        return cudaLaunchKernelEx(&cfg, quant_act_group_kernel<true>, static_cast<const uint16_t *>(x),
                                  static_cast<uint8_t *>(q), s, M, K, row_index, M_src, dev.err);
    return cudaLaunchKernelEx(&cfg, quant_act_group_kernel<false>, static_cast<const uint16_t *>(x),
                              static_cast<uint8_t *>(q), s, M, K, row_index, M, dev.err);
}

cudaError_t launch_quant_weight_block(const void *w, void *q, float *s, int64_t N, int64_t K,
                                      const DeviceInfo &dev, cudaStream_t stream) {
    (void)dev;
    const int64_t nb = (N + 127) / 128, kb = K / 128;
    if (nb == 0 || kb == 0) return cudaSuccess;
    if (nb > 65535 || kb > 0x7FFFFFFF) return cudaErrorInvalidValue;  // the entry point checks N first
    dim3 grid(static_cast<unsigned>(kb), static_cast<unsigned>(nb));
    quant_weight_block_kernel<<<grid, kWThreads, 0, stream>>>(static_cast<const uint16_t *>(w),
                                                              static_cast<uint8_t *>(q), s, N, K);
    return cudaGetLastError();
}

cudaError_t launch_quant_per_tensor(const void *x, void *q, float *scale, int64_t n, bool is_static,
                                    const DeviceInfo &dev, cudaStream_t stream) {
    const int64_t n8 = n / 8;  // n is a multiple of 16
    const uint16_t *xp = static_cast<const uint16_t *>(x);
    uint8_t *qp = static_cast<uint8_t *>(q);
    if (n8 == 0 && is_static) return cudaSuccess;
    if (n <= kSmallTensor) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(kTcCtas);
        cfg.blockDim = dim3(kTcThreads);
        cfg.stream = stream;
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = kTcCtas;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 2;
        return cudaLaunchKernelEx(&cfg, tensor_quant_cluster_kernel, xp, qp, n8, scale, is_static ? 1 : 0, dev.err);
    }
    // Each pass runs as one resident wave, and the quantize and finalize
    // kernels are programmatic dependents of their predecessors, so their
    // launches overlap the previous pass.
    static const int64_t kWant = kTThreads * kTUnroll;
    const int64_t want = (n8 + kWant - 1) / kWant;
    if (!is_static) {
        cudaError_t e = cudaMemsetAsync(scale, 0, sizeof(float), stream);
        if (e != cudaSuccess) return e;
        const unsigned ga = static_cast<unsigned>(tensor_grid(tensor_amax_kernel, want, dev));
        tensor_amax_kernel<<<ga, kTThreads, 0, stream>>>(xp, n8, reinterpret_cast<unsigned *>(scale));
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    const unsigned gq = static_cast<unsigned>(tensor_grid(tensor_quant_kernel, want, dev));
    int from_amax = is_static ? 0 : 1;
    const float *cscale = scale;
    unsigned *err = dev.err;
    void *qargs[] = {&xp, &qp, const_cast<int64_t *>(&n8), &cscale, &from_amax, &err};
    cudaError_t e = launch_pdl(reinterpret_cast<const void *>(tensor_quant_kernel), gq, kTThreads, qargs, stream);
    if (e != cudaSuccess || is_static) return e;
    void *fargs[] = {&scale};
    return launch_pdl(reinterpret_cast<const void *>(tensor_scale_finalize_kernel), 1, 1, fargs, stream);
}

}  // namespace fp8k
