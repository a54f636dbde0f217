// Weight-streaming FP8 GEMM for decode-shaped problems (M <= 16 tokens).
//
// Decode reads every weight once per step and does little arithmetic per
// byte, so it is bound by memory bandwidth ("FP8 serving slower than BF16",
// section "Arithmetic Intensity: decode가 FP8을 살리지 못하는 이유"; "서빙을
// 위한 양자화 가이드", item ② on decode being memory-bound). The design here:
//
//  - the weight matrix is the MMA's M side (128 weight rows per CTA) and the
//    tokens are its N side (N = 16), so no tensor-core rows are spent on
//    padding tokens to 128 and nothing padded is read from memory (the TMA
//    fills token rows >= M with zeros on chip);
//  - weights stream through a ring of TMA stages (16 KB of weights + 2 KB
//    of activation codes per 128-wide K block), one lane issuing, so many
//    bytes are in flight per SM with no register staging;
//  - K is split across the CTAs of a thread-block cluster (up to 8) so that
//    all CTAs of the grid are resident at once (one wave); each CTA promotes
//    its K blocks with the scales in FP32 registers. Each CTA of the cluster
//    owns a slice of the 128 rows: every CTA stages its partial sums in its
//    own shared memory in row order and pushes each rank's slice to that
//    rank with one bulk copy (counted on an mbarrier there); the owner sums
//    the slices in a fixed order and stores them. A rank waits only for the
//    bytes addressed to it and leaves once its own copies have read their
//    source, so no cluster-wide barrier sits on the critical path and no CTA
//    is addressed after it exits. No global scratch memory is used;
//  - launched as a programmatic dependent of the previous kernel in the
//    stream: before that kernel is known to be complete the CTA already
//    loads its first weight tiles into their stages and warms L2 with the
//    next few (weights are not written by any kernel that triggers this one
//    early); the activation codes and scales are read, and every global
//    write is made, after griddepcontrol.wait.
//
// Block mode applies Sw[n/128][kb] * Sa[kb][m] per K block; per-tensor mode
// accumulates all of the CTA's K range in TMEM and applies sa * sw once;
// row/column mode does the same with sa[m] * sw[n] (per-token activation and
// per-channel weight scales).
#include <mutex>

#include "common.cuh"
#include "launch.h"

namespace fp8k {
namespace {

constexpr int kRows = 128;      // weight rows per CTA (MMA M)
constexpr int kTok = 16;        // token slots (MMA N)
constexpr int BK = 128;
constexpr int kStages = 5;
constexpr int kWBytes = kRows * BK;
constexpr int kXBytes = kTok * BK;
constexpr int kThreads = 256;
// Two 16-column TMEM partial buffers: the MMA may run one K block ahead of
// the epilogue (4 and 8 buffers measured the same).
constexpr int kTBufs = 2;
constexpr int kTmemCols = kTBufs * kTok < 32 ? 32 : kTBufs * kTok;
// Before the upstream grid completes, the first kStages weight tiles go into
// their stages and one otherwise idle lane warms the next ones in L2, one tile
// every kWarmPaceNs, until the upstream wait returns (at most kWarmMax tiles).
// The amount therefore follows the upstream kernel's remaining time: a short
// quantizer in front of the GEMM leaves a few microseconds of idle HBM to
// fill, a previous GEMM that is still streaming leaves none.
constexpr int kWarmMax = 32;
constexpr unsigned kWarmPaceNs = 500;
constexpr int kScaleKb = 8;     // K blocks of activation/weight scales staged at a time per epilogue warp
constexpr int kScaleBytes = 4 * 4 * (kScaleKb * kTok + kScaleKb);
constexpr int kRecvBytes = kRows * kTok * 4;  // split-K partials addressed to this CTA
constexpr int kSmemBytes =
    1024 + kStages * (kWBytes + kXBytes) + kRecvBytes + 8 * (2 * kStages + 2 * kTBufs + 1) + 16 + kScaleBytes;

enum : unsigned { kSiteProdEmpty = 201, kSiteMmaTmem = 202, kSiteMmaFull = 203, kSiteEpiFull = 204,
                  kSiteDrain = 205, kSiteReduce = 206 };

template <int MODE>
__global__ void __launch_bounds__(kThreads, 2)
    gemm_decode_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                       const float *__restrict__ sa, const float *__restrict__ sw,
                       __nv_bfloat16 *__restrict__ y, int M, int N, int K, int splits, unsigned *err) {
    constexpr bool WHOLE_K = MODE != kScaleBlock;  // all of the CTA's K in one TMEM accumulator
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sW = smem;
    uint8_t *sX = smem + kStages * kWBytes;
    float *recv = reinterpret_cast<float *>(sX + kStages * kXBytes);  // [splits][rows_per][kTok]
    uint64_t *full = reinterpret_cast<uint64_t *>(reinterpret_cast<uint8_t *>(recv) + kRecvBytes);
    uint64_t *empty = full + kStages;
    uint64_t *tfull = empty + kStages;
    uint64_t *tempty = tfull + kTBufs;
    uint64_t *rbar = tempty + kTBufs;  // completes when all kRecvBytes have arrived
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(rbar + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    volatile int *waited = reinterpret_cast<volatile int *>(tmem_slot + 2);  // the producer passed the upstream wait
    float *scale_smem = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(tmem_slot) + 16);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nb = blockIdx.x / splits;
    const int split = blockIdx.x - nb * splits;
    const int n0 = nb * kRows;
    const int Kg = (K + BK - 1) / BK;
    const int kb0 = static_cast<int>((static_cast<int64_t>(split) * Kg) / splits);
    const int kb1 = static_cast<int>((static_cast<int64_t>(split + 1) * Kg) / splits);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
        for (int b = 0; b < kTBufs; ++b) { mbar_init(&tfull[b], 1); mbar_init(&tempty[b], 128); }
        mbar_init(rbar, 1);
        *abort_flag = 0;
        *waited = 0;
        fence_barrier_init();
        if (splits > 1) mbar_arrive_expect_tx(rbar, kRecvBytes);
    }
    if (warp == 0 && lane == 0) { tma_prefetch_desc(&tmW); tma_prefetch_desc(&tmX); }
    if (warp == 2) { tmem_alloc(tmem_slot, kTmemCols); tmem_relinquish(); }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // Every CTA's receive barrier is initialised before any rank pushes to it:
    // each thread passes this cluster barrier before the upstream wait, i.e.
    // while the previous kernel may still be running.
    if (splits > 1) cluster_arrive_relaxed();
    if (splits > 1 && !(warp == 0 && lane == 0)) cluster_wait_acquire();

    float acc[kTok];
#pragma unroll
    for (int j = 0; j < kTok; ++j) acc[j] = 0.0f;
    grid_dep_launch();

    if (warp == 0) {
        if (lane == 0) {
            // -------------------------------------------------- producer --
            // Weights are read before the upstream wait (the caller's contract:
            // no kernel that triggers this one early writes them): the first
            // kStages weight tiles go straight into their stages (warp 3 warms
            // the next ones in L2). Activation codes come after the wait.
            const uint64_t stream_once = policy_evict_first();
            const int nkb = kb1 - kb0;
            const int pre = nkb < kStages ? nkb : kStages;
            for (int i = 0; i < pre; ++i) {
                mbar_arrive_expect_tx(&full[i], kWBytes + kXBytes);
                tma_load_2d_hint(sW + i * kWBytes, &tmW, &full[i], (kb0 + i) * BK, n0, stream_once);
            }
            if (splits > 1) cluster_wait_acquire();
            grid_dep_wait();
            *waited = 1;
            for (int i = 0; i < pre; ++i) tma_load_2d(sX + i * kXBytes, &tmX, &full[i], (kb0 + i) * BK, 0);
            uint32_t stage = static_cast<uint32_t>(pre % kStages), phase = pre == kStages ? 1u : 0u;
            int issued = pre;
            for (int kb = kb0 + pre; kb < kb1; ++kb) {
                if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, err, kSiteProdEmpty)) break;
                mbar_arrive_expect_tx(&full[stage], kWBytes + kXBytes);
                tma_load_2d_hint(sW + stage * kWBytes, &tmW, &full[stage], kb * BK, n0, stream_once);
                tma_load_2d(sX + stage * kXBytes, &tmX, &full[stage], kb * BK, 0);
                ++issued;
                if (++stage == kStages) { stage = 0; phase ^= 1u; }
            }
            for (int i = 0; i < kStages && i < issued; ++i) {
                if (stage == 0) { stage = kStages; phase ^= 1u; }
                --stage;
                const uint64_t t0 = global_ns();
                while (!mbar_try_wait(&full[stage], phase)) {
                    if (global_ns() - t0 > kWaitLimitNs) { record_error(err, kErrTimeout, kSiteDrain); break; }
                }
            }
        }
    } else if (warp == 3) {
        if (lane == 0) {
            // ------------------------------------------------ L2 warming --
            const int nkb = kb1 - kb0;
            const int last = nkb < kStages + kWarmMax ? nkb : kStages + kWarmMax;
            for (int i = kStages; i < last && !*waited; ++i) {
                tma_prefetch_l2_2d(&tmW, (kb0 + i) * BK, n0);
                __nanosleep(kWarmPaceNs);
            }
        }
    } else if (warp == 1) {
        grid_dep_wait();
        if (lane == 0) {
            // ------------------------------------------------------- MMA --
            // spins (test_wait): the lane sits on the critical path of each K block
            constexpr uint32_t idesc = idesc_e4m3_f32(kRows, kTok);
            uint32_t stage = 0, phase = 0, buf = 0, bphase = 0, last_stage = 0, last_phase = 0;
            bool any = false;
            for (int kb = kb0; kb < kb1; ++kb) {
                const bool first = kb == kb0, last = kb == kb1 - 1;
                if (!WHOLE_K || first) {
                    if (!mbar_wait<true>(&tempty[buf], bphase ^ 1u, abort_flag, err, kSiteMmaTmem)) break;
                    tc_fence_after();
                }
                if (!mbar_wait<true>(&full[stage], phase, abort_flag, err, kSiteMmaFull)) break;
                tc_fence_after();
                const uint32_t w0 = smem_u32(sW + stage * kWBytes);
                const uint32_t x0 = smem_u32(sX + stage * kXBytes);
                const uint32_t d = tmem_base + buf * kTok;
#pragma unroll
                for (int k = 0; k < BK / 32; ++k) {
                    const uint32_t accum = (k > 0 || (WHOLE_K && !first)) ? 1u : 0u;
                    umma_e4m3(d, sdesc_k_sw128(w0 + k * 32), sdesc_k_sw128(x0 + k * 32), idesc, accum);
                }
                umma_commit(&empty[stage]);
                any = true;
                last_stage = stage;
                last_phase = phase;
                if (!WHOLE_K || last) {
                    umma_commit(&tfull[buf]);
                    if (++buf == kTBufs) { buf = 0; bphase ^= 1u; }
                }
                if (++stage == kStages) { stage = 0; phase ^= 1u; }
            }
            if (any) {
                const uint64_t t0 = global_ns();
                while (!mbar_try_wait(&empty[last_stage], last_phase)) {
                    if (global_ns() - t0 > kWaitLimitNs) { record_error(err, kErrTimeout, kSiteDrain); break; }
                }
            }
        }
    } else if (warp >= 4) {
        // ---------------------------------------------------------- epilogue --
        const int ep = warp - 4;
        const int r = ep * 32 + lane;  // weight row within the CTA's 128
        const uint32_t lane_addr = tmem_base + (static_cast<uint32_t>(ep * 32) << 16);
        uint32_t buf = 0, bphase = 0;
        grid_dep_wait();
        if (!WHOLE_K) {
            // Scales of kScaleKb K blocks at a time go through this warp's own
            // shared-memory slice; the next chunk is loaded into registers while
            // the current one is used (one L2 round trip per chunk, not per block).
            const float *swrow = sw + static_cast<int64_t>(nb) * Kg;
            float *w_sa = scale_smem + ep * (kScaleKb * kTok + kScaleKb);
            float *w_sw = w_sa + kScaleKb * kTok;
            float r_sa[kScaleKb * kTok / 32], r_sw = 0.0f;
            auto fetch = [&](int c0) {
                const int n = (min(kb1, c0 + kScaleKb) - c0);
#pragma unroll
                for (int i = 0; i < kScaleKb * kTok / 32; ++i) {
                    const int idx = lane + 32 * i;
                    r_sa[i] = idx < n * M ? __ldg(sa + static_cast<int64_t>(c0) * M + idx) : 0.0f;
                }
                r_sw = lane < n ? __ldg(swrow + c0 + lane) : 0.0f;
            };
            fetch(kb0);
            bool ok = true;
            for (int c0 = kb0; c0 < kb1 && ok; c0 += kScaleKb) {
                __syncwarp();
#pragma unroll
                for (int i = 0; i < kScaleKb * kTok / 32; ++i) w_sa[lane + 32 * i] = r_sa[i];
                if (lane < kScaleKb) w_sw[lane] = r_sw;
                __syncwarp();
                if (c0 + kScaleKb < kb1) fetch(c0 + kScaleKb);
                const int c1 = min(kb1, c0 + kScaleKb);
                for (int kb = c0; kb < c1; ++kb) {
                    const float wscale = w_sw[kb - c0];
                    const float *srow = w_sa + (kb - c0) * M;
                    if (!__all_sync(0xffffffffu, mbar_wait(&tfull[buf], bphase, abort_flag, err, kSiteEpiFull))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    float p[kTok];
                    tmem_ld16(lane_addr + buf * kTok, p);
                    tc_fence_before();
                    mbar_arrive(&tempty[buf]);
                    if (++buf == kTBufs) { buf = 0; bphase ^= 1u; }
#pragma unroll
                    for (int j = 0; j < kTok; ++j)
                        if (j < M) acc[j] = fmaf(p[j], wscale * srow[j], acc[j]);
                }
            }
        } else {
            if (__all_sync(0xffffffffu, mbar_wait(&tfull[0], 0, abort_flag, err, kSiteEpiFull))) {
                tc_fence_after();
                float p[kTok];
                tmem_ld16(lane_addr, p);
                tc_fence_before();
                if (MODE == kScaleTensor) {
                    const float sc = sa[0] * sw[0];
#pragma unroll
                    for (int j = 0; j < kTok; ++j) acc[j] = p[j] * sc;
                } else {  // per token (sa[j]) and per output channel (sw[n])
                    const int n = n0 + r;
                    const float swn = n < N ? __ldg(sw + n) : 0.0f;
#pragma unroll
                    for (int j = 0; j < kTok; ++j)
                        if (j < M) acc[j] = p[j] * (__ldg(sa + j) * swn);
                }
            }
        }
        if (splits == 1) {
            const int n = n0 + r;
            if (n < N) {
#pragma unroll
                for (int j = 0; j < kTok; ++j)
                    if (j < M) y[static_cast<int64_t>(j) * N + n] = __float2bfloat16_rn(acc[j]);
            }
        }
    }

    __syncwarp();  // lanes 1..31 of the producer and MMA warps wait for lane 0
    grid_dep_wait();  // every thread below may write Y

    if (splits > 1) {
        // ------------------------------------- cluster split-K reduction --
        // Rank q owns rows [q*rows_per, +rows_per). The operand stages are idle
        // once the last MMA has completed (the epilogue consumed its partial),
        // so they hold this CTA's partials in row order: rank q's slice is one
        // contiguous block, copied to [own rank] of q's receive buffer.
        const uint32_t rank = cluster_ctarank();
        const int rows_per = kRows / splits;
        const uint32_t slice_bytes = static_cast<uint32_t>(rows_per * kTok * 4);
        float *out = reinterpret_cast<float *>(sW);
        const bool issuer = warp == 4 && lane < splits;  // lane q copies rank q's slice
        if (warp >= 4) {
            const int r = (warp - 4) * 32 + lane;
            float4 *dst = reinterpret_cast<float4 *>(out + r * kTok);
#pragma unroll
            for (int j = 0; j < kTok / 4; ++j)
                dst[j] = make_float4(acc[4 * j], acc[4 * j + 1], acc[4 * j + 2], acc[4 * j + 3]);
            fence_proxy_async_smem();  // the bulk copies read these writes
            named_bar_sync(1, 128);
            if (issuer) {
                const uint32_t q = static_cast<uint32_t>(lane);
                bulk_copy_to_cluster(map_shared_rank(smem_u32(recv) + rank * slice_bytes, q),
                                     smem_u32(out) + q * slice_bytes, slice_bytes, map_shared_rank(smem_u32(rbar), q));
                bulk_commit();
            }
        }
        // Every rank pushes unconditionally, and a rank that stalls gives up
        // within one wait limit (the abort flag then short-circuits its other
        // waits), so this wait - which must not end before the data does, lest
        // a copy land in a CTA that has exited - takes a longer limit and does
        // not look at the abort flag.
        bool got = true;
        if (threadIdx.x % 32 == 0) {
            const uint64_t t0 = global_ns();
            while (!mbar_try_wait(rbar, 0)) {
                if (global_ns() - t0 > 4 * kWaitLimitNs) {
                    record_error(err, kErrTimeout, kSiteReduce);
                    got = false;
                    break;
                }
            }
        }
        got = __shfl_sync(0xffffffffu, got, 0) && mbar_try_wait(rbar, 0);
        if (__all_sync(0xffffffffu, got)) {
            const int row0 = static_cast<int>(rank) * rows_per;
            const int quads = (M + 3) / 4;
            const float4 *rv = reinterpret_cast<const float4 *>(recv);
            for (int idx = threadIdx.x; idx < rows_per * quads; idx += kThreads) {
                const int qd = idx / rows_per;
                const int rl = idx - qd * rows_per;
                float sum[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                for (int src = 0; src < splits; ++src) {  // fixed order: rank 0 first
                    const float4 v = rv[((src * rows_per + rl) * kTok) / 4 + qd];
                    sum[0] += v.x;
                    sum[1] += v.y;
                    sum[2] += v.z;
                    sum[3] += v.w;
                }
                const int n = n0 + row0 + rl;
                if (n < N) {
#pragma unroll
                    for (int t = 0; t < 4; ++t)
                        if (qd * 4 + t < M) y[static_cast<int64_t>(qd * 4 + t) * N + n] = __float2bfloat16_rn(sum[t]);
                }
            }
        }
        // The copies out of this CTA must have read their source before it
        // exits; everything addressed to it has landed (the wait above).
        if (issuer) bulk_wait_read();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

template <int MODE>
cudaError_t launch_variant(const void *qa, const float *sa, const void *qw, const float *sw, void *y, int64_t M,
                           int64_t N, int64_t K, const DeviceInfo &dev, cudaStream_t stream) {
    static std::once_flag attr_once[64];
    static cudaError_t attr_err[64];
    int device = 0;
    cudaGetDevice(&device);
    std::call_once(attr_once[device & 63], [&] {
        cudaError_t e = cudaFuncSetAttribute(gemm_decode_kernel<MODE>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        attr_err[device & 63] = e;
    });
    if (attr_err[device & 63] != cudaSuccess) return attr_err[device & 63];

    CUtensorMap tmW, tmX;
    if (encode_tma_2d_u8(&tmW, qw, K, N, K, BK, kRows) != CUDA_SUCCESS) return cudaErrorInvalidValue;
    if (encode_tma_2d_u8(&tmX, qa, K, M, K, BK, kTok) != CUDA_SUCCESS) return cudaErrorInvalidValue;

    const int64_t nblocks = (N + kRows - 1) / kRows;
    const int64_t Kg = (K + BK - 1) / BK;
    // Split K over a cluster as far as all CTAs still fit on the GPU at once
    // (two per SM), so that no CTA waits for a second wave.
    int splits = 1;
    while (splits < 8 && nblocks * splits * 2 <= 2 * dev.sm_count && splits * 2 <= Kg) splits *= 2;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(nblocks * splits));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(splits);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, gemm_decode_kernel<MODE>, tmW, tmX, sa, sw,
                              static_cast<__nv_bfloat16 *>(y), static_cast<int>(M), static_cast<int>(N),
                              static_cast<int>(K), splits, dev.err);
}

}  // namespace

cudaError_t launch_gemm_decode(const void *qa, const float *sa, const void *qw, const float *sw, void *y,
                               int64_t M, int64_t N, int64_t K, ScaleMode mode, const DeviceInfo &dev,
                               cudaStream_t stream) {
    if (mode == kScaleTensor) return launch_variant<kScaleTensor>(qa, sa, qw, sw, y, M, N, K, dev, stream);
    if (mode == kScaleRowCol) return launch_variant<kScaleRowCol>(qa, sa, qw, sw, y, M, N, K, dev, stream);
    return launch_variant<kScaleBlock>(qa, sa, qw, sw, y, M, N, K, dev, stream);
}

}  // namespace fp8k
