// Tile-persistent block-scaled FP8 GEMM for prefill-shaped (M > 16) and
// grouped (mixture-of-experts) problems, sm_103a.
//
//   Y[m,n] = bf16( sum_g Sa[g][m] Sw[n/128][g] sum_{k in g} dec(Qa[m,k]) dec(Qw[n,k]) )
//
// The pages only fix what is computed: FP8 operands into the tensor cores
// with high-precision accumulation ("FP8 and FP4: Throughput Needs Scaling",
// section "Kernel caveat가 마지막 관문이다") and 128x128 weight blocks with
// dynamic 128-groups for activations ("[vLLM] FP8", section "블록 양자화").
// The kernel below is this library's own design for GB300:
//
//  - one CTA per SM, persistent over output tiles of 128 x BN (BN = 128/256);
//  - warp 0 (one lane): TMA producer, fills a ring of shared-memory stages;
//    one stage = one 128-wide K block of A (128 x 128 B) and B (BN x 128 B),
//    both K-major with 128-byte swizzle;
//  - warp 1 owns TMEM; one lane of warp 1 (and, block-scaled, one of warp 2,
//    taking every other K block) issues 4 tcgen05.mma (K = 32 each) per stage
//    into a fresh TMEM accumulator, so a TMEM buffer holds the FP32 partial of
//    ONE K block; the 512 TMEM columns hold 512/BN such buffers, so the MMAs
//    run up to that many K blocks ahead of the promotion;
//  - warps 4..11 (two warpgroups): epilogue. Warp w reads TMEM lanes
//    32*(w%4).. (the lane quarter the hardware gives that warp) and one half
//    of the tile's columns; per K block each thread adds
//    partial * (Sa[m] * Sw) for its row into FP32 registers (the per-block
//    scale promotion). After the last K block the warp's 32 rows leave as BF16
//    through a 2 KB shared-memory buffer of its own, 32 columns at a time, by
//    TMA stores: the warp moves on to the next tile's K blocks while the
//    stores drain (a thread storing its own row instead wrote 32 rows per
//    instruction and held the promotion, and with it the MMAs, for the
//    whole drain);
//  - warpgroup 0 gives registers to the epilogue warpgroups (setmaxnreg);
//  - per-tensor mode: the MMAs accumulate all of K in TMEM; the epilogue
//    applies the single scale product once per tile, streaming TMEM to Y
//    through the same per-warp buffers and TMA stores;
//    row/column mode likewise, with sa[m] * sw[n] (per-token activation and
//    per-channel weight scales).
//
// Every wait is bounded (common.cuh); on expiry the CTA records an error,
// stops issuing, lets the copies and MMAs it issued finish and frees TMEM.
#include <mutex>

#include "common.cuh"
#include "launch.h"

namespace fp8k {
namespace {

constexpr int BM = 128;
constexpr int BK = 128;  // one K block: one stage, 4 MMAs of K = 32
constexpr int kThreads = 384;
constexpr int kEpiThreads = 256;
constexpr int kMaxGroups = 256;
constexpr int kTmemCols = 512;
// Output staging of the epilogue: per warp, 32 rows x 32 BF16
// columns (64-byte rows, 64-byte TMA swizzle), one TMA store box.
constexpr int kOutCols = 32;
constexpr int kOutWarpBytes = 32 * kOutCols * 2;
// Register split: warpgroup 0 shrinks, the two epilogue warpgroups grow.
// 128 * kLow + 256 * kHigh must not exceed 384 * (registers the kernel is
// compiled with); the launcher checks that before every launch. The 128 x 256
// block-scaled epilogue holds 128 accumulators and two 16-column load buffers
// per thread, so it takes the larger share.
template <int BN, bool WHOLE_K>
struct RegSplit {
    static constexpr bool kWide = BN == 256 && !WHOLE_K;
    static constexpr int kLow = kWide ? 56 : 72;
    static constexpr int kHigh = kWide ? 224 : 216;
    static_assert(128 * kLow + 256 * kHigh <= 384 * 168, "register split exceeds the launch budget");
};

// Bounded-wait sites reported through the error word.
enum : unsigned { kSiteProdEmpty = 101, kSiteMmaTmem = 102, kSiteMmaFull = 103, kSiteEpiFull = 104,
                  kSiteDrain = 105, kSiteOffsets = 106 };

template <int BN>
struct Cfg {
    static constexpr int kStages = BN == 128 ? 6 : 4;
    static constexpr int kABytes = BM * BK;
    static constexpr int kBBytes = BN * BK;
    static constexpr int kStageBytes = kABytes + kBBytes;
    static constexpr int kBufs = kTmemCols / BN;        // TMEM partial buffers
    static constexpr int kCols = BN / 2;                // columns per epilogue thread
    static constexpr int kChunk = BN == 128 ? 64 : 32;  // TMEM columns loaded per wait
    static constexpr int kBarrierBytes = 8 * (2 * kStages + 2 * kBufs) + 16;
    static constexpr int kTableBytes = 4 * (3 * kMaxGroups + 2);
    static constexpr int kOutBytes = 512 + 8 * kOutWarpBytes;  // output staging of the 8 epilogue warps, 512-byte aligned
    static constexpr int kSmemBytes = 1024 + kStages * kStageBytes + kBarrierBytes + kTableBytes + kOutBytes;
};

// Output tile of a linear tile index: rows [m0, m0+128) of which those below
// row_end are written, columns [n0, n0+BN), B rows from b_row, expert group.
struct Tile {
    int m0, row_end, n0, b_row, group;
};

template <int BN>
struct Sched {
    int M, N, num_n, num_m, raster, groups;
    const int *lo, *hi, *start;  // shared-memory tables (grouped only)

    __device__ __forceinline__ Tile get(int t) const {
        Tile r;
        int mt, nt;
        if (groups == 0) {
            if (raster == 0) { mt = t / num_n; nt = t - mt * num_n; }
            else             { nt = t / num_m; mt = t - nt * num_m; }
            r.m0 = mt * BM;
            r.row_end = M;
            r.group = 0;
        } else {
            int e = 0;
            while (e + 1 < groups && start[e + 1] <= t) ++e;
            const int local = t - start[e];
            mt = local / num_n;
            nt = local - mt * num_n;
            r.m0 = lo[e] + mt * BM;
            r.row_end = hi[e];
            r.group = e;
        }
        r.n0 = nt * BN;
        r.b_row = r.group * N + r.n0;
        return r;
    }
};

template <int CH>
__device__ __forceinline__ void tmem_ld_chunk(uint32_t taddr, float (&p)[CH]);
template <>
__device__ __forceinline__ void tmem_ld_chunk<64>(uint32_t taddr, float (&p)[64]) { tmem_ld64(taddr, p); }
template <>
__device__ __forceinline__ void tmem_ld_chunk<32>(uint32_t taddr, float (&p)[32]) { tmem_ld32(taddr, p); }

// Eight outputs p[j] * (s * sw[j]): one row scale, eight column scales.
__device__ __forceinline__ uint4 pack8_rowcol(const float *p, float s, const float *swp) {
    const float4 a = __ldg(reinterpret_cast<const float4 *>(swp));
    const float4 b = __ldg(reinterpret_cast<const float4 *>(swp + 4));
    uint4 v;
    v.x = pack_bf16x2(p[0] * (s * a.x), p[1] * (s * a.y));
    v.y = pack_bf16x2(p[2] * (s * a.z), p[3] * (s * a.w));
    v.z = pack_bf16x2(p[4] * (s * b.x), p[5] * (s * b.y));
    v.w = pack_bf16x2(p[6] * (s * b.z), p[7] * (s * b.w));
    return v;
}

__device__ __forceinline__ uint4 pack8_scaled(const float *p, float s) {
    uint4 v;
    v.x = pack_bf16x2(p[0] * s, p[1] * s);
    v.y = pack_bf16x2(p[2] * s, p[3] * s);
    v.z = pack_bf16x2(p[4] * s, p[5] * s);
    v.w = pack_bf16x2(p[6] * s, p[7] * s);
    return v;
}

// Bulk tensor store shared -> global (bulk async-group of the issuing thread).
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *map, uint32_t src, int x, int y) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(map), "r"(x),
                 "r"(y), "r"(src)
                 : "memory");
}

// Wait until this thread's bulk stores have completed (not only read shared memory).
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Columns [x, x + 32) of the warp's 32 output rows [row0, row0 + 32), lane l
// giving row l's four 16-byte chunks of BF16, through the warp's 2 KB buffer
// wbuf. Each lane writes its chunks in the 64-byte swizzle of the tensor map
// (chunk j of row r at j ^ ((r >> 1) & 3)), and lane 0 stores the 32 x 32 box;
// TMA leaves out rows >= M and columns >= N. Before refilling the buffer lane
// 0 waits until its previous store has read it. With use_tma false (rows that
// run past the end of an expert's range, which must not be written) the warp
// reads the buffer back and stores 8 rows x 64 bytes per instruction, each row
// checked against row_end.
__device__ __forceinline__ void store_box(const uint4 (&v)[4], uint8_t *wbuf, const CUtensorMap *tmY, int lane,
                                          int x, int row0, bool use_tma, __nv_bfloat16 *y, int M, int N,
                                          int row_end) {
    if (lane == 0) bulk_wait_read();
    __syncwarp();
#pragma unroll
    for (int j = 0; j < 4; ++j) *reinterpret_cast<uint4 *>(wbuf + lane * 64 + ((j ^ ((lane >> 1) & 3)) << 4)) = v[j];
    if (use_tma) {
        fence_proxy_async_smem();  // the TMA store reads these writes
        __syncwarp();
        if (lane == 0) {
            tma_store_2d(tmY, smem_u32(wbuf), x, row0);
            bulk_commit();
        }
    } else {
        __syncwarp();
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int rr = (lane >> 2) + 8 * i, jc = lane & 3;
            const uint4 w = *reinterpret_cast<const uint4 *>(wbuf + rr * 64 + ((jc ^ ((rr >> 1) & 3)) << 4));
            const int mr = row0 + rr, col = x + jc * 8;
            if (mr < M && mr < row_end && col < N) *reinterpret_cast<uint4 *>(y + static_cast<int64_t>(mr) * N + col) = w;
        }
        __syncwarp();
    }
}

template <int BN, int MODE>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_prefill_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmY,
                        const float *__restrict__ sa, const float *__restrict__ sw,
                        __nv_bfloat16 *__restrict__ y, int M, int N, int K, int groups,
                        const int32_t *__restrict__ offsets, int raster, unsigned *err) {
    using C = Cfg<BN>;
    constexpr bool WHOLE_K = MODE != kScaleBlock;  // all of K in one TMEM accumulator per tile
    constexpr uint32_t kIssuers = WHOLE_K ? 1u : 2u;  // MMA-issuing lanes
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sA = smem;
    uint8_t *sB = smem + C::kStages * C::kABytes;
    uint64_t *full = reinterpret_cast<uint64_t *>(sB + C::kStages * C::kBBytes);
    uint64_t *empty = full + C::kStages;
    uint64_t *tfull = empty + C::kStages;
    uint64_t *tempty = tfull + C::kBufs;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(tempty + C::kBufs);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    int *t_lo = reinterpret_cast<int *>(tmem_slot + 4);
    int *t_hi = t_lo + kMaxGroups;
    int *t_start = t_hi + kMaxGroups;
    uint8_t *s_out = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(t_lo) + C::kTableBytes + 511) & ~uintptr_t(511));

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int Kg = (K + BK - 1) / BK;
    const int num_n = (N + BN - 1) / BN;
    const int Nb = (N + 127) / 128;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
        for (int b = 0; b < C::kBufs; ++b) { mbar_init(&tfull[b], 1); mbar_init(&tempty[b], kEpiThreads); }
        *abort_flag = 0;
        fence_barrier_init();
        if (offsets != nullptr) {
            // Expert e owns rows [lo, hi) clamped into [0, M]; its tiles follow
            // those of experts < e (expert-major, n fastest within an expert).
            // Offsets that are not non-decreasing within [0, M] are a caller
            // error, recorded (by CTA 0) as FP8_ERR_ARG; they are clamped so
            // that no access leaves the buffers.
            int acc = 0;
            bool bad = false;
            for (int e = 0; e < groups; ++e) {
                int lo = offsets[e], hi = offsets[e + 1];
                bad |= lo < 0 || hi < lo || hi > M;
                lo = lo < 0 ? 0 : (lo > M ? M : lo);
                hi = hi < lo ? lo : (hi > M ? M : hi);
                t_lo[e] = lo;
                t_hi[e] = hi;
                t_start[e] = acc;
                acc += ((hi - lo + BM - 1) / BM) * num_n;
            }
            t_start[groups] = acc;
            if (bad && blockIdx.x == 0) record_error(err, kErrArg, kSiteOffsets);
        }
    }
    if (warp == 0 && lane == 0) { tma_prefetch_desc(&tmA); tma_prefetch_desc(&tmB); }
    if (warp == 1) { tmem_alloc(tmem_slot, kTmemCols); tmem_relinquish(); }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    Sched<BN> sched;
    sched.M = M; sched.N = N; sched.num_n = num_n; sched.num_m = (M + BM - 1) / BM; sched.raster = raster;
    sched.groups = offsets != nullptr ? groups : 0;
    sched.lo = t_lo; sched.hi = t_hi; sched.start = t_start;
    const int total = offsets != nullptr ? t_start[groups] : sched.num_m * num_n;

    if (warp < 4) {
        regs_shrink<RegSplit<BN, WHOLE_K>::kLow>();
        if (warp == 0 && lane == 0) {
            // ------------------------------------------------ TMA producer --
            uint32_t stage = 0, phase = 0;
            int issued = 0;
            for (int t = blockIdx.x; t < total && !*abort_flag; t += gridDim.x) {
                const Tile tl = sched.get(t);
                for (int kb = 0; kb < Kg; ++kb) {
                    if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, err, kSiteProdEmpty)) break;
                    mbar_arrive_expect_tx(&full[stage], C::kStageBytes);
                    tma_load_2d(sA + stage * C::kABytes, &tmA, &full[stage], kb * BK, tl.m0);
                    tma_load_2d(sB + stage * C::kBBytes, &tmB, &full[stage], kb * BK, tl.b_row);
                    ++issued;
                    if (++stage == C::kStages) { stage = 0; phase ^= 1u; }
                }
            }
            // Let the last fill of every stage land before the CTA can exit
            // (on the normal path these have all completed already).
            for (int i = 0; i < C::kStages && i < issued; ++i) {
                if (stage == 0) { stage = C::kStages; phase ^= 1u; }
                --stage;
                const uint64_t t0 = global_ns();
                while (!mbar_try_wait(&full[stage], phase)) {
                    if (global_ns() - t0 > kWaitLimitNs) { record_error(err, kErrTimeout, kSiteDrain); break; }
                }
            }
        } else if ((warp == 1 || (kIssuers == 2 && warp == 2)) && lane == 0) {
            // ------------------------------------------------ MMA issuers --
            // tcgen05.mma issue stalls while the tensor pipe is busy, so the
            // instructions an issuing lane runs between the last MMA of one K
            // block and the first of the next can leave the pipe idle. In
            // block-scaled mode every K block has a TMEM buffer of its own, so
            // two lanes (warps 1 and 2) take alternate K blocks: while one is
            // stalled feeding the pipe, the other has already waited for its
            // next buffer and stage. Each lane spins (test_wait), fences once
            // after both waits, and in block-scaled mode commits only to the
            // TMEM barrier (the epilogue, which learns from that barrier that
            // the K block's MMAs are done, frees the shared-memory stage). A
            // commit tracks the MMAs of the lane that issues it.
            constexpr uint32_t idesc = idesc_e4m3_f32(BM, BN);
            const uint32_t own = static_cast<uint32_t>(warp - 1);  // K blocks gi with gi % kIssuers == own
            uint32_t stage = 0, phase = 0, buf = 0, bphase = 0, gi = 0;
            uint64_t *last_bar = nullptr;
            uint32_t last_parity = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
                for (int kb = 0; kb < Kg && ok; ++kb, ++gi) {
                    if (gi % kIssuers == own) {
                        if (!WHOLE_K || kb == 0) {
                            ok = mbar_wait<true>(&tempty[buf], bphase ^ 1u, abort_flag, err, kSiteMmaTmem);
                            if (!ok) break;
                        }
                        ok = mbar_wait<true>(&full[stage], phase, abort_flag, err, kSiteMmaFull);
                        if (!ok) break;
                        tc_fence_after();
                        const uint32_t a0 = smem_u32(sA + stage * C::kABytes);
                        const uint32_t b0 = smem_u32(sB + stage * C::kBBytes);
                        const uint32_t d = tmem_base + buf * BN;
#pragma unroll
                        for (int k = 0; k < BK / 32; ++k) {
                            const uint32_t acc = (k > 0 || (WHOLE_K && kb > 0)) ? 1u : 0u;
                            umma_e4m3(d, sdesc_k_sw128(a0 + k * 32), sdesc_k_sw128(b0 + k * 32), idesc, acc);
                        }
                        if (WHOLE_K) {
                            umma_commit(&empty[stage]);
                            last_bar = &empty[stage];
                            last_parity = phase;
                        }
                        if (!WHOLE_K || kb == Kg - 1) {
                            umma_commit(&tfull[buf]);
                            last_bar = &tfull[buf];
                            last_parity = bphase;
                        }
                    }
                    if (!WHOLE_K || kb == Kg - 1) {
                        if (++buf == C::kBufs) { buf = 0; bphase ^= 1u; }
                    }
                    if (++stage == C::kStages) { stage = 0; phase ^= 1u; }
                }
            }
            // The last commit arrives once every MMA issued by this lane has
            // finished reading shared memory and writing TMEM; wait for it
            // before the CTA frees TMEM (already complete on the normal path).
            if (last_bar != nullptr) {
                const uint64_t t0 = global_ns();
                while (!mbar_try_wait(last_bar, last_parity)) {
                    if (global_ns() - t0 > kWaitLimitNs) { record_error(err, kErrTimeout, kSiteDrain); break; }
                }
            }
        }
        __syncwarp();  // lanes 1..31 wait for their lane 0
    } else {
        regs_grow<RegSplit<BN, WHOLE_K>::kHigh>();
        // ------------------------------------------------------ epilogue --
        const int quarter = warp & 3;      // TMEM lane quarter this warp may access
        const int half = (warp - 4) >> 2;  // which half of the tile's columns
        const int r = quarter * 32 + lane; // row within the tile
        const int c0 = half * C::kCols;    // first column within the tile
        const uint32_t lane_addr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + c0;
        uint32_t buf = 0, bphase = 0;
        uint32_t stage = 0;  // shared-memory stage of the current K block (block-scaled mode)
        const bool frees_stages = (warp == 4 && lane == 0);
        float tensor_scale = 0.0f;
        if (MODE == kScaleTensor) tensor_scale = sa[0] * sw[0];
        bool ok = true;
        for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
            const Tile tl = sched.get(t);
            const int m = tl.m0 + r;
            const bool row_in = m < M;
            const int row0 = tl.m0 + quarter * 32;                     // the warp's first output row
            uint8_t *const wbuf = s_out + (warp - 4) * kOutWarpBytes;  // its output staging buffer
            if (!WHOLE_K) {
                float acc[C::kCols];
#pragma unroll
                for (int j = 0; j < C::kCols; ++j) acc[j] = 0.0f;
                const int nb = (tl.n0 + c0) / 128;  // this half lies in one 128-column weight block
                const float *swp = sw + (static_cast<int64_t>(tl.group) * Nb + (nb < Nb ? nb : Nb - 1)) * Kg;
                const float *sap = sa + m;
                // Scales of K blocks kb+1 and kb+2 are in flight while block kb is promoted.
                float sa1 = row_in ? __ldg(sap) : 0.0f, sw1 = __ldg(swp);
                float sa2 = (row_in && Kg > 1) ? __ldg(sap + M) : 0.0f, sw2 = Kg > 1 ? __ldg(swp + 1) : 0.0f;
                for (int kb = 0; kb < Kg; ++kb) {
                    const float sc = sa1 * sw1;
                    sa1 = sa2;
                    sw1 = sw2;
                    if (kb + 2 < Kg) {
                        sa2 = row_in ? __ldg(sap + static_cast<int64_t>(kb + 2) * M) : 0.0f;
                        sw2 = __ldg(swp + kb + 2);
                    }
                    ok = __all_sync(0xffffffffu, mbar_wait(&tfull[buf], bphase, abort_flag, err, kSiteEpiFull));
                    if (!ok) break;
                    tc_fence_after();
                    // The K block's MMAs are complete, so its operand stage is free.
                    if (frees_stages) mbar_arrive(&empty[stage]);
                    if (++stage == C::kStages) stage = 0;
                    // 16-column chunks, software-pipelined: the load of chunk
                    // c+1 is in flight while chunk c is promoted. The buffer is
                    // released as soon as its last chunk is in registers. (The
                    // small chunks keep the 128-accumulator epilogue free of
                    // register spills; a spilled, reloaded scale in this loop
                    // cost a third of the kernel's throughput.)
                    constexpr int kCh = 16, kN = C::kCols / kCh;
                    const uint32_t base = lane_addr + buf * BN;
                    uint32_t u[2][kCh];
                    tmem_ld16_async(base, u[0]);
                    tmem_wait16(u[0]);
#pragma unroll
                    for (int c = 0; c < kN; ++c) {
                        if (c + 1 < kN) {
                            tmem_ld16_async(base + (c + 1) * kCh, u[(c + 1) & 1]);
                        } else {
                            tc_fence_before();
                            mbar_arrive(&tempty[buf]);
                        }
#pragma unroll
                        for (int j = 0; j < kCh; ++j)
                            acc[c * kCh + j] = fmaf(__uint_as_float(u[c & 1][j]), sc, acc[c * kCh + j]);
                        if (c + 1 < kN) tmem_wait16(u[(c + 1) & 1]);
                    }
                    if (++buf == C::kBufs) { buf = 0; bphase ^= 1u; }
                }
                if (!ok) break;
                // Output: the warp's 32 rows, 32 columns at a time.
                const bool use_tma = row0 + 32 <= tl.row_end || tl.row_end >= M;
#pragma unroll
                for (int q = 0; q < C::kCols / kOutCols; ++q) {
                    uint4 v[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j) v[j] = pack8_scaled(acc + q * kOutCols + j * 8, 1.0f);
                    store_box(v, wbuf, &tmY, lane, tl.n0 + c0 + q * kOutCols, row0, use_tma, y, M, N, tl.row_end);
                }
            } else {
                const float srow = (MODE == kScaleRowCol && row_in) ? __ldg(sa + m) : 0.0f;
                ok = __all_sync(0xffffffffu, mbar_wait(&tfull[buf], bphase, abort_flag, err, kSiteEpiFull));
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int c = 0; c < C::kCols / C::kChunk; ++c) {
                    float p[C::kChunk];
                    tmem_ld_chunk<C::kChunk>(lane_addr + buf * BN + c * C::kChunk, p);
                    if (c == C::kCols / C::kChunk - 1) {
                        tc_fence_before();
                        mbar_arrive(&tempty[buf]);
                    }
#pragma unroll
                    for (int q = 0; q < C::kChunk / kOutCols; ++q) {
                        // Row/column mode: this row's token scale times each
                        // column's channel scale (loaded per 8 columns; columns
                        // past N, which the store leaves out, read column 0's).
                        const int x = tl.n0 + c0 + c * C::kChunk + q * kOutCols;
                        uint4 v[4];
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const float *pj = p + q * kOutCols + j * 8;
                            if (MODE == kScaleRowCol)
                                v[j] = pack8_rowcol(pj, srow, sw + (x + j * 8 < N ? x + j * 8 : 0));
                            else
                                v[j] = pack8_scaled(pj, tensor_scale);
                        }
                        store_box(v, wbuf, &tmY, lane, x, row0, true, y, M, N, M);
                    }
                }
                if (++buf == C::kBufs) { buf = 0; bphase ^= 1u; }
            }
        }
    }

    if (warp >= 4 && lane == 0) bulk_wait_all();  // this warp's output stores have landed
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

template <int BN, int MODE>
cudaError_t launch_variant(const void *qa, const float *sa, const void *qw, const float *sw, void *y, int64_t M,
                           int64_t N, int64_t K, int num_groups, const int32_t *offsets, const DeviceInfo &dev,
                           cudaStream_t stream) {
    using C = Cfg<BN>;
    static std::once_flag attr_once[64];
    static cudaError_t attr_err[64];
    int device = 0;
    cudaGetDevice(&device);
    std::call_once(attr_once[device & 63], [&] {
        cudaError_t e = cudaFuncSetAttribute(gemm_prefill_kernel<BN, MODE>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
        // The register re-split inside the kernel needs the launch to hold at
        // least 128 * kLow + 256 * kHigh registers; refuse otherwise.
        using S = RegSplit<BN, MODE != kScaleBlock>;
        cudaFuncAttributes fa;
        if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, gemm_prefill_kernel<BN, MODE>);
        if (e == cudaSuccess && fa.numRegs * kThreads < 128 * S::kLow + 256 * S::kHigh)
            e = cudaErrorInvalidConfiguration;
        attr_err[device & 63] = e;
    });
    if (attr_err[device & 63] != cudaSuccess) return attr_err[device & 63];

    CUtensorMap tmA, tmB;
    if (encode_tma_2d_u8(&tmA, qa, K, M, K, BK, BM) != CUDA_SUCCESS) return cudaErrorInvalidValue;
    const int64_t b_rows = N * (offsets != nullptr ? num_groups : 1);
    if (encode_tma_2d_u8(&tmB, qw, K, b_rows, K, BK, BN) != CUDA_SUCCESS) return cudaErrorInvalidValue;
    CUtensorMap tmY;
    if (encode_tma_2d_bf16_sw64(&tmY, y, N, M, kOutCols, 32) != CUDA_SUCCESS) return cudaErrorInvalidValue;

    int64_t tiles;
    const int64_t num_n = (N + BN - 1) / BN;
    if (offsets == nullptr) tiles = ((M + BM - 1) / BM) * num_n;
    else tiles = ((M + BM - 1) / BM + num_groups) * num_n;  // upper bound
    const int64_t grid = tiles < dev.sm_count ? tiles : dev.sm_count;
    if (grid <= 0) return cudaSuccess;
    // Tiles sharing a row panel run together when the weight operand is the
    // smaller one (it stays in L2 while activations stream), else the reverse.
    const int raster = (N <= M) ? 0 : 1;
    gemm_prefill_kernel<BN, MODE><<<static_cast<unsigned>(grid), kThreads, C::kSmemBytes, stream>>>(
        tmA, tmB, tmY, sa, sw, static_cast<__nv_bfloat16 *>(y), static_cast<int>(M), static_cast<int>(N),
        static_cast<int>(K), num_groups, offsets, raster, dev.err);
    return cudaGetLastError();
}

// Tile width: 256 when N is a multiple of 256, else 128.
int pick_bn(int64_t N) { return (N % 256 == 0) ? 256 : 128; }

}  // namespace

cudaError_t launch_gemm_prefill(const void *qa, const float *sa, const void *qw, const float *sw, void *y,
                                int64_t M, int64_t N, int64_t K, int num_groups, const int32_t *offsets,
                                ScaleMode mode, const DeviceInfo &dev, cudaStream_t stream) {
    const int bn = pick_bn(N);
#define FP8_PREFILL_LAUNCH(MODE_)                                                                              \
    return bn == 256 ? launch_variant<256, MODE_>(qa, sa, qw, sw, y, M, N, K, num_groups, offsets, dev, stream) \
                     : launch_variant<128, MODE_>(qa, sa, qw, sw, y, M, N, K, num_groups, offsets, dev, stream)
    if (mode == kScaleTensor) FP8_PREFILL_LAUNCH(kScaleTensor);
    if (mode == kScaleRowCol) FP8_PREFILL_LAUNCH(kScaleRowCol);
    FP8_PREFILL_LAUNCH(kScaleBlock);
#undef FP8_PREFILL_LAUNCH
}

}  // namespace fp8k
