// Test hooks (not part of the computation):
//  - the bounded device waits: the same mbarrier wait, error word and abort
//    flag the GEMM kernels use, driven to expiry on purpose. Nothing in it
//    faults or hangs: the waits are on shared-memory mbarriers that nobody
//    arrives at, and each gives up by the %globaltimer limit;
//  - the hardware E4M3 conversion the quantizers use (round to nearest even,
//    saturating), applied to a range of FP32 bit patterns, so that it can be
//    compared with an independent encoder on every FP32 value.
#include "common.cuh"
#include "launch.h"

namespace fp8k {
namespace {

constexpr unsigned kSiteSelftest = 901;     // the first waiter, which times out
constexpr unsigned kSiteSelftestLate = 902; // the second, which should only see the abort
constexpr uint64_t kLateStartNs = kWaitLimitNs / 2;

// Thread 0 waits on bar[0]; thread 32 starts waiting on bar[1] half a wait
// limit later. Thread 0 gives up first, records FP8_ERR_TIMEOUT with its site
// and raises the CTA's abort flag; thread 32 then returns at the flag, half
// a limit before its own expiry, without recording anything.
__global__ void selftest_wait_kernel(unsigned *err) {
    __shared__ uint64_t bar[2];
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar[0], 1);
        mbar_init(&bar[1], 1);
        abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        mbar_wait(&bar[0], 0, &abort_flag, err, kSiteSelftest);
    } else if (threadIdx.x == 32) {
        const uint64_t t0 = global_ns();
        while (global_ns() - t0 < kLateStartNs) {
        }
        mbar_wait(&bar[1], 0, &abort_flag, err, kSiteSelftestLate);
    }
    __syncthreads();
}

// The two codes of the FP32 values with bit patterns a and b (low byte = a).
__device__ __forceinline__ uint32_t e4m3_of_bits(uint32_t a, uint32_t b) {
    return static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(make_float2(__uint_as_float(a), __uint_as_float(b)),
                                                          __NV_SATFINITE, __NV_E4M3));
}

// out[8i .. 8i+7] = codes of the patterns first + 8i .. first + 8i + 7, for
// i < n8, grid-stride; one 8-byte store per step. The caller keeps
// first + 8 * n8 <= 2^32, so no pattern wraps.
__global__ void selftest_encode_kernel(uint32_t first, int64_t n8, uint2 *out) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n8; i += stride) {
        const uint32_t b = first + static_cast<uint32_t>(i * 8);
        uint2 v;
        v.x = e4m3_of_bits(b, b + 1) | (e4m3_of_bits(b + 2, b + 3) << 16);
        v.y = e4m3_of_bits(b + 4, b + 5) | (e4m3_of_bits(b + 6, b + 7) << 16);
        out[i] = v;
    }
}

}  // namespace

cudaError_t launch_selftest_encode(uint32_t first, int64_t n, void *out, const DeviceInfo &dev,
                                   cudaStream_t stream) {
    const int64_t n8 = n / 8;  // n is a multiple of 8
    if (n8 == 0) return cudaSuccess;
    constexpr int kThreadsPerBlock = 256;
    const int64_t cap = static_cast<int64_t>(dev.sm_count) * 8;
    int64_t blocks = (n8 + kThreadsPerBlock - 1) / kThreadsPerBlock;
    if (blocks > cap) blocks = cap;
    selftest_encode_kernel<<<static_cast<unsigned>(blocks), kThreadsPerBlock, 0, stream>>>(
        first, n8, static_cast<uint2 *>(out));
    return cudaGetLastError();
}

cudaError_t launch_selftest_wait(const DeviceInfo &dev, cudaStream_t stream) {
    selftest_wait_kernel<<<1, 64, 0, stream>>>(dev.err);
    return cudaGetLastError();
}

}  // namespace fp8k
