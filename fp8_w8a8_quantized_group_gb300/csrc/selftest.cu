// Self-test of the bounded device waits: the same mbarrier wait, error word
// and abort flag the GEMM kernels use, driven to expiry on purpose. Nothing
// in it faults or hangs: the waits are on shared-memory mbarriers that nobody
// arrives at, and each gives up by the %globaltimer limit.
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

}  // namespace

cudaError_t launch_selftest_wait(const DeviceInfo &dev, cudaStream_t stream) {
    selftest_wait_kernel<<<1, 64, 0, stream>>>(dev.err);
    return cudaGetLastError();
}

}  // namespace fp8k
