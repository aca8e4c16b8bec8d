// selftest.cu -- skv_selftest_bounded_wait: runs the bounded mbarrier waits
// that every kernel of this library uses on barriers that nothing completes,
// so that the give-up path (error word, abort flag, return) is exercised
// without any fault: no copy is issued, nothing is left in flight, and the
// kernel returns normally.
#include "common.cuh"
#include "kernels.h"

namespace skv {
namespace {

// Detail codes recorded with SKV_ERR_TIMEOUT by the self-test waits.
constexpr int kWhereWait = 100;   // mbar_wait
constexpr int kWhereAbort = 101;  // wait_or_abort, the warp whose limit runs out

__global__ void __launch_bounds__(64) bounded_wait_selftest_kernel(int mode, uint64_t limit_ns,
                                                                   unsigned long long* err) {
    __shared__ __align__(8) uint64_t bars[2];
    __shared__ int abort_flag;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        mbar_init(&bars[0], 1);  // nothing ever arrives on either barrier
        mbar_init(&bars[1], 1);
        fence_mbar_init();
        abort_flag = 0;
    }
    __syncthreads();
    if (mode == 0) {
        // The wait of the decode and merge kernels: one lane of warp 0.
        if (warp == 0 && lane == 0) mbar_wait(&bars[0], 0, err, kWhereWait, limit_ns);
    } else if (lane == 0) {
        // The abort-aware wait of the warp-specialised kernels: warp 0's limit
        // runs out and raises the flag; warp 1, with a limit 100 times
        // longer, must leave as soon as it sees the flag, recording nothing.
        volatile int* flag = &abort_flag;
        if (warp == 0)
            wait_or_abort(&bars[0], 0, flag, err, kWhereAbort, limit_ns);
        else
            wait_or_abort(&bars[1], 0, flag, err, kWhereAbort + 1, 100 * limit_ns);
    }
}

}  // namespace
}  // namespace skv

using namespace skv;

extern "C" skv_status skv_selftest_bounded_wait(int32_t mode, int64_t limit_ns,
                                                skv_stream_t stream) {
    if ((mode != 0 && mode != 1) || limit_ns < 1000 || limit_ns > 10000000)
        return SKV_ERR_INVALID_ARG;
    const DeviceInfo* dev = nullptr;
    skv_status st = current_device(&dev);
    if (st != SKV_OK) return st;
    bounded_wait_selftest_kernel<<<1, 64, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        mode, (uint64_t)limit_ns, dev->err);
    return cudaGetLastError() == cudaSuccess ? SKV_OK : SKV_ERR_CUDA;
}
