// noalloc.cu -- skv_merge_states_noalloc: the N-state merge for callers that
// cannot allocate device memory.
//
// Some callers of this library have no way to call cudaMalloc: a plugin that
// runs inside another runtime which owns every allocation and hands the
// plugin only its input and output buffers, or a latency-critical decode loop
// where an allocation (which may synchronise the device) is not acceptable.
// skv_merge_states needs a caller-provided workspace for its two-level path;
// this entry point instead uses a fixed scratch array that lives in the
// library's own device memory, so the caller passes only inputs and outputs.
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace skv {
namespace {

// The scratch array: one per GPU that loads the library, held until exit.
constexpr size_t kScratchBytes = SKV_MERGE_STATES_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Device address of this device's scratch array.  In host code the array's
// name is only a host-side stand-in, so the address is looked up once per
// device, with that device current, and cached.
skv_status scratch_address(int device, void** out) {
    if (device < 0 || device >= kMaxDevices) return SKV_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (g_scratch_ptr[device] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
            return SKV_ERR_CUDA;
        g_scratch_ptr[device] = p;
    }
    *out = g_scratch_ptr[device];
    return SKV_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

}  // namespace
}  // namespace skv

using namespace skv;

extern "C" size_t skv_merge_states_noalloc_scratch_size(int64_t S, int64_t N, int64_t H,
                                                        int64_t D, skv_dtype dtype,
                                                        int32_t sm_count) {
    if (S <= 0 || H <= 0 || N < 1 || D < 1 || sm_count < 0) return 0;
    if (!(dtype == SKV_F32 || dtype == SKV_F16 || dtype == SKV_BF16)) return 0;
    const int64_t row_bytes = D * (int64_t)dtype_size(dtype);
    if (row_bytes % 16 != 0 || row_bytes > 512) return 0;
    if (sm_count == 0) {
        const DeviceInfo* dev = nullptr;
        if (current_device(&dev) != SKV_OK) return 0;
        sm_count = dev->sm_count;
    }
    return plan_merge_states(S * H, N, D, (int)(row_bytes / 16), sm_count, SIZE_MAX,
                             kMergeCtasPerSm, false).ws_bytes;
}

extern "C" skv_status skv_merge_states_noalloc(const void* v, const float* s, void* v_out,
                                               float* s_out, int64_t S, int64_t N, int64_t H,
                                               int64_t D, skv_dtype dtype, skv_stream_t stream) {
    if (S < 0 || H < 0 || N < 1) return SKV_ERR_INVALID_ARG;
    if (!(dtype == SKV_F32 || dtype == SKV_F16 || dtype == SKV_BF16) || D < 1)
        return SKV_ERR_INVALID_ARG;
    const int64_t row_bytes = D * (int64_t)dtype_size(dtype);
    if (row_bytes % 16 != 0) return SKV_ERR_INVALID_ARG;
    if (row_bytes > 512) return SKV_ERR_UNSUPPORTED;
    if (S * H == 0) return SKV_OK;
    if (N > (int64_t)INT32_MAX || S * H > (int64_t)INT32_MAX) return SKV_ERR_UNSUPPORTED;
    if (!v || !s || !v_out || !s_out) return SKV_ERR_INVALID_ARG;
    if (!aligned16(v) || !aligned16(v_out) || !aligned4(s) || !aligned4(s_out))
        return SKV_ERR_INVALID_ARG;
    const DeviceInfo* dev = nullptr;
    skv_status st = current_device(&dev);
    if (st != SKV_OK) return st;
    // The scratch this call would use with no size limit; reject what does
    // not fit in the fixed array rather than silently taking another path.
    const int chunks = (int)(row_bytes / 16);
    const MergeStatesPlan want =
        plan_merge_states(S * H, N, D, chunks, dev->sm_count, SIZE_MAX, kMergeCtasPerSm, false);
    if (want.ws_bytes > kScratchBytes) return SKV_ERR_UNSUPPORTED;
    void* scratch = nullptr;
    if ((st = scratch_address(dev->device, &scratch)) != SKV_OK) return st;
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    // The array keeps whatever the previous call left; the arrival counters
    // of the two-level merge must start at zero.
    if (want.ws_bytes > 0 && cudaMemsetAsync(scratch, 0, want.ws_bytes, cs) != cudaSuccess)
        return SKV_ERR_CUDA;
    cudaError_t e = launch_merge_states(v, s, v_out, s_out, S, N, H, D, dtype, scratch,
                                        kScratchBytes, kMergeCtasPerSm, false, *dev, cs);
    return e == cudaSuccess ? SKV_OK : SKV_ERR_CUDA;
}
