// common.cuh -- device helpers shared by the sm_103a kernels of libskv.
//
// 16-byte vector loads/stores with cache hints, dtype conversion to and from
// fp32, the merge guards ([FA] §2.2 sanitize, [F2] §⑤ fmax guard), mbarrier
// and bulk-copy (TMA) wrappers with bounded waits, programmatic dependent
// launch controls, and the per-device error word.
//
// Pages cited: [F2] "F2 讲解：merge_state，以 2 为底的 LSE 合并",
// [FA] "FlashAttention 的空行 LSE:FA-2 的 +inf 约定与后来的变化".
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/skv.h"

#define SKV_DEVINL __device__ __forceinline__

namespace skv {

// ------------------------------------------------------------------ error word
// One word per device (defined in api.cu, its address handed to every kernel
// that can detect an error): the first device-side error wins.  code in the
// low 8 bits, detail above.  Read and cleared by skv_get_device_error().
SKV_DEVINL void record_error(unsigned long long* word, int code, int detail) {
    unsigned long long w = ((unsigned long long)(unsigned)detail << 8) | (unsigned)code;
    atomicCAS(word, 0ull, w);
}

// ------------------------------------------------------------------ dtypes
template <typename T> struct Vec;  // 16-byte vector of T
template <> struct Vec<float> { static constexpr int N = 4; };
template <> struct Vec<__half> { static constexpr int N = 8; };
template <> struct Vec<__nv_bfloat16> { static constexpr int N = 8; };

SKV_DEVINL void unpack(const uint4& r, float (&f)[4]) {
    f[0] = __uint_as_float(r.x); f[1] = __uint_as_float(r.y);
    f[2] = __uint_as_float(r.z); f[3] = __uint_as_float(r.w);
}
SKV_DEVINL void unpack_h(const uint4& r, float (&f)[8]) {
    const __half2* h = reinterpret_cast<const __half2*>(&r);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float2 t = __half22float2(h[i]);
        f[2 * i] = t.x; f[2 * i + 1] = t.y;
    }
}
SKV_DEVINL void unpack_b(const uint4& r, float (&f)[8]) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&r);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float2 t = __bfloat1622float2(h[i]);
        f[2 * i] = t.x; f[2 * i + 1] = t.y;
    }
}

template <typename T> SKV_DEVINL void to_float(const uint4& r, float (&f)[Vec<T>::N]);
template <> SKV_DEVINL void to_float<float>(const uint4& r, float (&f)[4]) { unpack(r, f); }
template <> SKV_DEVINL void to_float<__half>(const uint4& r, float (&f)[8]) { unpack_h(r, f); }
template <> SKV_DEVINL void to_float<__nv_bfloat16>(const uint4& r, float (&f)[8]) { unpack_b(r, f); }

template <typename T> SKV_DEVINL uint4 from_float(const float (&f)[Vec<T>::N]);
template <> SKV_DEVINL uint4 from_float<float>(const float (&f)[4]) {
    return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                      __float_as_uint(f[3]));
}
template <> SKV_DEVINL uint4 from_float<__half>(const float (&f)[8]) {
    uint4 r;
    __half2* h = reinterpret_cast<__half2*>(&r);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2half2_rn(f[2 * i], f[2 * i + 1]);
    return r;
}
template <> SKV_DEVINL uint4 from_float<__nv_bfloat16>(const float (&f)[8]) {
    uint4 r;
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&r);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
    return r;
}

// ------------------------------------------------------------------ memory
// Streaming read of data that is read-only for the whole kernel: bypass L1,
// ask L2 to fetch the whole 256-byte line.
SKV_DEVINL uint4 ld_stream(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
    return r;
}
// Read-only load the compiler must keep in registers: volatile asm cannot be
// re-executed later to rematerialise the value (used for loop-invariant data
// such as the query of a decode CTA).
SKV_DEVINL uint4 ld_pinned(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
    return r;
}
// Read of data this kernel may later overwrite (in-place merge): coherent path.
SKV_DEVINL uint4 ld_coherent(const void* p) {
    uint4 r;
    asm volatile("ld.global.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p) : "memory");
    return r;
}
// Read of data written by another CTA of this grid or by a previous grid in
// the same stream (L2 is the point of coherence).
SKV_DEVINL uint4 ld_cg(const void* p) {
    uint4 r;
    asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p) : "memory");
    return r;
}
SKV_DEVINL float ld_cg_f32(const float* p) {
    float r;
    asm volatile("ld.global.cg.f32 %0, [%1];" : "=f"(r) : "l"(p) : "memory");
    return r;
}
// Streaming store (evict-first): outputs are not re-read by this kernel.
SKV_DEVINL void st_stream(void* p, const uint4& r) {
    asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};"
                 :: "l"(p), "r"(r.x), "r"(r.y), "r"(r.z), "r"(r.w) : "memory");
}

// ------------------------------------------------------------------ merge guards
// [FA] §2.2: an incoming LSE that is NaN or +inf carries no weight.
SKV_DEVINL float sanitize_lse(float s) {
    return (isnan(s) || s == INFINITY) ? -INFINITY : s;
}
// [F2] §⑤: 2^(s - m) with fmax(NaN, -inf) = -inf, so two empty states
// (s = m = -inf) get weight 0 instead of NaN.
SKV_DEVINL float merge_weight(float s, float m) {
    return exp2f(fmaxf(s - m, -INFINITY));
}

// 2^x by the hardware approximation (ex2.approx, relative error about
// 2^-22, subnormal results flushed to 0): softmax weights, where that error
// is far below the fp16 rounding of p.
SKV_DEVINL float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// ------------------------------------------------------------------ warp helpers
SKV_DEVINL float warp_max(float x, int width = 32) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1)
        if (o < width) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}
SKV_DEVINL float warp_sum(float x, int width = 32) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1)
        if (o < width) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// ------------------------------------------------------------------ PDL
// Programmatic dependent launch: the primary grid lets the dependent grid be
// scheduled early; the dependent grid waits here until the primary grid has
// completed and its writes are visible.
SKV_DEVINL void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
SKV_DEVINL void pdl_wait_primary() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
// Completion chaining for a grid launched as a programmatic dependent of
// the preceding grid in its stream without reading anything that grid
// writes: every CTA counts itself on *ctr (zeroed before this grid
// started) at its very end, and the last one to do so waits for the
// preceding grid to complete, so that this grid completes after it and a
// kernel that waits for this grid also sees the preceding grid's writes.
// Every CTA of the grid must call this exactly once; ctr == nullptr: no-op.
SKV_DEVINL void last_cta_waits_primary(unsigned int* ctr) {
    if (ctr == nullptr) return;
    __syncthreads();
    if (threadIdx.x == 0) {
        const unsigned total = gridDim.x * gridDim.y * gridDim.z;
        if (atomicAdd(ctr, 1u) == total - 1u) pdl_wait_primary();
    }
}

// ------------------------------------------------------------------ mbarrier / bulk copy
SKV_DEVINL uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
SKV_DEVINL void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(smem_addr(bar)), "r"(count)
                 : "memory");
}
SKV_DEVINL void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
SKV_DEVINL void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                 :: "r"(smem_addr(bar)), "r"(bytes) : "memory");
}
SKV_DEVINL void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(smem_addr(bar)) : "memory");
}
SKV_DEVINL bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok) : "r"(smem_addr(bar)), "r"(parity) : "memory");
    return ok != 0;
}
// As mbar_try_wait, but the thread may be suspended until the phase
// completes (at most about 20 us), so a waiting warp does not take issue
// slots from the warps doing the work.
SKV_DEVINL bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok) : "r"(smem_addr(bar)), "r"(parity), "r"(20000u) : "memory");
    return ok != 0;
}
SKV_DEVINL uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// Bounded wait: gives up after `limit_ns` of wall time (%globaltimer),
// records SKV_ERR_TIMEOUT with `where` as detail and returns false.  The
// kernels use kWaitLimitNs; skv_selftest_bounded_wait passes a short limit.
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s
static __device__ __noinline__ bool mbar_wait_slow(uint64_t* bar, uint32_t parity,
                                                    unsigned long long* err, int where,
                                                    uint64_t limit_ns) {
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (mbar_try_wait_sleep(bar, parity)) return true;
        if (globaltimer_ns() - t0 > limit_ns) {
            record_error(err, SKV_ERR_TIMEOUT, where);
            return false;
        }
    }
}
SKV_DEVINL bool mbar_wait(uint64_t* bar, uint32_t parity, unsigned long long* err, int where,
                          uint64_t limit_ns = kWaitLimitNs) {
    if (mbar_try_wait(bar, parity)) return true;
    return mbar_wait_slow(bar, parity, err, where, limit_ns);
}
// Bounded wait that also gives up as soon as another role of the CTA has
// raised the shared abort flag; a wait that runs out raises it.  The first
// poll is inline; the loop is a call, so the many wait sites of a
// warp-specialised kernel add little code (its warps run different code
// and share the instruction cache).
static __device__ __noinline__ bool wait_or_abort_slow(uint64_t* bar, uint32_t parity,
                                                 volatile int* abort_flag,
                                                 unsigned long long* err, int where,
                                                 uint64_t limit_ns) {
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (mbar_try_wait_sleep(bar, parity)) return true;
        if (*abort_flag) return false;
        if (globaltimer_ns() - t0 > limit_ns) {
            record_error(err, SKV_ERR_TIMEOUT, where);
            *abort_flag = 1;
            return false;
        }
    }
}
SKV_DEVINL bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                              unsigned long long* err, int where,
                              uint64_t limit_ns = kWaitLimitNs) {
    if (mbar_try_wait(bar, parity)) return true;
    return wait_or_abort_slow(bar, parity, abort_flag, err, where, limit_ns);
}
// 16-byte asynchronous global -> shared copy (cp.async, bypassing L1), and
// an arrive on `bar` once every cp.async of this thread so far has landed
// (the barrier's pending count is raised first, so its expected count is
// unchanged).
SKV_DEVINL void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" :: "r"(smem_addr(dst)), "l"(src)
                 : "memory");
}
SKV_DEVINL void cp_async_mbar_arrive(uint64_t* bar) {
    asm volatile("cp.async.mbarrier.arrive.shared::cta.b64 [%0];" :: "r"(smem_addr(bar)) : "memory");
}
// One contiguous global -> shared copy on the TMA engine, completion counted
// in bytes on `bar`.  dst, src 16-byte aligned, bytes a multiple of 16.
SKV_DEVINL void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                         uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;"
        :: "r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}
SKV_DEVINL uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

}  // namespace skv
