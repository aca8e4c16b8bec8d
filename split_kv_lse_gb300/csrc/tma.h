// tma.h -- host-side encoding of TMA tensor maps (CUtensorMap) and the
// device-side tiled bulk-tensor copy.
//
// The driver's cuTensorMapEncodeTiled is reached through the runtime's
// driver-entry-point query, so libskv needs no link against libcuda and
// still loads on a machine without a GPU.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace skv {

// 2-D tiled map over a row-major [rows, cols] array of 16-bit elements with
// `row_stride_bytes` between rows.  The box is box_cols x box_rows elements;
// swizzle128 selects the 128-byte swizzle (box_cols * 2 must then be 128).
// Returns cudaErrorInvalidValue if the driver entry point is missing or the
// encoding is rejected.
cudaError_t make_tmap_2d_16bit(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                               uint64_t row_stride_bytes, uint32_t box_cols, uint32_t box_rows,
                               bool swizzle128, bool bf16);

// 3-D tiled map over a [d2, d1, d0] array of 16-bit elements (d0 innermost,
// contiguous), strides in bytes for dims 1 and 2; box b0 x b1 x b2.
cudaError_t make_tmap_3d_16bit(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1,
                               uint64_t d2, uint64_t stride1_bytes, uint64_t stride2_bytes,
                               uint32_t b0, uint32_t b1, uint32_t b2, bool swizzle128);

}  // namespace skv

#ifdef __CUDACC__
namespace skv {
// Tiled 2-D TMA load of one box at element coordinates (x, y) into shared
// memory, completion counted in bytes on `bar`.  x * 2 bytes must be a
// multiple of 16.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;"
        :: "r"(static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
           "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y),
           "r"(static_cast<uint32_t>(__cvta_generic_to_shared(bar))), "l"(policy)
        : "memory");
}
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int x, int y, int z,
                                            uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];"
        :: "r"(static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
           "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z),
           "r"(static_cast<uint32_t>(__cvta_generic_to_shared(bar)))
        : "memory");
}
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
}  // namespace skv
#endif
