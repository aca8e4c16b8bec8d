// split_range.h -- page range of one split, shared by the decode kernel and
// the host query skv_split_page_range so the two can never disagree.
//
// Page: "L3 讲解：split-KV decode 与 LSE 合并", §②: each split owns the
// contiguous pages [p_start, p_end) with
//   num_pages = ceil(ctx / page), pages_per_split = ceil(num_pages / NS),
//   p_start = split * pages_per_split, p_end = min(p_start + pps, num_pages);
// p_end <= p_start is an empty split.  Computed per sequence from its own ctx.
#pragma once

#ifdef __CUDACC__
#define SKV_HD __host__ __device__ __forceinline__
#else
#define SKV_HD inline
#endif

namespace skv {

SKV_HD void split_page_range(int ctx, int page, int num_splits, int split, int* p_start,
                             int* p_end) {
    const int num_pages = (ctx + page - 1) / page;
    const int pps = (num_pages + num_splits - 1) / num_splits;
    const int start = split * pps;
    const int end = start + pps < num_pages ? start + pps : num_pages;
    *p_start = start;
    *p_end = end;
}

}  // namespace skv
