// api.cu -- the extern "C" entry points of libskv (declared in include/skv.h):
// argument checks on the host, then kernel launches on the caller's stream.
// Nothing here allocates memory; nothing here prints or aborts.
//
// Pages: [F2] "F2 讲解：merge_state，以 2 为底的 LSE 合并",
// [L3] "L3 讲解：split-KV decode 与 LSE 合并".
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>
#include <vector>

#include "common.cuh"
#include "kernels.h"
#include "split_range.h"

namespace skv {

__device__ unsigned long long g_skv_error_word = 0ull;

namespace {
constexpr int kMaxDevices = 64;
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;


// Share of the SMs the prefix pass is sized for (its CTAs hold a whole SM
// each); the suffix pass fills the rest of the GPU meanwhile.  Both passes
// are bound by how fast each SM takes in K/V (the prefix pass's tensor
// loads accept about 2 KB per 100 cycles), so the share balances their
// ends.  Measured on B=64 requests sharing 8192 tokens with suffixes of
// 1..2048 (median of 40): with 16 splits for every suffix, 1/5 (24 prefix
// CTAs) 62.5 us, 1/4 (32) 66.6 us, 1/3 (48) 66.6 us, 1/7 (16) 80.9 us;
// with per-sequence split counts (a faster suffix pass, which slows the
// prefix pass more beside it), 1/5 68.6-70.7 us, 1/4 60.4-62.5 us, 1/3
// 64.5 us.
constexpr int kPrefixSmNum = 1, kPrefixSmDen = 5;
constexpr int kPrefixSmDenVarlen = 4;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }
bool valid_dtype(skv_dtype t) { return t == SKV_F32 || t == SKV_F16 || t == SKV_BF16; }

skv_status from_cuda(cudaError_t e) { return e == cudaSuccess ? SKV_OK : SKV_ERR_CUDA; }

// Row length checks shared by the merges: D elements of `dt` must be whole
// 16-byte chunks and at most 32 of them (one chunk per lane of a warp).
skv_status check_merge_D(int64_t D, skv_dtype dt) {
    if (!valid_dtype(dt) || D < 1) return SKV_ERR_INVALID_ARG;
    const int64_t bytes = D * (int64_t)dtype_size(dt);
    if (bytes % 16 != 0) return SKV_ERR_INVALID_ARG;
    if (bytes > 512) return SKV_ERR_UNSUPPORTED;
    return SKV_OK;
}
}  // namespace

skv_status current_device(const DeviceInfo** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SKV_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_dev_mu);
    DeviceInfo& d = g_dev[dev];
    if (d.device != dev) {
        int sms = 0, smem = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return SKV_ERR_CUDA;
        if (cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
            return SKV_ERR_CUDA;
        void* word = nullptr;
        if (cudaGetSymbolAddress(&word, g_skv_error_word) != cudaSuccess) return SKV_ERR_CUDA;
        d.sm_count = sms;
        d.max_smem_optin = (size_t)smem;
        d.err = static_cast<unsigned long long*>(word);
        d.device = dev;
    }
    *out = &d;
    return SKV_OK;
}

}  // namespace skv

using namespace skv;

extern "C" {

const char* skv_status_string(skv_status status) {
    switch (status) {
        case SKV_OK: return "SKV_OK";
        case SKV_ERR_INVALID_ARG: return "SKV_ERR_INVALID_ARG";
        case SKV_ERR_UNSUPPORTED: return "SKV_ERR_UNSUPPORTED";
        case SKV_ERR_CUDA: return "SKV_ERR_CUDA";
        case SKV_ERR_TIMEOUT: return "SKV_ERR_TIMEOUT";
    }
    return "SKV_UNKNOWN_STATUS";
}

int32_t skv_abi_version(void) { return 2; }

skv_status skv_merge_state(const void* v_a, const float* s_a, const void* v_b, const float* s_b,
                           void* v_out, float* s_out, int64_t S, int64_t H, int64_t D,
                           skv_dtype dtype, skv_stream_t stream) {
    if (S < 0 || H < 0) return SKV_ERR_INVALID_ARG;
    skv_status st = check_merge_D(D, dtype);
    if (st != SKV_OK) return st;
    if (S * H == 0) return SKV_OK;
    if (!v_a || !s_a || !v_b || !s_b || !v_out || !s_out) return SKV_ERR_INVALID_ARG;
    if (!aligned16(v_a) || !aligned16(v_b) || !aligned16(v_out)) return SKV_ERR_INVALID_ARG;
    if (!aligned4(s_a) || !aligned4(s_b) || !aligned4(s_out)) return SKV_ERR_INVALID_ARG;
    const DeviceInfo* dev = nullptr;
    if ((st = current_device(&dev)) != SKV_OK) return st;
    return from_cuda(launch_merge_state(v_a, s_a, v_b, s_b, v_out, s_out, S * H, D, dtype,
                                        false, *dev, reinterpret_cast<cudaStream_t>(stream)));
}

skv_status skv_merge_state_in_place(void* v, float* s, const void* v_other, const float* s_other,
                                    int64_t S, int64_t H, int64_t D, skv_dtype dtype,
                                    skv_stream_t stream) {
    if (S < 0 || H < 0) return SKV_ERR_INVALID_ARG;
    skv_status st = check_merge_D(D, dtype);
    if (st != SKV_OK) return st;
    if (S * H == 0) return SKV_OK;
    if (!v || !s || !v_other || !s_other) return SKV_ERR_INVALID_ARG;
    if (!aligned16(v) || !aligned16(v_other) || !aligned4(s) || !aligned4(s_other))
        return SKV_ERR_INVALID_ARG;
    const DeviceInfo* dev = nullptr;
    if ((st = current_device(&dev)) != SKV_OK) return st;
    return from_cuda(launch_merge_state(v, s, v_other, s_other, v, s, S * H, D, dtype, true,
                                        *dev, reinterpret_cast<cudaStream_t>(stream)));
}

size_t skv_merge_states_workspace_size(int64_t S, int64_t N, int64_t H, int64_t D) {
    if (S <= 0 || H <= 0 || N < 1 || D < 1) return 0;
    return merge_states_ws_upper_bound(S * H, N, D);
}

skv_status skv_merge_states(const void* v, const float* s, void* v_out, float* s_out, int64_t S,
                            int64_t N, int64_t H, int64_t D, skv_dtype dtype, void* workspace,
                            size_t workspace_bytes, skv_stream_t stream) {
    if (S < 0 || H < 0 || N < 1) return SKV_ERR_INVALID_ARG;
    skv_status st = check_merge_D(D, dtype);
    if (st != SKV_OK) return st;
    if (S * H == 0) return SKV_OK;
    if (N > (int64_t)INT32_MAX || S * H > (int64_t)INT32_MAX) return SKV_ERR_UNSUPPORTED;
    if (!v || !s || !v_out || !s_out) return SKV_ERR_INVALID_ARG;
    if (!aligned16(v) || !aligned16(v_out) || !aligned4(s) || !aligned4(s_out))
        return SKV_ERR_INVALID_ARG;
    if (workspace != nullptr && !aligned16(workspace)) return SKV_ERR_INVALID_ARG;
    const DeviceInfo* dev = nullptr;
    if ((st = current_device(&dev)) != SKV_OK) return st;
    return from_cuda(launch_merge_states(v, s, v_out, s_out, S, N, H, D, dtype, workspace,
                                         workspace_bytes, kMergeCtasPerSm, true, *dev,
                                         reinterpret_cast<cudaStream_t>(stream)));
}

skv_status skv_split_page_range(int32_t ctx, int32_t page, int32_t num_splits, int32_t split,
                                int32_t* p_start, int32_t* p_end) {
    if (!p_start || !p_end || ctx < 0 || page < 1 || num_splits < 1 || split < 0 ||
        split >= num_splits)
        return SKV_ERR_INVALID_ARG;
    int a = 0, b = 0;
    split_page_range(ctx, page, num_splits, split, &a, &b);
    *p_start = a;
    *p_end = b;
    return SKV_OK;
}

skv_status skv_splitkv_decode_plan(int32_t B, const int32_t* ctx_host, int32_t Hkv, int32_t page,
                                   int32_t sm_count, int32_t* num_splits) {
    if (B < 0 || Hkv < 1 || page < 1 || sm_count < 0 || !num_splits) return SKV_ERR_INVALID_ARG;
    if (B > 0 && !ctx_host) return SKV_ERR_INVALID_ARG;
    if (sm_count == 0) {
        const DeviceInfo* dev = nullptr;
        skv_status st = current_device(&dev);
        if (st != SKV_OK) return st;
        sm_count = dev->sm_count;
    }
    int64_t max_pages = 0;
    for (int32_t b = 0; b < B; ++b) {
        if (ctx_host[b] < 0) return SKV_ERR_INVALID_ARG;
        const int64_t np = ((int64_t)ctx_host[b] + page - 1) / page;
        if (np > max_pages) max_pages = np;
    }
    // [L3] §⑥: no split when B*Hkv programs already fill the GPU several
    // times over; otherwise the smallest of the page's swept split counts
    // (4, 16, 64) that does, then fewer while a split would hold < 8 pages.
    const int64_t programs = (int64_t)B * Hkv;
    const int64_t target = 3LL * sm_count;
    int32_t ns = 1;
    if (programs < target) {
        ns = 4;
        while (ns < 64 && programs * ns < target) ns *= 4;
        while (ns > 1 && (max_pages + ns - 1) / ns < 8) ns /= 4;
    }
    *num_splits = ns;
    return SKV_OK;
}

}  // extern "C"

namespace {

// A per-sequence split plan as the decode kernels take it: the device copy
// of skv_splitkv_plan_varlen's buffer ([num_units][2] units, then [B] split
// counts), its unit count and its longest split.
struct VarlenPlan {
    const int32_t* plan = nullptr;
    int32_t num_units = 0;
    int32_t max_split_pages = 0;
};

skv_status check_varlen(const VarlenPlan* vl, int32_t B) {
    if (vl == nullptr) return SKV_OK;
    if (!vl->plan || !aligned16(vl->plan) || vl->num_units < B || vl->num_units < 1 ||
        vl->max_split_pages < 0)
        return SKV_ERR_INVALID_ARG;
    if ((int64_t)vl->num_units > (int64_t)INT32_MAX / 256) return SKV_ERR_UNSUPPORTED;
    return SKV_OK;
}

void apply_varlen(const VarlenPlan* vl, DecodeArgs* a) {
    if (vl == nullptr) return;
    a->units = vl->plan;
    a->num_units = vl->num_units;
    a->max_split_pages = vl->max_split_pages;
}

const int32_t* varlen_counts(const VarlenPlan* vl) {
    return vl == nullptr ? nullptr : vl->plan + 2 * (size_t)vl->num_units;
}

// Split-KV decode ([L3] §①-⑤): pass 1 over every (sequence, split) of the
// uniform count num_splits or of the per-sequence plan `vl`, then (out !=
// NULL) the combine, chained by programmatic dependent launch.
skv_status decode_run(const void* q, const void* k_cache, const void* v_cache,
                      int32_t num_pool_pages, const int32_t* block_table, int32_t max_pages,
                      const int32_t* ctx, int32_t B, int32_t Hq, int32_t Hkv, int32_t D,
                      int32_t page, int32_t num_splits, const VarlenPlan* vl, float sm_scale,
                      skv_dtype dtype, float* o_part, float* lse_part, void* out,
                      float* lse_out, int32_t* ranges_dbg, skv_stream_t stream) {
    if (B < 0 || Hq < 1 || Hkv < 1 || D < 1 || page < 1 || num_splits < 1 || max_pages < 1 ||
        num_pool_pages < 1 || !valid_dtype(dtype))
        return SKV_ERR_INVALID_ARG;
    if (Hq % Hkv != 0) return SKV_ERR_INVALID_ARG;
    const int G = Hq / Hkv;
    if ((dtype != SKV_F16 && dtype != SKV_BF16) || D != 128 || page != 16 ||
        !(G == 1 || G == 2 || G == 4 || G == 8) || num_splits > 256 || B > 65535 || Hkv > 65535)
        return SKV_ERR_UNSUPPORTED;
    if ((int64_t)max_pages * page > INT32_MAX) return SKV_ERR_UNSUPPORTED;
    if (B == 0) return SKV_OK;
    if (!q || !k_cache || !v_cache || !block_table || !ctx || !o_part || !lse_part)
        return SKV_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(o_part) ||
        !aligned4(lse_part) || !aligned4(block_table) || !aligned4(ctx))
        return SKV_ERR_INVALID_ARG;
    if (out && !aligned16(out)) return SKV_ERR_INVALID_ARG;
    if (lse_out && !aligned4(lse_out)) return SKV_ERR_INVALID_ARG;
    if (lse_out && !out) return SKV_ERR_INVALID_ARG;
    if (ranges_dbg && !aligned4(ranges_dbg)) return SKV_ERR_INVALID_ARG;
    skv_status st = check_varlen(vl, B);
    if (st != SKV_OK) return st;
    if (vl && (int64_t)vl->num_units * Hkv > INT32_MAX) return SKV_ERR_UNSUPPORTED;
    const DeviceInfo* dev = nullptr;
    if ((st = current_device(&dev)) != SKV_OK) return st;
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    DecodeArgs a;
    a.q = q;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.num_pool_pages = num_pool_pages;
    a.block_table = block_table;
    a.max_pages = max_pages;
    a.ctx = ctx;
    a.B = B;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.D = D;
    a.page = page;
    a.num_splits = num_splits;
    a.sm_scale = sm_scale;
    a.o_part = o_part;
    a.lse_part = lse_part;
    a.ranges_dbg = ranges_dbg;
    a.bf16 = dtype == SKV_BF16;
    apply_varlen(vl, &a);
    cudaError_t e = launch_splitkv_decode(a, *dev, cs);
    if (e != cudaSuccess) return SKV_ERR_CUDA;
    if (out != nullptr) {
        CombineArgs c = {};
        c.o_part = o_part;
        c.lse_part = lse_part;
        c.rows = (int64_t)B * Hq;
        c.NS = num_splits;
        c.seq_splits = varlen_counts(vl);
        c.Hq = Hq;
        c.D = D;
        c.out = out;
        c.out_dt = dtype;
        c.lse_out = lse_out;
        e = launch_combine(c, true, *dev, cs);
        if (e != cudaSuccess) return SKV_ERR_CUDA;
    }
    return SKV_OK;
}

}  // namespace

extern "C" {

skv_status skv_splitkv_decode(const void* q, const void* k_cache, const void* v_cache,
                              int32_t num_pool_pages, const int32_t* block_table,
                              int32_t max_pages, const int32_t* ctx, int32_t B, int32_t Hq,
                              int32_t Hkv, int32_t D, int32_t page, int32_t num_splits,
                              float sm_scale, skv_dtype dtype, float* o_part, float* lse_part,
                              void* out, float* lse_out, int32_t* ranges_dbg,
                              skv_stream_t stream) {
    return decode_run(q, k_cache, v_cache, num_pool_pages, block_table, max_pages, ctx, B, Hq,
                      Hkv, D, page, num_splits, nullptr, sm_scale, dtype, o_part, lse_part, out,
                      lse_out, ranges_dbg, stream);
}

skv_status skv_splitkv_decode_varlen(const void* q, const void* k_cache, const void* v_cache,
                                     int32_t num_pool_pages, const int32_t* block_table,
                                     int32_t max_pages, const int32_t* ctx, int32_t B,
                                     int32_t Hq, int32_t Hkv, int32_t D, int32_t page,
                                     int32_t max_splits, const int32_t* plan,
                                     int32_t num_units, int32_t max_split_pages,
                                     float sm_scale, skv_dtype dtype, float* o_part,
                                     float* lse_part, void* out, float* lse_out,
                                     int32_t* ranges_dbg, skv_stream_t stream) {
    VarlenPlan vl;
    vl.plan = plan;
    vl.num_units = num_units;
    vl.max_split_pages = max_split_pages;
    return decode_run(q, k_cache, v_cache, num_pool_pages, block_table, max_pages, ctx, B, Hq,
                      Hkv, D, page, max_splits, &vl, sm_scale, dtype, o_part, lse_part, out,
                      lse_out, ranges_dbg, stream);
}

skv_status skv_splitkv_plan_varlen(int32_t B, const int32_t* ctx_host, int32_t page,
                                   int32_t max_splits, int32_t pages_per_split,
                                   int32_t* plan_host, int64_t plan_capacity,
                                   int32_t* num_units, int32_t* max_split_pages) {
    if (B < 0 || page < 1 || max_splits < 1 || max_splits > 256 || pages_per_split < 1 ||
        !num_units || !max_split_pages || (B > 0 && !ctx_host))
        return SKV_ERR_INVALID_ARG;
    // [L3] §⑥ (a planner may give sequences of different lengths different
    // split counts), with the page's "several pages per split": sequence b
    // gets ceil(pages_b / pages_per_split) splits, clamped to [1, max_splits].
    std::vector<int32_t> ns((size_t)B);
    int64_t units = 0;
    for (int32_t b = 0; b < B; ++b) {
        if (ctx_host[b] < 0) return SKV_ERR_INVALID_ARG;
        const int32_t np = (int32_t)(((int64_t)ctx_host[b] + page - 1) / page);
        const int32_t want = (int32_t)(((int64_t)np + pages_per_split - 1) / pages_per_split);
        ns[b] = std::min(max_splits, std::max(1, want));
        units += ns[b];
    }
    if (units > (int64_t)INT32_MAX / 256) return SKV_ERR_UNSUPPORTED;
    if (plan_host == nullptr) {  // size query: the counts only
        int32_t longest = 0;
        for (int32_t b = 0; b < B; ++b) {
            int p0 = 0, p1 = 0;
            split_page_range(ctx_host[b], page, ns[b], 0, &p0, &p1);  // split 0 is the longest
            longest = std::max(longest, p1 > p0 ? p1 - p0 : 0);
        }
        *num_units = (int32_t)units;
        *max_split_pages = longest;
        return SKV_OK;
    }
    if (plan_capacity < 2 * units + B) return SKV_ERR_INVALID_ARG;
    // Units, longest first (a unit's pages from the [L3] §② range), so that
    // the short ones fill the end of the launch; ties keep (b, split) order.
    struct Unit {
        int32_t pages, b, split;
    };
    std::vector<Unit> list;
    list.reserve((size_t)units);
    int32_t longest = 0;
    for (int32_t b = 0; b < B; ++b)
        for (int32_t sp = 0; sp < ns[b]; ++sp) {
            int p0 = 0, p1 = 0;
            split_page_range(ctx_host[b], page, ns[b], sp, &p0, &p1);
            const int32_t n = p1 > p0 ? p1 - p0 : 0;
            longest = std::max(longest, n);
            list.push_back(Unit{n, b, sp});
        }
    std::stable_sort(list.begin(), list.end(),
                     [](const Unit& x, const Unit& y) { return x.pages > y.pages; });
    for (size_t i = 0; i < list.size(); ++i) {
        plan_host[2 * i] = list[i].b;
        plan_host[2 * i + 1] = list[i].split | (ns[list[i].b] << 16);
    }
    for (int32_t b = 0; b < B; ++b) plan_host[2 * units + b] = ns[b];
    *num_units = (int32_t)units;
    *max_split_pages = longest;
    return SKV_OK;
}

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

static skv_status cascade_chunks(int32_t B, int32_t Hq, int32_t Hkv, int32_t prefix_len,
                                 int32_t sm_count, int prefix_den, int* mtiles, int* bpc,
                                 int* nchunks) {
    if (sm_count == 0) {
        const DeviceInfo* dev = nullptr;
        skv_status st = current_device(&dev);
        if (st != SKV_OK) return st;
        sm_count = dev->sm_count;
    }
    const int budget = sm_count * kPrefixSmNum / prefix_den;
    cascade_prefix_geometry(B, Hq / Hkv, Hkv, prefix_len, budget > 0 ? budget : 1, mtiles, bpc,
                            nchunks);
    return SKV_OK;
}

}  // extern "C"

namespace {

// One group of a cascade level: requests [r0, r1) share `len` tokens on the
// pool pages `pages`.
struct CascadeGroup {
    int32_t r0, r1;
    const int32_t* pages;
    int32_t len;
};
using CascadeLevels = std::vector<std::vector<CascadeGroup>>;

// Chunk-state slots per row: each level gets as many as the most chunks any
// of its groups' prefixes needs.
struct LevelPlan {
    int slots = 0, offset = 0;
    std::vector<int> mt, bpc;
};

skv_status cascade_plan(const CascadeLevels& levels, int32_t Hq, int32_t Hkv, int32_t sm_count,
                        int prefix_den, std::vector<LevelPlan>* plan, int* total_slots) {
    plan->assign(levels.size(), LevelPlan());
    if (sm_count == 0) {  // the current device's
        const DeviceInfo* dev = nullptr;
        skv_status st = current_device(&dev);
        if (st != SKV_OK) return st;
        sm_count = dev->sm_count;
    }
    int total = 0;
    for (size_t l = 0; l < levels.size(); ++l) {
        LevelPlan& lp = (*plan)[l];
        // The groups of a level run side by side: each is sized for its
        // share of the prefix pass's SMs.
        const int share = std::max(1, sm_count / std::max(1, (int)levels[l].size()));
        for (const CascadeGroup& g : levels[l]) {
            int mt = 0, bpc = 0, nc = 0;
            skv_status st =
                cascade_chunks(g.r1 - g.r0, Hq, Hkv, g.len, share, prefix_den, &mt, &bpc, &nc);
            if (st != SKV_OK) return st;
            lp.mt.push_back(mt);
            lp.bpc.push_back(bpc);
            lp.slots = std::max(lp.slots, nc);
        }
        lp.offset = total;
        total += lp.slots;
    }
    *total_slots = total;
    return SKV_OK;
}

// Workspace: chunk states [rows, slots, D] fp32, their lse [rows, slots],
// then 256 bytes holding the suffix pass's completion counter.
size_t cascade_ws_bytes(size_t rows, int slots, int32_t D) {
    return align256(rows * slots * D * 4) + align256(rows * slots * 4) + 256;
}

// Converts the public level descriptions, checking them.
skv_status read_levels(int32_t num_levels, const skv_cascade_level* levels, int32_t B,
                       CascadeLevels* out) {
    if (num_levels < 0 || (num_levels > 0 && !levels)) return SKV_ERR_INVALID_ARG;
    out->assign((size_t)num_levels, {});
    for (int32_t l = 0; l < num_levels; ++l) {
        const skv_cascade_level& lv = levels[l];
        if (lv.num_groups < 1 || !lv.group_start || !lv.group_len || !lv.group_pages)
            return SKV_ERR_INVALID_ARG;
        if (lv.group_start[0] != 0 || lv.group_start[lv.num_groups] != B) return SKV_ERR_INVALID_ARG;
        for (int32_t g = 0; g < lv.num_groups; ++g) {
            const int32_t r0 = lv.group_start[g], r1 = lv.group_start[g + 1], len = lv.group_len[g];
            const int32_t* pages = lv.group_pages[g];
            if (r1 < r0 || len < 0) return SKV_ERR_INVALID_ARG;
            if (len > 0 && (!pages || !aligned4(pages))) return SKV_ERR_INVALID_ARG;
            if (r1 > r0) (*out)[l].push_back(CascadeGroup{r0, r1, pages, len});
        }
    }
    return SKV_OK;
}

// The cascade for any number of shared levels ([F2] §⑥ and the multi-level
// wrapper it names): each group's prefix pass writes its chunk states into
// its level's slots of every row it covers (beside the suffix pass), the
// suffixes run through the split-KV decode, and one combine merges all
// slots into the prefix state and that with the suffix splits.
skv_status cascade_run(const void* q, const void* k_cache, const void* v_cache,
                       int32_t num_pool_pages, const CascadeLevels& levels,
                       const int32_t* block_table, int32_t max_pages, const int32_t* ctx,
                       int32_t B, int32_t Hq, int32_t Hkv, int32_t D, int32_t page,
                       int32_t num_splits, const VarlenPlan* vl, float sm_scale,
                       skv_dtype dtype, float* o_pre, float* s_pre, float* o_part,
                       float* lse_part, void* out, float* lse_out, void* workspace,
                       size_t workspace_bytes, skv_stream_t stream) {
    if (B < 0 || Hq < 1 || Hkv < 1 || D < 1 || page < 1 || num_splits < 1 || max_pages < 1 ||
        num_pool_pages < 1 || !valid_dtype(dtype))
        return SKV_ERR_INVALID_ARG;
    if (Hq % Hkv != 0) return SKV_ERR_INVALID_ARG;
    const int G = Hq / Hkv;
    if ((dtype != SKV_F16 && dtype != SKV_BF16) || D != 128 || page != 16 ||
        !(G == 1 || G == 2 || G == 4 || G == 8) || num_splits > 256 || B > 65535 || Hkv > 65535)
        return SKV_ERR_UNSUPPORTED;
    if ((int64_t)max_pages * page > INT32_MAX ||
        (int64_t)num_pool_pages * Hkv * page > INT32_MAX - page)
        return SKV_ERR_UNSUPPORTED;
    if (B == 0) return SKV_OK;
    if (!q || !k_cache || !v_cache || !block_table || !ctx || !o_part || !lse_part || !out ||
        !workspace)
        return SKV_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(o_part) ||
        !aligned16(out) || !aligned16(workspace) || !aligned4(lse_part) || !aligned4(block_table) ||
        !aligned4(ctx))
        return SKV_ERR_INVALID_ARG;
    if ((o_pre && !aligned16(o_pre)) || (s_pre && !aligned4(s_pre)) ||
        (lse_out && !aligned4(lse_out)))
        return SKV_ERR_INVALID_ARG;
    skv_status st = check_varlen(vl, B);
    if (st != SKV_OK) return st;
    if (vl && (int64_t)vl->num_units * Hkv > INT32_MAX) return SKV_ERR_UNSUPPORTED;
    const DeviceInfo* dev = nullptr;
    if ((st = current_device(&dev)) != SKV_OK) return st;
    std::vector<LevelPlan> plan;
    int slots = 0;
    const int den = vl != nullptr ? kPrefixSmDenVarlen : kPrefixSmDen;
    if ((st = cascade_plan(levels, Hq, Hkv, dev->sm_count, den, &plan, &slots)) != SKV_OK) return st;
    const size_t rows = (size_t)B * Hq;
    if (workspace_bytes < cascade_ws_bytes(rows, slots, D)) return SKV_ERR_INVALID_ARG;
    float* pre_part = static_cast<float*>(workspace);
    float* pre_lse =
        reinterpret_cast<float*>(static_cast<char*>(workspace) + align256(rows * slots * D * 4));
    // Completion counter of the suffix pass (the workspace's last 256 bytes).
    unsigned int* done_ctr = reinterpret_cast<unsigned int*>(
        static_cast<char*>(workspace) + align256(rows * slots * D * 4) + align256(rows * slots * 4));
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    // 1. Shared prefixes on the tensor cores, one state per prefix chunk.
    // Every kernel of the cascade goes into the caller's stream, chained by
    // programmatic dependent launch: each prefix pass lets the next kernel
    // start at once, so the prefix passes and the suffix pass run side by
    // side (a prefix pass takes about a fifth of the SMs), and each
    // completes only after the kernel before it, so that the combine, which
    // waits for the suffix pass, sees every prefix state.  The first prefix
    // pass zeroes the suffix pass's completion counter.
    // A chained pass that ends before the pass launched ahead of it holds
    // its SMs until that one completes, so the passes go in order of their
    // work per CTA (prefix blocks per chunk), shortest first.
    int launched = 0;
    if (slots > 0) {
        const size_t elt = 2;  // fp16 / bf16
        std::vector<std::pair<int, std::pair<size_t, size_t>>> order;  // (bpc, (level, group))
        for (size_t l = 0; l < levels.size(); ++l)
            if (plan[l].slots > 0)
                for (size_t gi = 0; gi < levels[l].size(); ++gi)
                    order.push_back({plan[l].bpc[gi], {l, gi}});
        std::stable_sort(order.begin(), order.end(),
                         [](const auto& x, const auto& y) { return x.first < y.first; });
        for (const auto& o : order) {
            const size_t l = o.second.first, gi = o.second.second;
            const LevelPlan& lp = plan[l];
            {
                const CascadeGroup& g = levels[l][gi];
                CascadeArgs ca;
                ca.q = static_cast<const char*>(q) + (size_t)g.r0 * Hq * D * elt;
                ca.k_cache = k_cache;
                ca.v_cache = v_cache;
                ca.num_pool_pages = num_pool_pages;
                ca.prefix_pages = g.pages;
                ca.prefix_len = g.len;
                ca.B = g.r1 - g.r0;
                ca.Hq = Hq;
                ca.Hkv = Hkv;
                ca.bf16 = dtype == SKV_BF16;
                ca.sm_scale = sm_scale;
                ca.zero_ctr = launched == 0 ? done_ctr : nullptr;
                ca.chained = launched > 0;
                const size_t row0 = (size_t)g.r0 * Hq;
                if (launch_cascade_prefix(ca, *dev, pre_part + row0 * slots * D, pre_lse + row0 * slots,
                                          lp.slots, lp.bpc[gi], lp.mt[gi], slots, lp.offset,
                                          cs) != cudaSuccess)
                    return SKV_ERR_CUDA;
                ++launched;
            }
        }
    }
    // 2. Each request's own suffix through the split-KV decode.
    DecodeArgs a;
    a.q = q;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.num_pool_pages = num_pool_pages;
    a.block_table = block_table;
    a.max_pages = max_pages;
    a.ctx = ctx;
    a.B = B;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.D = D;
    a.page = page;
    a.num_splits = num_splits;
    a.sm_scale = sm_scale;
    a.o_part = o_part;
    a.lse_part = lse_part;
    a.ranges_dbg = nullptr;
    a.bf16 = dtype == SKV_BF16;
    a.done_ctr = launched > 0 ? done_ctr : nullptr;  // chained after the prefix passes
    apply_varlen(vl, &a);
    if (launch_splitkv_decode(a, *dev, cs) != cudaSuccess) return SKV_ERR_CUDA;
    // 3. Prefix chunks of every level -> prefix state; merge_state(prefix,
    // suffix) -> out.
    CombineArgs c = {};
    c.o_part = o_part;
    c.lse_part = lse_part;
    c.rows = (int64_t)rows;
    c.NS = num_splits;
    c.seq_splits = varlen_counts(vl);
    c.Hq = Hq;
    c.D = D;
    c.out = out;
    c.out_dt = dtype;
    c.lse_out = lse_out;
    c.pre_part = pre_part;
    c.pre_lse = pre_lse;
    c.C = slots;
    c.o_pre = o_pre;
    c.s_pre = s_pre;
    // The combine follows pass 1 directly (programmatic dependent launch) and
    // waits for it to complete (hence for the prefix passes too).
    if (launch_combine(c, true, *dev, cs) != cudaSuccess) return SKV_ERR_CUDA;
    return SKV_OK;
}

CascadeLevels two_level(int32_t B, const int32_t* prefix_pages, int32_t prefix_len) {
    CascadeLevels lv(1);
    if (B > 0) lv[0].push_back(CascadeGroup{0, B, prefix_pages, prefix_len});
    return lv;
}

}  // namespace

extern "C" {

size_t skv_cascade_workspace_size(int32_t B, int32_t Hq, int32_t Hkv, int32_t D,
                                  int32_t prefix_len, int32_t sm_count) {
    if (B < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || D < 1 || prefix_len < 0 || sm_count < 0)
        return 0;
    // Enough for the uniform and the per-sequence suffix plans (whose
    // prefix passes are sized for different shares of the SMs).
    size_t most = 0;
    for (int den : {kPrefixSmDen, kPrefixSmDenVarlen}) {
        std::vector<LevelPlan> plan;
        int slots = 0;
        if (cascade_plan(two_level(B, nullptr, prefix_len), Hq, Hkv, sm_count, den, &plan,
                         &slots) != SKV_OK)
            return 0;
        most = std::max(most, cascade_ws_bytes((size_t)B * Hq, slots, D));
    }
    return most;
}

skv_status skv_cascade_decode(const void* q, const void* k_cache, const void* v_cache,
                              int32_t num_pool_pages, const int32_t* prefix_pages,
                              int32_t prefix_len, const int32_t* block_table, int32_t max_pages,
                              const int32_t* ctx, int32_t B, int32_t Hq, int32_t Hkv, int32_t D,
                              int32_t page, int32_t num_splits, float sm_scale, skv_dtype dtype,
                              float* o_pre, float* s_pre, float* o_part, float* lse_part,
                              void* out, float* lse_out, void* workspace, size_t workspace_bytes,
                              skv_stream_t stream) {
    if (prefix_len < 0) return SKV_ERR_INVALID_ARG;
    if (prefix_len > 0 && (!prefix_pages || !aligned4(prefix_pages))) return SKV_ERR_INVALID_ARG;
    return cascade_run(q, k_cache, v_cache, num_pool_pages, two_level(B, prefix_pages, prefix_len),
                       block_table, max_pages, ctx, B, Hq, Hkv, D, page, num_splits, nullptr,
                       sm_scale, dtype, o_pre, s_pre, o_part, lse_part, out, lse_out, workspace,
                       workspace_bytes, stream);
}

skv_status skv_cascade_decode_varlen(const void* q, const void* k_cache, const void* v_cache,
                                     int32_t num_pool_pages, const int32_t* prefix_pages,
                                     int32_t prefix_len, const int32_t* block_table,
                                     int32_t max_pages, const int32_t* ctx, int32_t B,
                                     int32_t Hq, int32_t Hkv, int32_t D, int32_t page,
                                     int32_t max_splits, const int32_t* plan,
                                     int32_t num_units, int32_t max_split_pages,
                                     float sm_scale, skv_dtype dtype, float* o_pre,
                                     float* s_pre, float* o_part, float* lse_part, void* out,
                                     float* lse_out, void* workspace, size_t workspace_bytes,
                                     skv_stream_t stream) {
    if (prefix_len < 0) return SKV_ERR_INVALID_ARG;
    if (prefix_len > 0 && (!prefix_pages || !aligned4(prefix_pages))) return SKV_ERR_INVALID_ARG;
    VarlenPlan vl;
    vl.plan = plan;
    vl.num_units = num_units;
    vl.max_split_pages = max_split_pages;
    return cascade_run(q, k_cache, v_cache, num_pool_pages, two_level(B, prefix_pages, prefix_len),
                       block_table, max_pages, ctx, B, Hq, Hkv, D, page, max_splits, &vl,
                       sm_scale, dtype, o_pre, s_pre, o_part, lse_part, out, lse_out, workspace,
                       workspace_bytes, stream);
}

size_t skv_cascade_multilevel_workspace_size(int32_t num_levels, const skv_cascade_level* levels,
                                             int32_t B, int32_t Hq, int32_t Hkv, int32_t D,
                                             int32_t sm_count) {
    if (B < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || D < 1 || sm_count < 0) return 0;
    CascadeLevels lv;
    if (read_levels(num_levels, levels, B, &lv) != SKV_OK) return 0;
    std::vector<LevelPlan> plan;
    int slots = 0;
    if (cascade_plan(lv, Hq, Hkv, sm_count, kPrefixSmDen, &plan, &slots) != SKV_OK) return 0;
    return cascade_ws_bytes((size_t)B * Hq, slots, D);
}

skv_status skv_cascade_decode_multilevel(const void* q, const void* k_cache, const void* v_cache,
                                         int32_t num_pool_pages, int32_t num_levels,
                                         const skv_cascade_level* levels,
                                         const int32_t* block_table, int32_t max_pages,
                                         const int32_t* ctx, int32_t B, int32_t Hq, int32_t Hkv,
                                         int32_t D, int32_t page, int32_t num_splits,
                                         float sm_scale, skv_dtype dtype, float* o_pre,
                                         float* s_pre, float* o_part, float* lse_part, void* out,
                                         float* lse_out, void* workspace, size_t workspace_bytes,
                                         skv_stream_t stream) {
    CascadeLevels lv;
    skv_status st = read_levels(num_levels, levels, B, &lv);
    if (st != SKV_OK) return st;
    return cascade_run(q, k_cache, v_cache, num_pool_pages, lv, block_table, max_pages, ctx, B, Hq,
                       Hkv, D, page, num_splits, nullptr, sm_scale, dtype, o_pre, s_pre, o_part,
                       lse_part, out, lse_out, workspace, workspace_bytes, stream);
}

skv_status skv_get_device_error(int32_t* code, int32_t* detail) {
    if (!code || !detail) return SKV_ERR_INVALID_ARG;
    const DeviceInfo* dev = nullptr;
    skv_status st = current_device(&dev);
    if (st != SKV_OK) return st;
    if (cudaDeviceSynchronize() != cudaSuccess) return SKV_ERR_CUDA;
    unsigned long long w = 0, zero = 0;
    if (cudaMemcpy(&w, dev->err, sizeof(w), cudaMemcpyDeviceToHost) != cudaSuccess)
        return SKV_ERR_CUDA;
    if (cudaMemcpy(dev->err, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
        return SKV_ERR_CUDA;
    *code = (int32_t)(w & 0xffu);
    *detail = (int32_t)(w >> 8);
    return SKV_OK;
}

skv_status skv_poll_device_error(int32_t* code, int32_t* detail, skv_stream_t stream) {
    if (!code || !detail) return SKV_ERR_INVALID_ARG;
    const DeviceInfo* dev = nullptr;
    skv_status st = current_device(&dev);
    if (st != SKV_OK) return st;
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    // The copy to pageable host memory returns once it has run, i.e. after
    // the work queued on `stream` before it.  A non-zero word is never
    // overwritten (the first error wins), so clearing it after reading it
    // loses nothing.
    unsigned long long w = 0;
    if (cudaMemcpyAsync(&w, dev->err, sizeof(w), cudaMemcpyDeviceToHost, cs) != cudaSuccess)
        return SKV_ERR_CUDA;
    if (cudaStreamSynchronize(cs) != cudaSuccess) return SKV_ERR_CUDA;
    if (w != 0) {
        if (cudaMemsetAsync(dev->err, 0, sizeof(w), cs) != cudaSuccess) return SKV_ERR_CUDA;
        if (cudaStreamSynchronize(cs) != cudaSuccess) return SKV_ERR_CUDA;
    }
    *code = (int32_t)(w & 0xffu);
    *detail = (int32_t)(w >> 8);
    return SKV_OK;
}

}  // extern "C"
