/*
 * skv.h -- C ABI of the GB300 (sm_103a) split-KV decode and attention-state
 * merge library (libskv.so).
 *
 * Pages the operations follow, cited by title and section:
 *   [F2] "F2 讲解：merge_state，以 2 为底的 LSE 合并"
 *   [L3] "L3 讲解：split-KV decode 与 LSE 合并"
 *   [FA] "FlashAttention 的空行 LSE:FA-2 的 +inf 约定与后来的变化"
 *
 * Conventions shared by every entry point
 *   - An attention state is (v, s).  v is the softmax-normalised output over a
 *     subset of keys; s = log2( sum_j exp(score_j) ) is the BASE-2 log-sum-exp
 *     of those keys' scores ([F2] §②).  The natural-log form is s * ln 2.
 *     s is always fp32.  v is fp32, fp16 or bf16 (skv_dtype).
 *   - An empty state is s = -inf, v = 0 ([F2] §⑤).  Merging two empty states
 *     gives s = -inf, v = 0, never NaN.  An incoming s that is NaN or +inf is
 *     read as -inf, i.e. "no weight" ([FA] §2.2).
 *   - Pointers named v, s, q, *_cache, *_table, ctx, o_*, lse_*, out, workspace
 *     are DEVICE pointers; `*_host` pointers are host pointers.  The caller
 *     owns every buffer.  No entry point allocates device or host memory.
 *   - Every device entry point is asynchronous on `stream` (NULL = the legacy
 *     default stream) and returns as soon as its kernels are enqueued.
 *   - Arguments are checked on the host before anything is launched; a failed
 *     check returns SKV_ERR_INVALID_ARG (bad pointer, size, alignment) or
 *     SKV_ERR_UNSUPPORTED (a valid shape this library has no kernel for) and
 *     enqueues nothing.  A launch failure returns SKV_ERR_CUDA.  Errors that
 *     only the device can see (a page id outside the pool, a ctx larger than
 *     the page table, a bounded wait that gave up) are recorded in a per-device
 *     error word read by skv_get_device_error(); the kernel then clamps the
 *     offending index into range or skips the rest of its work, so it neither
 *     faults nor hangs, and its outputs are unspecified.
 *   - The library never aborts, never prints and keeps no state other than the
 *     per-device error word and cached device attributes.
 *   - 16-byte alignment is required for every v/q/cache/output pointer and for
 *     o_part; D * sizeof(element) must be a multiple of 16 bytes.
 */
#ifndef SKV_H_
#define SKV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream (cudaStream_t / CUstream); NULL is the legacy default stream. */
typedef struct CUstream_st* skv_stream_t;

typedef enum {
    SKV_OK = 0,
    SKV_ERR_INVALID_ARG = 1, /* a pointer, size or alignment check failed         */
    SKV_ERR_UNSUPPORTED = 2, /* a valid shape or dtype this library has no kernel for */
    SKV_ERR_CUDA = 3,        /* a CUDA runtime call or kernel launch failed         */
    SKV_ERR_TIMEOUT = 4      /* a bounded device wait gave up (device error word)   */
} skv_status;

typedef enum { SKV_F32 = 0, SKV_F16 = 1, SKV_BF16 = 2 } skv_dtype;

/* Human-readable name of a status code (static string, never NULL). */
const char* skv_status_string(skv_status status);

/* ABI version of this header (2); bumped on any signature change. */
int32_t skv_abi_version(void);

/*
 * Two-state merge ([F2] §③; guards of [F2] §⑤ and [FA] §2.2).
 * For every row r of R = S*H rows (row r = pos*H + h):
 *   a = sanitize(s_a[r]), b = sanitize(s_b[r]), m = max(a, b),
 *   w_x = 2^(x - m) (0 for an empty state), W = w_a + w_b,
 *   v_out[r, :] = (w_a v_a[r, :] + w_b v_b[r, :]) / W   (0 if W == 0),
 *   s_out[r]    = m + log2(W)                            (-inf if W == 0).
 * Layout: v_a, v_b, v_out are [S, H, D] contiguous in `dtype`; s_a, s_b, s_out
 * are [S, H] contiguous fp32.  Accumulation is fp32; v_out is rounded to
 * `dtype` (round to nearest even).  The formula is symmetric, so swapping the
 * two inputs gives bit-identical outputs.  Outputs must not overlap inputs
 * (use skv_merge_state_in_place for in-place merging).
 * Limits: S, H >= 0 (S*H == 0 is a no-op), 1 <= D, D*sizeof(dtype) % 16 == 0
 * (else SKV_ERR_INVALID_ARG), and a row of at most 512 bytes, D*sizeof(dtype)
 * <= 512 (D <= 128 in fp32, D <= 256 in fp16/bf16; a longer row returns
 * SKV_ERR_UNSUPPORTED).
 */
skv_status skv_merge_state(const void* v_a, const float* s_a,
                           const void* v_b, const float* s_b,
                           void* v_out, float* s_out,
                           int64_t S, int64_t H, int64_t D,
                           skv_dtype dtype, skv_stream_t stream);

/*
 * In-place two-state merge ([F2] §⑦ names merge_state_in_place; the page
 * gives no body, the reading taken is the unmasked update
 *   (v, s) <- merge_state((v, s), (v_other, s_other))
 * with exactly the arithmetic of skv_merge_state, a in the first operand.)
 * v is [S, H, D] in `dtype` and s is [S, H] fp32, both overwritten; v_other,
 * s_other are read only and must not overlap v, s.
 */
skv_status skv_merge_state_in_place(void* v, float* s,
                                    const void* v_other, const float* s_other,
                                    int64_t S, int64_t H, int64_t D,
                                    skv_dtype dtype, skv_stream_t stream);

/*
 * Device workspace, in bytes, that skv_merge_states may use for these sizes
 * (0 when it never needs any).  Few rows with many states are merged in two
 * levels: several CTAs per row each merge a chunk of the N states into a
 * partial state kept in the workspace, and the last CTA of the row merges the
 * partials (exact because merging is associative, [F2] §①).
 */
size_t skv_merge_states_workspace_size(int64_t S, int64_t N, int64_t H, int64_t D);

/*
 * N-state merge in the [S, N, H, D] / [S, N, H] layout ([F2] §④): element
 * s[pos, n, h] is at offset (pos*N + n)*H + h and v[pos, n, h, :] at that
 * offset times D.  For every (pos, h):
 *   m = max_n sanitize(s_n), w_n = 2^(s_n - m) (0 if empty), W = sum_n w_n,
 *   v_out[pos, h, :] = sum_n w_n v_n / W   (0 if W == 0),
 *   s_out[pos, h]    = m + log2(W)         (-inf if W == 0).
 * v_out is [S, H, D] in `dtype`, s_out [S, H] fp32; fp32 accumulation.
 * Zero-weight states are not read.
 * workspace: NULL, or a device buffer of workspace_bytes bytes.  If it is at
 *   least skv_merge_states_workspace_size(S, N, H, D) bytes the two-level
 *   path may be used; otherwise every row is merged by one CTA (same result
 *   up to fp32 rounding order).  The workspace MUST be zero-filled before its
 *   first use.  It holds per-row arrival counters that every completed call
 *   returns to zero, so one buffer serves consecutive calls on one stream
 *   without re-zeroing (zero it again after a call that did not complete).
 *   Calls that share a workspace must not overlap on the GPU.
 * Limits: S, H >= 0, N >= 1, D as for skv_merge_state (rows of at most 512
 * bytes).
 */
skv_status skv_merge_states(const void* v, const float* s,
                            void* v_out, float* s_out,
                            int64_t S, int64_t N, int64_t H, int64_t D,
                            skv_dtype dtype, void* workspace, size_t workspace_bytes,
                            skv_stream_t stream);

/*
 * Size of the fixed device scratch array used by skv_merge_states_noalloc
 * (one array per GPU that loads the library, held until the process exits).
 */
#define SKV_MERGE_STATES_NOALLOC_SCRATCH_BYTES (1u << 20)

/*
 * skv_merge_states without a workspace argument, for callers that cannot
 * allocate device memory.  (The pages have no counterpart: this is a
 * convenience of this library.)  Some callers have no way to call cudaMalloc:
 * a plugin inside another runtime that owns every allocation and only hands
 * over its inputs and outputs, or a latency-critical decode loop that must not
 * risk the device synchronisation an allocation can cause.  This entry point
 * computes exactly what skv_merge_states computes, with the same arguments
 * minus the workspace, and allocates nothing (no cudaMalloc, cudaFree or
 * allocating library call): when the merge runs in two levels its partial
 * states live in a file-scope device array of
 * SKV_MERGE_STATES_NOALLOC_SCRATCH_BYTES bytes inside the library.
 *   - Sizes whose two-level merge would need more scratch than that are
 *     rejected with SKV_ERR_UNSUPPORTED (nothing is enqueued);
 *     skv_merge_states_noalloc_scratch_size gives the need in advance.  The
 *     two-level path is only taken for fewer than 2 * SM-count rows (S*H),
 *     which it gives about 2 * SM-count CTAs, so at most about 4 * SM-count
 *     partial rows of D fp32 values (1 KB each at D = 256) plus 12 bytes per
 *     row.  On a GPU with up to about 250 SMs (a GB300 has 152) every
 *     supported shape fits; on larger GPUs the few-row, many-state shapes
 *     with D = 256 can be rejected.
 *   - The first call on a device looks up the array's device address with
 *     cudaGetSymbolAddress (with that device current) and caches it; make that
 *     first call before any stream capture on the device.
 *   - Every call shares the one array, which keeps the last call's contents;
 *     each call clears the part it needs (cudaMemsetAsync on `stream`) before
 *     using it.  Calls that overlap on the GPU (on different streams, or
 *     concurrently from several host threads) race on the array and must be
 *     serialised by the caller.
 */
skv_status skv_merge_states_noalloc(const void* v, const float* s,
                                    void* v_out, float* s_out,
                                    int64_t S, int64_t N, int64_t H, int64_t D,
                                    skv_dtype dtype, skv_stream_t stream);

/*
 * Bytes of the fixed scratch array that skv_merge_states_noalloc would use
 * for these sizes on a GPU with sm_count SMs (0 = the current device's);
 * 0 when the call needs none, or for invalid sizes.  A call whose need
 * exceeds SKV_MERGE_STATES_NOALLOC_SCRATCH_BYTES returns SKV_ERR_UNSUPPORTED.
 * Host only when sm_count > 0.
 */
size_t skv_merge_states_noalloc_scratch_size(int64_t S, int64_t N, int64_t H, int64_t D,
                                             skv_dtype dtype, int32_t sm_count);

/*
 * Page range of one split ([L3] §②), computed on the host with exactly the
 * integer arithmetic the decode kernel uses:
 *   num_pages = ceil(ctx / page), pps = ceil(num_pages / num_splits),
 *   p_start = split * pps, p_end = min(p_start + pps, num_pages).
 * The raw values are returned (p_end may be <= p_start: the split is empty).
 * Host only; needs no GPU.  Limits: ctx >= 0, page >= 1, num_splits >= 1,
 * 0 <= split < num_splits.
 */
skv_status skv_split_page_range(int32_t ctx, int32_t page, int32_t num_splits, int32_t split,
                                int32_t* p_start, int32_t* p_end);

/*
 * Split count for one decode step ([L3] §⑥): B*Hkv*NS several times the SM
 * count while every split keeps several pages; no split when B*Hkv already
 * fills the GPU.  Constants (the page prints none): candidates 1, 4, 16, 64
 * (the counts the page's sweep measures); NS = 1 if B*Hkv >= 3*sm_count, else
 * the smallest of 4, 16, 64 reaching 3*sm_count (64 if none does), then
 * stepped down while ceil(max_pages / NS) < 8.  This reproduces the page's
 * table exactly (170 SMs: B=1 ctx 32768 -> 64, B=8 ctx 4096 -> 16,
 * B=64 ctx 1024 -> 1).
 * ctx_host: host array of B context lengths.  sm_count > 0 is used as given;
 * sm_count == 0 means the current CUDA device's SM count (needs a GPU).
 * Result in *num_splits.
 */
skv_status skv_splitkv_decode_plan(int32_t B, const int32_t* ctx_host, int32_t Hkv,
                                   int32_t page, int32_t sm_count, int32_t* num_splits);

/*
 * Split-KV paged decode attention, Flash-Decoding style ([L3] §① two kernels,
 * §② ranges, §③ per-split state, §④ empty splits, §⑤ fp32 partials).
 * Pass 1, one CTA per (b, hkv, split): query heads hq = hkv*G .. hkv*G+G-1
 * (G = Hq/Hkv, grouped heads are contiguous) attend to the tokens
 * [p_start*page, min(p_end*page, ctx[b])) of sequence b, with
 * score = sm_scale * q . k, and write the split-normalised state
 *   o_part[b, hq, split, :] (fp32) and lse_part[b, hq, split] (fp32, base 2);
 * an empty split writes o = 0 and lse = -inf.
 * Pass 2 (only when out != NULL): merges the num_splits states of each
 * (b, hq) like skv_merge_states and writes out[b, hq, :] in `dtype` and, if
 * lse_out != NULL, lse_out[b, hq] (fp32, base 2).
 * Layouts: q [B, Hq, D]; k_cache, v_cache [num_pool_pages, Hkv, page, D]
 *   (`dtype`); block_table [B, max_pages] int32 pool-page ids, row-major;
 *   ctx [B] int32 context lengths (device); o_part [B, Hq, num_splits, D];
 *   lse_part [B, Hq, num_splits]; out [B, Hq, D]; lse_out [B, Hq].
 * ranges_dbg: NULL, or a device int32 [B, num_splits, 2] receiving the
 *   (p_start, p_end) each CTA computed.
 * Supported: dtype SKV_F16 or SKV_BF16 (q, K, V and out; the products are
 *   exact in fp32, p enters P.V rounded to the dtype), D = 128, page = 16,
 *   G in {1, 2, 4, 8}, 1 <= num_splits <= 256.  B = 0 is a no-op.
 * Device-side checks: a ctx outside [0, max_pages*page] or a page id outside
 *   [0, num_pool_pages) is clamped into range and flagged in the error word.
 * Rounding: when the longest split has 9..64 pages (max_pages / num_splits
 *   rounded up), the warps of a split's CTA take its pages in the order
 *   their copies land, so o_part and lse_part may differ between runs in
 *   the last bits (fp32 sums grouped differently); otherwise results are
 *   the same from run to run.
 */
skv_status skv_splitkv_decode(const void* q, const void* k_cache, const void* v_cache,
                              int32_t num_pool_pages,
                              const int32_t* block_table, int32_t max_pages,
                              const int32_t* ctx,
                              int32_t B, int32_t Hq, int32_t Hkv, int32_t D, int32_t page,
                              int32_t num_splits, float sm_scale, skv_dtype dtype,
                              float* o_part, float* lse_part,
                              void* out, float* lse_out,
                              int32_t* ranges_dbg, skv_stream_t stream);

/*
 * Per-sequence split counts ([L3] §⑥: a planner decides the splits before
 * each decode step from B, every sequence's ctx and the GPU, and may give
 * sequences of different lengths different split counts).  The page fixes
 * no rule for the per-sequence count; the rule taken keeps its "several
 * pages per split": sequence b, of n_b = ceil(ctx_host[b] / page) pages,
 * gets ns_b = ceil(n_b / pages_per_split) splits, clamped to
 * [1, max_splits], cut by the [L3] §② ranges with NUM_SPLITS = ns_b.
 * Host only; needs no GPU.
 * plan_host: NULL to query only *num_units and *max_split_pages (so that the
 *   buffer can be sized exactly), or a host int32 buffer of plan_capacity >=
 *   2 * sum_b ns_b + B elements (2 * B * max_splits + B always suffices).  It
 *   receives
 *   [*num_units][2] work units (b, split | ns_b << 16), one per split of
 *   every sequence, the longest splits first, followed by [B] the split
 *   counts ns_b.  Copy it as is into a 16-byte aligned device buffer for
 *   skv_splitkv_decode_varlen / skv_cascade_decode_varlen.
 * *num_units receives sum_b ns_b; *max_split_pages the most pages any one
 *   split holds (it sets the decode kernel's shape).
 * Limits: B >= 0, page >= 1, 1 <= max_splits <= 256, pages_per_split >= 1,
 *   ctx_host[b] >= 0.
 */
skv_status skv_splitkv_plan_varlen(int32_t B, const int32_t* ctx_host, int32_t page,
                                   int32_t max_splits, int32_t pages_per_split,
                                   int32_t* plan_host, int64_t plan_capacity,
                                   int32_t* num_units, int32_t* max_split_pages);

/*
 * Split-KV paged decode with a split count per sequence: as
 * skv_splitkv_decode, but sequence b is cut into ns_b splits (the plan's
 * counts) and pass 1 runs one CTA per (unit, kv head) of the plan's work list
 * only.  o_part [B, Hq, max_splits, D] and lse_part [B, Hq, max_splits] keep
 * the split axis max_splits long: split sp < ns_b of sequence b is written
 * there, slots sp >= ns_b are not written.  The combine (out != NULL) merges
 * the ns_b states of each (b, hq).  ranges_dbg [B, max_splits, 2] as for
 * skv_splitkv_decode, for sp < ns_b.
 * plan: device copy of skv_splitkv_plan_varlen's buffer (16-byte aligned),
 *   num_units and max_split_pages as that call returned them; the contexts
 *   in `ctx` (device) must be those the plan was made for (a longer one can
 *   make a split longer than max_split_pages, which is flagged in the error
 *   word and cut).  A unit naming a sequence outside [0, B) or a split count
 *   outside [1, max_splits] is flagged and skipped.
 * Other arguments, layouts, support and device-side checks as for
 * skv_splitkv_decode (with max_splits <= 256 in place of num_splits).
 */
skv_status skv_splitkv_decode_varlen(const void* q, const void* k_cache, const void* v_cache,
                                     int32_t num_pool_pages, const int32_t* block_table,
                                     int32_t max_pages, const int32_t* ctx, int32_t B,
                                     int32_t Hq, int32_t Hkv, int32_t D, int32_t page,
                                     int32_t max_splits, const int32_t* plan,
                                     int32_t num_units, int32_t max_split_pages,
                                     float sm_scale, skv_dtype dtype, float* o_part,
                                     float* lse_part, void* out, float* lse_out,
                                     int32_t* ranges_dbg, skv_stream_t stream);

/*
 * Device workspace, in bytes, that skv_cascade_decode and
 * skv_cascade_decode_varlen need for these sizes (the per-chunk states of the
 * shared-prefix pass; the two size that pass for different shares of the
 * SMs, and this is enough for either).  sm_count > 0 is used as given; 0
 * means the current device's SM count (the chunking depends on it).
 * Returns 0 for invalid sizes.
 */
size_t skv_cascade_workspace_size(int32_t B, int32_t Hq, int32_t Hkv, int32_t D,
                                  int32_t prefix_len, int32_t sm_count);

/*
 * Two-level cascade decode attention ([F2] §⑥): every request b attends to a
 * shared prefix of prefix_len tokens (pool pages prefix_pages[0 ..
 * ceil(prefix_len/page))) followed by its own suffix of ctx[b] tokens (pool
 * pages block_table[b][..]), as one softmax over prefix || suffix.
 *   1. Shared-prefix pass on the tensor cores (tcgen05): the prefix KV of each
 *      kv head is read once for all B*G query rows, as dense QK^T and PV
 *      products; it writes one state per prefix chunk into `workspace`.
 *   2. The suffixes run through the split-KV decode (as skv_splitkv_decode
 *      with `num_splits`), writing o_part / lse_part.
 *   3. One combine pass merges the prefix chunks into the prefix state
 *      (o_pre [B, Hq, D] fp32, s_pre [B, Hq] base 2, each written if not
 *      NULL), the splits into the suffix state, and the two with the
 *      two-state merge, prefix first, into out [B, Hq, D] (`dtype`) and, if
 *      not NULL, lse_out [B, Hq] (base 2).
 * Layouts as for skv_splitkv_decode; prefix_pages is a device int32 array.
 * prefix_len = 0 gives an empty prefix state (o = 0, s = -inf); ctx[b] = 0 an
 * empty suffix; both empty give out = 0, lse_out = -inf.
 * workspace: at least skv_cascade_workspace_size(B, Hq, Hkv, D, prefix_len, 0)
 *   bytes, 16-byte aligned; no initial contents are needed.  Calls that
 *   share a workspace must not overlap on the GPU.
 * All three steps are queued on `stream`, chained by programmatic dependent
 * launch: the suffix pass starts while the prefix pass runs (each sized to
 * share the GPU), and the combine waits for both.
 * Supported: dtype SKV_F16 or SKV_BF16 (the tensor-core products in the
 *   same type), D = 128, page = 16, G = Hq/Hkv in {1, 2, 4, 8},
 *   1 <= num_splits <= 256.  Device-side checks as for skv_splitkv_decode
 *   (prefix page ids included).
 */
skv_status skv_cascade_decode(const void* q, const void* k_cache, const void* v_cache,
                              int32_t num_pool_pages,
                              const int32_t* prefix_pages, int32_t prefix_len,
                              const int32_t* block_table, int32_t max_pages,
                              const int32_t* ctx,
                              int32_t B, int32_t Hq, int32_t Hkv, int32_t D, int32_t page,
                              int32_t num_splits, float sm_scale, skv_dtype dtype,
                              float* o_pre, float* s_pre,
                              float* o_part, float* lse_part,
                              void* out, float* lse_out,
                              void* workspace, size_t workspace_bytes, skv_stream_t stream);

/*
 * Two-level cascade decode whose suffixes have a split count per sequence:
 * as skv_cascade_decode, with the suffix pass and its merge as in
 * skv_splitkv_decode_varlen (plan, num_units, max_split_pages from
 * skv_splitkv_plan_varlen over the suffix contexts; o_part / lse_part with a
 * split axis max_splits long).  Workspace as for skv_cascade_decode.
 */
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
                                     skv_stream_t stream);

/*
 * One shared level of a multi-level cascade: the requests are cut into
 * num_groups contiguous groups, group g = requests [group_start[g],
 * group_start[g+1]), whose members all attend to the same group_len[g]
 * tokens on the pool pages group_pages[g][0 .. ceil(group_len[g]/page)).
 *   group_start: host int32 [num_groups + 1], non-decreasing, from 0 to B.
 *   group_len:   host int32 [num_groups], >= 0 (0: the group shares nothing
 *                at this level).
 *   group_pages: host array of num_groups device pointers (int32, 4-byte
 *                aligned; may be NULL where group_len is 0).
 */
typedef struct {
    int32_t num_groups;
    const int32_t* group_start;
    const int32_t* group_len;
    const int32_t* const* group_pages;
} skv_cascade_level;

/*
 * Device workspace, in bytes, that skv_cascade_decode_multilevel needs for
 * these levels and sizes (the prefix-chunk states of every level).  sm_count
 * as for skv_cascade_workspace_size.  Returns 0 for invalid arguments.
 */
size_t skv_cascade_multilevel_workspace_size(int32_t num_levels, const skv_cascade_level* levels,
                                             int32_t B, int32_t Hq, int32_t Hkv, int32_t D,
                                             int32_t sm_count);

/*
 * Multi-level cascade decode attention ([F2] §⑥: attention level by level,
 * then merge): request b attends, as one softmax, to the concatenation of
 * its group's shared tokens at level 0, 1, ..., num_levels - 1 and then its
 * own suffix of ctx[b] tokens (block_table[b][..]).  Each group's shared
 * tokens go through the tensor-core prefix pass for the group's requests
 * only (their K/V read once for the group); the suffixes through the
 * split-KV decode; one combine merges every level's chunk states into the
 * prefix state (o_pre, s_pre: over all shared levels) and that with the
 * suffix state into out and lse_out.  With one level of one group this is
 * skv_cascade_decode.  Arguments, layouts, workspace rules (sized by
 * skv_cascade_multilevel_workspace_size), support and device-side checks as
 * for skv_cascade_decode; a level list that does not cover [0, B) in order
 * returns SKV_ERR_INVALID_ARG.
 */
skv_status skv_cascade_decode_multilevel(const void* q, const void* k_cache, const void* v_cache,
                                         int32_t num_pool_pages, int32_t num_levels,
                                         const skv_cascade_level* levels,
                                         const int32_t* block_table, int32_t max_pages,
                                         const int32_t* ctx, int32_t B, int32_t Hq, int32_t Hkv,
                                         int32_t D, int32_t page, int32_t num_splits,
                                         float sm_scale, skv_dtype dtype, float* o_pre,
                                         float* s_pre, float* o_part, float* lse_part, void* out,
                                         float* lse_out, void* workspace, size_t workspace_bytes,
                                         skv_stream_t stream);

/*
 * Reads and clears the error word of the current CUDA device: *code is 0 or
 * the skv_status of the first device-side error since the last call, *detail
 * an index that identifies it (0 if none).  Synchronises the device.
 */
skv_status skv_get_device_error(int32_t* code, int32_t* detail);

/*
 * As skv_get_device_error, but waits only for the work queued on `stream`
 * (NULL: the legacy default stream, which waits for every blocking stream):
 * the word then holds every error of that work.  Kernels still running on
 * other streams may record an error later, which the next poll reports.
 * The first error since the word was last cleared wins; later ones are not
 * kept.
 */
skv_status skv_poll_device_error(int32_t* code, int32_t* detail, skv_stream_t stream);

/*
 * Self-test of the bounded device waits (the pages have no counterpart: it
 * checks this library's failure reporting without any fault).  Every
 * shared-memory barrier wait in the library's kernels gives up after a
 * limit (2 s), records SKV_ERR_TIMEOUT in the error word and returns, so a
 * lost copy can neither hang the GPU nor pass silently.  This call launches
 * one small kernel on `stream` that runs those same wait routines, with a
 * limit of limit_ns nanoseconds, on barriers that nothing ever completes (no
 * copy is issued, so nothing is left in flight):
 *   mode 0: the wait of the decode and merge kernels gives up and records
 *           SKV_ERR_TIMEOUT with detail 100;
 *   mode 1: the abort-aware wait of the warp-specialised kernels: one warp's
 *           limit runs out (SKV_ERR_TIMEOUT, detail 101) and raises the
 *           block's abort flag; a second warp, waiting on another barrier
 *           with a limit 100 times longer, sees the flag and returns without
 *           recording anything.
 * The kernel then returns normally and the context stays usable; read the
 * outcome with skv_get_device_error or skv_poll_device_error.
 * Limits: mode 0 or 1; 1000 <= limit_ns <= 10000000 (else SKV_ERR_INVALID_ARG).
 */
skv_status skv_selftest_bounded_wait(int32_t mode, int64_t limit_ns, skv_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* SKV_H_ */
