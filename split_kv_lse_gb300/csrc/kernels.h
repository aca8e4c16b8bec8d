// kernels.h -- internal launch interface between the C ABI (api.cu) and the
// kernel translation units.  Not installed; no torch types anywhere.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/skv.h"

namespace skv {

struct DeviceInfo {
    int device = -1;
    int sm_count = 0;
    size_t max_smem_optin = 0;
    unsigned long long* err = nullptr;  // device address of the error word
};
// Cached attributes of the current CUDA device (queried once per device).
skv_status current_device(const DeviceInfo** out);

inline size_t dtype_size(skv_dtype t) { return t == SKV_F32 ? 4 : 2; }

// ---------------------------------------------------------------- merges
cudaError_t launch_merge_state(const void* va, const float* sa, const void* vb, const float* sb,
                               void* vo, float* so, int64_t rows, int64_t D, skv_dtype dt,
                               bool in_place, const DeviceInfo& dev, cudaStream_t st);

// Which N-state merge path a call takes (host logic, shared with the
// workspace-size query so the two always agree).
struct MergeStatesPlan {
    bool team_kernel = false;  // warp-per-row bulk kernel (nsplit warps per row if > 1)
    bool row_cta = false;      // bulk CTA per row (per_split states per warp), no workspace
    int nsplit = 1;            // CTAs per row on the CTA path (>1 needs workspace)
    int per_split = 0;         // states per CTA on the CTA path
    size_t ws_bytes = 0;       // workspace the plan needs
};
// ctas_per_sm: CTAs the one-CTA-per-row path aims for per SM (the chunks of
// a row spread over that many).  allow_bulk_split: few rows with many states
// may instead take the two-level warp-per-row path (bulk copies), given the
// workspace; the fixed-scratch entry point keeps the CTA path.
constexpr int kMergeCtasPerSm = 2;
MergeStatesPlan plan_merge_states(int64_t rows, int64_t N, int64_t D, int chunks, int sm_count,
                                  size_t ws_available, int ctas_per_sm, bool allow_bulk_split);
size_t merge_states_ws_upper_bound(int64_t rows, int64_t N, int64_t D);

cudaError_t launch_merge_states(const void* v, const float* s, void* vo, float* so, int64_t S,
                                int64_t N, int64_t H, int64_t D, skv_dtype dt, void* ws,
                                size_t ws_bytes, int ctas_per_sm, bool allow_bulk_split,
                                const DeviceInfo& dev, cudaStream_t st);

// Combine pass of the split-KV decode: merges NS fp32 partial states per row
// (rows = B*Hq) into `out` (out_dt) and optional lse_out.  For the cascade,
// C fp32 prefix-chunk states per row (pre_part [rows, C, D], pre_lse
// [rows, C]) are first merged into the prefix state -- written to o_pre,
// s_pre when those are not null -- which is then merged with the split
// states (prefix first).  Launched as a programmatic dependent of the
// preceding kernel on `st` when pdl is set.
struct CombineArgs {
    const float* o_part;
    const float* lse_part;
    int64_t rows;
    int NS;  // split-axis length of o_part / lse_part
    // Per-sequence split counts ([B], row r reads seq_splits[r / Hq] states)
    // or nullptr (every row reads NS states).
    const int32_t* seq_splits;
    int Hq;
    int64_t D;
    void* out;
    skv_dtype out_dt;
    float* lse_out;
    const float* pre_part;
    const float* pre_lse;
    int C;
    float* o_pre;
    float* s_pre;
};
cudaError_t launch_combine(const CombineArgs& a, bool pdl, const DeviceInfo& dev, cudaStream_t st);

// ---------------------------------------------------------------- decode
struct DecodeArgs {
    const void* q;
    const void* k_cache;
    const void* v_cache;
    int32_t num_pool_pages;
    const int32_t* block_table;
    int32_t max_pages;
    const int32_t* ctx;
    int32_t B, Hq, Hkv, D, page, num_splits;
    float sm_scale;
    float* o_part;
    float* lse_part;
    int32_t* ranges_dbg;
    bool bf16;  // q, K, V are bf16 (else fp16)
    // Per-sequence split counts: `units` lists num_units (sequence, split)
    // pairs as int32 [b, split | splits_b << 16], one CTA per pair and kv
    // head, and num_splits is then the split-axis length of o_part;
    // max_split_pages is the longest split of the list (sets the CTA shape).
    // units == nullptr: every sequence has num_splits splits.
    const int32_t* units = nullptr;
    int32_t num_units = 0;
    int32_t max_split_pages = 0;
    // Cascade chaining (programmatic dependent launch): when set, the pass
    // is launched as a dependent of the preceding shared-prefix pass in the
    // same stream, so that the two run side by side, and the pass's last CTA
    // (counted on *done_ctr, zeroed by that prefix pass) waits for the
    // prefix pass to complete, so that the pass completes after it.
    unsigned int* done_ctr = nullptr;
};
cudaError_t launch_splitkv_decode(const DecodeArgs& a, const DeviceInfo& dev, cudaStream_t st);

// ---------------------------------------------------------------- cascade
struct CascadeArgs {
    const void* q;
    const void* k_cache;
    const void* v_cache;
    int32_t num_pool_pages;
    const int32_t* prefix_pages;
    int32_t prefix_len;
    int32_t B, Hq, Hkv;
    float sm_scale;
    bool bf16;  // q, K, V are bf16 (else fp16)
    // Chaining in one stream (programmatic dependent launch): every launch
    // lets the next kernel start at once.  zero_ctr (first launch of a
    // cascade): CTA 0 zeroes this counter before that.  chained (later
    // launches): launched as a dependent of the previous prefix pass, and
    // each CTA waits for that pass to complete before it exits.
    unsigned int* zero_ctr = nullptr;
    bool chained = false;
};
// Grid of the shared-prefix pass: M tiles of 128 query rows, prefix blocks
// of 128 keys per chunk, number of chunks.
void cascade_prefix_geometry(int B, int G, int Hkv, int prefix_len, int sm_count, int* mtiles,
                             int* blocks_per_chunk, int* nchunks);
// Launches nchunks chunk CTAs per (M-tile pair, kv head); chunk c writes
// slot chunk_offset + c of chunk_stride slots per row (slots past the
// prefix's last block get an empty state).
cudaError_t launch_cascade_prefix(const CascadeArgs& a, const DeviceInfo& dev, float* pre_part,
                                  float* pre_lse, int nchunks, int blocks_per_chunk, int mtiles,
                                  int chunk_stride, int chunk_offset, cudaStream_t st);

}  // namespace skv
