// merge.cu -- attention-state merge kernels for sm_103a.
//
// Pages: [F2] "F2 讲解：merge_state，以 2 为底的 LSE 合并" (§③ two states,
// §④ N states in the [S, N, H, D] layout, §⑤ empty states, §⑦ the
// vectorised CUDA kernels and the large-N kernel),
// [FA] "FlashAttention 的空行 LSE:FA-2 的 +inf 约定与后来的变化" (§2.2
// sanitize_lse, §4.1 the zero-reciprocal rule for an empty row).
//
// All three kernels are HBM-bound streams.  Design (GB300, not the pages'
// program-per-row Triton): a row's D elements are split into 16-byte chunks
// and a power-of-two "team" of lanes owns one row, so every load and store is
// a 128-bit coalesced access; each thread keeps several rows (or states) of
// loads in flight before it computes; all arithmetic is fp32.
//   merge_state_kernel        two states, team per row (in-place variant too)
//   merge_states_bulk_kernel  N states, warp per row, batches of TMA bulk copies: many rows
//   merge_states_cta_kernel   N states, one CTA (8 warps) per row or per chunk
//                             of a row's states: few rows, many states; the
//                             chunks of a row meet in a workspace and the
//                             last-arriving CTA merges them (associativity,
//                             [F2] §①) -- never a spin-wait.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace skv {
namespace {

#define SKV_HOSTDEV_CONST __host__ __device__ constexpr
constexpr int kThreads = 256;

// Lanes of this thread's team inside its warp (teams are aligned powers of 2).
SKV_DEVINL unsigned team_mask(int tpr) {
    if (tpr == 32) return 0xffffffffu;
    unsigned lane = threadIdx.x & 31;
    return ((1u << tpr) - 1u) << (lane & ~(unsigned)(tpr - 1));
}

// The two-state formula of [F2] §③ with the guards of [F2] §⑤ / [FA] §2.2.
// Written symmetrically (separate products, one rounded add) so that
// swapping the operands gives bit-identical results.
struct TwoWeights {
    float wa, wb, inv, s;
};
SKV_DEVINL TwoWeights two_weights(float sa, float sb) {
    float a = sanitize_lse(sa), b = sanitize_lse(sb);
    float m = fmaxf(a, b);
    TwoWeights t;
    t.wa = merge_weight(a, m);
    t.wb = merge_weight(b, m);
    float w = __fadd_rn(t.wa, t.wb);
    t.inv = w > 0.f ? 1.f / w : 0.f;  // [FA] §4.1: empty row -> reciprocal 0
    t.s = m + log2f(w);               // -inf + log2(0) = -inf for a double-empty row
    return t;
}
SKV_DEVINL float blend(float wa, float xa, float wb, float xb, float inv) {
    float ta = wa > 0.f ? __fmul_rn(wa, xa) : 0.f;  // a zero-weight state is not read
    float tb = wb > 0.f ? __fmul_rn(wb, xb) : 0.f;
    return __fmul_rn(__fadd_rn(ta, tb), inv);
}

// ---------------------------------------------------------------- two-state merge
// Coefficients of the merged row: v = ca * v_a + cb * v_b with
// ca = w_a / W, cb = w_b / W.  A zero-weight operand's vector is zeroed
// before use (it is never read into the result, even if not finite).
struct TwoCoef {
    float ca, cb, s;
};
SKV_DEVINL TwoCoef two_coef(float sa, float sb) {
    const TwoWeights t = two_weights(sa, sb);
    TwoCoef c;
    c.ca = __fmul_rn(t.wa, t.inv);
    c.cb = __fmul_rn(t.wb, t.inv);
    c.s = t.s;
    return c;
}

// Team of tpr lanes per row, each lane owning CPT 16-byte chunks
// (c = l + k*tpr); U rows in flight per lane.
template <typename T, int CPT, int U, bool kInPlace>
__global__ void __launch_bounds__(kThreads)
merge_state_kernel(const T* va, const float* sa, const T* __restrict__ vb,
                   const float* __restrict__ sb, T* vo, float* so, int64_t rows, int chunks,
                   int tpr_log2) {
    constexpr int E = Vec<T>::N;
    const int tpr = 1 << tpr_log2;
    const int64_t gt = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t team = gt >> tpr_log2;
    const int64_t nteams = ((int64_t)gridDim.x * blockDim.x) >> tpr_log2;
    const int l = (int)(gt & (tpr - 1));
    const unsigned tmask = team_mask(tpr);
    const int64_t row_stride = (int64_t)chunks * 16;  // bytes per row

    for (int64_t r0 = team; r0 < rows; r0 += (int64_t)U * nteams) {
        float xa[U], xb[U];
        uint4 ra[U][CPT], rb[U][CPT];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t r = r0 + u * nteams;
            const bool ok = r < rows;
            xa[u] = ok ? sa[r] : -INFINITY;
            xb[u] = ok ? sb[r] : -INFINITY;
#pragma unroll
            for (int k = 0; k < CPT; ++k) {
                const int c = l + k * tpr;
                ra[u][k] = rb[u][k] = make_uint4(0, 0, 0, 0);
                if (ok && c < chunks) {
                    const char* pa = reinterpret_cast<const char*>(va) + r * row_stride + c * 16;
                    const char* pb = reinterpret_cast<const char*>(vb) + r * row_stride + c * 16;
                    ra[u][k] = kInPlace ? ld_coherent(pa) : ld_stream(pa);
                    rb[u][k] = ld_stream(pb);
                }
            }
        }
        // In place, s_out aliases s_a: every lane of the team has read s_a[r]
        // before the team's first lane overwrites it.
        if (kInPlace) __syncwarp(tmask);
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t r = r0 + u * nteams;
            if (r >= rows) continue;
            const TwoCoef cf = two_coef(xa[u], xb[u]);
#pragma unroll
            for (int k = 0; k < CPT; ++k) {
                const int c = l + k * tpr;
                if (c >= chunks) continue;
                if (!(cf.ca > 0.f)) ra[u][k] = make_uint4(0, 0, 0, 0);
                if (!(cf.cb > 0.f)) rb[u][k] = make_uint4(0, 0, 0, 0);
                float fa[E], fb[E], fo[E];
                to_float<T>(ra[u][k], fa);
                to_float<T>(rb[u][k], fb);
#pragma unroll
                for (int e = 0; e < E; ++e)
                    fo[e] = __fadd_rn(__fmul_rn(cf.ca, fa[e]), __fmul_rn(cf.cb, fb[e]));
                char* po = reinterpret_cast<char*>(vo) + r * row_stride + c * 16;
                st_stream(po, from_float<T>(fo));
            }
            if (l == 0) so[r] = cf.s;
        }
    }
}

// ---------------------------------------------------------------- N-state, warp per row
// One warp per (pos, h) row.  The row's N LSEs are read once (lane n holds
// states n, n + 32, ...); the non-empty states are compacted (ballot) into a
// list of (index, weight) in shared memory -- a zero-weight state is never
// read, so its v cannot poison the sum.  Their v rows (D contiguous
// elements) then stream through a per-warp double buffer of two batches of
// kRowBatch rows: a batch is kRowBatch TMA bulk copies issued by kRowBatch
// lanes at once and completed on one mbarrier, so the ring bookkeeping is
// paid once per batch, not once per state.
// Warps (rows) per CTA, measured on the same shape (us, medians of 40, L2
// flushed): 2: 45.1, 4: 44.4-45.0, 8: 43.0-43.4, 16: 45.1 -- 8 warps, four
// CTAs (of about 53 KB of shared memory) resident per SM.
constexpr int kRowWarps = 8;
// Rows per batch, measured on S=256 N=64 H=32 D=128 fp32 (us, 30 steps, L2
// flushed): 3: 49.5, 4: 45.8-46.3, 5: 45.0, 6: 44.5-44.8, 7: 45.0, 8: 46.3.
constexpr int kRowBatch = 6;
constexpr int kBulkMaxN = 256;

// Entries per warp of the compacted state list: N rounded up to a warp.
SKV_HOSTDEV_CONST int rows_list_len(int N) { return (N + 31) & ~31; }

// Ring of NBUF batches of BATCH rows per warp: the many-rows path keeps
// (kRowBatch, 2); the two-level split, whose warps each stream only a chunk
// of a row, keeps more in flight per warp: (kSplitBatch, kSplitBufs).
constexpr int kSplitBatch = 8;
constexpr int kSplitBufs = 3;

template <int BATCH, int NBUF>
SKV_HOSTDEV_CONST size_t rows_smem_bytes(int row_bytes, int N) {
    return (size_t)kRowWarps * NBUF * BATCH * row_bytes +           // the batch ring
           (size_t)kRowWarps * NBUF * sizeof(uint64_t) +            // one mbarrier per buffer
           (size_t)kRowWarps * rows_list_len(N) * (sizeof(float) + sizeof(int));  // compacted list
}

// Two-level split of the warp-per-row merge (few rows, many states): warp
// (row, split) merges states [split * per, min(N, (split + 1) * per)) of its
// row into an unnormalised partial (m, W, sum w v) in the workspace, then
// takes a ticket; the row's last warp merges the nsplit partials
// (associativity, [F2] §①) and writes the row -- never a spin-wait.
struct BulkSplit {
    int nsplit = 1;       // warps per row; 1: no workspace, each warp writes its row
    int per = 0;          // states per warp (<= kBulkMaxN)
    float* ws_v = nullptr;       // [rows, nsplit, D] fp32 unnormalised sums
    float* ws_s = nullptr;       // [rows, nsplit, 2]: chunk max m, weight sum W
    unsigned* ws_cnt = nullptr;  // [rows] arrival tickets, zero between calls
};

// One warp streams states [n_begin, n_begin + n_cnt) of row (pos, h): their
// LSEs are read once (lane n holds states n, n + 32, ...), the non-empty
// ones are compacted (ballot) into a list of (index, weight) in shared
// memory -- a zero-weight state is never read, so its v cannot poison the
// sum -- and their v rows stream through the warp's ring of NBUF batches of
// BATCH rows (one TMA bulk copy per row, issued by BATCH lanes at once,
// completed on one mbarrier per batch).  Returns the chunk max m (log2
// units), W = sum 2^(s - m) and acc = sum 2^(s - m) v (this lane's 16-byte
// chunk of D).  The ring's barriers must be initialised.  Returns false if
// a bounded wait gave up (error recorded; every copy of the warp has landed
// or been waited for once more).
template <typename T, int BATCH, int NBUF>
SKV_DEVINL bool warp_stream_states(const T* __restrict__ v, const float* __restrict__ s,
                                   int64_t pos, int64_t h, int64_t H, int N, int n_begin,
                                   int n_cnt, int chunks, uint8_t* ring, uint64_t* bars,
                                   float* cw, int* cidx, unsigned long long* err, float& m_out,
                                   float& W_out, float (&acc)[Vec<T>::N]) {
    constexpr int E = Vec<T>::N;
    const int lane = threadIdx.x & 31;
    const int row_bytes = chunks * 16;
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = 0.f;
    // s[pos, n, h] at (pos*N + n)*H + h ([F2] §④).
    const float* srow = s + (pos * N + n_begin) * H + h;
    float sv[kBulkMaxN / 32];
    float m = -INFINITY;
#pragma unroll
    for (int k = 0; k < kBulkMaxN / 32; ++k) {
        const int n = lane + 32 * k;
        sv[k] = n < n_cnt ? sanitize_lse(__ldg(srow + (int64_t)n * H)) : -INFINITY;
        m = fmaxf(m, sv[k]);
    }
    m = warp_max(m);
    float W = 0.f;
    int nnz = 0;  // non-empty states, in state order
#pragma unroll
    for (int k = 0; k < kBulkMaxN / 32; ++k) {
        const float w = merge_weight(sv[k], m);  // 0 for empty states and n >= n_cnt
        W += w;
        const unsigned live = __ballot_sync(0xffffffffu, w > 0.f);
        if (w > 0.f) {
            const int at = nnz + __popc(live & ((1u << lane) - 1u));
            cidx[at] = lane + 32 * k;
            cw[at] = w;
        }
        nnz += __popc(live);
    }
    m_out = m;
    W_out = warp_sum(W);
    __syncwarp();

    const char* vrow = reinterpret_cast<const char*>(v) + ((pos * N + n_begin) * H + h) * (int64_t)row_bytes;
    const int64_t nstride = H * (int64_t)row_bytes;
    const uint64_t pol = policy_evict_first();
    const int nbatch = (nnz + BATCH - 1) / BATCH;
    auto issue = [&](int j) {  // batch j into buffer j % NBUF
        const int cnt = min(BATCH, nnz - j * BATCH);
        uint64_t* bar = &bars[j % NBUF];
        if (lane == 0) mbar_arrive_expect_tx(bar, (uint32_t)(cnt * row_bytes));
        __syncwarp();
        if (lane < cnt)
            bulk_g2s(ring + ((j % NBUF) * BATCH + lane) * row_bytes,
                     vrow + (int64_t)cidx[j * BATCH + lane] * nstride, row_bytes, bar, pol);
    };
    for (int j = 0; j < NBUF && j < nbatch; ++j) issue(j);
    for (int j = 0; j < nbatch; ++j) {
        const bool ok = mbar_wait(&bars[j % NBUF], (uint32_t)((j / NBUF) & 1), err, 6);
        if (!__all_sync(0xffffffffu, ok)) {
            // A bounded wait gave up (error recorded): one more bounded wait
            // for each other batch in flight, then stop.
            for (int jj = j + 1; jj < nbatch && jj < j + NBUF; ++jj)
                mbar_wait(&bars[jj % NBUF], (uint32_t)((jj / NBUF) & 1), err, 7);
            return false;
        }
        const int cnt = min(BATCH, nnz - j * BATCH);
        if (lane < chunks) {
            const uint8_t* buf = ring + (j % NBUF) * BATCH * row_bytes + lane * 16;
#pragma unroll
            for (int b = 0; b < BATCH; ++b) {
                if (b < cnt) {
                    const float w = cw[j * BATCH + b];
                    float f[E];
                    to_float<T>(*reinterpret_cast<const uint4*>(buf + b * row_bytes), f);
#pragma unroll
                    for (int e = 0; e < E; ++e) acc[e] = fmaf(w, f[e], acc[e]);
                }
            }
        }
        __syncwarp();  // buffer fully read
        if (j + NBUF < nbatch) issue(j + NBUF);
    }
    return true;
}

template <typename T, int BATCH, int NBUF>
__global__ void __launch_bounds__(kRowWarps * 32)
merge_states_bulk_kernel(const T* __restrict__ v, const float* __restrict__ s,
                         T* __restrict__ vo, float* __restrict__ so, int64_t rows, int N,
                         int64_t H, int chunks, unsigned long long* err, const BulkSplit bs) {
    constexpr int E = Vec<T>::N;
    extern __shared__ __align__(128) uint8_t smem[];
    const int row_bytes = chunks * 16;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int per = bs.nsplit > 1 ? bs.per : N;  // states this warp may own (<= kBulkMaxN)
    uint8_t* ring = smem + (size_t)warp * NBUF * BATCH * row_bytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (size_t)kRowWarps * NBUF * BATCH * row_bytes) +
                     warp * NBUF;
    float* cw = reinterpret_cast<float*>(smem + (size_t)kRowWarps * NBUF * BATCH * row_bytes +
                                         (size_t)kRowWarps * NBUF * sizeof(uint64_t)) + warp * rows_list_len(per);
    int* cidx = reinterpret_cast<int*>(cw + (kRowWarps - warp) * rows_list_len(per)) + warp * rows_list_len(per);

    // Warp wg: row wg (one warp per row), or with the split the warps of one
    // (pos, split) over consecutive heads h, so that a CTA's warps read
    // adjacent rows of each state (one contiguous run of the [S, N, H, D]
    // layout) as the many-rows path does.
    const int64_t wg = (int64_t)blockIdx.x * kRowWarps + warp;
    int64_t r = wg;
    int split = 0;
    if (bs.nsplit > 1) {
        const int64_t hh = wg % H, t = wg / H;
        split = (int)(t % bs.nsplit);
        r = (t / bs.nsplit) * H + hh;
    }
    if (r >= rows) return;  // whole warp; no block-wide barrier follows
    if (lane == 0) {
        for (int i = 0; i < NBUF; ++i) mbar_init(&bars[i], 1);
        fence_mbar_init();
    }
    __syncwarp();
    const int n_begin = split * per;
    const int n_cnt = min(per, N - n_begin);  // >= 1
    float m, W, acc[E];
    if (!warp_stream_states<T, BATCH, NBUF>(v, s, r / H, r % H, H, N, n_begin, n_cnt, chunks, ring,
                                            bars, cw, cidx, err, m, W, acc))
        return;
    if (bs.nsplit > 1) {
        // Publish this warp's partial unnormalised (an fp32 s = m + log2 W of
        // magnitude ~40 would carry ~1e-6 relative weight error), then take a
        // ticket; the warp that draws the row's last one merges.
        const int64_t slot = r * bs.nsplit + split;
        const int D = chunks * E;
        if (lane < chunks) {
            float* dst = bs.ws_v + slot * D + lane * E;
#pragma unroll
            for (int e = 0; e < E; e += 4)
                *reinterpret_cast<float4*>(dst + e) = make_float4(acc[e], acc[e + 1], acc[e + 2], acc[e + 3]);
        }
        if (lane == 0) {
            bs.ws_s[slot * 2 + 0] = m;
            bs.ws_s[slot * 2 + 1] = W;
        }
        __threadfence();  // every lane's partial is visible device-wide ...
        __syncwarp();     // ... before lane 0 takes the ticket
        unsigned last = 0;
        if (lane == 0) {
            const unsigned ticket = atomicAdd(&bs.ws_cnt[r], 1u);
            last = ticket == (unsigned)bs.nsplit - 1u;
            if (last) bs.ws_cnt[r] = 0u;  // every warp of the row has arrived
        }
        if (!__shfl_sync(0xffffffffu, last, 0)) return;
        __threadfence();
        // The row's partials: lane k holds partial k's (m, W) (nsplit <= 64).
        const float* ps = bs.ws_s + r * bs.nsplit * 2;
        float mk[2], wk[2];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int k = lane + 32 * i;
            mk[i] = k < bs.nsplit ? ld_cg_f32(ps + 2 * k) : -INFINITY;
            wk[i] = k < bs.nsplit ? ld_cg_f32(ps + 2 * k + 1) : 0.f;
        }
        const float M = warp_max(fmaxf(mk[0], mk[1]));
        float sc[2];
#pragma unroll
        for (int i = 0; i < 2; ++i) sc[i] = merge_weight(mk[i], M);
        const float WW = warp_sum(sc[0] * wk[0] + sc[1] * wk[1]);
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] = 0.f;
        const float* pv = bs.ws_v + r * bs.nsplit * (int64_t)D + lane * E;
        // kFinalBatch partials per L2 round trip: every load of a batch is
        // issued before any is used.
        constexpr int kFinalBatch = 16 * 4 / E;
        for (int k0 = 0; k0 < bs.nsplit; k0 += kFinalBatch) {
            float4 raw[kFinalBatch][E / 4];
            float c[kFinalBatch];
#pragma unroll
            for (int i = 0; i < kFinalBatch; ++i) {
                const int k = k0 + i;
                c[i] = __shfl_sync(0xffffffffu, k < 32 ? sc[0] : sc[1], k & 31);
                if (k >= bs.nsplit) c[i] = 0.f;
#pragma unroll
                for (int e = 0; e < E; e += 4)  // a zero-weight partial is not read
                    raw[i][e / 4] = (c[i] > 0.f && lane < chunks)
                                        ? __ldcg(reinterpret_cast<const float4*>(pv + (int64_t)k * D + e))
                                        : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int i = 0; i < kFinalBatch; ++i) {
                if (!(c[i] > 0.f)) continue;
#pragma unroll
                for (int e = 0; e < E; e += 4) {
                    acc[e] = fmaf(c[i], raw[i][e / 4].x, acc[e]);
                    acc[e + 1] = fmaf(c[i], raw[i][e / 4].y, acc[e + 1]);
                    acc[e + 2] = fmaf(c[i], raw[i][e / 4].z, acc[e + 2]);
                    acc[e + 3] = fmaf(c[i], raw[i][e / 4].w, acc[e + 3]);
                }
            }
        }
        m = M;
        W = WW;
    }
    const float inv = W > 0.f ? 1.f / W : 0.f;
    if (lane < chunks) {
        float f[E];
#pragma unroll
        for (int e = 0; e < E; ++e) f[e] = acc[e] * inv;
        st_stream(reinterpret_cast<char*>(vo) + r * row_bytes + lane * 16, from_float<T>(f));
    }
    if (lane == 0) so[r] = m + log2f(W);
}

// ---------------------------------------------------------------- N-state, bulk CTA per row
// Few rows, many states: one CTA of kRowCtaWarps warps per row, warp w
// streaming states [w * per, (w + 1) * per) through its own ring (as the
// warp-per-row kernel does), the warps' unnormalised partial states then
// merged in shared memory by warp 0 -- no workspace, no second pass through
// global memory ([F2] §① associativity; the large-N kernel of §⑦).
constexpr int kRowCtaWarps = 16;
constexpr int kRowCtaBatch = 8;
constexpr int kRowCtaBufs = 3;

SKV_HOSTDEV_CONST size_t rowcta_smem_bytes(int row_bytes, int per) {
    return (size_t)kRowCtaWarps * kRowCtaBufs * kRowCtaBatch * row_bytes +  // rings
           (size_t)kRowCtaWarps * kRowCtaBufs * sizeof(uint64_t) +          // barriers
           (size_t)kRowCtaWarps * rows_list_len(per) * (sizeof(float) + sizeof(int)) +
           (size_t)kRowCtaWarps * 2 * sizeof(float);                        // partial m, W
}

template <typename T>
__global__ void __launch_bounds__(kRowCtaWarps * 32, 1)
merge_states_rowcta_kernel(const T* __restrict__ v, const float* __restrict__ s,
                           T* __restrict__ vo, float* __restrict__ so, int N, int64_t H,
                           int chunks, int per, unsigned long long* err) {
    constexpr int E = Vec<T>::N;
    extern __shared__ __align__(128) uint8_t smem[];
    const int row_bytes = chunks * 16;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr size_t kRing = (size_t)kRowCtaBufs * kRowCtaBatch;
    uint8_t* rings = smem;
    uint64_t* bars_all = reinterpret_cast<uint64_t*>(smem + kRowCtaWarps * kRing * row_bytes);
    float* cw_all = reinterpret_cast<float*>(bars_all + kRowCtaWarps * kRowCtaBufs);
    int* cidx_all = reinterpret_cast<int*>(cw_all + kRowCtaWarps * rows_list_len(per));
    float* pm = reinterpret_cast<float*>(cidx_all + kRowCtaWarps * rows_list_len(per));
    float* pW = pm + kRowCtaWarps;

    const int64_t r = blockIdx.x;
    uint64_t* bars = bars_all + warp * kRowCtaBufs;
    if (lane == 0) {
        for (int i = 0; i < kRowCtaBufs; ++i) mbar_init(&bars[i], 1);
        fence_mbar_init();
    }
    __syncwarp();
    const int n_begin = warp * per;
    const int n_cnt = min(per, N - n_begin);
    float m = -INFINITY, W = 0.f, acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = 0.f;
    bool ok = true;
    if (n_cnt > 0)
        ok = warp_stream_states<T, kRowCtaBatch, kRowCtaBufs>(
            v, s, r / H, r % H, H, N, n_begin, n_cnt, chunks, rings + warp * kRing * row_bytes, bars,
            cw_all + warp * rows_list_len(per), cidx_all + warp * rows_list_len(per), err, m, W, acc);
    if (!ok) {  // a wait gave up (recorded): this warp adds nothing, the CTA still meets
        m = -INFINITY;
        W = 0.f;
    }
    __syncthreads();  // every ring is drained: reuse the first as [warps][D] partial sums
    float* pacc = reinterpret_cast<float*>(rings);
    const int D = chunks * E;
    if (lane < chunks) {
#pragma unroll
        for (int e = 0; e < E; e += 4)
            *reinterpret_cast<float4*>(pacc + warp * D + lane * E + e) =
                make_float4(acc[e], acc[e + 1], acc[e + 2], acc[e + 3]);
    }
    if (lane == 0) {
        pm[warp] = m;
        pW[warp] = W;
    }
    __syncthreads();
    if (warp != 0) return;
    // Warp 0 merges the kRowCtaWarps partial states and writes the row.
    const float mk = lane < kRowCtaWarps ? pm[lane] : -INFINITY;
    const float M = warp_max(mk);
    const float sc = merge_weight(mk, M);  // 0 for an empty partial
    const float WW = warp_sum(lane < kRowCtaWarps ? sc * pW[lane] : 0.f);
    float o[E];
#pragma unroll
    for (int e = 0; e < E; ++e) o[e] = 0.f;
#pragma unroll
    for (int k = 0; k < kRowCtaWarps; ++k) {
        const float c = __shfl_sync(0xffffffffu, sc, k);
        if (c > 0.f && lane < chunks) {
#pragma unroll
            for (int e = 0; e < E; ++e) o[e] = fmaf(c, pacc[k * D + lane * E + e], o[e]);
        }
    }
    const float inv = WW > 0.f ? 1.f / WW : 0.f;
    if (lane < chunks) {
#pragma unroll
        for (int e = 0; e < E; ++e) o[e] *= inv;
        st_stream(reinterpret_cast<char*>(vo) + r * row_bytes + lane * 16, from_float<T>(o));
    }
    if (lane == 0) so[r] = M + log2f(WW);
}

// ---------------------------------------------------------------- N-state, CTA per row
struct CtaParams {
    const void* v;        // Tin  [rows_outer.., N, H, D] (see row addressing below)
    const float* s;       // [S, N, H]
    void* vo;             // Tout [rows, D]
    float* so;            // [rows] or nullptr
    int64_t H;
    int N;
    int chunks;           // 16-byte chunks per row of D
    int tpr_log2;
    int nsplit;           // CTAs per row
    int per_split;        // states per CTA
    float* ws_v;          // [rows, nsplit, D] fp32 unnormalised chunk sums (nsplit > 1)
    float* ws_s;          // [rows, nsplit, 2]: chunk max m and weight sum W
    unsigned* ws_cnt;     // [rows] arrival tickets, zero between calls
    const float* extra_v; // [rows, D] fp32 state merged last, or nullptr
    const float* extra_s; // [rows]
    int pdl_wait;         // wait for the preceding grid (programmatic launch)
};



template <typename T>
SKV_DEVINL float block_reduce(float x, float* red, bool is_max) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    x = is_max ? warp_max(x) : warp_sum(x);
    __syncthreads();
    if (lane == 0) red[w] = x;
    __syncthreads();
    float r = red[0];
    for (int i = 1; i < (int)(blockDim.x >> 5); ++i) r = is_max ? fmaxf(r, red[i]) : r + red[i];
    return r;
}

template <typename Tin, typename Tout, int NB>
__global__ void __launch_bounds__(kThreads)
merge_states_cta_kernel(CtaParams p) {
    constexpr int E = Vec<Tin>::N;
    constexpr int EO = Vec<Tout>::N;
    __shared__ float red[32];
    // Team partial sums: nteams * D floats <= (256 / tpr) * (tpr * E) = 256 * E.
    __shared__ __align__(16) float part[kThreads * E];
    __shared__ int is_last;

    if (p.pdl_wait) pdl_wait_primary();

    const int64_t row = blockIdx.x;
    const int split = blockIdx.y;
    const int64_t pos = row / p.H, h = row % p.H;
    const int tpr = 1 << p.tpr_log2;
    const int nteams = kThreads >> p.tpr_log2;
    const int team = threadIdx.x >> p.tpr_log2;
    const int l = threadIdx.x & (tpr - 1);
    const int D = p.chunks * E;
    const int n_begin = split * p.per_split;
    const int n_end = min(p.N, n_begin + p.per_split);
    const float* srow = p.s + (pos * p.N) * p.H + h;

    // Chunk maximum and weight sum over this CTA's states.
    float m = -INFINITY;
    for (int n = n_begin + threadIdx.x; n < n_end; n += kThreads)
        m = fmaxf(m, sanitize_lse(srow[(int64_t)n * p.H]));
    m = block_reduce<float>(m, red, true);
    float W = 0.f;
    for (int n = n_begin + threadIdx.x; n < n_end; n += kThreads)
        W += merge_weight(sanitize_lse(srow[(int64_t)n * p.H]), m);
    W = block_reduce<float>(W, red, false);

    // Each team accumulates its states n = n_begin + team + k*nteams.
    float acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = 0.f;
    const int64_t row_bytes = (int64_t)p.chunks * 16;
    const char* vrow = reinterpret_cast<const char*>(p.v) + ((pos * p.N) * p.H + h) * row_bytes;
    const int64_t nstride = p.H * row_bytes;
    const bool lane_ok = l < p.chunks;
    for (int n0 = n_begin + team; n0 < n_end; n0 += NB * nteams) {
        float w[NB];
        uint4 raw[NB];
#pragma unroll
        for (int j = 0; j < NB; ++j) {
            const int n = n0 + j * nteams;
            w[j] = n < n_end ? merge_weight(sanitize_lse(srow[(int64_t)n * p.H]), m) : 0.f;
            raw[j] = (w[j] > 0.f && lane_ok)
                         ? (p.pdl_wait ? ld_cg(vrow + (int64_t)n * nstride + l * 16)
                                       : ld_stream(vrow + (int64_t)n * nstride + l * 16))
                         : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int j = 0; j < NB; ++j) {
            if (!(w[j] > 0.f)) continue;
            float f[E];
            to_float<Tin>(raw[j], f);
#pragma unroll
            for (int e = 0; e < E; ++e) acc[e] = fmaf(w[j], f[e], acc[e]);
        }
    }
    // Sum the teams' partial vectors through shared memory.
    if (lane_ok) {
#pragma unroll
        for (int e = 0; e < E; ++e) part[team * D + l * E + e] = acc[e];
    }
    __syncthreads();
    const float inv = W > 0.f ? 1.f / W : 0.f;
    const float s_chunk = m + log2f(W);
    // Thread d (< D) owns output element d.
    float vd = 0.f;
    if (threadIdx.x < D) {
        for (int t = 0; t < nteams; ++t) vd += part[t * D + threadIdx.x];
        vd *= inv;
    }
    float s_fin = s_chunk;

    if (p.nsplit > 1) {
        // Publish this chunk's partial state unnormalised -- (m, W, sum w v) --
        // so the final merge keeps single-pass accuracy (an fp32 s = m +
        // log2 W of magnitude ~40 would carry ~1e-6 relative weight error).
        // Then take a ticket; the CTA that draws the row's last ticket merges.
        if (threadIdx.x < D) {
            float raw = 0.f;
            for (int t = 0; t < nteams; ++t) raw += part[t * D + threadIdx.x];
            p.ws_v[(row * p.nsplit + split) * D + threadIdx.x] = raw;
        }
        if (threadIdx.x == 0) {
            p.ws_s[(row * p.nsplit + split) * 2 + 0] = m;
            p.ws_s[(row * p.nsplit + split) * 2 + 1] = W;
        }
        __threadfence();
        __syncthreads();
        if (threadIdx.x == 0) {
            const unsigned ticket = atomicAdd(&p.ws_cnt[row], 1u);
            is_last = (ticket == (unsigned)p.nsplit - 1u);
            if (is_last) p.ws_cnt[row] = 0u;  // every CTA of the row has arrived
        }
        __syncthreads();
        if (!is_last) return;
        __threadfence();
        float M = -INFINITY;
        for (int k = 0; k < p.nsplit; ++k) M = fmaxf(M, ld_cg_f32(&p.ws_s[(row * p.nsplit + k) * 2]));
        float WW = 0.f, a = 0.f;
        for (int k = 0; k < p.nsplit; ++k) {
            const float sc = merge_weight(ld_cg_f32(&p.ws_s[(row * p.nsplit + k) * 2]), M);
            if (!(sc > 0.f)) continue;
            WW = fmaf(sc, ld_cg_f32(&p.ws_s[(row * p.nsplit + k) * 2 + 1]), WW);
            if (threadIdx.x < D) a = fmaf(sc, ld_cg_f32(&p.ws_v[(row * p.nsplit + k) * D + threadIdx.x]), a);
        }
        vd = WW > 0.f ? a * (1.f / WW) : 0.f;
        s_fin = M + log2f(WW);
    }

    if (p.extra_v != nullptr) {
        // Final two-state merge with the extra state (cascade: prefix state
        // first, split states second).
        const TwoWeights t = two_weights(p.extra_s[row], s_fin);
        const float xe = threadIdx.x < D ? p.extra_v[row * D + threadIdx.x] : 0.f;
        vd = blend(t.wa, xe, t.wb, vd, t.inv);
        s_fin = t.s;
    }
    // Store: gather to shared memory, then 16-byte stores by `chunks` threads.
    __syncthreads();
    if (threadIdx.x < D) part[threadIdx.x] = vd;
    __syncthreads();
    if (threadIdx.x < D / EO) {
        float f[EO];
#pragma unroll
        for (int e = 0; e < EO; ++e) f[e] = part[threadIdx.x * EO + e];
        char* orow = reinterpret_cast<char*>(p.vo) + row * (int64_t)D * sizeof(Tout);
        st_stream(orow + threadIdx.x * 16, from_float<Tout>(f));
    }
    if (threadIdx.x == 0 && p.so != nullptr) p.so[row] = s_fin;
}

int log2_pow2_at_least(int x) {
    int l = 0;
    while ((1 << l) < x) ++l;
    return l;
}

template <typename T>
cudaError_t launch_merge_state_t(const void* va, const float* sa, const void* vb,
                                 const float* sb, void* vo, float* so, int64_t rows, int chunks,
                                 bool in_place, const DeviceInfo& dev, cudaStream_t st) {
    // Four 16-byte chunks per lane: a row's weights are computed by
    // ceil(chunks / 4) lanes, and each lane keeps 2 rows x 8 loads in flight.
    constexpr int CPT = 4, U = 2;
    const int tpr_log2 = log2_pow2_at_least((chunks + CPT - 1) / CPT);
    const int tpr = 1 << tpr_log2;
    const int64_t threads_needed = ((rows + U - 1) / U) * tpr;
    int64_t blocks = (threads_needed + kThreads - 1) / kThreads;
    const int64_t cap = (int64_t)dev.sm_count * 32;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    const T* a = static_cast<const T*>(va);
    const T* b = static_cast<const T*>(vb);
    T* o = static_cast<T*>(vo);
    if (in_place)
        merge_state_kernel<T, CPT, U, true><<<(unsigned)blocks, kThreads, 0, st>>>(
            a, sa, b, sb, o, so, rows, chunks, tpr_log2);
    else
        merge_state_kernel<T, CPT, U, false><<<(unsigned)blocks, kThreads, 0, st>>>(
            a, sa, b, sb, o, so, rows, chunks, tpr_log2);
    return cudaGetLastError();
}

template <typename Tin, typename Tout>
cudaError_t launch_cta(const CtaParams& p0, int64_t rows, const DeviceInfo& dev, cudaStream_t st,
                       bool pdl) {
    (void)dev;
    CtaParams p = p0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)rows, (unsigned)p.nsplit, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    p.pdl_wait = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, merge_states_cta_kernel<Tin, Tout, 4>, p);
}

}  // namespace

// ---------------------------------------------------------------- host entry points
cudaError_t launch_merge_state(const void* va, const float* sa, const void* vb, const float* sb,
                               void* vo, float* so, int64_t rows, int64_t D, skv_dtype dt,
                               bool in_place, const DeviceInfo& dev, cudaStream_t st) {
    const int chunks = (int)(D * (int64_t)dtype_size(dt) / 16);
    switch (dt) {
        case SKV_F32: return launch_merge_state_t<float>(va, sa, vb, sb, vo, so, rows, chunks, in_place, dev, st);
        case SKV_F16: return launch_merge_state_t<__half>(va, sa, vb, sb, vo, so, rows, chunks, in_place, dev, st);
        case SKV_BF16: return launch_merge_state_t<__nv_bfloat16>(va, sa, vb, sb, vo, so, rows, chunks, in_place, dev, st);
    }
    return cudaErrorInvalidValue;
}

static constexpr int64_t kTeamRows = 4096;  // rows at or above which the team kernel is used
static constexpr int kMaxSplit = 16;
// Two-level warp-per-row merge: at most kMaxBulkSplit warps per row, each
// with between kMinBulkPer and kBulkMaxN states, and about kBulkWarpsPerSm
// warps per SM in all (the bulk copies in flight per SM grow with them).
static constexpr int kMaxBulkSplit = 64;
static constexpr int kMinBulkPer = 16;
static constexpr int kBulkWarpsPerSm = 16;

static int max_split_for(int64_t N) {
    int64_t m = (N + 7) / 8;  // at least 8 states per CTA
    if (m > kMaxSplit) m = kMaxSplit;
    return (int)(m < 1 ? 1 : m);
}

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

static size_t ws_bytes_for(int64_t rows, int nsplit, int64_t D) {
    if (nsplit <= 1) return 0;
    return align256((size_t)rows * nsplit * D * 4) + align256((size_t)rows * nsplit * 8) +
           align256((size_t)rows * 4);
}

// The two-level warp-per-row split for these sizes (nsplit 1: none).
static void bulk_split_for(int64_t rows, int64_t N, int sm_count, int* nsplit, int* per) {
    const int64_t target = (int64_t)kBulkWarpsPerSm * (sm_count > 0 ? sm_count : 1);
    int64_t p = (N * rows + target - 1) / target;
    p = (p + kMinBulkPer - 1) / kMinBulkPer * kMinBulkPer;
    p = std::max<int64_t>(p, (N + kMaxBulkSplit - 1) / kMaxBulkSplit);
    p = std::min<int64_t>(std::max<int64_t>(p, kMinBulkPer), kBulkMaxN);
    const int64_t ns = (N + p - 1) / p;
    *nsplit = (int)ns;
    *per = (int)((N + ns - 1) / ns);  // the states spread evenly over the warps
}

static bool bulk_split_fits(int64_t N) { return N <= (int64_t)kBulkMaxN * kMaxBulkSplit; }

size_t merge_states_ws_upper_bound(int64_t rows, int64_t N, int64_t D) {
    if (rows <= 0) return 0;
    if (rows >= kTeamRows && N <= kBulkMaxN) return 0;
    size_t cta = rows < kTeamRows ? ws_bytes_for(rows, max_split_for(N), D) : 0;
    if (!bulk_split_fits(N)) return cta;
    // The most warps per row any SM count gives: kMinBulkPer states each.
    const int64_t most = std::min<int64_t>(kMaxBulkSplit, (N + kMinBulkPer - 1) / kMinBulkPer);
    return std::max(cta, ws_bytes_for(rows, (int)most, D));
}

MergeStatesPlan plan_merge_states(int64_t rows, int64_t N, int64_t D, int chunks, int sm_count,
                                  size_t ws_available, int ctas_per_sm, bool allow_bulk_split) {
    (void)chunks;
    MergeStatesPlan pl;
    if (rows >= kTeamRows && N <= kBulkMaxN) {
        pl.team_kernel = true;
        return pl;
    }
    if (allow_bulk_split && rows < kTeamRows && 2 * rows >= sm_count &&
        N <= (int64_t)kRowCtaWarps * kBulkMaxN) {
        // Enough rows for every SM to stream about one: a CTA per row.
        pl.row_cta = true;
        pl.per_split = (int)((N + kRowCtaWarps - 1) / kRowCtaWarps);
        return pl;
    }
    if (allow_bulk_split && bulk_split_fits(N)) {
        int nsplit = 1, per = 0;
        bulk_split_for(rows, N, sm_count, &nsplit, &per);
        if (nsplit > 1 && ws_bytes_for(rows, nsplit, D) <= ws_available) {
            pl.team_kernel = true;
            pl.nsplit = nsplit;
            pl.per_split = per;
            pl.ws_bytes = ws_bytes_for(rows, nsplit, D);
            return pl;
        }
    }
    // Enough CTAs to give every SM about ctas_per_sm: with few rows and many
    // states, the loads in flight per SM (and so the stream rate) grow with
    // the CTAs resident on it.
    int64_t want = ((int64_t)ctas_per_sm * sm_count + rows - 1) / (rows > 0 ? rows : 1);
    int nsplit = (int)(want < 1 ? 1 : (want > max_split_for(N) ? max_split_for(N) : want));
    if (nsplit > 1 && ws_bytes_for(rows, nsplit, D) > ws_available) nsplit = 1;
    pl.nsplit = nsplit;
    pl.per_split = (int)((N + nsplit - 1) / nsplit);
    pl.ws_bytes = ws_bytes_for(rows, nsplit, D);
    return pl;
}

template <typename T, int BATCH, int NBUF>
cudaError_t launch_rows_t(const T* v, const float* s, T* vo, float* so, int64_t rows, int N,
                          int64_t H, int chunks, int list_len, const BulkSplit& bs,
                          const DeviceInfo& dev, cudaStream_t st) {
    // The limit is set once per device, to the largest size any call can
    // ask for (rows of up to 128 fp32 values, up to kBulkMaxN states).
    constexpr size_t kMaxSmem = rows_smem_bytes<BATCH, NBUF>(128 * 4, kBulkMaxN);
    const size_t smem = rows_smem_bytes<BATCH, NBUF>(chunks * 16, list_len);
    if (smem > kMaxSmem) return cudaErrorInvalidValue;
    static bool attr_set[64] = {};
    if (dev.device >= 0 && dev.device < 64 && !attr_set[dev.device]) {
        cudaError_t e = cudaFuncSetAttribute(merge_states_bulk_kernel<T, BATCH, NBUF>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kMaxSmem);
        if (e != cudaSuccess) return e;
        attr_set[dev.device] = true;
    }
    const int64_t warps = rows * bs.nsplit;
    const unsigned blocks = (unsigned)((warps + kRowWarps - 1) / kRowWarps);
    merge_states_bulk_kernel<T, BATCH, NBUF><<<blocks, kRowWarps * 32, smem, st>>>(
        v, s, vo, so, rows, N, H, chunks, dev.err, bs);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_rowcta(const T* v, const float* s, T* vo, float* so, int64_t rows, int N,
                          int64_t H, int chunks, int per, size_t smem, const DeviceInfo& dev,
                          cudaStream_t st) {
    // The limit is set once per device, to the largest size any call can ask
    // for (rows of up to 512 bytes, kBulkMaxN states per warp).
    constexpr size_t kMaxSmem = rowcta_smem_bytes(512, kBulkMaxN);
    if (smem > kMaxSmem || kMaxSmem > dev.max_smem_optin) return cudaErrorInvalidValue;
    static bool attr_set[64] = {};
    if (dev.device >= 0 && dev.device < 64 && !attr_set[dev.device]) {
        cudaError_t e = cudaFuncSetAttribute(merge_states_rowcta_kernel<T>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kMaxSmem);
        if (e != cudaSuccess) return e;
        attr_set[dev.device] = true;
    }
    merge_states_rowcta_kernel<T><<<(unsigned)rows, kRowCtaWarps * 32, smem, st>>>(
        v, s, vo, so, N, H, chunks, per, dev.err);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_rows(const T* v, const float* s, T* vo, float* so, int64_t rows, int N, int64_t H,
                        int chunks, const BulkSplit& bs, const DeviceInfo& dev, cudaStream_t st) {
    if (bs.nsplit > 1)
        return launch_rows_t<T, kSplitBatch, kSplitBufs>(v, s, vo, so, rows, N, H, chunks, bs.per, bs,
                                                         dev, st);
    return launch_rows_t<T, kRowBatch, 2>(v, s, vo, so, rows, N, H, chunks, N, bs, dev, st);
}

cudaError_t launch_merge_states(const void* v, const float* s, void* vo, float* so, int64_t S,
                                int64_t N, int64_t H, int64_t D, skv_dtype dt, void* ws,
                                size_t ws_bytes, int ctas_per_sm, bool allow_bulk_split,
                                const DeviceInfo& dev, cudaStream_t st) {
    const int64_t rows = S * H;
    const int chunks = (int)(D * (int64_t)dtype_size(dt) / 16);
    const MergeStatesPlan pl = plan_merge_states(rows, N, D, chunks, dev.sm_count,
                                                 ws ? ws_bytes : 0, ctas_per_sm, allow_bulk_split);
    if (pl.row_cta) {
        const size_t smem = rowcta_smem_bytes(chunks * 16, pl.per_split);
#define SKV_ROWCTA(T_)                                                                        \
    launch_rowcta<T_>(static_cast<const T_*>(v), s, static_cast<T_*>(vo), so, rows, (int)N, H, \
                      chunks, pl.per_split, smem, dev, st)
        switch (dt) {
            case SKV_F32: return SKV_ROWCTA(float);
            case SKV_F16: return SKV_ROWCTA(__half);
            case SKV_BF16: return SKV_ROWCTA(__nv_bfloat16);
        }
#undef SKV_ROWCTA
        return cudaErrorInvalidValue;
    }
    if (pl.team_kernel) {
        BulkSplit bs;
        if (pl.nsplit > 1) {
            bs.nsplit = pl.nsplit;
            bs.per = pl.per_split;
            char* w = static_cast<char*>(ws);
            bs.ws_v = reinterpret_cast<float*>(w);
            w += align256((size_t)rows * pl.nsplit * D * 4);
            bs.ws_s = reinterpret_cast<float*>(w);
            w += align256((size_t)rows * pl.nsplit * 8);
            bs.ws_cnt = reinterpret_cast<unsigned*>(w);
        }
#define SKV_ROWS(T_)                                                                           \
    launch_rows<T_>(static_cast<const T_*>(v), s, static_cast<T_*>(vo), so, rows, (int)N, H,   \
                    chunks, bs, dev, st)
        switch (dt) {
            case SKV_F32: return SKV_ROWS(float);
            case SKV_F16: return SKV_ROWS(__half);
            case SKV_BF16: return SKV_ROWS(__nv_bfloat16);
        }
#undef SKV_ROWS
        return cudaErrorInvalidValue;
    }
    CtaParams p = {};
    p.v = v;
    p.s = s;
    p.vo = vo;
    p.so = so;
    p.H = H;
    p.N = (int)N;
    p.chunks = chunks;
    p.tpr_log2 = chunks >= 32 ? 5 : log2_pow2_at_least(chunks);
    p.nsplit = pl.nsplit;
    p.per_split = pl.per_split;
    if (pl.nsplit > 1) {
        char* w = static_cast<char*>(ws);
        p.ws_v = reinterpret_cast<float*>(w);
        w += align256((size_t)rows * pl.nsplit * D * 4);
        p.ws_s = reinterpret_cast<float*>(w);
        w += align256((size_t)rows * pl.nsplit * 8);
        p.ws_cnt = reinterpret_cast<unsigned*>(w);
    }
    switch (dt) {
        case SKV_F32: return launch_cta<float, float>(p, rows, dev, st, false);
        case SKV_F16: return launch_cta<__half, __half>(p, rows, dev, st, false);
        case SKV_BF16: return launch_cta<__nv_bfloat16, __nv_bfloat16>(p, rows, dev, st, false);
    }
    return cudaErrorInvalidValue;
}

}  // namespace skv
