// cascade.cu -- the shared-prefix pass of two-level cascade decode attention
// on the 5th-generation tensor cores (tcgen05) of sm_103a.
//
// Page: "F2 讲解：merge_state，以 2 为底的 LSE 合并", §⑥: when many requests
// share one prefix, the prefix KV is read once instead of once per request,
// and the queries that share it form a dense matrix product that can run on
// tensor cores; the prefix state is then merged with each request's own
// suffix state.  The suffix runs through the split-KV decode
// ("L3 讲解：split-KV decode 与 LSE 合并") and the merges through the combine
// kernel of decode.cu.
//
// One CTA per (kv head, 128-row M tile, chunk of the prefix).  The M tile's
// rows are (request, group head) pairs -- row = r_local * G + g -- so one KV
// tile serves 128 query rows.  Per 128-key block j:
//   S_j = Q K_j^T    tcgen05.mma kind::f16, Q [128 x 128] and the K block
//                    [128 keys x 128] K-major in shared memory; S fp32 in one
//                    of two TMEM buffers, so S_{j+1} runs on the tensor core
//                    while the warps do the softmax of block j
//   softmax          4 warps, thread i <-> row i <-> TMEM lane i: base-2
//                    online max/sum ([F2] §② exp2 trick); P written to shared
//                    memory as fp16 in the swizzled K-major operand layout
//   O += P_j V_j     tcgen05.mma with V as an MN-major operand, O fp32 stays
//                    in TMEM across blocks
// Lazy rescale: a row keeps the max it last rescaled to and only rescales
// O (in TMEM) and its sum when the block max exceeds it by more than 8 (log2
// units), so p <= 2^8 (exact in fp16 range) and the final normalisation by
// the same max keeps the result exact.
// Warp roles: warps 0-3 softmax and epilogue, warp 4 issues the MMAs, warp
// 5 issues the TMA copies; they meet on mbarriers (S full / free per S
// buffer, P full, PV done, K and V stage full / empty), so no role waits on
// another's serial work.  Q, K and V tiles arrive by TMA tensor loads with
// the 128-byte swizzle (a page is one 16 x 64 box per half of the head dim);
// two K and two V blocks are in flight.  Every wait is bounded; a wait that
// gives up raises a shared abort flag that ends every role's loop.  Each
// chunk writes its normalised state (o, s base 2) for the combine kernel,
// which merges the chunks into the prefix state.
#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"
#include "tma.h"

namespace skv {
namespace {

constexpr int kD = 128;
constexpr int kPage = 16;
constexpr int kBlockKeys = 128;                      // keys per block (N of QK^T, K of PV)
constexpr int kPagesPerBlock = kBlockKeys / kPage;   // 8
constexpr int kM = 128;                              // query rows per CTA
constexpr int kHalf = 128 * 128;                     // one [128 rows x 64] fp16 swizzled half tile
constexpr int kTile = 2 * kHalf;                     // one [128 x 128] fp16 operand tile (32 KB)
constexpr int kStages = 2;                           // K blocks and V blocks in flight
constexpr int kSoftmaxWarps = 4;                     // one thread per query row
constexpr int kMmaWarp = 8;
constexpr int kTmaWarp = 9;
constexpr int kThreads = 10 * 32;
constexpr uint32_t kTmemCols = 512;                  // S_w at 128 w, O_w at 256 + 128 w (w = softmax group)
constexpr float kRescaleThreshold = 8.f;             // log2 units

struct PrefixParams {
    const int32_t* prefix_pages;
    int32_t prefix_len;
    int32_t pool_rows;        // rows of the K/V tensor maps: num_pool_pages * Hkv * page
    int32_t num_pool_pages;
    int32_t B, Hq, Hkv, G;
    int32_t blocks_per_chunk, nchunks;
    float scale_log2;
    float* pre_part;          // [B*Hq, nchunks, D] split-normalised chunk states
    float* pre_lse;           // [B*Hq, nchunks] base 2
    unsigned long long* err;
};

constexpr size_t kSmemQ = 0;
constexpr size_t kSmemK = kSmemQ + kTile;
constexpr size_t kSmemV = kSmemK + (size_t)kStages * kTile;
constexpr size_t kSmemP = kSmemV + (size_t)kStages * kTile;
constexpr size_t kSmemBars = kSmemP + 2 * kTile;     // a P buffer per softmax group
// q_full, p_full[2], pv_done[2], s_full[2], s_free[2], merge, k_full[], k_empty[], v_full[], v_empty[]
constexpr int kNumBars = 10 + 4 * kStages;
constexpr size_t kSmemMl = kSmemBars + kNumBars * sizeof(uint64_t);  // group 1's (m, l) per row
constexpr size_t kSmemTmemSlot = kSmemMl + kM * 2 * sizeof(float);
constexpr size_t kSmemEnd = kSmemTmemSlot + 16;      // tmem address, abort flag

size_t prefix_smem_bytes(int) { return 1024 + kSmemEnd; }

__global__ void __launch_bounds__(kThreads, 1)
cascade_prefix_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                      const __grid_constant__ CUtensorMap tv, const PrefixParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    uint8_t* Qs = sm + kSmemQ;
    uint8_t* Ks = sm + kSmemK;
    uint8_t* Vs = sm + kSmemV;
    uint8_t* Ps = sm + kSmemP;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kSmemBars);
    uint64_t* q_full = bars + 0;
    uint64_t* p_full = bars + 1;   // [2], per softmax group
    uint64_t* pv_done = bars + 3;  // [2]
    uint64_t* s_full = bars + 5;   // [2]
    uint64_t* s_free = bars + 7;   // [2]
    uint64_t* merge_bar = bars + 9;
    uint64_t* k_full = bars + 10;
    uint64_t* k_empty = k_full + kStages;
    uint64_t* v_full = k_empty + kStages;
    uint64_t* v_empty = v_full + kStages;
    float* ml = reinterpret_cast<float*>(sm + kSmemMl);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + kSmemTmemSlot);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + kSmemTmemSlot + 4);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int chunk = blockIdx.x, mtile = blockIdx.y, hkv = blockIdx.z;
    const int nblocks_total = (p.prefix_len + kBlockKeys - 1) / kBlockKeys;
    const int blk0 = chunk * p.blocks_per_chunk;
    const int nb = min(p.blocks_per_chunk, nblocks_total - blk0);  // >= 1 (host sizing)
    const int npages_prefix = (p.prefix_len + kPage - 1) / kPage;

    if (tid == 0) {
        mbar_init(q_full, 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(&p_full[b], kSoftmaxWarps);
            mbar_init(&pv_done[b], 1);
            mbar_init(&s_full[b], 1);
            mbar_init(&s_free[b], kSoftmaxWarps);
        }
        mbar_init(merge_bar, kSoftmaxWarps);
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&k_full[i], 1);
            mbar_init(&k_empty[i], 1);
            mbar_init(&v_full[i], 1);
            mbar_init(&v_empty[i], 1);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0) tc::tmem_alloc(tmem_slot, kTmemCols);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    if (warp == kTmaWarp) {
        // ---------------------------------------------------------------- TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&tq);
            tma_prefetch_desc(&tk);
            tma_prefetch_desc(&tv);
        }
        const uint64_t pol = policy_evict_first();
        int win = -1, wid = -1;  // page-id window of the prefix list, id of page 32 * win + lane
        // A block's 16 boxes (8 pages x 2 halves of the head dim) go out from
        // 16 lanes at once: copies issued one after another by one thread
        // stream at about half the HBM bandwidth.
        auto load_block = [&](int j, bool is_v) {
            const int stage = j % kStages;
            uint64_t* bar = is_v ? &v_full[stage] : &k_full[stage];
            uint8_t* dst = (is_v ? Vs : Ks) + stage * kTile;
            const CUtensorMap* map = is_v ? &tv : &tk;
            if (lane == 0) mbar_arrive_expect_tx(bar, kTile);
            __syncwarp();
            const int pg = lane >> 1, h = lane & 1;
            // The block's 8 pages lie in one 32-page window of the prefix
            // page list, held one id per lane (reloaded every 4 blocks).
            const int g0 = (blk0 + j) * kPagesPerBlock;
            if ((g0 >> 5) != win) {
                win = g0 >> 5;
                const int gl = 32 * win + lane;
                wid = -1;  // past the prefix: loaded as zeros
                if (gl < npages_prefix) {
                    wid = __ldg(p.prefix_pages + gl);
                    if ((unsigned)wid >= (unsigned)p.num_pool_pages) {
                        record_error(p.err, SKV_ERR_INVALID_ARG, 2 << 20 | gl);
                        wid = 0;
                    }
                }
            }
            const int pid = __shfl_sync(0xffffffffu, wid, (g0 + (pg & 7)) & 31);
            if (pg < kPagesPerBlock) {
                // A page past the prefix is read from the row just past the
                // tensor: the TMA fills the whole box with zeros.
                const int row = pid >= 0 ? (pid * p.Hkv + hkv) * kPage : p.pool_rows;
                tma_load_2d(dst + h * kHalf + pg * (kPage * 128), map, h * 64, row, bar, pol);
            }
        };
        if (lane == 0) {
            mbar_arrive_expect_tx(q_full, kTile);
            const int z = mtile * (kM / p.G);
            tma_load_3d(Qs, &tq, 0, hkv * p.G, z, q_full);
            tma_load_3d(Qs + kHalf, &tq, 64, hkv * p.G, z, q_full);
        }
        for (int j = 0; j < nb; ++j) {
            bool ok = true;
            if (j >= kStages)
                ok = wait_or_abort(&k_empty[j % kStages], (uint32_t)((j / kStages - 1) & 1), abort_flag,
                                   p.err, 20);
            if (!__all_sync(0xffffffffu, ok)) break;
            load_block(j, false);
            if (j >= kStages)
                ok = wait_or_abort(&v_empty[j % kStages], (uint32_t)((j / kStages - 1) & 1), abort_flag,
                                   p.err, 21);
            if (!__all_sync(0xffffffffu, ok)) break;
            load_block(j, true);
        }
    } else if (warp == kMmaWarp) {
        // ---------------------------------------------------------------- MMA issuer
        // Block j belongs to softmax group w = j & 1: S_w = Q K_j^T, then
        // O_w += P_j V_j once the group has written P_j.
        if (lane == 0) {
            constexpr uint32_t idS = tc::idesc_f16_f32(kM, kBlockKeys, false);
            constexpr uint32_t idPV = tc::idesc_f16_f32(kM, kD, true);
            auto issue_pv = [&](int j) -> bool {  // O_w += P_j V_j
                const int st = j % kStages, w = j & 1;
                if (!wait_or_abort(&p_full[w], (uint32_t)((j >> 1) & 1), abort_flag, p.err, 22)) return false;
                if (!wait_or_abort(&v_full[st], (uint32_t)((j / kStages) & 1), abort_flag, p.err, 23))
                    return false;
                tc::fence_after_sync();
                const int tail = p.prefix_len % kPage;
                const int last_page = npages_prefix - 1 - (blk0 + j) * kPagesPerBlock;
                if (tail != 0 && last_page >= 0 && last_page < kPagesPerBlock) {
                    // The prefix ends inside this block's page `last_page`:
                    // its rows past the end hold whatever the pool has there.
                    // P is 0 for them, but 0 times a non-finite value is not
                    // 0, so the rows are zeroed (whole 128-byte rows: the
                    // swizzle only permutes chunks inside a row).
                    for (int t = tail; t < kPage; ++t)
                        for (int h = 0; h < 2; ++h) {
                            uint4* row = reinterpret_cast<uint4*>(Vs + st * kTile + h * kHalf +
                                                                  (last_page * kPage + t) * 128);
                            for (int c = 0; c < 8; ++c) row[c] = make_uint4(0, 0, 0, 0);
                        }
                    tc::fence_proxy_async_smem();
                }
                const uint32_t tOw = tmem + 256 + 128 * w;
                const uint8_t* Pw = Ps + w * kTile;
#pragma unroll
                for (int k = 0; k < kBlockKeys / 16; ++k) {
                    const int h = k >> 2, kk = k & 3;
                    const uint64_t ad = tc::sdesc_sw128(smem_addr(Pw + h * kHalf) + kk * 32, 16, 1024);
                    const uint64_t bd = tc::sdesc_sw128(smem_addr(Vs + st * kTile) + k * 2048, kHalf, 1024);
                    tc::mma_f16_ss(tOw, ad, bd, idPV, j >= 2 || k > 0);
                }
                tc::mma_commit(&pv_done[w]);
                tc::mma_commit(&v_empty[st]);
                return true;
            };
            bool ok = wait_or_abort(q_full, 0, abort_flag, p.err, 24);
            for (int j = 0; ok && j < nb; ++j) {
                // S_j into group (j & 1)'s buffer, then P_{j-1} V_{j-1}: the
                // tensor core computes S_j while the softmax of block j-1 runs.
                const int st = j % kStages, w = j & 1;
                ok = wait_or_abort(&k_full[st], (uint32_t)((j / kStages) & 1), abort_flag, p.err, 25);
                if (ok && j >= 2)
                    ok = wait_or_abort(&s_free[w], (uint32_t)(((j >> 1) - 1) & 1), abort_flag, p.err, 26);
                if (!ok) break;
                tc::fence_after_sync();
                const uint32_t tS = tmem + (uint32_t)w * 128;
#pragma unroll
                for (int k = 0; k < kD / 16; ++k) {
                    const int h = k >> 2, kk = k & 3;
                    const uint64_t ad = tc::sdesc_sw128(smem_addr(Qs + h * kHalf) + kk * 32, 16, 1024);
                    const uint64_t bd = tc::sdesc_sw128(smem_addr(Ks + st * kTile + h * kHalf) + kk * 32, 16, 1024);
                    tc::mma_f16_ss(tS, ad, bd, idS, k > 0);
                }
                tc::mma_commit(&s_full[w]);
                tc::mma_commit(&k_empty[st]);
                if (j >= 1) ok = issue_pv(j - 1);
            }
            if (ok) issue_pv(nb - 1);
        }
    } else {
        // ---------------------------------------------------------------- softmax, row = tid % 128
        // Group w (warps 4w .. 4w + 3) takes blocks w, w + 2, ... with its
        // own S, O and P; the two partial states of a row are merged at the
        // end, like two splits of the chunk.
        const int w = warp >> 2, row_t = tid & (kM - 1);
        const uint32_t tOw = tmem + 256 + 128 * w;
        uint8_t* Pw = Ps + w * kTile;
        float m_ref = -INFINITY;  // the max this row's O and l are scaled to (log2 units)
        float l_run = 0.f;
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        bool ok = true;
        int jl = -1;  // this group's last block
        for (int j = w; j < nb; j += 2) {
            jl = j;
            ok = wait_or_abort(&s_full[w], (uint32_t)((j >> 1) & 1), abort_flag, p.err, 27);
            if (!__all_sync(0xffffffffu, ok)) {
                ok = false;
                break;
            }
            tc::fence_after_sync();
            float x[kBlockKeys];
            tc::tmem_ld128(tmem + (uint32_t)w * 128 + lane_base, x);
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&s_free[w]);  // S buffer read by this warp
            // Row max in log2 units.  With a positive scale the max of the
            // raw scores is taken and scaled once, and the scale is folded
            // into the exponent below (p = 2^(x * sc - m)); only the block
            // that crosses the end of the prefix is masked.
            const int key0 = (blk0 + j) * kBlockKeys;
            float sc = p.scale_log2, mx;
            if (sc > 0.f) {
                if (key0 + kBlockKeys > p.prefix_len) {
#pragma unroll
                    for (int i = 0; i < kBlockKeys; ++i)
                        if (key0 + i >= p.prefix_len) x[i] = -INFINITY;
                }
                float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                for (int i = 0; i < kBlockKeys; ++i) m4[i & 3] = fmaxf(m4[i & 3], x[i]);
                mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) * sc;
            } else {
                mx = -INFINITY;
#pragma unroll
                for (int i = 0; i < kBlockKeys; ++i) {
                    x[i] = key0 + i < p.prefix_len ? x[i] * sc : -INFINITY;
                    mx = fmaxf(mx, x[i]);
                }
                sc = 1.f;
            }
            // PV of this group's previous block done: O_w is stable and P_w free.
            if (j >= 2) {
                ok = wait_or_abort(&pv_done[w], (uint32_t)(((j - 2) >> 1) & 1), abort_flag, p.err, 28);
                if (!__all_sync(0xffffffffu, ok)) {
                    ok = false;
                    break;
                }
                tc::fence_after_sync();
            }
            if (mx > m_ref + kRescaleThreshold) {  // also the first block (m_ref = -inf)
                if (j >= 2) {
                    const float alpha = exp2f(m_ref - mx);
                    l_run *= alpha;
#pragma unroll 1
                    for (int c = 0; c < kD / 32; ++c) {  // 32 columns at a time: x[] stays live
                        float ob[32];
                        tc::tmem_ld32(tOw + lane_base + 32 * c, ob);
#pragma unroll
                        for (int i = 0; i < 32; ++i) ob[i] *= alpha;
                        tc::tmem_st32(tOw + lane_base + 32 * c, ob);
                    }
                }
                m_ref = mx;
            }
            float ps4[4] = {0.f, 0.f, 0.f, 0.f};  // independent partial sums
            const float nm = -m_ref;
#pragma unroll
            for (int chunk16 = 0; chunk16 < 16; ++chunk16) {  // 8 keys = one 16-byte chunk of P
                uint32_t pk[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int i0 = chunk16 * 8 + 2 * e;
                    const float p0 = fast_exp2(fmaf(x[i0], sc, nm));  // masked keys: 2^-inf = 0
                    const float p1 = fast_exp2(fmaf(x[i0 + 1], sc, nm));
                    ps4[e] += p0 + p1;
                    const __half2 h2 = __floats2half2_rn(p0, p1);
                    pk[e] = *reinterpret_cast<const uint32_t*>(&h2);
                }
                const int half = chunk16 >> 3;
                const int pos = (chunk16 & 7) ^ (row_t & 7);  // 128-byte swizzle
                *reinterpret_cast<uint4*>(Pw + half * kHalf + row_t * 128 + pos * 16) =
                    make_uint4(pk[0], pk[1], pk[2], pk[3]);
            }
            l_run += (ps4[0] + ps4[1]) + (ps4[2] + ps4[3]);
            tc::fence_before_sync();
            tc::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&p_full[w]);  // P_j (and any O rescale) done by this warp
        }
        // ---- this group's state of row row_t, after its last PV
        if (ok && jl >= 0) ok = wait_or_abort(&pv_done[w], (uint32_t)((jl >> 1) & 1), abort_flag, p.err, 29);
        ok = __all_sync(0xffffffffu, ok);
        if (w == 1) {  // hand (m, l) to group 0 (l = 0: no block, O_1 unused)
            ml[2 * row_t] = ok ? m_ref : -INFINITY;
            ml[2 * row_t + 1] = ok ? l_run : 0.f;
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(merge_bar);
        } else {
            ok = __all_sync(0xffffffffu, ok && wait_or_abort(merge_bar, 0, abort_flag, p.err, 30));
            if (ok) {
                tc::fence_after_sync();
                const float m1 = ml[2 * row_t], l1 = ml[2 * row_t + 1];
                // Two-state merge of the groups' states ([F2] §③): weights
                // relative to the larger max; an empty state weighs 0.
                const float M = fmaxf(m_ref, m1);
                const float a0 = l_run > 0.f ? exp2f(m_ref - M) : 0.f;
                const float a1 = l1 > 0.f ? exp2f(m1 - M) : 0.f;
                const float L = a0 * l_run + a1 * l1;
                const float inv = L > 0.f ? 1.f / L : 0.f;
                const float c0 = a0 * inv, c1 = a1 * inv;
                const int rows_per_req = p.G;
                const int r = mtile * (kM / rows_per_req) + row_t / rows_per_req;
                const int g = row_t % rows_per_req;
                const int64_t row = (int64_t)r * p.Hq + hkv * p.G + g;
                float* dst = p.pre_part + (row * p.nchunks + chunk) * kD;
#pragma unroll 1
                for (int c = 0; c < kD / 32; ++c) {
                    float o0[32], o1[32];
                    tc::tmem_ld32(tmem + 256 + lane_base + 32 * c, o0);
                    if (l1 > 0.f) {
                        tc::tmem_ld32(tmem + 384 + lane_base + 32 * c, o1);
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i) o1[i] = 0.f;
                    }
                    if (r < p.B) {
#pragma unroll
                        for (int i = 0; i < 32; i += 4)
                            *reinterpret_cast<float4*>(dst + 32 * c + i) = make_float4(
                                c0 * o0[i] + c1 * o1[i], c0 * o0[i + 1] + c1 * o1[i + 1],
                                c0 * o0[i + 2] + c1 * o1[i + 2], c0 * o0[i + 3] + c1 * o1[i + 3]);
                    }
                }
                if (r < p.B) p.pre_lse[row * p.nchunks + chunk] = L > 0.f ? M + log2f(L) : -INFINITY;
            }
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc::fence_after_sync();
        tc::tmem_free(tmem, kTmemCols);
    }
}

}  // namespace

void cascade_prefix_geometry(int B, int G, int Hkv, int prefix_len, int sm_count, int* mtiles,
                             int* blocks_per_chunk, int* nchunks) {
    const int nblocks = (prefix_len + kBlockKeys - 1) / kBlockKeys;
    const int mt = (B * G + kM - 1) / kM;
    // About one CTA per SM: chunks = SMs / (Hkv * M tiles), at least one block each.
    int want = sm_count / (Hkv * mt > 0 ? Hkv * mt : 1);
    if (want < 1) want = 1;
    if (want > nblocks) want = nblocks;
    int bpc = nblocks > 0 ? (nblocks + want - 1) / want : 1;
    *mtiles = mt;
    *blocks_per_chunk = bpc;
    *nchunks = nblocks > 0 ? (nblocks + bpc - 1) / bpc : 0;
}

cudaError_t launch_cascade_prefix(const CascadeArgs& a, const DeviceInfo& dev, float* pre_part,
                                  float* pre_lse, int nchunks, int blocks_per_chunk, int mtiles,
                                  cudaStream_t st) {
    const int G = a.Hq / a.Hkv;
    CUtensorMap tq, tk, tv;
    cudaError_t e = make_tmap_3d_16bit(&tq, a.q, kD, a.Hq, a.B, (uint64_t)kD * 2,
                                       (uint64_t)a.Hq * kD * 2, 64, G, kM / G, true);
    if (e != cudaSuccess) return e;
    const uint64_t rows = (uint64_t)a.num_pool_pages * a.Hkv * kPage;
    if ((e = make_tmap_2d_16bit(&tk, a.k_cache, rows, kD, kD * 2, 64, kPage, true, false)) != cudaSuccess)
        return e;
    if ((e = make_tmap_2d_16bit(&tv, a.v_cache, rows, kD, kD * 2, 64, kPage, true, false)) != cudaSuccess)
        return e;
    PrefixParams p;
    p.prefix_pages = a.prefix_pages;
    p.prefix_len = a.prefix_len;
    p.pool_rows = (int32_t)rows;
    p.num_pool_pages = a.num_pool_pages;
    p.B = a.B;
    p.Hq = a.Hq;
    p.Hkv = a.Hkv;
    p.G = G;
    p.blocks_per_chunk = blocks_per_chunk;
    p.nchunks = nchunks;
    p.scale_log2 = a.sm_scale * 1.4426950408889634f;
    p.pre_part = pre_part;
    p.pre_lse = pre_lse;
    p.err = dev.err;
    const size_t smem = prefix_smem_bytes(blocks_per_chunk);
    if (smem > dev.max_smem_optin) return cudaErrorInvalidValue;
    e = cudaFuncSetAttribute(cascade_prefix_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
    if (e != cudaSuccess) return e;
    cascade_prefix_kernel<<<dim3(nchunks, mtiles, a.Hkv), kThreads, smem, st>>>(tq, tk, tv, p);
    return cudaGetLastError();
}

}  // namespace skv
