// decode_tc.cu -- split-KV paged decode attention, pass 1 (the per-split
// states), on the 5th-generation tensor cores (tcgen05) of sm_103a.
//
// Page: "L3 讲解：split-KV decode 与 LSE 合并" -- §① the two-pass scheme: a
// (request, kv head, split) work unit walks its own pages and writes that
// split's state; §② the page ranges; §③ the state o_s = acc / l, s = m2 +
// log2 l (base 2, [F2] §②); §④ an empty split is o = 0, s = -inf; §⑤ fp32
// partials.  Pass 2 (the merge of the NS states) is the combine kernel of
// decode.cu.
//
// Why tensor cores in a bandwidth-bound pass: the G = Hq / Hkv query heads of
// a KV head read the same K and V, so a work unit is the dense contraction
// S = q_G K^T, O = P V with q_G of G rows.  On CUDA cores its FMAs and the
// shared-memory reads that feed them take most of the issue slots, and the
// pass stops at the instruction issue rate instead of at HBM.  On tcgen05 the
// math costs 16 MMA instructions per 128 keys.
//
// Tile.  One tile is up to 8 pages (M = 128 keys) of K and V in shared
// memory, and N = 16 columns: column c belongs to unit slot c / G, head
// c % G.  Work units with at most 8 pages are packed into one tile, up to
// 16 / G of them: each slot brings its own q rows (the B operand), and a
// key row only counts in the columns of its own slot, so one set of MMAs
// serves several short splits.  A unit with more than 8 pages is a group of
// chunk tiles that accumulate into the same O; a packed tile is a group of
// its own.
//   S^T = K Q^T      M = 128 keys, N = 16, K = 128 dims (K-major operands)
//   softmax          thread i <-> key row i <-> TMEM lane i: column max per
//                    slot (per page over 16 lanes, then over the slot's
//                    pages), p = 2^(s - m); p as fp16 into P^T (K-major
//                    16 x 128), the fp32 p summed per thread; rows past ctx
//                    get p = 0
//   O^T += V^T P^T   M = 128 dims (V as an MN-major A operand), N = 16
// Lazy rescale: a chunk group keeps its reference max until a tile's max
// exceeds it by more than 8 (log2 units), then rescales O in TMEM and the
// sums; p <= 2^8 stays in range for fp16.
//
// Persistent CTAs (one per SM): CTA c takes units c, c + grid, ...  Fourteen
// warps:
//   0-3   softmax (one thread per key row)
//   4-7   epilogue: per group, o = O / L (thread i <-> dim i <-> TMEM lane i)
//         and s = m + log2 L, written to the split states
//   8     issues the S MMAs, 9 issues the PV MMAs
//   10-13 producers: all four walk the same deterministic packing of this
//         CTA's units into tiles; warps 10 and 11 load the K halves, q rows
//         and descriptors of the even and odd tiles, warps 12 and 13 their V
//         halves (q rows by cp.async, K and V as 16 x 64 boxes with the
//         128-byte swizzle, one box per lane)
// Copies, MMAs and TMEM loads issued one after another by a single thread
// cannot keep up with HBM, so each of these jobs has its own warp.  Three
// tile stages are in flight, each with its K (and q) half and its V half
// freed separately: K as soon as S is computed, V once PV is done, so the
// next K lands while this tile's softmax runs.  Every wait is bounded; a
// wait that gives up
// raises a shared abort flag that ends every role's loop, and each role
// waits (bounded) for its own copies or MMAs before the CTA frees its
// tensor memory.
#include "common.cuh"
#include "kernels.h"
#include "split_range.h"
#include "tc.cuh"
#include "tma.h"

namespace skv {
namespace {

constexpr int kD = 128;
constexpr int kPage = 16;
constexpr int kTilePages = 8;
constexpr int kM = kTilePages * kPage;           // 128 keys per tile
constexpr int kN = 16;                           // columns: slot * G + head
constexpr int kKVHalf = kM * 128;                // [128 rows x 64] fp16 swizzled: 16 KB
constexpr int kKVTile = 2 * kKVHalf;             // 32 KB
constexpr int kQHalf = kN * 128;                 // [16 rows x 64]: 2 KB
constexpr int kQTile = 2 * kQHalf;               // 4 KB
constexpr int kStageBytes = 2 * kKVTile + kQTile;  // K, V, Q^T
constexpr int kStages = 3;
constexpr int kDescs = 2 * kStages;              // a descriptor lives until its PV is issued
constexpr int kPHalf = kN * 128;                 // P^T [16 x 64 keys]: 2 KB
constexpr int kPTile = 2 * kPHalf;
constexpr int kPageBytes = 4 * kPage * 128;      // K and V of one page: 8 KB
constexpr int kSoftmaxWarps = 4;
constexpr int kEpiWarp0 = 4;
constexpr int kQkWarp = 8;
constexpr int kPvWarp = 9;
constexpr int kProdWarp0 = 10;                    // 10, 11: K + q; 12, 13: V
constexpr int kProdWarps = 4;
constexpr int kThreads = 14 * 32;
constexpr uint32_t kTmemCols = 64;  // S [0,16) [16,32); O [32,48) [48,64)
constexpr float kRescaleThreshold = 8.f;
constexpr unsigned kFull = 0xffffffffu;

enum : int16_t { kTileWork = 0, kTileEnd = 1 };
enum : int16_t { kFirst = 1, kLast = 2, kChunk = 4 };

// What the producers tell the other roles about one tile.
struct __align__(16) TileDesc {
    int32_t unit[kN];           // work unit of each slot
    int32_t slot_p0[kN];        // first page (index in the request's table) of the slot in this tile
    int32_t qrow[kN];           // q row of the slot's head 0: b * Hq + hkv * G
    int8_t slot_first[kN];      // first page of the slot inside the tile
    int8_t slot_pages[kN];      // pages of the slot inside the tile
    int8_t page_slot[kTilePages];
    int8_t page_valid[kTilePages];  // keys of the page before ctx (1..16)
    int16_t kind, npages, nunits, flags;
    int16_t slot_split[kN];     // split index of the slot's unit
    int32_t partial_mask;       // bit k: page k ends before its 16th key
    int32_t pad;
};
static_assert(sizeof(TileDesc) == 288, "descriptor size");

// What the softmax hands the epilogue at the end of a group.
struct __align__(16) GroupInfo {
    int32_t qrow[kN];                  // q row of the slot's head 0, -1 if the slot is unused
    int32_t split[kN];                 // split index of the slot's unit
    float m[kN];                       // reference max of each column
    float lpage[kTilePages][kN];       // per-page partial column sums
    int32_t nunits;                    // -1: no more groups
    int32_t has_o;                     // O holds this group's product
    int32_t pad[2];
};

struct TcParams {
    const uint16_t* q;  // fp16 or bf16 bit patterns
    const int32_t* block_table;
    const int32_t* ctx;
    float* o_part;
    float* lse_part;
    int32_t* ranges_dbg;
    unsigned long long* err;
    unsigned int* done_ctr;  // cascade chaining (DecodeArgs::done_ctr) or nullptr
    int32_t num_pool_pages, max_pages, B, Hq, Hkv, NS;
    int32_t units;  // B * Hkv * NS; unit u = ((b * NS) + split) * Hkv + hkv
    float scale_log2;
};

constexpr size_t kSmStages = 0;
constexpr size_t kSmP = kSmStages + (size_t)kStages * kStageBytes;
constexpr size_t kSmDesc = kSmP + 2 * kPTile;
constexpr size_t kSmScratch = kSmDesc + kDescs * sizeof(TileDesc);       // one per producer
constexpr size_t kSmInfo = kSmScratch + kProdWarps * sizeof(TileDesc);
constexpr size_t kSmRed = kSmInfo + 2 * sizeof(GroupInfo);              // [2][8 pages][8] floats
constexpr size_t kSmBars = kSmRed + 2 * kTilePages * 8 * sizeof(float);
// k_full[3], v_full[3], k_empty[3], v_empty[3], desc_full[6], desc_free[6],
// s_full[2], s_free[2], p_full[2], pv_done[2], o_full[2], o_free[2],
// epi_ready[2], red, mma_done[2]
constexpr int kNumBars = 4 * kStages + 2 * kDescs + 17;
constexpr size_t kSmMisc = kSmBars + kNumBars * sizeof(uint64_t);  // tmem address, abort flag
constexpr size_t kSmemBytes = 1024 + kSmMisc + 16;

SKV_DEVINL void decode_unit(const TcParams& p, int u, int* b, int* hkv, int* split) {
    *hkv = u % p.Hkv;
    const int r = u / p.Hkv;
    *split = r % p.NS;
    *b = r / p.NS;
}

template <int G, bool BF>
__global__ void __launch_bounds__(kThreads, 1)
splitkv_decode_tc_kernel(const __grid_constant__ CUtensorMap tk,
                         const __grid_constant__ CUtensorMap tv, const TcParams p) {
    constexpr int kSlots = kN / G;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    uint8_t* stages = sm + kSmStages;
    uint8_t* Ps = sm + kSmP;
    TileDesc* descs = reinterpret_cast<TileDesc*>(sm + kSmDesc);
    GroupInfo* info = reinterpret_cast<GroupInfo*>(sm + kSmInfo);
    float* redbuf = reinterpret_cast<float*>(sm + kSmRed);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kSmBars);
    uint64_t* k_full = bars;
    uint64_t* v_full = bars + kStages;
    uint64_t* k_empty = bars + 2 * kStages;
    uint64_t* v_empty = bars + 3 * kStages;
    // A tile's descriptor is published on its slot's barrier: the K barrier of
    // a stage can run a phase ahead of the softmax and PV roles (K is freed
    // early), a descriptor slot cannot (it is reused only after the PV of its
    // previous tile has been issued).
    uint64_t* desc_full = bars + 4 * kStages;
    uint64_t* desc_free = desc_full + kDescs;  // the PV issuer is done with the slot's descriptor
    uint64_t* s_full = desc_free + kDescs;
    uint64_t* s_free = s_full + 2;
    uint64_t* p_full = s_free + 2;
    uint64_t* pv_done = p_full + 2;
    uint64_t* o_full = pv_done + 2;
    uint64_t* o_free = o_full + 2;
    uint64_t* epi_ready = o_free + 2;
    uint64_t* red_bar = epi_ready + 2;
    uint64_t* mma_done = red_bar + 1;  // [2]: S issuer, PV issuer
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + kSmMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + kSmMisc + 4);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    // The combine grid may be scheduled now; it waits for this grid to finish.
    pdl_launch_dependents();

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&k_full[s], 1);
            mbar_init(&v_full[s], 1);
            mbar_init(&k_empty[s], 1);
            mbar_init(&v_empty[s], 1);
        }
        for (int i = 0; i < kDescs; ++i) {
            mbar_init(&desc_full[i], 1);
            mbar_init(&desc_free[i], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&s_full[b], 1);
            mbar_init(&s_free[b], kSoftmaxWarps);
            mbar_init(&p_full[b], kSoftmaxWarps);
            mbar_init(&pv_done[b], 1);
            mbar_init(&o_full[b], 1);
            mbar_init(&o_free[b], 4);
            mbar_init(&epi_ready[b], kSoftmaxWarps);
            mbar_init(&mma_done[b], 1);
        }
        mbar_init(red_bar, kSoftmaxWarps);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0) tc::tmem_alloc(tmem_slot, kTmemCols);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    if (warp >= kProdWarp0) {
        // ------------------------------------------------------------ producers
        const int pw = warp - kProdWarp0;
        const int par = pw & 1;        // this warp's tiles: tile & 1 == par
        const bool kprod = pw < 2;     // K half, q rows and descriptor; else the V half
        TileDesc* scratch = reinterpret_cast<TileDesc*>(sm + kSmScratch) + pw;
        if (lane == 0) {
            tma_prefetch_desc(&tk);
            tma_prefetch_desc(&tv);
        }
        const uint64_t pol = policy_evict_first();
        const int cap = p.max_pages * kPage;
        auto tma_row = [&](int pid, int hkv, int b) {  // first row of a (page, kv head) tile
            if ((unsigned)pid >= (unsigned)p.num_pool_pages) {
                record_error(p.err, SKV_ERR_INVALID_ARG, 1 << 20 | b);
                pid = 0;
            }
            return (pid * p.Hkv + hkv) * kPage;
        };
        // Lane l holds unit kb + l of this CTA's list (u = blockIdx.x + k *
        // gridDim.x) and, for a unit of at most 8 pages, the TMA rows of its
        // pages: one round of loads serves 32 units.
        int kb = 0, bu = -1, bb = 0, bhkv = 0, bsplit = 0, bp0 = 0, bnp = 0, bctx = 0;
        int brow[kTilePages];
        auto load_batch = [&]() {
            const long long uu = (long long)blockIdx.x + (long long)(kb + lane) * gridDim.x;
            bu = -1;
            bnp = 0;
            if (uu < p.units) {
                bu = (int)uu;
                decode_unit(p, bu, &bb, &bhkv, &bsplit);
                const int split = bsplit;
                int c = p.ctx[bb];
                if (c < 0 || c > cap) {
                    if (split == 0 && bhkv == 0) record_error(p.err, SKV_ERR_INVALID_ARG, bb);
                    c = c < 0 ? 0 : cap;
                }
                int p0, p1;
                split_page_range(c, kPage, p.NS, split, &p0, &p1);
                if (p.ranges_dbg != nullptr && bhkv == 0 && pw == 0) {
                    p.ranges_dbg[((int64_t)bb * p.NS + split) * 2 + 0] = p0;
                    p.ranges_dbg[((int64_t)bb * p.NS + split) * 2 + 1] = p1;
                }
                bp0 = p0;
                bnp = p1 > p0 ? p1 - p0 : 0;
                bctx = c;
            }
            int pid[kTilePages];
            const int32_t* bt = p.block_table + (int64_t)bb * p.max_pages + bp0;
#pragma unroll
            for (int k = 0; k < kTilePages; ++k) pid[k] = (bnp <= kTilePages && k < bnp) ? bt[k] : 0;
#pragma unroll
            for (int k = 0; k < kTilePages; ++k)
                brow[k] = (bnp <= kTilePages && k < bnp) ? tma_row(pid[k], bhkv, bb) : 0;
        };
        // A long unit's TMA rows, 32 pages at a time (lane l: page lbase + l).
        int lu = -1, lb = 0, lhkv = 0, lsplit = 0, lp0 = 0, lnp = 0, lctx = 0, lnext = 0, lbase = 0,
            lrow = 0;
        auto load_long = [&](int from) {
            lbase = from;
            lrow = 0;
            if (from + lane < lnp)
                lrow = tma_row(p.block_table[(int64_t)lb * p.max_pages + lp0 + from + lane], lhkv, lb);
        };
        load_batch();
        int ki = 0;  // next unit of the batch
        int last_fill[kStages] = {-1, -1, -1}, last_vfill[kStages] = {-1, -1, -1};
        bool ok = true;
        for (int tile = 0; ok; ++tile) {
            // ---- the tile's descriptor (both producers build every one, so
            // they stay in step); lane k < npages ends up with the TMA row of
            // the tile's page k
            int npages = 0, nunits = 0, flags = 0, my_row = 0;
            unsigned partial = 0;
            auto put_slot = [&](int slot, int u, int p0, int np, int c, int qrow, int split) {
                if (lane == 0) {
                    scratch->unit[slot] = u;
                    scratch->slot_p0[slot] = p0;
                    scratch->qrow[slot] = qrow;
                    scratch->slot_split[slot] = (int16_t)split;
                    scratch->slot_first[slot] = (int8_t)npages;
                    scratch->slot_pages[slot] = (int8_t)np;
                }
                const int nv = min(kPage, c - (p0 + lane) * kPage);
                if (lane < np) {
                    scratch->page_slot[npages + lane] = (int8_t)slot;
                    scratch->page_valid[npages + lane] = (int8_t)nv;
                }
                partial |= __ballot_sync(kFull, lane < np && nv < kPage) << npages;
            };
            if (lu < 0) {
                while (true) {  // pack short units
                    if (ki == 32) {
                        kb += 32;
                        ki = 0;
                        load_batch();
                    }
                    const int u = __shfl_sync(kFull, bu, ki);
                    if (u < 0) break;  // end of this CTA's list
                    const int np = __shfl_sync(kFull, bnp, ki);
                    const int p0 = __shfl_sync(kFull, bp0, ki);
                    const int c = __shfl_sync(kFull, bctx, ki);
                    const int b = __shfl_sync(kFull, bb, ki);
                    const int hkv = __shfl_sync(kFull, bhkv, ki);
                    const int split = __shfl_sync(kFull, bsplit, ki);
                    if (np > kTilePages) {
                        if (nunits == 0) {  // start chunking it
                            lu = u;
                            lb = b;
                            lhkv = hkv;
                            lp0 = p0;
                            lnp = np;
                            lctx = c;
                            lsplit = split;
                            lnext = 0;
                            load_long(0);
                            ++ki;
                        }
                        break;
                    }
                    if (nunits == kSlots || npages + np > kTilePages) break;
                    put_slot(nunits, u, p0, np, c, b * p.Hq + hkv * G, split);
#pragma unroll
                    for (int o = 0; o < kTilePages; ++o) {
                        const int r = __shfl_sync(kFull, brow[o], ki);
                        if (o < np && lane == npages + o) my_row = r;
                    }
                    npages += np;
                    ++nunits;
                    ++ki;
                }
                if (nunits > 0) flags = kFirst | kLast;
            }
            if (nunits == 0 && lu >= 0) {  // next chunk of the long unit
                const int np = min(kTilePages, lnp - lnext);
                if (lnext + np > lbase + 32) load_long(lnext);
                put_slot(0, lu, lp0 + lnext, np, lctx, lb * p.Hq + lhkv * G, lsplit);
#pragma unroll
                for (int o = 0; o < kTilePages; ++o) {
                    const int r = __shfl_sync(kFull, lrow, (lnext - lbase + o) & 31);
                    if (o < np && lane == o) my_row = r;
                }
                npages = np;
                nunits = 1;
                flags = kChunk | (lnext == 0 ? kFirst : 0) | (lnext + np == lnp ? kLast : 0);
                lnext += np;
                if (lnext == lnp) lu = -1;
            }
            const int kind = nunits > 0 ? kTileWork : kTileEnd;
            if ((tile & 1) != par) {  // another pair's tile
                if (kind == kTileEnd) break;
                continue;
            }
            const int s = tile % kStages;
            const uint32_t ph_prev = (uint32_t)((tile / kStages - 1) & 1);
            const int bk = lane >> 1, bh = lane & 1;  // one box per lane: page bk, half bh of the head dim
            const int rk = __shfl_sync(kFull, my_row, bk & 7);
            uint8_t* stg = stages + (size_t)s * kStageBytes;
            if (!kprod) {
                // ---- the V half, once PV three tiles back is done
                if (kind == kTileEnd) break;
                if (tile >= kStages) ok = wait_or_abort(&v_empty[s], ph_prev, abort_flag, p.err, 41);
                if (!__all_sync(kFull, ok)) break;
                if (lane == 0) mbar_arrive_expect_tx(&v_full[s], (uint32_t)(npages * kPageBytes / 2));
                __syncwarp();
                if (bk < npages)
                    tma_load_2d(stg + kKVTile + bh * kKVHalf + bk * 2048, &tv, bh * 64, rk, &v_full[s], pol);
                last_vfill[s] = tile;
                continue;
            }
            if (lane == 0) {
                scratch->kind = (int16_t)kind;
                scratch->npages = (int16_t)npages;
                scratch->nunits = (int16_t)nunits;
                scratch->flags = (int16_t)flags;
                scratch->partial_mask = (int32_t)partial;
            }
            __syncwarp();
            // ---- the K half (free once S three tiles back is computed) and
            // the descriptor slot (free once the PV issuer is done with tile - 6)
            if (tile >= kStages) ok = wait_or_abort(&k_empty[s], ph_prev, abort_flag, p.err, 40);
            if (ok && tile >= kDescs)
                ok = wait_or_abort(&desc_free[tile % kDescs], (uint32_t)((tile / kDescs - 1) & 1),
                                   abort_flag, p.err, 39);
            if (!__all_sync(kFull, ok)) break;
            TileDesc* d = descs + tile % kDescs;
            if (lane < (int)(sizeof(TileDesc) / 16))
                reinterpret_cast<uint4*>(d)[lane] = reinterpret_cast<const uint4*>(scratch)[lane];
            __syncwarp();
            if (lane == 0) mbar_arrive(&desc_full[tile % kDescs]);
            if (kind == kTileEnd) {
                if (lane == 0) mbar_arrive(&k_full[s]);
                break;
            }
            // q rows of the slots by cp.async, completion tracked on the stage's
            // barrier: row slot * G + g of Q^T, 16-byte chunk c at its
            // 128-byte-swizzle position (chunk c of a row sits at c ^ (row & 7)).
            uint8_t* Qs = stg + 2 * kKVTile;
            for (int idx = lane; idx < nunits * G * 16; idx += 32) {
                const int r = idx >> 4, c = idx & 15;
                const int64_t qr = scratch->qrow[r / G] + r % G;
                cp_async16(Qs + (c >> 3) * kQHalf + r * 128 + (((c & 7) ^ (r & 7)) << 4),
                           p.q + qr * kD + (c & 7) * 8 + (c >> 3) * 64);
            }
            cp_async_mbar_arrive(&k_full[s]);
            __syncwarp();
            if (lane == 0) mbar_arrive_expect_tx(&k_full[s], (uint32_t)(npages * kPageBytes / 2));
            __syncwarp();
            if (bk < npages) tma_load_2d(stg + bh * kKVHalf + bk * 2048, &tk, bh * 64, rk, &k_full[s], pol);
            last_fill[s] = tile;
        }
        // After an abort, copies still in flight land before the CTA ends
        // (without an abort every fill has been consumed, so has completed).
        if (lane == 0 && *abort_flag)
            for (int s = 0; s < kStages; ++s) {
                if (last_fill[s] >= 0) mbar_wait_quiet(&k_full[s], (uint32_t)((last_fill[s] / kStages) & 1));
                if (last_vfill[s] >= 0) mbar_wait_quiet(&v_full[s], (uint32_t)((last_vfill[s] / kStages) & 1));
            }
    } else if (warp == kQkWarp) {
        // ------------------------------------------------------------ S = K Q^T issuer
        constexpr uint32_t idQK = tc::idesc_f16_f32(kM, kN, false, false, BF);
        for (int i = 0;; ++i) {
            const int s = i % kStages, sb = i & 1;
            bool ok = wait_or_abort(&k_full[s], (uint32_t)((i / kStages) & 1), abort_flag, p.err, 44);
            if (!__all_sync(kFull, ok)) break;
            const TileDesc* d = descs + i % kDescs;
            if (d->kind == kTileEnd) break;
            if (i >= 2)
                ok = wait_or_abort(&s_free[sb], (uint32_t)(((i >> 1) - 1) & 1), abort_flag, p.err, 45);
            if (!__all_sync(kFull, ok)) break;
            tc::fence_after_sync();
            tc::fence_proxy_async_smem();  // q rows arrived through the generic proxy
            if (lane == 0) {
                if (d->npages > 0) {
                    const uint8_t* K = stages + (size_t)s * kStageBytes;
                    const uint8_t* Q = K + 2 * kKVTile;
#pragma unroll
                    for (int kk = 0; kk < kD / 16; ++kk) {
                        const int h = kk >> 2, k4 = kk & 3;
                        const uint64_t ad = tc::sdesc_sw128(smem_addr(K + h * kKVHalf) + k4 * 32, 16, 1024);
                        const uint64_t bd = tc::sdesc_sw128(smem_addr(Q + h * kQHalf) + k4 * 32, 16, 1024);
                        tc::mma_f16_ss(tmem + 16 * sb, ad, bd, idQK, kk > 0);
                    }
                }
                tc::mma_commit(&s_full[sb]);
                tc::mma_commit(&k_empty[s]);
            }
            __syncwarp();
        }
        if (lane == 0) {  // its MMAs have completed before TMEM is freed
            tc::mma_commit(&mma_done[0]);
            mbar_wait(&mma_done[0], 0, p.err, 46);
        }
        __syncwarp();
    } else if (warp == kPvWarp) {
        // ------------------------------------------------------------ O^T += V^T P^T issuer
        constexpr uint32_t idPV = tc::idesc_f16_f32(kM, kN, false, true, BF);
        int gcount = 0;
        for (int i = 0;; ++i) {
            const int s = i % kStages, pb = i & 1;
            bool ok = wait_or_abort(&desc_full[i % kDescs], (uint32_t)((i / kDescs) & 1), abort_flag,
                                    p.err, 53);
            if (!__all_sync(kFull, ok)) break;
            const TileDesc* d = descs + i % kDescs;
            if (d->kind == kTileEnd) break;
            const int np = d->npages, fl = d->flags;
            const int grp = (fl & kFirst) ? gcount++ : gcount - 1, ob = grp & 1;
            ok = wait_or_abort(&p_full[pb], (uint32_t)((i >> 1) & 1), abort_flag, p.err, 42);
            if (ok) ok = wait_or_abort(&v_full[s], (uint32_t)((i / kStages) & 1), abort_flag, p.err, 59);
            if (ok && (fl & kFirst) && grp >= 2)
                ok = wait_or_abort(&o_free[ob], (uint32_t)(((grp >> 1) - 1) & 1), abort_flag, p.err, 43);
            if (!__all_sync(kFull, ok)) break;
            tc::fence_after_sync();
            // Keys past ctx in a partial page: P is 0 there, but 0 times a
            // non-finite pool value is not 0, so their V rows are zeroed
            // (whole 128-byte rows: the swizzle only permutes inside a row).
            uint8_t* V = stages + (size_t)s * kStageBytes + kKVTile;
            if (d->partial_mask != 0) {
                for (int k = 0; k < np; ++k) {
                    const int nv = d->page_valid[k];
                    for (int idx = lane; idx < (kPage - nv) * 16; idx += 32) {
                        const int h = idx & 1, c = (idx >> 1) & 7, r = nv + (idx >> 4);
                        *reinterpret_cast<uint4*>(V + h * kKVHalf + (k * kPage + r) * 128 + c * 16) =
                            make_uint4(0u, 0u, 0u, 0u);
                    }
                }
                tc::fence_proxy_async_smem();
            }
            __syncwarp();
            if (lane == 0) {
                const uint32_t tO = tmem + 32 + 16 * ob;
                const uint8_t* P = Ps + pb * kPTile;
                for (int k = 0; k < np; ++k) {
                    const uint64_t bd = tc::sdesc_sw128(smem_addr(P + (k >> 2) * kPHalf) + (k & 3) * 32, 16, 1024);
                    const uint64_t ad = tc::sdesc_sw128(smem_addr(V + k * 2048), kKVHalf, 1024);
                    tc::mma_f16_ss(tO, ad, bd, idPV, !((fl & kFirst) && k == 0));
                }
                tc::mma_commit(&v_empty[s]);
                tc::mma_commit(&pv_done[pb]);
                if (fl & kLast) tc::mma_commit(&o_full[ob]);
                mbar_arrive(&desc_free[i % kDescs]);  // descriptor no longer read
            }
            __syncwarp();
        }
        if (lane == 0) {
            tc::mma_commit(&mma_done[1]);
            mbar_wait(&mma_done[1], 0, p.err, 54);
        }
        __syncwarp();
    } else if (warp < kSoftmaxWarps) {
        // ------------------------------------------------------------ softmax
        const int t = tid;  // key row of S^T, TMEM lane
        const int k = t >> 4;
        const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
        float m[G], l[G];  // reference max and this row's sum of p, of its column slot
#pragma unroll
        for (int g = 0; g < G; ++g) m[g] = l[g] = 0.f;
        int gcount = 0;
        for (int i = 0;; ++i) {
            const int sb = i & 1, pb = i & 1;
            if (!wait_or_abort(&desc_full[i % kDescs], (uint32_t)((i / kDescs) & 1), abort_flag, p.err, 47))
                break;
            const TileDesc* d = descs + i % kDescs;
            // kind, npages, nunits, flags in one load; page_slot[8] and
            // page_valid[8] in another
            const uint2 hd = *reinterpret_cast<const uint2*>(&d->kind);
            if ((int16_t)(hd.x & 0xffffu) == kTileEnd) {  // tell the epilogue there are no more groups
                const int ob = gcount & 1;
                if (gcount >= 2 &&
                    !wait_or_abort(&o_free[ob], (uint32_t)(((gcount >> 1) - 1) & 1), abort_flag, p.err, 55))
                    break;
                if (t == 0) info[ob].nunits = -1;
                __syncwarp();
                if (lane == 0) mbar_arrive(&epi_ready[ob]);
                break;
            }
            const int np = (int16_t)(hd.x >> 16), nun = (int16_t)(hd.y & 0xffffu), fl = (int16_t)(hd.y >> 16);
            const uint4 pp = *reinterpret_cast<const uint4*>(d->page_slot);
            auto page_slot_of = [&](int kk) {  // kk < kTilePages
                return (int)(int8_t)(((kk < 4 ? pp.x : pp.y) >> (8 * (kk & 3))) & 0xffu);
            };
            if (fl & kFirst) {
                ++gcount;
#pragma unroll
                for (int g = 0; g < G; ++g) l[g] = 0.f;
            }
            const int grp = gcount - 1, ob = grp & 1;
            const int pslot = k < np ? page_slot_of(k) : -1;
            const int pvalid = (int)(((k < 4 ? pp.z : pp.w) >> (8 * (k & 3))) & 0xffu);
            const bool valid = k < np && (t & 15) < pvalid;
            const int cslot = (fl & kChunk) ? 0 : pslot;  // the columns this key row counts in
            // the leader of the first page of its slot publishes the slot's max
            const bool m_writer = (t & 15) == 0 && pslot >= 0 && (k == 0 || page_slot_of(k - 1) != pslot);
            const int qrow_t = t < nun ? d->qrow[t] : -1;
            const int split_t = t < kN ? d->slot_split[t] : 0;

            // ---- S row (this key against the 16 columns)
            if (!wait_or_abort(&s_full[sb], (uint32_t)((i >> 1) & 1), abort_flag, p.err, 48)) break;
            tc::fence_after_sync();
            float sv[kN];
            tc::tmem_ld16(tmem + 16 * sb + lane_base, sv);
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&s_free[sb]);
            float v[G];
#pragma unroll
            for (int g = 0; g < G; ++g) v[g] = -INFINITY;
            if (valid) {
#pragma unroll
                for (int j = 0; j < kSlots; ++j)
                    if (cslot == j) {
#pragma unroll
                        for (int g = 0; g < G; ++g) v[g] = sv[j * G + g] * p.scale_log2;
                    }
            }
            // ---- column max over the key rows of this slot: per page (16
            // lanes), then over the tile's pages of the slot
            float pm[G];
#pragma unroll
            for (int g = 0; g < G; ++g) {
                pm[g] = v[g];
#pragma unroll
                for (int o = 8; o >= 1; o >>= 1) pm[g] = fmaxf(pm[g], __shfl_xor_sync(kFull, pm[g], o));
            }
            float* red = redbuf + (i & 1) * (kTilePages * 8);
            if ((t & 15) == 0) {
#pragma unroll
                for (int g = 0; g < G; ++g) red[k * 8 + g] = pm[g];
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(red_bar);
            if (!wait_or_abort(red_bar, (uint32_t)(i & 1), abort_flag, p.err, 49)) break;
            float tm[G];
#pragma unroll
            for (int g = 0; g < G; ++g) tm[g] = -INFINITY;
#pragma unroll
            for (int kk = 0; kk < kTilePages; ++kk) {
                if (kk < np && page_slot_of(kk) == cslot) {
                    float rv[G];
                    if constexpr (G >= 4) {
#pragma unroll
                        for (int g4 = 0; g4 < G; g4 += 4) {
                            const float4 x = *reinterpret_cast<const float4*>(&red[kk * 8 + g4]);
                            rv[g4] = x.x; rv[g4 + 1] = x.y; rv[g4 + 2] = x.z; rv[g4 + 3] = x.w;
                        }
                    } else {
#pragma unroll
                        for (int g = 0; g < G; ++g) rv[g] = red[kk * 8 + g];
                    }
#pragma unroll
                    for (int g = 0; g < G; ++g) tm[g] = fmaxf(tm[g], rv[g]);
                }
            }
            // ---- reference max; a chunk group's is the same in every thread
            bool rescale = false;
            float alpha[G];
#pragma unroll
            for (int g = 0; g < G; ++g) {
                alpha[g] = 1.f;
                if (fl & kFirst) {
                    m[g] = tm[g];
                } else if (tm[g] > m[g] + kRescaleThreshold) {
                    alpha[g] = exp2f(m[g] - tm[g]);
                    m[g] = tm[g];
                    rescale = true;
                }
            }
            if (rescale) {  // O is stable once PV of the previous tile is done
                if (!wait_or_abort(&pv_done[(i - 1) & 1], (uint32_t)(((i - 1) >> 1) & 1), abort_flag,
                                   p.err, 50))
                    break;
                tc::fence_after_sync();
                const uint32_t tO = tmem + 32 + 16 * ob + lane_base;
                float ov[kN];
                tc::tmem_ld16(tO, ov);
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    ov[g] *= alpha[g];
                    l[g] *= alpha[g];
                }
                tc::tmem_st16(tO, ov);
            }
            // ---- P^T (the P buffer is free once PV two tiles back is done)
            if (i >= 2 &&
                !wait_or_abort(&pv_done[pb], (uint32_t)(((i - 2) >> 1) & 1), abort_flag, p.err, 51))
                break;
            uint16_t ph[G];  // p in the operand type (fp16 or bf16, nearest even)
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const float pf = valid ? exp2f(v[g] - m[g]) : 0.f;
                l[g] += pf;
                ph[g] = BF ? __bfloat16_as_ushort(__float2bfloat16_rn(pf))
                           : __half_as_ushort(__float2half_rn(pf));
            }
            uint8_t* P = Ps + pb * kPTile + (t >> 6) * kPHalf + (t & 7) * 2;
            const int tq = (t & 63) >> 3;
#pragma unroll
            for (int c = 0; c < kN; ++c)  // +0 is all zero bits in both types
                *reinterpret_cast<uint16_t*>(P + c * 128 + ((tq ^ (c & 7)) << 4)) =
                    (c / G == cslot) ? ph[c % G] : (uint16_t)0;
            tc::fence_proxy_async_smem();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&p_full[pb]);

            // ---- end of a group: hand the epilogue its columns
            if (fl & kLast) {
                if (grp >= 2 &&
                    !wait_or_abort(&o_free[ob], (uint32_t)(((grp >> 1) - 1) & 1), abort_flag, p.err, 56))
                    break;
                GroupInfo& gi = info[ob];
                float ls[G];
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    ls[g] = l[g];
#pragma unroll
                    for (int o = 8; o >= 1; o >>= 1) ls[g] += __shfl_xor_sync(kFull, ls[g], o);
                }
                if ((t & 15) == 0) {  // this page's partial sums, 0 in other columns
#pragma unroll
                    for (int c = 0; c < kN; ++c) gi.lpage[k][c] = (c / G == cslot) ? ls[c % G] : 0.f;
                }
                if (m_writer) {
#pragma unroll
                    for (int g = 0; g < G; ++g) gi.m[pslot * G + g] = m[g];
                }
                if (t < kN) {
                    gi.qrow[t] = qrow_t;
                    gi.split[t] = split_t;
                }
                if (t == 0) {
                    gi.nunits = nun;
                    gi.has_o = np > 0 ? 1 : 0;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&epi_ready[ob]);
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int e = tid - kEpiWarp0 * 32;  // head-dim row of O^T, TMEM lane
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        for (int grp = 0;; ++grp) {
            const int ob = grp & 1;
            if (!wait_or_abort(&epi_ready[ob], (uint32_t)((grp >> 1) & 1), abort_flag, p.err, 57)) break;
            const GroupInfo& gi = info[ob];
            if (gi.nunits < 0) break;
            if (!wait_or_abort(&o_full[ob], (uint32_t)((grp >> 1) & 1), abort_flag, p.err, 58)) break;
            tc::fence_after_sync();
            float ov[kN];
#pragma unroll
            for (int c = 0; c < kN; ++c) ov[c] = 0.f;
            if (gi.has_o) tc::tmem_ld16(tmem + 32 + 16 * ob + lane_base, ov);
            float L[kN];
#pragma unroll
            for (int c = 0; c < kN; ++c) L[c] = 0.f;
#pragma unroll
            for (int kk = 0; kk < kTilePages; ++kk)
#pragma unroll
                for (int c = 0; c < kN; c += 4) {
                    const float4 x = *reinterpret_cast<const float4*>(&gi.lpage[kk][c]);
                    L[c] += x.x; L[c + 1] += x.y; L[c + 2] += x.z; L[c + 3] += x.w;
                }
#pragma unroll
            for (int j = 0; j < kSlots; ++j) {
                const int qr = gi.qrow[j];
                if (qr < 0) continue;
                const int split = gi.split[j];
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    const int c = j * G + g;
                    const int64_t row = (int64_t)(qr + g) * p.NS + split;
                    p.o_part[row * kD + e] = L[c] > 0.f ? __fdividef(ov[c], L[c]) : 0.f;
                    if (e == c) p.lse_part[row] = L[c] > 0.f ? gi.m[c] + __log2f(L[c]) : -INFINITY;
                }
            }
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&o_free[ob]);
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc::fence_after_sync();
        tc::tmem_free(tmem, kTmemCols);
    }
    last_cta_waits_primary(p.done_ctr);
}

template <int G, bool BF>
cudaError_t launch_tc_g(const CUtensorMap& tk, const CUtensorMap& tv, const TcParams& p, int grid,
                        const DeviceInfo& dev, cudaStream_t st) {
    auto kern = splitkv_decode_tc_kernel<G, BF>;
    static bool attr_set[64] = {};
    if (dev.device >= 0 && dev.device < 64 && !attr_set[dev.device]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_set[dev.device] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = p.done_ctr != nullptr ? 1 : 0;  // chained after a prefix pass
    return cudaLaunchKernelEx(&cfg, kern, tk, tv, p);
}

}  // namespace

cudaError_t launch_splitkv_decode_tc(const DecodeArgs& a, const DeviceInfo& dev, cudaStream_t st) {
    if (kSmemBytes > dev.max_smem_optin) return cudaErrorInvalidValue;
    const uint64_t rows = (uint64_t)a.num_pool_pages * a.Hkv * kPage;
    CUtensorMap tk, tv;
    cudaError_t e = make_tmap_2d_16bit(&tk, a.k_cache, rows, kD, kD * 2, 64, kPage, true, a.bf16);
    if (e != cudaSuccess) return e;
    if ((e = make_tmap_2d_16bit(&tv, a.v_cache, rows, kD, kD * 2, 64, kPage, true, a.bf16)) != cudaSuccess)
        return e;
    TcParams p;
    p.q = static_cast<const uint16_t*>(a.q);
    p.block_table = a.block_table;
    p.ctx = a.ctx;
    p.o_part = a.o_part;
    p.lse_part = a.lse_part;
    p.ranges_dbg = a.ranges_dbg;
    p.err = dev.err;
    p.done_ctr = a.done_ctr;
    p.num_pool_pages = a.num_pool_pages;
    p.max_pages = a.max_pages;
    p.B = a.B;
    p.Hq = a.Hq;
    p.Hkv = a.Hkv;
    p.NS = a.num_splits;
    const int64_t units = (int64_t)a.B * a.Hkv * a.num_splits;
    if (units <= 0 || units > INT32_MAX) return cudaErrorInvalidValue;
    p.units = (int32_t)units;
    p.scale_log2 = a.sm_scale * 1.4426950408889634f;
    // As few CTAs as give every CTA the same number of units (at most one
    // per SM): 512 equal units run as 128 CTAs x 4 rather than 152 CTAs of
    // which 56 take a fourth unit while the rest of the GPU idles.
    const int64_t per_cta = (units + dev.sm_count - 1) / dev.sm_count;
    const int grid = (int)((units + per_cta - 1) / per_cta);
#define SKV_LAUNCH_TC(BF_)                                            \
    switch (a.Hq / a.Hkv) {                                           \
        case 1: return launch_tc_g<1, BF_>(tk, tv, p, grid, dev, st); \
        case 2: return launch_tc_g<2, BF_>(tk, tv, p, grid, dev, st); \
        case 4: return launch_tc_g<4, BF_>(tk, tv, p, grid, dev, st); \
        case 8: return launch_tc_g<8, BF_>(tk, tv, p, grid, dev, st); \
    }
    if (a.bf16) SKV_LAUNCH_TC(true) else SKV_LAUNCH_TC(false)
#undef SKV_LAUNCH_TC
    return cudaErrorInvalidValue;
}

}  // namespace skv
