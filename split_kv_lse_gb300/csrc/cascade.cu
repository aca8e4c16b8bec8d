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
// One CTA per (kv head, pair of 128-row M tiles, chunk of the prefix).  An M
// tile's rows are (request, group head) pairs -- row = r_local * G + g -- and
// the CTA's two M tiles share every K and V block it loads, so each prefix
// block crosses HBM and the TMA unit once per 256 query rows.  Per 128-key
// block j and M tile w (softmax group w):
//   S_w = Q_w K_j^T  tcgen05.mma kind::f16, Q_w [128 x 128] and the K block
//                    [128 keys x 128] K-major in shared memory, S fp32 in TMEM
//   softmax          group w, thread i <-> row i <-> TMEM lane i: base-2
//                    online max/sum ([F2] §② exp2 trick); P = 2^(s - m) as
//                    fp16 pairs written back into TMEM over S
//   O_w += P V_j     tcgen05.mma with P from TMEM (A operand) and V an
//                    MN-major operand in shared memory; O fp32 stays in TMEM
// The MMAs are issued in the order S_0(j), S_1(j), PV_0(j), S_0(j+1),
// PV_1(j), S_1(j+1), ...: the tensor core computes one group's S while the
// other group runs its softmax, and an S MMA never overwrites a P that a
// PV issued before it has yet to read (tcgen05 MMAs of a thread run in order).
// Lazy rescale: a row keeps the max it last rescaled to and only rescales
// O and its sum when the block max exceeds it by more than 8 (log2 units),
// so p <= 2^8 (exact in fp16 range); the final normalisation by the same
// max keeps the result exact.
// Warp roles: warps 0-3 and 4-7 the two softmax groups (and their
// epilogues), warp 8 issues the MMAs, warp 9 loads Q and the K blocks,
// warp 10 the V blocks (16 lanes issue a block's boxes at once).  Two K and
// two V blocks are in flight.  Every wait is bounded; a wait that gives up
// raises a shared abort flag that ends every role's loop.  Each chunk writes
// its normalised state (o, s base 2) per row for the combine kernel, which
// merges the chunks into the prefix state.
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
constexpr int kM = 128;                              // query rows per M tile
constexpr int kHalf = 128 * 128;                     // one [128 rows x 64] fp16 swizzled half tile
constexpr int kTile = 2 * kHalf;                     // one [128 x 128] fp16 operand tile (32 KB)
constexpr int kStages = 2;                           // K blocks and V blocks in flight
constexpr int kSoftmaxWarps = 4;                     // per group: one thread per query row
constexpr int kMmaWarp = 8;
constexpr int kKWarp = 9;
constexpr int kVWarp = 10;
constexpr int kThreads = 11 * 32;
constexpr uint32_t kTmemCols = 512;                  // group w: S/P at 256 w, O at 256 w + 128
constexpr float kRescaleThreshold = 8.f;             // log2 units
constexpr unsigned kFull = 0xffffffffu;

struct PrefixParams {
    const int32_t* prefix_pages;
    int32_t prefix_len;
    int32_t pool_rows;        // rows of the K/V tensor maps: num_pool_pages * Hkv * page
    int32_t num_pool_pages;
    int32_t B, Hq, Hkv, G;
    int32_t blocks_per_chunk;
    int32_t chunk_stride;     // chunk-state slots per row in pre_part / pre_lse
    int32_t chunk_offset;     // slot of this launch's chunk 0
    float scale_log2;
    float* pre_part;          // [B*Hq, chunk_stride, D] split-normalised chunk states
    float* pre_lse;           // [B*Hq, chunk_stride] base 2
    unsigned long long* err;
    unsigned int* zero_ctr;   // CascadeArgs::zero_ctr or nullptr
    int32_t chained;          // CascadeArgs::chained
};

constexpr size_t kSmemQ = 0;                                   // Q_0, Q_1
constexpr size_t kSmemK = kSmemQ + 2 * (size_t)kTile;
constexpr size_t kSmemV = kSmemK + (size_t)kStages * kTile;
constexpr size_t kSmemBars = kSmemV + (size_t)kStages * kTile;
// q_full, s_full[2], p_full[2], pv_done[2], k_full[], k_empty[], v_full[], v_empty[]
constexpr int kNumBars = 7 + 4 * kStages;
constexpr size_t kSmemTmemSlot = kSmemBars + kNumBars * sizeof(uint64_t);
constexpr size_t kSmemEnd = kSmemTmemSlot + 16;      // tmem address, abort flag

size_t prefix_smem_bytes(int) { return 1024 + kSmemEnd; }

// D[tmem] (+)= A[tmem] * B[smem]^T: the A operand (M rows = TMEM lanes, K
// 16-bit elements packed two per 32-bit column) is read from tensor memory.
SKV_DEVINL void mma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                           bool accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
        :: "r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate ? 1u : 0u)
        : "memory");
}

template <bool BF>  // q, K, V (and so P) bf16, else fp16
__global__ void __launch_bounds__(kThreads, 1)
cascade_prefix_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                      const __grid_constant__ CUtensorMap tv, const PrefixParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    uint8_t* Qs = sm + kSmemQ;
    uint8_t* Ks = sm + kSmemK;
    uint8_t* Vs = sm + kSmemV;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kSmemBars);
    uint64_t* q_full = bars + 0;
    uint64_t* s_full = bars + 1;   // [2] per group
    uint64_t* p_full = bars + 3;   // [2]
    uint64_t* pv_done = bars + 5;  // [2]
    uint64_t* k_full = bars + 7;
    uint64_t* k_empty = k_full + kStages;
    uint64_t* v_full = k_empty + kStages;
    uint64_t* v_empty = v_full + kStages;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + kSmemTmemSlot);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + kSmemTmemSlot + 4);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int chunk = blockIdx.x, mpair = blockIdx.y, hkv = blockIdx.z;
    // Chaining in one stream: CTA 0 of a cascade's first prefix pass zeroes
    // the completion counter of the suffix pass before any dependent kernel
    // can start; then every CTA lets the next kernel start at once (nothing
    // launched after this pass reads what it writes before it completes).
    if (p.zero_ctr != nullptr && chunk == 0 && mpair == 0 && hkv == 0) {
        if (tid == 0) {
            *p.zero_ctr = 0u;
            __threadfence();
        }
        __syncthreads();
    }
    pdl_launch_dependents();
    const int nblocks_total = (p.prefix_len + kBlockKeys - 1) / kBlockKeys;
    const int blk0 = chunk * p.blocks_per_chunk;
    const int nb = min(p.blocks_per_chunk, nblocks_total - blk0);
    const int npages_prefix = (p.prefix_len + kPage - 1) / kPage;
    if (nb <= 0) {
        // A slot past this prefix's last block (the grid covers the most
        // chunks any prefix of its level has): an empty state, s = -inf, for
        // each of the CTA's rows (a zero-weight state's v is never read).
        for (int i = tid; i < 2 * kM; i += kThreads) {
            const int r = i / p.G, g = i % p.G;  // row i of the M pair: request, group head
            const int req = 2 * mpair * (kM / p.G) + r;
            if (req < p.B)
                p.pre_lse[((int64_t)req * p.Hq + hkv * p.G + g) * p.chunk_stride + p.chunk_offset +
                          chunk] = -INFINITY;
        }
        if (p.chained) pdl_wait_primary();  // complete after the previous prefix pass
        return;
    }

    if (tid == 0) {
        mbar_init(q_full, 1);
        for (int w = 0; w < 2; ++w) {
            mbar_init(&s_full[w], 1);
            mbar_init(&p_full[w], kSoftmaxWarps);
            mbar_init(&pv_done[w], 1);
        }
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

    if (warp == kKWarp || warp == kVWarp) {
        // ---------------------------------------------------------------- TMA producers
        const bool isk = warp == kKWarp;
        if (lane == 0) {
            if (isk) tma_prefetch_desc(&tq);
            tma_prefetch_desc(isk ? &tk : &tv);
        }
        const uint64_t pol = policy_evict_first();
        int win = -1, wid = -1;  // page-id window of the prefix list: id of page 32 * win + lane
        // A block's 16 boxes (8 pages x 2 halves of the head dim) go out from
        // 16 lanes at once: copies issued one after another by one thread
        // stream at about half the HBM bandwidth.
        auto load_block = [&](int j) {
            const int stage = j % kStages;
            uint64_t* bar = isk ? &k_full[stage] : &v_full[stage];
            uint8_t* dst = (isk ? Ks : Vs) + stage * kTile;
            const CUtensorMap* map = isk ? &tk : &tv;
            if (lane == 0) mbar_arrive_expect_tx(bar, kTile);
            __syncwarp();
            const int pg = lane >> 1, h = lane & 1;
            // The block's 8 pages lie in one 32-page window of the prefix page
            // list, held one id per lane (reloaded every 4 blocks).
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
            const int pid = __shfl_sync(kFull, wid, (g0 + (pg & 7)) & 31);
            if (pg < kPagesPerBlock) {
                // A page past the prefix is read from the row just past the
                // tensor: the TMA fills the whole box with zeros.
                const int row = pid >= 0 ? (pid * p.Hkv + hkv) * kPage : p.pool_rows;
                tma_load_2d(dst + h * kHalf + pg * (kPage * 128), map, h * 64, row, bar, pol);
            }
        };
        if (isk && lane == 0) {  // both M tiles' queries (a tile past B reads zeros)
            mbar_arrive_expect_tx(q_full, 2 * kTile);
            for (int w = 0; w < 2; ++w) {
                const int z = (2 * mpair + w) * (kM / p.G);
                tma_load_3d(Qs + w * kTile, &tq, 0, hkv * p.G, z, q_full);
                tma_load_3d(Qs + w * kTile + kHalf, &tq, 64, hkv * p.G, z, q_full);
            }
        }
        uint64_t* empty = isk ? k_empty : v_empty;
        for (int j = 0; j < nb; ++j) {
            bool ok = true;
            if (j >= kStages)
                ok = wait_or_abort(&empty[j % kStages], (uint32_t)((j / kStages - 1) & 1), abort_flag,
                                   p.err, isk ? 20 : 21);
            if (!__all_sync(kFull, ok)) break;
            load_block(j);
        }
    } else if (warp == kMmaWarp) {
        // ---------------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idS = tc::idesc_f16_f32(kM, kBlockKeys, false, false, BF);
            // A (P) from TMEM, B (V) MN-major
            constexpr uint32_t idPV = tc::idesc_f16_f32(kM, kD, true, false, BF);
            // The descriptors differ only in their start address (bits 0-13,
            // the byte address >> 4; shared addresses stay below 256 KB, so
            // an offset added there never carries out): built once, then
            // offset by constants, so that this thread -- which shares its
            // scheduler with two softmax warps -- spends few instructions
            // per MMA.
            const uint64_t q_desc = tc::sdesc_sw128(smem_addr(Qs), 16, 1024);
            const uint64_t k_desc = tc::sdesc_sw128(smem_addr(Ks), 16, 1024);
            const uint64_t v_desc = tc::sdesc_sw128(smem_addr(Vs), kHalf, 1024);
            auto qk = [&](int j, int w) {  // S_w = Q_w K_j^T
                const uint64_t ab = q_desc + (uint64_t)((w * kTile) >> 4);
                const uint64_t bb = k_desc + (uint64_t)(((j % kStages) * kTile) >> 4);
#pragma unroll
                for (int k = 0; k < kD / 16; ++k) {
                    // K step k: head-dim half k / 4 (a swizzled half tile),
                    // 32 bytes (16 elements) k % 4 into its 128-byte rows.
                    const uint64_t off = (uint64_t)(((k >> 2) * kHalf + (k & 3) * 32) >> 4);
                    tc::mma_f16_ss(tmem + 256 * w, ab + off, bb + off, idS, k > 0);
                }
                tc::mma_commit(&s_full[w]);
            };
            auto pv = [&](int j, int w) -> bool {  // O_w += P_w V_j
                if (!wait_or_abort(&p_full[w], (uint32_t)(j & 1), abort_flag, p.err, 22)) return false;
                tc::fence_after_sync();
                const uint64_t vb = v_desc + (uint64_t)(((j % kStages) * kTile) >> 4);
#pragma unroll
                for (int k = 0; k < kBlockKeys / 16; ++k)  // 16 keys (rows of 128 bytes) a step
                    mma_f16_ts(tmem + 256 * w + 128, tmem + 256 * w + 8 * k, vb + (uint64_t)((k * 2048) >> 4),
                               idPV, j > 0 || k > 0);
                tc::mma_commit(&pv_done[w]);
                return true;
            };
            bool ok = wait_or_abort(q_full, 0, abort_flag, p.err, 24);
            ok = ok && wait_or_abort(&k_full[0], 0, abort_flag, p.err, 25);
            if (ok) {
                tc::fence_after_sync();
                qk(0, 0);
                qk(0, 1);
                tc::mma_commit(&k_empty[0]);
            }
            // S_0(j+1) goes in after PV_0(j) and S_1(j+1) after PV_1(j): a PV
            // reads its P from the TMEM columns that the next S overwrites.
            for (int j = 0; ok && j < nb; ++j) {
                const int st = j % kStages;
                ok = wait_or_abort(&v_full[st], (uint32_t)((j / kStages) & 1), abort_flag, p.err, 23);
                if (!ok) break;
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
                if (!(ok = pv(j, 0))) break;
                const bool more = j + 1 < nb;
                if (more) {
                    ok = wait_or_abort(&k_full[(j + 1) % kStages], (uint32_t)(((j + 1) / kStages) & 1),
                                       abort_flag, p.err, 25);
                    if (!ok) break;
                    tc::fence_after_sync();
                    qk(j + 1, 0);
                }
                if (!(ok = pv(j, 1))) break;
                tc::mma_commit(&v_empty[st]);
                if (more) {
                    qk(j + 1, 1);
                    tc::mma_commit(&k_empty[(j + 1) % kStages]);
                }
            }
        }
    } else {
        // ---------------------------------------------------------------- softmax group w, row = tid % 128
        const int w = warp >> 2, row_t = tid & (kM - 1);
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t tS = tmem + 256 * w + lane_base;        // S, then P over it
        const uint32_t tO = tmem + 256 * w + 128 + lane_base;
        float m_ref = -INFINITY;  // the max this row's O and l are scaled to (log2 units)
        float l_run = 0.f;
        bool ok = true;
        for (int j = 0; j < nb; ++j) {
            // S_w(j) is complete; so is every MMA issued before it, PV_w(j-1)
            // included: O_w is stable and P_w's columns may be rewritten.
            ok = wait_or_abort(&s_full[w], (uint32_t)(j & 1), abort_flag, p.err, 27);
            if (!__all_sync(kFull, ok)) {
                ok = false;
                break;
            }
            tc::fence_after_sync();
            float x[kBlockKeys];
            tc::tmem_ld128(tS, x);
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
            // Lazy rescale, also the first block (m_ref = -inf).  The TMEM
            // loads and stores are warp-wide (.sync.aligned), so the warp
            // rescales O when any of its rows needs it, with alpha = 1 for
            // the rows that do not.
            const bool need = mx > m_ref + kRescaleThreshold;
            const float m_new = need ? mx : m_ref;
            if (j > 0 && __any_sync(kFull, need)) {
                const float alpha = need ? exp2f(m_ref - m_new) : 1.f;
                l_run *= alpha;
#pragma unroll 1
                for (int c = 0; c < kD / 32; ++c) {  // 32 columns at a time: x[] stays live
                    float ob[32];
                    tc::tmem_ld32(tO + 32 * c, ob);
#pragma unroll
                    for (int i = 0; i < 32; ++i) ob[i] *= alpha;
                    tc::tmem_st32(tO + 32 * c, ob);
                }
            }
            m_ref = m_new;
            // P as fp16 pairs, key 2c in the low half of column c, written
            // over S (this thread's own TMEM lane, already read).
            float ps4[4] = {0.f, 0.f, 0.f, 0.f};  // independent partial sums
            const float nm = -m_ref;
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                float pk[32];
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    const int i0 = 64 * hh + 2 * c;
                    const float p0 = fast_exp2(fmaf(x[i0], sc, nm));  // masked keys: 2^-inf = 0
                    const float p1 = fast_exp2(fmaf(x[i0 + 1], sc, nm));
                    ps4[c & 3] += p0 + p1;
                    uint32_t h2;  // (p0, p1) in the operand type, nearest even
                    if constexpr (BF) {
                        const __nv_bfloat162 b2 = __floats2bfloat162_rn(p0, p1);
                        h2 = *reinterpret_cast<const uint32_t*>(&b2);
                    } else {
                        const __half2 f2 = __floats2half2_rn(p0, p1);
                        h2 = *reinterpret_cast<const uint32_t*>(&f2);
                    }
                    pk[c] = __uint_as_float(h2);
                }
                tc::tmem_st32(tS + 32 * hh, pk);
            }
            l_run += (ps4[0] + ps4[1]) + (ps4[2] + ps4[3]);
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&p_full[w]);  // P_w(j) (and any O rescale) done by this warp
        }
        // ---- this chunk's state of row row_t of M tile w, after its last PV.
        // Every MMA of the CTA is complete once both groups' last PVs are,
        // and the last S MMAs were issued before them: Q_w and K stage w
        // (64 KB) are free and stage this group's 128 normalised rows, which
        // each warp then stores row by row with coalesced 512-byte writes
        // (one thread per row would write 16-byte pieces of 32 rows at once).
        if (ok) ok = wait_or_abort(&pv_done[w], (uint32_t)((nb - 1) & 1), abort_flag, p.err, 29);
        if (__all_sync(kFull, ok)) {
            tc::fence_after_sync();
            auto stage_row = [&](int r) -> uint8_t* {  // 512 bytes per row, chunks XOR-swizzled by row
                return r < 64 ? Qs + w * kTile + r * 512 : Ks + w * kTile + (r - 64) * 512;
            };
            const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
            uint8_t* mine = stage_row(row_t);
#pragma unroll 1
            for (int c = 0; c < kD / 32; ++c) {
                float ob[32];
                tc::tmem_ld32(tO + 32 * c, ob);
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    *reinterpret_cast<float4*>(mine + (((8 * c + q) ^ (row_t & 31)) << 4)) =
                        make_float4(ob[4 * q] * inv, ob[4 * q + 1] * inv, ob[4 * q + 2] * inv,
                                    ob[4 * q + 3] * inv);
            }
            const int rows_per_req = p.G;
            const int req0 = (2 * mpair + w) * (kM / rows_per_req);
            {
                const int r = req0 + row_t / rows_per_req, g = row_t % rows_per_req;
                if (r < p.B)
                    p.pre_lse[((int64_t)r * p.Hq + hkv * p.G + g) * p.chunk_stride + p.chunk_offset + chunk] =
                        l_run > 0.f ? m_ref + log2f(l_run) : -INFINITY;
            }
            __syncwarp();  // this warp's 32 rows are staged
#pragma unroll 4
            for (int i = 0; i < 32; ++i) {
                const int rt = (warp & 3) * 32 + i;
                const int r = req0 + rt / rows_per_req, g = rt % rows_per_req;
                if (r < p.B) {
                    const float4 v = *reinterpret_cast<const float4*>(stage_row(rt) + ((lane ^ (rt & 31)) << 4));
                    float* dst = p.pre_part +
                                 (((int64_t)r * p.Hq + hkv * p.G + g) * p.chunk_stride + p.chunk_offset + chunk) * kD;
                    *reinterpret_cast<float4*>(dst + 4 * lane) = v;
                }
            }
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc::fence_after_sync();
        tc::tmem_free(tmem, kTmemCols);
    }
    if (p.chained) pdl_wait_primary();  // complete after the previous prefix pass
}

}  // namespace

void cascade_prefix_geometry(int B, int G, int Hkv, int prefix_len, int sm_count, int* mtiles,
                             int* blocks_per_chunk, int* nchunks) {
    const int nblocks = (prefix_len + kBlockKeys - 1) / kBlockKeys;
    const int mt = (B * G + kM - 1) / kM;
    const int pairs = (mt + 1) / 2;  // a CTA takes two M tiles
    // About one CTA per SM: chunks = SMs / (Hkv * pairs), at least one block each.
    int want = sm_count / (Hkv * pairs > 0 ? Hkv * pairs : 1);
    if (want < 1) want = 1;
    if (want > nblocks) want = nblocks;
    int bpc = nblocks > 0 ? (nblocks + want - 1) / want : 1;
    *mtiles = mt;
    *blocks_per_chunk = bpc;
    *nchunks = nblocks > 0 ? (nblocks + bpc - 1) / bpc : 0;
}

cudaError_t launch_cascade_prefix(const CascadeArgs& a, const DeviceInfo& dev, float* pre_part,
                                  float* pre_lse, int nchunks, int blocks_per_chunk, int mtiles,
                                  int chunk_stride, int chunk_offset, cudaStream_t st) {
    const int G = a.Hq / a.Hkv;
    CUtensorMap tq, tk, tv;
    // (fp16 element type for bf16 q too: the copies are bitwise and the
    // out-of-range fill, zero bits, is +0 in both.)
    cudaError_t e = make_tmap_3d_16bit(&tq, a.q, kD, a.Hq, a.B, (uint64_t)kD * 2,
                                       (uint64_t)a.Hq * kD * 2, 64, G, kM / G, true);
    if (e != cudaSuccess) return e;
    const uint64_t rows = (uint64_t)a.num_pool_pages * a.Hkv * kPage;
    if ((e = make_tmap_2d_16bit(&tk, a.k_cache, rows, kD, kD * 2, 64, kPage, true, a.bf16)) != cudaSuccess)
        return e;
    if ((e = make_tmap_2d_16bit(&tv, a.v_cache, rows, kD, kD * 2, 64, kPage, true, a.bf16)) != cudaSuccess)
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
    p.chunk_stride = chunk_stride;
    p.chunk_offset = chunk_offset;
    p.scale_log2 = a.sm_scale * 1.4426950408889634f;
    p.pre_part = pre_part;
    p.pre_lse = pre_lse;
    p.err = dev.err;
    p.zero_ctr = a.zero_ctr;
    p.chained = a.chained ? 1 : 0;
    const size_t smem = prefix_smem_bytes(blocks_per_chunk);
    if (smem > dev.max_smem_optin) return cudaErrorInvalidValue;
    auto kern = a.bf16 ? cascade_prefix_kernel<true> : cascade_prefix_kernel<false>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(nchunks, (mtiles + 1) / 2, a.Hkv);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = a.chained ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, tq, tk, tv, p);
}

}  // namespace skv
