// decode.cu -- split-KV paged decode attention for sm_103a: pass 1 (the
// per-split states) and pass 2 (their merge, chained with programmatic
// dependent launch).
//
// Page: "L3 讲解：split-KV decode 与 LSE 合并" -- §① the two-pass
// Flash-Decoding scheme (grid (B, Hkv, NUM_SPLITS), each program walks its
// own pages and writes a split-normalised o and that split's lse), §② the
// page ranges, §③ the per-split state o_s = acc/l, lse_s = m + log l (here in
// base 2: s = m2 + log2 l), §④ empty splits (o = 0, lse = -inf), §⑤ fp32
// partials.
//
// GB300 design of pass 1 (not the page's Triton program):
//   * One CTA per (b, hkv, split) serves all G = Hq/Hkv query heads of that
//     KV head, so each K/V byte fetched from HBM feeds G heads.
//   * W warps, each with R/W ring slots.  Warp w takes the split's pages w,
//     w + W, ...; for splits of 9..64 pages (2 or 3 warps) the warps instead
//     claim the next page from a counter in shared memory whenever a slot
//     is free, so a warp whose copies land late does not hold the split
//     back (the fp32 sums are then grouped by arrival order, which can vary
//     in the last bits from run to run).
//     A slot holds one (page, kv-head) tile: K and V, each one contiguous
//     4 KB run of its cache, copied by two bulk copies (TMA engine) that two
//     lanes issue in one instruction, completion counted on the slot's
//     mbarrier.  The warp refills a slot as soon as it has consumed it.
//   * QK: lane (tg, dq) owns tokens tg + j*TG and part dq of the head dim
//     for all G heads, with q resident in registers; each K row is read
//     from shared memory once, and the G lanes of a token group sum their
//     partial dot products by a butterfly reduce-scatter that leaves head
//     dq's scores on lane dq.  The lanes of a quarter-warp walk their row
//     parts in rotated orders (q held rotated the same way), so they read
//     different banks.  fp16 x fp16 -> fp32 FMAs (fma.rn.f32.f16): the
//     products are exact, no conversions.
//   * Online softmax in base 2 ([F2] §② exp2 trick) per head, rescaled
//     lazily (only when a page's max passes the running max by 8); p goes
//     through shared memory as [token][head] 16-bit values to the PV
//     product, where lane l owns dims [4l, 4l + 4) of every head, so each V
//     row is read once.
//   * CUDA cores only (the pages put tensor cores in the shared-prefix pass).
#include "common.cuh"
#include "kernels.h"
#include "split_range.h"

namespace skv {
namespace {

constexpr int kD = 128;
constexpr int kPage = 16;
constexpr int kTileBytes = kPage * kD * 2;   // one (page, kv-head) tile of K or of V
constexpr int kStageBytes = 2 * kTileBytes;  // K tile then V tile
constexpr unsigned kFull = 0xffffffffu;

struct DecodeParams {
    const uint16_t* q;  // fp16 or bf16 bit patterns
    const uint16_t* k_cache;
    const uint16_t* v_cache;
    const int32_t* block_table;
    const int32_t* ctx;
    float* o_part;
    float* lse_part;
    int32_t* ranges_dbg;
    unsigned long long* err;
    unsigned int* done_ctr;  // cascade chaining (DecodeArgs::done_ctr) or nullptr
    const int2* units;       // per-sequence split counts: the (sequence, split) list, or nullptr
    int32_t num_pool_pages, max_pages, B, Hq, Hkv, NS;  // NS: split-axis length of o_part
    float scale_log2;  // sm_scale * log2(e)
};

// Mixed-precision FMAs on 16-bit operand pairs: fp16 (BF = false) or bf16
// (BF = true) products, exact in fp32, added into fp32 accumulators.
#define SKV_MIXED_FMA(TY) "fma.rn.f32." TY
// acc += a.lo * b.lo + a.hi * b.hi.
template <bool BF>
SKV_DEVINL float dot2_h(uint32_t a, uint32_t b, float acc) {
#define SKV_DOT2(TY)                                                  \
    asm("{\n\t.reg .b16 a0, a1, b0, b1;\n\t"                         \
        "mov.b32 {a0, a1}, %1;\n\t"                                   \
        "mov.b32 {b0, b1}, %2;\n\t" SKV_MIXED_FMA(TY) " %0, a0, b0, %0;\n\t" \
        SKV_MIXED_FMA(TY) " %0, a1, b1, %0;\n\t}"                     \
        : "+f"(acc) : "r"(a), "r"(b))
    if constexpr (BF) SKV_DOT2("bf16");
    else SKV_DOT2("f16");
#undef SKV_DOT2
    return acc;
}
// acc += a.lo * b.lo (HI = false) or a.hi * b.hi.
template <bool BF, bool HI>
SKV_DEVINL float fma_h(uint32_t a, uint32_t b, float acc) {
#define SKV_FMA1(TY, X, Y)                                            \
    asm("{\n\t.reg .b16 a0, a1, b0, b1;\n\t"                         \
        "mov.b32 {a0, a1}, %1;\n\t"                                   \
        "mov.b32 {b0, b1}, %2;\n\t" SKV_MIXED_FMA(TY) " %0, " X ", " Y ", %0;\n\t}" \
        : "+f"(acc) : "r"(a), "r"(b))
    if constexpr (BF && HI) SKV_FMA1("bf16", "a1", "b1");
    else if constexpr (BF) SKV_FMA1("bf16", "a0", "b0");
    else if constexpr (HI) SKV_FMA1("f16", "a1", "b1");
    else SKV_FMA1("f16", "a0", "b0");
#undef SKV_FMA1
    return acc;
}
// (o0, o1) += p * (v.lo, v.hi) where p is the low (HI = false) or high half
// of `pw`.
template <bool BF, bool HI>
SKV_DEVINL void axpy2_h(uint32_t pw, uint32_t v, float& o0, float& o1) {
#define SKV_AXPY2(TY, P)                                              \
    asm("{\n\t.reg .b16 v0, v1, p0, p1;\n\t"                         \
        "mov.b32 {v0, v1}, %2;\n\t"                                   \
        "mov.b32 {p0, p1}, %3;\n\t" SKV_MIXED_FMA(TY) " %0, " P ", v0, %0;\n\t" \
        SKV_MIXED_FMA(TY) " %1, " P ", v1, %1;\n\t}"                  \
        : "+f"(o0), "+f"(o1) : "r"(v), "r"(pw))
    if constexpr (BF && HI) SKV_AXPY2("bf16", "p1");
    else if constexpr (BF) SKV_AXPY2("bf16", "p0");
    else if constexpr (HI) SKV_AXPY2("f16", "p1");
    else SKV_AXPY2("f16", "p0");
#undef SKV_AXPY2
}
#undef SKV_MIXED_FMA
// p rounded to the operand type (nearest even).
template <bool BF>
SKV_DEVINL uint16_t to_p(float x) {
    if constexpr (BF) return __bfloat16_as_ushort(__float2bfloat16_rn(x));
    else return __half_as_ushort(__float2half_rn(x));
}

// Lane roles.  G >= 2: lane = tg * G + dq.  In QK the lane owns the tokens
// tg + j*TG (j < TPL) and, for all G heads, the dims of part dq of the head
// dim (128/G dims: P chunks of 16 bytes), so each K row is read from shared
// memory once, by the G lanes of its token group; the group's partial dot
// products are summed by a butterfly reduce-scatter that leaves head dq's
// scores on lane dq.  In PV the lane owns dims [4*lane, 4*lane + 4) of all G
// heads, so each V row is read once, by the whole warp.  G == 1: QK lane =
// dh*16 + t (token t, half dh of the head dim); PV as for G >= 2.
template <int G> struct Roles {
    static_assert(G == 1 || G == 2 || G == 4 || G == 8, "group size");
    static constexpr int TG = G == 1 ? 16 : 32 / G;  // token groups in QK
    static constexpr int TPL = G == 1 ? 1 : G / 2;   // tokens per lane in QK
    static constexpr int P = G == 1 ? 8 : 16 / G;    // 16-byte chunks of the lane's K row part
    static constexpr int NC = G == 2 ? 4 : (G == 4 ? 2 : 1);  // FMA chains per (token, head)
    static constexpr int QW = G == 1 ? 32 : 64;      // q registers (16-bit pairs)
};

// Lazy rescale ([F2] §② exp2 form): the running max moves only when a page's
// max exceeds it by more than this many log2 units, so p = 2^(x - m) <= 2^8
// (exact in fp16 and bf16 range) and the accumulators are rescaled rarely.
constexpr float kLazyRescale = 8.f;

// Registers per lane for the page ids loaded before ctx is known (up to
// 32 * kSpecRegs table entries per warp).
constexpr int kSpecRegs = 4;

// The barriers take R words, rounded up to 16 bytes: the p buffer after them
// is read with 16-byte loads.
template <int R>
constexpr size_t bars_bytes() {
    return ((size_t)R * sizeof(uint64_t) + 15) / 16 * 16;
}

// Page ids of a split held in shared memory when its warps claim pages
// dynamically (at most kDynMaxPages pages per split), then the claim counter.
constexpr int kDynMaxPages = 64;

template <int G, int W, int R, bool DYN>
constexpr size_t smem_bytes() {
    return 128 /* alignment slack */ + (size_t)R * kStageBytes + bars_bytes<R>() +
           (size_t)W * G * kPage * sizeof(uint16_t) + (DYN ? (kDynMaxPages + 4) * sizeof(int) : 0);
}

template <int G, int W, int R, bool BF, bool DYN, bool VAR>
__global__ void __launch_bounds__(W * 32)
splitkv_decode_kernel(const DecodeParams p) {
    using Ro = Roles<G>;
    constexpr int TG = Ro::TG, TPL = Ro::TPL, P = Ro::P, NC = Ro::NC, QW = Ro::QW;
    constexpr int SPW = R / W;  // ring slots per warp
    static_assert(R % W == 0, "each warp owns R/W slots");
    static_assert(R * kStageBytes >= W * G * (kD + 2) * (int)sizeof(float),
                  "the cross-warp merge buffer reuses the ring");
    extern __shared__ uint8_t smem_raw[];
    // The ring starts on a 128-byte boundary (bulk copies need 16).  Offset
    // the shared pointer itself (an integer round trip would lose the shared
    // address space and turn every K/V read into a generic load).
    uint8_t* ring = smem_raw + ((128u - (smem_addr(smem_raw) & 127u)) & 127u);
    uint64_t* bars = reinterpret_cast<uint64_t*>(ring + R * kStageBytes);
    uint16_t* ps_all = reinterpret_cast<uint16_t*>(reinterpret_cast<uint8_t*>(bars) + bars_bytes<R>());
    int* dyn_ids = reinterpret_cast<int*>(ps_all + W * kPage * G);  // DYN: [kDynMaxPages], then the counter
    int* dyn_next = dyn_ids + kDynMaxPages;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // Uniform splits: CTA (hkv, split, b), the kv head fastest, so that the
    // CTAs reading the Hkv tiles of one page (one contiguous run of the
    // cache) start together.  Per-sequence splits (VAR): CTA u*Hkv + hkv
    // takes unit u of the list, sequence b's split `split` of ns.
    // (Separate instantiations: the uniform kernel keeps its registers.)
    int split, hkv, b, ns;
    if constexpr (VAR) {
        const int u = blockIdx.x / p.Hkv;
        hkv = blockIdx.x - u * p.Hkv;
        const int2 wi = __ldg(p.units + u);
        b = wi.x;
        split = wi.y & 0xffff;
        ns = wi.y >> 16;
        if (b < 0 || b >= p.B || ns < 1 || ns > p.NS || split >= ns) {
            if (threadIdx.x == 0 && hkv == 0) record_error(p.err, SKV_ERR_INVALID_ARG, 2 << 20 | u);
            pdl_launch_dependents();
            last_cta_waits_primary(p.done_ctr);
            return;
        }
    } else {
        hkv = blockIdx.x;
        split = blockIdx.y;
        b = blockIdx.z;
        ns = p.NS;
    }

    // The combine grid may be scheduled now; it waits for this grid to finish.
    pdl_launch_dependents();

    // Page ids are loaded before ctx is known, so that the two loads overlap
    // instead of following one another.  The split's first page is split *
    // pps with 1 <= pps <= pps_max (pps_max: a full page table).  When the
    // entries [split, (split + 1) * pps_max) that any ctx could select are
    // few, they are all loaded (lane l holds entry split + l + 32 i);
    // otherwise the ids of a full table's split are, and reloaded if ctx
    // turns out shorter.
    const int32_t* bt = p.block_table + (int64_t)b * p.max_pages;
    const int pps_max = (p.max_pages + ns - 1) / ns;
    const int ulo = split, uhi = min((split + 1) * pps_max, p.max_pages);
    const bool spec_union = uhi - ulo <= 32 * kSpecRegs;
    int spec[kSpecRegs];
    if constexpr (DYN) {
        // The split's pages are claimed by whichever warp is free: thread t
        // loads entry t of a full table's split (pps_max <= kDynMaxPages).
        const int e = split * pps_max + (int)threadIdx.x;
        spec[0] = ((int)threadIdx.x < pps_max && e < p.max_pages) ? bt[e] : 0;
    } else {
#pragma unroll
        for (int i = 0; i < kSpecRegs; ++i) {
            const int e = spec_union ? ulo + lane + 32 * i : (i == 0 ? split * pps_max + warp + lane * W : -1);
            spec[i] = (e >= 0 && e < uhi) ? bt[e] : 0;
        }
    }

    int ctx = p.ctx[b];
    const int cap = p.max_pages * kPage;
    if (ctx < 0 || ctx > cap) {
        if (threadIdx.x == 0 && split == 0 && hkv == 0) record_error(p.err, SKV_ERR_INVALID_ARG, b);
        ctx = ctx < 0 ? 0 : cap;
    }
    int p0, p1;
    split_page_range(ctx, kPage, ns, split, &p0, &p1);
    if (p.ranges_dbg != nullptr && hkv == 0 && threadIdx.x == 0) {
        p.ranges_dbg[((int64_t)b * p.NS + split) * 2 + 0] = p0;
        p.ranges_dbg[((int64_t)b * p.NS + split) * 2 + 1] = p1;
    }
    int npages = p1 > p0 ? p1 - p0 : 0;
    if constexpr (DYN) {
        // The shape was chosen for splits of at most kDynMaxPages pages; a
        // longer one (a split list planned for shorter contexts than ctx
        // holds) is flagged and cut, so no page id is read past the
        // shared-memory list.
        if (npages > kDynMaxPages) {
            if (threadIdx.x == 0) record_error(p.err, SKV_ERR_INVALID_ARG, 3 << 20 | b);
            npages = kDynMaxPages;
        }
    }
    const int nw = npages > warp ? (npages - warp + W - 1) / W : 0;  // this warp's pages

    if constexpr (DYN) {
        static_assert(W * 32 >= kDynMaxPages, "one page id per thread");
        const int t = threadIdx.x;
        if (t < kDynMaxPages) dyn_ids[t] = t < npages ? (p0 == split * pps_max ? spec[0] : bt[p0 + t]) : 0;
        if (t == 0) *dyn_next = 0;
    }
    if (threadIdx.x == 0) {
        for (int i = 0; i < R; ++i) mbar_init(&bars[i], 1);
        fence_mbar_init();
    }
    __syncthreads();

    const uint64_t pol = policy_evict_first();
    uint8_t* my_ring = ring + warp * SPW * kStageBytes;
    uint64_t* my_bars = bars + warp * SPW;
    // Page ids of this warp's pages k in [kb, kb + 32), one per lane: entry
    // p0 + warp + lane * W of the table row, from the speculative loads when
    // they hold it.
    int kb = 0;
    int my_id = 0;
    if constexpr (!DYN) {
        const int e = p0 + warp + lane * W;
        if (spec_union) {
            // e lies in [ulo, uhi) for lane < nw (p0 >= split, e < p1).
            const int off = lane < nw ? e - ulo : 0;
#pragma unroll
            for (int i = 0; i < kSpecRegs; ++i) {
                const int v = __shfl_sync(kFull, spec[i], off & 31);
                my_id = (off >> 5) == i ? v : my_id;
            }
        } else if (p0 == split * pps_max) {
            my_id = spec[0];
        } else if (lane < nw) {
            my_id = bt[e];
        }
    }
    // DYN: page index of each of the warp's ring slots (claimed dynamically).
    int claimed[SPW];
#pragma unroll
    for (int i = 0; i < SPW; ++i) claimed[i] = 0;
    // Issues the copies of the warp's k-th page into slot k % SPW; with DYN
    // the page is first claimed from the split's counter, and false is
    // returned (nothing issued) once every page is taken.
    auto issue = [&](int k) -> bool {  // warp-uniform call; lanes 0 and 1 issue the copies
        int pid;
        if constexpr (DYN) {
            int j = 0;
            if (lane == 0) j = atomicAdd(dyn_next, 1);
            j = __shfl_sync(kFull, j, 0);
            if (j >= npages) return false;
#pragma unroll
            for (int i = 0; i < SPW; ++i)
                if (i == k % SPW) claimed[i] = j;
            pid = dyn_ids[j];
        } else {
            if (k - kb >= 32) {
                kb += 32;
                my_id = (kb + lane < nw) ? bt[p0 + warp + (kb + lane) * W] : 0;
            }
            pid = __shfl_sync(kFull, my_id, k - kb);
        }
        if ((unsigned)pid >= (unsigned)p.num_pool_pages) {
            if (lane == 0) record_error(p.err, SKV_ERR_INVALID_ARG, 1 << 20 | b);
            pid = 0;
        }
        const int slot = k % SPW;
        uint64_t* bar = &my_bars[slot];
        uint8_t* dst = my_ring + slot * kStageBytes;
        const int64_t row = ((int64_t)pid * p.Hkv + hkv) * kPage;  // first row of the tile
        if (lane == 0) mbar_arrive_expect_tx(bar, kStageBytes);
        __syncwarp();
        // The K and V tiles are each one contiguous 4 KB run of the cache:
        // two bulk copies, issued by two lanes in one instruction (one thread
        // issuing its copies back to back is held up by the copy engine).
        if (lane < 2)
            bulk_g2s(dst + lane * kTileBytes, (lane == 0 ? p.k_cache : p.v_cache) + row * kD,
                     kTileBytes, bar, pol);
        return true;
    };
    // Pages of this warp issued so far: static, pages warp, warp + W, ...
    // (nw of them); DYN, as many as it has claimed.
    int nseq = 0;
#pragma unroll 1
    while (nseq < SPW && (DYN || nseq < nw) && issue(nseq)) ++nseq;

    // q pinned in registers for the whole split, as 16-bit pairs, loaded
    // while the first pages are in flight.  G == 1: the 64 dims of the
    // lane's half dh, 16-byte chunk i in register chunk (i - r) mod 8, r =
    // the lane's token.  G >= 2: for each head h the P chunks of part dq,
    // chunk c of the part in register chunk (c - r) mod P, r the lane's
    // rotation (below).
    const int tg = G == 1 ? (lane & 15) : lane / G;
    const int dq = G == 1 ? (lane >> 4) : lane % G;
    // Rotation of the lane's walk over its K row part: the 8 lanes of a
    // quarter-warp then read 8 different 16-byte bank groups.
    const int rot = G == 1 ? (lane & 7) : (lane / (G / 2)) % P;
    uint32_t qh[QW];
    if (npages > 0) {  // an empty split reads no q
        const uint16_t* qbase = p.q + ((int64_t)b * p.Hq + hkv * G) * kD;
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
            for (int i = 0; i < P; ++i) {
                const int c = (i + rot) & (P - 1);
                const uint4 a = ld_pinned(qbase + h * kD + dq * (kD / (G == 1 ? 2 : G)) + 8 * c);
                qh[(h * P + i) * 4 + 0] = a.x; qh[(h * P + i) * 4 + 1] = a.y;
                qh[(h * P + i) * 4 + 2] = a.z; qh[(h * P + i) * 4 + 3] = a.w;
            }
    }

    float o[G][4];  // PV: head h, dims [4*lane, 4*lane + 4)
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
        for (int i = 0; i < 4; ++i) o[h][i] = 0.f;
    float m_run = -INFINITY;  // running max (log2 units) of the lane's QK head
    float l_run = 0.f;        // the lane's share of that head's running sum
    uint16_t* ps = ps_all + warp * (kPage * G);  // p[token][head], 16-bit

#pragma unroll 1
    for (int k = 0; k < nseq; ++k) {
        const int slot = k % SPW;
        const bool ok = mbar_wait(&my_bars[slot], (uint32_t)((k / SPW) & 1), p.err, 2);
        if (!__all_sync(kFull, ok)) {
            // A bounded wait gave up (error recorded).  Give the copies this
            // warp still has in flight one more bounded wait each before the
            // ring is reused, then stop.
            for (int kk = k + 1; kk < nseq; ++kk)
                mbar_wait(&my_bars[kk % SPW], (uint32_t)((kk / SPW) & 1), p.err, 3);
            break;
        }
        int pj = warp + k * W;  // index of the page in the split
        if constexpr (DYN) {
#pragma unroll
            for (int i = 0; i < SPW; ++i)
                if (i == slot) pj = claimed[i];
        }
        const int nvalid = min(kPage, ctx - (p0 + pj) * kPage);  // >= 1
        const uint8_t* Kb = my_ring + slot * kStageBytes;
        const uint8_t* Vs = Kb + kTileBytes;

        // ---- scores of the lane's tokens for its QK head (log2 units, masked)
        float x[TPL];
        if constexpr (G == 1) {
            const uint8_t* rowp = Kb + tg * (kD * 2) + dq * 128;
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const uint4 kv = *reinterpret_cast<const uint4*>(rowp + (((c + rot) & 7) << 4));
                acc[c & 3] = dot2_h<BF>(qh[4 * c + 0], kv.x, acc[c & 3]);
                acc[c & 3] = dot2_h<BF>(qh[4 * c + 1], kv.y, acc[c & 3]);
                acc[c & 3] = dot2_h<BF>(qh[4 * c + 2], kv.z, acc[c & 3]);
                acc[c & 3] = dot2_h<BF>(qh[4 * c + 3], kv.w, acc[c & 3]);
            }
            float sc = (acc[0] + acc[1]) + (acc[2] + acc[3]);
            sc += __shfl_xor_sync(kFull, sc, 16);
            x[0] = tg < nvalid ? sc * p.scale_log2 : -INFINITY;
        } else {
            // Partial dot products over part dq for every (token j, head h),
            // NC independent FMA chains each (low and high 16-bit halves,
            // and for G = 2 even and odd words, apart).
            float acc[TPL][G][NC];
#pragma unroll
            for (int j = 0; j < TPL; ++j)
#pragma unroll
                for (int h = 0; h < G; ++h)
#pragma unroll
                    for (int c = 0; c < NC; ++c) acc[j][h][c] = 0.f;
#pragma unroll
            for (int i = 0; i < P; ++i) {
                uint4 kv[TPL];
#pragma unroll
                for (int j = 0; j < TPL; ++j)
                    kv[j] = *reinterpret_cast<const uint4*>(
                        Kb + (tg + j * TG) * (kD * 2) + ((dq * P + ((i + rot) & (P - 1))) << 4));
#pragma unroll
                for (int j = 0; j < TPL; ++j) {
                    const uint32_t kw[4] = {kv[j].x, kv[j].y, kv[j].z, kv[j].w};
#pragma unroll
                    for (int h = 0; h < G; ++h)
#pragma unroll
                        for (int w = 0; w < 4; ++w) {
                            const uint32_t qw = qh[(h * P + i) * 4 + w];
                            float& a0 = acc[j][h][(2 * w) % NC];
                            a0 = fma_h<BF, false>(qw, kw[w], a0);
                            float& a1 = acc[j][h][(2 * w + 1) % NC];
                            a1 = fma_h<BF, true>(qw, kw[w], a1);
                        }
                }
            }
#pragma unroll
            for (int j = 0; j < TPL; ++j) {
                float cur[G];
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    float s = acc[j][h][0];
#pragma unroll
                    for (int c = 1; c < NC; ++c) s += acc[j][h][c];
                    cur[h] = s;
                }
                // Reduce-scatter over the G lanes of the token group: at step
                // m the lane keeps the half of its heads whose bit m matches
                // its own and sends the other half to lane ^ m.
#pragma unroll
                for (int m = G / 2; m >= 1; m >>= 1) {
                    const bool up = (dq & m) != 0;
#pragma unroll
                    for (int kk = 0; kk < m; ++kk) {
                        const float send = up ? cur[kk] : cur[kk + m];
                        const float keep = up ? cur[kk + m] : cur[kk];
                        cur[kk] = keep + __shfl_xor_sync(kFull, send, m);
                    }
                }
                x[j] = tg + j * TG < nvalid ? cur[0] * p.scale_log2 : -INFINITY;
            }
        }

        // ---- online softmax of the lane's QK head (its lanes agree on m),
        // lazily rescaled
        constexpr int MLO = G == 1 ? 1 : G, MHI = G == 1 ? 16 : 32;  // lanes of one head
        float mx = x[0];
#pragma unroll
        for (int j = 1; j < TPL; ++j) mx = fmaxf(mx, x[j]);
#pragma unroll
        for (int mm = MLO; mm < MHI; mm <<= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, mm));
        // mx is finite: token 0 of the page is valid.
        const bool need = mx > m_run + kLazyRescale;
        const float m_new = need ? mx : m_run;
        const float alpha = need ? exp2f(m_run - m_new) : 1.f;
        float psum = 0.f;
#pragma unroll
        for (int j = 0; j < TPL; ++j) {
            const float pj = exp2f(x[j] - m_new);
            psum += pj;
            if constexpr (G == 1) {
                if (lane < 16) ps[lane] = to_p<BF>(pj);
            } else {
                ps[(tg + j * TG) * G + dq] = to_p<BF>(pj);
            }
        }
        l_run = fmaf(l_run, alpha, psum);
        m_run = m_new;
        if (__any_sync(kFull, need)) {
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const float a = G == 1 ? alpha : __shfl_sync(kFull, alpha, h);  // lane h: head h
#pragma unroll
                for (int i = 0; i < 4; ++i) o[h][i] *= a;
            }
        }
        __syncwarp();

        // ---- o += p V: head h, dims [4*lane, 4*lane + 4)
        auto pv_token = [&](int t) {
            uint32_t pw[(G + 1) / 2];
            if constexpr (G == 1) {
                pw[0] = ps[t];
            } else if constexpr (G == 2) {
                pw[0] = *reinterpret_cast<const uint32_t*>(ps + t * G);
            } else if constexpr (G == 4) {
                const uint2 a = *reinterpret_cast<const uint2*>(ps + t * G);
                pw[0] = a.x; pw[1] = a.y;
            } else {
                const uint4 a = *reinterpret_cast<const uint4*>(ps + t * G);
                pw[0] = a.x; pw[1] = a.y; pw[2] = a.z; pw[3] = a.w;
            }
            const uint2 vv = *reinterpret_cast<const uint2*>(Vs + t * (kD * 2) + 8 * lane);
#pragma unroll
            for (int h = 0; h < G; ++h) {
                if (h & 1) {
                    axpy2_h<BF, true>(pw[h >> 1], vv.x, o[h][0], o[h][1]);
                    axpy2_h<BF, true>(pw[h >> 1], vv.y, o[h][2], o[h][3]);
                } else {
                    axpy2_h<BF, false>(pw[h >> 1], vv.x, o[h][0], o[h][1]);
                    axpy2_h<BF, false>(pw[h >> 1], vv.y, o[h][2], o[h][3]);
                }
            }
        };
        if (nvalid == kPage) {
#pragma unroll
            for (int t = 0; t < kPage; ++t) pv_token(t);
        } else {
            // Partial last page: tokens past ctx are never read (p = 0 must
            // not meet a stale value).
#pragma unroll
            for (int t = 0; t < kPage; ++t)
                if (t < nvalid) pv_token(t);
        }
        __syncwarp();  // slot and p buffer fully read
        if ((DYN || k + SPW < nw) && issue(k + SPW)) ++nseq;  // refills this slot (nseq == k + SPW)
    }

    // This warp's per-head totals: l over the lanes of the head.
#pragma unroll
    for (int mm = (G == 1 ? 1 : G); mm < (G == 1 ? 16 : 32); mm <<= 1)
        l_run += __shfl_xor_sync(kFull, l_run, mm);

    if constexpr (W == 1) {
        // One warp: its state is the split's.  Lane h holds head h's m and
        // l; lane l writes dims [4l, 4l + 4) of every head (an empty split
        // ends as o = 0, lse = -inf, [L3] §④).
#pragma unroll
        for (int h = 0; h < G; ++h) {
            const float M = __shfl_sync(kFull, m_run, G == 1 ? 0 : h);
            const float L = __shfl_sync(kFull, l_run, G == 1 ? 0 : h);
            const float inv = L > 0.f ? 1.f / L : 0.f;
            const int64_t row = ((int64_t)b * p.Hq + hkv * G + h) * p.NS + split;
            *reinterpret_cast<float4*>(p.o_part + row * kD + 4 * lane) =
                make_float4(o[h][0] * inv, o[h][1] * inv, o[h][2] * inv, o[h][3] * inv);
            if (lane == 0) p.lse_part[row] = L > 0.f ? M + log2f(L) : -INFINITY;
        }
    } else {
        __syncthreads();  // every warp is done with its ring: reuse it
        float* wo = reinterpret_cast<float*>(ring);  // [W][G][kD]
        float* wm = wo + W * G * kD;                 // [W][G]
        float* wl = wm + W * G;                      // [W][G]
#pragma unroll
        for (int h = 0; h < G; ++h)
            *reinterpret_cast<float4*>(wo + (warp * G + h) * kD + 4 * lane) =
                make_float4(o[h][0], o[h][1], o[h][2], o[h][3]);
        if (lane < G) {  // lane h holds head h's m and l
            wm[warp * G + lane] = m_run;
            wl[warp * G + lane] = l_run;
        }
        __syncthreads();
        // Merge the W warp states of each head ([F2] §③ over W states) and write
        // the split state; an empty split ends as o = 0, lse = -inf ([L3] §④).
        for (int idx = threadIdx.x; idx < G * (kD / 4); idx += W * 32) {
            const int g = idx / (kD / 4), d4 = idx % (kD / 4);
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < W; ++w) M = fmaxf(M, wm[w * G + g]);
            float L = 0.f;
            float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int w = 0; w < W; ++w) {
                const float sc = merge_weight(wm[w * G + g], M);
                L = fmaf(sc, wl[w * G + g], L);
                const float4 t4 = *reinterpret_cast<const float4*>(wo + (w * G + g) * kD + 4 * d4);
                a.x = fmaf(sc, t4.x, a.x); a.y = fmaf(sc, t4.y, a.y);
                a.z = fmaf(sc, t4.z, a.z); a.w = fmaf(sc, t4.w, a.w);
            }
            const float inv = L > 0.f ? 1.f / L : 0.f;
            const int64_t row = ((int64_t)b * p.Hq + hkv * G + g) * p.NS + split;
            *reinterpret_cast<float4*>(p.o_part + row * kD + 4 * d4) =
                make_float4(a.x * inv, a.y * inv, a.z * inv, a.w * inv);
            if (d4 == 0) p.lse_part[row] = L > 0.f ? M + log2f(L) : -INFINITY;
        }
    }
    last_cta_waits_primary(p.done_ctr);
}

template <int G, int W, int R, bool BF, bool DYN, bool VAR>
cudaError_t launch_gwr_t(const DecodeParams& p, int B, int Hkv, int NS, int num_units,
                         cudaStream_t st) {
    constexpr size_t smem = smem_bytes<G, W, R, DYN>();
    auto kern = splitkv_decode_kernel<G, W, R, BF, DYN, VAR>;
    static bool attr_set[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 64 && !attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = VAR ? dim3((unsigned)num_units * (unsigned)Hkv, 1, 1) : dim3(Hkv, NS, B);
    cfg.blockDim = dim3(W * 32, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = p.done_ctr != nullptr ? 1 : 0;  // chained after a prefix pass
    return cudaLaunchKernelEx(&cfg, kern, p);
}

template <int G, int W, int R, bool BF, bool DYN = false>
cudaError_t launch_gwr(const DecodeParams& p, int B, int Hkv, int NS, int num_units,
                       cudaStream_t st) {
    return p.units != nullptr ? launch_gwr_t<G, W, R, BF, DYN, true>(p, B, Hkv, NS, num_units, st)
                              : launch_gwr_t<G, W, R, BF, DYN, false>(p, B, Hkv, NS, num_units, st);
}

// Warps per CTA follow the longest possible split (the page table's width
// over NUM_SPLITS): a CTA of 3 warps with a 6-page ring for long splits; for
// short splits smaller CTAs, so that many more of them are resident per SM
// and their fixed latencies (q, page table, first copies) overlap.
template <int G, bool BF>
cudaError_t launch_g(const DecodeParams& p, int B, int Hkv, int NS, int num_units,
                     int pps, cudaStream_t st) {
    // Measured on the cascade suffixes (<= 8 pages per split, B=64, NS=16):
    // pass 1 takes 53 us with 1 warp and a 2-page ring (about 13 CTAs per
    // SM), 64 us with 2 warps, 72 us with 3; a 4-page ring for the 1-warp
    // CTA (fewer CTAs per SM) takes 74 us.  On long splits (32 pages, B=1,
    // NS=64) 3 warps with a 6-page ring, 2 with 6 and 2 with 4 are level
    // (27.6-28.0 us): the pages in flight per SM, not the warps, set the
    // pace there; 1 warp with 4 takes 33 us.
    // Splits of 9..kDynMaxPages pages: the warps claim pages one at a time
    // from the split's counter (DYN), so that a warp whose copies land late
    // does not hold the split back while its neighbours idle (long context,
    // 32 pages: 30.5-30.9 -> 29.5-29.7 us for the decode).
    if (pps <= 8) return launch_gwr<G, 1, 2, BF>(p, B, Hkv, NS, num_units, st);
    if (pps <= 16) return launch_gwr<G, 2, 4, BF, true>(p, B, Hkv, NS, num_units, st);
    if (pps <= kDynMaxPages) return launch_gwr<G, 3, 6, BF, true>(p, B, Hkv, NS, num_units, st);
    return launch_gwr<G, 3, 6, BF>(p, B, Hkv, NS, num_units, st);
}

// ---------------------------------------------------------------- combine (pass 2)
// [L3] §③ merge of the split states (base 2).  For the cascade ([F2] §⑥) the
// prefix-chunk states are merged first into the prefix state, which is then
// merged with the merged split state by the two-state formula (prefix first).
// WPR warps per (b, hq) row (1 for many rows, 4 for few rows); within a row,
// warp w takes states w, w + WPR, ...; lane l owns dims [4l, 4l + 4).  A
// warp requests the lse and v chunk of up to kCombBatch states at once (one
// L2 round trip per batch), keeps an online (m, W, acc) across batches, and
// with WPR > 1 the warp states meet in shared memory.
constexpr int kCombWarps = 4;
constexpr int kCombBatch = 16;

struct CombineParams {
    const float* o_part;   // [rows, NS, D]
    const float* lse_part; // [rows, NS]
    const int32_t* seq_splits;  // [rows / Hq] states per row, or nullptr (NS each)
    unsigned long long* err;
    void* out;             // [rows, D] Tout
    float* lse_out;        // [rows] or nullptr
    const float* pre_part; // [rows, C, D] prefix-chunk states or nullptr
    const float* pre_lse;  // [rows, C]
    float* o_pre;          // [rows, D] merged prefix state or nullptr
    float* s_pre;          // [rows]
    int64_t rows;
    int NS, C, D, Hq;
};

// States of `row` (at most NS): its sequence's split count with per-sequence
// splits (a count outside [1, NS] is flagged and clamped), else NS.
template <bool VAR>
SKV_DEVINL int row_splits(const CombineParams& p, int64_t row) {
    if (!VAR) return p.NS;
    const int b = (int)row / p.Hq;  // rows = B * Hq < 2^31
    const int n = __ldg(p.seq_splits + b);
    if (n < 1 || n > p.NS) {
        if ((threadIdx.x & 31) == 0) record_error(p.err, SKV_ERR_INVALID_ARG, 4 << 20 | b);
        return n < 1 ? 1 : p.NS;
    }
    return n;
}

struct WarpState {
    float m, W;
    float4 acc;
};

// This warp's share (states sub, sub + WPR, ...) of the first N of the
// `stride` states of `row`.
// Per batch of kCombBatch states: lane k (and lane k + 16) reads state k's
// lse and computes its weight, the batch max and weight sum go through
// shuffles, and every lane then accumulates its 4 dims of the batch's v rows
// with the weights broadcast from their lanes.
template <int WPR, int BATCH = kCombBatch>
SKV_DEVINL WarpState warp_merge(const float* o, const float* lse, int stride, int N, int D,
                                int64_t row, int sub) {
    static_assert(BATCH == 8 || BATCH == 16, "lanes k, k + BATCH, ... read state k of a batch");
    const int lane = threadIdx.x & 31;
    const bool has = 4 * lane < D;
    WarpState st{-INFINITY, 0.f, make_float4(0.f, 0.f, 0.f, 0.f)};
    for (int n0 = sub; n0 < N; n0 += WPR * BATCH) {
        const int nk = n0 + (lane & (BATCH - 1)) * WPR;
        const float lk = nk < N ? sanitize_lse(__ldcg(lse + row * stride + nk)) : -INFINITY;
        float4 x[BATCH];
#pragma unroll
        for (int k = 0; k < BATCH; ++k) {
            const int n = n0 + k * WPR;
            x[k] = (n < N && has) ? __ldcg(reinterpret_cast<const float4*>(o + (row * stride + n) * D) + lane)
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        float mb = lk;
#pragma unroll
        for (int mm = 1; mm < BATCH; mm <<= 1) mb = fmaxf(mb, __shfl_xor_sync(kFull, mb, mm));
        mb = fmaxf(mb, st.m);
        const float wk = merge_weight(lk, mb);
        float ws = wk;
#pragma unroll
        for (int mm = 1; mm < BATCH; mm <<= 1) ws += __shfl_xor_sync(kFull, ws, mm);
        const float sc = merge_weight(st.m, mb);  // rescale of the running state
        st.W = fmaf(st.W, sc, ws);
        st.acc.x *= sc; st.acc.y *= sc; st.acc.z *= sc; st.acc.w *= sc;
#pragma unroll
        for (int k = 0; k < BATCH; ++k) {
            const float w = __shfl_sync(kFull, wk, k);
            if (w > 0.f) {  // a zero-weight state is not read into the result
                st.acc.x = fmaf(w, x[k].x, st.acc.x); st.acc.y = fmaf(w, x[k].y, st.acc.y);
                st.acc.z = fmaf(w, x[k].z, st.acc.z); st.acc.w = fmaf(w, x[k].w, st.acc.w);
            }
        }
        st.m = mb;
    }
    return st;
}

struct CombSmem {
    float wm[kCombWarps], wW[kCombWarps];
    __align__(16) float wacc[kCombWarps][kD];
};

// Merged state of `row` over the first N of its `stride` states: v (this
// lane's 4 dims) and s.  With WPR > 1 every thread of the CTA must call this
// (block barriers).
template <int WPR, int BATCH = kCombBatch>
SKV_DEVINL void merge_row(const float* o, const float* lse, int stride, int N, int D,
                          int64_t row, int sub, CombSmem& sm, float (&v)[4], float& s_out) {
    WarpState st = warp_merge<WPR, BATCH>(o, lse, stride, N, D, row, sub);
    if constexpr (WPR > 1) {
        const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
        __syncthreads();  // the buffers may still be read from a previous merge
        if (lane == 0) {
            sm.wm[w] = st.m;
            sm.wW[w] = st.W;
        }
        if (4 * lane < D) *reinterpret_cast<float4*>(&sm.wacc[w][4 * lane]) = st.acc;
        __syncthreads();
        float M = sm.wm[0];
#pragma unroll
        for (int i = 1; i < WPR; ++i) M = fmaxf(M, sm.wm[i]);
        float WW = 0.f;
        float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int i = 0; i < WPR; ++i) {
            const float sc = merge_weight(sm.wm[i], M);
            WW = fmaf(sc, sm.wW[i], WW);
            if (4 * lane < D) {
                const float4 t = *reinterpret_cast<const float4*>(&sm.wacc[i][4 * lane]);
                a.x = fmaf(sc, t.x, a.x); a.y = fmaf(sc, t.y, a.y);
                a.z = fmaf(sc, t.z, a.z); a.w = fmaf(sc, t.w, a.w);
            }
        }
        st.m = M;
        st.W = WW;
        st.acc = a;
    }
    const float inv = st.W > 0.f ? 1.f / st.W : 0.f;
    v[0] = st.acc.x * inv; v[1] = st.acc.y * inv; v[2] = st.acc.z * inv; v[3] = st.acc.w * inv;
    s_out = st.m + log2f(st.W);  // -inf when every state is empty
}

template <typename Tout, int WPR, bool VAR>
__global__ void __launch_bounds__(kCombWarps * 32)
combine_kernel(const CombineParams p) {
    pdl_wait_primary();  // the states are written by the preceding grids
    __shared__ CombSmem sm;
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr int kRowsPerCta = kCombWarps / WPR;
    const int64_t row_raw = (int64_t)blockIdx.x * kRowsPerCta + w / WPR;
    const bool row_ok = row_raw < p.rows;
    const int64_t row = row_ok ? row_raw : p.rows - 1;  // keep every warp on the barriers
    const int sub = w % WPR;
    const bool has = 4 * lane < p.D;
    float vd[4], sd;
    merge_row<WPR>(p.o_part, p.lse_part, p.NS, row_splits<VAR>(p, row), p.D, row, sub, sm, vd, sd);
    if (p.pre_part != nullptr) {
        float vp[4] = {0.f, 0.f, 0.f, 0.f}, sp = -INFINITY;  // empty prefix when C == 0
        if (p.C > 0) merge_row<WPR>(p.pre_part, p.pre_lse, p.C, p.C, p.D, row, sub, sm, vp, sp);
        if (sub == 0 && row_ok) {
            if (p.o_pre != nullptr && has)
                *reinterpret_cast<float4*>(p.o_pre + row * p.D + 4 * lane) =
                    make_float4(vp[0], vp[1], vp[2], vp[3]);
            if (p.s_pre != nullptr && lane == 0) p.s_pre[row] = sp;
        }
        // Two-state merge, prefix first ([F2] §③, guards of §⑤ and [FA] §2.2).
        const float se = sanitize_lse(sp), sb = sanitize_lse(sd);
        const float mm = fmaxf(se, sb);
        const float we = merge_weight(se, mm), wb = merge_weight(sb, mm);
        const float ws = __fadd_rn(we, wb);
        const float iv = ws > 0.f ? 1.f / ws : 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float te = we > 0.f ? __fmul_rn(we, vp[i]) : 0.f;
            const float tb = wb > 0.f ? __fmul_rn(wb, vd[i]) : 0.f;
            vd[i] = __fmul_rn(__fadd_rn(te, tb), iv);
        }
        sd = mm + log2f(ws);
    }
    if (sub != 0 || !row_ok) return;
    if (lane == 0 && p.lse_out != nullptr) p.lse_out[row] = sd;
    // Lane l holds dims [4l, 4l + 4): write them in the output dtype.
    constexpr int EO = Vec<Tout>::N;
    char* orow = reinterpret_cast<char*>(p.out) + row * p.D * (int64_t)sizeof(Tout);
    if constexpr (EO == 4) {
        if (has) *reinterpret_cast<float4*>(orow + lane * 16) = make_float4(vd[0], vd[1], vd[2], vd[3]);
    } else {
        // Two lanes form one 16-byte chunk of 8 elements.
        float f[8];
        const float o0 = __shfl_down_sync(0xffffffffu, vd[0], 1);
        const float o1 = __shfl_down_sync(0xffffffffu, vd[1], 1);
        const float o2 = __shfl_down_sync(0xffffffffu, vd[2], 1);
        const float o3 = __shfl_down_sync(0xffffffffu, vd[3], 1);
        f[0] = vd[0]; f[1] = vd[1]; f[2] = vd[2]; f[3] = vd[3];
        f[4] = o0; f[5] = o1; f[6] = o2; f[7] = o3;
        if ((lane & 1) == 0 && 4 * lane < p.D) st_stream(orow + lane * 8, from_float<Tout>(f));
    }
}

// States a warp of the cascade combine requests per L2 round trip: 8 keeps
// the kernel under 64 registers, so that all of its CTAs are resident at once.
constexpr int kCascadeBatch = 8;

// Cascade combine with many rows: two warps per row, so that the row's two
// lists are read at once -- warp 0 merges the suffix's split states, warp 1
// the prefix chunks' states into the prefix state (written to o_pre/s_pre)
// -- and they meet in shared memory for the two-state merge, prefix first.
template <typename Tout, bool VAR>
__global__ void __launch_bounds__(kCombWarps * 32, 8)
cascade_combine_kernel(const CombineParams p) {
    pdl_wait_primary();  // the states are written by the preceding grids
    __shared__ CombSmem sm;  // unused by merge_row<1>
    __shared__ __align__(16) float pre_v[kCombWarps / 2][kD];
    __shared__ float pre_s[kCombWarps / 2];
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int sub = w & 1, slot = w >> 1;
    const int64_t row_raw = (int64_t)blockIdx.x * (kCombWarps / 2) + slot;
    const bool row_ok = row_raw < p.rows;
    const int64_t row = row_ok ? row_raw : p.rows - 1;  // every warp reaches the barrier
    const bool has = 4 * lane < p.D;
    float v[4] = {0.f, 0.f, 0.f, 0.f}, s = -INFINITY;
    if (sub == 0) {
        merge_row<1, kCascadeBatch>(p.o_part, p.lse_part, p.NS, row_splits<VAR>(p, row), p.D, row, 0,
                                    sm, v, s);
    } else {
        if (p.C > 0)
            merge_row<1, kCascadeBatch>(p.pre_part, p.pre_lse, p.C, p.C, p.D, row, 0, sm, v, s);
        if (row_ok) {
            if (p.o_pre != nullptr && has)
                *reinterpret_cast<float4*>(p.o_pre + row * p.D + 4 * lane) = make_float4(v[0], v[1], v[2], v[3]);
            if (p.s_pre != nullptr && lane == 0) p.s_pre[row] = s;
        }
        if (has) *reinterpret_cast<float4*>(&pre_v[slot][4 * lane]) = make_float4(v[0], v[1], v[2], v[3]);
        if (lane == 0) pre_s[slot] = s;
    }
    __syncthreads();
    if (sub != 0 || !row_ok) return;
    float vp[4] = {0.f, 0.f, 0.f, 0.f};
    if (has) {
        const float4 t = *reinterpret_cast<const float4*>(&pre_v[slot][4 * lane]);
        vp[0] = t.x; vp[1] = t.y; vp[2] = t.z; vp[3] = t.w;
    }
    // Two-state merge, prefix first ([F2] §③, guards of §⑤ and [FA] §2.2).
    const float se = sanitize_lse(pre_s[slot]), sb = sanitize_lse(s);
    const float mm = fmaxf(se, sb);
    const float we = merge_weight(se, mm), wb = merge_weight(sb, mm);
    const float ws = __fadd_rn(we, wb);
    const float iv = ws > 0.f ? 1.f / ws : 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float te = we > 0.f ? __fmul_rn(we, vp[i]) : 0.f;
        const float tb = wb > 0.f ? __fmul_rn(wb, v[i]) : 0.f;
        v[i] = __fmul_rn(__fadd_rn(te, tb), iv);
    }
    const float so = mm + log2f(ws);
    if (lane == 0 && p.lse_out != nullptr) p.lse_out[row] = so;
    constexpr int EO = Vec<Tout>::N;
    char* orow = reinterpret_cast<char*>(p.out) + row * p.D * (int64_t)sizeof(Tout);
    if constexpr (EO == 4) {
        if (has) *reinterpret_cast<float4*>(orow + lane * 16) = make_float4(v[0], v[1], v[2], v[3]);
    } else {
        float f[8];
        const float o0 = __shfl_down_sync(0xffffffffu, v[0], 1);
        const float o1 = __shfl_down_sync(0xffffffffu, v[1], 1);
        const float o2 = __shfl_down_sync(0xffffffffu, v[2], 1);
        const float o3 = __shfl_down_sync(0xffffffffu, v[3], 1);
        f[0] = v[0]; f[1] = v[1]; f[2] = v[2]; f[3] = v[3];
        f[4] = o0; f[5] = o1; f[6] = o2; f[7] = o3;
        if ((lane & 1) == 0 && 4 * lane < p.D) st_stream(orow + lane * 8, from_float<Tout>(f));
    }
}

}  // namespace

cudaError_t launch_splitkv_decode(const DecodeArgs& a, const DeviceInfo& dev, cudaStream_t st) {
    DecodeParams p;
    p.q = static_cast<const uint16_t*>(a.q);
    p.k_cache = static_cast<const uint16_t*>(a.k_cache);
    p.v_cache = static_cast<const uint16_t*>(a.v_cache);
    p.block_table = a.block_table;
    p.ctx = a.ctx;
    p.o_part = a.o_part;
    p.lse_part = a.lse_part;
    p.ranges_dbg = a.ranges_dbg;
    p.err = dev.err;
    p.done_ctr = a.done_ctr;
    p.units = reinterpret_cast<const int2*>(a.units);
    p.num_pool_pages = a.num_pool_pages;
    p.max_pages = a.max_pages;
    p.B = a.B;
    p.Hq = a.Hq;
    p.Hkv = a.Hkv;
    p.NS = a.num_splits;
    p.scale_log2 = a.sm_scale * 1.4426950408889634f;
    // The CTA shape follows the longest split: the page table's width over
    // the split count, or the longest split of the per-sequence list.
    if (a.units != nullptr && a.num_units < 1) return cudaErrorInvalidValue;
    const int pps = a.units != nullptr ? a.max_split_pages
                                       : (a.max_pages + a.num_splits - 1) / a.num_splits;
#define SKV_LAUNCH_G(BF_)                                                             \
    switch (a.Hq / a.Hkv) {                                                           \
        case 1: return launch_g<1, BF_>(p, a.B, a.Hkv, a.num_splits, a.num_units, pps, st); \
        case 2: return launch_g<2, BF_>(p, a.B, a.Hkv, a.num_splits, a.num_units, pps, st); \
        case 4: return launch_g<4, BF_>(p, a.B, a.Hkv, a.num_splits, a.num_units, pps, st); \
        case 8: return launch_g<8, BF_>(p, a.B, a.Hkv, a.num_splits, a.num_units, pps, st); \
    }
    if (a.bf16) SKV_LAUNCH_G(true) else SKV_LAUNCH_G(false)
#undef SKV_LAUNCH_G
    return cudaErrorInvalidValue;
}

}  // namespace skv

namespace skv {

cudaError_t launch_combine(const CombineArgs& a, bool pdl, const DeviceInfo& dev, cudaStream_t st) {
    if (a.D > kD || a.D % 8 != 0) return cudaErrorInvalidValue;
    CombineParams p;
    p.o_part = a.o_part;
    p.lse_part = a.lse_part;
    p.seq_splits = a.seq_splits;
    p.err = dev.err;
    p.Hq = a.Hq > 0 ? a.Hq : 1;
    p.out = a.out;
    p.lse_out = a.lse_out;
    p.pre_part = a.pre_part;
    p.pre_lse = a.pre_lse;
    p.o_pre = a.o_pre;
    p.s_pre = a.s_pre;
    p.NS = a.NS;
    p.C = a.C;
    p.D = (int)a.D;
    p.rows = a.rows;
    // Many rows: one warp per row (4 rows per CTA).  Few rows: 4 warps per row.
    const bool wide = a.rows >= 2LL * dev.sm_count * 4;
    const bool cascade = wide && a.pre_part != nullptr && a.NS <= kCombBatch && a.C <= kCombBatch;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(cascade ? (a.rows + kCombWarps / 2 - 1) / (kCombWarps / 2)
                                          : (wide ? (a.rows + kCombWarps - 1) / kCombWarps : a.rows)),
                       1, 1);
    cfg.blockDim = dim3(kCombWarps * 32, 1, 1);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
#define SKV_COMB(T_, V_) \
    (cascade ? cudaLaunchKernelEx(&cfg, cascade_combine_kernel<T_, V_>, p) \
             : (wide ? cudaLaunchKernelEx(&cfg, combine_kernel<T_, 1, V_>, p) \
                     : cudaLaunchKernelEx(&cfg, combine_kernel<T_, kCombWarps, V_>, p)))
    // Per-sequence split counts are separate instantiations: a count that
    // varies by row costs the uniform kernels registers.
    const bool var = a.seq_splits != nullptr;
    switch (a.out_dt) {
        case SKV_F32: return var ? SKV_COMB(float, true) : SKV_COMB(float, false);
        case SKV_F16: return var ? SKV_COMB(__half, true) : SKV_COMB(__half, false);
        case SKV_BF16: return var ? SKV_COMB(__nv_bfloat16, true) : SKV_COMB(__nv_bfloat16, false);
    }
#undef SKV_COMB
    return cudaErrorInvalidValue;
}

}  // namespace skv
