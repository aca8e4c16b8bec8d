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
//   * W warps; warp w owns the split's pages w, w + W, ... and R/W ring slots.
//     A slot holds one (page, kv-head) tile: K and V, each one contiguous
//     4 KB run of its cache, copied by two bulk copies (TMA engine) that two
//     lanes issue in one instruction, completion counted on the slot's
//     mbarrier.  The warp refills a slot as soon as it has consumed it.
//   * QK: lane (g, tg) owns whole dot products -- head g, tokens tg + j*TGN --
//     over all 128 dims, with q resident in registers, so no cross-lane
//     reduction.  A lane walks the 16-byte chunks of its rows in an order
//     rotated by its token (q is held rotated the same way), so the lanes'
//     reads of different rows fall in different banks.  fp16 x fp16 -> fp32
//     FMAs (fma.rn.f32.f16): the products are exact, no conversions.
//   * Online softmax in base 2 ([F2] §② exp2 trick) per head; the lanes of
//     a head hold its running max, so the rescale factor never crosses lanes.
//     p goes through shared memory as fp16 to the PV product, where lane
//     (g, dc) owns head g's dims of 16-byte chunks dc, dc + TGN, ....
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
    int32_t num_pool_pages, max_pages, Hq, Hkv, NS;
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

// Lane roles.  G >= 2: lane = g * TGN + x, x in [0, TGN) -- in QK x = tg (the
// lane's tokens are tg + j*TGN, j < G/2), in PV x = dc (the lane's V chunks
// are dc + j*TGN, j < G/2).  G == 1: QK lane = dh*16 + t (token t, dims of
// K box dh, two lanes per token); PV lane = dims [4*lane, 4*lane + 4).
template <int G> struct Roles {
    static_assert(G == 1 || G == 2 || G == 4 || G == 8, "group size");
    static constexpr int TGN = G == 1 ? 32 : 32 / G;  // lanes per head
    static constexpr int TPL = G == 1 ? 1 : G / 2;    // tokens per lane in QK
    static constexpr int CPL = G == 1 ? 1 : G / 2;    // V chunks per lane in PV
    static constexpr int DPL = G == 1 ? 4 : 8 * CPL;  // output dims per lane
};


// The barriers take R words, rounded up to 16 bytes: the p buffer after them
// is read with 16-byte loads.
template <int R>
constexpr size_t bars_bytes() {
    return ((size_t)R * sizeof(uint64_t) + 15) / 16 * 16;
}

template <int G, int W, int R>
constexpr size_t smem_bytes() {
    return 1024 /* alignment slack */ + (size_t)R * kStageBytes + bars_bytes<R>() +
           (size_t)W * G * kPage * sizeof(uint16_t);
}

template <int G, int W, int R, bool BF>
__global__ void __launch_bounds__(W * 32)
splitkv_decode_kernel(const DecodeParams p) {
    using Ro = Roles<G>;
    constexpr int TGN = Ro::TGN, TPL = Ro::TPL, CPL = Ro::CPL, DPL = Ro::DPL;
    constexpr int SPW = R / W;  // ring slots per warp
    static_assert(R % W == 0, "each warp owns R/W slots");
    static_assert(R * kStageBytes >= W * G * (kD + 2) * (int)sizeof(float),
                  "the cross-warp merge buffer reuses the ring");
    extern __shared__ uint8_t smem_raw[];
    // The swizzled K boxes need 1024-byte alignment.  Offset the shared
    // pointer itself (an integer round trip would lose the shared address
    // space and turn every K/V read into a generic load).
    uint8_t* ring = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    uint64_t* bars = reinterpret_cast<uint64_t*>(ring + R * kStageBytes);
    uint16_t* ps_all = reinterpret_cast<uint16_t*>(reinterpret_cast<uint8_t*>(bars) + bars_bytes<R>());

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int split = blockIdx.x, hkv = blockIdx.y, b = blockIdx.z;

    // The combine grid may be scheduled now; it waits for this grid to finish.
    pdl_launch_dependents();

    int ctx = p.ctx[b];
    const int cap = p.max_pages * kPage;
    if (ctx < 0 || ctx > cap) {
        if (threadIdx.x == 0 && split == 0 && hkv == 0) record_error(p.err, SKV_ERR_INVALID_ARG, b);
        ctx = ctx < 0 ? 0 : cap;
    }
    int p0, p1;
    split_page_range(ctx, kPage, p.NS, split, &p0, &p1);
    if (p.ranges_dbg != nullptr && hkv == 0 && threadIdx.x == 0) {
        p.ranges_dbg[((int64_t)b * p.NS + split) * 2 + 0] = p0;
        p.ranges_dbg[((int64_t)b * p.NS + split) * 2 + 1] = p1;
    }
    const int npages = p1 > p0 ? p1 - p0 : 0;
    const int nw = npages > warp ? (npages - warp + W - 1) / W : 0;  // this warp's pages

    if (threadIdx.x == 0) {
        for (int i = 0; i < R; ++i) mbar_init(&bars[i], 1);
        fence_mbar_init();
    }
    __syncthreads();

    // q of this lane's head, all 128 dims, as fp16 pairs (G == 1: the 64
    // dims of K box dh), pinned in registers for the whole split.
    const int g_lane = G == 1 ? 0 : lane / TGN;
    const int x_lane = G == 1 ? lane : lane % TGN;
    constexpr int QW = G == 1 ? 32 : 64;
    uint32_t qh[QW];
    {
        // Rotated: register chunk i holds q chunk (i + r) mod n, r = the
        // lane's token (G == 1: within its half of the head dim).
        const uint16_t* qrow = p.q + ((int64_t)b * p.Hq + hkv * G + g_lane) * kD +
                             (G == 1 ? 64 * (lane >> 4) : 0);
        constexpr int nq = QW / 4;
        const int r = G == 1 ? (lane & 15) : x_lane;
#pragma unroll
        for (int i = 0; i < nq; ++i) {
            const uint4 a = ld_pinned(qrow + 8 * ((i + r) & (nq - 1)));
            qh[4 * i + 0] = a.x; qh[4 * i + 1] = a.y; qh[4 * i + 2] = a.z; qh[4 * i + 3] = a.w;
        }
    }

    const int32_t* bt = p.block_table + (int64_t)b * p.max_pages;
    const uint64_t pol = policy_evict_first();
    uint8_t* my_ring = ring + warp * SPW * kStageBytes;
    uint64_t* my_bars = bars + warp * SPW;
    // Page ids of this warp's pages k in [kb, kb + 32), one per lane.
    int kb = 0;
    int my_id = (lane < nw) ? bt[p0 + warp + lane * W] : 0;
    auto issue = [&](int k) {  // warp-uniform call; lanes 0 and 1 issue the copies
        if (k - kb >= 32) {
            kb += 32;
            my_id = (kb + lane < nw) ? bt[p0 + warp + (kb + lane) * W] : 0;
        }
        int pid = __shfl_sync(kFull, my_id, k - kb);
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
    };
#pragma unroll 1
    for (int k = 0; k < SPW && k < nw; ++k) issue(k);

    float o[DPL];
#pragma unroll
    for (int i = 0; i < DPL; ++i) o[i] = 0.f;
    float m_run = -INFINITY;  // running max (log2 units) of this lane's head
    float l_run = 0.f;        // this lane's share of the running sum
    uint16_t* ps = ps_all + warp * (G * kPage);  // p[g][token], fp16

#pragma unroll 1
    for (int k = 0; k < nw; ++k) {
        const int slot = k % SPW;
        const bool ok = mbar_wait(&my_bars[slot], (uint32_t)((k / SPW) & 1), p.err, 2);
        if (!__all_sync(kFull, ok)) {
            // A bounded wait gave up (error recorded).  Give the copies this
            // warp still has in flight one more bounded wait each before the
            // ring is reused, then stop.
            for (int kk = k + 1; kk < nw && kk < k + SPW; ++kk)
                mbar_wait(&my_bars[kk % SPW], (uint32_t)((kk / SPW) & 1), p.err, 3);
            break;
        }
        const int nvalid = min(kPage, ctx - (p0 + warp + k * W) * kPage);  // >= 1
        const uint8_t* Kb = my_ring + slot * kStageBytes;  // two swizzled boxes
        const uint8_t* Vs = Kb + kTileBytes;

        // ---- scores of this lane's tokens (log2 units, masked)
        float x[TPL];
        if constexpr (G == 1) {
            const int t = lane & 15, dh = lane >> 4;
            const uint8_t* rowp = Kb + t * (kD * 2) + dh * 128;
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                // Step c reads chunk (c + t) & 7 of the lane's half row (q is
                // held rotated to match), so lanes of different rows read
                // different banks.
                const uint4 kv = *reinterpret_cast<const uint4*>(rowp + (((c + t) & 7) << 4));
                acc[c & 3] = dot2_h<BF>(qh[4 * c + 0], kv.x, acc[c & 3]);
                acc[c & 3] = dot2_h<BF>(qh[4 * c + 1], kv.y, acc[c & 3]);
                acc[c & 3] = dot2_h<BF>(qh[4 * c + 2], kv.z, acc[c & 3]);
                acc[c & 3] = dot2_h<BF>(qh[4 * c + 3], kv.w, acc[c & 3]);
            }
            float sc = (acc[0] + acc[1]) + (acc[2] + acc[3]);
            sc += __shfl_xor_sync(kFull, sc, 16);
            x[0] = t < nvalid ? sc * p.scale_log2 : -INFINITY;
        } else {
            // The lane's TPL tokens side by side, and the low and high fp16
            // halves of each word into separate sums: 8 * TPL independent
            // FMA chains, each advanced once per 16-byte chunk of K.
            float acc[TPL][8];
#pragma unroll
            for (int j = 0; j < TPL; ++j)
#pragma unroll
                for (int i = 0; i < 8; ++i) acc[j][i] = 0.f;
            // Step c reads chunk (c + t) & 15 of row t: the lanes of a head
            // read different banks.  The lane's q is held rotated by x_lane,
            // so token t = x_lane + j * TGN meets q chunk (c + j * TGN) & 15.
#pragma unroll
            for (int c = 0; c < 16; ++c) {
                uint4 kv[TPL];
#pragma unroll
                for (int j = 0; j < TPL; ++j) {
                    const int t = x_lane + j * TGN;
                    kv[j] = *reinterpret_cast<const uint4*>(Kb + t * (kD * 2) + (((c + t) & 15) << 4));
                }
#pragma unroll
                for (int j = 0; j < TPL; ++j) {
                    const int qi = 4 * ((c + j * TGN) & 15);
                    const uint32_t kw[4] = {kv[j].x, kv[j].y, kv[j].z, kv[j].w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        acc[j][2 * i] = fma_h<BF, false>(qh[qi + i], kw[i], acc[j][2 * i]);
                        acc[j][2 * i + 1] = fma_h<BF, true>(qh[qi + i], kw[i], acc[j][2 * i + 1]);
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < TPL; ++j) {
                const int t = x_lane + j * TGN;
                const float sc = ((acc[j][0] + acc[j][1]) + (acc[j][2] + acc[j][3])) +
                                 ((acc[j][4] + acc[j][5]) + (acc[j][6] + acc[j][7]));
                x[j] = t < nvalid ? sc * p.scale_log2 : -INFINITY;
            }
        }

        // ---- online softmax of this lane's head (its lanes agree on m)
        float mx = x[0];
#pragma unroll
        for (int j = 1; j < TPL; ++j) mx = fmaxf(mx, x[j]);
#pragma unroll
        for (int mm = 1; mm < (G == 1 ? 16 : TGN); mm <<= 1)
            mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, mm));
        const float m_new = fmaxf(m_run, mx);  // finite: token 0 of the page is valid
        const float alpha = exp2f(m_run - m_new);
        float psum = 0.f;
#pragma unroll
        for (int j = 0; j < TPL; ++j) {
            const float pj = exp2f(x[j] - m_new);
            psum += pj;
            if constexpr (G == 1) {
                if (lane < 16) ps[lane] = to_p<BF>(pj);
            } else {
                ps[g_lane * kPage + x_lane + j * TGN] = to_p<BF>(pj);
            }
        }
        l_run = fmaf(l_run, alpha, psum);
        m_run = m_new;
        __syncwarp();

        // ---- o = alpha * o + p V for this lane's head and dims
        if (__any_sync(kFull, alpha != 1.f)) {
#pragma unroll
            for (int i = 0; i < DPL; ++i) o[i] *= alpha;
        }
        const uint4 pa = *reinterpret_cast<const uint4*>(ps + g_lane * kPage);
        const uint4 pb = *reinterpret_cast<const uint4*>(ps + g_lane * kPage + 8);
        const uint32_t pw[8] = {pa.x, pa.y, pa.z, pa.w, pb.x, pb.y, pb.z, pb.w};
        auto pv_token = [&](int t) {
            const uint8_t* vrow = Vs + t * (kD * 2);
            if constexpr (G == 1) {
                const uint2 vv = *reinterpret_cast<const uint2*>(vrow + 8 * lane);
                if (t & 1) {
                    axpy2_h<BF, true>(pw[t >> 1], vv.x, o[0], o[1]);
                    axpy2_h<BF, true>(pw[t >> 1], vv.y, o[2], o[3]);
                } else {
                    axpy2_h<BF, false>(pw[t >> 1], vv.x, o[0], o[1]);
                    axpy2_h<BF, false>(pw[t >> 1], vv.y, o[2], o[3]);
                }
            } else {
#pragma unroll
                for (int j = 0; j < CPL; ++j) {
                    const uint4 vv = *reinterpret_cast<const uint4*>(vrow + (x_lane + j * TGN) * 16);
                    const uint32_t w4[4] = {vv.x, vv.y, vv.z, vv.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        if (t & 1)
                            axpy2_h<BF, true>(pw[t >> 1], w4[i], o[8 * j + 2 * i], o[8 * j + 2 * i + 1]);
                        else
                            axpy2_h<BF, false>(pw[t >> 1], w4[i], o[8 * j + 2 * i], o[8 * j + 2 * i + 1]);
                    }
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
        if (k + SPW < nw) issue(k + SPW);
    }

    // This warp's per-head totals: l over the lanes of the head.
#pragma unroll
    for (int mm = 1; mm < (G == 1 ? 16 : TGN); mm <<= 1) l_run += __shfl_xor_sync(kFull, l_run, mm);

    __syncthreads();  // every warp is done with its ring: reuse it
    float* wo = reinterpret_cast<float*>(ring);  // [W][G][kD]
    float* wm = wo + W * G * kD;                 // [W][G]
    float* wl = wm + W * G;                      // [W][G]
    if constexpr (G == 1) {
        *reinterpret_cast<float4*>(wo + warp * kD + 4 * lane) = make_float4(o[0], o[1], o[2], o[3]);
        if (lane == 0) {
            wm[warp] = m_run;
            wl[warp] = l_run;
        }
    } else {
        float* dst = wo + (warp * G + g_lane) * kD;
#pragma unroll
        for (int j = 0; j < CPL; ++j) {
            float4* d4 = reinterpret_cast<float4*>(dst + 8 * (x_lane + j * TGN));
            d4[0] = make_float4(o[8 * j + 0], o[8 * j + 1], o[8 * j + 2], o[8 * j + 3]);
            d4[1] = make_float4(o[8 * j + 4], o[8 * j + 5], o[8 * j + 6], o[8 * j + 7]);
        }
        if (x_lane == 0) {
            wm[warp * G + g_lane] = m_run;
            wl[warp * G + g_lane] = l_run;
        }
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

template <int G, int W, int R, bool BF>
cudaError_t launch_gwr(const DecodeParams& p, int B, int Hkv, int NS,
                       cudaStream_t st) {
    constexpr size_t smem = smem_bytes<G, W, R>();
    auto kern = splitkv_decode_kernel<G, W, R, BF>;
    static bool attr_set[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 64 && !attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    kern<<<dim3(NS, Hkv, B), W * 32, smem, st>>>(p);
    return cudaGetLastError();
}

// Warps per CTA follow the longest possible split (the page table's width
// over NUM_SPLITS): a CTA of 3 warps with a 6-page ring for long splits; for
// short splits smaller CTAs, so that many more of them are resident per SM
// and their fixed latencies (q, page table, first copies) overlap.
template <int G, bool BF>
cudaError_t launch_g(const DecodeParams& p, int B, int Hkv, int NS,
                     int max_pages, cudaStream_t st) {
    // Measured on the cascade suffixes (<= 8 pages per split, B=64, NS=16):
    // pass 1 takes 53 us with 1 warp and a 2-page ring (about 13 CTAs per
    // SM), 64 us with 2 warps, 72 us with 3; a 4-page ring for the 1-warp
    // CTA (fewer CTAs per SM) takes 74 us.  Long splits (32 pages) keep 3.
    const int pps = (max_pages + NS - 1) / NS;
    if (pps <= 8) return launch_gwr<G, 1, 2, BF>(p, B, Hkv, NS, st);
    if (pps <= 16) return launch_gwr<G, 2, 4, BF>(p, B, Hkv, NS, st);
    return launch_gwr<G, 3, 6, BF>(p, B, Hkv, NS, st);
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
    void* out;             // [rows, D] Tout
    float* lse_out;        // [rows] or nullptr
    const float* pre_part; // [rows, C, D] prefix-chunk states or nullptr
    const float* pre_lse;  // [rows, C]
    float* o_pre;          // [rows, D] merged prefix state or nullptr
    float* s_pre;          // [rows]
    int64_t rows;
    int NS, C, D;
};

struct WarpState {
    float m, W;
    float4 acc;
};

// This warp's share (states sub, sub + WPR, ...) of the N states of `row`.
// Per batch of kCombBatch states: lane k (and lane k + 16) reads state k's
// lse and computes its weight, the batch max and weight sum go through
// shuffles, and every lane then accumulates its 4 dims of the batch's v rows
// with the weights broadcast from their lanes.
template <int WPR>
SKV_DEVINL WarpState warp_merge(const float* o, const float* lse, int N, int D, int64_t row,
                                int sub) {
    static_assert(kCombBatch == 16, "two lanes per state in a batch");
    const int lane = threadIdx.x & 31;
    const bool has = 4 * lane < D;
    WarpState st{-INFINITY, 0.f, make_float4(0.f, 0.f, 0.f, 0.f)};
    for (int n0 = sub; n0 < N; n0 += WPR * kCombBatch) {
        const int nk = n0 + (lane & 15) * WPR;
        const float lk = nk < N ? sanitize_lse(__ldcg(lse + row * N + nk)) : -INFINITY;
        float4 x[kCombBatch];
#pragma unroll
        for (int k = 0; k < kCombBatch; ++k) {
            const int n = n0 + k * WPR;
            x[k] = (n < N && has) ? __ldcg(reinterpret_cast<const float4*>(o + (row * N + n) * D) + lane)
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        float mb = lk;
#pragma unroll
        for (int mm = 1; mm < 16; mm <<= 1) mb = fmaxf(mb, __shfl_xor_sync(kFull, mb, mm));
        mb = fmaxf(mb, st.m);
        const float wk = merge_weight(lk, mb);
        float ws = wk;
#pragma unroll
        for (int mm = 1; mm < 16; mm <<= 1) ws += __shfl_xor_sync(kFull, ws, mm);
        const float sc = merge_weight(st.m, mb);  // rescale of the running state
        st.W = fmaf(st.W, sc, ws);
        st.acc.x *= sc; st.acc.y *= sc; st.acc.z *= sc; st.acc.w *= sc;
#pragma unroll
        for (int k = 0; k < kCombBatch; ++k) {
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

// Merged state of `row` over N states: v (this lane's 4 dims) and s.  With
// WPR > 1 every thread of the CTA must call this (block barriers).
template <int WPR>
SKV_DEVINL void merge_row(const float* o, const float* lse, int N, int D, int64_t row, int sub,
                          CombSmem& sm, float (&v)[4], float& s_out) {
    WarpState st = warp_merge<WPR>(o, lse, N, D, row, sub);
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

template <typename Tout, int WPR>
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
    merge_row<WPR>(p.o_part, p.lse_part, p.NS, p.D, row, sub, sm, vd, sd);
    if (p.pre_part != nullptr) {
        float vp[4] = {0.f, 0.f, 0.f, 0.f}, sp = -INFINITY;  // empty prefix when C == 0
        if (p.C > 0) merge_row<WPR>(p.pre_part, p.pre_lse, p.C, p.D, row, sub, sm, vp, sp);
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

// Cascade combine with many rows: two warps per row, so that the row's two
// lists are read at once -- warp 0 merges the suffix's split states, warp 1
// the prefix chunks' states into the prefix state (written to o_pre/s_pre)
// -- and they meet in shared memory for the two-state merge, prefix first.
template <typename Tout>
__global__ void __launch_bounds__(kCombWarps * 32)
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
        merge_row<1>(p.o_part, p.lse_part, p.NS, p.D, row, 0, sm, v, s);
    } else {
        if (p.C > 0) merge_row<1>(p.pre_part, p.pre_lse, p.C, p.D, row, 0, sm, v, s);
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
    p.num_pool_pages = a.num_pool_pages;
    p.max_pages = a.max_pages;
    p.Hq = a.Hq;
    p.Hkv = a.Hkv;
    p.NS = a.num_splits;
    p.scale_log2 = a.sm_scale * 1.4426950408889634f;
#define SKV_LAUNCH_G(BF_)                                                             \
    switch (a.Hq / a.Hkv) {                                                           \
        case 1: return launch_g<1, BF_>(p, a.B, a.Hkv, a.num_splits, a.max_pages, st); \
        case 2: return launch_g<2, BF_>(p, a.B, a.Hkv, a.num_splits, a.max_pages, st); \
        case 4: return launch_g<4, BF_>(p, a.B, a.Hkv, a.num_splits, a.max_pages, st); \
        case 8: return launch_g<8, BF_>(p, a.B, a.Hkv, a.num_splits, a.max_pages, st); \
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
#define SKV_COMB(T_) \
    (cascade ? cudaLaunchKernelEx(&cfg, cascade_combine_kernel<T_>, p) \
             : (wide ? cudaLaunchKernelEx(&cfg, combine_kernel<T_, 1>, p) \
                     : cudaLaunchKernelEx(&cfg, combine_kernel<T_, kCombWarps>, p)))
    switch (a.out_dt) {
        case SKV_F32: return SKV_COMB(float);
        case SKV_F16: return SKV_COMB(__half);
        case SKV_BF16: return SKV_COMB(__nv_bfloat16);
    }
#undef SKV_COMB
    return cudaErrorInvalidValue;
}

}  // namespace skv
