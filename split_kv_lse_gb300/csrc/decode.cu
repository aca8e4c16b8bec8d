// decode.cu -- split-KV paged decode attention, pass 1, for sm_103a.
//
// Page: "L3 讲解：split-KV decode 与 LSE 合并" -- §① the two-pass
// Flash-Decoding scheme (grid (B, Hkv, NUM_SPLITS), each program walks its
// own pages and writes a split-normalised o and that split's lse), §② the
// page ranges, §③ the per-split state o_s = acc/l, lse_s = m + log l (here in
// base 2: s = m2 + log2 l), §④ empty splits (o = 0, lse = -inf), §⑤ fp32
// partials.  The combine pass is merge.cu's CTA kernel, chained with
// programmatic dependent launch.
//
// GB300 design (not the page's Triton program):
//   * One CTA per (b, hkv, split) serves all G = Hq/Hkv query heads of that
//     KV head, so each K/V byte fetched from HBM feeds G heads.
//   * W warps per CTA; warp w owns pages p_start + w, + w + W, ... of the
//     split and streams them through its own ring of R slots.  A slot is the
//     (page, hkv) tile of K and of V: two contiguous 4 KB blocks copied by the
//     TMA engine (cp.async.bulk) with completion counted on an mbarrier; the
//     warp refills a slot right after consuming it, so up to R pages per warp
//     are in flight.  No cross-warp synchronisation in the main loop.
//   * Lane (c, th) = (lane % 16, lane / 16) owns dims [8c, 8c+8) and tokens
//     [8th, 8th+8) of a page: every 16-byte shared-memory read of a warp then
//     covers two full 256-byte rows, i.e. is bank-conflict free without a
//     swizzle.  q (pre-scaled by sm_scale*log2 e) and the output accumulators
//     for the lane's 8 dims of all G heads live in registers.
//   * Scores: per-lane partial dot products over 8 dims, then a shuffle
//     reduce-scatter over the 16 dim-lanes leaves each lane complete scores
//     for 8G/16 (token, head) pairs.  Online softmax in base 2 ([F2] §②
//     exp2 trick): page max per head by shuffles, p = 2^(x - m), running l
//     kept per lane and reduced once at the end.  p reaches the PV product
//     through a per-warp shared-memory buffer.
//   * CUDA cores only (fp32 FMA): this pass is bound by HBM, not by math.
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
    const __half* q;
    const __half* k_cache;
    const __half* v_cache;
    const int32_t* block_table;
    const int32_t* ctx;
    float* o_part;
    float* lse_part;
    int32_t* ranges_dbg;
    unsigned long long* err;
    int32_t num_pool_pages, max_pages, Hq, Hkv, NS;
    float scale_log2;  // sm_scale * log2(e)
};

// Reduce-scatter of L values over the lanes that differ in bits MASK, MASK/2,
// ..., 1: at each step a lane keeps the half of its array selected by its
// lane bit and adds the partner's copy of that half.  After the steps with
// L >= 2 lane c holds in v[i] the complete sum for original index
// i + (L_final) * c; once L reaches 1 the remaining steps are plain
// butterflies (both partners end with the same total).
template <int L, int MASK>
SKV_DEVINL void reduce_scatter(float* v, int lane) {
    if constexpr (MASK >= 1) {
        if constexpr (L >= 2) {
            constexpr int H = L / 2;
            const bool upper = (lane & MASK) != 0;
#pragma unroll
            for (int i = 0; i < H; ++i) {
                const float send = upper ? v[i] : v[i + H];
                const float keep = upper ? v[i + H] : v[i];
                v[i] = keep + __shfl_xor_sync(kFull, send, MASK);
            }
            reduce_scatter<H, MASK / 2>(v, lane);
        } else {
            v[0] += __shfl_xor_sync(kFull, v[0], MASK);
            reduce_scatter<1, MASK / 2>(v, lane);
        }
    }
}

template <int G> struct Layout {
    static constexpr int NV = 8 * G;                 // partial dots per lane per page
    static constexpr int LF = NV >= 16 ? NV / 16 : 1;  // complete scores per lane
    static constexpr int LPH = G == 1 ? 16 : 8 / LF; // dim-lanes sharing one head
};

template <int G, int W, int R>
constexpr size_t smem_bytes() {
    return (size_t)W * R * kStageBytes + (size_t)W * R * sizeof(uint64_t) +
           (size_t)W * 2 * 8 * G * sizeof(float);
}

template <int G, int W, int R>
__global__ void __launch_bounds__(W * 32)
splitkv_decode_kernel(const DecodeParams p) {
    using Lay = Layout<G>;
    constexpr int NV = Lay::NV, LF = Lay::LF, LPH = Lay::LPH;
    static_assert(W * R * kStageBytes >= W * G * (kD + 2) * (int)sizeof(float),
                  "the cross-warp merge buffer reuses the ring");
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t* ring = smem;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + W * R * kStageBytes);
    float* ps_all = reinterpret_cast<float*>(bars + W * R);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c = lane & 15, th = lane >> 4;
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
        for (int i = 0; i < W * R; ++i) mbar_init(&bars[i], 1);
        fence_mbar_init();
    }
    __syncthreads();

    // q for the lane's 8 dims of every head of the group, scaled so that
    // scores come out in log2 units.
    float qf[G][8];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        const uint4 raw = *reinterpret_cast<const uint4*>(
            p.q + ((int64_t)b * p.Hq + hkv * G + g) * kD + 8 * c);
        unpack_h(raw, qf[g]);
#pragma unroll
        for (int i = 0; i < 8; ++i) qf[g][i] *= p.scale_log2;
    }

    const int32_t* bt = p.block_table + (int64_t)b * p.max_pages;
    const uint64_t pol = policy_evict_first();
    uint8_t* my_ring = ring + warp * R * kStageBytes;
    uint64_t* my_bars = bars + warp * R;
    // Page ids of this warp's pages k in [kb, kb + 32), one per lane.
    int kb = 0;
    int my_id = (lane < nw) ? bt[p0 + warp + lane * W] : 0;
    auto issue = [&](int k) {  // warp-uniform
        if (k - kb >= 32) {
            kb += 32;
            my_id = (kb + lane < nw) ? bt[p0 + warp + (kb + lane) * W] : 0;
        }
        int pid = __shfl_sync(kFull, my_id, k - kb);
        if (lane == 0) {
            if ((unsigned)pid >= (unsigned)p.num_pool_pages) {
                record_error(p.err, SKV_ERR_INVALID_ARG, 1 << 20 | b);
                pid = 0;
            }
            const int slot = k % R;
            uint64_t* bar = &my_bars[slot];
            uint8_t* dst = my_ring + slot * kStageBytes;
            const int64_t off = ((int64_t)pid * p.Hkv + hkv) * (kPage * kD);
            mbar_arrive_expect_tx(bar, kStageBytes);
            bulk_g2s(dst, p.k_cache + off, kTileBytes, bar, pol);
            bulk_g2s(dst + kTileBytes, p.v_cache + off, kTileBytes, bar, pol);
        }
    };
#pragma unroll 1
    for (int k = 0; k < R && k < nw; ++k) issue(k);

    float o[G][8];
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
        for (int i = 0; i < 8; ++i) o[g][i] = 0.f;
    float m_own = -INFINITY;  // running max (log2 units) of this lane's head
    float l_own = 0.f;        // this lane's share of the running sum
    const int g_own = G == 1 ? 0 : (LF * c) / 8;
    float* ps = ps_all + warp * (2 * 8 * G);  // p[th][tl][g]

#pragma unroll 1
    for (int k = 0; k < nw; ++k) {
        const int slot = k % R;
        const bool ok = mbar_wait(&my_bars[slot], (uint32_t)((k / R) & 1), p.err, 2);
        if (!__all_sync(kFull, ok)) {
            // A bounded wait gave up (error recorded).  Give the copies this
            // warp still has in flight one more bounded wait each before the
            // ring is reused, then stop.
            for (int kk = k + 1; kk < nw && kk < k + R; ++kk)
                mbar_wait(&my_bars[kk % R], (uint32_t)((kk / R) & 1), p.err, 3);
            break;
        }
        const int page_idx = p0 + warp + k * W;
        const int nvalid = min(kPage, ctx - page_idx * kPage);  // >= 1 inside the range
        const uint8_t* Ks = my_ring + slot * kStageBytes;
        const uint8_t* Vs = Ks + kTileBytes;

        // Partial scores, head-major: part[g * 8 + tl].
        float part[NV];
#pragma unroll
        for (int tl = 0; tl < 8; ++tl) {
            const uint4 kr = *reinterpret_cast<const uint4*>(Ks + (8 * th + tl) * (kD * 2) + c * 16);
            float kf[8];
            unpack_h(kr, kf);
#pragma unroll
            for (int g = 0; g < G; ++g) {
                float a = qf[g][0] * kf[0];
#pragma unroll
                for (int i = 1; i < 8; ++i) a = fmaf(qf[g][i], kf[i], a);
                part[g * 8 + tl] = a;
            }
        }
        reduce_scatter<NV, 8>(part, lane);

        // Complete scores x[i] for (token 8th + tl_i, head g_own), masked.
        float x[LF];
        float mx = -INFINITY;
#pragma unroll
        for (int i = 0; i < LF; ++i) {
            const int j = G == 1 ? (c >> 1) : LF * c + i;
            const int t = 8 * th + (j & 7);
            x[i] = t < nvalid ? part[i] : -INFINITY;
            mx = fmaxf(mx, x[i]);
        }
#pragma unroll
        for (int mm = 1; mm < LPH; mm <<= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, mm));
        mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 16));
        const float m_new = fmaxf(m_own, mx);  // finite: token 0 of the page is valid
        const float alpha_own = exp2f(m_own - m_new);
        float psum = 0.f;
#pragma unroll
        for (int i = 0; i < LF; ++i) {
            const float pv = exp2f(x[i] - m_new);
            psum += pv;
            const int j = G == 1 ? (c >> 1) : LF * c + i;
            if (G != 1 || (c & 1) == 0) ps[(th * 8 + (j & 7)) * G + g_own] = pv;
        }
        l_own = l_own * alpha_own + psum;
        m_own = m_new;
        float alpha[G];
        bool rescale = false;
#pragma unroll
        for (int g = 0; g < G; ++g) {
            alpha[g] = __shfl_sync(kFull, alpha_own, g * LPH);
            rescale |= alpha[g] != 1.f;
        }
        __syncwarp();
        if (__any_sync(kFull, rescale)) {
#pragma unroll
            for (int g = 0; g < G; ++g)
#pragma unroll
                for (int i = 0; i < 8; ++i) o[g][i] *= alpha[g];
        }
        const bool ragged = nvalid < kPage;
#pragma unroll
        for (int tl = 0; tl < 8; ++tl) {
            const int t = 8 * th + tl;
            const uint4 vr = *reinterpret_cast<const uint4*>(Vs + t * (kD * 2) + c * 16);
            float vf[8];
            unpack_h(vr, vf);
            if (ragged && t >= nvalid) {
#pragma unroll
                for (int i = 0; i < 8; ++i) vf[i] = 0.f;  // never multiply 0 by a stale value
            }
            float pg[G];
            const float* pp = ps + (th * 8 + tl) * G;
            if constexpr (G % 4 == 0) {
#pragma unroll
                for (int g = 0; g < G; g += 4) {
                    const float4 t4 = *reinterpret_cast<const float4*>(pp + g);
                    pg[g] = t4.x; pg[g + 1] = t4.y; pg[g + 2] = t4.z; pg[g + 3] = t4.w;
                }
            } else if constexpr (G == 2) {
                const float2 t2 = *reinterpret_cast<const float2*>(pp);
                pg[0] = t2.x; pg[1] = t2.y;
            } else {
                pg[0] = pp[0];
            }
#pragma unroll
            for (int g = 0; g < G; ++g)
#pragma unroll
                for (int i = 0; i < 8; ++i) o[g][i] = fmaf(pg[g], vf[i], o[g][i]);
        }
        __syncwarp();  // slot and p buffer fully read
        if (k + R < nw) issue(k + R);
    }

    // Per-head totals of this warp: l over the lanes of the head (each lane
    // pair of G == 1 holds duplicates), o over the two token halves.
#pragma unroll
    for (int mm = (G == 1 ? 2 : 1); mm < LPH; mm <<= 1) l_own += __shfl_xor_sync(kFull, l_own, mm);
    l_own += __shfl_xor_sync(kFull, l_own, 16);
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
        for (int i = 0; i < 8; ++i) o[g][i] += __shfl_xor_sync(kFull, o[g][i], 16);

    __syncthreads();  // every warp is done with its ring: reuse it
    float* wo = reinterpret_cast<float*>(ring);  // [W][G][kD]
    float* wm = wo + W * G * kD;                 // [W][G]
    float* wl = wm + W * G;                      // [W][G]
    if (th == 0) {
#pragma unroll
        for (int g = 0; g < G; ++g) {
            float4* dst = reinterpret_cast<float4*>(wo + (warp * G + g) * kD + 8 * c);
            dst[0] = make_float4(o[g][0], o[g][1], o[g][2], o[g][3]);
            dst[1] = make_float4(o[g][4], o[g][5], o[g][6], o[g][7]);
        }
        if (c % LPH == 0) {
            wm[warp * G + g_own] = m_own;
            wl[warp * G + g_own] = l_own;
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

constexpr int kWarps = 2;
constexpr int kRing = 3;

template <int G>
cudaError_t launch_g(const DecodeParams& p, int B, int Hkv, int NS, cudaStream_t st) {
    constexpr size_t smem = smem_bytes<G, kWarps, kRing>();
    auto kern = splitkv_decode_kernel<G, kWarps, kRing>;
    static bool attr_set[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 64 && !attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    kern<<<dim3(NS, Hkv, B), kWarps * 32, smem, st>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_splitkv_decode(const DecodeArgs& a, const DeviceInfo& dev, cudaStream_t st) {
    DecodeParams p;
    p.q = static_cast<const __half*>(a.q);
    p.k_cache = static_cast<const __half*>(a.k_cache);
    p.v_cache = static_cast<const __half*>(a.v_cache);
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
    switch (a.Hq / a.Hkv) {
        case 1: return launch_g<1>(p, a.B, a.Hkv, a.num_splits, st);
        case 2: return launch_g<2>(p, a.B, a.Hkv, a.num_splits, st);
        case 4: return launch_g<4>(p, a.B, a.Hkv, a.num_splits, st);
        case 8: return launch_g<8>(p, a.B, a.Hkv, a.num_splits, st);
    }
    return cudaErrorInvalidValue;
}

}  // namespace skv
