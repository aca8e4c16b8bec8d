/*
 * oracle.c -- plain, slow, single-threaded fp64 CPU reference for split-KV
 * decode attention and attention-state merging.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file: only the test suite, the smoke check and the CPU-baseline
 * leg of the benchmark use it.  It shares no code, header, table or helper
 * with the CUDA library; the two meet only through seeded input arrays.
 *
 * Pages this file follows (cited by title and section):
 *   [F2]  "F2 讲解：merge_state，以 2 为底的 LSE 合并"
 *         (gpu-kernel-drills hints page for merge_state)
 *   [L3]  "L3 讲解：split-KV decode 与 LSE 合并"
 *         (gpu-kernel-drills hints page for split-KV decode)
 *   [FA]  "FlashAttention 的空行 LSE:FA-2 的 +inf 约定与后来的变化"
 *
 * Conventions (every function):
 *   - All floating point is double.  Inputs arrive already widened to double.
 *   - An attention state is (v, s): v is the softmax-normalised output over a
 *     key subset, s = log2( sum_j exp(score_j) ) is its base-2 log-sum-exp
 *     ([F2] §① and §②).  The natural-log form is lse = s * ln 2.
 *   - An empty state is s = -inf, v = 0 ([F2] §⑤).
 *   - An incoming s that is NaN or +inf means "no weight" and is read as
 *     -inf ([FA] §2.2).
 *   - Where the pages are silent the readings are stated at the function.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* [FA] §2.2: an incoming LSE that is NaN or +inf folds to -inf. */
static double sanitize(double s) {
    if (isnan(s) || s == INFINITY) return -INFINITY;
    return s;
}

/*
 * Two-state merge, one call for R = S*H rows of D elements ([F2] §③).
 *   m = max(s_a, s_b);  w_x = 2^(s_x - m);  v = (w_a v_a + w_b v_b)/(w_a + w_b);
 *   s = m + log2(w_a + w_b).
 * An empty operand gets weight exactly 0 and its v is not read ([F2] §⑤: one
 * empty state merged with a normal one gives the normal one).  Two empty
 * operands give v = 0, s = -inf: the page guards only the weights; the
 * reading taken here is the zero-reciprocal rule of [FA] §4.1 (inv_sum = 0
 * when the weight sum is 0), which zeroes v, and log2(0) = -inf for s.
 */
void oracle_merge_state(int64_t R, int64_t D,
                        const double* va, const double* sa,
                        const double* vb, const double* sb,
                        double* v, double* s) {
    for (int64_t r = 0; r < R; ++r) {
        double a = sanitize(sa[r]);
        double b = sanitize(sb[r]);
        if (a == -INFINITY && b == -INFINITY) {
            for (int64_t d = 0; d < D; ++d) v[r * D + d] = 0.0;
            s[r] = -INFINITY;
            continue;
        }
        double m = a > b ? a : b;
        double wa = (a == -INFINITY) ? 0.0 : exp2(a - m);
        double wb = (b == -INFINITY) ? 0.0 : exp2(b - m);
        double wsum = wa + wb;
        for (int64_t d = 0; d < D; ++d) {
            double acc = 0.0;
            if (wa > 0.0) acc += wa * va[r * D + d];
            if (wb > 0.0) acc += wb * vb[r * D + d];
            v[r * D + d] = acc / wsum;
        }
        s[r] = m + log2(wsum);
    }
}

/*
 * N-state merge in the [S, N, H, D] / [S, N, H] layout ([F2] §④): element
 * s[pos, n, h] sits at offset (pos*N + n)*H + h, v[pos, n, h, :] at that
 * offset times D.  Output v_out [S, H, D], s_out [S, H].
 *   m = max_n s_n;  w_n = 2^(s_n - m);  v = sum_n w_n v_n / sum_n w_n;
 *   s = m + log2(sum_n w_n).
 * Empty inputs get weight 0 and their v is not read; all-empty rows give
 * v = 0, s = -inf (same reading as oracle_merge_state).  If w_out is not
 * NULL it receives every unnormalised weight 2^(s_n - m) in the [S, N, H]
 * layout (0 for empty inputs and for all-empty rows).
 */
void oracle_merge_states(int64_t S, int64_t N, int64_t H, int64_t D,
                         const double* v, const double* s,
                         double* v_out, double* s_out, double* w_out) {
    double* acc = (double*)malloc(sizeof(double) * (size_t)(D > 0 ? D : 1));
    for (int64_t pos = 0; pos < S; ++pos) {
        for (int64_t h = 0; h < H; ++h) {
            double m = -INFINITY;
            for (int64_t n = 0; n < N; ++n) {
                double x = sanitize(s[(pos * N + n) * H + h]);
                if (x > m) m = x;
            }
            double* vo = v_out + (pos * H + h) * D;
            if (m == -INFINITY) {
                for (int64_t d = 0; d < D; ++d) vo[d] = 0.0;
                s_out[pos * H + h] = -INFINITY;
                if (w_out)
                    for (int64_t n = 0; n < N; ++n) w_out[(pos * N + n) * H + h] = 0.0;
                continue;
            }
            double wsum = 0.0;
            for (int64_t d = 0; d < D; ++d) acc[d] = 0.0;
            for (int64_t n = 0; n < N; ++n) {
                int64_t off = (pos * N + n) * H + h;
                double x = sanitize(s[off]);
                double w = (x == -INFINITY) ? 0.0 : exp2(x - m);
                if (w_out) w_out[off] = w;
                if (w > 0.0) {
                    wsum += w;
                    for (int64_t d = 0; d < D; ++d) acc[d] += w * v[off * D + d];
                }
            }
            for (int64_t d = 0; d < D; ++d) vo[d] = acc[d] / wsum;
            s_out[pos * H + h] = m + log2(wsum);
        }
    }
    free(acc);
}

/*
 * Page range of one split ([L3] §②):
 *   num_pages = ceil(ctx / page);  pages_per_split = ceil(num_pages / NS);
 *   p_start = split * pages_per_split;  p_end = min(p_start + pps, num_pages).
 * The raw values are reported; the split is empty when p_end <= p_start.
 */
void oracle_split_range(int32_t ctx, int32_t page, int32_t num_splits, int32_t split,
                        int32_t* p_start, int32_t* p_end) {
    int32_t num_pages = (ctx + page - 1) / page;
    int32_t pps = (num_pages + num_splits - 1) / num_splits;
    int32_t start = split * pps;
    int32_t end = start + pps;
    if (end > num_pages) end = num_pages;
    *p_start = start;
    *p_end = end;
}

/*
 * Split-count choice ([L3] §⑥): make B*Hkv*NS several times the SM count
 * while every split keeps several pages; do not split when B*Hkv already
 * fills the GPU.  The page prints no constants, only its sweep (unsplit, 4,
 * 16 and 64 splits) and the count it judges suitable for three workloads.
 * The reading taken, which reproduces that table exactly:
 *   - candidates are the swept counts 1, 4, 16, 64;
 *   - "several times the SM count" is 3x: NS = 1 if B*Hkv >= 3*SM, else the
 *     smallest of 4, 16, 64 with B*Hkv*NS >= 3*SM (64 if none reaches it);
 *   - "several pages per split" is 8: while NS > 1 and
 *     ceil(max_pages / NS) < 8, step down to the next smaller candidate.
 */
int32_t oracle_plan(int32_t B, const int32_t* ctx, int32_t Hkv, int32_t page, int32_t sm_count) {
    int32_t max_pages = 0;
    for (int32_t b = 0; b < B; ++b) {
        int32_t np = (ctx[b] + page - 1) / page;
        if (np > max_pages) max_pages = np;
    }
    int64_t programs = (int64_t)B * Hkv;
    int64_t target = 3 * (int64_t)sm_count;
    if (programs >= target) return 1;
    int32_t ns = 4;
    while (ns < 64 && programs * ns < target) ns *= 4;
    while (ns > 1 && (max_pages + ns - 1) / ns < 8) ns /= 4;
    return ns;
}

/*
 * Attention of one query row over an explicit list of n key/value rows
 * ([FA] §0 equation): Z = sum_j e^{S_j}, L = log Z, P_j = e^{S_j - L},
 * O = sum_j P_j V_j, with S_j = sm_scale * q . k_j (the softmax scale is
 * inside the scores).  Returns O and s = L / ln 2.  n = 0 is the empty
 * state ([L3] §④): O = 0, s = -inf.
 */
static void attend_rows(int32_t D, const double* q, int32_t n,
                        const double* const* krows, const double* const* vrows,
                        double sm_scale, double* o, double* s_out) {
    for (int32_t d = 0; d < D; ++d) o[d] = 0.0;
    if (n == 0) {
        *s_out = -INFINITY;
        return;
    }
    double* score = (double*)malloc(sizeof(double) * (size_t)n);
    double mx = -INFINITY;
    for (int32_t j = 0; j < n; ++j) {
        double dot = 0.0;
        for (int32_t d = 0; d < D; ++d) dot += q[d] * krows[j][d];
        score[j] = sm_scale * dot;
        if (score[j] > mx) mx = score[j];
    }
    double z = 0.0;
    for (int32_t j = 0; j < n; ++j) z += exp(score[j] - mx);
    double L = mx + log(z);
    for (int32_t j = 0; j < n; ++j) {
        double p = exp(score[j] - L);
        for (int32_t d = 0; d < D; ++d) o[d] += p * vrows[j][d];
    }
    *s_out = L / log(2.0);
    free(score);
}

/*
 * Address of token t of sequence b in a paged cache laid out
 * [num_pool_pages, Hkv, page, D] with block_table [B, max_pages]: token t
 * lives in pool page block_table[b][t / page], slot t % page.  ([L3] §②
 * fixes pages of PAGE tokens walked through a per-sequence page list; the
 * exact tensor layout is not printed, this is the reading taken.)
 */
static const double* token_row(const double* cache, const int32_t* pages, int32_t t,
                               int32_t Hkv, int32_t hk, int32_t page, int32_t D) {
    int64_t pid = pages[t / page];
    return cache + (((pid * Hkv + hk) * page) + (t % page)) * (int64_t)D;
}

/*
 * Unsplit decode attention (the plain definition the split method must
 * reproduce exactly, [FA] §0.2): for every (b, hq), query head hq reads
 * KV head hq / (Hq/Hkv) (grouped query heads are contiguous: a reading, the
 * pages are silent), over tokens [0, ctx[b]).
 *   q [B, Hq, D]; k_cache, v_cache [P, Hkv, page, D]; block_table [B, max_pages]
 *   out [B, Hq, D]; s_out [B, Hq] base-2.
 */
void oracle_attend_full(int32_t B, int32_t Hq, int32_t Hkv, int32_t D, int32_t page,
                        const double* q, const double* k_cache, const double* v_cache,
                        const int32_t* block_table, int32_t max_pages, const int32_t* ctx,
                        double sm_scale, double* out, double* s_out) {
    int32_t G = Hq / Hkv;
    int32_t maxn = 0;
    for (int32_t b = 0; b < B; ++b) if (ctx[b] > maxn) maxn = ctx[b];
    const double** kr = (const double**)malloc(sizeof(double*) * (size_t)(maxn > 0 ? maxn : 1));
    const double** vr = (const double**)malloc(sizeof(double*) * (size_t)(maxn > 0 ? maxn : 1));
    for (int32_t b = 0; b < B; ++b) {
        const int32_t* pages = block_table + (int64_t)b * max_pages;
        for (int32_t hq = 0; hq < Hq; ++hq) {
            int32_t hk = hq / G;
            for (int32_t t = 0; t < ctx[b]; ++t) {
                kr[t] = token_row(k_cache, pages, t, Hkv, hk, page, D);
                vr[t] = token_row(v_cache, pages, t, Hkv, hk, page, D);
            }
            int64_t row = (int64_t)b * Hq + hq;
            attend_rows(D, q + row * D, ctx[b], kr, vr, sm_scale, out + row * D, s_out + row);
        }
    }
    free(kr);
    free(vr);
}

/*
 * Per-split partial states of the split-KV decode ([L3] §① first kernel,
 * §② ranges, §③ per-split output, §④ empty splits): split `sp` of sequence
 * b attends only to tokens [p_start*page, min(p_end*page, ctx)) and writes
 * the state normalised within the split.  An empty split writes o = 0 and
 * s = -inf.  Outputs o_part [B, Hq, NS, D], lse_part [B, Hq, NS] (base 2).
 */
void oracle_attend_splits(int32_t B, int32_t Hq, int32_t Hkv, int32_t D, int32_t page,
                          const double* q, const double* k_cache, const double* v_cache,
                          const int32_t* block_table, int32_t max_pages, const int32_t* ctx,
                          double sm_scale, int32_t num_splits,
                          double* o_part, double* lse_part) {
    int32_t G = Hq / Hkv;
    int32_t maxn = 0;
    for (int32_t b = 0; b < B; ++b) if (ctx[b] > maxn) maxn = ctx[b];
    const double** kr = (const double**)malloc(sizeof(double*) * (size_t)(maxn > 0 ? maxn : 1));
    const double** vr = (const double**)malloc(sizeof(double*) * (size_t)(maxn > 0 ? maxn : 1));
    for (int32_t b = 0; b < B; ++b) {
        const int32_t* pages = block_table + (int64_t)b * max_pages;
        for (int32_t hq = 0; hq < Hq; ++hq) {
            int32_t hk = hq / G;
            for (int32_t sp = 0; sp < num_splits; ++sp) {
                int32_t p0, p1;
                oracle_split_range(ctx[b], page, num_splits, sp, &p0, &p1);
                int32_t t0 = p0 * page;
                int32_t t1 = p1 * page;
                if (t1 > ctx[b]) t1 = ctx[b];
                int32_t n = (p1 > p0 && t1 > t0) ? t1 - t0 : 0;
                for (int32_t j = 0; j < n; ++j) {
                    kr[j] = token_row(k_cache, pages, t0 + j, Hkv, hk, page, D);
                    vr[j] = token_row(v_cache, pages, t0 + j, Hkv, hk, page, D);
                }
                int64_t row = ((int64_t)b * Hq + hq) * num_splits + sp;
                attend_rows(D, q + ((int64_t)b * Hq + hq) * D, n, kr, vr, sm_scale,
                            o_part + row * D, lse_part + row);
            }
        }
    }
    free(kr);
    free(vr);
}

/*
 * Per-sequence split counts ([L3] §⑥: a real planner decides the splits from
 * B, each sequence's ctx and the SM count, and can give sequences of
 * different lengths different split counts).  The page fixes no rule for
 * the per-sequence count; the reading taken keeps its other rule, every
 * split holds several pages: sequence b's n_b = ceil(ctx_b / page) pages
 * get ns_b = ceil(n_b / pages_per_split) splits, so that no split holds
 * more than pages_per_split pages, clamped to [1, max_splits] (a sequence
 * with no pages has one, empty, split; at the clamp a split holds
 * ceil(n_b / max_splits) pages).
 */
void oracle_plan_varlen(int32_t B, const int32_t* ctx, int32_t page, int32_t max_splits,
                        int32_t pages_per_split, int32_t* num_splits) {
    for (int32_t b = 0; b < B; ++b) {
        int32_t n = (ctx[b] + page - 1) / page;
        int32_t ns = (n + pages_per_split - 1) / pages_per_split;
        if (ns < 1) ns = 1;
        if (ns > max_splits) ns = max_splits;
        num_splits[b] = ns;
    }
}

/*
 * Per-split partial states with a split count per sequence: as
 * oracle_attend_splits, but sequence b is cut into num_splits[b] splits by
 * the [L3] §② formula with NS = num_splits[b].  Outputs keep the split axis
 * max_splits long: o_part [B, Hq, max_splits, D], lse_part [B, Hq,
 * max_splits]; entries sp >= num_splits[b] are not splits of the sequence
 * and are written as empty states (o = 0, s = -inf).
 */
void oracle_attend_splits_varlen(int32_t B, int32_t Hq, int32_t Hkv, int32_t D, int32_t page,
                                 const double* q, const double* k_cache, const double* v_cache,
                                 const int32_t* block_table, int32_t max_pages,
                                 const int32_t* ctx, double sm_scale,
                                 const int32_t* num_splits, int32_t max_splits,
                                 double* o_part, double* lse_part) {
    int32_t G = Hq / Hkv;
    int32_t maxn = 0;
    for (int32_t b = 0; b < B; ++b) if (ctx[b] > maxn) maxn = ctx[b];
    const double** kr = (const double**)malloc(sizeof(double*) * (size_t)(maxn > 0 ? maxn : 1));
    const double** vr = (const double**)malloc(sizeof(double*) * (size_t)(maxn > 0 ? maxn : 1));
    for (int32_t b = 0; b < B; ++b) {
        const int32_t* pages = block_table + (int64_t)b * max_pages;
        int32_t ns = num_splits[b];
        for (int32_t hq = 0; hq < Hq; ++hq) {
            int32_t hk = hq / G;
            for (int32_t sp = 0; sp < max_splits; ++sp) {
                int32_t n = 0, t0 = 0;
                if (sp < ns) {
                    int32_t p0, p1;
                    oracle_split_range(ctx[b], page, ns, sp, &p0, &p1);
                    int32_t t1 = p1 * page;
                    t0 = p0 * page;
                    if (t1 > ctx[b]) t1 = ctx[b];
                    n = (p1 > p0 && t1 > t0) ? t1 - t0 : 0;
                }
                for (int32_t j = 0; j < n; ++j) {
                    kr[j] = token_row(k_cache, pages, t0 + j, Hkv, hk, page, D);
                    vr[j] = token_row(v_cache, pages, t0 + j, Hkv, hk, page, D);
                }
                int64_t row = ((int64_t)b * Hq + hq) * max_splits + sp;
                attend_rows(D, q + ((int64_t)b * Hq + hq) * D, n, kr, vr, sm_scale,
                            o_part + row * D, lse_part + row);
            }
        }
    }
    free(kr);
    free(vr);
}

/*
 * Two-level cascade ([F2] §⑥): every request b attends to a shared prefix
 * of prefix_len tokens (pool pages prefix_pages[0..]) followed by its own
 * suffix of ctx[b] tokens (pool pages block_table[b][..]).  The plain
 * definition is one softmax over the concatenation prefix || suffix:
 *   out [B, Hq, D], s_out [B, Hq].
 * Also returned: the prefix-only state o_pre [B, Hq, D], s_pre [B, Hq]
 * (the state the shared-prefix pass emits before the merge).
 */
void oracle_cascade(int32_t B, int32_t Hq, int32_t Hkv, int32_t D, int32_t page,
                    const double* q, const double* k_cache, const double* v_cache,
                    const int32_t* prefix_pages, int32_t prefix_len,
                    const int32_t* block_table, int32_t max_pages, const int32_t* ctx,
                    double sm_scale, double* out, double* s_out,
                    double* o_pre, double* s_pre) {
    int32_t G = Hq / Hkv;
    int32_t maxn = 0;
    for (int32_t b = 0; b < B; ++b) if (ctx[b] > maxn) maxn = ctx[b];
    int32_t cap = prefix_len + maxn;
    const double** kr = (const double**)malloc(sizeof(double*) * (size_t)(cap > 0 ? cap : 1));
    const double** vr = (const double**)malloc(sizeof(double*) * (size_t)(cap > 0 ? cap : 1));
    for (int32_t b = 0; b < B; ++b) {
        const int32_t* pages = block_table + (int64_t)b * max_pages;
        for (int32_t hq = 0; hq < Hq; ++hq) {
            int32_t hk = hq / G;
            int32_t n = 0;
            for (int32_t t = 0; t < prefix_len; ++t, ++n) {
                kr[n] = token_row(k_cache, prefix_pages, t, Hkv, hk, page, D);
                vr[n] = token_row(v_cache, prefix_pages, t, Hkv, hk, page, D);
            }
            int64_t row = (int64_t)b * Hq + hq;
            attend_rows(D, q + row * D, prefix_len, kr, vr, sm_scale, o_pre + row * D, s_pre + row);
            for (int32_t t = 0; t < ctx[b]; ++t, ++n) {
                kr[n] = token_row(k_cache, pages, t, Hkv, hk, page, D);
                vr[n] = token_row(v_cache, pages, t, Hkv, hk, page, D);
            }
            attend_rows(D, q + row * D, n, kr, vr, sm_scale, out + row * D, s_out + row);
        }
    }
    free(kr);
    free(vr);
}

/*
 * Multi-level cascade ([F2] §⑥: attention level by level, then merge): as
 * oracle_cascade, with L shared segments before each request's suffix.
 * Request b's keys are, in order, seg_len[b*L + l] tokens on the pages
 * seg_pages + seg_page_off[b*L + l] for l = 0 .. L-1 (its group's shared
 * tokens at level l), then its ctx[b] suffix tokens.  out/s_out: one softmax
 * over all of them (the plain definition); o_pre/s_pre: one softmax over the
 * shared tokens only (the prefix state the merge combines with the suffix).
 */
void oracle_cascade_multilevel(int32_t B, int32_t Hq, int32_t Hkv, int32_t D, int32_t page,
                               const double* q, const double* k_cache, const double* v_cache,
                               int32_t L, const int32_t* seg_pages, const int64_t* seg_page_off,
                               const int32_t* seg_len, const int32_t* block_table,
                               int32_t max_pages, const int32_t* ctx, double sm_scale,
                               double* out, double* s_out, double* o_pre, double* s_pre) {
    int32_t G = Hq / Hkv;
    int64_t cap = 1;
    for (int32_t b = 0; b < B; ++b) {
        int64_t n = ctx[b];
        for (int32_t l = 0; l < L; ++l) n += seg_len[(int64_t)b * L + l];
        if (n > cap) cap = n;
    }
    const double** kr = (const double**)malloc(sizeof(double*) * (size_t)cap);
    const double** vr = (const double**)malloc(sizeof(double*) * (size_t)cap);
    for (int32_t b = 0; b < B; ++b) {
        const int32_t* sfx = block_table + (int64_t)b * max_pages;  /* the suffix's pages */
        for (int32_t hq = 0; hq < Hq; ++hq) {
            int32_t hk = hq / G;
            int32_t n = 0;
            for (int32_t l = 0; l < L; ++l) {
                const int32_t* sp = seg_pages + seg_page_off[(int64_t)b * L + l];
                for (int32_t t = 0; t < seg_len[(int64_t)b * L + l]; ++t, ++n) {
                    kr[n] = token_row(k_cache, sp, t, Hkv, hk, page, D);
                    vr[n] = token_row(v_cache, sp, t, Hkv, hk, page, D);
                }
            }
            int64_t row = (int64_t)b * Hq + hq;
            attend_rows(D, q + row * D, n, kr, vr, sm_scale, o_pre + row * D, s_pre + row);
            for (int32_t t = 0; t < ctx[b]; ++t, ++n) {
                kr[n] = token_row(k_cache, sfx, t, Hkv, hk, page, D);
                vr[n] = token_row(v_cache, sfx, t, Hkv, hk, page, D);
            }
            attend_rows(D, q + row * D, n, kr, vr, sm_scale, out + row * D, s_out + row);
        }
    }
    free(kr);
    free(vr);
}
