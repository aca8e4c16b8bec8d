"""Pins for the fp64 oracle: facts fixed by the pages and by mathematics.

Each pin is a function ``pin_xxx(orc)`` that raises AssertionError when the
oracle ``orc`` (an ``oracle.Oracle``) disagrees with a printed value, a closed
form, an invariant, a special case that reduces to a library routine, or brute
force on a tiny input.  ``test_oracle_pins.py`` runs them on the committed
oracle; ``test_oracle_mutants.py`` runs them on copies of the oracle with a
planted mistake and requires that some pin fails for each.

Pages cited (by title and section):
  [F2] "F2 讲解：merge_state，以 2 为底的 LSE 合并"
  [L3] "L3 讲解：split-KV decode 与 LSE 合并"
  [FA] "FlashAttention 的空行 LSE:FA-2 的 +inf 约定与后来的变化"
"""
import math

import numpy as np

from conftest import read_golden, read_golden_table

LN2 = math.log(2.0)
NEG = -math.inf


def _printed(value, printed, decimals):
    """|value - printed| <= half a unit in the last printed place."""
    tol = 0.5 * 10.0 ** (-decimals) + 1e-12
    assert abs(value - printed) <= tol, (value, printed, decimals)


def _one_row_decode(scores, values, page):
    """Decode inputs whose single query reproduces given scores exactly.

    q = e0, k_j = scores[j] * e0, v_j = values[j] * e0, sm_scale = 1, D = 4,
    one head, pages of `page` tokens laid out in order.
    """
    n = len(scores)
    D = 4
    npages = -(-n // page)
    kc = np.zeros((npages, 1, page, D))
    vc = np.zeros((npages, 1, page, D))
    for j in range(n):
        kc[j // page, 0, j % page, 0] = scores[j]
        vc[j // page, 0, j % page, 0] = values[j]
    q = np.zeros((1, 1, D))
    q[0, 0, 0] = 1.0
    bt = np.arange(npages, dtype=np.int32).reshape(1, npages)
    ctx = np.array([n], dtype=np.int32)
    return q, kc, vc, bt, ctx


# ---------------------------------------------------------------- printed values
def pin_worked_example(orc):
    """[L3] §③ table and [F2] §② table: split [1,2] | [3,0] of scores [1,2,3,0]."""
    g = read_golden("worked_example.txt")
    scores = [float(x) for x in g["scores"][0]]
    values = [float(x) for x in g["values"][0]]
    val = lambda k: (float(g[k][0][0]), int(g[k][0][1]))
    q, kc, vc, bt, ctx = _one_row_decode(scores, values, page=2)
    o_part, s_part = orc.attend_splits(q, kc, vc, bt, ctx, 1.0, 2)
    _printed(o_part[0, 0, 0, 0], *val("split0_o"))
    _printed(o_part[0, 0, 1, 0], *val("split1_o"))
    _printed(s_part[0, 0, 0] * LN2, *val("split0_lse"))
    _printed(s_part[0, 0, 1] * LN2, *val("split1_lse"))
    _printed(s_part[0, 0, 0], *val("split0_s"))
    _printed(s_part[0, 0, 1], *val("split1_s"))
    # Merge the two split states in the [S, N, H, D] layout with S = H = 1.
    vo, so, w = orc.merge_states(o_part.reshape(1, 2, 1, 4), s_part.reshape(1, 2, 1),
                                 return_weights=True)
    _printed(w[0, 0, 0], *val("weight0"))
    _printed(w[0, 1, 0], *val("weight1"))
    _printed(vo[0, 0, 0], *val("merged_v"))
    _printed(so[0, 0], *val("merged_s"))
    _printed(so[0, 0] * LN2, *val("merged_lse"))
    # The two-state API gives the same numbers.
    v2, s2 = orc.merge_state(o_part[0, 0, 0:1], s_part[0, 0, 0:1],
                             o_part[0, 0, 1:2], s_part[0, 0, 1:2])
    _printed(v2[0, 0], *val("merged_v"))
    _printed(s2[0], *val("merged_s"))
    # The unsplit definition gives them as well ("和 T5 里一次算完的结果相同").
    of, sf = orc.attend_full(q, kc, vc, bt, ctx, 1.0)
    _printed(of[0, 0, 0], *val("merged_v"))
    _printed(sf[0, 0], *val("merged_s"))
    _printed(sf[0, 0] * LN2, *val("merged_lse"))


def pin_merge_selftest1(orc):
    """[F2] §⑧ 自测 1: equal s = 10 -> v = [0.5, 0.5], s = 11."""
    g = read_golden("merge_selftests.txt")
    f = lambda k: np.array([float(x) for x in g[k][0]])
    v, s = orc.merge_state(f("selftest1_v_a")[None], f("selftest1_s_a"),
                           f("selftest1_v_b")[None], f("selftest1_s_b"))
    assert np.array_equal(v[0], f("selftest1_v")), v
    assert s[0] == f("selftest1_s")[0], s


def pin_merge_selftest2(orc):
    """[F2] §⑧ 自测 2: a natural lse of 5 is s = 7.21 in base 2.

    A single key with score 5 has natural lse exactly 5; the oracle's s for
    it must read 7.21.
    """
    g = read_golden("merge_selftests.txt")
    lse = float(g["selftest2_lse"][0][0])
    q, kc, vc, bt, ctx = _one_row_decode([lse], [1.0], page=1)
    _, s = orc.attend_full(q, kc, vc, bt, ctx, 1.0)
    _printed(s[0, 0], float(g["selftest2_s"][0][0]), int(g["selftest2_s"][0][1]))


def pin_split_weights(orc):
    """[FA] §0.2: natural LSEs 1 and 0 get weights about 0.731 and 0.269."""
    g = read_golden("split_weights.txt")
    lse = np.array([float(x) for x in g["lse"][0]])
    want = [float(x) for x in g["weights"][0][:2]]
    dec = int(g["weights"][0][2])
    v = np.zeros((1, 2, 1, 1))
    _, _, w = orc.merge_states(v, (lse / LN2).reshape(1, 2, 1), return_weights=True)
    wn = w[0, :, 0] / w[0, :, 0].sum()
    _printed(wn[0], want[0], dec)
    _printed(wn[1], want[1], dec)


def pin_l3_selftest(orc):
    """[L3] §⑧ 自测 2: lse 0 and 10; equal o merge to themselves, else ~[0.00005, 0.99995]."""
    g = read_golden("l3_selftest_merge.txt")
    f = lambda k: np.array([float(x) for x in g[k][0]])
    s = f("lse") / LN2
    v, _ = orc.merge_state(f("same_o")[None], s[:1], f("same_o")[None], s[1:])
    assert np.allclose(v[0], f("same_result"), rtol=0, atol=1e-15), v
    v, _ = orc.merge_state(f("diff_o_a")[None], s[:1], f("diff_o_b")[None], s[1:])
    res = g["diff_result"][0]
    _printed(v[0, 0], float(res[0]), int(res[2]))
    _printed(v[0, 1], float(res[1]), int(res[2]))


def pin_poisoned_merge(orc):
    """[FA] §1 and §2.2: +inf or NaN incoming LSE must not poison the merge."""
    g = read_golden("poisoned_merge.txt")
    lse = [float(x) for x in g["lse"][0]]
    assert lse[1] == math.inf
    va = np.array([[1.5, -2.0, 3.25]])
    vb = np.array([[7.0, 8.0, 9.0]])
    for bad in (math.inf, math.nan):
        v, s = orc.merge_state(va, np.array([lse[0]]), vb, np.array([bad]))
        assert np.array_equal(v, va) and s[0] == lse[0], (v, s)
        v, s = orc.merge_state(vb, np.array([bad]), va, np.array([lse[0]]))
        assert np.array_equal(v, va) and s[0] == lse[0], (v, s)
    # N-state: +inf and NaN next to one finite state reduce to that state.
    v3 = np.stack([vb[0], va[0], vb[0]])[None, :, None, :]
    s3 = np.array([math.inf, lse[0], math.nan]).reshape(1, 3, 1)
    vo, so = orc.merge_states(v3, s3)
    assert np.array_equal(vo[0, 0], va[0]) and so[0, 0] == lse[0]
    # All poisoned -> empty.
    vo, so = orc.merge_states(v3, np.array([math.inf, math.nan, math.inf]).reshape(1, 3, 1))
    assert np.all(vo == 0) and so[0, 0] == NEG


def pin_split_ranges(orc):
    """[L3] §② examples (ctx 1000, 37) and §⑧ 自测 1 (ctx 100), bit-exact."""
    rows = read_golden_table("split_ranges.txt")
    for ctx, page, ns, num_pages, pps, split, p0, p1, ntok in rows:
        a, b = orc.split_range(ctx, page, ns, split)
        assert (a, b) == (p0, p1), (ctx, split, a, b)
        # num_pages and pages_per_split follow from the ranges.
        assert orc.split_range(ctx, page, ns, 0)[1] == min(pps, num_pages)
        assert orc.split_range(ctx, page, ns, ns - 1)[1] == num_pages
        got_tok = max(0, min(b * page, ctx) - a * page) if b > a else 0
        assert got_tok == ntok, (ctx, split, got_tok, ntok)


def pin_empty_splits_in_decode(orc):
    """[L3] §④: an empty split writes o = 0 and s = -inf (ctx = 37, 4 splits)."""
    rng = np.random.default_rng(1)
    D, page = 8, 16
    for ctx_len, ns in ((37, 4), (1, 8), (16, 2), (17, 4)):
        npg = -(-ctx_len // page)
        kc = rng.standard_normal((npg, 1, page, D))
        vc = rng.standard_normal((npg, 1, page, D))
        q = rng.standard_normal((1, 1, D))
        bt = np.arange(npg, dtype=np.int32)[None]
        o, s = orc.attend_splits(q, kc, vc, bt, np.array([ctx_len], np.int32), 0.3, ns)
        for sp in range(ns):
            a, b = orc.split_range(ctx_len, page, ns, sp)
            if b <= a:
                assert s[0, 0, sp] == NEG and np.all(o[0, 0, sp] == 0.0)
            else:
                assert np.isfinite(s[0, 0, sp]) and np.all(np.isfinite(o[0, 0, sp]))


def pin_plan_table(orc):
    """[L3] §⑥: the suitable split counts of the page's table, exactly."""
    for B, ctx, Hkv, page, sm, want in read_golden_table("plan_table.txt"):
        assert orc.plan([ctx] * B, Hkv, page, sm) == want, (B, ctx)


# ---------------------------------------------------------------- merge identities
def _rand_states(rng, shape, D, empty_p=0.0):
    v = rng.standard_normal(shape + (D,))
    s = rng.uniform(-20, 20, shape)
    e = rng.random(shape) < empty_p
    s[e] = NEG
    v[e] = 0.0
    return v, s


def pin_empty_and_double_empty(orc):
    """[F2] §⑤: empty + normal = normal (bit-exact); empty + empty = (0, -inf), no NaN."""
    rng = np.random.default_rng(2)
    va, sa = _rand_states(rng, (64,), 16)
    ve = np.zeros_like(va)
    se = np.full(64, NEG)
    v, s = orc.merge_state(va, sa, ve, se)
    assert np.array_equal(v, va) and np.array_equal(s, sa)
    v, s = orc.merge_state(ve, se, va, sa)
    assert np.array_equal(v, va) and np.array_equal(s, sa)
    v, s = orc.merge_state(ve, se, ve, se)
    assert np.all(v == 0.0) and np.all(s == NEG)
    vo, so = orc.merge_states(np.zeros((3, 5, 2, 4)), np.full((3, 5, 2), NEG))
    assert np.all(vo == 0.0) and np.all(so == NEG)


def pin_commutative(orc):
    """[F2] §①: merging is commutative (bit-exact, the formula is symmetric)."""
    rng = np.random.default_rng(3)
    va, sa = _rand_states(rng, (256,), 32, 0.1)
    vb, sb = _rand_states(rng, (256,), 32, 0.1)
    v1, s1 = orc.merge_state(va, sa, vb, sb)
    v2, s2 = orc.merge_state(vb, sb, va, sa)
    assert np.array_equal(v1, v2) and np.array_equal(s1, s2)


def pin_associative(orc):
    """[F2] §①: any grouping gives the same state (to fp64 rounding)."""
    rng = np.random.default_rng(4)
    (va, sa), (vb, sb), (vc, sc) = (_rand_states(rng, (128,), 8, 0.1) for _ in range(3))
    l_v, l_s = orc.merge_state(*orc.merge_state(va, sa, vb, sb), vc, sc)
    r_v, r_s = orc.merge_state(va, sa, *orc.merge_state(vb, sb, vc, sc))
    n_v, n_s = orc.merge_states(np.stack([va, vb, vc], 1)[:, :, None, :],
                                np.stack([sa, sb, sc], 1)[:, :, None])
    for v, s in ((r_v, r_s), (n_v[:, 0], n_s[:, 0])):
        assert np.allclose(l_v, v, rtol=1e-12, atol=1e-12)
        fin = np.isfinite(l_s)
        assert np.array_equal(fin, np.isfinite(s))
        assert np.allclose(l_s[fin], s[fin], rtol=0, atol=1e-12)


def pin_equal_states(orc):
    """K identical states: v unchanged, s + log2 K (the denominator is K times larger)."""
    rng = np.random.default_rng(5)
    v1, s1 = _rand_states(rng, (4, 3), 16)
    for K in (1, 2, 3, 7, 64):
        v = np.repeat(v1[:, None], K, axis=1)
        s = np.repeat(s1[:, None], K, axis=1)
        vo, so = orc.merge_states(v, s)
        assert np.allclose(vo, v1, rtol=1e-14, atol=1e-14)
        assert np.allclose(so, s1 + math.log2(K), rtol=0, atol=1e-12)


def pin_shift_invariance(orc):
    """Adding c to every s leaves v unchanged and adds c to the merged s."""
    rng = np.random.default_rng(6)
    v, s = _rand_states(rng, (3, 9, 2), 8, 0.2)
    vo, so = orc.merge_states(v, s)
    for c in (-50.0, 0.75, 300.0):
        vc, sc = orc.merge_states(v, s + c)
        assert np.allclose(vc, vo, rtol=1e-12, atol=1e-13)
        fin = np.isfinite(so)
        assert np.allclose(sc[fin], so[fin] + c, rtol=0, atol=1e-11)


def pin_merge_states_layout(orc):
    """[F2] §④ figure: with S=2, N=3, H=2 the program (pos=1, h=1) reads offsets 7, 9, 11."""
    S, N, H, D = 2, 3, 2, 4
    s = np.full((S, N, H), NEG)
    v = np.zeros((S, N, H, D))
    flat_s = s.reshape(-1)
    flat_v = v.reshape(-1, D)
    for k, off in enumerate((7, 9, 11)):
        flat_s[off] = 0.0
        flat_v[off] = k + 1.0
    vo, so = orc.merge_states(v, s)
    assert np.allclose(vo[1, 1], 2.0, rtol=0, atol=1e-15)  # mean of 1, 2, 3
    assert abs(so[1, 1] - math.log2(3.0)) < 1e-15
    for pos, h in ((0, 0), (0, 1), (1, 0)):
        assert so[pos, h] == NEG and np.all(vo[pos, h] == 0.0)


def pin_two_state_forms_agree(orc):
    """merge_states with N = 2 equals merge_state; N = 1 is the identity (empty -> (0,-inf))."""
    rng = np.random.default_rng(7)
    va, sa = _rand_states(rng, (5, 6), 16, 0.2)
    vb, sb = _rand_states(rng, (5, 6), 16, 0.2)
    sa[0, 0] = sb[0, 0] = NEG
    v2, s2 = orc.merge_state(va, sa, vb, sb)
    vn, sn = orc.merge_states(np.stack([va, vb], 1), np.stack([sa, sb], 1))
    assert np.array_equal(v2, vn) and np.array_equal(s2, sn)
    v1, s1 = orc.merge_states(va[:, None], sa[:, None])
    ne = np.isfinite(sa)
    assert np.array_equal(v1[ne], va[ne]) and np.array_equal(s1[ne], sa[ne])
    assert np.all(v1[~ne] == 0) and np.all(s1[~ne] == NEG)


# ---------------------------------------------------------------- decode attention
def _rand_decode(rng, B, Hq, Hkv, D, page, ctx, pool_extra=3):
    need = sum(-(-c // page) for c in ctx)
    P = need + pool_extra
    perm = rng.permutation(P).astype(np.int32)
    maxp = max(1, max(-(-c // page) for c in ctx))
    bt = np.zeros((B, maxp), np.int32)
    k = 0
    for b, c in enumerate(ctx):
        n = -(-c // page)
        bt[b, :n] = perm[k:k + n]
        k += n
    kc = rng.standard_normal((P, Hkv, page, D))
    vc = rng.standard_normal((P, Hkv, page, D))
    q = rng.standard_normal((B, Hq, D))
    return q, kc, vc, bt, np.array(ctx, np.int32)


def pin_closed_forms(orc):
    """q = 0: every score is 0, so o = mean of v and s = log2(ctx); one key: o = v, s = score/ln2."""
    rng = np.random.default_rng(8)
    q, kc, vc, bt, ctx = _rand_decode(rng, 2, 4, 2, 8, 4, [7, 13])
    o, s = orc.attend_full(np.zeros_like(q), kc, vc, bt, ctx, 0.5)
    for b in range(2):
        n = int(ctx[b])
        for hq in range(4):
            rows = np.stack([vc[bt[b, t // 4], hq // 2, t % 4] for t in range(n)])
            assert np.allclose(o[b, hq], rows.mean(0), rtol=1e-13, atol=1e-14)
            assert abs(s[b, hq] - math.log2(n)) < 1e-13
    q, kc, vc, bt, ctx = _rand_decode(rng, 1, 2, 1, 8, 4, [1])
    o, s = orc.attend_full(q, kc, vc, bt, ctx, 0.7)
    for hq in range(2):
        k0 = kc[bt[0, 0], 0, 0]
        assert np.allclose(o[0, hq], vc[bt[0, 0], 0, 0], rtol=0, atol=1e-15)
        assert abs(s[0, hq] - 0.7 * float(q[0, hq] @ k0) / LN2) < 1e-13


def pin_brute_force(orc):
    """Tiny inputs against scipy's logsumexp and softmax over explicitly gathered keys."""
    from scipy.special import logsumexp, softmax
    rng = np.random.default_rng(9)
    for (B, Hq, Hkv, D, page, ctx, ns) in (
            (2, 4, 2, 8, 4, [5, 11], 3), (3, 6, 3, 4, 2, [1, 2, 9], 4),
            (1, 8, 1, 16, 16, [37], 4), (2, 2, 2, 8, 8, [64, 3], 8)):
        q, kc, vc, bt, cx = _rand_decode(rng, B, Hq, Hkv, D, page, ctx)
        scale = 0.37
        o, s = orc.attend_full(q, kc, vc, bt, cx, scale)
        op, sp = orc.attend_splits(q, kc, vc, bt, cx, scale, ns)
        G = Hq // Hkv
        for b in range(B):
            n = ctx[b]
            for hq in range(Hq):
                K = np.stack([kc[bt[b, t // page], hq // G, t % page] for t in range(n)])
                V = np.stack([vc[bt[b, t // page], hq // G, t % page] for t in range(n)])
                x = scale * (K @ q[b, hq])
                assert abs(s[b, hq] - logsumexp(x) / LN2) < 1e-12
                assert np.allclose(o[b, hq], softmax(x) @ V, rtol=1e-12, atol=1e-13)
                for spl in range(ns):
                    a, e = orc.split_range(n, page, ns, spl)
                    t0, t1 = a * page, min(e * page, n)
                    if e <= a:
                        continue
                    xs = x[t0:t1]
                    assert abs(sp[b, hq, spl] - logsumexp(xs) / LN2) < 1e-12
                    assert np.allclose(op[b, hq, spl], softmax(xs) @ V[t0:t1], rtol=1e-12,
                                       atol=1e-13)


def pin_split_merge_identity(orc):
    """[FA] §0.2 / [L3] §③: merging the split states reproduces unsplit attention."""
    rng = np.random.default_rng(10)
    for ctx, ns in (([37, 1000, 1], 4), ([100, 16, 17], 64), ([0, 5], 3), ([2048], 1)):
        q, kc, vc, bt, cx = _rand_decode(rng, len(ctx), 4, 2, 16, 16, ctx)
        o, s = orc.attend_full(q, kc, vc, bt, cx, 0.25)
        op, sp = orc.attend_splits(q, kc, vc, bt, cx, 0.25, ns)
        B, Hq = o.shape[:2]
        vo, so = orc.merge_states(op.reshape(B * Hq, ns, 1, -1), sp.reshape(B * Hq, ns, 1))
        vo = vo.reshape(o.shape)
        so = so.reshape(s.shape)
        assert np.allclose(vo, o, rtol=1e-12, atol=1e-13)
        fin = np.isfinite(s)
        assert np.array_equal(fin, np.isfinite(so))
        assert np.allclose(so[fin], s[fin], rtol=0, atol=1e-12)
        for b, c in enumerate(ctx):
            if c == 0:
                assert np.all(o[b] == 0) and np.all(s[b] == NEG)


def pin_gqa_mapping(orc):
    """Query head hq reads KV head hq // (Hq/Hkv): contiguous groups."""
    Hq, Hkv, D, page = 8, 2, 4, 4
    kc = np.zeros((2, Hkv, page, D))
    vc = np.zeros((2, Hkv, page, D))
    for hk in range(Hkv):
        vc[:, hk] = hk + 1.0
    q = np.ones((1, Hq, D))
    bt = np.array([[0, 1]], np.int32)
    o, _ = orc.attend_full(q, kc, vc, bt, np.array([6], np.int32), 1.0)
    for hq in range(Hq):
        assert np.allclose(o[0, hq], hq // (Hq // Hkv) + 1.0, rtol=0, atol=1e-15)


def pin_page_table_permutation(orc):
    """Moving pages around the pool (and the table with them) changes nothing."""
    rng = np.random.default_rng(11)
    q, kc, vc, bt, cx = _rand_decode(rng, 2, 4, 2, 8, 4, [13, 6])
    o, s = orc.attend_full(q, kc, vc, bt, cx, 0.3)
    perm = rng.permutation(kc.shape[0])
    inv = np.argsort(perm)
    o2, s2 = orc.attend_full(q, kc[perm], vc[perm], inv[bt].astype(np.int32), cx, 0.3)
    assert np.array_equal(o, o2) and np.array_equal(s, s2)


def pin_scale_and_large_scores(orc):
    """Scale folds into q; a huge common score offset shifts s and leaves o alone."""
    rng = np.random.default_rng(12)
    q, kc, vc, bt, cx = _rand_decode(rng, 1, 2, 1, 8, 4, [9])
    o, s = orc.attend_full(q, kc, vc, bt, cx, 0.5)
    o2, s2 = orc.attend_full(2.0 * q, kc, vc, bt, cx, 0.25)
    assert np.allclose(o, o2, rtol=1e-13, atol=1e-14) and np.allclose(s, s2, rtol=0, atol=1e-12)
    scores = rng.uniform(-3, 3, 9)
    vals = rng.standard_normal(9)
    base = _one_row_decode(list(scores), list(vals), 4)
    big = _one_row_decode(list(scores + 1000.0), list(vals), 4)
    ob, sb = orc.attend_full(*base, 1.0)
    og, sg = orc.attend_full(*big, 1.0)
    assert np.all(np.isfinite(og)) and np.isfinite(sg[0, 0])
    assert np.allclose(og, ob, rtol=1e-11, atol=1e-12)
    assert abs(sg[0, 0] - sb[0, 0] - 1000.0 / LN2) < 1e-9


def pin_cascade(orc):
    """[F2] §⑥: prefix || suffix equals one softmax; prefix state then merge reproduces it."""
    rng = np.random.default_rng(13)
    Hq, Hkv, D, page = 4, 2, 8, 4
    for prefix_len, ctx in ((12, [5, 0, 9]), (0, [3, 7, 1]), (7, [0, 0, 4])):
        npre = -(-prefix_len // page)
        q, kc, vc, bt, cx = _rand_decode(rng, 3, Hq, Hkv, D, page, ctx, pool_extra=npre + 2)
        used = set(bt[bt >= 0].reshape(-1).tolist()) if max(ctx) > 0 else set()
        free = [p for p in range(kc.shape[0]) if p not in used]
        pre = np.array(free[:npre], np.int32)
        out, s, o_pre, s_pre = orc.cascade(q, kc, vc, pre, prefix_len, bt, cx, 0.4)
        # Concatenated block tables: prefix pages then suffix pages, when the
        # prefix fills whole pages the token order is the same.
        if prefix_len % page == 0:
            cat = np.concatenate([np.repeat(pre[None], 3, 0), bt], 1).astype(np.int32)
            of, sf = orc.attend_full(q, kc, vc, cat, cx + prefix_len, 0.4)
            assert np.allclose(out, of, rtol=1e-13, atol=1e-14)
            assert np.allclose(s[np.isfinite(s)], sf[np.isfinite(sf)], rtol=0, atol=1e-12)
        pt = np.repeat(pre[None], 3, 0) if npre else np.zeros((3, 1), np.int32)
        op, sp = orc.attend_full(q, kc, vc, pt, np.full(3, prefix_len, np.int32), 0.4)
        assert np.allclose(o_pre, op, rtol=1e-13, atol=1e-14)
        assert np.array_equal(np.isfinite(s_pre), np.isfinite(sp))
        ns = 4
        osu, ssu = orc.attend_splits(q, kc, vc, bt, cx, 0.4, ns)
        vsu, ssm = orc.merge_states(osu.reshape(-1, ns, 1, D), ssu.reshape(-1, ns, 1))
        mv, ms = orc.merge_state(o_pre.reshape(-1, D), s_pre.reshape(-1),
                                 vsu.reshape(-1, D), ssm.reshape(-1))
        assert np.allclose(mv.reshape(out.shape), out, rtol=1e-12, atol=1e-13)
        fin = np.isfinite(s)
        assert np.array_equal(fin, np.isfinite(ms.reshape(s.shape)))
        assert np.allclose(ms.reshape(s.shape)[fin], s[fin], rtol=0, atol=1e-12)


def pin_cascade_multilevel(orc):
    """[F2] §⑥ (attention level by level, then merge): shared tokens at several
    levels, then the suffix, equal one softmax over their concatenation; one
    level of one group is the two-level cascade; the prefix state is the merge
    of the levels' own states."""
    rng = np.random.default_rng(17)
    B, Hq, Hkv, D, page = 5, 4, 2, 8, 4
    ctx = [5, 0, 9, 3, 6]
    # levels[l] = groups (r0, r1, length); pages drawn after the suffix pages.
    for spec in (
            [[(0, 5, 12)]],                                    # one level, one group
            [[(0, 5, 8)], [(0, 2, 4), (2, 5, 12)], [(0, 3, 0), (3, 5, 8)]],   # whole pages
            [[(0, 5, 7)], [(0, 1, 5), (1, 4, 0), (4, 5, 10)]],  # partial pages, an empty group
    ):
        npg = sum(-(-ln // page) for lv in spec for (_, _, ln) in lv)
        q, kc, vc, bt, cx = _rand_decode(rng, B, Hq, Hkv, D, page, ctx, pool_extra=npg + 1)
        used = set(bt.reshape(-1).tolist()) if max(ctx) > 0 else set()
        free = [p for p in range(kc.shape[0]) if p not in used]
        levels, at = [], 0
        for lv in spec:
            groups = []
            for (r0, r1, ln) in lv:
                n = -(-ln // page)
                groups.append((r0, r1, np.array(free[at:at + n], np.int32), ln))
                at += n
            levels.append(groups)
        out, s, o_pre, s_pre = orc.cascade_multilevel(q, kc, vc, levels, bt, cx, 0.4)
        if len(spec) == 1 and len(spec[0]) == 1:
            o2, s2, op2, sp2 = orc.cascade(q, kc, vc, levels[0][0][2], spec[0][0][2], bt, cx, 0.4)
            assert np.allclose(out, o2, rtol=1e-13, atol=1e-14)
            assert np.allclose(s, s2, rtol=0, atol=1e-12)
            assert np.allclose(o_pre, op2, rtol=1e-13, atol=1e-14)
            assert np.allclose(s_pre, sp2, rtol=0, atol=1e-12)
        if all(ln % page == 0 for lv in spec for (_, _, ln) in lv):
            # Whole pages: one block table per request, shared pages first.
            rows, lens = [], []
            for b in range(B):
                pg, n = [], 0
                for groups in levels:
                    for (r0, r1, pages, ln) in groups:
                        if r0 <= b < r1:
                            pg += pages.tolist()
                            n += ln
                pg += bt[b, :-(-int(cx[b]) // page)].tolist() if cx[b] else []
                rows.append(pg)
                lens.append(n + int(cx[b]))
            cat = np.zeros((B, max(1, max(len(r) for r in rows))), np.int32)
            for b, r in enumerate(rows):
                cat[b, :len(r)] = r
            of, sf = orc.attend_full(q, kc, vc, cat, np.array(lens, np.int32), 0.4)
            assert np.allclose(out, of, rtol=1e-13, atol=1e-14)
            fin = np.isfinite(sf)
            assert np.array_equal(np.isfinite(s), fin)
            assert np.allclose(s[fin], sf[fin], rtol=0, atol=1e-12)
        # The prefix state is the merge of each level's own state (each
        # group's tokens alone, through the unsplit definition), and out is
        # that merged with the suffix state.
        acc_v = np.zeros((B * Hq, D))
        acc_s = np.full(B * Hq, -np.inf)
        for groups in levels:
            lv_v = np.zeros((B, Hq, D))
            lv_s = np.full((B, Hq), -np.inf)
            for (r0, r1, pages, ln) in groups:
                nb = r1 - r0
                tab = np.repeat(pages[None], nb, 0) if pages.size else np.zeros((nb, 1), np.int32)
                ov, sv = orc.attend_full(q[r0:r1], kc, vc, tab, np.full(nb, ln, np.int32), 0.4)
                lv_v[r0:r1], lv_s[r0:r1] = ov, sv
            acc_v, acc_s = orc.merge_state(acc_v, acc_s, lv_v.reshape(-1, D), lv_s.reshape(-1))
        assert np.allclose(acc_v.reshape(o_pre.shape), o_pre, rtol=1e-12, atol=1e-13)
        fin = np.isfinite(s_pre)
        assert np.array_equal(np.isfinite(acc_s.reshape(s_pre.shape)), fin)
        assert np.allclose(acc_s.reshape(s_pre.shape)[fin], s_pre[fin], rtol=0, atol=1e-12)
        ov, sv = orc.attend_full(q, kc, vc, bt, cx, 0.4)
        mv, ms = orc.merge_state(o_pre.reshape(-1, D), s_pre.reshape(-1), ov.reshape(-1, D),
                                 sv.reshape(-1))
        assert np.allclose(mv.reshape(out.shape), out, rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------- per-sequence split counts
def pin_plan_varlen(orc):
    """[L3] §⑥ per-sequence split counts, read as: n pages get ceil(n / P)
    splits of at most P pages, clamped to [1, max_splits].  Values worked by
    hand for page 16: ctx 0, 1, 128, 129, 1000, 2048, 4096 are 0, 1, 8, 9, 63,
    128, 256 pages."""
    ctx = [0, 1, 128, 129, 1000, 2048, 4096]
    assert orc.plan_varlen(ctx, 16, 16, 8).tolist() == [1, 1, 1, 2, 8, 16, 16]
    assert orc.plan_varlen(ctx, 16, 4, 8).tolist() == [1, 1, 1, 2, 4, 4, 4]
    assert orc.plan_varlen(ctx, 16, 64, 8).tolist() == [1, 1, 1, 2, 8, 16, 32]
    assert orc.plan_varlen(ctx, 16, 16, 1).tolist() == [1, 1, 8, 9, 16, 16, 16]
    assert orc.plan_varlen(ctx, 16, 256, 64).tolist() == [1, 1, 1, 1, 1, 2, 4]


def pin_varlen_splits_printed_ranges(orc):
    """Per-sequence split counts reuse the [L3] §② ranges with each sequence's
    own count: a batch of ctx 100, 37, 1000 (page 16) with 4, 1 and 4 splits.
    Sequence 0 is §⑧ 自测 1 (pages [0,2), [2,4), [4,6), [6,7)), sequence 2 the
    §② ctx = 1000 example (split 3 is pages 48-62), sequence 1 is not split, so
    its one state is the whole sequence's; the slots past a sequence's count
    hold empty states.  Every state is checked by brute force over the tokens
    of the printed page ranges."""
    from scipy.special import logsumexp, softmax
    rows = read_golden_table("split_ranges.txt")
    printed = {}
    for ctx, page, ns, _, _, split, p0, p1, _ in rows:
        printed[(ctx, split)] = (p0, p1)
    rng = np.random.default_rng(31)
    ctx = [100, 37, 1000]
    ns = np.array([4, 1, 4], np.int32)
    q, kc, vc, bt, cx = _rand_decode(rng, 3, 4, 2, 8, 16, ctx)
    scale = 0.3
    op, sp = orc.attend_splits_varlen(q, kc, vc, bt, cx, scale, ns, 4)
    for b, c in enumerate(ctx):
        for hq in range(4):
            K = np.stack([kc[bt[b, t // 16], hq // 2, t % 16] for t in range(c)])
            V = np.stack([vc[bt[b, t // 16], hq // 2, t % 16] for t in range(c)])
            x = scale * (K @ q[b, hq])
            for spl in range(4):
                if spl >= ns[b]:
                    assert sp[b, hq, spl] == NEG and np.all(op[b, hq, spl] == 0.0)
                    continue
                p0, p1 = printed[(c, spl)] if ns[b] == 4 else (0, -(-c // 16))
                t0, t1 = p0 * 16, min(p1 * 16, c)
                assert abs(sp[b, hq, spl] - logsumexp(x[t0:t1]) / LN2) < 1e-12
                assert np.allclose(op[b, hq, spl], softmax(x[t0:t1]) @ V[t0:t1], rtol=1e-12,
                                   atol=1e-13)
    # With the same count for every sequence it is the uniform split.
    op4, sp4 = orc.attend_splits(q, kc, vc, bt, cx, scale, 4)
    o4, s4 = orc.attend_splits_varlen(q, kc, vc, bt, cx, scale, np.full(3, 4, np.int32), 4)
    assert np.array_equal(op4, o4) and np.array_equal(sp4, s4)


def pin_varlen_split_merge_identity(orc):
    """Merging the first ns_b states of each sequence gives unsplit attention
    ([FA] §0.2), whatever the per-sequence counts."""
    rng = np.random.default_rng(32)
    ctx = [0, 5, 37, 300, 1000, 16, 17]
    q, kc, vc, bt, cx = _rand_decode(rng, len(ctx), 4, 2, 8, 16, ctx)
    ns = orc.plan_varlen(ctx, 16, 8, 2)
    assert ns.tolist() == [1, 1, 2, 8, 8, 1, 1]
    op, sp = orc.attend_splits_varlen(q, kc, vc, bt, cx, 0.25, ns, 8)
    o, s = orc.attend_full(q, kc, vc, bt, cx, 0.25)
    for b in range(len(ctx)):
        n = int(ns[b])
        vo, so = orc.merge_states(op[b, :, :n].transpose(1, 0, 2)[None], sp[b, :, :n].T[None])
        fin = np.isfinite(s[b])
        assert np.array_equal(fin, np.isfinite(so[0]))
        assert np.allclose(vo[0], o[b], rtol=1e-12, atol=1e-13)
        assert np.allclose(so[0][fin], s[b][fin], rtol=0, atol=1e-12)


PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
