"""Parity of the two-level cascade (tcgen05 shared-prefix pass + split-KV suffix +
merges) with the fp64 oracle: the prefix state, the suffix split states and the
merged output, on small and ragged cases, every group size, empty prefixes and
suffixes, and the full B=64 / 8192-token-prefix workload.

Pages: "F2 讲解：merge_state，以 2 为底的 LSE 合并" §⑥ (cascade);
"L3 讲解：split-KV decode 与 LSE 合并" §①-④ (the suffix)."""
import math

import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import (DEC_LSE_ATOL, DEC_O_TOL, assert_s_close, assert_v_close,
                         require_gpu, skv)
from split_kv_lse_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def lib():
    require_gpu()
    return skv()


def poison_unused(d):
    """NaN in every pool slot no request may read: tails of partial last pages
    (prefix and suffixes) and unused pages."""
    kc, vc = d["k_cache"], d["v_cache"]
    used = set()
    npre = -(-d["prefix_len"] // 16)
    pre = d["prefix_pages"][:npre].tolist()
    used.update(pre)
    if d["prefix_len"] % 16 and npre:
        kc[pre[-1], :, d["prefix_len"] % 16:] = float("nan")
        vc[pre[-1], :, d["prefix_len"] % 16:] = float("nan")
    for b, c in enumerate(d["ctx"].tolist()):
        n = -(-c // 16)
        pages = d["block_table"][b, :n].tolist()
        used.update(pages)
        if c % 16:
            kc[pages[-1], :, c % 16:] = float("nan")
            vc[pages[-1], :, c % 16:] = float("nan")
    for pid in range(kc.shape[0]):
        if pid not in used:
            kc[pid] = float("nan")
            vc[pid] = float("nan")


def run_and_check(lib, d, ns, poison=True):
    if poison:
        poison_unused(d)
    g = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
    pp = g["prefix_pages"] if g["prefix_pages"].numel() else torch.zeros(1, dtype=torch.int32,
                                                                       device=DEV)
    out, lse, o_pre, s_pre, o_part, lse_part = lib.cascade_decode(
        g["q"], g["k_cache"], g["v_cache"], pp, d["prefix_len"], g["block_table"], g["ctx"], ns,
        d["sm_scale"])
    torch.cuda.synchronize()
    assert lib.get_device_error() == (0, 0)
    o_r, s_r, op_r, sp_r = oracle.cascade(d["q"], d["k_cache"], d["v_cache"], d["prefix_pages"],
                                          d["prefix_len"], d["block_table"], d["ctx"],
                                          d["sm_scale"])
    atol, rtol_part, rtol_out = DEC_O_TOL[d["q"].dtype]
    assert out.dtype == d["q"].dtype
    assert_s_close(s_pre, sp_r, DEC_LSE_ATOL, "s_pre")
    assert_v_close(o_pre, op_r, atol, rtol_part, "o_pre", empty_rows=(sp_r == -math.inf))
    opr, lpr = oracle.attend_splits(d["q"], d["k_cache"], d["v_cache"], d["block_table"],
                                    d["ctx"], d["sm_scale"], ns)
    assert_s_close(lse_part, lpr, DEC_LSE_ATOL, "lse_part")
    assert_v_close(o_part, opr, atol, rtol_part, "o_part", empty_rows=(lpr == -math.inf))
    assert_s_close(lse, s_r, DEC_LSE_ATOL, "lse_out")
    assert_v_close(out, o_r, atol, rtol_out, "out", empty_rows=(s_r == -math.inf))
    return out, lse, o_pre, s_pre


@pytest.mark.parametrize("prefix_len", [128, 200, 1000, 16])
def test_cascade_small(lib, prefix_len):
    d = W.cascade_inputs(3, 8, 2, 128, 16, prefix_len, [5, 0, 37], seed=prefix_len)
    run_and_check(lib, d, 4)


@pytest.mark.parametrize("G", [1, 2, 4, 8])
def test_cascade_group_sizes(lib, G):
    # B*G rows spanning two M tiles of 128 rows, the second partial.
    B = (160 + G - 1) // G
    ctx = [int(x) for x in np.random.default_rng(G).integers(0, 300, B)]
    d = W.cascade_inputs(B, 2 * G, 2, 128, 16, 777, ctx, seed=10 + G)
    run_and_check(lib, d, 8)


def test_cascade_empty_prefix(lib):
    d = W.cascade_inputs(2, 8, 2, 128, 16, 0, [40, 3], seed=20)
    out, lse, o_pre, s_pre = run_and_check(lib, d, 4)
    assert torch.all(s_pre.cpu() == -math.inf) and torch.all(o_pre.cpu() == 0)


def test_cascade_empty_suffixes(lib):
    d = W.cascade_inputs(2, 8, 2, 128, 16, 300, [0, 0], seed=21)
    run_and_check(lib, d, 4)


def test_cascade_everything_empty(lib):
    d = W.cascade_inputs(2, 8, 2, 128, 16, 0, [0, 0], seed=22)
    out, lse, _, _ = run_and_check(lib, d, 2, poison=False)
    assert torch.all(lse.cpu() == -math.inf) and torch.all(out.cpu() == 0)


def test_cascade_prefix_rescale_in_some_rows_only(lib):
    """Scores that rise along the prefix for the even query heads only: their
    rows pass the running max by more than the lazy-rescale threshold in
    block after block while the odd heads' rows, in the same warps, never
    do (the rescale of O in TMEM is warp-wide)."""
    B, G, Hkv, plen = 40, 4, 2, 1000
    ctx = [int(x) for x in np.random.default_rng(31).integers(0, 200, B)]
    d = W.cascade_inputs(B, G * Hkv, Hkv, 128, 16, plen, ctx, seed=31)
    pages = d["prefix_pages"].tolist()
    for t in range(plen):
        d["k_cache"][pages[t // 16], :, t % 16, 0] = t / 16.0  # exact in fp16 and bf16
    d["q"][:, 0::2, 0] = 8.0
    d["q"][:, 1::2, 0] = 0.0
    run_and_check(lib, d, 4)


def test_cascade_full_workload(lib):
    """B=64, Hq=32, Hkv=8, an 8192-token shared prefix, suffixes of 1..2048 tokens, NS=16."""
    d = W.cascade_mixed()
    run_and_check(lib, d, d["num_splits"], poison=False)


@pytest.mark.parametrize("G", [1, 4])
def test_cascade_bf16(lib, G):
    """bf16 q/K/V: the prefix pass on the tensor cores with bf16 operands (P in
    bf16), bf16 suffix decode, bf16 output."""
    B = (160 + G - 1) // G
    ctx = [int(x) for x in np.random.default_rng(30 + G).integers(0, 300, B)]
    d = W.cascade_inputs(B, 2 * G, 2, 128, 16, 777, ctx, seed=30 + G, dtype=torch.bfloat16)
    run_and_check(lib, d, 8)


def test_cascade_bf16_full_workload(lib):
    """The B=64 cascade workload in bf16."""
    fp16 = W.cascade_mixed()
    suffix = fp16["ctx"].tolist()  # the same suffix lengths as the fp16 workload
    d = W.cascade_inputs(64, 32, 8, 128, 16, 8192, suffix, 0, dtype=torch.bfloat16)
    run_and_check(lib, d, 16, poison=False)


# ---------------------------------------------------------------- multi-level cascade
def poison_multilevel(d):
    """NaN into every cache slot no request may read: the tails of partial last
    pages of every shared list and suffix, and unused pool pages."""
    kc, vc = d["k_cache"], d["v_cache"]
    used = set()
    segs = [(pages.tolist(), length) for groups in d["levels"] for (_, _, pages, length) in groups]
    segs += [(d["block_table"][b].tolist(), c) for b, c in enumerate(d["ctx"].tolist())]
    for pages, length in segs:
        n = -(-length // 16)
        used.update(pages[:n])
        if length % 16:
            kc[pages[n - 1], :, length % 16:] = float("nan")
            vc[pages[n - 1], :, length % 16:] = float("nan")
    for pid in range(kc.shape[0]):
        if pid not in used:
            kc[pid] = float("nan")
            vc[pid] = float("nan")


def run_multilevel(lib, d, ns, poison=True):
    if poison:
        poison_multilevel(d)
    g = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
    levels = [[(r0, r1, pages.to(DEV) if pages.numel() else None, length)
               for (r0, r1, pages, length) in groups] for groups in d["levels"]]
    res = lib.cascade_decode_multilevel(g["q"], g["k_cache"], g["v_cache"], levels,
                                        g["block_table"], g["ctx"], ns, d["sm_scale"])
    torch.cuda.synchronize()
    assert lib.get_device_error() == (0, 0)
    out, lse, o_pre, s_pre, o_part, lse_part = res
    o_r, s_r, op_r, sp_r = oracle.cascade_multilevel(d["q"], d["k_cache"], d["v_cache"],
                                                     d["levels"], d["block_table"], d["ctx"],
                                                     d["sm_scale"])
    atol, rtol_part, rtol_out = DEC_O_TOL[d["q"].dtype]
    assert out.dtype == d["q"].dtype
    assert_s_close(s_pre, sp_r, DEC_LSE_ATOL, "s_pre")
    assert_v_close(o_pre, op_r, atol, rtol_part, "o_pre", empty_rows=(sp_r == -math.inf))
    opr, lpr = oracle.attend_splits(d["q"], d["k_cache"], d["v_cache"], d["block_table"],
                                    d["ctx"], d["sm_scale"], ns)
    assert_s_close(lse_part, lpr, DEC_LSE_ATOL, "lse_part")
    assert_v_close(o_part, opr, atol, rtol_part, "o_part", empty_rows=(lpr == -math.inf))
    assert_s_close(lse, s_r, DEC_LSE_ATOL, "lse_out")
    assert_v_close(out, o_r, atol, rtol_out, "out", empty_rows=(s_r == -math.inf))
    return res


THREE_LEVELS = [[(0, 12, 1000)], [(0, 5, 300), (5, 9, 0), (9, 12, 77)],
                [(0, 3, 16), (3, 12, 200)]]


def test_cascade_multilevel_three_levels(lib):
    """A level shared by all 12 requests, a level of three groups (one sharing
    nothing), a third level of two groups, ragged suffixes (one empty)."""
    ctx = [5, 0, 37, 100, 16, 1, 250, 17, 64, 3, 90, 31]
    d = W.cascade_multilevel_inputs(12, 16, 4, 128, 16, THREE_LEVELS, ctx, seed=40)
    run_multilevel(lib, d, 4)


@pytest.mark.parametrize("G", [1, 8])
def test_cascade_multilevel_group_sizes_bf16(lib, G):
    ctx = [int(x) for x in np.random.default_rng(41 + G).integers(0, 200, 12)]
    d = W.cascade_multilevel_inputs(12, 2 * G, 2, 128, 16, THREE_LEVELS, ctx, seed=41 + G,
                                    dtype=torch.bfloat16)
    run_multilevel(lib, d, 8)


def test_cascade_multilevel_no_shared_level(lib):
    """No shared level: the prefix state is empty and out is the suffix alone."""
    d = W.cascade_multilevel_inputs(3, 8, 2, 128, 16, [], [40, 0, 7], seed=43)
    out, lse, o_pre, s_pre, _, _ = run_multilevel(lib, d, 4)
    assert torch.all(s_pre.cpu() == -math.inf) and torch.all(o_pre.cpu() == 0)


def test_cascade_multilevel_one_level_is_the_two_level_cascade(lib):
    """One level of one group runs exactly the two-level cascade: equal bits."""
    d = W.cascade_multilevel_inputs(6, 16, 4, 128, 16, [[(0, 6, 777)]], [9, 0, 33, 200, 1, 64],
                                    seed=44)
    g = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
    r0, r1, pages, length = d["levels"][0][0]
    a = lib.cascade_decode_multilevel(g["q"], g["k_cache"], g["v_cache"],
                                      [[(r0, r1, pages.to(DEV), length)]], g["block_table"],
                                      g["ctx"], 4, d["sm_scale"])
    b = lib.cascade_decode(g["q"], g["k_cache"], g["v_cache"], pages.to(DEV), length,
                           g["block_table"], g["ctx"], 4, d["sm_scale"])
    torch.cuda.synchronize()
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_cascade_multilevel_full_size(lib):
    """B=64: an 8192-token level shared by all, then eight groups of eight
    requests sharing 512 tokens each, then suffixes of 1..2048 tokens."""
    suffix = W.cascade_mixed()["ctx"].tolist()
    levels = [[(0, 64, 8192)], [(8 * i, 8 * i + 8, 512) for i in range(8)]]
    d = W.cascade_multilevel_inputs(64, 32, 8, 128, 16, levels, suffix, seed=45)
    run_multilevel(lib, d, 16, poison=False)


def test_cascade_back_to_back_on_a_side_stream_sharing_a_workspace(lib):
    """The cascade's kernels are chained in the caller's stream (the suffix
    pass's last CTA waits for the prefix pass, counted on a word of the
    workspace that the prefix pass zeroes): two calls of different sizes
    queued back to back on a non-default stream, sharing one workspace, each
    match the oracle."""
    cases = [W.cascade_inputs(6, 32, 8, 128, 16, 1000, [40, 1, 300, 0, 17, 129], seed=61),
             W.cascade_inputs(20, 16, 4, 128, 16, 333, [5 * i + 3 for i in range(20)], seed=62)]
    need = max(lib.cascade_workspace_size(d["q"].shape[0], d["q"].shape[1], d["k_cache"].shape[1],
                                          128, d["prefix_len"]) for d in cases)
    st = torch.cuda.Stream()
    outs = []
    with torch.cuda.stream(st):
        ws = torch.empty(max(need, 256), dtype=torch.uint8, device=DEV)
        for d in cases:
            g = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
            outs.append(lib.cascade_decode(g["q"], g["k_cache"], g["v_cache"], g["prefix_pages"],
                                           d["prefix_len"], g["block_table"], g["ctx"], 4,
                                           d["sm_scale"], workspace=ws)[:2])
    st.synchronize()
    assert lib.get_device_error() == (0, 0)
    for d, (out, lse) in zip(cases, outs):
        o_r, s_r, _, _ = oracle.cascade(d["q"], d["k_cache"], d["v_cache"], d["prefix_pages"],
                                        d["prefix_len"], d["block_table"], d["ctx"], d["sm_scale"])
        atol, _, rtol_out = DEC_O_TOL[d["q"].dtype]
        assert_s_close(lse, s_r, DEC_LSE_ATOL, "lse_out")
        assert_v_close(out, o_r, atol, rtol_out, "out", empty_rows=(s_r == -math.inf))


def test_cascade_bad_prefix_page_id_is_flagged_not_faulted(lib):
    """A prefix page id outside the pool is replaced by page 0 and reported
    in the device error word (detail 2 << 20 | the entry); the call
    completes and the context stays usable."""
    lib.get_device_error()  # clear
    d = W.cascade_inputs(4, 16, 4, 128, 16, 300, [20, 1, 0, 77], seed=63)
    d["prefix_pages"][2] = 10_000_000
    g = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
    lib.cascade_decode(g["q"], g["k_cache"], g["v_cache"], g["prefix_pages"], d["prefix_len"],
                       g["block_table"], g["ctx"], 4, d["sm_scale"])
    torch.cuda.synchronize()
    code, detail = lib.get_device_error()
    assert code == 1 and detail == (2 << 20 | 2)  # SKV_ERR_INVALID_ARG, prefix entry 2
    assert lib.get_device_error() == (0, 0)
    # The next call on clean inputs is correct.
    run_and_check(lib, W.cascade_inputs(4, 16, 4, 128, 16, 300, [20, 1, 0, 77], seed=63), 4)


# ---------------------------------------------------------------- per-sequence split counts
def run_and_check_varlen(lib, d, max_splits, pps, poison=True):
    """skv_cascade_decode_varlen: prefix state, the written suffix split
    states (per-sequence counts) and the merged output against the oracle."""
    if poison:
        poison_unused(d)
    g = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
    pp = g["prefix_pages"] if g["prefix_pages"].numel() else torch.zeros(1, dtype=torch.int32,
                                                                       device=DEV)
    plan = lib.splitkv_plan_varlen(d["ctx"], 16, max_splits, pps)
    ns = plan.num_splits.numpy()
    out, lse, o_pre, s_pre, o_part, lse_part = lib.cascade_decode_varlen(
        g["q"], g["k_cache"], g["v_cache"], pp, d["prefix_len"], g["block_table"], g["ctx"],
        plan, d["sm_scale"])
    torch.cuda.synchronize()
    assert lib.get_device_error() == (0, 0)
    o_r, s_r, op_r, sp_r = oracle.cascade(d["q"], d["k_cache"], d["v_cache"], d["prefix_pages"],
                                          d["prefix_len"], d["block_table"], d["ctx"],
                                          d["sm_scale"])
    atol, rtol_part, rtol_out = DEC_O_TOL[d["q"].dtype]
    assert_s_close(s_pre, sp_r, DEC_LSE_ATOL, "s_pre")
    assert_v_close(o_pre, op_r, atol, rtol_part, "o_pre", empty_rows=(sp_r == -math.inf))
    opr, lpr = oracle.attend_splits_varlen(d["q"], d["k_cache"], d["v_cache"], d["block_table"],
                                           d["ctx"], d["sm_scale"], ns, max_splits)
    B, Hq = d["q"].shape[:2]
    w = np.broadcast_to((np.arange(max_splits)[None, :] < ns[:, None])[:, None, :],
                        (B, Hq, max_splits))
    lp = lse_part.cpu().double().numpy()
    assert_s_close(lp[w], lpr[w], DEC_LSE_ATOL, "lse_part")
    assert_v_close(o_part.cpu().double().numpy()[w], opr[w], atol, rtol_part, "o_part",
                   empty_rows=(lpr[w] == -math.inf))
    assert_s_close(lse, s_r, DEC_LSE_ATOL, "lse_out")
    assert_v_close(out, o_r, atol, rtol_out, "out", empty_rows=(s_r == -math.inf))


@pytest.mark.parametrize("G", [1, 4, 8])
def test_cascade_varlen_small(lib, G):
    """Per-sequence suffix splits ([L3] §⑥ F1) under a 777-token shared prefix,
    ragged suffixes including empty ones."""
    B = (160 + G - 1) // G
    ctx = [int(x) for x in np.random.default_rng(50 + G).integers(0, 700, B)]
    ctx[0], ctx[1] = 0, 1
    d = W.cascade_inputs(B, 2 * G, 2, 128, 16, 777, ctx, seed=50 + G)
    run_and_check_varlen(lib, d, 16, 8)


def test_cascade_varlen_full_workload(lib):
    """The B=64 cascade workload (8192 shared tokens, suffixes of 1..2048
    tokens) with at most 16 suffix splits of at most 8 pages each."""
    d = W.cascade_mixed()
    run_and_check_varlen(lib, d, 16, 8, poison=False)


def test_cascade_varlen_bf16(lib):
    B = 40
    ctx = [int(x) for x in np.random.default_rng(60).integers(0, 900, B)]
    d = W.cascade_inputs(B, 8, 2, 128, 16, 300, ctx, seed=60, dtype=torch.bfloat16)
    run_and_check_varlen(lib, d, 8, 4)


def test_cascade_varlen_empty_prefix_and_empty_suffixes(lib):
    """Per-sequence suffix splits with no shared prefix (no prefix pass is
    launched: the suffix pass is not chained), and with a prefix but every
    suffix empty (one empty split each)."""
    d = W.cascade_inputs(6, 16, 4, 128, 16, 0, [40, 0, 3, 300, 17, 129], seed=61)
    run_and_check_varlen(lib, d, 8, 2)
    d = W.cascade_inputs(5, 8, 2, 128, 16, 500, [0] * 5, seed=62)
    run_and_check_varlen(lib, d, 4, 8)
