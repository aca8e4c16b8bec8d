"""Parity of the split-KV paged decode (pass 1 partials, page ranges, combined
output) with the fp64 oracle, at the full long-context size and on small
cases that cover ragged pages, empty splits, ctx = 0, every supported group
size and the device-side bounds checks.

Page: "L3 讲解：split-KV decode 与 LSE 合并" §①-⑤."""
import math

import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import (DEC_LSE_ATOL, DEC_O_TOL, assert_s_close, assert_v_close, np64,
                         require_gpu, skv)
from split_kv_lse_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def lib():
    require_gpu()
    return skv()


def to_dev(d, nan_tail=False):
    g = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
    if nan_tail:
        # Poison every cache slot past each sequence's end (inside its last
        # page) and every pool page no sequence uses: none may be read.
        kc, vc = g["k_cache"], g["v_cache"]
        used = set()
        for b, c in enumerate(d["ctx"].tolist()):
            npg = -(-c // 16)
            used.update(d["block_table"][b, :npg].tolist())
            if c % 16:
                pid = int(d["block_table"][b, npg - 1])
                kc[pid, :, c % 16:] = float("nan")
                vc[pid, :, c % 16:] = float("nan")
        for pid in range(kc.shape[0]):
            if pid not in used:
                kc[pid] = float("nan")
                vc[pid] = float("nan")
    return g


def run_decode(lib, d, ns, nan_tail=False):
    g = to_dev(d, nan_tail)
    B = d["q"].shape[0]
    rd = torch.full((B, ns, 2), -7, dtype=torch.int32, device=DEV)
    out, lse, o_part, lse_part = lib.splitkv_decode(
        g["q"], g["k_cache"], g["v_cache"], g["block_table"], g["ctx"], ns, d["sm_scale"],
        ranges_dbg=rd)
    torch.cuda.synchronize()
    return out, lse, o_part, lse_part, rd


def check_decode(lib, d, ns, nan_tail=False):
    out, lse, o_part, lse_part, rd = run_decode(lib, d, ns, nan_tail)
    args = (d["q"], d["k_cache"], d["v_cache"], d["block_table"], d["ctx"], d["sm_scale"])
    op_r, lp_r = oracle.attend_splits(*args, ns)
    o_r, s_r = oracle.attend_full(*args)
    empty = lp_r == -math.inf
    atol, rtol_part, rtol_out = DEC_O_TOL[d["q"].dtype]
    assert out.dtype == d["q"].dtype
    assert_s_close(lse_part, lp_r, DEC_LSE_ATOL, "lse_part")
    assert_v_close(o_part, op_r, atol, rtol_part, "o_part", empty_rows=empty)
    assert_s_close(lse, s_r, DEC_LSE_ATOL, "lse_out")
    assert_v_close(out, o_r, atol, rtol_out, "out", empty_rows=(s_r == -math.inf))
    # Page ranges, bit-exact against the oracle's integer formula.
    ranges = rd.cpu().numpy()
    for b, c in enumerate(d["ctx"].tolist()):
        for sp in range(ns):
            assert tuple(ranges[b, sp]) == orc_range(c, ns, sp), (b, sp)
    return out, lse, o_part, lse_part


def orc_range(ctx, ns, sp):
    return oracle.split_range(int(ctx), 16, ns, sp)


def test_decode_long_context_full(lib):
    """B=1, ctx=32768, Hq=32, Hkv=8, D=128, 64 splits: every partial, range and output."""
    d = W.decode_long()
    check_decode(lib, d, d["num_splits"])


@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("ns", [1, 3, 4, 64])
def test_decode_small(lib, G, ns):
    ctx = [1, 15, 16, 17, 37, 100, 1000, 0]
    Hkv = 2
    d = W.decode_inputs(len(ctx), Hkv * G, Hkv, 128, 16, ctx, seed=G * 100 + ns, pool_extra=3)
    check_decode(lib, d, ns, nan_tail=True)


def test_decode_empty_splits_write_neg_inf_and_zero(lib):
    """L3 §④: ctx = 37 with 4 splits leaves split 3 empty; ctx < page*NS everywhere."""
    d = W.decode_inputs(3, 32, 8, 128, 16, [37, 5, 200], seed=5)
    out, lse, o_part, lse_part = check_decode(lib, d, 16, nan_tail=True)
    lp = lse_part.cpu()
    assert torch.all(lp[0, :, 3:] == -math.inf) and torch.all(o_part.cpu()[0, :, 3:] == 0)


def test_decode_all_empty_sequence(lib):
    d = W.decode_inputs(2, 8, 2, 128, 16, [0, 0], seed=6, pool_extra=2)
    out, lse, o_part, lse_part = check_decode(lib, d, 4)
    assert torch.all(lse.cpu() == -math.inf) and torch.all(out.cpu() == 0)


def test_decode_plan_choice_runs(lib):
    ctx = [4096] * 8
    ns = lib.splitkv_decode_plan(ctx, 8, 16, 0)
    assert ns in (4, 16, 64)
    d = W.decode_inputs(8, 32, 8, 128, 16, ctx, seed=7)
    check_decode(lib, d, ns)


def test_decode_bad_page_id_is_flagged_not_faulted(lib):
    """A page id outside the pool is clamped and reported in the error word."""
    lib.get_device_error()  # clear
    d = W.decode_inputs(1, 8, 2, 128, 16, [40], seed=8)
    d["block_table"][0, 1] = 10_000_000
    run_decode(lib, d, 2)
    code, detail = lib.get_device_error()
    assert code == 1  # SKV_ERR_INVALID_ARG
    assert lib.get_device_error() == (0, 0)


def test_decode_ctx_past_table_is_flagged(lib):
    lib.get_device_error()
    d = W.decode_inputs(1, 8, 2, 128, 16, [40], seed=9)
    d["ctx"][0] = 40 * 100  # more tokens than the table has pages for
    run_decode(lib, d, 2)
    assert lib.get_device_error()[0] == 1


def test_decode_partials_only(lib):
    """combine=False: pass 1 alone writes the same partials."""
    d = W.decode_inputs(2, 16, 4, 128, 16, [300, 77], seed=10)
    g = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
    out, lse, op, lp = lib.splitkv_decode(g["q"], g["k_cache"], g["v_cache"], g["block_table"],
                                          g["ctx"], 8, d["sm_scale"], combine=False)
    assert out is None and lse is None
    _, _, op2, lp2 = lib.splitkv_decode(g["q"], g["k_cache"], g["v_cache"], g["block_table"],
                                        g["ctx"], 8, d["sm_scale"])
    assert torch.equal(op, op2) and torch.equal(lp, lp2)


def test_decode_many_short_splits(lib):
    """Far more (request, kv head, split) CTAs than fit on the GPU at once
    (several waves), with short ragged contexts, empty splits and ctx = 0."""
    rng = np.random.default_rng(11)
    ctx = rng.integers(0, 130, size=300).tolist()
    ctx[5], ctx[17], ctx[18] = 0, 128, 129
    d = W.decode_inputs(len(ctx), 32, 8, 128, 16, ctx, seed=11, pool_extra=2)
    check_decode(lib, d, 16, nan_tail=True)


def test_decode_short_splits_many_requests(lib):
    """Over a thousand requests (the grid's request dimension) with contexts
    of 0 to 39 tokens."""
    rng = np.random.default_rng(12)
    ctx = rng.integers(0, 40, size=1100).tolist()
    d = W.decode_inputs(len(ctx), 2, 1, 128, 16, ctx, seed=12)
    check_decode(lib, d, 4)


@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("ns,ctx", [
    (2, [0, 1, 16, 130, 255, 256]),
    (6, [0, 1, 17, 100, 129, 500, 767, 768]),
    (7, [0, 3, 100, 700]),
])
def test_decode_short_split_boundaries(lib, G, ns, ctx):
    """One-warp CTAs (splits of at most 8 pages) at split counts that are not
    powers of two: split boundaries on page edges, a last split that is empty
    or ends in a partial page, whole sequences empty."""
    d = W.decode_inputs(len(ctx), 2 * G, 2, 128, 16, ctx, seed=40 + G * 7 + ns, pool_extra=2)
    assert -(-d["block_table"].shape[1] // ns) <= 8
    check_decode(lib, d, ns, nan_tail=True)


@pytest.mark.parametrize("G", [1, 4, 8])
@pytest.mark.parametrize("ns", [3, 64])
def test_decode_bf16_small(lib, G, ns):
    """bf16 q/K/V end to end: bf16 x bf16 -> fp32 products, bf16 output."""
    ctx = [1, 15, 16, 17, 37, 100, 1000, 0]
    Hkv = 2
    d = W.decode_inputs(len(ctx), Hkv * G, Hkv, 128, 16, ctx, seed=G * 100 + ns + 7,
                        dtype=torch.bfloat16, pool_extra=3)
    check_decode(lib, d, ns, nan_tail=True)


def test_decode_bf16_long_context(lib):
    """The long-context workload (B=1, ctx=32768, Hq=32, Hkv=8, NS=64) in bf16."""
    d = W.decode_inputs(1, 32, 8, 128, 16, [32768], seed=0, dtype=torch.bfloat16)
    check_decode(lib, d, 64)


@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("ns", [1, 2])
def test_decode_long_splits(lib, G, ns):
    """Splits of more than 64 pages (the CTA shape whose warps take fixed
    pages w, w+3, ...): the unsplit decode ([L3] §⑥, no split) and a two-way
    split.  ctx 4096 is 256 pages: unsplit, each of the 3 warps owns about 86
    pages, so its page ids are reloaded past 32 and 64; ctx 2500 and 1100
    (157 and 69 pages) end on partial pages whose tails hold NaN, as does
    every pool page no sequence uses."""
    ctx = [4096, 2500, 1100]
    Hkv = 2
    d = W.decode_inputs(len(ctx), Hkv * G, Hkv, 128, 16, ctx, seed=300 + 10 * G + ns,
                        pool_extra=3)
    check_decode(lib, d, ns, nan_tail=True)


def test_decode_plan_unsplit_batch(lib):
    """The plan chooses no split when B*Hkv already fills the GPU ([L3] §⑥):
    B=64, Hkv=8 (512 programs) with 1100..1900-token contexts on this GPU's
    SMs gives NS=1 (the oracle's plan agrees), and the unsplit decode of that
    batch (69..119 pages per split) matches the oracle."""
    rng = np.random.default_rng(13)
    ctx = [int(c) for c in rng.integers(1100, 1901, size=64)]
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    ns = lib.splitkv_decode_plan(ctx, 8, 16, 0)
    assert ns == oracle.plan(ctx, 8, 16, sms)
    assert ns == 1 or 64 * 8 < 3 * sms
    d = W.decode_inputs(len(ctx), 32, 8, 128, 16, ctx, seed=13)
    check_decode(lib, d, ns, nan_tail=True)


@pytest.mark.parametrize("mode,detail", [(0, 100), (1, 101)])
def test_bounded_wait_gives_up_and_reports(lib, mode, detail):
    """A barrier wait that nothing completes gives up after its limit (1 ms
    here), records SKV_ERR_TIMEOUT with the wait's detail code and returns:
    the kernel completes, the error is read on the host, and the GPU goes on
    working (a decode right after is exact)."""
    lib.get_device_error()  # clear
    lib.selftest_bounded_wait(mode, 1_000_000)
    assert lib.poll_device_error() == (4, detail)
    assert lib.poll_device_error() == (0, 0)
    d = W.decode_inputs(2, 8, 2, 128, 16, [100, 37], seed=14)
    check_decode(lib, d, 4)
    assert lib.get_device_error() == (0, 0)


# ---------------------------------------------------------------- per-sequence split counts
def check_decode_varlen(lib, d, max_splits, pps, nan_tail=False):
    """skv_splitkv_decode_varlen against the oracle's per-sequence split
    states (the written slots), the unsplit attention (merged output) and the
    per-sequence page ranges (bit-exact; unwritten slots keep their fill)."""
    g = to_dev(d, nan_tail)
    B, Hq = d["q"].shape[:2]
    plan = lib.splitkv_plan_varlen(d["ctx"], 16, max_splits, pps)
    ns = plan.num_splits.numpy()
    assert np.array_equal(ns, oracle.plan_varlen(d["ctx"], 16, max_splits, pps))
    rd = torch.full((B, max_splits, 2), -7, dtype=torch.int32, device=DEV)
    op = torch.full((B, Hq, max_splits, 128), 5.0, device=DEV)
    out, lse, o_part, lse_part = lib.splitkv_decode_varlen(
        g["q"], g["k_cache"], g["v_cache"], g["block_table"], g["ctx"], plan, d["sm_scale"],
        o_part=op, ranges_dbg=rd)
    torch.cuda.synchronize()
    args = (d["q"], d["k_cache"], d["v_cache"], d["block_table"], d["ctx"], d["sm_scale"])
    op_r, lp_r = oracle.attend_splits_varlen(*args, ns, max_splits)
    o_r, s_r = oracle.attend_full(*args)
    atol, rtol_part, rtol_out = DEC_O_TOL[d["q"].dtype]
    written = np.arange(max_splits)[None, :] < ns[:, None]            # [B, max_splits]
    wmask = np.broadcast_to(written[:, None, :], (B, Hq, max_splits))
    lp = np64(lse_part)
    assert_s_close(lp[wmask], lp_r[wmask], DEC_LSE_ATOL, "lse_part")
    assert_v_close(np64(o_part)[wmask], op_r[wmask], atol, rtol_part, "o_part",
                   empty_rows=(lp_r[wmask] == -math.inf))
    assert np.all(np64(o_part)[~wmask] == 5.0), "a slot past a sequence's split count was written"
    assert_s_close(lse, s_r, DEC_LSE_ATOL, "lse_out")
    assert_v_close(out, o_r, atol, rtol_out, "out", empty_rows=(s_r == -math.inf))
    ranges = rd.cpu().numpy()
    for b, c in enumerate(d["ctx"].tolist()):
        for sp in range(max_splits):
            want = oracle.split_range(int(c), 16, int(ns[b]), sp) if sp < ns[b] else (-7, -7)
            assert tuple(ranges[b, sp]) == want, (b, sp)
    return plan


VARLEN_CTX = [0, 1, 15, 16, 17, 100, 129, 1000, 2500, 4096]


@pytest.mark.parametrize("G", [1, 4, 8])
@pytest.mark.parametrize("max_splits,pps", [(16, 8), (4, 2), (64, 1), (2, 64)])
def test_decode_varlen_ragged(lib, G, max_splits, pps):
    """Per-sequence split counts ([L3] §⑥ F1) on a ragged batch: ctx 0..4096
    with NaN in every slot that must not be read.  The four plans give splits
    of at most 16, 64, 4 and 128 pages (each CTA shape of pass 1)."""
    Hkv = 2
    d = W.decode_inputs(len(VARLEN_CTX), Hkv * G, Hkv, 128, 16, VARLEN_CTX,
                        seed=400 + G + max_splits + pps, pool_extra=3)
    plan = check_decode_varlen(lib, d, max_splits, pps, nan_tail=True)
    assert plan.max_split_pages == {(16, 8): 16, (4, 2): 64, (64, 1): 4, (2, 64): 128}[
        (max_splits, pps)]


def test_decode_varlen_cascade_suffix_mix(lib):
    """The cascade workload's suffixes (B=64, Hq=32, Hkv=8, 1..2048 tokens) with
    at most 16 splits of at most 8 pages each: every written partial, range
    and output at full size."""
    d5 = W.cascade_mixed()
    ctx = d5["ctx"].tolist()
    d = W.decode_inputs(64, 32, 8, 128, 16, ctx, seed=41)
    check_decode_varlen(lib, d, 16, 8)


@pytest.mark.parametrize("G", [1, 8])
def test_decode_varlen_bf16(lib, G):
    d = W.decode_inputs(len(VARLEN_CTX), 2 * G, 2, 128, 16, VARLEN_CTX, seed=430 + G,
                        dtype=torch.bfloat16, pool_extra=2)
    check_decode_varlen(lib, d, 16, 8, nan_tail=True)


def test_decode_varlen_plan_for_shorter_contexts_is_flagged(lib):
    """A plan made for 200 tokens (one split of 13 pages: the two-warp CTA
    shape, which holds at most 64 page ids) run on a 2000-token context: the
    125-page split is flagged in the error word and cut, nothing faults, and
    the GPU goes on working."""
    lib.get_device_error()
    plan = lib.splitkv_plan_varlen([200], 16, 16, 16)
    assert plan.max_split_pages == 13
    d = W.decode_inputs(1, 8, 2, 128, 16, [2000], seed=44)
    g = to_dev(d)
    lib.splitkv_decode_varlen(g["q"], g["k_cache"], g["v_cache"], g["block_table"], g["ctx"],
                              plan, d["sm_scale"])
    code, detail = lib.get_device_error()
    assert code == 1 and detail == (3 << 20)
    d2 = W.decode_inputs(2, 8, 2, 128, 16, [100, 37], seed=45)
    check_decode_varlen(lib, d2, 4, 2)
    assert lib.get_device_error() == (0, 0)
