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
from gpu_helpers import (DECODE_KERNELS, select_decode_kernel, DEC_LSE_ATOL, DEC_O_TOL, assert_s_close, assert_v_close, np64,
                         require_gpu, skv)
from split_kv_lse_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(params=DECODE_KERNELS, autouse=True)
def decode_kernel(request):
    """Every test runs once per pass-1 kernel."""
    select_decode_kernel(request.param)
    yield request.param
    select_decode_kernel("cuda_cores")


@pytest.fixture(scope="module")
def lib():
    require_gpu()
    return skv()


def run_decode(lib, d, ns, nan_tail=False):
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
