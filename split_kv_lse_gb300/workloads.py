"""Seeded synthetic inputs with the shapes and distributions of the workloads.

Every generator draws from a ``torch.Generator`` on the CPU with a fixed seed
and returns CPU tensors; callers move them to the GPU (library path) or widen
them to float64 (oracle).  This module contains no attention or merge
arithmetic: only shapes, distributions, empty-state patterns and page tables.

Named workloads (sizes of the split-KV decode and state-merge workloads):
  merge_state_tiny      S=16, H=4, D=64 fp32; rows 3, 7 one state empty, row 11 both
  merge_state_large     S=8192, H=32, D=128 fp16; s = 40 + N(0, 6); 1% empty
                        states, 0.1% double-empty rows, 0.1% of s +inf or NaN
  merge_states_main     S=256, N=64, H=32, D=128 fp32; s = 30 + N(0, 8), 5% empty
  merge_states_sweep    S=16, H=8, D=128 fp32, N in {1, 2, 3, 128, 1024}
  decode_long           B=1, ctx=32768, Hq=32, Hkv=8, D=128, page 16, fp16,
                        page table a random permutation of 2048 pool pages, NS=64
  cascade_mixed         B=64, Hq=32, Hkv=8, D=128, page 16, fp16; one shared
                        8192-token prefix + suffixes of 1..2048 tokens, NS=16
"""
from __future__ import annotations

import math

import torch

NEG_INF = float("-inf")


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return g


def _empty(s: torch.Tensor, v: torch.Tensor, mask: torch.Tensor) -> None:
    """Mark states empty: s = -inf and v = 0."""
    s[mask] = NEG_INF
    v[mask] = 0


# ---------------------------------------------------------------- merge_state
def merge_state_inputs(S, H, D, dtype=torch.float32, seed=0, s_mean=0.0, s_std=None,
                       s_lo=-20.0, s_hi=20.0, empty_p=0.0, double_empty_p=0.0, poison_p=0.0):
    """Two states [S, H, D] / [S, H].

    s ~ U(s_lo, s_hi) when s_std is None, else s_mean + N(0, s_std).
    Each state is independently empty with probability empty_p; each row is
    double-empty with probability double_empty_p; each incoming s is
    independently +inf with probability poison_p/2 and NaN with poison_p/2
    (its v stays random: such a state must be read as empty).
    """
    g = _gen(seed)
    va = torch.randn(S, H, D, generator=g, dtype=torch.float32)
    vb = torch.randn(S, H, D, generator=g, dtype=torch.float32)
    if s_std is None:
        sa = torch.rand(S, H, generator=g) * (s_hi - s_lo) + s_lo
        sb = torch.rand(S, H, generator=g) * (s_hi - s_lo) + s_lo
    else:
        sa = s_mean + s_std * torch.randn(S, H, generator=g)
        sb = s_mean + s_std * torch.randn(S, H, generator=g)
    if empty_p > 0:
        _empty(sa, va, torch.rand(S, H, generator=g) < empty_p)
        _empty(sb, vb, torch.rand(S, H, generator=g) < empty_p)
    if double_empty_p > 0:
        both = torch.rand(S, H, generator=g) < double_empty_p
        _empty(sa, va, both)
        _empty(sb, vb, both)
    if poison_p > 0:
        for s in (sa, sb):
            u = torch.rand(S, H, generator=g)
            s[u < poison_p / 2] = float("inf")
            s[(u >= poison_p / 2) & (u < poison_p)] = float("nan")
    return {"v_a": va.to(dtype), "s_a": sa.float(), "v_b": vb.to(dtype), "s_b": sb.float()}


def merge_state_tiny(seed=0):
    """S=16, H=4, D=64 fp32, s ~ U(-20, 20); rows 3 and 7 have one empty
    state (a and b respectively), row 11 has both empty (row = pos*H + h)."""
    d = merge_state_inputs(16, 4, 64, torch.float32, seed)
    fa, fb = d["s_a"].view(-1), d["s_b"].view(-1)
    va, vb = d["v_a"].view(-1, 64), d["v_b"].view(-1, 64)
    fa[3] = NEG_INF; va[3] = 0
    fb[7] = NEG_INF; vb[7] = 0
    fa[11] = NEG_INF; va[11] = 0
    fb[11] = NEG_INF; vb[11] = 0
    return d


def merge_state_large(seed=0):
    return merge_state_inputs(8192, 32, 128, torch.float16, seed, s_mean=40.0, s_std=6.0,
                              empty_p=0.01, double_empty_p=0.001, poison_p=0.001)


# ---------------------------------------------------------------- merge_states
def merge_states_inputs(S, N, H, D, dtype=torch.float32, seed=0, s_mean=30.0, s_std=8.0,
                        empty_p=0.05):
    """v [S, N, H, D] ~ N(0,1), s [S, N, H] = s_mean + N(0, s_std); each state
    empty (s = -inf, v = 0) with probability empty_p."""
    g = _gen(seed)
    v = torch.randn(S, N, H, D, generator=g, dtype=torch.float32)
    s = s_mean + s_std * torch.randn(S, N, H, generator=g)
    if empty_p > 0:
        _empty(s, v, torch.rand(S, N, H, generator=g) < empty_p)
    return {"v": v.to(dtype), "s": s.float()}


def merge_states_main(seed=0):
    return merge_states_inputs(256, 64, 32, 128, torch.float32, seed)


MERGE_STATES_SWEEP_N = (1, 2, 3, 128, 1024)


def merge_states_sweep(N, seed=0):
    return merge_states_inputs(16, N, 8, 128, torch.float32, seed)


# ---------------------------------------------------------------- paged decode
def decode_inputs(B, Hq, Hkv, D, page, ctx, seed=0, dtype=torch.float16, pool_extra=0,
                  max_pages=None):
    """Paged KV cache [P, Hkv, page, D] and a page table of distinct random pool
    pages per sequence (a random permutation of the pool); q [B, Hq, D].
    q, K, V ~ N(0, 1).  ctx: list of B context lengths.  Unused table entries
    are 0 (never read: they lie beyond ctx)."""
    g = _gen(seed)
    need = [math.ceil(c / page) for c in ctx]
    P = sum(need) + pool_extra
    P = max(P, 1)
    perm = torch.randperm(P, generator=g).to(torch.int32)
    mp = max(1, max(need) if need else 1) if max_pages is None else max_pages
    table = torch.zeros(B, mp, dtype=torch.int32)
    k = 0
    for b, n in enumerate(need):
        table[b, :n] = perm[k:k + n]
        k += n
    q = torch.randn(B, Hq, D, generator=g, dtype=torch.float32).to(dtype)
    kc = torch.randn(P, Hkv, page, D, generator=g, dtype=torch.float32).to(dtype)
    vc = torch.randn(P, Hkv, page, D, generator=g, dtype=torch.float32).to(dtype)
    return {"q": q, "k_cache": kc, "v_cache": vc, "block_table": table,
            "ctx": torch.tensor(ctx, dtype=torch.int32), "sm_scale": 1.0 / math.sqrt(D),
            "page": page}


def decode_long(seed=0, dtype=torch.float16):
    """B=1, ctx=32768 (2048 pages = the whole pool, randomly permuted), NS=64."""
    d = decode_inputs(1, 32, 8, 128, 16, [32768], seed, dtype=dtype)
    d["num_splits"] = 64
    return d


# ---------------------------------------------------------------- cascade
def cascade_inputs(B, Hq, Hkv, D, page, prefix_len, suffix_ctx, seed=0, dtype=torch.float16):
    """One shared prefix of prefix_len tokens (its own random pool pages) plus a
    suffix of suffix_ctx[b] tokens per request (random pages of a separate
    part of the pool)."""
    g = _gen(seed)
    npre = math.ceil(prefix_len / page)
    need = [math.ceil(c / page) for c in suffix_ctx]
    nsuf = sum(need)
    P = max(1, npre + nsuf)
    prefix_pages = torch.randperm(npre, generator=g).to(torch.int32) if npre else torch.zeros(0, dtype=torch.int32)
    suffix_pool = (torch.randperm(nsuf, generator=g) + npre).to(torch.int32)
    mp = max(1, max(need) if need else 1)
    table = torch.zeros(B, mp, dtype=torch.int32)
    k = 0
    for b, n in enumerate(need):
        table[b, :n] = suffix_pool[k:k + n]
        k += n
    q = torch.randn(B, Hq, D, generator=g, dtype=torch.float32).to(dtype)
    kc = torch.randn(P, Hkv, page, D, generator=g, dtype=torch.float32).to(dtype)
    vc = torch.randn(P, Hkv, page, D, generator=g, dtype=torch.float32).to(dtype)
    return {"q": q, "k_cache": kc, "v_cache": vc, "prefix_pages": prefix_pages,
            "prefix_len": prefix_len, "block_table": table,
            "ctx": torch.tensor(suffix_ctx, dtype=torch.int32), "sm_scale": 1.0 / math.sqrt(D),
            "page": page}


def cascade_multilevel_inputs(B, Hq, Hkv, D, page, levels, suffix_ctx, seed=0,
                              dtype=torch.float16):
    """Shared tokens at several levels plus a per-request suffix.  levels[l] is a
    list of groups (r0, r1, length): requests [r0, r1) share `length` tokens at
    level l.  Every group's tokens and every suffix get their own pool pages, in
    one random permutation of the pool.  Returns the cascade inputs with
    "levels" = [[(r0, r1, pages int32 tensor, length), ...], ...]."""
    g = _gen(seed)
    sizes = [math.ceil(length / page) for groups in levels for (_, _, length) in groups]
    need = [math.ceil(c / page) for c in suffix_ctx]
    P = max(1, sum(sizes) + sum(need))
    perm = torch.randperm(P, generator=g).to(torch.int32)
    at = 0
    out_levels = []
    for groups in levels:
        lv = []
        for (r0, r1, length) in groups:
            n = math.ceil(length / page)
            lv.append((r0, r1, perm[at:at + n].clone(), length))
            at += n
        out_levels.append(lv)
    mp = max(1, max(need) if need else 1)
    table = torch.zeros(B, mp, dtype=torch.int32)
    for b, n in enumerate(need):
        table[b, :n] = perm[at:at + n]
        at += n
    q = torch.randn(B, Hq, D, generator=g, dtype=torch.float32).to(dtype)
    kc = torch.randn(P, Hkv, page, D, generator=g, dtype=torch.float32).to(dtype)
    vc = torch.randn(P, Hkv, page, D, generator=g, dtype=torch.float32).to(dtype)
    return {"q": q, "k_cache": kc, "v_cache": vc, "levels": out_levels, "block_table": table,
            "ctx": torch.tensor(suffix_ctx, dtype=torch.int32), "sm_scale": 1.0 / math.sqrt(D),
            "page": page}


def cascade_mixed(seed=0, dtype=torch.float16):
    """B=64 requests sharing an 8192-token prefix; suffix lengths uniform in
    [1, 2048] (so some have fewer tokens than page*NS and get empty splits);
    NS=16 for the suffix."""
    g = _gen(seed + 1000)
    suffix = torch.randint(1, 2049, (64,), generator=g).tolist()
    d = cascade_inputs(64, 32, 8, 128, 16, 8192, suffix, seed, dtype=dtype)
    d["num_splits"] = 16
    return d
