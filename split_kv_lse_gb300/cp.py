"""Context-parallel split-KV decode: the KV cache of every sequence is cut into
contiguous page ranges, one per rank; each rank attends to its own range, the
per-rank attention states are exchanged with one all-gather, and every rank
merges them exactly.

Pages: "FlashAttention 的空行 LSE:FA-2 的 +inf 约定与后来的变化" §2.2 (the
cross-GPU LSE merge of decode context parallelism sanitises every incoming
LSE, because a shard that contributed nothing may report -inf, NaN or +inf);
"L3 讲解：split-KV decode 与 LSE 合并" §② (the page ranges, here at the rank
level) and §③ (a state is (o, lse); merging needs both);
"F2 讲解：merge_state，以 2 为底的 LSE 合并" §④ (the [S, N, H, D] merge).

Design: the rank shards are the [L3] §② split ranges with NUM_SPLITS = world
size, so rank r owns pages [r * pps, min((r + 1) * pps, num_pages)) of a
sequence of num_pages pages, pps = ceil(num_pages / world).  A rank whose range
is empty for a sequence contributes the empty state (o = 0, s = -inf).  Each
rank's state is fp32 [B, Hq, D] plus its base-2 s [B, Hq]; the all-gather
stacks them as [world, B*Hq, D], which is exactly the [S=1, N=world, H=B*Hq, D]
layout merge_states takes, so no transpose is needed.  Only the all-gather
crosses ranks; everything else is this library's kernels on each rank's GPU.

The two compute steps are parameters (`attend`, `merge`), defaulting to this
library's GPU calls, so that the sharding, the exchange and the merge order can
be exercised on CPU process groups with any stand-in computation.
"""
from __future__ import annotations

import torch


def shard_range(ctx: int, page: int, world: int, rank: int):
    """Pages [p_start, p_end) of a ctx-token sequence that `rank` owns
    ([L3] §② with NUM_SPLITS = world; p_end <= p_start: the rank holds none)."""
    num_pages = -(-int(ctx) // page)
    pps = -(-num_pages // world)
    p0 = rank * pps
    return p0, min(p0 + pps, num_pages)


def shard_sequences(block_table: torch.Tensor, ctx, page: int, world: int, rank: int):
    """This rank's page table and contexts: row b holds the pool pages of the
    rank's range of sequence b (the rest of the row 0), ctx_local[b] the
    tokens of that range.  Returns (block_table_local int32 [B, max_local],
    ctx_local int32 [B]) on the CPU."""
    ctx = [int(c) for c in (ctx.tolist() if hasattr(ctx, "tolist") else ctx)]
    B = len(ctx)
    ranges = [shard_range(c, page, world, rank) for c in ctx]
    width = max(1, max((max(0, e - a) for a, e in ranges), default=1))
    bt = torch.zeros(B, width, dtype=torch.int32)
    cl = torch.zeros(B, dtype=torch.int32)
    src = block_table.detach().cpu()
    for b, (a, e) in enumerate(ranges):
        if e > a:
            bt[b, :e - a] = src[b, a:e]
            cl[b] = min(ctx[b], e * page) - a * page
    return bt, cl


def local_state_gpu(q, k_cache, v_cache, block_table, ctx, num_splits: int, sm_scale: float):
    """This rank's state over its shard, on the GPU: split-KV pass 1, then the
    num_splits states of each (b, hq) merged in fp32 (merge_states over
    o_part viewed as [B*Hq, num_splits, 1, D]).  Returns (o fp32 [B, Hq, D],
    s fp32 [B, Hq])."""
    from . import merge_states, splitkv_decode
    B, Hq, D = q.shape
    _, _, o_part, lse_part = splitkv_decode(q, k_cache, v_cache, block_table, ctx, num_splits,
                                            sm_scale, combine=False)
    o, s = merge_states(o_part.view(B * Hq, num_splits, 1, D),
                        lse_part.view(B * Hq, num_splits, 1))
    return o.view(B, Hq, D), s.view(B, Hq)


def merge_rank_states_gpu(o_all: torch.Tensor, s_all: torch.Tensor):
    """Merge of the gathered states o_all [W, B, Hq, D], s_all [W, B, Hq]
    (fp32, CUDA) with this library's merge_states, whose sanitiser reads a
    NaN or +inf s as an empty state ([FA] §2.2).  Returns (o [B, Hq, D],
    s [B, Hq])."""
    from . import merge_states
    W, B, Hq, D = o_all.shape
    o, s = merge_states(o_all.reshape(1, W, B * Hq, D).contiguous(),
                        s_all.reshape(1, W, B * Hq).contiguous())
    return o.view(B, Hq, D), s.view(B, Hq)


def all_gather_states(o: torch.Tensor, s: torch.Tensor, group=None):
    """One exchange of every rank's state: returns o_all [W, B, Hq, D] and
    s_all [W, B, Hq], rank r's state at index r on every rank."""
    import torch.distributed as dist
    W = dist.get_world_size(group)
    o_all = [torch.empty_like(o) for _ in range(W)]
    s_all = [torch.empty_like(s) for _ in range(W)]
    dist.all_gather(o_all, o.contiguous(), group=group)
    dist.all_gather(s_all, s.contiguous(), group=group)
    return torch.stack(o_all), torch.stack(s_all)


def cp_decode(q, k_cache, v_cache, block_table_local, ctx_local, sm_scale: float,
              num_splits: int = 1, group=None, attend=None, merge=None):
    """Context-parallel decode step on this rank: the state over the rank's
    shard (attend), one all-gather of the states, and their merge (merge).

    q [B, Hq, D] is the full query (every rank holds it); k_cache, v_cache,
    block_table_local, ctx_local describe this rank's shard (shard_sequences).
    attend(q, k_cache, v_cache, block_table_local, ctx_local, num_splits,
    sm_scale) -> (o fp32 [B, Hq, D], s fp32 [B, Hq]); default local_state_gpu.
    merge(o_all, s_all) -> (o, s); default merge_rank_states_gpu.
    The states are exchanged in the type attend returns (fp32 on the GPU).
    Returns (o [B, Hq, D], s [B, Hq] base 2), the same on every rank.
    """
    attend = local_state_gpu if attend is None else attend
    merge = merge_rank_states_gpu if merge is None else merge
    o, s = attend(q, k_cache, v_cache, block_table_local, ctx_local, num_splits, sm_scale)
    o_all, s_all = all_gather_states(o, s, group)
    return merge(o_all, s_all)
