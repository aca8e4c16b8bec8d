"""Context-parallel decode on CPU process groups (gloo): every rank holds one
contiguous page range of each sequence ([L3] §② ranges with NUM_SPLITS = world
size), computes the attention state over it, the states are exchanged with one
all-gather and merged with the sanitising N-state merge ([FA] §2.2).  The fp64
oracle stands in for each rank's GPU computation; the sharding, the exchange
and the merge order are the library's (split_kv_lse_gb300.cp).  The result must
equal unsplit attention over the whole context, also when a rank reports NaN
or +inf for a shard it holds nothing of, and for sequences too short to reach
every rank."""
import math
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

from conftest import ROOT

CTX = [0, 1, 17, 37, 300, 1000, 2049]


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, poison, out_q):
    import sys
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle
        from split_kv_lse_gb300 import cp
        from split_kv_lse_gb300 import workloads as W
        d = W.decode_inputs(len(CTX), 8, 2, 16, 16, CTX, seed=70 + world, pool_extra=2)
        bt_l, ctx_l = cp.shard_sequences(d["block_table"], d["ctx"], 16, world, rank)

        def attend(q, kc, vc, bt, cx, ns, scale):
            o, s = oracle.attend_full(q, kc, vc, bt, cx, scale)
            if poison and rank == world - 1:
                # A backend that reports an empty shard as NaN or +inf (and
                # leaves garbage in its o): the merge must read it as empty.
                empty = np.asarray(cx) == 0
                s[empty] = math.nan if world % 2 == 0 else math.inf
                o[empty] = math.nan
            return torch.from_numpy(o), torch.from_numpy(s)

        def merge(o_all, s_all):
            Wn, B, Hq, D = o_all.shape
            vo, so = oracle.merge_states(o_all.reshape(1, Wn, B * Hq, D).numpy(),
                                         s_all.reshape(1, Wn, B * Hq).numpy())
            return torch.from_numpy(vo).view(B, Hq, D), torch.from_numpy(so).view(B, Hq)

        o, s = cp.cp_decode(d["q"], d["k_cache"], d["v_cache"], bt_l, ctx_l, d["sm_scale"],
                            attend=attend, merge=merge)
        o_r, s_r = oracle.attend_full(d["q"], d["k_cache"], d["v_cache"], d["block_table"],
                                      d["ctx"], d["sm_scale"])
        o, s = o.numpy(), s.numpy()
        fin = np.isfinite(s_r)
        ok = (np.array_equal(fin, np.isfinite(s)) and np.allclose(o, o_r, rtol=1e-12, atol=1e-13)
              and np.allclose(s[fin], s_r[fin], rtol=0, atol=1e-12)
              and np.all(o[~fin] == 0) and np.all(s[~fin] == -math.inf))
        # Which ranks held something of each sequence (the shard ranges).
        held = [int(c) for c in ctx_l.tolist()]
        out_q.put((rank, bool(ok), held))
    except Exception as e:  # reported to the parent, which fails the test
        out_q.put((rank, repr(e), None))
    finally:
        dist.destroy_process_group()


def _run(world, poison):
    import oracle
    oracle.build()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, poison, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=300) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
    return sorted(res)


@pytest.mark.parametrize("world", [2, 3])
@pytest.mark.parametrize("poison", [False, True])
def test_cp_decode_equals_unsplit_attention(world, poison):
    res = _run(world, poison)
    for rank, ok, held in res:
        assert ok is True, (rank, ok)
    # The shards partition every sequence's tokens: their lengths add up to ctx.
    tot = np.sum([held for _, _, held in res], axis=0)
    assert tot.tolist() == CTX


def test_shard_ranges_are_the_split_ranges():
    """Rank r's pages are the [L3] §② range of split r with NUM_SPLITS = world
    (the printed ctx = 100, 4 ranges: [0,2) [2,4) [4,6) [6,7); ctx = 37 leaves
    rank 3 empty)."""
    from split_kv_lse_gb300 import cp
    assert [cp.shard_range(100, 16, 4, r) for r in range(4)] == [(0, 2), (2, 4), (4, 6), (6, 7)]
    assert cp.shard_range(37, 16, 4, 3) == (3, 3)
    bt = torch.arange(20, dtype=torch.int32).view(2, 10)
    t, c = cp.shard_sequences(bt, [100, 37], 16, 4, 1)
    assert c.tolist() == [32, 16] and t[0, :2].tolist() == [2, 3] and t[1, :1].tolist() == [11]
    t, c = cp.shard_sequences(bt, [100, 37], 16, 4, 3)
    assert c.tolist() == [4, 0] and t[0, :1].tolist() == [6]
