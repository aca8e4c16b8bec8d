"""Context-parallel decode on one GPU: the per-rank computations of
split_kv_lse_gb300.cp (the state over one contiguous page range of every
sequence, then the merge of the gathered states) run here for every rank of a
4-way split in turn, with the all-gather replaced by stacking, and are checked
against the fp64 oracle's unsplit attention.  The merge sanitises: a rank that
reports NaN or +inf (with NaN in o) for a shard it holds nothing of changes
nothing ([FA] §2.2).  The exchange itself is tested on CPU process groups."""
import math

import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import DEC_LSE_ATOL, assert_s_close, assert_v_close, require_gpu, skv
from split_kv_lse_gb300 import cp
from split_kv_lse_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def lib():
    require_gpu()
    return skv()


@pytest.mark.parametrize("poison", [None, "nan", "inf"])
def test_cp_rank_states_merge_to_unsplit_attention(lib, poison):
    world = 4
    ctx = [0, 1, 17, 37, 300, 1000, 4096, 2049]
    d = W.decode_inputs(len(ctx), 32, 8, 128, 16, ctx, seed=80, pool_extra=2)
    g = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
    os_, ss_ = [], []
    for r in range(world):
        bt_l, ctx_l = cp.shard_sequences(d["block_table"], d["ctx"], 16, world, r)
        o, s = cp.local_state_gpu(g["q"], g["k_cache"], g["v_cache"], bt_l.to(DEV),
                                  ctx_l.to(DEV), 4, d["sm_scale"])
        if poison is not None:
            empty = (ctx_l == 0).to(DEV)
            s[empty] = math.nan if poison == "nan" else math.inf
            o[empty] = math.nan
        os_.append(o)
        ss_.append(s)
    o, s = cp.merge_rank_states_gpu(torch.stack(os_), torch.stack(ss_))
    torch.cuda.synchronize()
    assert lib.get_device_error() == (0, 0)
    o_r, s_r = oracle.attend_full(d["q"], d["k_cache"], d["v_cache"], d["block_table"],
                                  d["ctx"], d["sm_scale"])
    assert o.dtype == torch.float32
    assert_s_close(s, s_r, DEC_LSE_ATOL, "s")
    assert_v_close(o, o_r, 2e-3, 0.0, "o", empty_rows=(s_r == -math.inf))
