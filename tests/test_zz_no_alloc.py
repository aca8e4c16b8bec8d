"""skv_merge_states_noalloc: the N-state merge for callers that cannot allocate.

Some callers cannot call cudaMalloc (a plugin inside a runtime that owns all
device memory, a decode loop that must not risk an allocation's device
synchronisation), so this entry point keeps its scratch in a fixed array inside
the library instead of taking a workspace.  The tests call it through the C ABI
twice in a row, on shapes that take the two-level (scratch-using) path --
including the heaviest one a GB300 allows, fp16 rows of 256 values with just
under 2 x SM-count rows -- and on one that does not, and check every result
against the fp64 oracle at the merge tolerances of the other tests and against
skv_merge_states with a caller-provided workspace.  A smaller shape right after
a larger one checks that the partials a previous call left in the shared array
are not read.  This file is collected last so that a run stopping at the first
failure has already run every other test; it also passes when run on its own.
"""
import ctypes

import pytest
import torch

import oracle
from gpu_helpers import V_TOL, assert_s_close, assert_states, assert_v_close, require_gpu, skv

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
DT = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2}


@pytest.fixture(scope="module")
def lib():
    require_gpu()
    return skv()


def noalloc(m, v, s):
    S, N, H, D = v.shape
    vo = torch.empty(S, H, D, dtype=v.dtype, device=DEV)
    so = torch.empty(S, H, dtype=torch.float32, device=DEV)
    st = m._ffi.lib().skv_merge_states_noalloc(
        v.data_ptr(), s.data_ptr(), vo.data_ptr(), so.data_ptr(), S, N, H, D, DT[v.dtype],
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, m._ffi.STATUS.get(st, st)
    return vo, so


def scratch_need(m, S, N, H, D, dtype):
    return int(m._ffi.lib().skv_merge_states_noalloc_scratch_size(S, N, H, D, DT[dtype], 0))


def heaviest_rows():
    """S*H just under 2 x SM count: the most two-level partials a call can need."""
    return 2 * torch.cuda.get_device_properties(0).multi_processor_count - 1


def check_shape(m, S, N, H, D, dtype, seed):
    from split_kv_lse_gb300 import workloads as W
    d = W.merge_states_inputs(S, N, H, D, dtype, seed=seed, empty_p=0.1)
    v, s = d["v"].to(DEV), d["s"].to(DEV)
    vr, sr = oracle.merge_states(d["v"], d["s"])
    need = m.merge_states_workspace_size(S, N, H, D)
    ws = torch.zeros(max(need, 16), dtype=torch.uint8, device=DEV)
    vw, sw = m.merge_states(v, s, workspace=ws)
    atol, rtol = V_TOL[dtype]
    for _ in range(2):  # the shared scratch keeps the previous call's contents
        vo, so = noalloc(m, v, s)
        torch.cuda.synchronize()
        assert_states(vo, so, vr, sr, dtype)
        assert_s_close(so, sw.double().cpu().numpy(), 1e-5)
        assert_v_close(vo, vw.double().cpu().numpy(), atol, rtol)


@pytest.mark.parametrize("S,N,H,D,dtype", [(16, 1024, 8, 128, torch.float32),
                                           (8, 200, 2, 64, torch.float16),
                                           (300, 40, 16, 128, torch.float32)])
def test_noalloc_matches_oracle_twice(lib, S, N, H, D, dtype):
    check_shape(lib, S, N, H, D, dtype, seed=S + N + D)


def test_noalloc_heaviest_shape_then_smaller(lib):
    """fp16 D=256 with S*H = 2*SM - 1 rows (about 612 KB of scratch on a GB300),
    then a smaller two-level shape that reuses the front of the array."""
    rows = heaviest_rows()
    need = scratch_need(lib, rows, 64, 1, 256, torch.float16)
    assert 0 < need <= 1 << 20
    check_shape(lib, rows, 64, 1, 256, torch.float16, seed=21)
    assert 0 < scratch_need(lib, 4, 300, 4, 64, torch.bfloat16) < need
    check_shape(lib, 4, 300, 4, 64, torch.bfloat16, seed=22)


def test_noalloc_rejects_bad_arguments(lib):
    f = lib._ffi.lib().skv_merge_states_noalloc
    assert f(None, None, None, None, 4, 3, 2, 64, 0, None) == 1       # null pointers
    assert f(None, None, None, None, 4, 0, 2, 64, 0, None) == 1       # N = 0
    assert f(None, None, None, None, 0, 3, 2, 64, 0, None) == 0       # empty: no-op
