"""skv_merge_states_noalloc: the N-state merge for callers that cannot allocate.

Some callers cannot call cudaMalloc (a plugin inside a runtime that owns all
device memory, a decode loop that must not risk an allocation's device
synchronisation), so this entry point keeps its scratch in a fixed array inside
the library instead of taking a workspace.  The test calls it through the C ABI
twice in a row on a shape that takes the two-level (scratch-using) path and on
one that does not, and checks each result against skv_merge_states with a
caller-provided workspace, within the merge tolerances of the other tests.
This file is collected last so that a run stopping at the first failure has
already run every other test; it also passes when run on its own.
"""
import ctypes

import pytest
import torch

from gpu_helpers import V_TOL, assert_s_close, assert_v_close, require_gpu, skv

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


@pytest.mark.parametrize("S,N,H,D,dtype", [(16, 1024, 8, 128, torch.float32),
                                           (8, 200, 2, 64, torch.float16),
                                           (300, 40, 16, 128, torch.float32)])
def test_noalloc_matches_workspace_merge_twice(lib, S, N, H, D, dtype):
    from split_kv_lse_gb300 import workloads as W
    d = W.merge_states_inputs(S, N, H, D, dtype, seed=S + N + D, empty_p=0.1)
    v, s = d["v"].to(DEV), d["s"].to(DEV)
    need = lib.merge_states_workspace_size(S, N, H, D)
    ws = torch.zeros(max(need, 16), dtype=torch.uint8, device=DEV)
    vr, sr = lib.merge_states(v, s, workspace=ws)
    atol, rtol = V_TOL[dtype]
    for _ in range(2):  # the shared scratch keeps the previous call's contents
        vo, so = noalloc(lib, v, s)
        torch.cuda.synchronize()
        assert_s_close(so, sr.double().cpu().numpy(), 1e-5)
        assert_v_close(vo, vr.double().cpu().numpy(), atol, rtol)


def test_noalloc_rejects_bad_arguments(lib):
    f = lib._ffi.lib().skv_merge_states_noalloc
    assert f(None, None, None, None, 4, 3, 2, 64, 0, None) == 1       # null pointers
    assert f(None, None, None, None, 4, 0, 2, 64, 0, None) == 1       # N = 0
    assert f(None, None, None, None, 0, 3, 2, 64, 0, None) == 0       # empty: no-op
