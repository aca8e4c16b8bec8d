"""Parity of the merge kernels (merge_state, merge_state_in_place, merge_states)
with the fp64 oracle, element by element, on the seeded workloads at full size
and on edge cases; plus the identities the pages fix, checked on the GPU
(commutativity and the empty-state identity bit-exact).

Pages: "F2 讲解：merge_state，以 2 为底的 LSE 合并" §①, §③, §④, §⑤;
"FlashAttention 的空行 LSE:FA-2 的 +inf 约定与后来的变化" §2.2."""
import math

import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import assert_states, np64, require_gpu, skv
from split_kv_lse_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def lib():
    require_gpu()
    return skv()


def _cuda(d):
    return {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in d.items()}


def _check_merge_state(lib, d, dtype):
    g = _cuda(d)
    v, s = lib.merge_state(g["v_a"], g["s_a"], g["v_b"], g["s_b"])
    torch.cuda.synchronize()
    vr, sr = oracle.merge_state(d["v_a"], d["s_a"], d["v_b"], d["s_b"])
    assert_states(v, s, vr, sr, dtype)
    return v, s


def test_merge_state_tiny(lib):
    d = W.merge_state_tiny()
    v, s = _check_merge_state(lib, d, torch.float32)
    sf, vf = np64(s).reshape(-1), np64(v).reshape(-1, 64)
    # Row 3 (a empty) equals b exactly, row 7 (b empty) equals a, row 11 is (0, -inf).
    assert np.array_equal(vf[3], np64(d["v_b"]).reshape(-1, 64)[3])
    assert sf[3] == np64(d["s_b"]).reshape(-1)[3]
    assert np.array_equal(vf[7], np64(d["v_a"]).reshape(-1, 64)[7])
    assert sf[11] == -math.inf and np.all(vf[11] == 0)


def test_merge_state_large_fp16(lib):
    """S=8192, H=32, D=128 fp16 with empty, double-empty and +inf/NaN inputs."""
    d = W.merge_state_large()
    assert torch.isinf(d["s_a"]).any() and torch.isnan(d["s_b"]).any()
    _check_merge_state(lib, d, torch.float16)


def test_merge_state_in_place_large(lib):
    d = W.merge_state_large()
    g = _cuda(d)
    v, s = g["v_a"].clone(), g["s_a"].clone()
    r = lib.merge_state_in_place(v, s, g["v_b"], g["s_b"])
    assert r[0].data_ptr() == v.data_ptr()
    torch.cuda.synchronize()
    vr, sr = oracle.merge_state(d["v_a"], d["s_a"], d["v_b"], d["s_b"])
    assert_states(v, s, vr, sr, torch.float16)
    # Same bits as the out-of-place kernel.
    vo, so = lib.merge_state(g["v_a"], g["s_a"], g["v_b"], g["s_b"])
    assert torch.equal(vo, v) and torch.equal(so.isnan(), s.isnan())
    assert torch.equal(torch.nan_to_num(so), torch.nan_to_num(s))


@pytest.mark.parametrize("dtype", [torch.float32, torch.float16, torch.bfloat16])
@pytest.mark.parametrize("S,H,D", [(1, 1, 64), (7, 3, 8 * 4), (33, 5, 96), (129, 2, 128),
                                   (5, 3, 256)])
def test_merge_state_shapes(lib, dtype, S, H, D):
    if D * torch.tensor([], dtype=dtype).element_size() > 512:
        pytest.skip("rows over 512 bytes are unsupported")
    d = W.merge_state_inputs(S, H, D, dtype, seed=S * 131 + D, empty_p=0.1,
                             double_empty_p=0.05, poison_p=0.05)
    _check_merge_state(lib, d, dtype)


def test_merge_state_zero_rows_is_noop(lib):
    v = torch.zeros(0, 4, 64, device=DEV)
    s = torch.zeros(0, 4, device=DEV)
    lib.merge_state(v, s, v, s)


def test_merge_state_identities_bit_exact(lib):
    """Commutative (bit-exact) and empty + x = x (bit-exact) on the GPU."""
    d = _cuda(W.merge_state_inputs(512, 8, 128, torch.float16, seed=3, empty_p=0.1))
    v1, s1 = lib.merge_state(d["v_a"], d["s_a"], d["v_b"], d["s_b"])
    v2, s2 = lib.merge_state(d["v_b"], d["s_b"], d["v_a"], d["s_a"])
    assert torch.equal(v1, v2) and torch.equal(s1, s2)
    ve = torch.zeros_like(d["v_a"])
    se = torch.full_like(d["s_a"], -math.inf)
    v3, s3 = lib.merge_state(d["v_a"], d["s_a"], ve, se)
    assert torch.equal(v3, d["v_a"]) and torch.equal(s3, d["s_a"])
    v4, s4 = lib.merge_state(ve, se, ve, se)
    assert torch.all(v4 == 0) and torch.all(s4 == -math.inf)
    # +inf / NaN incoming s behave exactly like an empty state.
    for bad in (math.inf, math.nan):
        sb = torch.full_like(d["s_a"], bad)
        v5, s5 = lib.merge_state(d["v_a"], d["s_a"], d["v_b"], sb)
        assert torch.equal(v5, d["v_a"]) and torch.equal(s5, d["s_a"])


def test_merge_state_printed_selftest(lib):
    """F2 §⑧ 自测 1 on the GPU: s = 10, 10; v = [1,0], [0,1] -> [0.5, 0.5], 11."""
    va = torch.zeros(1, 1, 4, device=DEV)
    vb = torch.zeros(1, 1, 4, device=DEV)
    va[0, 0, 0] = 1
    vb[0, 0, 1] = 1
    s = torch.full((1, 1), 10.0, device=DEV)
    v, so = lib.merge_state(va, s, vb, s)
    assert v.cpu().tolist() == [[[0.5, 0.5, 0.0, 0.0]]] and so.item() == 11.0


def _check_merge_states(lib, d, dtype, workspace=None):
    g = _cuda(d)
    v, s = lib.merge_states(g["v"], g["s"], workspace=workspace)
    torch.cuda.synchronize()
    vr, sr = oracle.merge_states(d["v"], d["s"])
    assert_states(v, s, vr, sr, dtype)
    return v, s


def test_merge_states_main(lib):
    """S=256, N=64, H=32, D=128 fp32, 5% empty states."""
    _check_merge_states(lib, W.merge_states_main(), torch.float32)


def _ws(lib, S, N, H, D):
    n = lib.merge_states_workspace_size(S, N, H, D)
    return torch.zeros(max(n, 16), dtype=torch.uint8, device=DEV), n


@pytest.mark.parametrize("N", W.MERGE_STATES_SWEEP_N)
@pytest.mark.parametrize("use_ws", [False, True])
def test_merge_states_sweep(lib, N, use_ws):
    """S=16, H=8, D=128, N in {1, 2, 3, 128, 1024}: one CTA per row, or the
    two-level split through a workspace (which must be reusable without
    re-zeroing: its arrival tickets are reset by the last CTA of each row)."""
    d = W.merge_states_sweep(N)
    ws = None
    if use_ws:
        ws, need = _ws(lib, 16, N, 8, 128)
    _check_merge_states(lib, d, torch.float32, ws)
    if use_ws:
        # A second call on the same workspace gives the same answer, and the
        # workspace's ticket counters are back to zero.
        v1, s1 = lib.merge_states(d["v"].to(DEV), d["s"].to(DEV), workspace=ws)
        v2, s2 = lib.merge_states(d["v"].to(DEV), d["s"].to(DEV), workspace=ws)
        assert torch.equal(v1, v2) and torch.equal(s1, s2)
        torch.cuda.synchronize()


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16, torch.float32])
@pytest.mark.parametrize("S,N,H,D", [(3, 1, 2, 64), (5, 7, 3, 128), (1, 300, 1, 128),
                                     (2, 33, 4, 64), (4097, 2, 1, 64), (9, 5, 7, 96)])
def test_merge_states_shapes(lib, dtype, S, N, H, D):
    d = W.merge_states_inputs(S, N, H, D, dtype, seed=S + N * 7 + D, empty_p=0.2)
    ws, _ = _ws(lib, S, N, H, D)
    _check_merge_states(lib, d, dtype, ws)
    _check_merge_states(lib, d, dtype, None)


def test_merge_states_all_empty_and_poisoned(lib):
    S, N, H, D = 6, 5, 3, 64
    v = torch.randn(S, N, H, D)
    s = torch.full((S, N, H), -math.inf)
    s[0, 2, 1] = 3.0
    s[1, :, 0] = math.inf
    s[2, :, 2] = math.nan
    s[3, 1, 1] = math.nan
    s[3, 4, 1] = 7.5
    _check_merge_states(lib, {"v": v, "s": s}, torch.float32)


def test_merge_states_two_equals_merge_state(lib):
    d = _cuda(W.merge_state_inputs(300, 4, 128, torch.float32, seed=9, empty_p=0.2))
    v2, s2 = lib.merge_state(d["v_a"], d["s_a"], d["v_b"], d["s_b"])
    vn, sn = lib.merge_states(torch.stack([d["v_a"], d["v_b"]], 1).contiguous(),
                              torch.stack([d["s_a"], d["s_b"]], 1).contiguous())
    torch.testing.assert_close(vn, v2, rtol=1e-6, atol=1e-7)
    torch.testing.assert_close(sn, s2, rtol=0, atol=1e-6)


_ROW_SIZES_SCRIPT = r"""
import sys, torch
sys.path.insert(0, sys.argv[1]); sys.path.insert(0, sys.argv[1] + "/tests")
import oracle
from gpu_helpers import assert_states, skv
from split_kv_lse_gb300 import workloads as W
lib = skv()
# Short rows and few states first (a small shared-memory need of the
# many-rows kernel, 4096 rows), then long rows with more states.
for (S, N, H, D, dt) in ((128, 2, 32, 64, torch.float16), (128, 32, 32, 128, torch.float32)):
    d = W.merge_states_inputs(S, N, H, D, dt, seed=N)
    v, s = lib.merge_states(d["v"].to("cuda:0"), d["s"].to("cuda:0"))
    torch.cuda.synchronize()
    vr, sr = oracle.merge_states(d["v"], d["s"])
    assert_states(v, s, vr, sr, dt)
print("ok")
"""


def test_merge_states_row_sizes_in_a_fresh_process(lib):
    """The many-rows N-state kernel takes more shared memory for longer rows
    and more states: a first call with the smallest need must not cap a
    later call with the largest (run in a fresh process, where the first
    call is known)."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", _ROW_SIZES_SCRIPT, root], capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout + r.stderr


@pytest.mark.parametrize("dtype", [torch.float32, torch.float16, torch.bfloat16])
@pytest.mark.parametrize("S,N,H,D", [(16, 1024, 8, 128), (2, 5000, 3, 64), (32, 260, 128, 64),
                                     (1, 16384, 1, 64), (1, 16385, 1, 64), (3, 40, 1, 128)])
def test_merge_states_two_level_warp_split(lib, dtype, S, N, H, D):
    """Few rows with many states through a workspace: each row's states are
    cut over up to 64 warps, whose unnormalised partials the row's last warp
    merges ([F2] §① associativity, §⑦ the large-N kernel).  Shapes cover the
    large-N sweep's N = 1024, 4096 rows with N > 256, the largest N the warp
    split takes (16384) and one past it (the CTA path), and few states.  The
    workspace is reused without re-zeroing for a second call, which must give
    the same bits."""
    if dtype == torch.float32 and D * 4 > 512:
        pytest.skip("fp32 rows of more than 512 bytes are not supported")
    d = W.merge_states_inputs(S, N, H, D, dtype, seed=S * 31 + N + D, empty_p=0.05)
    ws, need = _ws(lib, S, N, H, D)
    assert need > 0
    v1, s1 = _check_merge_states(lib, d, dtype, ws)
    v2, s2 = lib.merge_states(d["v"].to(DEV), d["s"].to(DEV), workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(v1, v2) and torch.equal(s1, s2)
    assert lib.get_device_error() == (0, 0)


def test_merge_states_two_level_empty_chunks_and_poison(lib):
    """Rows whose states are all empty, all poisoned (+inf or NaN s), or empty
    except for one state in one chunk: every warp's partial of such a row may
    be empty, and the row's merge must still be exact (v = 0, s = -inf when
    nothing is left)."""
    S, N, H, D = 8, 2048, 2, 128
    g = torch.Generator().manual_seed(77)
    v = torch.randn(S, N, H, D, generator=g)
    s = 30 + 8 * torch.randn(S, N, H, generator=g)
    s[0] = -math.inf                   # all empty
    s[1, :, 0] = math.inf              # all +inf (read as empty)
    s[1, :, 1] = math.nan              # all NaN
    s[2] = -math.inf
    s[2, 1999, 1] = 4.0                # one state, in the last chunk
    v[2, :, 0] = math.nan              # empty states' v are never read
    s[3, ::3, :] = math.nan            # a third poisoned
    ws, _ = _ws(lib, S, N, H, D)
    _check_merge_states(lib, {"v": v, "s": s}, torch.float32, ws)


@pytest.mark.parametrize("dtype", [torch.float32, torch.float16, torch.bfloat16])
@pytest.mark.parametrize("S,N,H,D", [(100, 3, 1, 128), (80, 33, 1, 64), (10, 4096, 9, 64),
                                     (90, 4097, 1, 64), (16, 17, 8, 128)])
@pytest.mark.parametrize("use_ws", [False, True])
def test_merge_states_row_per_cta(lib, dtype, S, N, H, D, use_ws):
    """Enough rows for about one per SM and up to 16 x 256 states: one CTA per
    row, 16 warps each streaming a chunk of the states, their partials merged
    in shared memory (warps past N hold nothing); N = 4097 and above takes the
    other paths.  Same result with or without a workspace."""
    d = W.merge_states_inputs(S, N, H, D, dtype, seed=S + 3 * N + D, empty_p=0.1)
    ws = _ws(lib, S, N, H, D)[0] if use_ws else None
    _check_merge_states(lib, d, dtype, ws)
    assert lib.get_device_error() == (0, 0)
