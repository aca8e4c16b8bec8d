"""GB300 (sm_103a) split-KV decode attention and attention-state merging.

A thin Python binding over the C ABI of libskv.so (include/skv.h): every
function here only checks tensor metadata, passes device pointers, sizes and
the current CUDA stream to the library, and returns the output tensors.  All
arithmetic runs in the library's CUDA kernels; there is no CPU or PyTorch
fallback, and a missing library raises.

States follow the pages' convention: v is the softmax-normalised output over a
key subset, s = log2(sum exp(score)) its base-2 log-sum-exp (fp32); an empty
state is (v = 0, s = -inf).
"""
from __future__ import annotations

import ctypes

import torch

from . import _ffi
from ._ffi import SkvError

__all__ = [
    "SkvError", "merge_state", "merge_state_in_place", "merge_states",
    "merge_states_workspace_size", "split_page_range", "splitkv_decode_plan",
    "splitkv_decode", "SplitPlan", "splitkv_plan_varlen", "splitkv_decode_varlen",
    "cascade_workspace_size", "cascade_decode", "cascade_decode_varlen", "get_device_error",
    "poll_device_error", "selftest_bounded_wait", "abi_version", "library_path",
]

_DT = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2}


def library_path() -> str:
    return _ffi.LIB


def abi_version() -> int:
    return int(_ffi.lib().skv_abi_version())


def _stream(t: torch.Tensor) -> int:
    return torch.cuda.current_stream(t.device).cuda_stream


def _ptr(t):
    return None if t is None else t.data_ptr()


def _need(t: torch.Tensor, name: str, dtype=None, shape=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def merge_state(v_a, s_a, v_b, s_b, v_out=None, s_out=None):
    """Two-state merge of [S, H, D] / [S, H] states -> (v, s)."""
    S, H, D = v_a.shape
    _need(v_a, "v_a")
    dt = v_a.dtype
    _need(v_b, "v_b", dt, (S, H, D))
    _need(s_a, "s_a", torch.float32, (S, H))
    _need(s_b, "s_b", torch.float32, (S, H))
    v_out = torch.empty_like(v_a) if v_out is None else v_out
    s_out = torch.empty_like(s_a) if s_out is None else s_out
    _need(v_out, "v_out", dt, (S, H, D))
    _need(s_out, "s_out", torch.float32, (S, H))
    _ffi.check("skv_merge_state", _ffi.lib().skv_merge_state(
        v_a.data_ptr(), s_a.data_ptr(), v_b.data_ptr(), s_b.data_ptr(), v_out.data_ptr(),
        s_out.data_ptr(), S, H, D, _DT[dt], _stream(v_a)))
    return v_out, s_out


def merge_state_in_place(v, s, v_other, s_other):
    """(v, s) <- merge_state((v, s), (v_other, s_other)), in place."""
    S, H, D = v.shape
    _need(v, "v")
    _need(v_other, "v_other", v.dtype, (S, H, D))
    _need(s, "s", torch.float32, (S, H))
    _need(s_other, "s_other", torch.float32, (S, H))
    _ffi.check("skv_merge_state_in_place", _ffi.lib().skv_merge_state_in_place(
        v.data_ptr(), s.data_ptr(), v_other.data_ptr(), s_other.data_ptr(), S, H, D,
        _DT[v.dtype], _stream(v)))
    return v, s


def merge_states_workspace_size(S: int, N: int, H: int, D: int) -> int:
    return int(_ffi.lib().skv_merge_states_workspace_size(S, N, H, D))


def merge_states(v, s, workspace=None, v_out=None, s_out=None):
    """N-state merge of v [S, N, H, D], s [S, N, H] -> (v [S, H, D], s [S, H]).

    workspace: optional zero-filled uint8 CUDA tensor of at least
    merge_states_workspace_size(S, N, H, D) bytes; it is left zero-filled.
    """
    S, N, H, D = v.shape
    _need(v, "v")
    _need(s, "s", torch.float32, (S, N, H))
    v_out = torch.empty((S, H, D), dtype=v.dtype, device=v.device) if v_out is None else v_out
    s_out = torch.empty((S, H), dtype=torch.float32, device=v.device) if s_out is None else s_out
    _need(v_out, "v_out", v.dtype, (S, H, D))
    _need(s_out, "s_out", torch.float32, (S, H))
    ws_bytes = 0
    if workspace is not None:
        _need(workspace, "workspace")
        ws_bytes = workspace.numel() * workspace.element_size()
    _ffi.check("skv_merge_states", _ffi.lib().skv_merge_states(
        v.data_ptr(), s.data_ptr(), v_out.data_ptr(), s_out.data_ptr(), S, N, H, D,
        _DT[v.dtype], _ptr(workspace), ws_bytes, _stream(v)))
    return v_out, s_out


def split_page_range(ctx: int, page: int, num_splits: int, split: int):
    """Raw (p_start, p_end) of one split, computed by the library on the host."""
    a, b = ctypes.c_int32(), ctypes.c_int32()
    _ffi.check("skv_split_page_range", _ffi.lib().skv_split_page_range(
        ctx, page, num_splits, split, ctypes.byref(a), ctypes.byref(b)))
    return a.value, b.value


def splitkv_decode_plan(ctx, Hkv: int, page: int = 16, sm_count: int = 0) -> int:
    """Split count for one decode step (host; sm_count 0 = current device)."""
    vals = [int(x) for x in (ctx.tolist() if hasattr(ctx, "tolist") else ctx)]
    arr = (ctypes.c_int32 * max(1, len(vals)))(*vals)
    ns = ctypes.c_int32()
    _ffi.check("skv_splitkv_decode_plan", _ffi.lib().skv_splitkv_decode_plan(
        len(vals), arr, Hkv, page, sm_count, ctypes.byref(ns)))
    return ns.value


class SplitPlan:
    """A per-sequence split plan from skv_splitkv_plan_varlen: the host int32
    buffer ([num_units][2] work units, longest first, then [B] split counts),
    its unit count, longest split and split-axis length, and a cached device
    copy per device."""

    def __init__(self, host: torch.Tensor, num_units: int, max_split_pages: int,
                 max_splits: int, B: int):
        self.host = host
        self.num_units = num_units
        self.max_split_pages = max_split_pages
        self.max_splits = max_splits
        self.B = B
        self._dev = {}

    @property
    def num_splits(self) -> torch.Tensor:
        """Split count of each sequence (host int32 [B])."""
        return self.host[2 * self.num_units:2 * self.num_units + self.B]

    def device(self, dev) -> torch.Tensor:
        dev = torch.device(dev)
        if dev not in self._dev:
            t = torch.empty(max(4, self.host.numel()), dtype=torch.int32, device=dev)
            t[:self.host.numel()].copy_(self.host)
            self._dev[dev] = t
        return self._dev[dev]


def splitkv_plan_varlen(ctx, page: int = 16, max_splits: int = 16,
                        pages_per_split: int = 8) -> SplitPlan:
    """Per-sequence split counts and work list (host; see skv_splitkv_plan_varlen)."""
    vals = [int(x) for x in (ctx.tolist() if hasattr(ctx, "tolist") else ctx)]
    B = len(vals)
    arr = (ctypes.c_int32 * max(1, B))(*vals)
    nu, msp = ctypes.c_int32(), ctypes.c_int32()
    f = _ffi.lib().skv_splitkv_plan_varlen
    _ffi.check("skv_splitkv_plan_varlen", f(B, arr, page, max_splits, pages_per_split, None, 0,
                                            ctypes.byref(nu), ctypes.byref(msp)))
    cap = 2 * nu.value + B
    host = torch.zeros(max(1, cap), dtype=torch.int32)
    _ffi.check("skv_splitkv_plan_varlen", f(
        B, arr, page, max_splits, pages_per_split,
        ctypes.cast(host.data_ptr(), ctypes.POINTER(ctypes.c_int32)), cap, ctypes.byref(nu),
        ctypes.byref(msp)))
    return SplitPlan(host[:cap], nu.value, msp.value, max_splits, B)


def _decode_bufs(q, k_cache, v_cache, block_table, ctx, ns, o_part, lse_part, out, lse_out,
                 combine, ranges_dbg):
    B, Hq, D = q.shape
    _need(q, "q")
    _need(k_cache, "k_cache", q.dtype)
    _need(v_cache, "v_cache", q.dtype, tuple(k_cache.shape))
    _need(block_table, "block_table", torch.int32)
    _need(ctx, "ctx", torch.int32, (B,))
    if k_cache.shape[3] != D or block_table.dim() != 2 or block_table.shape[0] != B:
        raise ValueError("inconsistent decode shapes")
    dev = q.device
    if o_part is None:
        o_part = torch.empty((B, Hq, ns, D), dtype=torch.float32, device=dev)
    if lse_part is None:
        lse_part = torch.empty((B, Hq, ns), dtype=torch.float32, device=dev)
    _need(o_part, "o_part", torch.float32, (B, Hq, ns, D))
    _need(lse_part, "lse_part", torch.float32, (B, Hq, ns))
    if combine:
        out = torch.empty((B, Hq, D), dtype=q.dtype, device=dev) if out is None else out
        lse_out = torch.empty((B, Hq), dtype=torch.float32, device=dev) if lse_out is None else lse_out
        _need(out, "out", q.dtype, (B, Hq, D))
        _need(lse_out, "lse_out", torch.float32, (B, Hq))
    else:
        out = lse_out = None
    if ranges_dbg is not None:
        _need(ranges_dbg, "ranges_dbg", torch.int32, (B, ns, 2))
    return o_part, lse_part, out, lse_out


def splitkv_decode_varlen(q, k_cache, v_cache, block_table, ctx, plan: SplitPlan,
                          sm_scale: float, o_part=None, lse_part=None, out=None, lse_out=None,
                          combine: bool = True, ranges_dbg=None):
    """Split-KV paged decode with the per-sequence split counts of `plan`.
    Returns (out, lse_out, o_part, lse_part); o_part has plan.max_splits slots
    per (b, hq), of which the first plan.num_splits[b] are written."""
    B, Hq, D = q.shape
    P, Hkv, page, _ = k_cache.shape
    if plan.B != B:
        raise ValueError("the plan was made for another batch size")
    o_part, lse_part, out, lse_out = _decode_bufs(q, k_cache, v_cache, block_table, ctx,
                                                  plan.max_splits, o_part, lse_part, out,
                                                  lse_out, combine, ranges_dbg)
    dplan = plan.device(q.device)
    _ffi.check("skv_splitkv_decode_varlen", _ffi.lib().skv_splitkv_decode_varlen(
        q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), P, block_table.data_ptr(),
        block_table.shape[1], ctx.data_ptr(), B, Hq, Hkv, D, page, plan.max_splits,
        dplan.data_ptr(), plan.num_units, plan.max_split_pages, float(sm_scale), _DT[q.dtype],
        o_part.data_ptr(), lse_part.data_ptr(), _ptr(out), _ptr(lse_out), _ptr(ranges_dbg),
        _stream(q)))
    return out, lse_out, o_part, lse_part


def splitkv_decode(q, k_cache, v_cache, block_table, ctx, num_splits: int, sm_scale: float,
                   o_part=None, lse_part=None, out=None, lse_out=None, combine: bool = True,
                   ranges_dbg=None):
    """Split-KV paged decode.

    q [B, Hq, D] fp16; k_cache, v_cache [P, Hkv, page, D] fp16; block_table
    [B, max_pages] int32; ctx [B] int32 (device).  Returns
    (out, lse_out, o_part, lse_part); out/lse_out are None when combine=False.
    """
    B, Hq, D = q.shape
    P, Hkv, page, D2 = k_cache.shape
    _need(q, "q")
    _need(k_cache, "k_cache", q.dtype)
    _need(v_cache, "v_cache", q.dtype, tuple(k_cache.shape))
    _need(block_table, "block_table", torch.int32)
    _need(ctx, "ctx", torch.int32, (B,))
    if D2 != D or block_table.dim() != 2 or block_table.shape[0] != B:
        raise ValueError("inconsistent decode shapes")
    dev = q.device
    if o_part is None:
        o_part = torch.empty((B, Hq, num_splits, D), dtype=torch.float32, device=dev)
    if lse_part is None:
        lse_part = torch.empty((B, Hq, num_splits), dtype=torch.float32, device=dev)
    _need(o_part, "o_part", torch.float32, (B, Hq, num_splits, D))
    _need(lse_part, "lse_part", torch.float32, (B, Hq, num_splits))
    if combine:
        out = torch.empty((B, Hq, D), dtype=q.dtype, device=dev) if out is None else out
        lse_out = torch.empty((B, Hq), dtype=torch.float32, device=dev) if lse_out is None else lse_out
        _need(out, "out", q.dtype, (B, Hq, D))
        _need(lse_out, "lse_out", torch.float32, (B, Hq))
    else:
        out = lse_out = None
    if ranges_dbg is not None:
        _need(ranges_dbg, "ranges_dbg", torch.int32, (B, num_splits, 2))
    _ffi.check("skv_splitkv_decode", _ffi.lib().skv_splitkv_decode(
        q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), P, block_table.data_ptr(),
        block_table.shape[1], ctx.data_ptr(), B, Hq, Hkv, D, page, num_splits, float(sm_scale),
        _DT[q.dtype], o_part.data_ptr(), lse_part.data_ptr(), _ptr(out), _ptr(lse_out),
        _ptr(ranges_dbg), _stream(q)))
    return out, lse_out, o_part, lse_part


def cascade_workspace_size(B: int, Hq: int, Hkv: int, D: int, prefix_len: int,
                           sm_count: int = 0) -> int:
    return int(_ffi.lib().skv_cascade_workspace_size(B, Hq, Hkv, D, prefix_len, sm_count))


def cascade_decode(q, k_cache, v_cache, prefix_pages, prefix_len: int, block_table, ctx,
                   num_splits: int, sm_scale: float, out=None, lse_out=None, o_pre=None,
                   s_pre=None, o_part=None, lse_part=None, workspace=None):
    """Two-level cascade decode: shared prefix (tensor cores) + per-request suffix.

    Returns (out, lse_out, o_pre, s_pre, o_part, lse_part).  prefix_pages is a
    device int32 tensor of the prefix's pool pages.
    """
    B, Hq, D = q.shape
    P, Hkv, page, D2 = k_cache.shape
    _need(q, "q")
    _need(k_cache, "k_cache", q.dtype)
    _need(v_cache, "v_cache", q.dtype, tuple(k_cache.shape))
    _need(block_table, "block_table", torch.int32)
    _need(ctx, "ctx", torch.int32, (B,))
    _need(prefix_pages, "prefix_pages", torch.int32)
    if D2 != D or block_table.dim() != 2 or block_table.shape[0] != B:
        raise ValueError("inconsistent cascade shapes")
    dev = q.device
    f32 = torch.float32
    out = torch.empty((B, Hq, D), dtype=q.dtype, device=dev) if out is None else out
    lse_out = torch.empty((B, Hq), dtype=f32, device=dev) if lse_out is None else lse_out
    o_pre = torch.empty((B, Hq, D), dtype=f32, device=dev) if o_pre is None else o_pre
    s_pre = torch.empty((B, Hq), dtype=f32, device=dev) if s_pre is None else s_pre
    if o_part is None:
        o_part = torch.empty((B, Hq, num_splits, D), dtype=f32, device=dev)
    if lse_part is None:
        lse_part = torch.empty((B, Hq, num_splits), dtype=f32, device=dev)
    for t, n, shp in ((out, "out", (B, Hq, D)), (lse_out, "lse_out", (B, Hq)),
                      (o_pre, "o_pre", (B, Hq, D)), (s_pre, "s_pre", (B, Hq)),
                      (o_part, "o_part", (B, Hq, num_splits, D)),
                      (lse_part, "lse_part", (B, Hq, num_splits))):
        _need(t, n, None, shp)
    need = cascade_workspace_size(B, Hq, Hkv, D, prefix_len)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    _need(workspace, "workspace")
    ws_bytes = workspace.numel() * workspace.element_size()
    _ffi.check("skv_cascade_decode", _ffi.lib().skv_cascade_decode(
        q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), P, prefix_pages.data_ptr(),
        int(prefix_len), block_table.data_ptr(), block_table.shape[1], ctx.data_ptr(), B, Hq,
        Hkv, D, page, num_splits, float(sm_scale), _DT[q.dtype], o_pre.data_ptr(),
        s_pre.data_ptr(), o_part.data_ptr(), lse_part.data_ptr(), out.data_ptr(),
        lse_out.data_ptr(), workspace.data_ptr(), ws_bytes, _stream(q)))
    return out, lse_out, o_pre, s_pre, o_part, lse_part


def cascade_decode_varlen(q, k_cache, v_cache, prefix_pages, prefix_len: int, block_table, ctx,
                          plan: SplitPlan, sm_scale: float, out=None, lse_out=None, o_pre=None,
                          s_pre=None, o_part=None, lse_part=None, workspace=None):
    """Two-level cascade whose suffixes use the per-sequence split counts of
    `plan` (made over the suffix contexts).  Returns
    (out, lse_out, o_pre, s_pre, o_part, lse_part)."""
    B, Hq, D = q.shape
    P, Hkv, page, D2 = k_cache.shape
    if plan.B != B:
        raise ValueError("the plan was made for another batch size")
    _need(prefix_pages, "prefix_pages", torch.int32)
    ns = plan.max_splits
    o_part, lse_part, out, lse_out = _decode_bufs(q, k_cache, v_cache, block_table, ctx, ns,
                                                  o_part, lse_part, out, lse_out, True, None)
    dev = q.device
    f32 = torch.float32
    o_pre = torch.empty((B, Hq, D), dtype=f32, device=dev) if o_pre is None else o_pre
    s_pre = torch.empty((B, Hq), dtype=f32, device=dev) if s_pre is None else s_pre
    _need(o_pre, "o_pre", f32, (B, Hq, D))
    _need(s_pre, "s_pre", f32, (B, Hq))
    need = cascade_workspace_size(B, Hq, Hkv, D, prefix_len)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    _need(workspace, "workspace")
    ws_bytes = workspace.numel() * workspace.element_size()
    dplan = plan.device(dev)
    _ffi.check("skv_cascade_decode_varlen", _ffi.lib().skv_cascade_decode_varlen(
        q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), P, prefix_pages.data_ptr(),
        int(prefix_len), block_table.data_ptr(), block_table.shape[1], ctx.data_ptr(), B, Hq,
        Hkv, D, page, ns, dplan.data_ptr(), plan.num_units, plan.max_split_pages,
        float(sm_scale), _DT[q.dtype], o_pre.data_ptr(), s_pre.data_ptr(), o_part.data_ptr(),
        lse_part.data_ptr(), out.data_ptr(), lse_out.data_ptr(), workspace.data_ptr(), ws_bytes,
        _stream(q)))
    return out, lse_out, o_pre, s_pre, o_part, lse_part


def _levels_struct(levels, B):
    """ctypes array of skv_cascade_level for levels = [[(r0, r1, pages, length), ...], ...]
    (pages: device int32 tensor or None); returns it with the buffers it points into."""
    keep = []
    arr = (_ffi.CascadeLevel * max(1, len(levels)))()
    for li, groups in enumerate(levels):
        n = len(groups)
        starts = (ctypes.c_int32 * (n + 1))()
        lens = (ctypes.c_int32 * n)()
        pages = (ctypes.c_void_p * n)()
        for gi, (r0, r1, pg, length) in enumerate(groups):
            if gi == 0 and r0 != 0:
                raise ValueError("level groups must start at request 0")
            if gi > 0 and r0 != groups[gi - 1][1]:
                raise ValueError("level groups must be contiguous")
            starts[gi] = int(r0)
            lens[gi] = int(length)
            if pg is not None:
                _need(pg, "group pages", torch.int32)
                pages[gi] = pg.data_ptr()
        starts[n] = int(groups[-1][1]) if n else 0
        if n and starts[n] != B:
            raise ValueError("level groups must end at request B")
        arr[li].num_groups = n
        arr[li].group_start = ctypes.cast(starts, ctypes.POINTER(ctypes.c_int32))
        arr[li].group_len = ctypes.cast(lens, ctypes.POINTER(ctypes.c_int32))
        arr[li].group_pages = ctypes.cast(pages, ctypes.POINTER(ctypes.c_void_p))
        keep += [starts, lens, pages]
    return arr, keep


def cascade_multilevel_workspace_size(levels, B: int, Hq: int, Hkv: int, D: int,
                                      sm_count: int = 0) -> int:
    arr, _keep = _levels_struct(levels, B)
    return int(_ffi.lib().skv_cascade_multilevel_workspace_size(
        len(levels), ctypes.cast(arr, ctypes.c_void_p), B, Hq, Hkv, D, sm_count))


def cascade_decode_multilevel(q, k_cache, v_cache, levels, block_table, ctx, num_splits: int,
                              sm_scale: float, out=None, lse_out=None, o_pre=None, s_pre=None,
                              o_part=None, lse_part=None, workspace=None):
    """Multi-level cascade decode.  levels[l] is a list of groups (r0, r1, pages, length):
    requests [r0, r1) share `length` tokens on the device int32 page list `pages` at level l
    (the groups of a level cover 0..B in order).  Returns
    (out, lse_out, o_pre, s_pre, o_part, lse_part)."""
    B, Hq, D = q.shape
    P, Hkv, page, D2 = k_cache.shape
    _need(q, "q")
    _need(k_cache, "k_cache", q.dtype)
    _need(v_cache, "v_cache", q.dtype, tuple(k_cache.shape))
    _need(block_table, "block_table", torch.int32)
    _need(ctx, "ctx", torch.int32, (B,))
    if D2 != D or block_table.dim() != 2 or block_table.shape[0] != B:
        raise ValueError("inconsistent cascade shapes")
    dev = q.device
    f32 = torch.float32
    out = torch.empty((B, Hq, D), dtype=q.dtype, device=dev) if out is None else out
    lse_out = torch.empty((B, Hq), dtype=f32, device=dev) if lse_out is None else lse_out
    o_pre = torch.empty((B, Hq, D), dtype=f32, device=dev) if o_pre is None else o_pre
    s_pre = torch.empty((B, Hq), dtype=f32, device=dev) if s_pre is None else s_pre
    if o_part is None:
        o_part = torch.empty((B, Hq, num_splits, D), dtype=f32, device=dev)
    if lse_part is None:
        lse_part = torch.empty((B, Hq, num_splits), dtype=f32, device=dev)
    for t, n, shp in ((out, "out", (B, Hq, D)), (lse_out, "lse_out", (B, Hq)),
                      (o_pre, "o_pre", (B, Hq, D)), (s_pre, "s_pre", (B, Hq)),
                      (o_part, "o_part", (B, Hq, num_splits, D)),
                      (lse_part, "lse_part", (B, Hq, num_splits))):
        _need(t, n, None, shp)
    arr, keep = _levels_struct(levels, B)
    need = int(_ffi.lib().skv_cascade_multilevel_workspace_size(
        len(levels), ctypes.cast(arr, ctypes.c_void_p), B, Hq, Hkv, D, 0))
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    _need(workspace, "workspace")
    ws_bytes = workspace.numel() * workspace.element_size()
    _ffi.check("skv_cascade_decode_multilevel", _ffi.lib().skv_cascade_decode_multilevel(
        q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), P, len(levels),
        ctypes.cast(arr, ctypes.c_void_p), block_table.data_ptr(), block_table.shape[1],
        ctx.data_ptr(), B, Hq, Hkv, D, page, num_splits, float(sm_scale), _DT[q.dtype],
        o_pre.data_ptr(), s_pre.data_ptr(), o_part.data_ptr(), lse_part.data_ptr(),
        out.data_ptr(), lse_out.data_ptr(), workspace.data_ptr(), ws_bytes, _stream(q)))
    del keep
    return out, lse_out, o_pre, s_pre, o_part, lse_part


def get_device_error():
    """(code, detail) of the first device-side error since the last call; clears it."""
    code, detail = ctypes.c_int32(), ctypes.c_int32()
    _ffi.check("skv_get_device_error", _ffi.lib().skv_get_device_error(
        ctypes.byref(code), ctypes.byref(detail)))
    return code.value, detail.value


def poll_device_error(stream=None):
    """As get_device_error, waiting only for the work queued on `stream`
    (default: the current stream)."""
    if stream is None:
        stream = torch.cuda.current_stream()
    code, detail = ctypes.c_int32(), ctypes.c_int32()
    _ffi.check("skv_poll_device_error", _ffi.lib().skv_poll_device_error(
        ctypes.byref(code), ctypes.byref(detail), stream.cuda_stream))
    return code.value, detail.value


def selftest_bounded_wait(mode: int, limit_ns: int, stream=None):
    """Runs the library's bounded barrier waits on barriers nothing completes
    (see skv_selftest_bounded_wait); the outcome is read from the error word."""
    if stream is None:
        stream = torch.cuda.current_stream()
    _ffi.check("skv_selftest_bounded_wait", _ffi.lib().skv_selftest_bounded_wait(
        int(mode), int(limit_ns), stream.cuda_stream))
