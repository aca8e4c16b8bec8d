"""fp64 CPU oracle for split-KV decode and attention-state merging.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product path
(``split_kv_lse_gb300``) never imports, loads or calls it, and the two share no
code: they meet only through the seeded arrays of ``split_kv_lse_gb300.workloads``.

The arithmetic lives in ``oracle.c`` (plain C, double precision, one thread);
this module compiles it with gcc and marshals numpy arrays to it.  Every
function widens its inputs to float64 before the call.

Pages followed (cited by title and section):
  [F2] "F2 讲解：merge_state，以 2 为底的 LSE 合并"
  [L3] "L3 讲解：split-KV decode 与 LSE 合并"
  [FA] "FlashAttention 的空行 LSE:FA-2 的 +inf 约定与后来的变化"
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_default = None

_dp = ctypes.POINTER(ctypes.c_double)
_ip = ctypes.POINTER(ctypes.c_int32)
_i64 = ctypes.c_int64
_i32 = ctypes.c_int32

GCC_FLAGS = ["-std=c11", "-O2", "-fPIC", "-shared", "-fno-fast-math", "-ffp-contract=off"]


def compile_c(src: str, out: str) -> str:
    """Compile one oracle C source into a shared library at ``out``."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *GCC_FLAGS, "-o", tmp, src, "-lm"], check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile oracle.c (gcc -O2, no fast-math, no FMA contraction)."""
    stale = (not os.path.exists(_LIB_PATH)) or (
        os.path.getmtime(_LIB_PATH) < os.path.getmtime(SOURCE))
    if force or stale:
        compile_c(SOURCE, _LIB_PATH)
    return _LIB_PATH


def _f64(a) -> np.ndarray:
    if hasattr(a, "detach"):  # a torch CPU tensor
        a = a.detach().cpu().double().numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _i32a(a) -> np.ndarray:
    if hasattr(a, "detach"):
        a = a.detach().cpu().numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _p(a):
    return None if a is None else a.ctypes.data_as(_dp)


def _pi(a: np.ndarray):
    return a.ctypes.data_as(_ip)


class Oracle:
    """Bindings to one compiled copy of the oracle library."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        lib.oracle_merge_state.argtypes = [_i64, _i64, _dp, _dp, _dp, _dp, _dp, _dp]
        lib.oracle_merge_state.restype = None
        lib.oracle_merge_states.argtypes = [_i64, _i64, _i64, _i64, _dp, _dp, _dp, _dp, _dp]
        lib.oracle_merge_states.restype = None
        lib.oracle_split_range.argtypes = [_i32, _i32, _i32, _i32, _ip, _ip]
        lib.oracle_split_range.restype = None
        lib.oracle_plan.argtypes = [_i32, _ip, _i32, _i32, _i32]
        lib.oracle_plan.restype = _i32
        common = [_i32, _i32, _i32, _i32, _i32, _dp, _dp, _dp]
        lib.oracle_attend_full.argtypes = common + [_ip, _i32, _ip, ctypes.c_double, _dp, _dp]
        lib.oracle_attend_full.restype = None
        lib.oracle_attend_splits.argtypes = common + [_ip, _i32, _ip, ctypes.c_double, _i32,
                                                      _dp, _dp]
        lib.oracle_attend_splits.restype = None
        lib.oracle_plan_varlen.argtypes = [_i32, _ip, _i32, _i32, _i32, _ip]
        lib.oracle_plan_varlen.restype = None
        lib.oracle_attend_splits_varlen.argtypes = common + [_ip, _i32, _ip, ctypes.c_double,
                                                             _ip, _i32, _dp, _dp]
        lib.oracle_attend_splits_varlen.restype = None
        lib.oracle_cascade.argtypes = common + [_ip, _i32, _ip, _i32, _ip, ctypes.c_double,
                                                _dp, _dp, _dp, _dp]
        lib.oracle_cascade.restype = None
        lib.oracle_cascade_multilevel.argtypes = common + [
            _i32, _ip, ctypes.POINTER(ctypes.c_int64), _ip, _ip, _i32, _ip, ctypes.c_double,
            _dp, _dp, _dp, _dp]
        lib.oracle_cascade_multilevel.restype = None
        self.lib = lib
        self.path = path

    def merge_state(self, v_a, s_a, v_b, s_b):
        """Two-state merge ([F2] §③, §⑤; [FA] §2.2).  v [..., D], s [...] -> (v, s)."""
        va, vb = _f64(v_a), _f64(v_b)
        sa, sb = _f64(s_a), _f64(s_b)
        D = va.shape[-1]
        R = int(np.prod(va.shape[:-1], dtype=np.int64))
        assert vb.shape == va.shape and sa.shape == va.shape[:-1] and sb.shape == sa.shape
        v = np.empty_like(va)
        s = np.empty_like(sa)
        self.lib.oracle_merge_state(R, D, _p(va), _p(sa), _p(vb), _p(sb), _p(v), _p(s))
        return v, s

    def merge_states(self, v, s, return_weights: bool = False):
        """N-state merge in the [S, N, H, D] / [S, N, H] layout ([F2] §④)."""
        v, s = _f64(v), _f64(s)
        S, N, H, D = v.shape
        assert s.shape == (S, N, H)
        vo = np.empty((S, H, D))
        so = np.empty((S, H))
        w = np.empty((S, N, H)) if return_weights else None
        self.lib.oracle_merge_states(S, N, H, D, _p(v), _p(s), _p(vo), _p(so), _p(w))
        return (vo, so, w) if return_weights else (vo, so)

    def split_range(self, ctx: int, page: int, num_splits: int, split: int):
        """Raw [p_start, p_end) page range of one split ([L3] §②)."""
        a = ctypes.c_int32()
        b = ctypes.c_int32()
        self.lib.oracle_split_range(ctx, page, num_splits, split, ctypes.byref(a),
                                    ctypes.byref(b))
        return a.value, b.value

    def plan(self, ctx, Hkv: int, page: int, sm_count: int) -> int:
        """Split count for one decode step ([L3] §⑥, constants as read)."""
        c = _i32a(ctx)
        return int(self.lib.oracle_plan(len(c), _pi(c), Hkv, page, sm_count))

    @staticmethod
    def _decode_args(q, k_cache, v_cache, block_table, ctx):
        q = _f64(q)
        kc, vc = _f64(k_cache), _f64(v_cache)
        bt = _i32a(block_table)
        cx = _i32a(ctx)
        B, Hq, D = q.shape
        P, Hkv, page, D2 = kc.shape
        assert D2 == D and vc.shape == kc.shape and bt.shape[0] == B and cx.shape == (B,)
        assert bt.ndim == 2
        return q, kc, vc, bt, cx, B, Hq, Hkv, D, page

    def attend_full(self, q, k_cache, v_cache, block_table, ctx, sm_scale: float):
        """Unsplit paged decode attention -> (out [B,Hq,D], s [B,Hq] base 2)."""
        q, kc, vc, bt, cx, B, Hq, Hkv, D, page = self._decode_args(
            q, k_cache, v_cache, block_table, ctx)
        out = np.empty((B, Hq, D))
        s = np.empty((B, Hq))
        self.lib.oracle_attend_full(B, Hq, Hkv, D, page, _p(q), _p(kc), _p(vc), _pi(bt),
                                    bt.shape[1], _pi(cx), float(sm_scale), _p(out), _p(s))
        return out, s

    def attend_splits(self, q, k_cache, v_cache, block_table, ctx, sm_scale: float,
                      num_splits: int):
        """Per-split partial states -> (o_part [B,Hq,NS,D], lse_part [B,Hq,NS] base 2)."""
        q, kc, vc, bt, cx, B, Hq, Hkv, D, page = self._decode_args(
            q, k_cache, v_cache, block_table, ctx)
        o = np.empty((B, Hq, num_splits, D))
        lse = np.empty((B, Hq, num_splits))
        self.lib.oracle_attend_splits(B, Hq, Hkv, D, page, _p(q), _p(kc), _p(vc), _pi(bt),
                                      bt.shape[1], _pi(cx), float(sm_scale), num_splits,
                                      _p(o), _p(lse))
        return o, lse

    def plan_varlen(self, ctx, page: int, max_splits: int, pages_per_split: int):
        """Split count of each sequence ([L3] §⑥, per-sequence reading) -> int32 [B]."""
        c = _i32a(ctx).reshape(-1)
        ns = np.zeros(c.size, dtype=np.int32)
        self.lib.oracle_plan_varlen(c.size, _pi(c), page, max_splits, pages_per_split, _pi(ns))
        return ns

    def attend_splits_varlen(self, q, k_cache, v_cache, block_table, ctx, sm_scale: float,
                             num_splits, max_splits: int):
        """Per-split states with num_splits[b] splits for sequence b ->
        (o_part [B,Hq,max_splits,D], lse_part [B,Hq,max_splits]); entries past a
        sequence's count are empty states."""
        q, kc, vc, bt, cx, B, Hq, Hkv, D, page = self._decode_args(
            q, k_cache, v_cache, block_table, ctx)
        ns = _i32a(num_splits).reshape(-1)
        assert ns.size == B and np.all(ns >= 1) and np.all(ns <= max_splits)
        o = np.empty((B, Hq, max_splits, D))
        lse = np.empty((B, Hq, max_splits))
        self.lib.oracle_attend_splits_varlen(B, Hq, Hkv, D, page, _p(q), _p(kc), _p(vc),
                                             _pi(bt), bt.shape[1], _pi(cx), float(sm_scale),
                                             _pi(ns), max_splits, _p(o), _p(lse))
        return o, lse

    def cascade(self, q, k_cache, v_cache, prefix_pages, prefix_len: int, block_table, ctx,
                sm_scale: float):
        """Two-level cascade ([F2] §⑥) -> (out, s, o_pre, s_pre)."""
        q, kc, vc, bt, cx, B, Hq, Hkv, D, page = self._decode_args(
            q, k_cache, v_cache, block_table, ctx)
        pp = _i32a(prefix_pages).reshape(-1)
        if pp.size == 0:
            pp = np.zeros(1, dtype=np.int32)
        out = np.empty((B, Hq, D))
        s = np.empty((B, Hq))
        o_pre = np.empty((B, Hq, D))
        s_pre = np.empty((B, Hq))
        self.lib.oracle_cascade(B, Hq, Hkv, D, page, _p(q), _p(kc), _p(vc), _pi(pp),
                                int(prefix_len), _pi(bt), bt.shape[1], _pi(cx),
                                float(sm_scale), _p(out), _p(s), _p(o_pre), _p(s_pre))
        return out, s, o_pre, s_pre


    def cascade_multilevel(self, q, k_cache, v_cache, levels, block_table, ctx,
                           sm_scale: float):
        """Multi-level cascade ([F2] §⑥) -> (out, s, o_pre, s_pre).  levels[l] is a
        list of groups (r0, r1, pages, length): requests [r0, r1) share `length`
        tokens on the page list `pages` at level l."""
        q, kc, vc, bt, cx, B, Hq, Hkv, D, page = self._decode_args(
            q, k_cache, v_cache, block_table, ctx)
        L = len(levels)
        lens = np.zeros((B, max(L, 1)), dtype=np.int32)
        offs = np.zeros((B, max(L, 1)), dtype=np.int64)
        chunks = [np.zeros(1, dtype=np.int32)]
        at = 1
        for li, groups in enumerate(levels):
            for r0, r1, pages, length in groups:
                pg = _i32a(pages).reshape(-1) if pages is not None else np.zeros(0, np.int32)
                for b in range(int(r0), int(r1)):
                    lens[b, li] = int(length)
                    offs[b, li] = at
                chunks.append(pg)
                at += pg.size
        segp = np.ascontiguousarray(np.concatenate(chunks).astype(np.int32))
        out = np.empty((B, Hq, D))
        s = np.empty((B, Hq))
        o_pre = np.empty((B, Hq, D))
        s_pre = np.empty((B, Hq))
        self.lib.oracle_cascade_multilevel(
            B, Hq, Hkv, D, page, _p(q), _p(kc), _p(vc), L, _pi(segp),
            offs.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), _pi(lens), _pi(bt), bt.shape[1],
            _pi(cx), float(sm_scale), _p(out), _p(s), _p(o_pre), _p(s_pre))
        return out, s, o_pre, s_pre


def default() -> Oracle:
    """The oracle built from the committed oracle.c."""
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
    return _default


def merge_state(*a, **k):
    return default().merge_state(*a, **k)


def merge_states(*a, **k):
    return default().merge_states(*a, **k)


def split_range(*a, **k):
    return default().split_range(*a, **k)


def plan(*a, **k):
    return default().plan(*a, **k)


def attend_full(*a, **k):
    return default().attend_full(*a, **k)


def attend_splits(*a, **k):
    return default().attend_splits(*a, **k)


def plan_varlen(*a, **k):
    return default().plan_varlen(*a, **k)


def attend_splits_varlen(*a, **k):
    return default().attend_splits_varlen(*a, **k)


def cascade(*a, **k):
    return default().cascade(*a, **k)


def cascade_multilevel(*a, **k):
    return default().cascade_multilevel(*a, **k)
