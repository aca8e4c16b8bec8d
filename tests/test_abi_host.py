"""The C-ABI library on the CPU: it builds, loads without a GPU, exports every
entry point include/skv.h declares, and its host logic (split page ranges, the
split-count plan, argument checks) is bit-exact against the oracle and the
pages' printed values.  No compute call is made here."""
import ctypes
import os
import re

import pytest

from conftest import ROOT, read_golden_table

HEADER = os.path.join(ROOT, "include", "skv.h")


@pytest.fixture(scope="session")
def lib():
    from split_kv_lse_gb300 import _ffi, build
    build.build()
    return _ffi.lib()


def declared_symbols():
    text = open(HEADER, encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(skv_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_symbols()
    for n in ("skv_merge_state", "skv_merge_state_in_place", "skv_merge_states",
              "skv_merge_states_workspace_size", "skv_split_page_range",
              "skv_splitkv_decode_plan", "skv_splitkv_decode", "skv_get_device_error"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    from split_kv_lse_gb300 import _ffi
    for name in declared_symbols():
        assert hasattr(lib, name), f"{name} declared in skv.h but not exported"
        assert name in _ffi.SIGNATURES, f"{name} has no ctypes declaration"


def test_status_strings_and_version(lib):
    assert lib.skv_abi_version() == 2
    for code, name in ((0, b"SKV_OK"), (1, b"SKV_ERR_INVALID_ARG"), (2, b"SKV_ERR_UNSUPPORTED"),
                       (3, b"SKV_ERR_CUDA"), (4, b"SKV_ERR_TIMEOUT")):
        assert lib.skv_status_string(code) == name


def _range(lib, ctx, page, ns, split):
    a, b = ctypes.c_int32(), ctypes.c_int32()
    st = lib.skv_split_page_range(ctx, page, ns, split, ctypes.byref(a), ctypes.byref(b))
    return st, a.value, b.value


def test_split_ranges_printed(lib):
    """L3 讲解 §② and §⑧ 自测 1: the printed ranges, bit-exact."""
    for ctx, page, ns, _, _, split, p0, p1, _ in read_golden_table("split_ranges.txt"):
        assert _range(lib, ctx, page, ns, split) == (0, p0, p1)


def test_split_ranges_match_oracle(lib, orc):
    import numpy as np
    rng = np.random.default_rng(0)
    cases = [(c, 16, ns) for c in (0, 1, 15, 16, 17, 37, 100, 255, 256, 257, 1000, 32768)
             for ns in (1, 2, 3, 4, 7, 16, 64, 256)]
    cases += [(int(rng.integers(0, 100000)), int(rng.integers(1, 64)), int(rng.integers(1, 300)))
              for _ in range(300)]
    for ctx, page, ns in cases:
        for split in range(ns):
            st, a, b = _range(lib, ctx, page, ns, split)
            assert st == 0 and (a, b) == orc.split_range(ctx, page, ns, split), (ctx, page, ns, split)


def test_split_range_argument_checks(lib):
    assert _range(lib, -1, 16, 4, 0)[0] == 1
    assert _range(lib, 10, 0, 4, 0)[0] == 1
    assert _range(lib, 10, 16, 0, 0)[0] == 1
    assert _range(lib, 10, 16, 4, 4)[0] == 1
    assert lib.skv_split_page_range(10, 16, 4, 0, None, None) == 1


def _plan(lib, ctx, Hkv, page, sm):
    arr = (ctypes.c_int32 * max(1, len(ctx)))(*ctx)
    ns = ctypes.c_int32(-1)
    st = lib.skv_splitkv_decode_plan(len(ctx), arr, Hkv, page, sm, ctypes.byref(ns))
    return st, ns.value


def test_plan_printed_table(lib):
    """L3 讲解 §⑥: the suitable split counts of the page's table (170 SMs)."""
    for B, ctx, Hkv, page, sm, want in read_golden_table("plan_table.txt"):
        assert _plan(lib, [ctx] * B, Hkv, page, sm) == (0, want)


def test_plan_matches_oracle(lib, orc):
    import numpy as np
    rng = np.random.default_rng(1)
    for _ in range(500):
        B = int(rng.integers(1, 80))
        ctx = [int(x) for x in rng.integers(0, 40000, B)]
        Hkv = int(rng.choice([1, 2, 4, 8, 16]))
        sm = int(rng.choice([1, 16, 132, 148, 152, 170]))
        assert _plan(lib, ctx, Hkv, 16, sm) == (0, orc.plan(ctx, Hkv, 16, sm))
    # GB300 (152 SMs) on the long-context decode workload: 64 splits.
    assert _plan(lib, [32768], 8, 16, 152) == (0, 64)


def test_plan_argument_checks(lib):
    assert _plan(lib, [10], 0, 16, 152)[0] == 1
    assert _plan(lib, [-5], 8, 16, 152)[0] == 1
    assert _plan(lib, [10], 8, 0, 152)[0] == 1


def test_device_entry_points_reject_bad_arguments_before_any_cuda_call(lib):
    """Checks that fail on the host return before the library touches CUDA.

    Every call below breaks at least one host-side check, so none of them can
    reach a kernel launch even on a machine with a GPU (the pointers are fake).
    """
    fake = ctypes.c_void_p(0x10000)      # 16-byte aligned, never dereferenced
    odd = ctypes.c_void_p(0x10004)       # not 16-byte aligned
    F32, F16 = 0, 1
    ms = lib.skv_merge_state
    assert ms(None, fake, fake, fake, fake, fake, 4, 2, 64, F32, None) == 1
    assert ms(fake, fake, fake, fake, fake, fake, -1, 2, 64, F32, None) == 1
    assert ms(fake, fake, fake, fake, fake, fake, 4, 2, 3, F32, None) == 1      # 12 bytes/row
    assert ms(fake, fake, fake, fake, fake, fake, 4, 2, 256, F32, None) == 2    # 1 KB rows
    assert ms(odd, fake, fake, fake, fake, fake, 4, 2, 64, F32, None) == 1
    assert ms(fake, fake, fake, fake, fake, fake, 4, 2, 64, 7, None) == 1       # bad dtype
    assert ms(None, None, None, None, None, None, 0, 2, 64, F16, None) == 0     # empty: no-op
    ip = lib.skv_merge_state_in_place
    assert ip(None, fake, fake, fake, 4, 2, 64, F32, None) == 1
    mss = lib.skv_merge_states
    assert mss(fake, fake, fake, fake, 4, 0, 2, 64, F32, None, 0, None) == 1    # N = 0
    assert mss(None, fake, fake, fake, 4, 3, 2, 64, F32, None, 0, None) == 1
    assert mss(fake, fake, fake, fake, 4, 3, 2, 64, F32, odd, 64, None) == 1
    dec = lib.skv_splitkv_decode

    def d(**kw):
        a = dict(q=fake, k=fake, v=fake, P=4, bt=fake, mp=4, ctx=fake, B=1, Hq=32, Hkv=8, D=128,
                 page=16, ns=4, scale=0.1, dt=F16, op=fake, lp=fake, out=None, lo=None, rd=None)
        a.update(kw)
        return dec(a["q"], a["k"], a["v"], a["P"], a["bt"], a["mp"], a["ctx"], a["B"], a["Hq"],
                   a["Hkv"], a["D"], a["page"], a["ns"], a["scale"], a["dt"], a["op"], a["lp"],
                   a["out"], a["lo"], a["rd"], None)
    assert d(B=0) == 0
    assert d(Hq=30) == 1          # Hq % Hkv
    assert d(D=64) == 2           # unsupported head size
    assert d(page=32) == 2        # unsupported page size
    assert d(Hq=8 * 16) == 2      # G = 16
    assert d(dt=F32) == 2
    assert d(ns=0) == 1
    assert d(ns=257) == 2
    assert d(q=None) == 1
    assert d(q=odd) == 1
    assert d(op=odd) == 1
    assert d(P=0) == 1
    assert d(lo=fake) == 1        # lse_out without out
    code = ctypes.c_int32()
    assert lib.skv_get_device_error(None, ctypes.byref(code)) == 1
    assert lib.skv_poll_device_error(None, ctypes.byref(code), None) == 1
    st = lib.skv_selftest_bounded_wait
    assert st(2, 1_000_000, None) == 1           # unknown mode
    assert st(0, 999, None) == 1                 # limit below 1 us
    assert st(1, 10_000_001, None) == 1          # limit above 10 ms


def test_merge_states_workspace_size(lib):
    f = lib.skv_merge_states_workspace_size
    assert f(256, 64, 32, 128) == 0          # many rows: one lane team per row, no workspace
    assert f(16, 1024, 8, 128) > 0           # few rows, many states: two-level merge
    assert f(16, 1024, 8, 128) >= 16 * 8 * 16 * 128 * 4
    assert f(0, 4, 4, 64) == 0 and f(4, 0, 4, 64) == 0


def _level(starts, lens):
    from split_kv_lse_gb300 import _ffi
    n = len(lens)
    s = (ctypes.c_int32 * (n + 1))(*starts)
    ln = (ctypes.c_int32 * n)(*lens)
    pg = (ctypes.c_void_p * n)(*[16 if x > 0 else None for x in lens])  # never dereferenced here
    lv = _ffi.CascadeLevel(n, ctypes.cast(s, ctypes.POINTER(ctypes.c_int32)),
                           ctypes.cast(ln, ctypes.POINTER(ctypes.c_int32)),
                           ctypes.cast(pg, ctypes.POINTER(ctypes.c_void_p)))
    return lv, (s, ln, pg)


def test_cascade_multilevel_workspace_size(lib):
    """One level of one group needs no more than the two-level cascade's size
    query gives (which also covers per-sequence suffix splits); more levels
    add their chunk-state slots; a level that does not cover 0..B in order is
    rejected (size 0)."""
    from split_kv_lse_gb300 import _ffi
    lv, keep = _level([0, 64], [8192])
    arr = (_ffi.CascadeLevel * 1)(lv)
    two = lib.skv_cascade_multilevel_workspace_size(1, arr, 64, 32, 8, 128, 152)
    assert 0 < two <= lib.skv_cascade_workspace_size(64, 32, 8, 128, 8192, 152)
    lv1, k1 = _level([0, 30, 64], [1000, 0])
    arr2 = (_ffi.CascadeLevel * 2)(lv, lv1)
    assert lib.skv_cascade_multilevel_workspace_size(2, arr2, 64, 32, 8, 128, 152) > two
    bad, kb = _level([0, 40, 30, 64], [5, 5, 5])     # decreasing boundary
    assert lib.skv_cascade_multilevel_workspace_size(1, (_ffi.CascadeLevel * 1)(bad), 64, 32, 8,
                                                     128, 152) == 0
    short, ks = _level([0, 60], [5])                 # does not reach B
    assert lib.skv_cascade_multilevel_workspace_size(1, (_ffi.CascadeLevel * 1)(short), 64, 32,
                                                     8, 128, 152) == 0
    # No shared level: the suffix alone, no slots.
    assert lib.skv_cascade_multilevel_workspace_size(0, None, 64, 32, 8, 128, 152) > 0


def test_product_path_never_imports_the_oracle():
    """The library package must not reference the oracle in any form."""
    pkg = os.path.join(ROOT, "split_kv_lse_gb300")
    for dirpath, _, files in os.walk(pkg):
        if "_build" in dirpath:
            continue
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f), encoding="utf-8").read()
                assert not re.search(r"\bimport\s+oracle\b|\bfrom\s+oracle\b|oracle\.c\b|liboracle",
                                     text), f


def test_cascade_prefix_sizing_on_the_cascade_workload(lib):
    """The shared-prefix pass is sized for about a fifth of the SMs (a quarter
    when the suffixes have per-sequence split counts) so that it runs beside
    the suffix pass: for B=64 requests sharing 8192 tokens (Hq=32, Hkv=8) on
    152 SMs that is 3 (4) prefix chunks x 8 kv heads = 24 (32) CTAs, i.e. 3
    (4) chunk-state slots per row in the workspace ([rows, slots, D] fp32
    states, [rows, slots] LSEs, then 256 bytes of counters); the size query
    covers both.  A one-level multi-level cascade takes the uniform sizing."""
    from split_kv_lse_gb300 import _ffi
    def align256(x):
        return (x + 255) // 256 * 256
    rows, D = 64 * 32, 128
    want = lambda slots: align256(rows * slots * D * 4) + align256(rows * slots * 4) + 256
    assert lib.skv_cascade_workspace_size(64, 32, 8, D, 8192, 152) == want(4)
    lv, keep = _level([0, 64], [8192])
    assert lib.skv_cascade_multilevel_workspace_size(1, (_ffi.CascadeLevel * 1)(lv), 64, 32, 8, D,
                                                     152) == want(3)
    # No prefix: no slots.
    assert lib.skv_cascade_workspace_size(64, 32, 8, D, 0, 152) == want(0)


def test_noalloc_scratch_fits_every_shape_on_gb300(lib):
    """skv_merge_states_noalloc keeps its two-level partials in a fixed 1 MiB
    array.  The heaviest shape is fp16 D=256 (1 KB fp32 partial rows) with
    S*H = 2*SM - 1 rows, just below the count at which every row gets one CTA:
    on a GB300 (152 SMs) it needs about 612 KB, which fits, and a few-row
    shape needs less.  On a GPU with 300 SMs the same kind of shape no longer
    fits, so there the call returns SKV_ERR_UNSUPPORTED."""
    cap = 1 << 20
    f = lib.skv_merge_states_noalloc_scratch_size
    F16 = 1
    sm = 152
    worst = max(f(rows, 1024, 1, 256, F16, sm) for rows in range(1, 2 * sm + 1))
    assert worst == f(2 * sm - 1, 1024, 1, 256, F16, sm)
    assert 600_000 < worst < cap
    assert f(2 * sm, 1024, 1, 256, F16, sm) == 0      # one CTA per row: no scratch
    assert f(16, 1024, 8, 128, 0, sm) > 0             # the large-N sweep shape (fp32, D=128)
    assert f(8, 1, 4, 128, 0, sm) == 0                # N = 1: one CTA per row
    big = 300
    assert f(2 * big - 1, 1024, 1, 256, F16, big) > cap
    assert f(0, 4, 4, 64, 0, sm) == 0 and f(4, 4, 4, 3, 0, sm) == 0   # invalid sizes


def _plan_varlen(ctx, page, max_splits, pps):
    import split_kv_lse_gb300 as m
    return m.splitkv_plan_varlen(ctx, page, max_splits, pps)


def test_plan_varlen_matches_oracle_and_lists_every_split(lib, orc):
    """skv_splitkv_plan_varlen: the split counts bit-exact against the
    oracle's per-sequence reading ([L3] §⑥); the work list holds every
    (sequence, split < ns_b) exactly once, longest splits first, each unit
    carrying its sequence's count; max_split_pages is the longest split."""
    import numpy as np
    rng = np.random.default_rng(5)
    cases = [([0, 1, 128, 129, 1000, 2048, 4096], 16, 16, 8), ([37], 16, 4, 1),
             ([0, 0], 16, 3, 2), ([32768], 16, 64, 8)]
    for _ in range(200):
        B = int(rng.integers(1, 70))
        cases.append(([int(x) for x in rng.integers(0, 5000, B)], 16,
                      int(rng.integers(1, 257)), int(rng.integers(1, 20))))
    for ctx, page, ms, pps in cases:
        plan = _plan_varlen(ctx, page, ms, pps)
        ns = plan.num_splits.numpy()
        assert np.array_equal(ns, orc.plan_varlen(ctx, page, ms, pps)), (ctx, ms, pps)
        assert plan.num_units == int(ns.sum())
        units = plan.host[:2 * plan.num_units].view(-1, 2).numpy()
        b, word = units[:, 0], units[:, 1]
        split, cnt = word & 0xFFFF, word >> 16
        assert np.array_equal(cnt, ns[b])
        assert sorted(zip(b.tolist(), split.tolist())) == [
            (i, s) for i in range(len(ctx)) for s in range(int(ns[i]))]
        pages = []
        for bi, sp in zip(b.tolist(), split.tolist()):
            a, e = orc.split_range(ctx[bi], page, int(ns[bi]), sp)
            pages.append(max(0, e - a))
        assert pages == sorted(pages, reverse=True)
        assert plan.max_split_pages == max(pages)


def test_plan_varlen_argument_checks(lib):
    f = lib.skv_splitkv_plan_varlen
    c = ctypes.c_int32
    ctx = (c * 2)(10, 20)
    buf = (c * 64)()
    nu, mp = c(), c()
    ok = f(2, ctx, 16, 4, 8, buf, 64, ctypes.byref(nu), ctypes.byref(mp))
    assert ok == 0 and nu.value == 2 and mp.value == 2
    assert f(2, ctx, 16, 0, 8, buf, 64, ctypes.byref(nu), ctypes.byref(mp)) == 1    # max_splits 0
    assert f(2, ctx, 16, 257, 8, buf, 64, ctypes.byref(nu), ctypes.byref(mp)) == 1  # > 256
    assert f(2, ctx, 16, 4, 0, buf, 64, ctypes.byref(nu), ctypes.byref(mp)) == 1    # pps 0
    assert f(2, ctx, 16, 4, 8, buf, 5, ctypes.byref(nu), ctypes.byref(mp)) == 1     # too small
    nu.value = mp.value = -1
    assert f(2, ctx, 16, 4, 8, None, 0, ctypes.byref(nu), ctypes.byref(mp)) == 0    # size query
    assert nu.value == 2 and mp.value == 2
    neg = (c * 2)(10, -1)
    assert f(2, neg, 16, 4, 8, buf, 64, ctypes.byref(nu), ctypes.byref(mp)) == 1
