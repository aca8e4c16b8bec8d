"""Comparison helpers for the GPU parity tests (CUDA path vs the fp64 oracle).

Tolerances (written here once, used by every parity test):
  merges, fp32 v      rtol 1e-5, atol 1e-6
  merges, fp16 v      atol 2e-3 + 2^-11 * |ref|   (2^-11: fp16 rounding of the output)
  merges, bf16 v      atol 8e-3 + 2^-8  * |ref|   (2^-8:  bf16 rounding of the output)
  merged s            atol 1e-5
  decode o, fp16 q/K/V (fp32 partials and the fp16 output)
                      atol 2e-3 (+ 2^-11 * |ref| on the fp16 output)
  decode o, bf16 q/K/V
                      atol 8e-3 + 2^-8 * |ref|: p enters P.V rounded to bf16
                      (relative 2^-9, so the error is at most 2^-9 times the
                      v values it weights) and the output is rounded to bf16
  decode lse (base 2) atol 1e-4 (the sums use the unrounded p)
  -inf must be -inf exactly; an empty state's v must be exactly 0; integer
  page ranges bit-exact.
"""
import math

import numpy as np
import pytest
import torch

V_TOL = {torch.float32: (1e-6, 1e-5), torch.float16: (2e-3, 2.0 ** -11),
         torch.bfloat16: (8e-3, 2.0 ** -8)}
S_ATOL = 1e-5
DEC_O_ATOL = 2e-3
DEC_LSE_ATOL = 1e-4
# (atol, rtol of the fp32 partials, rtol of the output) per q/K/V dtype.
DEC_O_TOL = {torch.float16: (2e-3, 0.0, 2.0 ** -11), torch.bfloat16: (8e-3, 2.0 ** -8, 2.0 ** -8)}


def skv():
    """The library binding, built on first use (fails loudly if it cannot build)."""
    import split_kv_lse_gb300 as m
    from split_kv_lse_gb300 import build
    build.build()
    return m


def require_gpu():
    if not torch.cuda.is_available():
        pytest.fail("a CUDA GPU is required for tests marked gpu")


def np64(t):
    return t.detach().cpu().double().numpy()


def assert_s_close(s_gpu, s_ref, atol, what="s"):
    s = np64(s_gpu) if isinstance(s_gpu, torch.Tensor) else np.asarray(s_gpu, np.float64)
    r = np.asarray(s_ref, np.float64)
    assert s.shape == r.shape, (s.shape, r.shape)
    ref_empty = r == -math.inf
    got_empty = s == -math.inf
    bad = np.nonzero(ref_empty != got_empty)
    assert bad[0].size == 0, f"{what}: -inf pattern differs at {tuple(i[:5] for i in bad)}"
    fin = ~ref_empty
    assert np.all(np.isfinite(s[fin])), f"{what}: non-finite where the oracle is finite"
    if fin.any():
        err = np.abs(s[fin] - r[fin]).max()
        assert err <= atol, f"{what}: max |err| {err:.3g} > {atol}"


def assert_v_close(v_gpu, v_ref, atol, rtol, what="v", empty_rows=None):
    v = np64(v_gpu) if isinstance(v_gpu, torch.Tensor) else np.asarray(v_gpu, np.float64)
    r = np.asarray(v_ref, np.float64)
    assert v.shape == r.shape, (v.shape, r.shape)
    assert np.all(np.isfinite(v)), f"{what}: non-finite values"
    err = np.abs(v - r)
    lim = atol + rtol * np.abs(r)
    worst = np.argmax(err - lim)
    assert np.all(err <= lim), (
        f"{what}: |err| {err.flat[worst]:.3g} > {lim.flat[worst]:.3g} at flat index {worst}")
    if empty_rows is not None:
        assert np.all(v[empty_rows] == 0.0), f"{what}: empty state with non-zero v"


def assert_states(v_gpu, s_gpu, v_ref, s_ref, dtype):
    atol, rtol = V_TOL[dtype]
    r = np.asarray(s_ref)
    assert_s_close(s_gpu, r, S_ATOL)
    assert_v_close(v_gpu, v_ref, atol, rtol, empty_rows=(r == -math.inf))
