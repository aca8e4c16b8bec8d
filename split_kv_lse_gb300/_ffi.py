"""ctypes declarations of the libskv C ABI (include/skv.h).

Loading fails loudly when the library has not been built: there is no
fallback implementation of any operation.
"""
from __future__ import annotations

import ctypes
import os
import threading

from .build import LIB

_lock = threading.Lock()
_lib = None

c_void_p = ctypes.c_void_p
c_float_p = ctypes.POINTER(ctypes.c_float)
c_int32_p = ctypes.POINTER(ctypes.c_int32)
i64 = ctypes.c_int64
i32 = ctypes.c_int32
f32 = ctypes.c_float
size_t = ctypes.c_size_t

STATUS = {0: "SKV_OK", 1: "SKV_ERR_INVALID_ARG", 2: "SKV_ERR_UNSUPPORTED", 3: "SKV_ERR_CUDA",
          4: "SKV_ERR_TIMEOUT"}

# name -> (restype, argtypes), exactly the declarations of include/skv.h
SIGNATURES = {
    "skv_status_string": (ctypes.c_char_p, [i32]),
    "skv_abi_version": (i32, []),
    "skv_merge_state": (i32, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                              i64, i64, i64, i32, c_void_p]),
    "skv_merge_state_in_place": (i32, [c_void_p, c_void_p, c_void_p, c_void_p, i64, i64, i64,
                                       i32, c_void_p]),
    "skv_merge_states_workspace_size": (size_t, [i64, i64, i64, i64]),
    "skv_merge_states": (i32, [c_void_p, c_void_p, c_void_p, c_void_p, i64, i64, i64, i64, i32,
                               c_void_p, size_t, c_void_p]),
    "skv_merge_states_noalloc": (i32, [c_void_p, c_void_p, c_void_p, c_void_p, i64, i64, i64,
                                        i64, i32, c_void_p]),
    "skv_split_page_range": (i32, [i32, i32, i32, i32, c_int32_p, c_int32_p]),
    "skv_splitkv_decode_plan": (i32, [i32, c_int32_p, i32, i32, i32, c_int32_p]),
    "skv_splitkv_decode": (i32, [c_void_p, c_void_p, c_void_p, i32, c_void_p, i32, c_void_p,
                                 i32, i32, i32, i32, i32, i32, f32, i32, c_void_p, c_void_p,
                                 c_void_p, c_void_p, c_void_p, c_void_p]),
    "skv_splitkv_plan_varlen": (i32, [i32, c_int32_p, i32, i32, i32, c_int32_p, i64, c_int32_p,
                                      c_int32_p]),
    "skv_splitkv_decode_varlen": (i32, [c_void_p, c_void_p, c_void_p, i32, c_void_p, i32,
                                        c_void_p, i32, i32, i32, i32, i32, i32, c_void_p, i32,
                                        i32, f32, i32, c_void_p, c_void_p, c_void_p, c_void_p,
                                        c_void_p, c_void_p]),
    "skv_cascade_decode_varlen": (i32, [c_void_p, c_void_p, c_void_p, i32, c_void_p, i32,
                                        c_void_p, i32, c_void_p, i32, i32, i32, i32, i32, i32,
                                        c_void_p, i32, i32, f32, i32, c_void_p, c_void_p,
                                        c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                        size_t, c_void_p]),
    "skv_cascade_workspace_size": (size_t, [i32, i32, i32, i32, i32, i32]),
    "skv_cascade_decode": (i32, [c_void_p, c_void_p, c_void_p, i32, c_void_p, i32, c_void_p, i32,
                                 c_void_p, i32, i32, i32, i32, i32, i32, f32, i32, c_void_p,
                                 c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                 size_t, c_void_p]),
    "skv_cascade_multilevel_workspace_size": (size_t, [i32, c_void_p, i32, i32, i32, i32, i32]),
    "skv_cascade_decode_multilevel": (i32, [c_void_p, c_void_p, c_void_p, i32, i32, c_void_p,
                                            c_void_p, i32, c_void_p, i32, i32, i32, i32, i32, i32,
                                            f32, i32, c_void_p, c_void_p, c_void_p, c_void_p,
                                            c_void_p, c_void_p, c_void_p, size_t, c_void_p]),
    "skv_merge_states_noalloc_scratch_size": (size_t, [i64, i64, i64, i64, i32, i32]),
    "skv_get_device_error": (i32, [c_int32_p, c_int32_p]),
    "skv_poll_device_error": (i32, [c_int32_p, c_int32_p, c_void_p]),
    "skv_selftest_bounded_wait": (i32, [i32, i64, c_void_p]),
}


class CascadeLevel(ctypes.Structure):
    """skv_cascade_level: host arrays (group_start, group_len, group_pages)."""
    _fields_ = [("num_groups", i32), ("group_start", c_int32_p), ("group_len", c_int32_p),
                ("group_pages", ctypes.POINTER(c_void_p))]


class SkvError(RuntimeError):
    def __init__(self, fn: str, code: int):
        self.code = code
        super().__init__(f"{fn} returned {STATUS.get(code, code)}")


def lib():
    """The loaded libskv.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB):
                raise RuntimeError(
                    f"libskv.so is not built ({LIB}); run split_kv_lse_gb300.build.build() "
                    "or __graft_entry__.build() first")
            h = ctypes.CDLL(LIB)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(h, name)
                fn.restype = res
                fn.argtypes = args
            _lib = h
    return _lib


def check(fn: str, code: int) -> None:
    if code != 0:
        raise SkvError(fn, code)
