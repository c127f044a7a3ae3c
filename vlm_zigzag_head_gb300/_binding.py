"""ctypes binding of libcpattn.so: signatures of the C ABI in include/cpattn.h.

Loading fails loudly when the library has not been built: there is no
fallback implementation anywhere in the package.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import threading

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_lib", "libcpattn.so")
_CHECKED_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_lib",
                             "libcpattn_checked.so")
_lock = threading.Lock()
_lib = None
_checked = None
_use_checked = False

c_i32p = ctypes.POINTER(ctypes.c_int32)
c_i64p = ctypes.POINTER(ctypes.c_int64)
c_vp = ctypes.c_void_p

STATUS = {0: "CP_OK", 1: "CP_ERR_INVALID_ARG", 2: "CP_ERR_SHAPE", 3: "CP_ERR_DTYPE",
          4: "CP_ERR_ALIGNMENT", 5: "CP_ERR_WORKSPACE", 6: "CP_ERR_CUDA", 7: "CP_ERR_TIMEOUT",
          8: "CP_ERR_UNSUPPORTED", 9: "CP_ERR_BOUNDS"}
CP_F32, CP_BF16 = 0, 1

# name -> (restype, argtypes)
SIGNATURES = {
    "cp_last_error": (ctypes.c_char_p, []),
    "cp_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "cp_version": (ctypes.c_int, []),
    "cp_zigzag_index": (ctypes.c_int, [c_i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int, c_vp,
                                       c_vp, ctypes.c_int, c_vp]),
    "cp_zigzag_gather": (ctypes.c_int, [c_vp, c_vp, ctypes.c_size_t, c_vp, ctypes.c_int, c_vp]),
    "cp_zigzag_scatter": (ctypes.c_int, [c_vp, c_vp, ctypes.c_size_t, c_vp, ctypes.c_int, c_vp]),
    "cp_copy_rows": (ctypes.c_int, [c_vp, ctypes.c_size_t, c_vp, ctypes.c_size_t, ctypes.c_size_t,
                                    ctypes.c_size_t, c_vp]),
    "cp_attn_fwd_workspace_size": (ctypes.c_size_t, [ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                     ctypes.c_int, c_i32p, ctypes.c_int,
                                                     ctypes.c_int, ctypes.c_int, ctypes.c_float]),
    "cp_attn_fwd": (ctypes.c_int, [c_vp, c_vp, c_vp, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                   ctypes.c_int, c_i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                   ctypes.c_float, c_vp, c_vp, c_vp, c_vp, ctypes.c_size_t,
                                   c_vp]),
    "cp_attn_fwd_noalloc": (ctypes.c_int, [c_vp, c_vp, c_vp, ctypes.c_int, ctypes.c_int,
                                           ctypes.c_int, ctypes.c_int, c_i32p, ctypes.c_int,
                                           ctypes.c_int, ctypes.c_int, ctypes.c_float, c_vp, c_vp,
                                           c_vp, c_vp]),
    "cp_attn_fwd_workspace_size_gqa": (ctypes.c_size_t, [ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                         ctypes.c_int, ctypes.c_int, c_i32p,
                                                         ctypes.c_int, ctypes.c_int,
                                                         ctypes.c_int, ctypes.c_float]),
    "cp_attn_fwd_gqa": (ctypes.c_int, [c_vp, c_vp, c_vp, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                       ctypes.c_int, ctypes.c_int, c_i32p, ctypes.c_int,
                                       ctypes.c_int, ctypes.c_int, ctypes.c_float, c_vp, c_vp,
                                       c_vp, c_vp, ctypes.c_size_t, c_vp]),
    "cp_attn_bwd_workspace_size_gqa": (ctypes.c_size_t, [ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                         ctypes.c_int, ctypes.c_int, c_i32p,
                                                         ctypes.c_int, ctypes.c_int,
                                                         ctypes.c_int, ctypes.c_float]),
    "cp_attn_bwd_gqa": (ctypes.c_int, [c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, ctypes.c_int,
                                       ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                       c_i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                       ctypes.c_float, c_vp, c_vp, c_vp, c_vp, c_vp,
                                       ctypes.c_size_t, c_vp]),
    "cp_lse_merge": (ctypes.c_int, [ctypes.c_int, c_vp, c_vp, ctypes.c_int, ctypes.c_int,
                                    ctypes.c_int, c_vp, ctypes.c_int, c_vp, c_vp]),
    "cp_attn_bwd_workspace_size": (ctypes.c_size_t, [ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                     ctypes.c_int, c_i32p, ctypes.c_int,
                                                     ctypes.c_int, ctypes.c_int, ctypes.c_float]),
    "cp_attn_bwd": (ctypes.c_int, [c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, ctypes.c_int,
                                   ctypes.c_int,
                                   ctypes.c_int, ctypes.c_int, c_i32p, ctypes.c_int, ctypes.c_int,
                                   ctypes.c_int, ctypes.c_float, c_vp, c_vp, c_vp, c_vp, c_vp,
                                   ctypes.c_size_t, c_vp]),
    "cp_workspace_status": (ctypes.c_int, [c_vp, c_vp]),
    "cp_plan_pairs": (ctypes.c_int, [c_i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int, c_i64p,
                                     c_i64p, c_i64p, c_i64p]),
    "cp_plan_unit_lists": (ctypes.c_int, [c_i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                          ctypes.c_int, ctypes.c_int, c_i64p, c_i32p, c_i32p,
                                          c_i32p]),
    "cp_set_wait_limit": (None, [ctypes.c_longlong]),
    "cp_profile_begin": (None, []),
    "cp_profile_end": (ctypes.c_int, [ctypes.POINTER(ctypes.c_double), c_i64p]),
}


class CpError(RuntimeError):
    def __init__(self, status, message):
        self.status = status
        super().__init__("%s: %s" % (STATUS.get(status, status), message))


def lib_path() -> str:
    return _LIB_PATH


def _load(path, how):
    if not os.path.exists(path):
        raise RuntimeError("%s is not built; run %s" % (path, how))
    L = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    return L


def lib():
    """The loaded library (raises if it was never built).  Inside
    ``bounds_checked()`` this is the bounds-checked debug build."""
    global _lib, _checked
    if _use_checked:
        if _checked is None:
            with _lock:
                if _checked is None:
                    _checked = _load(_CHECKED_PATH, "`python vlm_zigzag_head_gb300/build.py "
                                     "--checked`")
        return _checked
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            _lib = _load(_LIB_PATH, "`python -c 'import __graft_entry__ as g; g.build()'`")
    return _lib


@contextlib.contextmanager
def bounds_checked():
    """Route every call of the package, from any thread, through
    libcpattn_checked.so while the block runs: the same kernels with each row
    and head index tested before a TMA load, TMA reduce or global store (a
    failure is skipped and reported as CP_ERR_BOUNDS by cp_workspace_status).
    A debugging aid: the two libraries keep separate plan caches, wait limits
    and fixed scratch."""
    global _use_checked
    prev = _use_checked
    _use_checked = True
    try:
        yield lib()
    finally:
        _use_checked = prev


def check(status: int):
    if status != 0:
        raise CpError(status, lib().cp_last_error().decode(errors="replace"))


def cu_array(cu_seqlens):
    arr = (ctypes.c_int32 * len(cu_seqlens))(*[int(x) for x in cu_seqlens])
    return arr
