"""ctypes view of libdvl.so (the C ABI declared in include/dvl.h).

Loading fails loudly: there is no fallback path.  The library is built in
place by ``draft_vocab_lm_gb300.build`` (or ``__graft_entry__.build()``)."""
from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdvl.so")

DVL_BF16 = 0
DVL_NVFP4 = 1
DVL_FP8 = 2
DVL_MAX_M = 32
DVL_MAX_TOPK = 4
DVL_K_MULTIPLE = 64
DVL_MAX_K = 24576
DVL_HEAD_STATIC = 1

STATUS_NAMES = {
    0: "DVL_OK", 1: "DVL_ERR_INVALID_ARG", 2: "DVL_ERR_OUT_OF_RANGE",
    3: "DVL_ERR_UNSUPPORTED", 4: "DVL_ERR_WORKSPACE", 5: "DVL_ERR_CUDA",
    6: "DVL_ERR_TIMEOUT",
}

# every symbol include/dvl.h declares
EXPORTS = (
    "dvl_status_string", "dvl_version", "dvl_last_error", "dvl_workspace_bytes", "dvl_workspace_init",
    "dvl_workspace_status",
    "dvl_draft_argmax", "dvl_draft_topk", "dvl_draft_argmax_noalloc", "dvl_noalloc_status",
    "dvl_draft_plan",
    "dvl_score_ids",
    "dvl_trim_head", "dvl_learn_rows", "dvl_learn_missing", "dvl_quantize_head",
    "dvl_histogram",
    "dvl_build_ranks", "dvl_union_sorted",
)


class DvlHead(ctypes.Structure):
    _fields_ = [
        ("dtype", ctypes.c_int32),
        ("N", ctypes.c_int32),
        ("K", ctypes.c_int32),
        ("flags", ctypes.c_int32),
        ("V", ctypes.c_int64),
        ("id_base", ctypes.c_int64),
        ("w", ctypes.c_void_p),
        ("scales", ctypes.c_void_p),
        ("global_scale", ctypes.c_float),
        ("reserved2", ctypes.c_int32),
        ("d2t", ctypes.c_void_p),
    ]


class DvlError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: {STATUS_NAMES.get(status, status)}")


_lock = threading.Lock()
_lib = None


def lib():
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(LIB_PATH)
        p, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
        hp = ctypes.POINTER(DvlHead)
        L.dvl_status_string.argtypes = [ctypes.c_int]
        L.dvl_status_string.restype = ctypes.c_char_p
        L.dvl_version.argtypes = []
        L.dvl_version.restype = ctypes.c_int
        L.dvl_last_error.argtypes = []
        L.dvl_last_error.restype = ctypes.c_char_p
        L.dvl_workspace_bytes.argtypes = [i32, i32]
        L.dvl_workspace_bytes.restype = sz
        L.dvl_workspace_init.argtypes = [p, sz, p]
        L.dvl_workspace_status.argtypes = [p, p, p]
        L.dvl_draft_argmax.argtypes = [hp, p, i32, p, p, p, sz, p]
        L.dvl_draft_topk.argtypes = [hp, p, i32, i32, p, p, p, sz, p]
        L.dvl_draft_argmax_noalloc.argtypes = [hp, p, i32, p, p, p]
        L.dvl_noalloc_status.argtypes = [p, p]
        L.dvl_draft_plan.argtypes = [hp, i32, i32, p, p]
        L.dvl_score_ids.argtypes = [hp, p, i32, p, i32, p, p]
        L.dvl_trim_head.argtypes = [hp, p, i32, p, p, p, p, p]
        L.dvl_learn_rows.argtypes = [hp, p, i32, i32, p, p, p, p]
        L.dvl_learn_missing.argtypes = [hp, p, i32, p, p, i32, p, p, p, p, p, p]
        L.dvl_quantize_head.argtypes = [hp, i32, p, p, p, p, sz, p]
        L.dvl_histogram.argtypes = [p, i64, i64, p]
        L.dvl_build_ranks.argtypes = [p, i64, p, i32, i32, i32, p, p]
        L.dvl_union_sorted.argtypes = [p, i32, p, i32, p, p]
        for fn in ("dvl_workspace_init", "dvl_workspace_status", "dvl_draft_argmax", "dvl_draft_topk",
                   "dvl_draft_argmax_noalloc", "dvl_noalloc_status",
                   "dvl_draft_plan", "dvl_score_ids",
                   "dvl_trim_head", "dvl_learn_rows", "dvl_learn_missing", "dvl_quantize_head", "dvl_histogram", "dvl_build_ranks", "dvl_union_sorted"):
            getattr(L, fn).restype = ctypes.c_int
        _lib = L
        return L


def check(fn: str, status: int) -> None:
    if status != 0:
        err = DvlError(fn, status)
        if status == 5:
            err.args = (f"{err.args[0]} ({lib().dvl_last_error().decode()})",)
        raise err
