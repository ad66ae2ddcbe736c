"""GB300-native draft-head argmax: Python binding of libdvl.so.

The library computes, for M hidden rows of a speculative-decoding draft head,
the best token of logits = h . W^T over a bf16 or NVFP4 head -- the full
vocabulary or a frequency-ranked shortlist with its d2t map -- fused on the
device so no logit tensor is written (see include/dvl.h for the C ABI).

This module only marshals arguments: PyTorch provides device memory and the
current CUDA stream, and every step of the computation runs in the library's
CUDA kernels.  There is no CPU fallback; calls fail loudly if the library is
not built.

    head = Head(w, V=248_320, d2t=d2t)            # w: CUDA bf16 [N][K]
    ids, logits = draft_argmax(head, h)            # h: CUDA bf16 [M][K]
    ids, logits = draft_topk(head, h, k=4)
    logits = score_ids(head, h, cand)              # cand: CUDA int32 [M][c]
    w_trim, _, d2t, n_dup = trim_head(w_full, ranks)
"""
from __future__ import annotations

import ctypes

import numpy as np

from . import roofline
from ._native import (DVL_BF16, DVL_FP8, DVL_HEAD_STATIC, DVL_K_MULTIPLE, DVL_MAX_K, DVL_MAX_M,
                      DVL_MAX_TOPK, DVL_NVFP4, DvlError, DvlHead, check, lib)

__all__ = [
    "Head", "DvlError", "workspace_status", "draft_argmax", "draft_topk", "draft_plan", "score_ids", "trim_head",
    "learn_rows",
    "quantize_head",
    "Shortlist", "workspace_bytes",
    "make_workspace", "workspace_init", "histogram", "build_ranks", "union_sorted",
    "read_ranks_txt", "write_ranks_txt", "roofline", "version",
]


def _torch():
    import torch
    return torch


def _stream_handle(stream, device) -> int:
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


_raw_stream_fn = None


def _call_stream(stream, t) -> int:
    """The stream handle for a draft call on tensor t's device: the given
    stream, or the device's current one.  A short draft call takes about as
    long on the GPU as building a torch Stream object takes on the host, so
    the current stream is read as a raw handle when torch offers that."""
    global _raw_stream_fn
    if stream is None:
        if _raw_stream_fn is None:
            _raw_stream_fn = getattr(_torch()._C, "_cuda_getCurrentRawStream", False)
        if _raw_stream_fn:
            return int(_raw_stream_fn(t.get_device()))
    return _stream_handle(stream, t.device)


def version() -> int:
    return int(lib().dvl_version())


class Head:
    """A draft head resident on one CUDA device.

    w:        bf16 [N][K] (any 2-byte dtype holding bfloat16 bits); for
              NVFP4 uint8 codes [N][K/2] (two E2M1 per byte, low nibble = even
              k); for FP8 uint8 E4M3 codes [N][K] (with fmt="fp8").
    V:        full vocabulary size (ids lie in [0, V)); defaults to N.
    d2t:      int32 [N] full-vocabulary id of each row, or None (identity,
              shifted by id_base).
    scales:   NVFP4 only: uint8 E4M3 [N][K/16].
    global_scale: NVFP4 / FP8 tensor scale.
    fmt:      "bf16", "nvfp4" or "fp8"; by default NVFP4 when scales are
              given, else bf16.
    static:   promise that no work still pending on the stream writes w,
              scales or d2t when a call is enqueued (weights loaded earlier;
              not a head trim_head has just filled on the same stream).  The
              kernel may then start streaming the head while the preceding
              kernel on the stream finishes.
    """

    def __init__(self, w, *, V: int | None = None, d2t=None, scales=None,
                 global_scale: float = 1.0, id_base: int = 0, static: bool = False,
                 fmt: str | None = None):
        torch = _torch()
        if not w.is_cuda or w.dim() != 2 or not w.is_contiguous():
            raise ValueError("w must be a contiguous 2-D CUDA tensor")
        fmt = fmt or ("nvfp4" if scales is not None else "bf16")
        if fmt not in ("bf16", "nvfp4", "fp8"):
            raise ValueError("fmt must be bf16, nvfp4 or fp8")
        if (fmt == "nvfp4") != (scales is not None):
            raise ValueError("scales go with, and only with, an NVFP4 head")
        self.fmt = fmt
        if fmt == "fp8":
            if w.element_size() != 1:
                raise ValueError("FP8 codes must be a uint8 tensor")
            self.dtype = DVL_FP8
            self.K = w.shape[1]
        elif scales is not None:
            if w.element_size() != 1:
                raise ValueError("NVFP4 codes must be a uint8 tensor")
            self.dtype = DVL_NVFP4
            self.K = 2 * w.shape[1]
            if (not scales.is_cuda or not scales.is_contiguous()
                    or tuple(scales.shape) != (w.shape[0], self.K // 16)):
                raise ValueError("scales must be a contiguous CUDA uint8 [N][K/16] tensor")
        else:
            if w.element_size() != 2:
                raise ValueError("a bf16 head needs a 2-byte dtype")
            self.dtype = DVL_BF16
            self.K = w.shape[1]
        self.w = w
        self.scales = scales
        self.N = w.shape[0]
        self.V = int(V) if V is not None else self.N
        self.id_base = int(id_base)
        self.global_scale = float(global_scale)
        if d2t is not None:
            if (not d2t.is_cuda or d2t.dtype != torch.int32 or not d2t.is_contiguous()
                    or tuple(d2t.shape) != (self.N,)):
                raise ValueError("d2t must be a contiguous CUDA int32 [N] tensor")
        self.d2t = d2t
        self.static = bool(static)
        self.device = w.device
        self._struct = None
        self._on_enqueue = None  # called after a draft call with this head is enqueued

    def struct(self) -> DvlHead:
        if self._struct is None:
            self._struct = self._make_struct()
        self._struct.flags = DVL_HEAD_STATIC if self.static else 0  # static may change
        return self._struct

    def _make_struct(self) -> DvlHead:
        s = DvlHead()
        s.dtype = self.dtype
        s.N = self.N
        s.K = self.K
        s.V = self.V
        s.id_base = self.id_base
        s.w = self.w.data_ptr()
        s.scales = self.scales.data_ptr() if self.scales is not None else None
        s.global_scale = self.global_scale
        s.d2t = self.d2t.data_ptr() if self.d2t is not None else None
        s.flags = DVL_HEAD_STATIC if self.static else 0
        return s

    def slice_rows(self, n0: int, n1: int) -> "Head":
        """Rows [n0, n1) as a head of their own (views, no copy); ids keep
        their full-vocabulary values."""
        h = Head.__new__(Head)
        h.__dict__.update(self.__dict__)
        h.w = self.w[n0:n1]
        h.scales = self.scales[n0:n1] if self.scales is not None else None
        h.d2t = self.d2t[n0:n1] if self.d2t is not None else None
        h.id_base = self.id_base + (n0 if self.d2t is None else 0)
        h.N = n1 - n0
        h._struct = None
        return h


def workspace_bytes(M: int, k: int = 1) -> int:
    return int(lib().dvl_workspace_bytes(int(M), int(k)))


def workspace_init(ws, stream=None) -> None:
    check("dvl_workspace_init",
          lib().dvl_workspace_init(ws.data_ptr(), ws.numel() * ws.element_size(),
                                   _stream_handle(stream, ws.device)))


def workspace_status(ws, stream=None) -> int:
    """Device-side failures recorded in `ws` since the last read, as a bitmask
    of 1 << status (DVL_ERR_TIMEOUT: a bounded device wait gave up and that
    call's results are not valid); reading synchronizes the stream and
    clears the word."""
    bits = ctypes.c_uint32(0)
    check("dvl_workspace_status",
          lib().dvl_workspace_status(ws.data_ptr(), ctypes.byref(bits),
                                     _stream_handle(stream, ws.device)))
    return int(bits.value)


def make_workspace(M: int = DVL_MAX_M, k: int = DVL_MAX_TOPK, device=None, stream=None):
    """A zeroed device workspace big enough for calls with up to M rows and k."""
    torch = _torch()
    n = workspace_bytes(M, k)
    if n == 0:
        raise ValueError("M or k outside the library's limits")
    ws = torch.empty(n, dtype=torch.uint8, device=device or "cuda")
    workspace_init(ws, stream)
    return ws


def _check_h(head: Head, h):
    if not h.is_cuda or h.dim() != 2 or not h.is_contiguous() or h.element_size() != 2:
        raise ValueError("h must be a contiguous 2-D CUDA bf16 tensor")
    if h.shape[1] != head.K:
        raise ValueError("h width must equal the head's K")


def draft_topk(head: Head, h, k: int, *, ids=None, logits=None, ws=None, stream=None):
    """Per hidden row: the k best (full id, logit), best first."""
    _check_h(head, h)
    M = h.shape[0]
    if ids is None:
        ids = _torch().empty((M, k), dtype=_torch().int32, device=h.device)
    if logits is None:
        logits = _torch().empty((M, k), dtype=_torch().float32, device=h.device)
    if ws is None:
        ws = make_workspace(M, k, device=h.device, stream=stream)
    check("dvl_draft_topk",
          lib().dvl_draft_topk(ctypes.byref(head.struct()), h.data_ptr(), M, int(k), ids.data_ptr(),
                               logits.data_ptr(), ws.data_ptr(), ws.numel(),
                               _call_stream(stream, h)))
    if head._on_enqueue is not None:
        head._on_enqueue()
    return ids, logits


def draft_argmax(head: Head, h, *, ids=None, logits=None, ws=None, stream=None):
    """Per hidden row: (full id, max logit) of the best head row."""
    _check_h(head, h)
    M = h.shape[0]
    if ids is None:
        ids = _torch().empty(M, dtype=_torch().int32, device=h.device)
    if logits is None:
        logits = _torch().empty(M, dtype=_torch().float32, device=h.device)
    if ws is None:
        ws = make_workspace(M, 1, device=h.device, stream=stream)
    check("dvl_draft_argmax",
          lib().dvl_draft_argmax(ctypes.byref(head.struct()), h.data_ptr(), M, ids.data_ptr(),
                                 logits.data_ptr(), ws.data_ptr(), ws.numel(),
                                 _call_stream(stream, h)))
    if head._on_enqueue is not None:
        head._on_enqueue()
    return ids, logits


def draft_plan(head: Head, M: int, k: int = 1):
    """(kernel family, launches) of a draft_argmax (k = 1) / draft_topk call
    with this head and M hidden rows on the current device; launches
    nothing."""
    name = ctypes.c_char_p()
    n = ctypes.c_int32()
    check("dvl_draft_plan", lib().dvl_draft_plan(ctypes.byref(head.struct()), int(M), int(k),
                                                 ctypes.byref(name), ctypes.byref(n)))
    return name.value.decode(), n.value


def score_ids(head: Head, h, ids, *, logits=None, stream=None):
    """Per hidden row m and candidate j: the logit of the head row that
    ids[m][j] names (ids id_base .. id_base + N - 1; NaN outside).  The head
    has no d2t; ids is a CUDA int32 [M][c] tensor."""
    torch = _torch()
    _check_h(head, h)
    M = h.shape[0]
    if (not ids.is_cuda or ids.dtype != torch.int32 or ids.dim() != 2
            or not ids.is_contiguous() or ids.shape[0] != M):
        raise ValueError("ids must be a contiguous CUDA int32 [M][c] tensor")
    c = ids.shape[1]
    if logits is None:
        logits = torch.empty((M, c), dtype=torch.float32, device=h.device)
    check("dvl_score_ids",
          lib().dvl_score_ids(ctypes.byref(head.struct()), h.data_ptr(), M, ids.data_ptr(), c,
                              logits.data_ptr(), _stream_handle(stream, h.device)))
    return logits


def trim_head(w_full, ranks, *, scales=None, fmt=None, stream=None):
    """Gather the rows `ranks` names (in its order) from a full head.

    w_full: CUDA bf16 [V][K], NVFP4 codes [V][K/2] (then `scales` [V][K/16])
            or FP8 codes [V][K] (fmt="fp8").
    ranks:  host ids (list, NumPy or CPU tensor).
    Returns (w_trim, scales_trim or None, d2t int32 CUDA [n], n_duplicates)."""
    torch = _torch()
    r = np.ascontiguousarray(np.asarray(ranks, dtype=np.int32))
    n = r.shape[0]
    full = Head(w_full, scales=scales, fmt=fmt)
    w_trim = torch.empty((n, w_full.shape[1]), dtype=w_full.dtype, device=w_full.device)
    s_trim = None
    if scales is not None:
        s_trim = torch.empty((n, scales.shape[1]), dtype=scales.dtype, device=scales.device)
    d2t = torch.empty(n, dtype=torch.int32, device=w_full.device)
    dup = ctypes.c_int32(0)
    st = full.struct()
    check("dvl_trim_head",
          lib().dvl_trim_head(ctypes.byref(st), r.ctypes.data, n, w_trim.data_ptr(),
                              s_trim.data_ptr() if s_trim is not None else None,
                              d2t.data_ptr(), ctypes.byref(dup),
                              _stream_handle(stream, w_full.device)))
    return w_trim, s_trim, d2t, int(dup.value)


def quantize_head(w, fmt: str = "nvfp4", *, ws=None, stream=None):
    """Requantize a bf16 head [N][K] (CUDA) to NVFP4 or FP8 on the device
    (dvl_quantize_head; synchronizes the stream once, to read the head's
    maximum back).  Returns (codes, scales or None, global_scale); pass them
    to Head(codes, scales=..., global_scale=..., fmt=fmt)."""
    torch = _torch()
    src = Head(w)
    N, K = src.N, src.K
    if fmt == "nvfp4":
        dtype, codes = DVL_NVFP4, torch.empty((N, K // 2), dtype=torch.uint8, device=w.device)
        scales = torch.empty((N, K // 16), dtype=torch.uint8, device=w.device)
    elif fmt == "fp8":
        dtype, codes, scales = DVL_FP8, torch.empty((N, K), dtype=torch.uint8, device=w.device), None
    else:
        raise ValueError("fmt must be nvfp4 or fp8")
    if ws is None:
        ws = make_workspace(1, 1, device=w.device, stream=stream)
    g = ctypes.c_float(0.0)
    check("dvl_quantize_head",
          lib().dvl_quantize_head(ctypes.byref(src.struct()), dtype, codes.data_ptr(),
                                  scales.data_ptr() if scales is not None else None,
                                  ctypes.byref(g), ws.data_ptr(), ws.numel(),
                                  _stream_handle(stream, w.device)))
    return codes, scales, float(g.value)


def learn_rows(w_full, ids, w_trim, d2t, row0: int, *, scales=None, scales_trim=None,
               fmt=None, stream=None) -> None:
    """Copy the full head's rows `ids` (host ids) into rows row0 .. row0 + n - 1
    of trimmed buffers and set their d2t entries (dvl_learn_rows).  The first
    call on the stream afterwards must not treat the trimmed head as static;
    Shortlist takes care of that."""
    r = np.ascontiguousarray(np.asarray(ids, dtype=np.int32))
    full = Head(w_full, scales=scales, fmt=fmt)
    check("dvl_learn_rows",
          lib().dvl_learn_rows(ctypes.byref(full.struct()), r.ctypes.data, r.shape[0], int(row0),
                               w_trim.data_ptr(),
                               scales_trim.data_ptr() if scales_trim is not None else None,
                               d2t.data_ptr(), _stream_handle(stream, w_full.device)))


class Shortlist:
    """A trimmed head with spare rows that learns escaped ids while serving.

    ("Masked MTP drafts", section "Update (November 2026)": a static trim can
    miss; learning the escaped ids into spare head rows recovered the loss.)
    The head is trimmed to `ranks` into buffers of `capacity` rows; learn()
    hands the emitted ids to dvl_learn_missing, which appends the full
    head's rows of the ids the list does not hold yet, in stream order,
    until the spare rows run out.

        sl = Shortlist(w_full, ranks, capacity=len(ranks) + 1024)
        ids, logits = draft_argmax(sl.head(), h)
        sl.learn(emitted_ids)        # host ids the target produced
    """

    def __init__(self, w_full, ranks, capacity: int, *, scales=None, global_scale: float = 1.0,
                 fmt=None, stream=None):
        torch = _torch()
        r = np.ascontiguousarray(np.asarray(ranks, dtype=np.int32))
        if capacity < r.shape[0]:
            raise ValueError("capacity below the number of ranks")
        self.V = w_full.shape[0]
        self.capacity = int(capacity)
        self.w_full, self.scales_full = w_full, scales
        self.fmt = fmt or ("nvfp4" if scales is not None else "bf16")
        self.global_scale = float(global_scale)
        self.stream = stream
        self.w = torch.empty((capacity, w_full.shape[1]), dtype=w_full.dtype, device=w_full.device)
        self.scales = None
        if scales is not None:
            self.scales = torch.empty((capacity, scales.shape[1]), dtype=scales.dtype,
                                      device=scales.device)
        self.d2t = torch.empty(capacity, dtype=torch.int32, device=w_full.device)
        # full id -> trimmed row (-1: not in the list), the table the C call keeps
        self.row_of = np.full(self.V, -1, dtype=np.int32)
        learn_rows(self.w_full, r, self.w, self.d2t, 0, scales=self.scales_full,
                   scales_trim=self.scales, fmt=self.fmt, stream=self.stream)
        # a padded list may repeat ids: each maps to its first row
        first = np.unique(r, return_index=True)
        self.row_of[first[0]] = first[1].astype(np.int32)
        self.n = int(r.shape[0])
        self._pending = True  # rows written by kernels that may still run

    def learn(self, ids) -> np.ndarray:
        """Learn the ids (host, any order, repeats allowed) the list does not
        hold, as many as spare rows remain; returns the ids learned."""
        x = np.asarray(ids, dtype=np.int64).ravel()
        if x.size and (x.min() < 0 or x.max() >= self.V):
            raise ValueError("ids outside the vocabulary")
        x = np.ascontiguousarray(x.astype(np.int32))
        learned = np.empty(max(1, x.size), dtype=np.int32)
        n_rows = ctypes.c_int32(self.n)
        n_learned = ctypes.c_int32(0)
        full = Head(self.w_full, scales=self.scales_full, fmt=self.fmt)
        check("dvl_learn_missing",
              lib().dvl_learn_missing(ctypes.byref(full.struct()),
                                      x.ctypes.data if x.size else None, x.size,
                                      self.row_of.ctypes.data, ctypes.byref(n_rows),
                                      self.capacity, self.w.data_ptr(),
                                      self.scales.data_ptr() if self.scales is not None else None,
                                      self.d2t.data_ptr(), learned.ctypes.data,
                                      ctypes.byref(n_learned),
                                      _stream_handle(self.stream, self.w_full.device)))
        self.n = int(n_rows.value)
        if n_learned.value:
            self._pending = True
        return learned[:n_learned.value].copy()

    def _enqueued(self) -> None:
        # a draft call that waits for the stream's preceding work has been
        # enqueued after the last learn: later calls may stream the head
        # before their wait
        self._pending = False

    def head(self, *, static: bool = True) -> Head:
        """The active rows as a Head.  Heads handed out between a learn and
        the first draft call enqueued after it are not static (the rows were
        written by the stream's latest kernels); later ones are, unless
        static=False."""
        hd = Head(self.w[:self.n], V=self.V, d2t=self.d2t[:self.n],
                  scales=self.scales[:self.n] if self.scales is not None else None,
                  global_scale=self.global_scale, static=static and not self._pending,
                  fmt=self.fmt)
        if self._pending:
            hd._on_enqueue = self._enqueued
        return hd


# ---------------------------------------------------------------------------
# Host-only ranks builder
# ---------------------------------------------------------------------------

def histogram(tokens, V: int, counts: np.ndarray | None = None) -> np.ndarray:
    t = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
    if counts is None:
        counts = np.zeros(V, dtype=np.int64)
    assert counts.dtype == np.int64 and counts.flags["C_CONTIGUOUS"] and counts.shape == (V,)
    check("dvl_histogram", lib().dvl_histogram(t.ctypes.data, t.shape[0], V, counts.ctypes.data))
    return counts


def build_ranks(counts: np.ndarray, N: int, forced=None, sorted_ids: bool = False) -> np.ndarray:
    c = np.ascontiguousarray(counts, dtype=np.int64)
    f = np.ascontiguousarray(np.asarray([] if forced is None else forced, dtype=np.int32))
    out = np.empty(max(1, min(N, c.shape[0])), dtype=np.int32)
    n = ctypes.c_int32(0)
    check("dvl_build_ranks",
          lib().dvl_build_ranks(c.ctypes.data, c.shape[0], f.ctypes.data if f.size else None,
                                f.shape[0], int(N), 1 if sorted_ids else 0, out.ctypes.data,
                                ctypes.byref(n)))
    return out[:n.value].copy()


def union_sorted(a, b) -> np.ndarray:
    a = np.ascontiguousarray(np.asarray(a, dtype=np.int32))
    b = np.ascontiguousarray(np.asarray(b, dtype=np.int32))
    out = np.empty(max(1, a.shape[0] + b.shape[0]), dtype=np.int32)
    n = ctypes.c_int32(0)
    check("dvl_union_sorted",
          lib().dvl_union_sorted(a.ctypes.data if a.size else None, a.shape[0],
                                 b.ctypes.data if b.size else None, b.shape[0],
                                 out.ctypes.data, ctypes.byref(n)))
    return out[:n.value].copy()


def read_ranks_txt(path: str) -> np.ndarray:
    """A ranks list: one decimal id per line (blank lines ignored)."""
    with open(path) as f:
        return np.array([int(x) for x in f if x.strip()], dtype=np.int32)


def write_ranks_txt(path: str, ids) -> None:
    with open(path, "w") as f:
        f.writelines(f"{int(x)}\n" for x in ids)
