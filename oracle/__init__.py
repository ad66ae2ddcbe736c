"""Plain CPU oracle for the draft-head argmax path (NumPy-facing wrapper).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, the smoke check in
``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may import this
package.  The product library (``draft_vocab_lm_gb300``) never imports it and
shares no code with it; the oracle is compiled from ``oracle.c`` with gcc,
independently of the CUDA build.

Every function states what it computes; ``oracle.c`` holds the definitions
and the passages of the pages they follow.  Pins that tie the oracle to
something other than itself live in ``tests/test_oracle_*.py``.

Parity pins, per function (all in ``tests/``):
  logits_bf16   exact integer brute force (matmul of small integers), one-hot
                and all-ones closed forms, the fp32 summation error bound
                against an fp64 dot, the shortlist masking invariant.
  topk/argmax   brute-force sort on tiny inputs, planted exact ties with a
                non-monotone d2t, NaN and signed-zero cases.
  e2m1/e4m3     hand-computed values from the format definitions
                (tests/golden/nvfp4_values.txt).
  logits_nvfp4  one-hot and all-ones closed forms built from those values.
  check_trim    planted byte and d2t corruptions.
  ranks builder the pages' printed counts (union 47,149 + 9,749 -> 52,755;
                16k composition), brute force against Python's sorted().
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

# -ffp-contract=off: every multiply and every add rounds separately, in the
# order written (no fused multiply-add), on x86-64 and on aarch64 alike.
CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
          "-shared", "-pthread"]


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (gcc) if it is missing or stale."""
    with _lock:
        stale = (not os.path.exists(_LIB_PATH)
                 or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)
                 or os.path.getmtime(_LIB_PATH) < os.path.getmtime(
                     os.path.join(_HERE, "oracle.h")))
        if force or stale:
            tmp = _LIB_PATH + f".tmp{os.getpid()}"
            subprocess.run(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"], check=True)
            os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build()
    lib = ctypes.CDLL(_LIB_PATH)
    p = ctypes.c_void_p
    i64 = ctypes.c_int64
    lib.oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
    lib.oracle_bf16_to_f32.restype = ctypes.c_float
    lib.oracle_e2m1.argtypes = [ctypes.c_uint8]
    lib.oracle_e2m1.restype = ctypes.c_float
    lib.oracle_e4m3.argtypes = [ctypes.c_uint8]
    lib.oracle_e4m3.restype = ctypes.c_float
    lib.oracle_nvfp4_weight.argtypes = [p, p, ctypes.c_float, i64, i64, i64]
    lib.oracle_nvfp4_weight.restype = ctypes.c_float
    lib.oracle_num_cores.argtypes = []
    lib.oracle_num_cores.restype = ctypes.c_int
    lib.oracle_logits_bf16.argtypes = [p, i64, i64, p, i64, p, ctypes.c_int]
    lib.oracle_logits_bf16.restype = ctypes.c_int
    lib.oracle_logits_nvfp4.argtypes = [p, p, ctypes.c_float, i64, i64, p, i64, p,
                                        ctypes.c_int]
    lib.oracle_logits_nvfp4.restype = ctypes.c_int
    lib.oracle_logits_fp8.argtypes = [p, ctypes.c_float, i64, i64, p, i64, p, ctypes.c_int]
    lib.oracle_logits_fp8.restype = ctypes.c_int
    lib.oracle_score_ids_fp8.argtypes = [p, ctypes.c_float, i64, i64, i64, p, i64, p, i64, p]
    lib.oracle_score_ids_fp8.restype = None
    lib.oracle_score_ids_bf16.argtypes = [p, i64, i64, i64, p, i64, p, i64, p]
    lib.oracle_score_ids_bf16.restype = None
    lib.oracle_score_ids_nvfp4.argtypes = [p, p, ctypes.c_float, i64, i64, i64, p, i64, p,
                                           i64, p]
    lib.oracle_score_ids_nvfp4.restype = None
    lib.oracle_quantize_nvfp4.argtypes = [p, i64, i64, p, p]
    lib.oracle_quantize_nvfp4.restype = ctypes.c_float
    lib.oracle_quantize_fp8.argtypes = [p, i64, i64, p]
    lib.oracle_quantize_fp8.restype = ctypes.c_float
    lib.oracle_topk.argtypes = [p, i64, i64, p, ctypes.c_int, p, p, p]
    lib.oracle_topk.restype = None
    lib.oracle_check_trim.argtypes = [p, i64, i64, p, i64, p, p]
    lib.oracle_check_trim.restype = i64
    lib.oracle_histogram.argtypes = [p, i64, i64, p]
    lib.oracle_histogram.restype = ctypes.c_int
    lib.oracle_build_ranks.argtypes = [p, i64, p, i64, i64, ctypes.c_int, p]
    lib.oracle_build_ranks.restype = i64
    lib.oracle_union_sorted.argtypes = [p, i64, p, i64, p]
    lib.oracle_union_sorted.restype = i64
    _lib = lib
    return lib


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data


def num_cores() -> int:
    """Host cores the oracle's threads would use by default."""
    return int(_load().oracle_num_cores())


def bf16_to_f32(bits: int) -> float:
    return float(_load().oracle_bf16_to_f32(int(bits)))


def e2m1(code: int) -> float:
    return float(_load().oracle_e2m1(int(code)))


def e4m3(byte: int) -> float:
    return float(_load().oracle_e4m3(int(byte)))


def logits_bf16(w: np.ndarray, h: np.ndarray, nthreads: int = 0):
    """fp32 logits[M][N] = W[N][K] . h[M][K]^T, ascending k, no FMA.

    w, h: uint16 arrays of bfloat16 bit patterns.  Returns (logits, threads)."""
    w = np.ascontiguousarray(w, dtype=np.uint16)
    h = np.ascontiguousarray(h, dtype=np.uint16)
    N, K = w.shape
    M, K2 = h.shape
    assert K == K2
    out = np.empty((M, N), dtype=np.float32)
    t = _load().oracle_logits_bf16(_ptr(w), N, K, _ptr(h), M, _ptr(out), nthreads)
    return out, int(t)


def logits_nvfp4(q: np.ndarray, scales: np.ndarray, g: float, h: np.ndarray,
                 nthreads: int = 0):
    """fp32 logits of an NVFP4 head: q uint8[N][K/2] (low nibble = even k),
    scales uint8[N][K/16] (e4m3), g the fp32 tensor scale, h bf16 bits[M][K]."""
    q = np.ascontiguousarray(q, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    h = np.ascontiguousarray(h, dtype=np.uint16)
    N, Kh = q.shape
    K = 2 * Kh
    assert scales.shape == (N, K // 16)
    M = h.shape[0]
    assert h.shape[1] == K
    out = np.empty((M, N), dtype=np.float32)
    t = _load().oracle_logits_nvfp4(_ptr(q), _ptr(scales), float(g), N, K, _ptr(h),
                                    M, _ptr(out), nthreads)
    return out, int(t)


def score_ids_bf16(w: np.ndarray, h: np.ndarray, ids: np.ndarray, id_base: int = 0):
    """fp32 scores[M][c]: the logit of head row ids[m][j] - id_base against
    h[m] (the same dot as logits_bf16); NaN for an id outside the head."""
    w = np.ascontiguousarray(w, dtype=np.uint16)
    h = np.ascontiguousarray(h, dtype=np.uint16)
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    N, K = w.shape
    M = h.shape[0]
    assert h.shape[1] == K and ids.ndim == 2 and ids.shape[0] == M
    c = ids.shape[1]
    out = np.empty((M, c), dtype=np.float32)
    _load().oracle_score_ids_bf16(_ptr(w), N, K, int(id_base), _ptr(h), M, _ptr(ids), c,
                                  _ptr(out))
    return out


def score_ids_nvfp4(q: np.ndarray, scales: np.ndarray, g: float, h: np.ndarray,
                    ids: np.ndarray, id_base: int = 0):
    """score_ids_bf16 for an NVFP4 head (the same weight decode as
    logits_nvfp4)."""
    q = np.ascontiguousarray(q, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    h = np.ascontiguousarray(h, dtype=np.uint16)
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    N, Kh = q.shape
    K = 2 * Kh
    assert scales.shape == (N, K // 16)
    M = h.shape[0]
    assert h.shape[1] == K and ids.ndim == 2 and ids.shape[0] == M
    c = ids.shape[1]
    out = np.empty((M, c), dtype=np.float32)
    _load().oracle_score_ids_nvfp4(_ptr(q), _ptr(scales), float(g), N, K, int(id_base),
                                   _ptr(h), M, _ptr(ids), c, _ptr(out))
    return out


def logits_fp8(q: np.ndarray, g: float, h: np.ndarray, nthreads: int = 0):
    """fp32 logits of an FP8 head: q uint8[N][K] (E4M3 codes), g the fp32
    tensor scale, h bf16 bits[M][K].  Returns (logits, threads)."""
    q = np.ascontiguousarray(q, dtype=np.uint8)
    h = np.ascontiguousarray(h, dtype=np.uint16)
    N, K = q.shape
    M = h.shape[0]
    assert h.shape[1] == K
    out = np.empty((M, N), dtype=np.float32)
    t = _load().oracle_logits_fp8(_ptr(q), float(g), N, K, _ptr(h), M, _ptr(out), nthreads)
    return out, int(t)


def score_ids_fp8(q: np.ndarray, g: float, h: np.ndarray, ids: np.ndarray, id_base: int = 0):
    """score_ids_bf16 for an FP8 head (the same weight decode as logits_fp8)."""
    q = np.ascontiguousarray(q, dtype=np.uint8)
    h = np.ascontiguousarray(h, dtype=np.uint16)
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    N, K = q.shape
    M = h.shape[0]
    assert h.shape[1] == K and ids.ndim == 2 and ids.shape[0] == M
    c = ids.shape[1]
    out = np.empty((M, c), dtype=np.float32)
    _load().oracle_score_ids_fp8(_ptr(q), float(g), N, K, int(id_base), _ptr(h), M, _ptr(ids),
                                 c, _ptr(out))
    return out


def quantize_nvfp4(w: np.ndarray):
    """Requantize a bf16 head [N][K] (bits) to NVFP4 by the plain recipe:
    returns (codes uint8[N][K/2], scales uint8[N][K/16], g)."""
    w = np.ascontiguousarray(w, dtype=np.uint16)
    N, K = w.shape
    q = np.empty((N, K // 2), dtype=np.uint8)
    sc = np.empty((N, K // 16), dtype=np.uint8)
    g = _load().oracle_quantize_nvfp4(_ptr(w), N, K, _ptr(q), _ptr(sc))
    return q, sc, float(g)


def quantize_fp8(w: np.ndarray):
    """Requantize a bf16 head [N][K] (bits) to FP8 E4M3 with one tensor
    scale: returns (codes uint8[N][K], g)."""
    w = np.ascontiguousarray(w, dtype=np.uint16)
    N, K = w.shape
    q = np.empty((N, K), dtype=np.uint8)
    g = _load().oracle_quantize_fp8(_ptr(w), N, K, _ptr(q))
    return q, float(g)


def nvfp4_weight(q, scales, g, n, k) -> float:
    q = np.ascontiguousarray(q, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    K = 2 * q.shape[1]
    return float(_load().oracle_nvfp4_weight(_ptr(q), _ptr(scales), float(g), K,
                                             int(n), int(k)))


def topk(logits: np.ndarray, k: int, d2t: np.ndarray | None = None):
    """Per row m: the k best n by (logit desc, full id asc); NaN ranks last.

    Returns (ids int32[M][k], vals float32[M][k], rows int64[M][k])."""
    logits = np.ascontiguousarray(logits, dtype=np.float32)
    M, N = logits.shape
    if d2t is not None:
        d2t = np.ascontiguousarray(d2t, dtype=np.int32)
        assert d2t.shape == (N,)
    ids = np.empty((M, k), dtype=np.int32)
    vals = np.empty((M, k), dtype=np.float32)
    rows = np.empty((M, k), dtype=np.int64)
    _load().oracle_topk(_ptr(logits), N, M, _ptr(d2t), int(k), _ptr(ids), _ptr(vals),
                        _ptr(rows))
    return ids, vals, rows


def argmax(logits: np.ndarray, d2t: np.ndarray | None = None):
    """Per row m: (full id, logit) of the best n; ties to the lowest full id."""
    ids, vals, _ = topk(logits, 1, d2t)
    return ids[:, 0].copy(), vals[:, 0].copy()


def row_stats(logits: np.ndarray):
    """Per row m: (gap = best - second best logit, max |logit|), NaNs ignored."""
    lg = np.where(np.isnan(logits), -np.inf, logits.astype(np.float64))
    part = -np.sort(-lg, axis=1)
    gap = part[:, 0] - part[:, 1] if lg.shape[1] > 1 else np.full(lg.shape[0], np.inf)
    maxabs = np.max(np.abs(np.where(np.isnan(logits), 0.0, logits)), axis=1)
    return gap, maxabs


def check_trim(w_full: np.ndarray, ranks: np.ndarray, w_trim: np.ndarray,
               d2t: np.ndarray | None) -> int:
    """Rows i where W_trim[i] != W_full[ranks[i]] bytewise or d2t[i] != ranks[i]
    (-1 if a rank is out of range)."""
    w_full = np.ascontiguousarray(w_full)
    w_trim = np.ascontiguousarray(w_trim)
    ranks = np.ascontiguousarray(ranks, dtype=np.int32)
    V = w_full.shape[0]
    row_bytes = w_full.nbytes // V if V else 0
    assert w_trim.shape[0] == ranks.shape[0]
    assert w_trim.nbytes == row_bytes * ranks.shape[0]
    if d2t is not None:
        d2t = np.ascontiguousarray(d2t, dtype=np.int32)
    return int(_load().oracle_check_trim(_ptr(w_full), V, row_bytes, _ptr(ranks),
                                         ranks.shape[0], _ptr(w_trim), _ptr(d2t)))


def histogram(tokens: np.ndarray, V: int, counts: np.ndarray | None = None):
    tokens = np.ascontiguousarray(tokens, dtype=np.int32)
    if counts is None:
        counts = np.zeros(V, dtype=np.int64)
    rc = _load().oracle_histogram(_ptr(tokens), tokens.shape[0], V, _ptr(counts))
    if rc != 0:
        raise ValueError("token id outside [0, V)")
    return counts


def build_ranks(counts: np.ndarray, N: int, forced: np.ndarray | None = None,
                sorted_ids: bool = False) -> np.ndarray:
    counts = np.ascontiguousarray(counts, dtype=np.int64)
    V = counts.shape[0]
    if forced is None:
        forced = np.zeros(0, dtype=np.int32)
    forced = np.ascontiguousarray(forced, dtype=np.int32)
    out = np.empty(max(min(N, V), 1), dtype=np.int32)
    n = _load().oracle_build_ranks(_ptr(counts), V, _ptr(forced), forced.shape[0], N,
                                   1 if sorted_ids else 0, _ptr(out))
    if n < 0:
        raise ValueError("bad argument to build_ranks")
    return out[:n].copy()


def union_sorted(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a, dtype=np.int32)
    b = np.ascontiguousarray(b, dtype=np.int32)
    out = np.empty(max(a.shape[0] + b.shape[0], 1), dtype=np.int32)
    n = _load().oracle_union_sorted(_ptr(a), a.shape[0], _ptr(b), b.shape[0], _ptr(out))
    return out[:n].copy()
