"""Parity rules between the CUDA library's results and the CPU oracle's.

Ids: the GPU id must equal the oracle's whenever the oracle's top-1/top-2 gap
exceeds 1e-3 * max|logit| of the row; otherwise any id whose oracle logit is
within that threshold of the oracle's maximum is accepted (both sides decide
on fp32 sums, added in different orders).
Logits: |gpu - oracle| <= 2e-3 * max(|oracle|, 1e-6) for the argmax logit,
measured against the oracle logit of the row the GPU picked; for top-k
entries against 2e-3 * max|logit| of the row (a k-th logit near 0 has no
meaningful relative error).
"""
from __future__ import annotations

import numpy as np

ID_GAP_REL = 1e-3
LOGIT_REL = 2e-3


def _rows_of_id(d2t, N):
    if d2t is None:
        return lambda i: [int(i)] if 0 <= i < N else []
    table = {}
    for n, i in enumerate(np.asarray(d2t).tolist()):
        table.setdefault(i, []).append(n)
    return lambda i: table.get(int(i), [])


def check_argmax(oracle, L, d2t, gpu_ids, gpu_logits, id_base=0):
    """Apply the parity rule; returns a small report dict.  L: oracle
    logits [M][N]; d2t: int32 [N] or None (ids = id_base + n)."""
    L = np.asarray(L, dtype=np.float32)
    M, N = L.shape
    d2t_full = None if d2t is None else np.asarray(d2t, dtype=np.int32)
    o_ids, o_vals = oracle.argmax(L, d2t_full)
    if d2t_full is None:
        o_ids = o_ids + id_base
    gap, mx = oracle.row_stats(L)
    rows_of = _rows_of_id(d2t_full, N) if d2t_full is not None else (
        lambda i: [int(i) - id_base] if 0 <= int(i) - id_base < N else [])
    exact = exempt = 0
    max_rel = 0.0
    for m in range(M):
        thr = ID_GAP_REL * mx[m]
        gid = int(gpu_ids[m])
        rows = rows_of(gid)
        assert rows, f"row {m}: GPU id {gid} is not an id of this head"
        if gap[m] > thr:
            assert gid == int(o_ids[m]), (
                f"row {m}: GPU id {gid} != oracle id {o_ids[m]} (gap {gap[m]:.3g} > {thr:.3g})")
            exact += 1
        else:
            assert max(L[m, r] for r in rows) >= o_vals[m] - thr, (
                f"row {m}: GPU id {gid} is not within the near-tie set")
            exempt += 1
        ref = max(float(L[m, r]) for r in rows)
        err = abs(float(gpu_logits[m]) - ref)
        assert err <= LOGIT_REL * max(abs(ref), 1e-6), (
            f"row {m}: GPU logit {gpu_logits[m]!r} vs oracle {ref!r}")
        max_rel = max(max_rel, err / max(abs(ref), 1e-6))
    return {"rows_exact": exact, "rows_exempt": exempt, "max_rel_logit_err": max_rel}


def check_topk(oracle, L, d2t, k, gpu_ids, gpu_logits, id_base=0):
    L = np.asarray(L, dtype=np.float32)
    M, N = L.shape
    d2t_full = None if d2t is None else np.asarray(d2t, dtype=np.int32)
    kk = min(k + 1, N)  # one more, for the gap below the k-th entry
    o_ids, o_vals, _ = oracle.topk(L, kk, d2t_full)
    if d2t_full is None:
        o_ids = o_ids + id_base
    _, mx = oracle.row_stats(L)
    rows_of = _rows_of_id(d2t_full, N) if d2t_full is not None else (
        lambda i: [int(i) - id_base] if 0 <= int(i) - id_base < N else [])
    exact = exempt = 0
    for m in range(M):
        thr = ID_GAP_REL * mx[m]
        used = set()
        prev = np.inf
        for j in range(k):
            gid = int(gpu_ids[m, j])
            rows = [r for r in rows_of(gid) if r not in used]
            assert rows, f"row {m} slot {j}: id {gid} unknown or repeated"
            # the row this entry stands for: the one whose oracle logit is closest
            r = min(rows, key=lambda r: abs(float(L[m, r]) - float(gpu_logits[m, j])))
            used.add(r)
            assert abs(float(L[m, r]) - float(o_vals[m, j])) <= thr, (
                f"row {m} slot {j}: oracle logit {L[m, r]} of GPU id {gid} is not "
                f"within {thr:.3g} of the oracle's {j}-th best {o_vals[m, j]}")
            lo_gap = (o_vals[m, j] - o_vals[m, j + 1]) if j + 1 < kk else np.inf
            hi_gap = (o_vals[m, j - 1] - o_vals[m, j]) if j > 0 else np.inf
            if min(lo_gap, hi_gap) > thr:
                assert gid == int(o_ids[m, j]), f"row {m} slot {j}: {gid} != {o_ids[m, j]}"
                exact += 1
            else:
                exempt += 1
            assert abs(float(gpu_logits[m, j]) - float(L[m, r])) <= LOGIT_REL * max(mx[m], 1e-6)
            assert float(gpu_logits[m, j]) <= prev
            prev = float(gpu_logits[m, j])
    return {"entries_exact": exact, "entries_exempt": exempt}
