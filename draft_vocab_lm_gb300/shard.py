"""Combining the argmax of a head split by rows across devices.

When the vocabulary rows of a head are split over G devices (as the pages do
at TP=2: "[DGX Spark] Qwen3.8-Flash-Next on two DGX Sparks", section "Decode
runs at 80-87% of memory bandwidth", 124,160 of 248,320 rows per GPU; the
shortlist split evenly over the ranks in section "Build the draft vocabulary
from your own text"), each part's draft_argmax yields a local (id, logit) per
hidden row -- the local argmax reduction of "Shortlist MTP", section
"Re-running the comparison fairly" -- and one exchange picks the global best.

The exchange packs each (logit, id) into one signed 64-bit key whose order is
the result order (logit descending, then id ascending; NaN below every number;
-0 folded onto +0), so a single MAX all-reduce of M keys combines the parts.
A part is a row slice of the head (``Head.slice_rows`` keeps full ids).
"""
from __future__ import annotations

import numpy as np

_SIGN = np.uint64(1 << 63)


def pack_keys(ids, logits) -> np.ndarray:
    """int64 keys whose signed order is (logit desc, id asc)."""
    ids = np.asarray(ids, dtype=np.int64).ravel()
    lg = np.ascontiguousarray(np.asarray(logits, dtype=np.float32).ravel())
    b = lg.view(np.uint32).astype(np.uint64)
    mag = b & np.uint64(0x7FFFFFFF)
    neg = (b & np.uint64(0x80000000)) != 0
    hi = np.where(neg, (~b) & np.uint64(0xFFFFFFFF), b | np.uint64(0x80000000))
    hi = np.where(mag == 0, np.uint64(0x80000000), hi)
    hi = np.where(mag > np.uint64(0x7F800000), np.uint64(0), hi)
    lo = np.uint64(0xFFFFFFFF) - (ids.astype(np.uint64) & np.uint64(0xFFFFFFFF))
    key = (hi << np.uint64(32)) | lo
    return (key ^ _SIGN).view(np.int64)


def unpack_keys(keys):
    """Inverse of pack_keys: (ids int32, logits float32)."""
    k = (np.asarray(keys, dtype=np.int64).view(np.uint64) ^ _SIGN)
    hi = (k >> np.uint64(32)).astype(np.uint64)
    bits = np.where((hi & np.uint64(0x80000000)) != 0, hi & np.uint64(0x7FFFFFFF),
                    (~hi) & np.uint64(0xFFFFFFFF)).astype(np.uint32)
    ids = (np.uint64(0xFFFFFFFF) - (k & np.uint64(0xFFFFFFFF))).astype(np.uint32).view(np.int32)
    return ids, bits.view(np.float32)


def combine(parts):
    """The global (ids, logits) from a list of per-part (ids, logits)."""
    keys = np.stack([pack_keys(i, v) for i, v in parts])
    return unpack_keys(keys.max(axis=0))


def allreduce_argmax(ids, logits, group=None):
    """Combine this rank's (ids, logits) with every other rank's by one MAX
    all-reduce of packed keys (torch.distributed, any backend)."""
    import torch
    import torch.distributed as dist
    keys = torch.from_numpy(pack_keys(ids, logits))
    dist.all_reduce(keys, op=dist.ReduceOp.MAX, group=group)
    return unpack_keys(keys.numpy())
