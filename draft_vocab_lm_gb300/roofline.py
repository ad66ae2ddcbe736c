"""Byte and bandwidth accounting for the draft-head argmax path.

The pages define a kernel's effective bandwidth as the weight bytes it must
read divided by its time ("[DGX Spark] Qwen3.8-Flash-Next on two DGX Sparks",
section "Decode runs at 80-87% of memory bandwidth": the BF16 lm_head of
124,160 x 2,560 rows per GPU is 635.7 MB, read in 2,677 us, i.e. 237 GB/s,
87% of GB10's 273 GB/s).  This module applies that definition to one call of
``draft_argmax`` / ``draft_topk``: the algorithmic bytes are what the method
must move -- the head, the hidden rows, the d2t entry of each reported id and
the outputs -- not the logits, which are never written, and not the rows a
shortlist skips.
"""
from __future__ import annotations

NOMINAL_HBM_GBS = 8000.0  # GB300 HBM3e, nominal


def head_bytes(N: int, K: int, dtype: str = "bf16") -> int:
    """Bytes of an N x K head: bf16 2 B per weight; NVFP4 half a byte per
    weight plus one E4M3 scale per 16 weights plus the fp32 tensor scale;
    FP8 one byte per weight plus the fp32 tensor scale."""
    if dtype == "bf16":
        return N * K * 2
    if dtype == "nvfp4":
        return N * K // 2 + N * K // 16 + 4
    if dtype == "fp8":
        return N * K + 4
    raise ValueError(dtype)


def call_bytes(N: int, K: int, M: int, dtype: str = "bf16", k: int = 1) -> int:
    """Algorithmic bytes of one argmax (k = 1) or top-k call: head + hidden
    rows (bf16) + for each of the M*k results its d2t entry (4 B), id (4 B)
    and logit (4 B)."""
    return head_bytes(N, K, dtype) + M * K * 2 + M * k * 12


def score_bytes(M: int, c: int, K: int, dtype: str = "bf16") -> int:
    """Algorithmic bytes of one candidate-scoring call: each named head row
    (M*c rows, repeats counted once per candidate), the hidden rows, the ids
    and the fp32 scores."""
    row = head_bytes(1, K, dtype) - (0 if dtype == "bf16" else 4)
    return M * c * row + M * K * 2 + M * c * 8


def quantize_bytes(N: int, K: int, dtype: str) -> int:
    """Algorithmic bytes of requantizing a bf16 N x K head: the head read
    once and the NVFP4 or FP8 head written.  (The recipe needs the head's
    maximum before any code, so a head larger than L2 is read twice: its
    traffic is N K 2 bytes more, and half the copy peak is its ceiling on
    this count.)"""
    return N * K * 2 + head_bytes(N, K, dtype) - 4


def call_flops(N: int, K: int, M: int) -> int:
    """Multiply-adds of the projection, counted as 2 flops each."""
    return 2 * M * N * K


def trim_bytes(n_rows: int, row_bytes: int) -> int:
    """Algorithmic bytes of a load-time trim: each kept row read once and
    written once, plus the d2t write (4 B per row)."""
    return 2 * n_rows * row_bytes + 4 * n_rows


def effective_gbs(nbytes: float, seconds: float) -> float:
    """Effective bandwidth in GB/s (10^9 bytes per second)."""
    return nbytes / seconds / 1e9
