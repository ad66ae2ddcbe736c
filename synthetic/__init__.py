"""Seeded synthetic inputs for the draft-head argmax path.

This module is shared by the tests, the smoke check and the benchmark, and it
serves both the CUDA library and the CPU oracle with identical bytes.  It
holds none of the method's arithmetic: no dot product over the head, no
argmax, no NVFP4 decode.  It only draws random numbers, rounds them to the
storage formats (bfloat16 by round-to-nearest-even on the bits; NVFP4 by the
quantizer below) and lays out ids.

The five workloads mirror the shapes on the pages:
  c1  shortlist of a 248,320-row head, K=2,560: every id below 8,192 plus
      7,808 random ids, sorted (the 16k list of "Shortlist MTP", section
      "Building the 16k shortlist"); W ~ N(0, 0.02), h ~ N(0, 1).
  c2  the full 248,320-row head, K=2,560, M in {1, 3} (draft / MTP2 verify,
      "Shortlist MTP", section "What I was testing").
  c3  FR-Spec trim to 32,768 rows by emitted-token frequency, K=5,120
      ("Masked MTP drafts": 248,320 / 32,768 = 7.6x); the token stream is a
      bounded Zipf(1.1) sample mapped through a seeded permutation of ids.
  c4  union list 47,149 + 9,749 ids sharing 4,143 -> 52,755 sorted ids
      ("[DGX Spark] Qwen3.8-Flash-Next on two DGX Sparks", section "Build the
      draft vocabulary from your own text"), M in {8, 16, 32}, with a planted
      top-2 pair per row whose gap spans 1e-4 .. 1.
  c5  NVFP4 trimmed head, 32,768 x 5,120, quantized from N(0, 0.02) bf16.
"""
from __future__ import annotations

import concurrent.futures as _cf
import os
from dataclasses import dataclass, field

import numpy as np

V_FULL = 248_320
BLOCK_ROWS = 2048  # rows per independently seeded generator block


# ---------------------------------------------------------------------------
# Storage formats (encoding only)
# ---------------------------------------------------------------------------

def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round binary32 values to bfloat16 bit patterns, nearest-even.
    Inputs are finite (normals from a generator)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bfloat16 bit patterns to binary32 (append sixteen zero bits)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(
        np.float32)


def _e4m3_encode(x: np.ndarray):
    """Non-negative float64 -> (E4M3 byte, its value), round-to-nearest-even,
    saturating at 448; 2^-9 is the smallest subnormal."""
    x = np.clip(np.asarray(x, dtype=np.float64), 0.0, 448.0)
    _, p = np.frexp(np.where(x > 0, x, 2.0 ** -10))  # zero takes the subnormal path: byte 0
    e = np.maximum(p - 1, -6)              # binade exponent, floor at the subnormal one
    spacing = np.ldexp(1.0, e - 3)         # 3 mantissa bits
    units = np.rint(x / spacing)           # ties to even
    value = units * spacing
    carry = units >= 16
    e = np.where(carry, e + 1, e)
    units = np.where(carry, 8, units).astype(np.int64)
    sub = (e == -6) & (units < 8)
    byte = np.where(sub, units, ((e + 7) << 3) | (units - 8))
    return byte.astype(np.uint8), value


_E2M1_GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def _e2m1_encode(x: np.ndarray) -> np.ndarray:
    """float64 -> E2M1 4-bit code (bit 3 sign), nearest-even, saturating at 6."""
    x = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(x), 6.0)
    _, p = np.frexp(np.where(a > 0, a, 1.0))
    e = np.clip(p - 1, 0, 2)               # binades [1,2), [2,4), [4,8); below 1: step 0.5
    spacing = np.ldexp(1.0, e - 1)
    spacing = np.where(a < 1.0, 0.5, spacing)
    v = np.minimum(np.rint(a / spacing) * spacing, 6.0)
    code = np.searchsorted(_E2M1_GRID, v).astype(np.uint8)
    return np.where(x < 0, code | np.uint8(8), code).astype(np.uint8)


def quantize_nvfp4(wbits: np.ndarray):
    """Quantize a bf16 head [N][K] to NVFP4: g = amax / (6 * 448) (fp32);
    per 16-element block s = e4m3(amax_b / (6 g)); q = e2m1(w / (s g)).
    A block whose scale rounds to zero gets zero codes.
    Returns (q uint8[N][K/2], low nibble = even k; scales uint8[N][K/16]; g)."""
    w = bf16_bits_to_f32(wbits).astype(np.float64)
    N, K = w.shape
    assert K % 32 == 0
    amax = float(np.max(np.abs(w))) if w.size else 0.0
    g = np.float32(amax / (6.0 * 448.0)) if amax > 0 else np.float32(1.0)
    blocks = w.reshape(N, K // 16, 16)
    amax_b = np.max(np.abs(blocks), axis=2)
    s_byte, s_val = _e4m3_encode(amax_b / (6.0 * float(g)))
    denom = (s_val * float(g))[:, :, None]
    x = np.where(denom > 0, blocks / np.where(denom > 0, denom, 1.0), 0.0)
    codes = _e2m1_encode(x).reshape(N, K)
    q = (codes[:, 0::2] | (codes[:, 1::2] << np.uint8(4))).astype(np.uint8)
    return q, s_byte.reshape(N, K // 16), float(g)


def quantize_fp8(wbits: np.ndarray, g: float | None = None):
    """Quantize a bf16 head [N][K] to FP8 E4M3 with one fp32 tensor scale:
    g = amax / 448 unless given; q = e4m3(|w| / g) with the sign in bit 7,
    nearest-even, saturating at 448.  Returns (q uint8[N][K], g)."""
    wbits = np.asarray(wbits, dtype=np.uint16)
    if g is None:
        amax = float(np.max(np.abs(bf16_bits_to_f32(wbits)))) if wbits.size else 0.0
        g = float(np.float32(amax / 448.0)) if amax > 0 else 1.0
    # a bf16 weight has 65,536 possible bit patterns: encode each once
    with np.errstate(invalid="ignore"):  # the signalling-NaN patterns
        v = bf16_bits_to_f32(np.arange(65536, dtype=np.uint32).astype(np.uint16)).astype(
            np.float64)
        finite = np.isfinite(v)
        byte, _ = _e4m3_encode(np.where(finite, np.abs(v), 0.0) / float(g))
    lut = np.where(v < 0, byte | np.uint8(0x80), byte).astype(np.uint8)
    lut[~finite] = 0x7F
    return lut[wbits], float(g)


# ---------------------------------------------------------------------------
# Random tensors
# ---------------------------------------------------------------------------

def _block_normals(seed: int, tag: int, b: int, rows: int, K: int, std: float):
    rng = np.random.default_rng([seed, tag, b])
    x = rng.standard_normal((rows, K), dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return f32_to_bf16_bits(x)


def normal_bf16_rows(seed: int, rows: int, K: int, std: float, tag: int = 0,
                     threads: int | None = None) -> np.ndarray:
    """bf16 bits [rows][K] of N(0, std^2), drawn in blocks of BLOCK_ROWS rows,
    each from its own generator seeded by (seed, tag, block), so the bytes do
    not depend on the thread count."""
    out = np.empty((rows, K), dtype=np.uint16)
    nblk = (rows + BLOCK_ROWS - 1) // BLOCK_ROWS

    def work(b):
        r0 = b * BLOCK_ROWS
        r1 = min(rows, r0 + BLOCK_ROWS)
        out[r0:r1] = _block_normals(seed, tag, b, r1 - r0, K, std)

    threads = threads or min(16, os.cpu_count() or 1)
    if nblk <= 1 or threads <= 1:
        for b in range(nblk):
            work(b)
    else:
        with _cf.ThreadPoolExecutor(threads) as ex:
            list(ex.map(work, range(nblk)))
    return out


def normal_fp8_rows(seed: int, rows: int, K: int, std: float, tag: int = 0,
                    threads: int | None = None):
    """An FP8 head: the rows of normal_bf16_rows(seed, rows, K, std, tag),
    quantized block by block with the fixed tensor scale g = 6 std / 448 (so
    no pass over the whole head is needed; |w| > 6 std saturates).
    Returns (q uint8[rows][K], g)."""
    g = float(np.float32(6.0 * std / 448.0))
    out = np.empty((rows, K), dtype=np.uint8)
    nblk = (rows + BLOCK_ROWS - 1) // BLOCK_ROWS

    def work(b):
        r0 = b * BLOCK_ROWS
        r1 = min(rows, r0 + BLOCK_ROWS)
        out[r0:r1] = quantize_fp8(_block_normals(seed, tag, b, r1 - r0, K, std), g)[0]

    threads = threads or min(16, os.cpu_count() or 1)
    if nblk <= 1 or threads <= 1:
        for b in range(nblk):
            work(b)
    else:
        with _cf.ThreadPoolExecutor(threads) as ex:
            list(ex.map(work, range(nblk)))
    return out, g


def hidden_bf16(seed: int, M: int, K: int) -> np.ndarray:
    """h[M][K] ~ N(0, 1) as bf16 bits (tag 1, independent of the head)."""
    rng = np.random.default_rng([seed, 1])
    return f32_to_bf16_bits(rng.standard_normal((M, K), dtype=np.float32))


# ---------------------------------------------------------------------------
# Id lists and token streams
# ---------------------------------------------------------------------------

def shortlist_low_plus_random(seed: int, V: int, n_low: int, n_rand: int) -> np.ndarray:
    """Every id below n_low plus n_rand distinct random ids from [n_low, V),
    sorted ascending."""
    rng = np.random.default_rng([seed, 2])
    extra = rng.choice(np.arange(n_low, V, dtype=np.int64), size=n_rand, replace=False)
    return np.sort(np.concatenate([np.arange(n_low, dtype=np.int64), extra])).astype(
        np.int32)


def zipf_permutation(seed: int, V: int, tag: int = 3) -> np.ndarray:
    """The seeded permutation that maps Zipf rank r (1-based) to id perm[r-1]."""
    return np.random.default_rng([seed, tag, 7]).permutation(V).astype(np.int32)


def zipf_tokens(seed: int, V: int, S: int, s: float = 1.1, tag: int = 3) -> np.ndarray:
    """S tokens from a Zipf(s) law bounded to ranks 1..V (inverse-CDF sampling
    of p_r ~ r^-s), rank r mapped to id perm[r-1] for a seeded permutation of
    [0, V).  Returns int32[S]."""
    rng = np.random.default_rng([seed, tag])
    perm = zipf_permutation(seed, V, tag)
    p = np.arange(1, V + 1, dtype=np.float64) ** (-s)
    cdf = np.cumsum(p)
    cdf /= cdf[-1]
    out = np.empty(S, dtype=np.int32)
    chunk = 1 << 22
    for i in range(0, S, chunk):
        u = rng.random(min(chunk, S - i))
        r = np.minimum(np.searchsorted(cdf, u, side="right"), V - 1)
        out[i:i + r.shape[0]] = perm[r]
    return out


def candidate_ids(seed: int, V: int, M: int, c: int, s: float = 1.1, tag: int = 5) -> np.ndarray:
    """A drafter's candidates: for each of M rows, c distinct ids drawn from
    the bounded Zipf(s) law of zipf_tokens (frequent tokens are likely
    candidates).  Returns int32[M][c]."""
    rng = np.random.default_rng([seed, tag])
    perm = zipf_permutation(seed, V, tag)
    p = np.arange(1, V + 1, dtype=np.float64) ** (-s)
    cdf = np.cumsum(p)
    cdf /= cdf[-1]
    out = np.empty((M, c), dtype=np.int32)
    for m in range(M):
        got: list[int] = []
        seen: set[int] = set()
        while len(got) < c:
            r = np.minimum(np.searchsorted(cdf, rng.random(2 * c), side="right"), V - 1)
            for x in perm[r].tolist():
                if x not in seen and len(got) < c:
                    seen.add(x)
                    got.append(x)
        out[m] = got
    return out


def union_sets(seed: int, V: int, na: int, nb: int, n_shared: int):
    """Two id sets A (|A| = na) and B (|B| = nb) with |A & B| = n_shared, drawn
    without replacement from [0, V).  Returns (A, B) as unsorted int32."""
    rng = np.random.default_rng([seed, 4])
    pool = rng.choice(V, size=na + nb - n_shared, replace=False).astype(np.int32)
    A = pool[:na]
    B = np.concatenate([pool[:n_shared], pool[na:]])
    return rng.permutation(A).astype(np.int32), rng.permutation(B).astype(np.int32)


def structural_forced_set(seed: int, V: int, n_low: int, core: int, core_above: int):
    """A stand-in for the 16k list's forced groups: every id below n_low, plus a
    'structural core' of `core` ids of which `core_above` lie above n_low and
    the rest below it.  (The real core needs a tokenizer.)"""
    rng = np.random.default_rng([seed, 5])
    low = np.arange(n_low, dtype=np.int32)
    above = rng.choice(np.arange(n_low + 1, V), size=core_above, replace=False)
    below = rng.choice(np.arange(n_low), size=core - core_above, replace=False)
    return low, np.concatenate([above, below]).astype(np.int32)


# ---------------------------------------------------------------------------
# Near-tie planting (c4)
# ---------------------------------------------------------------------------

def plant_near_ties(W: np.ndarray, h: np.ndarray, gaps: np.ndarray, seed: int,
                    level_sigmas: float = 8.0):
    """For each hidden row m, overwrite two head rows p_m, q_m so that they
    become row m's top two with a logit gap close to gaps[m].

    W[p_m] = bf16(c h_m) with c = L / |h_m|^2, L = level_sigmas * 0.02 |h_m|
    (well above the natural maximum of N(0, (0.02 |h_m|)^2) logits).  W[q_m]
    is W[p_m] with one element k* lowered so that (W[p][k*] - W[q][k*]) h[k*]
    is as close as bf16 allows to the target gap; k* is chosen per row for
    that.  p_m < q_m for even m and p_m > q_m for odd m, so the lower-id row
    of the pair alternates between winner and runner-up.  The achieved gaps
    depend on rounding and are measured by the oracle, not assumed here.
    Returns (p, q) row positions.  W is modified in place."""
    N, K = W.shape
    M = h.shape[0]
    rng = np.random.default_rng([seed, 6])
    pos = rng.choice(N, size=2 * M, replace=False)
    p = np.empty(M, dtype=np.int64)
    q = np.empty(M, dtype=np.int64)
    for m in range(M):
        a, b = sorted(pos[2 * m:2 * m + 2])
        p[m], q[m] = (a, b) if m % 2 == 0 else (b, a)
        hm = bf16_bits_to_f32(h[m]).astype(np.float64)
        nrm2 = float(hm @ hm)  # a norm of the hidden row, not a logit
        level = level_sigmas * 0.02 * np.sqrt(nrm2)
        wp_bits = f32_to_bf16_bits((level / nrm2 * hm).astype(np.float32))
        wp = bf16_bits_to_f32(wp_bits).astype(np.float64)
        if gaps[m] >= 1e-2:
            # wide gap: the whole row scaled to level - gap (bf16 rounding of
            # the row moves the result by a few 1e-4)
            wq_bits = f32_to_bf16_bits(((level - gaps[m]) / nrm2 * hm).astype(np.float32))
        else:
            # narrow gap: one element lowered; among elements with |h_k| >= 1
            # (so the change stays small) keep the one closest to the target
            safe = np.where(np.abs(hm) >= 1.0, hm, 1.0)
            tgt = wp - gaps[m] / safe
            cand_bits = f32_to_bf16_bits(tgt.astype(np.float32))
            cand = bf16_bits_to_f32(cand_bits).astype(np.float64)
            achieved = (wp - cand) * hm
            ok = (np.abs(hm) >= 1.0) & (achieved > 0)
            err = np.full(K, np.inf)
            err[ok] = np.abs(np.log(achieved[ok] / gaps[m]))
            kstar = int(np.argmin(err))
            wq_bits = wp_bits.copy()
            wq_bits[kstar] = cand_bits[kstar]
        W[p[m]] = wp_bits
        W[q[m]] = wq_bits
    return p, q


# ---------------------------------------------------------------------------
# The five workloads
# ---------------------------------------------------------------------------

@dataclass
class Workload:
    name: str
    V: int
    K: int
    Ms: tuple
    topk: int
    seed: int
    dtype: str = "bf16"
    # filled by build()
    w_full: np.ndarray | None = None      # bf16 bits [V][K] (when the head is trimmed)
    ranks: np.ndarray | None = None       # int32 ids (trimmed heads)
    w: np.ndarray | None = None           # the head the argmax reads: bf16 bits [N][K]
    q: np.ndarray | None = None           # NVFP4 codes [N][K/2]
    scales: np.ndarray | None = None      # NVFP4 e4m3 scales [N][K/16]
    g: float = 1.0
    d2t: np.ndarray | None = None         # int32[N] or None (identity)
    h: dict = field(default_factory=dict)  # M -> bf16 bits [M][K]
    extra: dict = field(default_factory=dict)

    @property
    def N(self) -> int:
        if self.w is not None:
            return self.w.shape[0]
        return self.q.shape[0]


def c1(V=V_FULL, K=2560, n_low=8192, n_rand=7808, seed=0, with_full=True) -> Workload:
    wl = Workload("c1_shortlist16k_bf16", V, K, (1,), 1, seed)
    wl.ranks = shortlist_low_plus_random(seed, V, n_low, n_rand)
    if with_full:
        wl.w_full = normal_bf16_rows(seed, V, K, 0.02)
        wl.w = wl.w_full[wl.ranks]
    else:  # same bytes, rows drawn only for the listed ids' blocks
        wl.w = _rows_of_full(seed, V, K, wl.ranks)
    wl.d2t = wl.ranks.copy()
    wl.h = {1: hidden_bf16(seed, 1, K)}
    return wl


def _rows_of_full(seed, V, K, ids):
    out = np.empty((ids.shape[0], K), dtype=np.uint16)
    blocks = np.unique(ids // BLOCK_ROWS)
    for b in blocks:
        r0 = int(b) * BLOCK_ROWS
        rows = min(V, r0 + BLOCK_ROWS) - r0
        blk = _block_normals(seed, 0, int(b), rows, K, 0.02)
        sel = np.nonzero(ids // BLOCK_ROWS == b)[0]
        out[sel] = blk[ids[sel] - r0]
    return out


def c2(V=V_FULL, K=2560, Ms=(1, 3), seed=1) -> Workload:
    wl = Workload("c2_fullvocab_bf16", V, K, tuple(Ms), 4, seed)
    wl.w = normal_bf16_rows(seed, V, K, 0.02)
    wl.d2t = None
    wl.h = {M: hidden_bf16(seed + 100 * M, M, K) for M in Ms}
    return wl


def c3(V=V_FULL, K=5120, N=32768, Ms=(1, 2, 3, 4), S=10_000_000, seed=2) -> Workload:
    wl = Workload("c3_frspec_trim32k_bf16", V, K, tuple(Ms), 1, seed)
    wl.w_full = normal_bf16_rows(seed, V, K, 0.02)
    wl.extra["tokens"] = zipf_tokens(seed, V, S)
    wl.extra["N"] = N
    wl.h = {M: hidden_bf16(seed + 100 * M, M, K) for M in Ms}
    return wl


def c4(V=V_FULL, K=2560, na=47149, nb=9749, n_shared=4143, Ms=(8, 16, 32), seed=3,
       gap_lo=1e-4, gap_hi=1.0) -> Workload:
    wl = Workload("c4_batched_union53k_bf16", V, K, tuple(Ms), 1, seed)
    A, B = union_sets(seed, V, na, nb, n_shared)
    wl.extra["A"], wl.extra["B"] = A, B
    ids = np.union1d(A, B).astype(np.int32)
    wl.ranks = ids
    wl.d2t = ids.copy()
    base = normal_bf16_rows(seed, ids.shape[0], K, 0.02)
    wl.extra["w_by_M"] = {}
    wl.extra["planted"] = {}
    for M in Ms:
        h = hidden_bf16(seed + 100 * M, M, K)
        W = base.copy()
        gaps = np.geomspace(gap_lo, gap_hi, M) if M > 1 else np.array([gap_lo])
        p, q = plant_near_ties(W, h, gaps, seed + M)
        wl.h[M] = h
        wl.extra["w_by_M"][M] = W
        wl.extra["planted"][M] = (p, q, gaps)
    wl.w = wl.extra["w_by_M"][Ms[0]]
    return wl


def c5(V=V_FULL, K=5120, N=32768, Ms=(1, 3), seed=4) -> Workload:
    wl = Workload("c5_nvfp4_trim32k", V, K, tuple(Ms), 1, seed, dtype="nvfp4")
    wbits = normal_bf16_rows(seed, N, K, 0.02)
    wl.q, wl.scales, wl.g = quantize_nvfp4(wbits)
    # d2t: a frequency-ranked id list in rank order (not monotone): the first
    # N ids of the Zipf rank -> id permutation, i.e. the ids a Zipf(1.1)
    # token stream would rank highest.
    wl.d2t = zipf_permutation(seed, V)[:N].copy()
    wl.extra["w_bf16_source"] = wbits
    wl.h = {M: hidden_bf16(seed + 100 * M, M, K) for M in Ms}
    return wl
