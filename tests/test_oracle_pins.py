"""Pins of the CPU oracle's logits, argmax/top-k and NVFP4 decode to things
other than itself: exact integer arithmetic, closed forms, the fp32
summation error bound against an fp64 dot, brute-force sorts, hand-computed
format values and the shortlist masking invariant."""
import math
import os

import numpy as np
import pytest

from conftest import GOLDEN
import synthetic as S


def _int_bf16(rng, shape, lo=-8, hi=8):
    """Small integers, exactly representable in bf16; returned as (bits, ints)."""
    x = rng.integers(lo, hi + 1, size=shape).astype(np.int64)
    return S.f32_to_bf16_bits(x.astype(np.float32)), x


# --------------------------------------------------------------------------
# logits
# --------------------------------------------------------------------------

@pytest.mark.parametrize("N,K,M", [(1, 64, 1), (37, 64, 3), (64, 128, 4), (5, 128, 2)])
def test_logits_exact_integer_bruteforce(oracle_mod, N, K, M):
    # every partial sum is an integer below 2^24: exact in any order, so the
    # oracle must equal the integer matrix product bit for bit
    rng = np.random.default_rng(N * 1000 + K + M)
    wb, wi = _int_bf16(rng, (N, K))
    hb, hi = _int_bf16(rng, (M, K))
    got, _ = oracle_mod.logits_bf16(wb, hb, nthreads=3)
    want = (hi @ wi.T).astype(np.float32)
    assert np.array_equal(got, want)


def test_logits_onehot_and_ones_closed_forms(oracle_mod):
    rng = np.random.default_rng(5)
    N, K = 50, 192
    wb = S.normal_bf16_rows(5, N, K, 0.02)
    w = S.bf16_bits_to_f32(wb)
    for j in (0, 7, K - 1):
        h = np.zeros((1, K), np.float32)
        h[0, j] = 1.0
        got, _ = oracle_mod.logits_bf16(wb, S.f32_to_bf16_bits(h))
        assert np.array_equal(got[0], w[:, j])
    # all-ones against small-integer rows: the row sums, exactly
    wb2, wi2 = _int_bf16(rng, (N, K))
    ones = S.f32_to_bf16_bits(np.ones((1, K), np.float32))
    got, _ = oracle_mod.logits_bf16(wb2, ones)
    assert np.array_equal(got[0], wi2.sum(axis=1).astype(np.float32))


def test_logits_within_fp32_summation_bound_of_fp64(oracle_mod):
    # recursive fp32 summation of exact products: |fl - exact| <= gamma_K * sum|x|
    N, K, M = 300, 2560, 3
    wb = S.normal_bf16_rows(11, N, K, 0.02)
    hb = S.hidden_bf16(11, M, K)
    got, _ = oracle_mod.logits_bf16(wb, hb, nthreads=4)
    w = S.bf16_bits_to_f32(wb).astype(np.float64)
    h = S.bf16_bits_to_f32(hb).astype(np.float64)
    exact = h @ w.T
    u = 2.0 ** -24
    gamma = K * u / (1 - K * u)
    bound = gamma * (np.abs(h) @ np.abs(w).T)
    assert np.all(np.abs(got - exact) <= bound)
    # and the error is far below the parity tolerance (2e-3 relative)
    assert np.max(np.abs(got - exact)) < 1e-4


def test_logits_thread_count_invariant(oracle_mod):
    wb = S.normal_bf16_rows(12, 101, 256, 0.02)
    hb = S.hidden_bf16(12, 2, 256)
    a, _ = oracle_mod.logits_bf16(wb, hb, nthreads=1)
    b, t = oracle_mod.logits_bf16(wb, hb, nthreads=7)
    assert t == 7 and np.array_equal(a, b)


# --------------------------------------------------------------------------
# argmax / top-k and the tie rule
# --------------------------------------------------------------------------

def _brute_topk(lrow, ids, k):
    def key(n):
        v = lrow[n]
        return (1, 0.0, ids[n]) if math.isnan(v) else (0, -float(v), ids[n])
    order = sorted(range(len(lrow)), key=key)
    return order[:k]


@pytest.mark.parametrize("seed", range(6))
def test_topk_bruteforce_with_ties_and_nonmonotone_d2t(oracle_mod, seed):
    rng = np.random.default_rng(seed)
    M, N, k = 3, 40, 4
    # few distinct values -> many exact ties; d2t a permutation of distinct ids
    logits = rng.integers(-3, 4, size=(M, N)).astype(np.float32)
    d2t = rng.permutation(1000)[:N].astype(np.int32)
    ids, vals, rows = oracle_mod.topk(logits, k, d2t)
    for m in range(M):
        want_rows = _brute_topk(logits[m], d2t, k)
        assert list(rows[m]) == want_rows
        assert list(ids[m]) == [int(d2t[n]) for n in want_rows]
        assert list(vals[m]) == [float(logits[m, n]) for n in want_rows]


def test_argmax_tie_goes_to_lowest_full_id_not_lowest_row(oracle_mod):
    logits = np.array([[1.0, 5.0, 2.0, 5.0, 5.0]], np.float32)
    d2t = np.array([9, 70, 3, 12, 40], np.int32)
    ids, vals = oracle_mod.argmax(logits, d2t)
    assert ids[0] == 12 and vals[0] == 5.0
    ids, _ = oracle_mod.argmax(logits, None)
    assert ids[0] == 1


def test_nan_never_wins_and_signed_zeros_tie(oracle_mod):
    logits = np.array([[np.nan, -1.0, np.nan], [0.0, -0.0, -5.0]], np.float32)
    d2t = np.array([0, 5, 1], np.int32)
    ids, vals, _ = oracle_mod.topk(logits, 3, d2t)
    assert list(ids[0][:1]) == [5]
    assert list(ids[0][1:]) == [0, 1]  # NaNs last, by id
    # +0 and -0 are equal logits: the lower full id (0, then 5) wins
    assert list(ids[1]) == [0, 5, 1]


def test_topk_k1_is_argmax(oracle_mod):
    rng = np.random.default_rng(3)
    logits = rng.standard_normal((4, 500)).astype(np.float32)
    a, av = oracle_mod.argmax(logits)
    assert np.array_equal(a, np.argmax(logits, axis=1))
    assert np.array_equal(av, logits.max(axis=1))


def test_shortlist_masking_invariant(oracle_mod):
    # the shortlist's argmax (through d2t) equals the full head's argmax with
    # every id outside the list set to -inf
    V, K, M = 3000, 128, 3
    wfull = S.normal_bf16_rows(21, V, K, 0.02)
    hb = S.hidden_bf16(21, M, K)
    rng = np.random.default_rng(21)
    ranks = rng.permutation(V)[:700].astype(np.int32)  # rank order, not sorted
    lt, _ = oracle_mod.logits_bf16(wfull[ranks], hb)
    lf, _ = oracle_mod.logits_bf16(wfull, hb)
    masked = np.full_like(lf, -np.inf)
    masked[:, ranks] = lf[:, ranks]
    ids_t, vals_t = oracle_mod.argmax(lt, ranks)
    ids_f, vals_f = oracle_mod.argmax(masked)
    assert np.array_equal(ids_t, ids_f) and np.array_equal(vals_t, vals_f)
    # identity ranks: the trimmed head is the full head
    ident = np.arange(V, dtype=np.int32)
    li, _ = oracle_mod.logits_bf16(wfull[ident], hb)
    assert np.array_equal(oracle_mod.argmax(li, ident)[0], oracle_mod.argmax(lf)[0])


def test_row_stats(oracle_mod):
    logits = np.array([[1.0, 4.0, -6.0, 3.5]], np.float32)
    gap, mx = oracle_mod.row_stats(logits)
    assert gap[0] == 0.5 and mx[0] == 6.0


# --------------------------------------------------------------------------
# NVFP4
# --------------------------------------------------------------------------

def _read_values():
    rows = []
    with open(os.path.join(GOLDEN, "nvfp4_values.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            kind, byte, val = line.split()[:3]
            rows.append((kind, int(byte, 16), float(val)))
    return rows


def test_format_values_match_hand_computed(oracle_mod):
    rows = _read_values()
    assert len(rows) == 30
    for kind, byte, val in rows:
        got = oracle_mod.e2m1(byte) if kind == "e2m1" else oracle_mod.e4m3(byte)
        if math.isnan(val):
            assert math.isnan(got)
        else:
            assert got == val and math.copysign(1, got) == math.copysign(1, val), (kind, byte)


def _read_block():
    g = None
    q, sc, ones, onehot = [], [], {}, []
    with open(os.path.join(GOLDEN, "nvfp4_block.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            t = line.split()
            if t[0] == "g":
                g = float(t[1])
            elif t[0] == "row":
                i = t.index("bytes")
                sc.append([int(x, 16) for x in t[3:i]])
                q.append([int(x, 16) for x in t[i + 1:]])
            elif t[0] == "ones":
                ones[int(t[1])] = float(t[2])
            elif t[0] == "onehot":
                onehot.append((int(t[1]), int(t[2]), float(t[3])))
    return (np.array(q, np.uint8), np.array(sc, np.uint8), g, ones, onehot)


def test_nvfp4_hand_built_block(oracle_mod):
    q, sc, g, ones, onehot = _read_block()
    K = 32
    h1 = S.f32_to_bf16_bits(np.ones((1, K), np.float32))
    got, _ = oracle_mod.logits_nvfp4(q, sc, g, h1)
    for n, v in ones.items():
        assert got[0, n] == v
    for n, k, v in onehot:
        h = np.zeros((1, K), np.float32)
        h[0, k] = 1.0
        got, _ = oracle_mod.logits_nvfp4(q, sc, g, S.f32_to_bf16_bits(h))
        assert got[0, n] == v
        assert oracle_mod.nvfp4_weight(q, sc, g, n, k) == v


def test_nvfp4_dequant_of_quantized_head_is_close(oracle_mod):
    # the generator's quantizer and the oracle's decode agree to within the
    # format's rounding: |w - deq| <= 1.5 * s_block * g (half the widest E2M1
    # step is one unit; the scale's own rounding adds at most 1/16 of 6 units)
    N, K = 8, 64
    wb = S.normal_bf16_rows(31, N, K, 0.02)
    q, sc, g = S.quantize_nvfp4(wb)
    w = S.bf16_bits_to_f32(wb).astype(np.float64)
    for n in range(N):
        for k in range(K):
            deq = oracle_mod.nvfp4_weight(q, sc, g, n, k)
            s = oracle_mod.e4m3(int(sc[n, k // 16]))
            assert abs(w[n, k] - deq) <= 1.5 * s * g + 1e-12
    # largest-magnitude weight of each block lands within 1/16 relative
    for n in range(N):
        for b in range(K // 16):
            blk = w[n, 16 * b:16 * b + 16]
            j = int(np.argmax(np.abs(blk)))
            deq = oracle_mod.nvfp4_weight(q, sc, g, n, 16 * b + j)
            assert abs(deq - blk[j]) <= abs(blk[j]) / 8 + 1e-12


# --------------------------------------------------------------------------
# trim check
# --------------------------------------------------------------------------

def test_check_trim_detects_planted_faults(oracle_mod):
    V, K = 500, 64
    wfull = S.normal_bf16_rows(41, V, K, 0.02)
    rng = np.random.default_rng(41)
    ranks = np.concatenate([rng.permutation(V)[:120], [7, 7]]).astype(np.int32)  # duplicates
    wtrim = wfull[ranks].copy()
    d2t = ranks.copy()
    assert oracle_mod.check_trim(wfull, ranks, wtrim, d2t) == 0
    bad = wtrim.copy()
    bad[5, 3] ^= 1
    assert oracle_mod.check_trim(wfull, ranks, bad, d2t) == 1
    badd = d2t.copy()
    badd[0] += 1
    assert oracle_mod.check_trim(wfull, ranks, wtrim, badd) == 1
    oob = ranks.copy()
    oob[3] = V
    assert oracle_mod.check_trim(wfull, oob, wtrim, None) == -1
