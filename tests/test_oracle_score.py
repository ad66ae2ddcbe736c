"""Pins of the oracle's candidate scores ("Masked MTP drafts", section
"Update (November 2026)": a drafter's candidates scored through the target's
own LM head, bf16 or NVFP4) to things other than itself: exact integer
arithmetic, the hand-built NVFP4 block, the fp32 summation error bound
against an fp64 dot, and the NaN rule for ids outside the head."""
import numpy as np
import pytest

from test_oracle_pins import _int_bf16, _read_block
import synthetic as S


@pytest.mark.parametrize("N,K,M,c", [(1, 64, 1, 1), (37, 64, 3, 9), (64, 128, 4, 40)])
def test_score_exact_integer_bruteforce(oracle_mod, N, K, M, c):
    # integer weights and hidden values below 8: every partial sum is an
    # integer under 2^24, exact in any order, so each score must equal the
    # integer dot of the named row bit for bit
    rng = np.random.default_rng(7 * N + K + M + c)
    wb, wi = _int_bf16(rng, (N, K))
    hb, hi = _int_bf16(rng, (M, K))
    ids = rng.integers(0, N, size=(M, c)).astype(np.int32)
    got = oracle_mod.score_ids_bf16(wb, hb, ids)
    for m in range(M):
        for j in range(c):
            want = int(np.dot(wi[ids[m, j]], hi[m]))
            assert got[m, j] == np.float32(want)


def test_score_ids_outside_the_head_are_nan(oracle_mod):
    rng = np.random.default_rng(3)
    wb, wi = _int_bf16(rng, (10, 64))
    hb, hi = _int_bf16(rng, (2, 64))
    ids = np.array([[-1, 0, 9, 10], [2147483647, -2147483648, 5, 5]], np.int32)
    got = oracle_mod.score_ids_bf16(wb, hb, ids)
    assert np.isnan(got[0, 0]) and np.isnan(got[0, 3])
    assert np.isnan(got[1, 0]) and np.isnan(got[1, 1])
    assert got[0, 1] == np.dot(wi[0], hi[0]) and got[0, 2] == np.dot(wi[9], hi[0])
    assert got[1, 2] == got[1, 3] == np.dot(wi[5], hi[1])


def test_score_id_base_names_rows_from_the_base(oracle_mod):
    # a head holding rows id_base .. id_base + N - 1 of a vocabulary: id x is
    # row x - id_base; ids below the base fall outside
    rng = np.random.default_rng(11)
    wb, wi = _int_bf16(rng, (16, 64))
    hb, hi = _int_bf16(rng, (1, 64))
    base = 1000
    ids = np.array([[1000, 1015, 999, 1016, 1007]], np.int32)
    got = oracle_mod.score_ids_bf16(wb, hb, ids, id_base=base)
    assert got[0, 0] == np.dot(wi[0], hi[0])
    assert got[0, 1] == np.dot(wi[15], hi[0])
    assert np.isnan(got[0, 2]) and np.isnan(got[0, 3])
    assert got[0, 4] == np.dot(wi[7], hi[0])


def test_score_nvfp4_hand_built_block(oracle_mod):
    # the 2 x 32 block worked out by hand from the format definitions
    q, sc, g, ones, onehot = _read_block()
    K = 32
    h1 = S.f32_to_bf16_bits(np.ones((1, K), np.float32))
    ids = np.array([[1, 0, 1, 2]], np.int32)
    got = oracle_mod.score_ids_nvfp4(q, sc, g, h1, ids)
    assert got[0, 0] == ones[1] and got[0, 1] == ones[0] and got[0, 2] == ones[1]
    assert np.isnan(got[0, 3])
    for n, k, v in onehot:
        h = np.zeros((1, K), np.float32)
        h[0, k] = 1.0
        got = oracle_mod.score_ids_nvfp4(q, sc, g, S.f32_to_bf16_bits(h),
                                         np.array([[n]], np.int32))
        assert got[0, 0] == v


def test_score_within_fp32_summation_bound_of_fp64(oracle_mod):
    # |fp32 ascending sum - exact| <= (K - 1) u sum|w h| (u = 2^-24), with the
    # products exact in fp32 (bf16 x bf16); the fp64 dot stands in for exact
    N, K, M, c = 200, 2560, 2, 64
    wb = S.normal_bf16_rows(5, N, K, 0.02)
    hb = S.hidden_bf16(6, M, K)
    rng = np.random.default_rng(8)
    ids = rng.integers(0, N, size=(M, c)).astype(np.int32)
    got = oracle_mod.score_ids_bf16(wb, hb, ids)
    w = S.bf16_bits_to_f32(wb).astype(np.float64)
    h = S.bf16_bits_to_f32(hb).astype(np.float64)
    for m in range(M):
        for j in range(c):
            prod = w[ids[m, j]] * h[m]
            bound = (K - 1) * 2.0 ** -24 * np.abs(prod).sum()
            assert abs(float(got[m, j]) - prod.sum()) <= bound
