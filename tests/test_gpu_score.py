"""GPU parity of candidate scoring (dvl_score_ids) against the oracle:
exact-integer heads bit for bit at the unrolled widths and at ragged
run-time widths, NaN for ids outside the head, head slices (id_base), the
hand-built NVFP4 block exactly, and gaussian / quantized heads within the
fp32 summation bound.

Tolerance (floating point): both sides sum the same exact products (bf16 x
bf16 is exact in fp32) in different orders, so each lies within
(K - 1) u sum_k |w_k h_k| of the exact dot (u = 2^-24) and they differ by at
most twice that.  The NVFP4 kernel also rounds each 16-weight block sum once
more when it applies the block scale, and the oracle rounds each weight
times the tensor scale: the bound is doubled again for NVFP4."""
import numpy as np
import pytest

import synthetic as S

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

U = 2.0 ** -24


@pytest.fixture(scope="module")
def dvl():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from draft_vocab_lm_gb300 import build
    build.build()
    import draft_vocab_lm_gb300 as d
    return d


def dev(a):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).cuda()


def int_bf16(rng, shape, lo=-8, hi=8):
    return S.f32_to_bf16_bits(rng.integers(lo, hi + 1, size=shape).astype(np.float32))


def abs_dot(w_f64, h_f64, ids, id_base=0):
    """sum_k |w[id - id_base][k] h[m][k]| per (m, j); 0 where the id is outside."""
    M, c = ids.shape
    N = w_f64.shape[0]
    out = np.zeros((M, c))
    for m in range(M):
        for j in range(c):
            r = int(ids[m, j]) - id_base
            if 0 <= r < N:
                out[m, j] = np.abs(w_f64[r] * h_f64[m]).sum()
    return out


def assert_scores(got, want, bound):
    nan_w = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan_w)
    err = np.abs(got[~nan_w].astype(np.float64) - want[~nan_w])
    assert np.all(err <= bound[~nan_w]), float((err - bound[~nan_w]).max())


@pytest.mark.parametrize("N,K,M,c", [
    (1, 2560, 1, 1), (300, 2560, 3, 7), (5000, 5120, 4, 100), (64, 5120, 32, 9),
    (70, 64, 2, 33), (513, 320, 5, 17), (100, 1088, 1, 200), (40, 24576, 2, 3),
])
def test_score_exact_integer_bit_exact(dvl, oracle_mod, N, K, M, c):
    # small integers: every partial sum is an integer below 2^24 in any order
    rng = np.random.default_rng(N + 3 * K + 7 * M + c)
    lo, hi = (-2, 2) if K > 8192 else (-8, 8)
    w = int_bf16(rng, (N, K), lo, hi)
    h = int_bf16(rng, (M, K), lo, hi)
    ids = rng.integers(-2, N + 2, size=(M, c)).astype(np.int32)
    ids[0, 0] = N - 1
    head = dvl.Head(dev(w))
    got = dvl.score_ids(head, dev(h), dev(ids)).cpu().numpy()
    want = oracle_mod.score_ids_bf16(w, h, ids)
    assert np.array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    assert np.array_equal(got[ok], want[ok])


def test_score_extreme_ids_are_nan(dvl, oracle_mod):
    rng = np.random.default_rng(1)
    w = int_bf16(rng, (50, 2560))
    h = int_bf16(rng, (2, 2560))
    ids = np.array([[-2147483648, 2147483647, 50, -1, 0, 49]] * 2, np.int32)
    got = dvl.score_ids(dvl.Head(dev(w)), dev(h), dev(ids)).cpu().numpy()
    want = oracle_mod.score_ids_bf16(w, h, ids)
    assert np.isnan(got[:, :4]).all() and np.array_equal(got[:, 4:], want[:, 4:])


def test_score_head_slice_uses_id_base(dvl, oracle_mod):
    # a slice of a head keeps full ids: rows n0 .. n1 - 1 answer ids n0 .. n1 - 1
    rng = np.random.default_rng(2)
    N, K = 1000, 2560
    w = int_bf16(rng, (N, K))
    h = int_bf16(rng, (3, K))
    full = dvl.Head(dev(w))
    part = full.slice_rows(200, 700)
    ids = rng.integers(150, 750, size=(3, 64)).astype(np.int32)
    got = dvl.score_ids(part, dev(h), dev(ids)).cpu().numpy()
    want = oracle_mod.score_ids_bf16(w[200:700], h, ids, id_base=200)
    assert np.array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    assert np.array_equal(got[ok], want[ok])
    assert np.isnan(got[ids < 200]).all() and np.isnan(got[ids >= 700]).all()


@pytest.mark.parametrize("N,K,M,c", [(20000, 2560, 16, 64), (4096, 5120, 4, 128),
                                     (3000, 448, 3, 50)])
def test_score_gaussian_within_summation_bound(dvl, oracle_mod, N, K, M, c):
    w = S.normal_bf16_rows(40 + K, N, K, 0.02)
    h = S.hidden_bf16(41, M, K)
    ids = S.candidate_ids(42, N, M, c)
    got = dvl.score_ids(dvl.Head(dev(w)), dev(h), dev(ids)).cpu().numpy()
    want = oracle_mod.score_ids_bf16(w, h, ids)
    wf = S.bf16_bits_to_f32(w).astype(np.float64)
    hf = S.bf16_bits_to_f32(h).astype(np.float64)
    assert_scores(got, want, 2 * (K - 1) * U * abs_dot(wf, hf, ids))


def test_score_nvfp4_hand_built_block(dvl, oracle_mod):
    from test_oracle_pins import _read_block
    q, sc, g, ones, onehot = _read_block()
    # repeat the two 32-wide rows along K so the width is a multiple of 64
    q2 = np.tile(q, (1, 2))
    sc2 = np.tile(sc, (1, 2))
    K = 64
    head = dvl.Head(dev(q2), scales=dev(sc2), global_scale=g)
    h1 = S.f32_to_bf16_bits(np.ones((1, K), np.float32))
    ids = np.array([[0, 1, 2, -1, 1]], np.int32)
    got = dvl.score_ids(head, dev(h1), dev(ids)).cpu().numpy()
    assert got[0, 0] == 2 * ones[0] and got[0, 1] == 2 * ones[1] and got[0, 4] == 2 * ones[1]
    assert np.isnan(got[0, 2]) and np.isnan(got[0, 3])
    for n, k, v in onehot:
        h = np.zeros((1, K), np.float32)
        h[0, k] = 1.0
        got = dvl.score_ids(head, dev(S.f32_to_bf16_bits(h)),
                            dev(np.array([[n]], np.int32))).cpu().numpy()
        assert got[0, 0] == v


@pytest.mark.parametrize("N,K,M,c", [(4096, 5120, 3, 50), (2000, 2560, 8, 40),
                                     (1500, 320, 2, 30)])
def test_score_nvfp4_within_bound(dvl, oracle_mod, N, K, M, c):
    wb = S.normal_bf16_rows(50 + K, N, K, 0.02)
    q, sc, g = S.quantize_nvfp4(wb)
    h = S.hidden_bf16(51, M, K)
    ids = S.candidate_ids(52, N, M, c)
    ids[0, :3] = [-1, N, 0]
    head = dvl.Head(dev(q), scales=dev(sc), global_scale=g)
    got = dvl.score_ids(head, dev(h), dev(ids)).cpu().numpy()
    want = oracle_mod.score_ids_nvfp4(q, sc, g, h, ids)
    # |w| per weight from the oracle's decode tables, for the bound only
    e2m1 = np.array([oracle_mod.e2m1(x) for x in range(16)])
    e4m3 = np.array([oracle_mod.e4m3(x) for x in range(256)])
    codes = np.stack([q & 0xF, q >> 4], axis=-1).reshape(N, K)
    wdeq = e2m1[codes] * np.repeat(e4m3[sc], 16, axis=1) * g
    hf = S.bf16_bits_to_f32(h).astype(np.float64)
    assert_scores(got, want, 4 * (K + 16) * U * abs_dot(wdeq, hf, ids))
