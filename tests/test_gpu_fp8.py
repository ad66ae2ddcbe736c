"""GPU parity of the FP8 (E4M3, one tensor scale) head against the oracle:
bit-exact argmax, top-k and logits on integer heads with power-of-two
scales, at the unrolled widths and at ragged run-time widths, chunked hidden
rows; quantized gaussian heads under the parity rule; candidate scores; the
trim gather; and a full-vocabulary 248,320 x 2,560 FP8 head in the shape the
benchmark times (M = 1 and 3, argmax and top-4)."""
import numpy as np
import pytest

import synthetic as S
from parity import check_argmax, check_topk
from test_oracle_fp8 import _int_e4m3

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


CASES = [
    # N, K, M, g: unrolled widths at M <= 4, run-time widths, chunked M
    (1, 2560, 1, 1.0), (300, 2560, 3, 0.5), (4099, 5120, 4, 2.0), (2047, 5120, 1, 0.25),
    (513, 320, 5, 1.0), (70, 64, 8, 1.0), (1000, 1088, 2, 4.0), (3001, 2560, 13, 1.0),
]


@pytest.mark.parametrize("N,K,M,g", CASES)
def test_fp8_exact_integer_head_bit_exact(dvl, oracle_mod, N, K, M, g):
    # integer codes (|w| <= 16) and hidden values (|h| <= 8), a power-of-two
    # scale: every sum is an exact multiple of a power of two on both sides,
    # so ids, logits and ties agree bit for bit
    rng = np.random.default_rng(N + K + M)
    q, _ = _int_e4m3(rng, (N, K))
    h = S.f32_to_bf16_bits(rng.integers(-8, 9, size=(M, K)).astype(np.float32))
    d2t = rng.permutation(3 * N + 7)[:N].astype(np.int32)
    head = dvl.Head(dev(q), fmt="fp8", global_scale=g, V=3 * N + 7, d2t=dev(d2t))
    L, _ = oracle_mod.logits_fp8(q, g, h)
    ids, vals = dvl.draft_argmax(head, dev(h))
    o_ids, o_vals = oracle_mod.argmax(L, d2t)
    assert np.array_equal(ids.cpu().numpy(), o_ids)
    assert np.array_equal(vals.cpu().numpy(), o_vals)
    k = min(4, N)
    ids, vals = dvl.draft_topk(head, dev(h), k)
    o_ids, o_vals, _ = oracle_mod.topk(L, k, d2t)
    assert np.array_equal(ids.cpu().numpy(), o_ids)
    assert np.array_equal(vals.cpu().numpy(), o_vals)


@pytest.mark.parametrize("N,K,M", [(40, 64, 1), (3000, 5120, 3), (777, 1088, 4), (2000, 2560, 6)])
def test_fp8_quantized_head(dvl, oracle_mod, N, K, M):
    wb = S.normal_bf16_rows(N + 7, N, K, 0.02)
    q, g = S.quantize_fp8(wb)
    h = S.hidden_bf16(N + 8, M, K)
    rng = np.random.default_rng(N + 9)
    d2t = rng.permutation(100_000)[:N].astype(np.int32)
    head = dvl.Head(dev(q), fmt="fp8", global_scale=g, V=100_000, d2t=dev(d2t))
    L, _ = oracle_mod.logits_fp8(q, g, h)
    ids, vals = dvl.draft_argmax(head, dev(h))
    check_argmax(oracle_mod, L, d2t, ids.cpu().numpy(), vals.cpu().numpy())
    if N >= 4:
        ids, vals = dvl.draft_topk(head, dev(h), 4)
        check_topk(oracle_mod, L, d2t, 4, ids.cpu().numpy(), vals.cpu().numpy())


def test_fp8_scores(dvl, oracle_mod):
    # exact on an integer head; within twice the fp32 summation bound on a
    # quantized one (both sides sum exact products)
    rng = np.random.default_rng(21)
    q, _ = _int_e4m3(rng, (500, 2560))
    h = S.f32_to_bf16_bits(rng.integers(-8, 9, size=(3, 2560)).astype(np.float32))
    ids = rng.integers(-3, 503, size=(3, 40)).astype(np.int32)
    head = dvl.Head(dev(q), fmt="fp8", global_scale=0.5)
    got = dvl.score_ids(head, dev(h), dev(ids)).cpu().numpy()
    want = oracle_mod.score_ids_fp8(q, 0.5, h, ids)
    assert np.array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    assert np.array_equal(got[ok], want[ok])
    N, K = 3000, 5120
    qn, g = S.normal_fp8_rows(22, N, K, 0.02)
    hn = S.hidden_bf16(23, 4, K)
    idn = S.candidate_ids(24, N, 4, 32)
    got = dvl.score_ids(dvl.Head(dev(qn), fmt="fp8", global_scale=g), dev(hn),
                        dev(idn)).cpu().numpy()
    want = oracle_mod.score_ids_fp8(qn, g, hn, idn)
    e4 = np.array([oracle_mod.e4m3(b) for b in range(256)])
    hf = S.bf16_bits_to_f32(hn).astype(np.float64)
    for m in range(4):
        for j in range(32):
            prod = e4[qn[idn[m, j]]] * g * hf[m]
            assert abs(float(got[m, j]) - float(want[m, j])) <= 2 * K * U * np.abs(prod).sum()


def test_fp8_trim_and_learn_copy_rows(dvl, oracle_mod):
    V, K = 2000, 640
    q, g = S.normal_fp8_rows(30, V, K, 0.02)
    rng = np.random.default_rng(31)
    ranks = rng.permutation(V)[:300].astype(np.int32)
    w_trim, s_trim, d2t, ndup = dvl.trim_head(dev(q), ranks, fmt="fp8")
    assert s_trim is None and ndup == 0
    assert oracle_mod.check_trim(q, ranks, w_trim.cpu().numpy(), d2t.cpu().numpy()) == 0
    sl = dvl.Shortlist(dev(q), ranks, capacity=350, fmt="fp8", global_scale=g)
    learned = sl.learn(rng.integers(0, V, size=100))
    torch.cuda.synchronize()
    all_ids = np.concatenate([ranks, learned]).astype(np.int32)
    assert oracle_mod.check_trim(q, all_ids, sl.w[:sl.n].cpu().numpy(),
                                 sl.d2t[:sl.n].cpu().numpy()) == 0
    h = S.hidden_bf16(32, 2, K)
    L, _ = oracle_mod.logits_fp8(q[all_ids], g, h)
    ids, vals = dvl.draft_argmax(sl.head(), dev(h))
    check_argmax(oracle_mod, L, all_ids, ids.cpu().numpy(), vals.cpu().numpy())


@pytest.fixture(scope="module")
def fp8_full(dvl):
    q, g = S.normal_fp8_rows(1, S.V_FULL, 2560, 0.02)
    return q, g, dvl.Head(dev(q), fmt="fp8", global_scale=g, V=S.V_FULL)


@pytest.mark.parametrize("M", [1, 3])
def test_fp8_fullvocab_argmax_and_top4(dvl, oracle_mod, fp8_full, M):
    q, g, head = fp8_full
    h = S.hidden_bf16(101 + M, M, 2560)
    L, _ = oracle_mod.logits_fp8(q, g, h)
    ids, vals = dvl.draft_argmax(head, dev(h), ws=dvl.make_workspace(M, 1))
    rep = check_argmax(oracle_mod, L, None, ids.cpu().numpy(), vals.cpu().numpy())
    print(f"[parity] fp8 full vocab M={M}: {rep}")
    ids, vals = dvl.draft_topk(head, dev(h), 4, ws=dvl.make_workspace(M, 4))
    check_topk(oracle_mod, L, None, 4, ids.cpu().numpy(), vals.cpu().numpy())


@pytest.mark.parametrize("K,M", [(2560, 1), (5120, 3)])
def test_fp8_head_16_byte_aligned_only(dvl, oracle_mod, K, M):
    # the same rows at a 32-byte aligned address and 16 bytes into a buffer
    # (the least alignment a head may have): identical, exact results
    N = 3001
    rng = np.random.default_rng(K + M + 5)
    q, _ = _int_e4m3(rng, (N, K))
    h = S.f32_to_bf16_bits(rng.integers(-8, 9, size=(M, K)).astype(np.float32))
    flat = torch.empty(N * K + 16, dtype=torch.uint8, device="cuda")
    flat[16:] = dev(q).view(-1)
    q16 = flat[16:].view(N, K)
    assert q16.data_ptr() % 32 == 16
    L, _ = oracle_mod.logits_fp8(q, 0.5, h)
    for wq in (dev(q), q16):
        head = dvl.Head(wq, fmt="fp8", global_scale=0.5)
        ids, vals = dvl.draft_topk(head, dev(h), 4)
        o_ids, o_vals, _ = oracle_mod.topk(L, 4, None)
        assert np.array_equal(ids.cpu().numpy(), o_ids)
        assert np.array_equal(vals.cpu().numpy(), o_vals)
        ids, vals = dvl.draft_argmax(head, dev(h))
        o_ids, o_vals = oracle_mod.argmax(L, None)
        assert np.array_equal(ids.cpu().numpy(), o_ids)
        assert np.array_equal(vals.cpu().numpy(), o_vals)
