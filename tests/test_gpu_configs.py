"""GPU parity on the five workloads at their full sizes, through the same
library calls (and so the same launch configuration) the benchmark times,
against the oracle run in full on every row.

c1  16,000-row shortlist of a 248,320 x 2,560 head (trim, then argmax, M=1)
c2  the full 248,320 x 2,560 head, M in {1, 3}, argmax and top-4; candidate
    scores of 16 hidden rows x 32 candidates through it
c3  32,768-row FR-Spec trim of a 248,320 x 5,120 head, ranks built on the
    host from a Zipf token stream, M in {1, 2, 3, 4}
c4  52,755-row union list, M in {8, 16, 32}, planted near-ties, argmax and
    top-4
c5  NVFP4 32,768 x 5,120 head with a rank-order d2t, M in {1, 3}
"""
import numpy as np
import pytest

import synthetic as S
from parity import check_argmax, check_topk

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


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


def report(name, rep):
    print(f"[parity] {name}: {rep}")


def test_c1_shortlist16k(dvl, oracle_mod):
    wl = S.c1()
    wfull_d = dev(wl.w_full)
    w_trim, _, d2t, ndup = dvl.trim_head(wfull_d, wl.ranks)
    assert ndup == 0
    got = w_trim.cpu().numpy().view(np.uint16)
    assert oracle_mod.check_trim(wl.w_full, wl.ranks, got, d2t.cpu().numpy()) == 0
    del wfull_d
    head = dvl.Head(w_trim, V=wl.V, d2t=d2t)
    h = wl.h[1]
    L, _ = oracle_mod.logits_bf16(wl.w, h)
    ws = dvl.make_workspace(1, 1)
    ids, vals = dvl.draft_argmax(head, dev(h), ws=ws)
    report("c1", check_argmax(oracle_mod, L, wl.d2t, ids.cpu().numpy(), vals.cpu().numpy()))
    # shortlist semantics: the same id as the full head with off-list rows masked
    Lf, _ = oracle_mod.logits_bf16(wl.w_full, h)
    masked = np.full_like(Lf, -np.inf)
    masked[:, wl.ranks] = Lf[:, wl.ranks]
    assert oracle_mod.argmax(masked)[0][0] == oracle_mod.argmax(L, wl.d2t)[0][0]


@pytest.fixture(scope="module")
def c2(dvl):
    wl = S.c2()
    return wl, dvl.Head(dev(wl.w), V=wl.V)


def test_c2_candidate_scores(dvl, oracle_mod, c2):
    # candidate scoring through the full head, in the benchmark's shape: 16
    # hidden rows x 32 Zipf-drawn candidates; every score against the oracle
    # within twice the fp32 summation bound (both sides sum exact products)
    wl, head = c2
    M, c = 16, 32
    h = S.hidden_bf16(91, M, wl.K)
    ids = S.candidate_ids(92, wl.V, M, c)
    got = dvl.score_ids(head, dev(h), dev(ids)).cpu().numpy()
    want = oracle_mod.score_ids_bf16(wl.w, h, ids)
    hf = S.bf16_bits_to_f32(h).astype(np.float64)
    worst = 0.0
    for m in range(M):
        for j in range(c):
            prod = S.bf16_bits_to_f32(wl.w[ids[m, j]]).astype(np.float64) * hf[m]
            bound = 2 * (wl.K - 1) * 2.0 ** -24 * np.abs(prod).sum()
            err = abs(float(got[m, j]) - float(want[m, j]))
            assert err <= bound
            worst = max(worst, err / bound)
    report("c2 scores 16x32", {"pairs": M * c, "worst err / bound": round(worst, 4)})


@pytest.mark.parametrize("M", [1, 3])
def test_c2_fullvocab_argmax_and_top4(dvl, oracle_mod, c2, M):
    wl, head = c2
    h = wl.h[M]
    L, _ = oracle_mod.logits_bf16(wl.w, h)
    ids, vals = dvl.draft_argmax(head, dev(h), ws=dvl.make_workspace(M, 1))
    report(f"c2 M={M}", check_argmax(oracle_mod, L, None, ids.cpu().numpy(), vals.cpu().numpy()))
    ids, vals = dvl.draft_topk(head, dev(h), 4, ws=dvl.make_workspace(M, 4))
    report(f"c2 M={M} top4", check_topk(oracle_mod, L, None, 4, ids.cpu().numpy(),
                                          vals.cpu().numpy()))


def test_c3_frspec_trim(dvl, oracle_mod):
    wl = S.c3()
    counts = dvl.histogram(wl.extra["tokens"], wl.V)
    ranks = dvl.build_ranks(counts, wl.extra["N"])
    assert np.array_equal(ranks, oracle_mod.build_ranks(oracle_mod.histogram(
        wl.extra["tokens"], wl.V), wl.extra["N"]))
    assert np.any(np.diff(ranks) < 0)  # rank order, not sorted
    wfull_d = dev(wl.w_full)
    w_trim, _, d2t, ndup = dvl.trim_head(wfull_d, ranks)
    assert ndup == 0
    got = w_trim.cpu().numpy().view(np.uint16)
    assert oracle_mod.check_trim(wl.w_full, ranks, got, d2t.cpu().numpy()) == 0
    del wfull_d
    head = dvl.Head(w_trim, V=wl.V, d2t=d2t)
    for M in wl.Ms:
        h = wl.h[M]
        L, _ = oracle_mod.logits_bf16(got, h)
        ids, vals = dvl.draft_argmax(head, dev(h))
        report(f"c3 M={M}", check_argmax(oracle_mod, L, ranks, ids.cpu().numpy(),
                                          vals.cpu().numpy()))


def test_c4_batched_near_ties(dvl, oracle_mod):
    wl = S.c4()
    d2t = dev(wl.d2t)
    exempt_total = exact_total = 0
    for M in wl.Ms:
        W = wl.extra["w_by_M"][M]
        h = wl.h[M]
        head = dvl.Head(dev(W), V=wl.V, d2t=d2t)
        L, _ = oracle_mod.logits_bf16(W, h)
        gap, mx = oracle_mod.row_stats(L)
        assert (gap < 1e-3 * mx).any() and (gap > 1e-3 * mx).any()
        assert np.log10(gap.max() / gap.min()) >= 3
        ids, vals = dvl.draft_argmax(head, dev(h), ws=dvl.make_workspace(M, 1))
        rep = check_argmax(oracle_mod, L, wl.d2t, ids.cpu().numpy(), vals.cpu().numpy())
        report(f"c4 M={M}", rep)
        exempt_total += rep["rows_exempt"]
        exact_total += rep["rows_exact"]
        # batched top-4 in the same single pass over the head
        ids, vals = dvl.draft_topk(head, dev(h), 4, ws=dvl.make_workspace(M, 4))
        report(f"c4 M={M} top4", check_topk(oracle_mod, L, wl.d2t, 4, ids.cpu().numpy(),
                                              vals.cpu().numpy()))
    assert exempt_total > 0 and exact_total > 0


def test_c5_nvfp4(dvl, oracle_mod):
    wl = S.c5()
    head = dvl.Head(dev(wl.q), scales=dev(wl.scales), global_scale=wl.g, V=wl.V,
                    d2t=dev(wl.d2t))
    for M in wl.Ms:
        h = wl.h[M]
        L, _ = oracle_mod.logits_nvfp4(wl.q, wl.scales, wl.g, h)
        ids, vals = dvl.draft_argmax(head, dev(h))
        report(f"c5 M={M}", check_argmax(oracle_mod, L, wl.d2t, ids.cpu().numpy(),
                                          vals.cpu().numpy()))
        ids, vals = dvl.draft_topk(head, dev(h), 4)
        report(f"c5 M={M} top4", check_topk(oracle_mod, L, wl.d2t, 4, ids.cpu().numpy(),
                                             vals.cpu().numpy()))
