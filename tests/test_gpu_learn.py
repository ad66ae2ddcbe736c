"""GPU checks of learning escaped ids into spare rows of a trimmed head
(dvl_learn_rows and the Shortlist helper): the learned rows are the full
head's rows byte for byte with d2t set, in bf16 and NVFP4; after a learn
the draft argmax covers the list plus the learned ids exactly as the oracle
over that id set says, with no synchronisation between the learn and the
next call on the stream."""
import numpy as np
import pytest

import synthetic as S
from parity import check_argmax

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


@pytest.mark.parametrize("dtype", ["bf16", "nvfp4"])
def test_learned_rows_are_the_full_rows(dvl, oracle_mod, dtype):
    V, K = 3000, 512
    wb = S.normal_bf16_rows(60, V, K, 0.02)
    rng = np.random.default_rng(61)
    ranks = rng.permutation(V)[:1000].astype(np.int32)
    if dtype == "bf16":
        sl = dvl.Shortlist(dev(wb), ranks, capacity=1200)
        full_rows, row_bytes = wb, K * 2
    else:
        q, sc, g = S.quantize_nvfp4(wb)
        sl = dvl.Shortlist(dev(q), ranks, capacity=1200, scales=dev(sc), global_scale=g)
        full_rows = q
    # a batch of emitted ids: some already listed, repeats, some new
    emitted = np.concatenate([ranks[:20], rng.integers(0, V, size=400), ranks[5:9]])
    learned = sl.learn(emitted)
    listed = set(ranks.tolist())
    expect, seen = [], set()
    for x in emitted.tolist():
        if x not in listed and x not in seen and len(expect) < 200:
            expect.append(x)
            seen.add(x)
    assert learned.tolist() == expect
    assert sl.n == 1000 + len(expect)
    torch.cuda.synchronize()
    all_ids = np.concatenate([ranks, learned]).astype(np.int32)
    got_w = sl.w[:sl.n].cpu().numpy()
    if dtype == "bf16":
        got_w = got_w.view(np.uint16)
    assert oracle_mod.check_trim(full_rows, all_ids, got_w, sl.d2t[:sl.n].cpu().numpy()) == 0
    if dtype == "nvfp4":
        assert oracle_mod.check_trim(sc, all_ids, sl.scales[:sl.n].cpu().numpy(),
                                     sl.d2t[:sl.n].cpu().numpy()) == 0
    # learning stops at the capacity
    more = sl.learn(np.arange(V))
    assert sl.n == 1200 and more.size == 1200 - 1000 - len(expect)
    assert sl.learn(np.arange(V)).size == 0


def test_learning_the_missed_ids_recovers_the_full_argmax(dvl, oracle_mod):
    # a shortlist that misses each row's full-head winner; once the winners
    # are learned the shortlist's argmax is the full head's argmax
    V, K, M = 20000, 2560, 4
    wb = S.normal_bf16_rows(70, V, K, 0.02)
    h = S.hidden_bf16(71, M, K)
    Lf, _ = oracle_mod.logits_bf16(wb, h)
    best = oracle_mod.argmax(Lf)[0]
    rng = np.random.default_rng(72)
    ranks = np.setdiff1d(rng.permutation(V)[:2000], best).astype(np.int32)
    sl = dvl.Shortlist(dev(wb), ranks, capacity=len(ranks) + 16)
    hd = dev(h)
    ws = dvl.make_workspace(M, 1)
    ids0, _ = dvl.draft_argmax(sl.head(), hd, ws=ws)
    assert not set(ids0.cpu().numpy().tolist()) & set(best.tolist())
    sl.learn(best)  # no synchronisation before the next call
    head = sl.head()
    assert not head.static
    ids, vals = dvl.draft_argmax(head, hd, ws=ws)
    active = np.concatenate([ranks, np.unique(best)]).astype(np.int32)
    L, _ = oracle_mod.logits_bf16(wb[active], h)
    check_argmax(oracle_mod, L, active, ids.cpu().numpy(), vals.cpu().numpy())
    assert np.array_equal(oracle_mod.argmax(L, active)[0], best)
    # back to static once the learned rows are in stream order
    assert sl.head().static


def test_learn_and_draft_in_a_loop_without_syncs(dvl, oracle_mod):
    # emitted token -> learn -> next draft on one stream, repeatedly
    V, K, M = 8000, 256, 1
    wb = S.normal_bf16_rows(80, V, K, 0.02)
    hs = [S.hidden_bf16(81 + i, M, K) for i in range(12)]
    rng = np.random.default_rng(82)
    ranks = rng.permutation(V)[:500].astype(np.int32)
    sl = dvl.Shortlist(dev(wb), ranks, capacity=600)
    ws = dvl.make_workspace(M, 1)
    outs = []
    for i, h in enumerate(hs):
        Lf, _ = oracle_mod.logits_bf16(wb, h)
        sl.learn(oracle_mod.argmax(Lf)[0])
        ids, vals = dvl.draft_argmax(sl.head(), dev(h), ws=ws)
        outs.append((ids, vals, sl.n))
    torch.cuda.synchronize()
    active = sl.d2t.cpu().numpy()
    for (ids, vals, n), h in zip(outs, hs):
        L, _ = oracle_mod.logits_bf16(wb[active[:n]], h)
        check_argmax(oracle_mod, L, active[:n], ids.cpu().numpy(), vals.cpu().numpy())


def test_heads_handed_out_before_the_next_draft_are_not_static(dvl, oracle_mod):
    # every head taken between a learn and the first draft call enqueued
    # after it streams nothing before its wait; once such a call is
    # enqueued, later heads may
    V, K, M = 4000, 256, 1
    wb = S.normal_bf16_rows(90, V, K, 0.02)
    h = S.hidden_bf16(91, M, K)
    ranks = np.arange(0, V, 7, dtype=np.int32)
    sl = dvl.Shortlist(dev(wb), ranks, capacity=len(ranks) + 8)
    a, b = sl.head(), sl.head()
    assert not a.static and not b.static
    dvl.draft_argmax(b, dev(h))
    assert sl.head().static
    assert sl.learn([1, 2, 1, 7]).tolist() == [1, 2]  # 7 is in the list already
    c, d = sl.head(), sl.head()
    assert not c.static and not d.static
    ids, vals = dvl.draft_argmax(d, dev(h))
    assert sl.head().static
    active = sl.d2t[:sl.n].cpu().numpy()
    L, _ = oracle_mod.logits_bf16(wb[active], h)
    check_argmax(oracle_mod, L, active, ids.cpu().numpy(), vals.cpu().numpy())
    assert sl.row_of[1] == len(ranks) and sl.row_of[2] == len(ranks) + 1
