"""GPU parity at small sizes: exact-integer heads (bit-exact ids and logits,
many exact ties, non-monotone d2t), ragged tails, the degenerate shapes, the
NVFP4 hand-built block, a self-cleaning workspace and a head split by rows
whose parts are combined on the host."""
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


def int_bf16(rng, shape, lo=-4, hi=4):
    x = rng.integers(lo, hi + 1, size=shape).astype(np.float32)
    return S.f32_to_bf16_bits(x)


CASES = [
    # N, K, M, d2t kind
    (1, 64, 1, "none"), (2, 64, 3, "perm"), (5, 128, 2, "perm"), (31, 192, 4, "none"),
    (64, 256, 1, "perm"), (257, 320, 3, "perm"), (1000, 64, 8, "none"),
    (3001, 256, 5, "perm"), (4099, 576, 1, "perm"), (777, 128, 9, "perm"),
    (2048, 192, 13, "none"), (513, 64, 32, "perm"), (20000, 128, 2, "perm"),
    # short heads at the unrolled widths, one and two rows: the grid that
    # gives every warp two full row groups (fewer blocks than the full grid)
    (15000, 2560, 2, "perm"), (16000, 5120, 1, "none"),
    # three rows at 2,560: h staged in two parts around a block barrier,
    # reached by warps without rows too (40 rows leave most of them empty)
    (16000, 2560, 3, "perm"), (40, 2560, 3, "none"),
]


@pytest.mark.parametrize("N,K,M,kind", CASES)
def test_exact_integer_head_bit_exact(dvl, oracle_mod, N, K, M, kind):
    # small-integer weights and hidden values: every sum is an integer below
    # 2^24, so both sides are exact and must agree bit for bit, ties included
    rng = np.random.default_rng(N * 7 + K + M)
    w = int_bf16(rng, (N, K))
    h = int_bf16(rng, (M, K))
    d2t = rng.permutation(5 * N + 10)[:N].astype(np.int32) if kind == "perm" else None
    V = 5 * N + 10 if kind == "perm" else N
    head = dvl.Head(dev(w), V=V, d2t=dev(d2t) if d2t is not None else None)
    L, _ = oracle_mod.logits_bf16(w, h)
    ids, vals = dvl.draft_argmax(head, dev(h))
    o_ids, o_vals = oracle_mod.argmax(L, d2t)
    assert np.array_equal(ids.cpu().numpy(), o_ids)
    assert np.array_equal(vals.cpu().numpy(), o_vals)
    for k in sorted({1, 2, min(4, N)}):
        if k > N:
            continue
        ids, vals = dvl.draft_topk(head, dev(h), k)
        o_ids, o_vals, _ = oracle_mod.topk(L, k, d2t)
        assert np.array_equal(ids.cpu().numpy(), o_ids), k
        assert np.array_equal(vals.cpu().numpy(), o_vals), k


@pytest.mark.parametrize("N,K,M", [(50, 64, 1), (4000, 2560, 3), (1001, 5120, 4), (300, 24576, 2),
                                   (9000, 2560, 32)])
def test_gaussian_head_within_tolerance(dvl, oracle_mod, N, K, M):
    w = S.normal_bf16_rows(N + K, N, K, 0.02)
    h = S.hidden_bf16(N + K, M, K)
    rng = np.random.default_rng(N)
    d2t = rng.permutation(300_000)[:N].astype(np.int32)
    head = dvl.Head(dev(w), V=300_000, d2t=dev(d2t))
    L, _ = oracle_mod.logits_bf16(w, h)
    ids, vals = dvl.draft_argmax(head, dev(h))
    check_argmax(oracle_mod, L, d2t, ids.cpu().numpy(), vals.cpu().numpy())
    ids, vals = dvl.draft_topk(head, dev(h), 4)
    check_topk(oracle_mod, L, d2t, 4, ids.cpu().numpy(), vals.cpu().numpy())


def _golden_block_padded():
    """The hand-built NVFP4 block (K=32) padded to K=64 with zero blocks."""
    import test_oracle_pins as P
    q, sc, g, ones, onehot = P._read_block()
    q64 = np.zeros((q.shape[0], 32), np.uint8)
    q64[:, :16] = q
    s64 = np.zeros((sc.shape[0], 4), np.uint8)
    s64[:, :2] = sc
    return q64, s64, g, ones, onehot


def test_nvfp4_hand_built_block_on_gpu(dvl):
    q, sc, g, ones, onehot = _golden_block_padded()
    K = 64
    head = dvl.Head(dev(q), scales=dev(sc), global_scale=g, V=2)
    h1 = S.f32_to_bf16_bits(np.ones((1, K), np.float32))
    ids, vals = dvl.draft_topk(head, dev(h1), 2)
    want = sorted(ones.items(), key=lambda t: -t[1])
    assert ids.cpu().tolist()[0] == [n for n, _ in want]
    assert vals.cpu().tolist()[0] == [v for _, v in want]
    for n, k, v in onehot:
        h = np.zeros((1, K), np.float32)
        h[0, k] = 1.0
        ids, vals = dvl.draft_topk(head, dev(S.f32_to_bf16_bits(h)), 2)
        got = dict(zip(ids.cpu().tolist()[0], vals.cpu().tolist()[0]))
        assert got[n] == v, (n, k)


@pytest.mark.parametrize("N,K,M", [(40, 64, 1), (3000, 5120, 3), (777, 1088, 4), (2000, 2560, 6)])
def test_nvfp4_random_head(dvl, oracle_mod, N, K, M):
    wb = S.normal_bf16_rows(N, N, K, 0.02)
    q, sc, g = S.quantize_nvfp4(wb)
    h = S.hidden_bf16(N + 1, M, K)
    rng = np.random.default_rng(N + 5)
    d2t = rng.permutation(100_000)[:N].astype(np.int32)
    head = dvl.Head(dev(q), scales=dev(sc), global_scale=g, V=100_000, d2t=dev(d2t))
    L, _ = oracle_mod.logits_nvfp4(q, sc, g, h)
    ids, vals = dvl.draft_argmax(head, dev(h))
    check_argmax(oracle_mod, L, d2t, ids.cpu().numpy(), vals.cpu().numpy())
    if N >= 4:
        ids, vals = dvl.draft_topk(head, dev(h), 4)
        check_topk(oracle_mod, L, d2t, 4, ids.cpu().numpy(), vals.cpu().numpy())


def test_workspace_is_self_cleaning_and_recovers_from_a_stale_ticket(dvl, oracle_mod):
    rng = np.random.default_rng(9)
    N, K, M = 5000, 256, 3
    ws = dvl.make_workspace(8, 4)
    for it in range(3):
        w = int_bf16(rng, (N, K))
        h = int_bf16(rng, (M, K))
        head = dvl.Head(dev(w))
        L, _ = oracle_mod.logits_bf16(w, h)
        ids, vals = dvl.draft_argmax(head, dev(h), ws=ws)
        assert np.array_equal(ids.cpu().numpy(), oracle_mod.argmax(L)[0])
        ids, vals = dvl.draft_topk(head, dev(h), 3, ws=ws)
        assert np.array_equal(ids.cpu().numpy(), oracle_mod.topk(L, 3)[0])
    torch.cuda.synchronize()
    assert int(ws[:8].view(torch.int64).item()) == 0  # ticket and status back to 0
    assert bool((ws[256:512] == 0).all())             # best keys swapped back to 0
    # a stale ticket (as a call cut short would leave): the call returns (no
    # block waits), and re-initialising the workspace restores exact results
    ws[0] = 5
    dvl.draft_argmax(head, dev(h), ws=ws)
    torch.cuda.synchronize()
    dvl.workspace_init(ws)
    ids, _ = dvl.draft_argmax(head, dev(h), ws=ws)
    assert np.array_equal(ids.cpu().numpy(), oracle_mod.argmax(L)[0])


def test_row_split_combined_on_host_equals_whole_head(dvl, oracle_mod):
    # the head split by rows over G parts (as G GPUs would hold it): each
    # part's argmax, combined by (logit desc, id asc), is the whole head's
    N, K, M, G = 10_000, 512, 3, 3
    w = S.normal_bf16_rows(77, N, K, 0.02)
    h = S.hidden_bf16(77, M, K)
    head = dvl.Head(dev(w))
    hd = dev(h)
    whole = dvl.draft_argmax(head, hd)
    parts = []
    for g in range(G):
        n0, n1 = N * g // G, N * (g + 1) // G
        parts.append(dvl.draft_argmax(head.slice_rows(n0, n1), hd))
    for m in range(M):
        cands = [(-float(v[m]), int(i[m])) for i, v in parts]
        best = min(cands)
        assert best[1] == int(whole[0][m]) and -best[0] == float(whole[1][m])


def test_non_default_stream_and_preallocated_outputs(dvl, oracle_mod):
    rng = np.random.default_rng(4)
    w = int_bf16(rng, (3000, 256))
    h = int_bf16(rng, (2, 256))
    L, _ = oracle_mod.logits_bf16(w, h)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        head = dvl.Head(dev(w))
        ids = torch.full((2,), -7, dtype=torch.int32, device="cuda")
        vals = torch.zeros(2, dtype=torch.float32, device="cuda")
        ws = dvl.make_workspace(2, 1)
        dvl.draft_argmax(head, dev(h), ids=ids, logits=vals, ws=ws)
    s.synchronize()
    assert np.array_equal(ids.cpu().numpy(), oracle_mod.argmax(L)[0])


def test_gpu_side_argument_errors(dvl):
    w = torch.zeros((100, 256), dtype=torch.int16, device="cuda")
    head = dvl.Head(w)
    h = torch.zeros((2, 256), dtype=torch.int16, device="cuda")
    small = torch.zeros(64, dtype=torch.uint8, device="cuda")
    with pytest.raises(dvl.DvlError) as e:
        dvl.draft_argmax(head, h, ws=small)
    assert e.value.status == 4
    with pytest.raises(dvl.DvlError) as e:
        dvl.trim_head(w, [0, 5, 100])
    assert e.value.status == 2


def test_trim_head_small_with_duplicates(dvl, oracle_mod):
    V, K = 3000, 320
    wfull = S.normal_bf16_rows(5, V, K, 0.02)
    rng = np.random.default_rng(5)
    ranks = np.concatenate([rng.permutation(V)[:900], [11, 11, 2999]]).astype(np.int32)
    w_trim, _, d2t, ndup = dvl.trim_head(dev(wfull), ranks)
    assert ndup == 1 + int(11 in ranks[:900]) + int(2999 in ranks[:900])
    got = w_trim.cpu().numpy().view(np.uint16)
    assert oracle_mod.check_trim(wfull, ranks, got, d2t.cpu().numpy()) == 0
    # NVFP4: codes and scales gathered together
    q, sc, g = S.quantize_nvfp4(wfull)
    q_t, s_t, d2t2, _ = dvl.trim_head(dev(q), ranks, scales=dev(sc))
    assert oracle_mod.check_trim(q, ranks, q_t.cpu().numpy(), d2t2.cpu().numpy()) == 0
    assert oracle_mod.check_trim(sc, ranks, s_t.cpu().numpy(), None) == 0


@pytest.mark.parametrize("static", [False, True])
def test_back_to_back_calls_with_overlapping_launches(dvl, oracle_mod, static):
    # consecutive calls may overlap (programmatic dependent launch); each must
    # still see its own hidden rows and a clean workspace, and a static head
    # may be streamed before the previous call ends
    rng = np.random.default_rng(21 + static)
    N, K = 16000, 2560
    w = int_bf16(rng, (N, K))
    head = dvl.Head(dev(w), static=static)
    ws = dvl.make_workspace(4, 4)
    hs = [int_bf16(rng, (M, K)) for M in (1, 3, 2, 1, 3, 4)]
    outs = []
    for h in hs:
        ids = torch.empty(h.shape[0], dtype=torch.int32, device="cuda")
        vals = torch.empty(h.shape[0], dtype=torch.float32, device="cuda")
        dvl.draft_argmax(head, dev(h), ids=ids, logits=vals, ws=ws)
        outs.append((ids, vals))
    for h, (ids, vals) in zip(hs, outs):
        L, _ = oracle_mod.logits_bf16(w, h)
        o_ids, o_vals = oracle_mod.argmax(L)
        assert np.array_equal(ids.cpu().numpy(), o_ids)
        assert np.array_equal(vals.cpu().numpy(), o_vals)


def test_trim_then_argmax_without_synchronizing(dvl, oracle_mod):
    # the argmax right after trim_head on the same stream must read the
    # trimmed rows, not what the buffer held before
    V, K = 6000, 2560
    rng = np.random.default_rng(33)
    wfull = int_bf16(rng, (V, K))
    wfull_d = dev(wfull)
    h = int_bf16(rng, (2, K))
    hd = dev(h)
    for it in range(3):
        ranks = rng.permutation(V)[:2500].astype(np.int32)
        w_trim, _, d2t, _ = dvl.trim_head(wfull_d, ranks)
        ids, vals = dvl.draft_argmax(dvl.Head(w_trim, V=V, d2t=d2t), hd)
        L, _ = oracle_mod.logits_bf16(wfull[ranks], h)
        o_ids, o_vals = oracle_mod.argmax(L, ranks)
        assert np.array_equal(ids.cpu().numpy(), o_ids), it
        assert np.array_equal(vals.cpu().numpy(), o_vals), it


def test_workspace_status_reads_and_clears(dvl, oracle_mod):
    # a fresh workspace reports nothing; a status bit written from the host
    # (standing in for a kernel's record) is reported once, then cleared;
    # ordinary calls, the tensor-core one included, record nothing
    ws = dvl.make_workspace(8, 4)
    assert dvl.workspace_status(ws) == 0
    ws[4:8].view(torch.int32)[0] = 1 << 6  # DVL_ERR_TIMEOUT
    assert dvl.workspace_status(ws) == 1 << 6
    assert dvl.workspace_status(ws) == 0
    rng = np.random.default_rng(12)
    w = int_bf16(rng, (3000, 256))
    head = dvl.Head(dev(w))
    for M in (1, 8):
        h = int_bf16(rng, (M, 256))
        L, _ = oracle_mod.logits_bf16(w, h)
        ids, _ = dvl.draft_argmax(head, dev(h), ws=ws)
        assert np.array_equal(ids.cpu().numpy(), oracle_mod.argmax(L)[0])
    assert dvl.workspace_status(ws) == 0


def test_two_streams_with_their_own_workspaces(dvl, oracle_mod):
    # calls interleaved on two streams, each with its own workspace (the
    # documented rule for concurrent calls): CUDA-core, tensor-core and
    # low-bit kernels, argmax and top-k, all as the oracle says
    rng = np.random.default_rng(33)
    N, K = 6000, 256
    w = int_bf16(rng, (N, K))
    head = dvl.Head(dev(w))
    q, sc, g = S.quantize_nvfp4(S.normal_bf16_rows(34, N, K, 0.02))
    head4 = dvl.Head(dev(q), scales=dev(sc), global_scale=g)
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    wss = [dvl.make_workspace(32, 4), dvl.make_workspace(32, 4)]
    torch.cuda.synchronize()
    inputs = []
    for it in range(12):
        M = [1, 3, 8, 20][it % 4]
        h = int_bf16(rng, (M, K))
        inputs.append((it, h, dev(h)))
    torch.cuda.synchronize()  # every input in place; the launches below overlap
    jobs = []
    for it, h, hd in inputs:
        sidx = it % 2
        k = 1 if it % 3 else 4
        hh = head4 if it % 5 == 4 else head
        with torch.cuda.stream(streams[sidx]):
            ids = torch.empty((h.shape[0], k), dtype=torch.int32, device="cuda")
            vals = torch.empty((h.shape[0], k), dtype=torch.float32, device="cuda")
            if k == 1:
                dvl.draft_argmax(hh, hd, ids=ids.view(-1), logits=vals.view(-1), ws=wss[sidx],
                                 stream=streams[sidx])
            else:
                dvl.draft_topk(hh, hd, k, ids=ids, logits=vals, ws=wss[sidx], stream=streams[sidx])
        jobs.append((hh is head4, h, k, (ids, vals)))
    torch.cuda.synchronize()
    from parity import check_argmax, check_topk
    for is4, h, k, (ids, vals) in jobs:
        if is4:
            L, _ = oracle_mod.logits_nvfp4(q, sc, g, h)
            if k == 1:
                check_argmax(oracle_mod, L, None, ids.cpu().numpy().ravel(),
                             vals.cpu().numpy().ravel())
            else:
                check_topk(oracle_mod, L, None, k, ids.cpu().numpy(), vals.cpu().numpy())
        else:
            L, _ = oracle_mod.logits_bf16(w, h)
            o_ids, o_vals, _ = oracle_mod.topk(L, k)
            got = ids.cpu().numpy().reshape(o_ids.shape)
            assert np.array_equal(got, o_ids)
    for ws in wss:
        assert dvl.workspace_status(ws) == 0
