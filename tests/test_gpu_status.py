"""Device-side checks of the draft calls, read through dvl_workspace_status,
and canaries around their outputs and workspace.

- A d2t entry outside [0, V) on the winning row: every kernel family
  returns the id as it is and sets the DVL_ERR_OUT_OF_RANGE bit of the
  workspace's status word; the next clean call leaves the word at 0 once it
  was read.  (The kernels read no memory through d2t entries, so the
  planted entry is harmless to run.)
- Canaries: ids, logits and the workspace are carved out of larger buffers
  filled with a known byte pattern; after calls of every family, every byte
  outside the call's own ranges is unchanged.
"""
import numpy as np
import pytest

import synthetic as S
from parity import check_argmax, check_topk

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

OUT_OF_RANGE_BIT = 1 << 2  # 1 << DVL_ERR_OUT_OF_RANGE


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
    return torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).cuda()


# (expected kernel family, M, N, K, dtype)
FAMILIES = [
    ("bf16-cuda-cores", 1, 3001, 2560, "bf16"),
    ("bf16-mma", 3, 20000, 2560, "bf16"),
    ("bf16-tcgen05", 8, 3001, 256, "bf16"),
    ("nvfp4-mma", 1, 3001, 5120, "nvfp4"),
    ("fp8-mma", 3, 3001, 2560, "fp8"),
]


def make_head(dvl, oracle_mod, N, K, M, dtype, seed, V):
    w = S.normal_bf16_rows(seed, N, K, 0.02)
    h = S.hidden_bf16(seed, M, K)
    if dtype == "bf16":
        L, _ = oracle_mod.logits_bf16(w, h)
        return (lambda d2t: dvl.Head(dev(w), V=V, d2t=dev(d2t))), h, L
    if dtype == "nvfp4":
        q, sc, g = S.quantize_nvfp4(w)
        L, _ = oracle_mod.logits_nvfp4(q, sc, g, h)
        return (lambda d2t: dvl.Head(dev(q), scales=dev(sc), global_scale=g, V=V,
                                     d2t=dev(d2t))), h, L
    q, g = S.quantize_fp8(w)
    L, _ = oracle_mod.logits_fp8(q, g, h)
    return (lambda d2t: dvl.Head(dev(q), fmt="fp8", global_scale=g, V=V, d2t=dev(d2t))), h, L


@pytest.mark.parametrize("family,M,N,K,dtype", FAMILIES)
@pytest.mark.parametrize("k", [1, 4])
def test_out_of_range_d2t_winner_is_reported(dvl, oracle_mod, family, M, N, K, dtype, k):
    V = 300_000
    mk, h, L = make_head(dvl, oracle_mod, N, K, M, dtype, 40 + M, V)
    d2t = np.random.default_rng(N + M).permutation(V)[:N].astype(np.int32)
    bad = d2t.copy()
    win = int(np.argmax(L[0]))
    bad[win] = -7 if k == 1 else V  # below and at the bound
    head_bad, head_ok = mk(bad), mk(d2t)
    if k == 1:
        assert dvl.draft_plan(head_ok, M, 1)[0] == family
    ws = dvl.make_workspace(M, 4)
    hd = dev(h)
    if k == 1:
        ids, _ = dvl.draft_argmax(head_bad, hd, ws=ws)
    else:
        ids, _ = dvl.draft_topk(head_bad, hd, k, ws=ws)
    torch.cuda.synchronize()
    assert int(ids.view(-1)[0]) == int(bad[win])
    assert dvl.workspace_status(ws) == OUT_OF_RANGE_BIT
    assert dvl.workspace_status(ws) == 0
    if k == 1:
        ids, vals = dvl.draft_argmax(head_ok, hd, ws=ws)
        check_argmax(oracle_mod, L, d2t, ids.cpu().numpy(), vals.cpu().numpy())
    else:
        ids, vals = dvl.draft_topk(head_ok, hd, k, ws=ws)
        check_topk(oracle_mod, L, d2t, k, ids.cpu().numpy(), vals.cpu().numpy())
    assert dvl.workspace_status(ws) == 0


PAD = 4096  # canary bytes on each side


def carve(nbytes, fill):
    """A buffer of nbytes with PAD canary bytes on both sides; returns
    (whole buffer, the inner view)."""
    whole = torch.full((PAD + nbytes + PAD,), fill, dtype=torch.uint8, device="cuda")
    return whole, whole[PAD:PAD + nbytes]


def test_canaries_around_outputs_and_workspace(dvl, oracle_mod):
    V = 300_000
    for family, M, N, K, dtype in FAMILIES + [("bf16-tcgen05", 32, 3001, 2560, "bf16")]:
        mk, h, L = make_head(dvl, oracle_mod, N, K, M, dtype, 60 + M, V)
        d2t = np.random.default_rng(N).permutation(V)[:N].astype(np.int32)
        head = mk(d2t)
        hd = dev(h)
        for k in (1, 4):
            nws = dvl.workspace_bytes(M, k)
            ws_whole, ws = carve(nws, 0)
            dvl.workspace_init(ws)
            # the workspace's own bytes start at zero, the pads at 0xA5
            ws_whole[:PAD].fill_(0xA5)
            ws_whole[PAD + nws:].fill_(0xA5)
            id_whole, id_bytes = carve(4 * M * k, 0x5A)
            lg_whole, lg_bytes = carve(4 * M * k, 0x3C)
            ids = id_bytes.view(torch.int32).view(M, k)
            lg = lg_bytes.view(torch.float32).view(M, k)
            for _ in range(2):
                if k == 1:
                    dvl.draft_argmax(head, hd, ids=ids.view(-1), logits=lg.view(-1), ws=ws)
                else:
                    dvl.draft_topk(head, hd, k, ids=ids, logits=lg, ws=ws)
            torch.cuda.synchronize()
            for whole, n, fill in ((ws_whole, nws, 0xA5), (id_whole, 4 * M * k, 0x5A),
                                   (lg_whole, 4 * M * k, 0x3C)):
                b = whole.cpu().numpy()
                assert np.all(b[:PAD] == fill), family
                assert np.all(b[PAD + n:] == fill), family
            # the ticket, status word and best keys are left at zero (the
            # top-k slots after them are rewritten by every call)
            assert not ws[:512].cpu().numpy().any(), family
            if k == 1:
                check_argmax(oracle_mod, L, d2t, ids.view(-1).cpu().numpy(),
                             lg.view(-1).cpu().numpy())
            else:
                check_topk(oracle_mod, L, d2t, k, ids.cpu().numpy(), lg.cpu().numpy())
