"""The tcgen05 kernel with a head flagged static, against the oracle: the
first ring stages' head boxes are loaded before the wait on the preceding
kernel and the hidden-row boxes after it.  Each call follows another draft
call on the same stream (a different head and different hidden rows), so
its early part overlaps running work.  Cases: 32 and 20 hidden rows on
the 32-column tiles, argmax and top-4; a width whose last stage holds one
64-wide box; a head so short that the whole call is fewer stages than the
ring; 5 rows on a head below the register-path threshold (16 columns)."""
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
    return torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).cuda()


# N, K, M, k
CASES = [(20000, 2560, 32, 1), (20000, 2560, 32, 4), (9000, 2496, 20, 1), (9000, 2496, 20, 4),
         (100, 256, 24, 4), (3001, 2560, 5, 1)]


@pytest.mark.parametrize("N,K,M,k", CASES)
def test_static_head_on_tcgen05_after_another_call(dvl, oracle_mod, N, K, M, k):
    w = S.normal_bf16_rows(N + 7, N, K, 0.02)
    h = S.hidden_bf16(N + 8, M, K)
    d2t = np.random.default_rng(N + 9).permutation(300_000)[:N].astype(np.int32)
    head = dvl.Head(dev(w), V=300_000, d2t=dev(d2t), static=True)
    assert dvl.draft_plan(head, M, k)[0] == "bf16-tcgen05"
    # the preceding kernel: a draft call on another head
    w0 = S.normal_bf16_rows(N + 10, 4000, K, 0.02)
    h0 = S.hidden_bf16(N + 11, 3, K)
    other = dvl.Head(dev(w0), static=True)
    L, _ = oracle_mod.logits_bf16(w, h)
    ws0, ws = dvl.make_workspace(3, 1), dvl.make_workspace(M, k)
    hd, hd0 = dev(h), dev(h0)
    for _ in range(3):
        dvl.draft_argmax(other, hd0, ws=ws0)
        if k == 1:
            ids, vals = dvl.draft_argmax(head, hd, ws=ws)
        else:
            ids, vals = dvl.draft_topk(head, hd, k, ws=ws)
    torch.cuda.synchronize()
    if k == 1:
        check_argmax(oracle_mod, L, d2t, ids.cpu().numpy(), vals.cpu().numpy())
    else:
        check_topk(oracle_mod, L, d2t, k, ids.cpu().numpy(), vals.cpu().numpy())
    assert dvl.workspace_status(ws) == 0
