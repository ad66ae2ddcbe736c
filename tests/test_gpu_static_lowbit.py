"""GPU parity of the static-head mode of the NVFP4 and FP8 kernels, the mode
the benchmark times: with DVL_HEAD_STATIC the kernel fills its load ring
from the head before it waits for the preceding kernel on the stream, and
reads h, d2t and the workspace only after that wait.

Each call here follows, on the same stream, a long reduction kernel whose
output IS the call's h (a sum over 2,048 terms of which exactly one is the
wanted value, so the bf16 result is exact).  h holds a different, wrong
vector before that kernel runs; a call that read h before its wait would
see it and miss the oracle.  Workloads: the NVFP4 32,768 x 5,120 trimmed head
(rank-order d2t) and the 248,320 x 2,560 FP8 full-vocabulary head, M = 1
and 3, argmax and top-4, several calls back to back, against the oracle by
the parity rule."""
import numpy as np
import pytest

import synthetic as S
from parity import check_argmax, check_topk

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

TERMS = 2048  # summands per element of the reduction that writes h


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


def spread(h_bits, slot):
    """A [M*K][TERMS] bf16 tensor that is zero except h at column `slot`:
    its sum over the last axis is h exactly."""
    M, K = h_bits.shape
    big = torch.zeros((M * K, TERMS), dtype=torch.bfloat16, device="cuda")
    big[:, slot] = dev(h_bits).view(torch.bfloat16).reshape(-1)
    return big


def calls_after_h_writer(dvl, head, hs, k, ws):
    """For each h of hs: poison the h buffer, let a long reduction write the
    real h into it, then enqueue the draft call right behind it."""
    M, K = hs[0].shape
    hbuf = torch.empty((M, K), dtype=torch.bfloat16, device="cuda")
    bigs = [spread(h, 17 + 301 * i) for i, h in enumerate(hs)]
    poison = torch.full((M, K), -3.0, dtype=torch.bfloat16, device="cuda")
    torch.cuda.synchronize()
    outs = []
    for big in bigs:
        hbuf.copy_(poison)
        torch.sum(big, dim=1, out=hbuf.view(-1))  # the kernel right before the call
        if k == 1:
            ids, vals = dvl.draft_argmax(head, hbuf.view(torch.int16), ws=ws)
        else:
            ids, vals = dvl.draft_topk(head, hbuf.view(torch.int16), k, ws=ws)
        outs.append((ids, vals))
    torch.cuda.synchronize()
    return [(i.cpu().numpy(), v.cpu().numpy()) for i, v in outs]


@pytest.mark.parametrize("k", [1, 4])
def test_nvfp4_trimmed_head_static(dvl, oracle_mod, k):
    wl = S.c5()
    head = dvl.Head(dev(wl.q), scales=dev(wl.scales), global_scale=wl.g, V=wl.V,
                    d2t=dev(wl.d2t), static=True)
    ws = dvl.make_workspace(4, 4)
    torch.cuda.synchronize()  # the head is complete before any static call
    for M in (1, 3):
        hs = [S.hidden_bf16(700 + 10 * M + i, M, wl.K) for i in range(3)]
        assert dvl.draft_plan(head, M, k) == ("nvfp4-mma", 1)
        got = calls_after_h_writer(dvl, head, hs, k, ws)
        for h, (ids, vals) in zip(hs, got):
            L, _ = oracle_mod.logits_nvfp4(wl.q, wl.scales, wl.g, h)
            if k == 1:
                check_argmax(oracle_mod, L, wl.d2t, ids, vals)
            else:
                check_topk(oracle_mod, L, wl.d2t, k, ids, vals)
    assert dvl.workspace_status(ws) == 0


@pytest.fixture(scope="module")
def fp8_full():
    q8, g8 = S.normal_fp8_rows(1, S.V_FULL, 2560, 0.02)
    return q8, g8


@pytest.mark.parametrize("k", [1, 4])
def test_fp8_full_vocabulary_head_static(dvl, oracle_mod, fp8_full, k):
    q8, g8 = fp8_full
    head = dvl.Head(dev(q8), fmt="fp8", global_scale=g8, V=S.V_FULL, static=True)
    ws = dvl.make_workspace(4, 4)
    torch.cuda.synchronize()
    for M in (1, 3):
        hs = [S.hidden_bf16(800 + 10 * M + i, M, 2560) for i in range(2)]
        assert dvl.draft_plan(head, M, k) == ("fp8-mma", 1)
        got = calls_after_h_writer(dvl, head, hs, k, ws)
        for h, (ids, vals) in zip(hs, got):
            L, _ = oracle_mod.logits_fp8(q8, g8, h)
            if k == 1:
                check_argmax(oracle_mod, L, None, ids, vals)
            else:
                check_topk(oracle_mod, L, None, k, ids, vals)
    assert dvl.workspace_status(ws) == 0
