"""GPU parity at batched-drafting sizes where M x K exceeds 98,304 (the most a
block could stage when every hidden row sat in shared memory at once):
bf16 at M = 32, K = 5,120 and at M = 20, K = 24,576 (one pass on the tcgen05
kernel, which streams tiles of h with the head), and NVFP4 / FP8 at M = 24
and 32, K = 5,120 (chunks of 8 rows on the low-bit kernel).  Integer heads
and hidden rows make every sum exact, so ids, logits and ties must agree
with the oracle bit for bit; each case also checks the plan it ran on."""
import numpy as np
import pytest

import synthetic as S
from test_gpu_sweep import _int_nvfp4
from test_oracle_fp8 import _int_e4m3

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


def exact(dvl, oracle_mod, head, L, h, M, d2t, ws):
    ids, vals = dvl.draft_argmax(head, dev(h), ws=ws)
    o_ids, o_vals = oracle_mod.argmax(L, d2t)
    assert np.array_equal(ids.cpu().numpy(), o_ids)
    assert np.array_equal(vals.cpu().numpy(), o_vals)
    ids, vals = dvl.draft_topk(head, dev(h), 4, ws=ws)
    o_ids, o_vals, _ = oracle_mod.topk(L, 4, d2t)
    assert np.array_equal(ids.cpu().numpy(), o_ids)
    assert np.array_equal(vals.cpu().numpy(), o_vals)
    torch.cuda.synchronize()
    assert dvl.workspace_status(ws) == 0


@pytest.mark.parametrize("N,K,M", [(3001, 5120, 32), (500, 24576, 20)])
def test_bf16_batched_one_pass(dvl, oracle_mod, N, K, M):
    rng = np.random.default_rng(N + K + M)
    w = S.f32_to_bf16_bits(rng.integers(-4, 5, size=(N, K)).astype(np.float32))
    h = S.f32_to_bf16_bits(rng.integers(-2, 3, size=(M, K)).astype(np.float32))
    V = 2 * N + 1
    d2t = rng.permutation(V)[:N].astype(np.int32)
    head = dvl.Head(dev(w), V=V, d2t=dev(d2t))
    assert dvl.draft_plan(head, M, 4) == ("bf16-tcgen05", 1)
    L, _ = oracle_mod.logits_bf16(w, h)
    exact(dvl, oracle_mod, head, L, h, M, d2t, dvl.make_workspace(M, 4))


@pytest.mark.parametrize("fmt,N,M", [("fp8", 3001, 32), ("nvfp4", 1000, 24)])
def test_lowbit_batched_in_chunks(dvl, oracle_mod, fmt, N, M):
    K = 5120
    rng = np.random.default_rng(N + M + 11)
    h = S.f32_to_bf16_bits(rng.integers(-3, 4, size=(M, K)).astype(np.float32))
    d2t = rng.permutation(3 * N)[:N].astype(np.int32)
    if fmt == "fp8":
        q, _ = _int_e4m3(rng, (N, K), -8, 8)
        g = 0.5
        head = dvl.Head(dev(q), fmt="fp8", global_scale=g, V=3 * N, d2t=dev(d2t))
        L, _ = oracle_mod.logits_fp8(q, g, h)
    else:
        q, sc = _int_nvfp4(rng, N, K)
        g = 0.25
        head = dvl.Head(dev(q), scales=dev(sc), global_scale=g, V=3 * N, d2t=dev(d2t))
        L, _ = oracle_mod.logits_nvfp4(q, sc, g, h)
    assert dvl.draft_plan(head, M, 4) == (f"{fmt}-mma", (M + 7) // 8)
    exact(dvl, oracle_mod, head, L, h, M, d2t, dvl.make_workspace(M, 4))
