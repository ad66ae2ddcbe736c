"""GPU parity at batched-drafting sizes where M x K exceeds 98,304 (the most a
block could stage when every hidden row sat in shared memory at once):
bf16 at M = 32, K = 5,120 and at M = 20, K = 24,576 (one pass on the tcgen05
kernel, which streams tiles of h with the head), and NVFP4 / FP8 at 9 to 32
hidden rows (one pass at K = 2,560, groups of 16 rows at 5,120, on the
low-bit kernel with two or four groups of 8 MMA columns), and 5 to 8 rows
(one launch of its run-time-width instantiation).  Integer heads and
hidden rows make every sum exact, so ids, logits and ties must agree with the
oracle bit for bit; each case also checks the plan it ran on.  Gaussian
NVFP4 / FP8 heads of the workloads' shapes (the 32,768 x 5,120 trimmed head,
the 248,320 x 2,560 full vocabulary) follow the parity rule at 16 and 32
rows."""
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


def lowbit_int_head(dvl, oracle_mod, fmt, N, K, M, seed):
    rng = np.random.default_rng(seed)
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
    return head, L, h, d2t


@pytest.mark.parametrize("fmt", ["fp8", "nvfp4"])
@pytest.mark.parametrize("K,M", [(2560, 5), (2560, 8), (2560, 9), (2560, 16), (2560, 17),
                                 (2560, 32), (5120, 7), (5120, 12), (5120, 16), (5120, 24),
                                 (5120, 32)])
def test_lowbit_batched_one_pass(dvl, oracle_mod, fmt, K, M):
    # one launch for up to 32 rows (argmax) at 2,560, else one per 16 rows:
    # the head is read once per launch
    N = 3001 if K == 2560 else 1000
    head, L, h, d2t = lowbit_int_head(dvl, oracle_mod, fmt, N, K, M, N + K + M + 11)
    assert dvl.draft_plan(head, M, 4) == (f"{fmt}-mma", (M + 15) // 16)
    assert dvl.draft_plan(head, M, 1) == (f"{fmt}-mma", 1 if K == 2560 else (M + 15) // 16)
    exact(dvl, oracle_mod, head, L, h, M, d2t, dvl.make_workspace(M, 4))


@pytest.mark.parametrize("fmt", ["fp8", "nvfp4"])
def test_lowbit_batched_ragged_rows_and_tiles(dvl, oracle_mod, fmt):
    # a head whose rows end mid-tile and a few rows per warp, row counts
    # that fill a group partly, and calls back to back on one workspace
    ws = dvl.make_workspace(32, 4)
    for N, M in ((37, 25), (4099, 10), (20011, 31)):
        head, L, h, d2t = lowbit_int_head(dvl, oracle_mod, fmt, N, 2560, M, N + M)
        exact(dvl, oracle_mod, head, L, h, M, d2t, ws)


def test_lowbit_batched_gaussian_workload_shapes(dvl, oracle_mod):
    from parity import check_argmax, check_topk
    wl = S.c5(Ms=())
    head = dvl.Head(dev(wl.q), scales=dev(wl.scales), global_scale=wl.g, V=wl.V,
                    d2t=dev(wl.d2t), static=True)
    q8, g8 = S.normal_fp8_rows(1, S.V_FULL, 2560, 0.02)
    head8 = dvl.Head(dev(q8), fmt="fp8", global_scale=g8, V=S.V_FULL, static=True)
    torch.cuda.synchronize()
    ws = dvl.make_workspace(32, 4)
    for hd, K, M, name in ((head, 5120, 16, "nvfp4"), (head8, 2560, 32, "fp8")):
        h = S.hidden_bf16(600 + M, M, K)
        if name == "nvfp4":
            L, _ = oracle_mod.logits_nvfp4(wl.q, wl.scales, wl.g, h)
            d2t = wl.d2t
        else:
            L, _ = oracle_mod.logits_fp8(q8, g8, h)
            d2t = None
        assert dvl.draft_plan(hd, M, 1) == (f"{name}-mma", 1)
        ids, vals = dvl.draft_argmax(hd, dev(h), ws=ws)
        check_argmax(oracle_mod, L, d2t, ids.cpu().numpy(), vals.cpu().numpy())
        ids, vals = dvl.draft_topk(hd, dev(h), 4, ws=ws)
        check_topk(oracle_mod, L, d2t, 4, ids.cpu().numpy(), vals.cpu().numpy())
    assert dvl.workspace_status(ws) == 0


@pytest.mark.parametrize("N,M", [(40000, 32), (40000, 20), (33001, 25)])
def test_bf16_topk_two_level_merge_bit_exact(dvl, oracle_mod, N, M):
    # grids whose top-k merge is two-level (M x blocks >= 2,560: groups of 16
    # blocks, the last group partial), exact integer sums with many ties
    K = 256
    rng = np.random.default_rng(N + M + 5)
    w = S.f32_to_bf16_bits(rng.integers(-4, 5, size=(N, K)).astype(np.float32))
    h = S.f32_to_bf16_bits(rng.integers(-2, 3, size=(M, K)).astype(np.float32))
    V = 2 * N + 1
    d2t = rng.permutation(V)[:N].astype(np.int32)
    head = dvl.Head(dev(w), V=V, d2t=dev(d2t))
    assert dvl.draft_plan(head, M, 4) == ("bf16-tcgen05", 1)
    L, _ = oracle_mod.logits_bf16(w, h)
    ws = dvl.make_workspace(M, 4)
    for _ in range(2):  # the group tickets leave the workspace clean
        exact(dvl, oracle_mod, head, L, h, M, d2t, ws)
