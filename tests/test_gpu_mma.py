"""GPU parity of the register-path tensor-core kernel for bf16 heads (3 .. 16
hidden rows at width 2,560, 3 .. 8 at 5,120, heads of at least one full
8-row tile per warp; top-k above 8 rows runs on the tcgen05 kernel),
against the oracle: bit-exact argmax and top-4 on integer heads with a d2t map and with id_base, ragged tiles at the end of
each warp's range, the same head one row short of the threshold (CUDA
cores), a head that is 16-byte but not 32-byte aligned (CUDA cores),
gaussian heads under the parity rule, and the plan each case reports."""
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


def threshold_rows():
    """Smallest head that gives every warp of the two-blocks-per-SM grid a
    full 8-row tile."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    return 8 * 8 * 2 * sms


def int_case(seed, N, K, M):
    rng = np.random.default_rng(seed)
    w = S.f32_to_bf16_bits(rng.integers(-4, 5, size=(N, K)).astype(np.float32))
    h = S.f32_to_bf16_bits(rng.integers(-3, 4, size=(M, K)).astype(np.float32))
    return rng, w, h


@pytest.mark.parametrize("K,M", [(2560, 3), (2560, 4), (2560, 5), (2560, 8), (2560, 12), (2560, 16),
                                 (5120, 3), (5120, 4), (5120, 5), (5120, 8)])
def test_mma_integer_head_bit_exact(dvl, oracle_mod, K, M):
    N = threshold_rows() + 555  # ragged: warps end on partial tiles
    rng, w, h = int_case(K + M, N, K, M)
    L, _ = oracle_mod.logits_bf16(w, h)
    V = 2 * N + 3
    d2t = rng.permutation(V)[:N].astype(np.int32)
    head = dvl.Head(dev(w), V=V, d2t=dev(d2t))
    ws = dvl.make_workspace(M, 4)
    ids, vals = dvl.draft_argmax(head, dev(h), ws=ws)
    o_ids, o_vals = oracle_mod.argmax(L, d2t)
    assert np.array_equal(ids.cpu().numpy(), o_ids)
    assert np.array_equal(vals.cpu().numpy(), o_vals)
    ids, vals = dvl.draft_topk(head, dev(h), 4, ws=ws)
    o_ids, o_vals, _ = oracle_mod.topk(L, 4, d2t)
    assert np.array_equal(ids.cpu().numpy(), o_ids)
    assert np.array_equal(vals.cpu().numpy(), o_vals)
    # identity ids with an offset
    head = dvl.Head(dev(w), V=N + 1000, id_base=1000)
    ids, vals = dvl.draft_topk(head, dev(h), 3, ws=ws)
    o_ids, o_vals, _ = oracle_mod.topk(L, 3, None)
    assert np.array_equal(ids.cpu().numpy(), o_ids + 1000)
    assert np.array_equal(vals.cpu().numpy(), o_vals)
    torch.cuda.synchronize()
    assert dvl.workspace_status(ws) == 0


def test_mma_and_cuda_core_paths_agree_and_dispatch(dvl, oracle_mod):
    """The same integer head at the threshold (tensor cores), one row short
    (CUDA cores) and 16-byte aligned only (CUDA cores): every result exact,
    and each call planned on the kernel the rule names."""
    T, K, M = threshold_rows(), 2560, 3
    rng, w, h = int_case(7, T, K, M)
    hd = dev(h)
    ws = dvl.make_workspace(M, 4)
    # 16-byte aligned only: the same rows 8 elements into a flat buffer
    flat = torch.empty(T * K + 8, dtype=torch.int16, device="cuda")
    flat[8:] = dev(w).view(-1)
    w16 = flat[8:].view(T, K)
    assert w16.data_ptr() % 32 == 16
    cases = {"mma": (dev(w), w, "bf16-mma"),
             "short": (dev(w[: T - 1]), w[: T - 1], "bf16-cuda-cores"),
             "align16": (w16, w, "bf16-cuda-cores")}
    for name, (wd, wn, plan) in cases.items():
        head = dvl.Head(wd)
        assert dvl.draft_plan(head, M, 4) == (plan, 1), name
        assert dvl.draft_plan(head, M, 1) == (plan, 1), name
        L, _ = oracle_mod.logits_bf16(wn, h)
        o_ids, o_vals, _ = oracle_mod.topk(L, 4, None)
        ids, vals = dvl.draft_topk(head, hd, 4, ws=ws)
        assert np.array_equal(ids.cpu().numpy(), o_ids), name
        assert np.array_equal(vals.cpu().numpy(), o_vals), name
        o_ids, o_vals = oracle_mod.argmax(L, None)
        ids, vals = dvl.draft_argmax(head, hd, ws=ws)
        assert np.array_equal(ids.cpu().numpy(), o_ids), name
        assert np.array_equal(vals.cpu().numpy(), o_vals), name
    # the other plans on the same head
    head = dvl.Head(cases["mma"][0])
    assert dvl.draft_plan(head, 1) == ("bf16-cuda-cores", 1)
    assert dvl.draft_plan(head, 2, 4) == ("bf16-cuda-cores", 1)
    assert dvl.draft_plan(head, 4) == ("bf16-mma", 1)
    assert dvl.draft_plan(head, 8, 4) == ("bf16-mma", 1)
    assert dvl.draft_plan(head, 9) == ("bf16-mma", 1)
    assert dvl.draft_plan(head, 16) == ("bf16-mma", 1)
    assert dvl.draft_plan(head, 9, 4) == ("bf16-tcgen05", 1)
    assert dvl.draft_plan(head, 17) == ("bf16-tcgen05", 1)
    assert dvl.draft_plan(head, 32, 4) == ("bf16-tcgen05", 1)
    wide = dvl.Head(torch.empty((T, 5120), dtype=torch.int16, device="cuda"))
    assert dvl.draft_plan(wide, 8) == ("bf16-mma", 1)
    assert dvl.draft_plan(wide, 9) == ("bf16-tcgen05", 1)
    short = dvl.Head(cases["short"][0])
    assert dvl.draft_plan(short, 8) == ("bf16-tcgen05", 1)
    torch.cuda.synchronize()
    assert dvl.workspace_status(ws) == 0


@pytest.mark.parametrize("N,K,M", [(20011, 2560, 3), (32768, 5120, 4), (40000, 2560, 4),
                                   (52755, 2560, 8), (20011, 5120, 6), (52755, 2560, 16),
                                   (24000, 2560, 11)])
def test_mma_gaussian_head_parity(dvl, oracle_mod, N, K, M):
    if N < threshold_rows():
        pytest.skip("head below the tensor-core threshold on this device")
    w = S.normal_bf16_rows(N + 1, N, K, 0.02)
    h = S.hidden_bf16(N + 2, M, K)
    rng = np.random.default_rng(N + 3)
    d2t = rng.permutation(248_320)[:N].astype(np.int32)
    head = dvl.Head(dev(w), V=248_320, d2t=dev(d2t), static=True)
    L, _ = oracle_mod.logits_bf16(w, h)
    ids, vals = dvl.draft_argmax(head, dev(h))
    check_argmax(oracle_mod, L, d2t, ids.cpu().numpy(), vals.cpu().numpy())
    ids, vals = dvl.draft_topk(head, dev(h), 4)
    check_topk(oracle_mod, L, d2t, 4, ids.cpu().numpy(), vals.cpu().numpy())
