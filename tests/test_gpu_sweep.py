"""A seeded sweep over the library's dispatch space, bit for bit against the
oracle: dtype (bf16, NVFP4, FP8), head rows N (1 .. 70,000, ragged), width K
(multiples of 64, the unrolled widths 2,560 and 5,120 included), hidden rows
M (1 .. 32), k (1 .. 4), with or without a d2t map, and id_base offsets of
row slices.  Every head holds small integers (and power-of-two scales), so
every dot is exact on both sides and ids, logits and ties must agree
exactly; the same heads are scored through dvl_score_ids where they have no
d2t.  Together the cases reach the CUDA-core, tensor-core and low-bit
kernels, their unrolled and run-time widths, and the chunked paths."""
import numpy as np
import pytest

import synthetic as S
from test_oracle_fp8 import _int_e4m3

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

E2M1_INT = {0: 0x0, 1: 0x2, 2: 0x4, 3: 0x5, 4: 0x6, 6: 0x7}  # exact E2M1 integers


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


def _int_nvfp4(rng, N, K):
    """NVFP4 codes of small integers (E2M1 values 0..6 and signs) with block
    scales 1 or 2 (E4M3 0x38, 0x40)."""
    mags = np.array(sorted(E2M1_INT))
    lut = np.zeros(7, np.uint8)
    for v, c in E2M1_INT.items():
        lut[v] = c
    x = rng.choice(mags, size=(N, K)) * rng.choice([-1, 1], size=(N, K))
    codes = (lut[np.abs(x)] | np.where(x < 0, 8, 0)).astype(np.uint8)
    q = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    sc = rng.choice(np.array([0x38, 0x40], np.uint8), size=(N, K // 16))
    return q, sc


def _cases():
    rng = np.random.default_rng(2024)
    out = []
    for i in range(40):
        dtype = ["bf16", "bf16", "nvfp4", "fp8"][i % 4]
        K = int(rng.choice([64, 128, 320, 1024, 2560, 2560, 5120]))
        N = int(rng.choice([1, 7, 129, 1000, 4097, 20000, 70000]))
        if K >= 5120 and N > 20000:
            N = 20000
        if dtype != "bf16":  # the low-bit oracle decodes every weight: keep it small
            N = min(N, 4097)
        M = int(rng.choice([1, 2, 3, 4, 5, 8, 9, 16, 31, 32]))
        k = int(min(rng.integers(1, 5), N))
        mode = ["none", "d2t", "base"][int(rng.integers(0, 3))]
        out.append((i, dtype, N, K, M, k, mode))
    # NVFP4 at one hidden row and the unrolled widths (block scales applied
    # to the MMA results): heads long enough for every warp of the full grid
    # to take one or two 16-row tiles
    out += [(40, "nvfp4", 40000, 2560, 1, 4, "d2t"), (41, "nvfp4", 20000, 5120, 1, 1, "base"),
            (42, "nvfp4", 20000, 5120, 1, 3, "none")]
    return out


@pytest.mark.parametrize("i,dtype,N,K,M,k,mode", _cases())
def test_sweep_bit_exact(dvl, oracle_mod, i, dtype, N, K, M, k, mode):
    rng = np.random.default_rng(1000 + i)
    h = S.f32_to_bf16_bits(rng.integers(-3, 4, size=(M, K)).astype(np.float32))
    if dtype == "bf16":
        w = S.f32_to_bf16_bits(rng.integers(-4, 5, size=(N, K)).astype(np.float32))
        L, _ = oracle_mod.logits_bf16(w, h)
        head_kw = dict()
        w_dev = dev(w)
        score = lambda ids, base: oracle_mod.score_ids_bf16(w, h, ids, base)
    elif dtype == "nvfp4":
        q, sc = _int_nvfp4(rng, N, K)
        g = 0.5
        L, _ = oracle_mod.logits_nvfp4(q, sc, g, h)
        head_kw = dict(scales=dev(sc), global_scale=g)
        w_dev = dev(q)
        score = lambda ids, base: oracle_mod.score_ids_nvfp4(q, sc, g, h, ids, base)
    else:
        q, _ = _int_e4m3(rng, (N, K), -8, 8)
        g = 2.0
        L, _ = oracle_mod.logits_fp8(q, g, h)
        head_kw = dict(fmt="fp8", global_scale=g)
        w_dev = dev(q)
        score = lambda ids, base: oracle_mod.score_ids_fp8(q, g, h, ids, base)
    d2t, base, V = None, 0, N
    if mode == "d2t":
        V = 3 * N + 11
        d2t = rng.permutation(V)[:N].astype(np.int32)
    elif mode == "base":
        base, V = 977, N + 977 + 5
    head = dvl.Head(w_dev, V=V, d2t=dev(d2t) if d2t is not None else None, id_base=base,
                    **head_kw)
    ws = dvl.make_workspace(M, k)
    ids, vals = dvl.draft_topk(head, dev(h), k, ws=ws)
    o_ids, o_vals, _ = oracle_mod.topk(L, k, d2t)
    if d2t is None:
        o_ids = o_ids + base
    assert np.array_equal(ids.cpu().numpy(), o_ids), (i, dtype, N, K, M, k, mode)
    assert np.array_equal(vals.cpu().numpy(), o_vals), (i, dtype, N, K, M, k, mode)
    a_ids, a_vals = dvl.draft_argmax(head, dev(h), ws=ws)
    assert np.array_equal(a_ids.cpu().numpy(), o_ids[:, 0])
    assert np.array_equal(a_vals.cpu().numpy(), o_vals[:, 0])
    if d2t is None:
        cand = rng.integers(base - 2, base + N + 2, size=(M, 6)).astype(np.int32)
        got = dvl.score_ids(head, dev(h), dev(cand)).cpu().numpy()
        want = score(cand, base)
        assert np.array_equal(np.isnan(got), np.isnan(want))
        ok = ~np.isnan(want)
        assert np.array_equal(got[ok], want[ok])
    torch.cuda.synchronize()
    assert dvl.workspace_status(ws) == 0
