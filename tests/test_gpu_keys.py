"""The key rules of the draft calls, on every kernel family, against the
oracle: an exactly equal logit goes to the lowest full-vocabulary id, a NaN
logit ranks below every number (among NaNs the lowest id wins), +inf and
-inf rank as numbers, and -0 and +0 are equal with +0 reported.

Every input is finite-time and host-planted: special values come from bf16
weights that are +inf, -inf or NaN, from E4M3 scale or code bytes that
encode NaN, and, for NVFP4 and FP8 heads (whose codes hold no infinity), from
a tensor scale so large that a planted row's dot product overflows to
+-inf while every other row stays finite.  Ids and logits must match the
oracle exactly (NaN matching NaN); a zero logit must come back as +0.
"""
import functools

import numpy as np
import pytest

import synthetic as S

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

BF16_PINF, BF16_NINF, BF16_NAN, BF16_NZERO = 0x7F80, 0xFF80, 0x7FC0, 0x8000
CASES = ("inf", "zero", "nan", "ninf")


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


def planted_rows(rng, N, n):
    """n distinct rows spread over the head (so several blocks hold some)."""
    return rng.choice(N, size=n, replace=False)


def hidden(rng, M, K):
    # positive small integers: a planted special weight meets a positive
    # hidden value in every hidden row; columns 0 and 1 equal so that a row
    # (1, -1, 0, ...) cancels to an exact zero
    h = rng.integers(1, 4, size=(M, K)).astype(np.float32)
    h[:, 1] = h[:, 0]
    return S.f32_to_bf16_bits(h)


@functools.lru_cache(maxsize=None)
def bf16_head(case, N, K, M, seed):
    """(W bits [N][K], h bits [M][K], d2t [N], V) for one key case."""
    rng = np.random.default_rng([seed, N, K, M, CASES.index(case)])
    V = 4 * N + 7
    d2t = rng.permutation(V)[:N].astype(np.int32)  # not monotone in the row
    if case == "zero":
        # every logit <= 0: negative weights, a few rows of zeros, of -0
        # and of two weights that cancel; the best logit is exactly 0
        w = S.f32_to_bf16_bits(-rng.integers(1, 4, size=(N, K)).astype(np.float32))
        rows = planted_rows(rng, N, 9)
        w[rows[:3]] = 0
        w[rows[3:6]] = BF16_NZERO
        for r in rows[6:]:
            w[r] = 0
            w[r, 0] = S.f32_to_bf16_bits(np.float32([1.0]))[0]
            w[r, 1] = S.f32_to_bf16_bits(np.float32([-1.0]))[0]
    else:
        w = S.f32_to_bf16_bits(rng.integers(-3, 4, size=(N, K)).astype(np.float32))
        if case == "inf":
            rows = planted_rows(rng, N, 8)
            w[rows[:3], 0] = BF16_PINF            # three +inf rows
            w[rows[3:5], 0] = BF16_NINF           # -inf rows
            w[rows[5:7], 0] = BF16_NAN            # NaN rows
            w[rows[7], 0] = BF16_PINF             # +inf + -inf = NaN
            w[rows[7], 1] = BF16_NINF
        elif case == "nan":
            w[:, 0] = BF16_NAN                    # every logit NaN
        elif case == "ninf":
            w[:, 0] = BF16_NAN                    # NaN everywhere but a few
            rows = planted_rows(rng, N, 5)
            w[rows, 0] = BF16_NINF                # rows at -inf
    h = hidden(rng, M, K)
    return w, h, d2t, V


# E2M1 nibbles and E4M3 bytes used below (values from the format definitions)
E2M1_POS = np.array([0x0, 0x1, 0x2, 0x3], np.uint8)      # 0, 0.5, 1, 1.5
E2M1_SIX, E2M1_NSIX = 0x7, 0xF                            # +6, -6
E4M3_ONE, E4M3_448, E4M3_NAN = 0x38, 0x7E, 0x7F
FP8_SMALL = np.array([0x00, 0x30, 0x38, 0x3C, 0xB0, 0xB8, 0xBC], np.uint8)  # 0, +-0.5, +-1, +-1.5
# A tensor scale of 2^112: |ordinary logit| <= K * 3 * 1.5 * 2^112 < 2^126 at
# K = 2,560, while a row of 6 * 448 (NVFP4) or 448 (FP8) weights against
# hidden values >= 1 sums past 2^128 and overflows to +-inf.
G_HUGE = float(2.0 ** 112)


def pack_nibbles(nib):
    nib = np.asarray(nib, np.uint8)
    return (nib[:, 0::2] | (nib[:, 1::2] << 4)).astype(np.uint8)


@functools.lru_cache(maxsize=None)
def lowbit_head(fmt, case, N, K, M, seed):
    """(codes, scales or None, g, h bits, d2t, V) for one key case."""
    rng = np.random.default_rng([seed, N, K, M, CASES.index(case), 4 if fmt == "nvfp4" else 8])
    V = 4 * N + 7
    d2t = rng.permutation(V)[:N].astype(np.int32)
    h = hidden(rng, M, K)
    nv = fmt == "nvfp4"
    if nv:
        nib = rng.choice(E2M1_POS, size=(N, K))
        nib = nib | (rng.integers(0, 2, size=(N, K)).astype(np.uint8) << 3)  # random signs
        sc = np.full((N, K // 16), E4M3_ONE, np.uint8)
    else:
        q = rng.choice(FP8_SMALL, size=(N, K))
    g = G_HUGE
    if case == "zero":
        # a negative tensor scale flips every sign: non-negative codes give
        # logits <= 0, all-zero rows give a zero dot (the kernel's product
        # with g is then -0; the oracle's sum is +0)
        g = -1.0
        rows = planted_rows(rng, N, 6)
        if nv:
            nib = nib & 0x7
            nib[rows[:3]] = 0
            nib[rows[3:]] = 0x8                   # -0 codes
        else:
            q = q & 0x7F
            q[rows[:3]] = 0
            q[rows[3:]] = 0x80                    # -0 codes
    elif case == "inf":
        rows = planted_rows(rng, N, 7)
        if nv:
            nib[rows[:3]] = E2M1_SIX
            sc[rows[:3]] = E4M3_448
            nib[rows[3:5]] = E2M1_NSIX
            sc[rows[3:5]] = E4M3_448
            sc[rows[5:], 0] = E4M3_NAN
        else:
            q[rows[:3]] = E4M3_448
            q[rows[3:5]] = E4M3_448 | 0x80
            q[rows[5:], 0] = E4M3_NAN
    elif case == "nan":
        if nv:
            sc[:, 0] = E4M3_NAN
        else:
            q[:, 0] = E4M3_NAN
    elif case == "ninf":
        rows = planted_rows(rng, N, 5)
        if nv:
            sc[:, 0] = E4M3_NAN
            nib[rows] = E2M1_NSIX
            sc[rows] = E4M3_448
        else:
            q[:, 0] = E4M3_NAN
            q[rows] = E4M3_448 | 0x80
    if nv:
        return pack_nibbles(nib), sc, g, h, d2t, V
    return q.astype(np.uint8), None, g, h, d2t, V


def assert_same(gpu_ids, gpu_vals, o_ids, o_vals):
    gpu_ids, o_ids = np.asarray(gpu_ids), np.asarray(o_ids)
    gpu_vals = np.asarray(gpu_vals, np.float32)
    o_vals = np.asarray(o_vals, np.float32)
    assert np.array_equal(gpu_ids, o_ids), (gpu_ids, o_ids)
    nan = np.isnan(o_vals)
    assert np.array_equal(np.isnan(gpu_vals), nan), (gpu_vals, o_vals)
    assert np.array_equal(gpu_vals[~nan], o_vals[~nan]), (gpu_vals, o_vals)
    zero = gpu_vals == 0
    assert not np.any(np.signbit(gpu_vals[zero])), "a zero logit must be reported as +0"


def run_and_check(dvl, oracle_mod, head, h, L, d2t, M, plan_kernel):
    kernel, _ = dvl.draft_plan(head, M, 1)
    assert kernel == plan_kernel
    hd = dev(h)
    ids, vals = dvl.draft_argmax(head, hd)
    o_ids, o_vals = oracle_mod.argmax(L, d2t)
    assert_same(ids.cpu().numpy(), vals.cpu().numpy(), o_ids, o_vals)
    ids, vals = dvl.draft_topk(head, hd, 4)
    o_ids, o_vals, _ = oracle_mod.topk(L, 4, d2t)
    assert_same(ids.cpu().numpy(), vals.cpu().numpy(), o_ids, o_vals)
    return o_vals


# (kernel family, M, N, K): the family draft_plan reports for the argmax
BF16_FAMILIES = [
    ("bf16-cuda-cores", 1, 3001, 2560), ("bf16-cuda-cores", 2, 3001, 320),
    ("bf16-mma", 3, 20000, 2560), ("bf16-mma", 8, 20000, 5120),
    ("bf16-tcgen05", 8, 3001, 256), ("bf16-tcgen05", 32, 3001, 2560),
]


@pytest.mark.parametrize("case", CASES)
@pytest.mark.parametrize("family,M,N,K", BF16_FAMILIES)
def test_bf16_key_rules(dvl, oracle_mod, family, M, N, K, case):
    w, h, d2t, V = bf16_head(case, N, K, M, 7)
    L, _ = oracle_mod.logits_bf16(w, h)
    head = dvl.Head(dev(w), V=V, d2t=dev(d2t))
    o_vals = run_and_check(dvl, oracle_mod, head, h, L, d2t, M, family)
    # the case really plants what it names
    best = o_vals[:, 0]
    if case == "inf":
        assert np.all(np.isposinf(best))
    elif case == "zero":
        assert np.all(best == 0)
    elif case == "nan":
        assert np.all(np.isnan(best))
    else:
        assert np.all(np.isneginf(best))


LOWBIT_FAMILIES = [
    ("nvfp4", 1, 3001, 2560), ("nvfp4", 3, 3001, 5120), ("nvfp4", 5, 2049, 128),
    ("fp8", 1, 3001, 2560), ("fp8", 3, 3001, 2560), ("fp8", 2, 2049, 192),
]


@pytest.mark.parametrize("case", CASES)
@pytest.mark.parametrize("fmt,M,N,K", LOWBIT_FAMILIES)
def test_lowbit_key_rules(dvl, oracle_mod, fmt, M, N, K, case):
    q, sc, g, h, d2t, V = lowbit_head(fmt, case, N, K, M, 11)
    if fmt == "nvfp4":
        L, _ = oracle_mod.logits_nvfp4(q, sc, g, h)
        head = dvl.Head(dev(q), scales=dev(sc), global_scale=g, V=V, d2t=dev(d2t))
    else:
        L, _ = oracle_mod.logits_fp8(q, g, h)
        head = dvl.Head(dev(q), fmt="fp8", global_scale=g, V=V, d2t=dev(d2t))
    o_vals = run_and_check(dvl, oracle_mod, head, h, L, d2t, M, f"{fmt}-mma")
    best = o_vals[:, 0]
    if case == "inf":
        assert np.all(np.isposinf(best))
        # the huge tensor scale leaves every row but the seven planted finite
        assert int((~np.isfinite(L).all(axis=0)).sum()) == 7
    elif case == "zero":
        assert np.all(best == 0)
    elif case == "nan":
        assert np.all(np.isnan(best))
    else:
        assert np.all(np.isneginf(best))
