"""Pins of the oracle's FP8 (E4M3) head ("[DGX Spark] Qwen3.8-Flash-Next on
two DGX Sparks", section "The costs: a 69% smaller KV pool and FP8 GDN
weights": weights read as FP8 E4M3 halve the bytes; "Masked MTP drafts": a
drafter shipping an FP8 head) to things other than itself: exact integer
arithmetic, power-of-two tensor scales, the hand-computed E4M3 values, the
fp32 summation bound against an fp64 dot, and the test-data quantizer's
rounding bound."""
import numpy as np
import pytest

from test_oracle_pins import _read_values
import synthetic as S


def _int_e4m3(rng, shape, lo=-16, hi=16):
    """Small integers (every integer up to 16 is exact in E4M3) as codes,
    with the codes built from the format definition by hand: sign bit 7,
    exponent e (bias 7) in bits 3-6, mantissa m in bits 0-2."""
    x = rng.integers(lo, hi + 1, size=shape)
    codes = np.zeros(shape, np.uint8)
    for v in range(1, 17):
        e = int(np.floor(np.log2(v)))
        m = v * 8 // (1 << e) - 8  # v = 2^e * (1 + m/8)
        code = ((e + 7) << 3) | m
        codes[x == v] = code
        codes[x == -v] = code | 0x80
    return codes, x


@pytest.mark.parametrize("N,K,M,g", [(1, 64, 1, 1.0), (37, 128, 3, 1.0), (64, 256, 4, 0.25),
                                     (9, 2560, 2, 2.0)])
def test_fp8_logits_exact_integer_bruteforce(oracle_mod, N, K, M, g):
    # integer weights times a power-of-two tensor scale, integer hidden
    # values: every partial sum is exact, so the oracle equals g * (W h)
    rng = np.random.default_rng(N + K + M)
    q, wi = _int_e4m3(rng, (N, K))
    hi = rng.integers(-8, 9, size=(M, K))
    hb = S.f32_to_bf16_bits(hi.astype(np.float32))
    got, _ = oracle_mod.logits_fp8(q, g, hb)
    want = (hi @ wi.T).astype(np.float64) * g
    assert np.array_equal(got.astype(np.float64), want)


def test_fp8_decode_is_the_hand_computed_e4m3(oracle_mod):
    # one-hot hidden rows pick single weights: each code decodes to the
    # hand-computed E4M3 value times g
    rows = [(b, v) for kind, b, v in _read_values() if kind == "e4m3" and not np.isnan(v)]
    q = np.array([[b for b, _ in rows] + [0] * (64 - len(rows))], np.uint8)
    g = 0.5
    for k, (_, v) in enumerate(rows):
        h = np.zeros((1, 64), np.float32)
        h[0, k] = 1.0
        got, _ = oracle_mod.logits_fp8(q, g, S.f32_to_bf16_bits(h))
        assert got[0, 0] == np.float32(v * g)


def test_fp8_scores_are_gathered_logits(oracle_mod):
    rng = np.random.default_rng(4)
    q, _ = _int_e4m3(rng, (30, 128))
    hb = S.f32_to_bf16_bits(rng.integers(-4, 5, size=(2, 128)).astype(np.float32))
    L, _ = oracle_mod.logits_fp8(q, 0.125, hb)
    ids = np.array([[3, 29, 30, -1, 0], [7, 7, 12, 28, 1]], np.int32)
    got = oracle_mod.score_ids_fp8(q, 0.125, hb, ids)
    for m in range(2):
        for j in range(5):
            i = ids[m, j]
            if 0 <= i < 30:
                assert got[m, j] == L[m, i]
            else:
                assert np.isnan(got[m, j])


def test_fp8_within_fp32_summation_bound_of_fp64(oracle_mod):
    N, K, M = 50, 2560, 2
    q, g = S.normal_fp8_rows(9, N, K, 0.02)
    hb = S.hidden_bf16(10, M, K)
    got, _ = oracle_mod.logits_fp8(q, g, hb)
    e4 = np.array([oracle_mod.e4m3(b) for b in range(256)])
    w = (e4[q] * g).astype(np.float32).astype(np.float64)  # one rounding per weight
    h = S.bf16_bits_to_f32(hb).astype(np.float64)
    for m in range(M):
        prod = w * h[m]
        # against the exact dot of the fp32-rounded weights: one rounding per
        # product and K - 1 per sum, to first order K u sum|w h|
        bound = K * 2.0 ** -24 * np.abs(prod).sum(axis=1)
        assert np.all(np.abs(got[m] - prod.sum(axis=1)) <= bound)


def test_fp8_quantizer_error_bound_and_zero(oracle_mod):
    # nearest rounding: |w - deq| <= half the E4M3 spacing at w (times g);
    # zeros map to code 0
    wb = S.normal_bf16_rows(11, 16, 256, 0.02)
    wb[0, :4] = S.f32_to_bf16_bits(np.array([0.0, -0.0, 0.0, 0.0], np.float32))
    q, g = S.quantize_fp8(wb)
    e4 = np.array([oracle_mod.e4m3(b) for b in range(256)])
    w = S.bf16_bits_to_f32(wb).astype(np.float64)
    deq = e4[q] * g
    a = np.abs(w) / g
    _, p = np.frexp(np.where(a > 0, a, 1.0))
    spacing = np.ldexp(1.0, np.maximum(p - 1, -6) - 3) * g
    assert np.all(np.abs(w - deq) <= spacing / 2 + 1e-30)
    assert np.all(q[0, :4] & 0x7F == 0)
