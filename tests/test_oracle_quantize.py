"""Pins of the oracle's requantization of a bf16 head to NVFP4 and FP8
("Masked MTP drafts": the trimmed head requantized to NVFP4 at load) to
things other than itself: blocks worked by hand from the recipe and the
format definitions (tests/golden/quantize_blocks.txt), covering ties to even,
signed zero, subnormals and saturation; the half-step rounding bound; and
the all-zero block."""
import os

import numpy as np

from conftest import GOLDEN
import synthetic as S


def _golden():
    d = {}
    with open(os.path.join(GOLDEN, "quantize_blocks.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            t = line.split()
            d[t[0]] = t[1:]
    return d


def test_nvfp4_hand_worked_blocks(oracle_mod):
    d = _golden()
    w = S.f32_to_bf16_bits(np.array([[float(x) for x in d["nvfp4_w"]]], np.float32))
    q, sc, g = oracle_mod.quantize_nvfp4(w)
    assert g == float(d["nvfp4_g"][0])
    assert sc[0].tolist() == [int(x, 16) for x in d["nvfp4_scales"]]
    assert q[0].tolist() == [int(x, 16) for x in d["nvfp4_bytes"]]


def test_fp8_hand_worked_row(oracle_mod):
    d = _golden()
    vals = [float(x) for x in d["fp8_w"]]
    w = S.f32_to_bf16_bits(np.array([vals * 8], np.float32))  # K = 64
    q, g = oracle_mod.quantize_fp8(w)
    assert g == float(d["fp8_g"][0])
    assert q[0, :8].tolist() == [int(x, 16) for x in d["fp8_bytes"]]
    assert q[0].tolist() == q[0, :8].tolist() * 8


def test_requantized_heads_round_to_nearest(oracle_mod):
    # every decoded weight lies within half a step of the format at its
    # quotient (E2M1 steps 0.5 / 1 / 2; E4M3 spacing 2^(e-3), subnormal 2^-9),
    # and saturation only at the largest value
    wb = S.normal_bf16_rows(3, 64, 512, 0.02)
    w = S.bf16_bits_to_f32(wb).astype(np.float64)
    q, sc, g = oracle_mod.quantize_nvfp4(wb)
    e2 = np.array([oracle_mod.e2m1(c) for c in range(16)])
    e4 = np.array([oracle_mod.e4m3(c) for c in range(256)])
    s = np.repeat(e4[sc], 16, axis=1)
    codes = np.stack([q & 0xF, q >> 4], axis=-1).reshape(w.shape)
    x = w / (s * g)
    step = np.where(np.abs(x) < 2, 0.5, np.where(np.abs(x) < 4, 1.0, 2.0))
    assert np.all(np.abs(e2[codes] - np.clip(x, -6, 6)) <= step / 2 + 1e-12)
    q8, g8 = oracle_mod.quantize_fp8(wb)
    x8 = np.abs(w) / g8
    _, p = np.frexp(np.where(x8 > 0, x8, 1.0))
    spacing = np.ldexp(1.0, np.maximum(p - 1, -6) - 3)
    assert np.all(np.abs(np.abs(e4[q8]) - np.minimum(x8, 448)) <= spacing / 2 + 1e-12)
    assert np.all(np.sign(e4[q8]) * np.sign(w) >= 0)


def test_zero_head_and_zero_block(oracle_mod):
    wb = np.zeros((2, 64), np.uint16)
    q, sc, g = oracle_mod.quantize_nvfp4(wb)
    assert g == 1.0 and not q.any() and not sc.any()
    q8, g8 = oracle_mod.quantize_fp8(wb)
    assert g8 == 1.0 and not q8.any()
    wb[0, 20] = S.f32_to_bf16_bits(np.array([3.0], np.float32))[0]
    q, sc, g = oracle_mod.quantize_nvfp4(wb)
    assert sc[0, 0] == 0 and sc[1].tolist() == [0] * 4 and not q[0, :8].any()
