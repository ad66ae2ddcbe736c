"""GPU requantization of bf16 heads (dvl_quantize_head) against the oracle's
recipe, bit for bit: NVFP4 codes and block scales and FP8 codes, and the
tensor scale, on the hand-worked blocks, on gaussian heads with planted
ties, zero blocks and signed zeros, and on the 32,768 x 5,120 trimmed head
of the FR-Spec workload shape; then the requantized heads drive the argmax
like host-quantized ones."""
import numpy as np
import pytest

import synthetic as S
from parity import check_argmax
from test_oracle_quantize import _golden

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


def test_hand_worked_blocks_on_gpu(dvl):
    d = _golden()
    w = S.f32_to_bf16_bits(np.array([[float(x) for x in d["nvfp4_w"]] * 2], np.float32))  # K = 64
    q, sc, g = dvl.quantize_head(dev(w), "nvfp4")
    assert g == float(d["nvfp4_g"][0])
    assert sc.cpu().numpy()[0].tolist() == [int(x, 16) for x in d["nvfp4_scales"]] * 2
    assert q.cpu().numpy()[0].tolist() == [int(x, 16) for x in d["nvfp4_bytes"]] * 2
    w8 = S.f32_to_bf16_bits(np.array([[float(x) for x in d["fp8_w"]] * 8], np.float32))
    q8, _, g8 = dvl.quantize_head(dev(w8), "fp8")
    assert g8 == float(d["fp8_g"][0])
    assert q8.cpu().numpy()[0, :8].tolist() == [int(x, 16) for x in d["fp8_bytes"]]


def _planted(seed, N, K):
    # gaussian rows plus ties on both grids, an all-zero block, signed zeros
    wb = S.normal_bf16_rows(seed, N, K, 0.02)
    w = S.bf16_bits_to_f32(wb).copy()
    w[0, :16] = 0.0
    w[1, 16:32] = -0.0
    w[2, :8] = [0.375, 0.125, -0.625, 0.875, 0.0625, -0.1875, 0.25, 0.3125]
    return S.f32_to_bf16_bits(w)


@pytest.mark.parametrize("N,K", [(3, 64), (257, 320), (1000, 2560), (64, 24576)])
def test_requantized_heads_match_the_oracle_bit_for_bit(dvl, oracle_mod, N, K):
    wb = _planted(N + K, N, K)
    q, sc, g = dvl.quantize_head(dev(wb), "nvfp4")
    oq, osc, og = oracle_mod.quantize_nvfp4(wb)
    assert g == og
    assert np.array_equal(sc.cpu().numpy(), osc)
    assert np.array_equal(q.cpu().numpy(), oq)
    q8, _, g8 = dvl.quantize_head(dev(wb), "fp8")
    oq8, og8 = oracle_mod.quantize_fp8(wb)
    assert g8 == og8
    assert np.array_equal(q8.cpu().numpy(), oq8)


def test_trimmed_head_requantized_on_gpu_then_drafted(dvl, oracle_mod):
    # the load-time path: trim a bf16 head, requantize the trimmed rows, draft
    N, K, M = 32768, 5120, 3
    wb = S.normal_bf16_rows(7, N, K, 0.02)
    ws = dvl.make_workspace(M, 1)
    q, sc, g = dvl.quantize_head(dev(wb), "nvfp4", ws=ws)
    oq, osc, og = oracle_mod.quantize_nvfp4(wb)
    assert g == og and np.array_equal(sc.cpu().numpy(), osc) and np.array_equal(q.cpu().numpy(), oq)
    torch.cuda.synchronize()
    assert bool((ws[:256] == 0).all())  # the workspace is left as it was found
    h = S.hidden_bf16(8, M, K)
    head = dvl.Head(q, scales=sc, global_scale=g)
    L, _ = oracle_mod.logits_nvfp4(oq, osc, og, h)
    ids, vals = dvl.draft_argmax(head, dev(h), ws=ws)
    check_argmax(oracle_mod, L, None, ids.cpu().numpy(), vals.cpu().numpy())
    q8, _, g8 = dvl.quantize_head(dev(wb), "fp8", ws=ws)
    oq8, og8 = oracle_mod.quantize_fp8(wb)
    assert g8 == og8 and np.array_equal(q8.cpu().numpy(), oq8)
