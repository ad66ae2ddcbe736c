"""dvl_draft_argmax_noalloc and dvl_noalloc_status, called through the C ABI.

Some callers cannot allocate device memory: plugins inside an inference
engine that owns every allocation, and decode loops that cannot afford
cudaMalloc's stall.  For them the library keeps the argmax's reduction
scratch in its own static device array.  Here every kernel family reaches
that entry point (CUDA cores at 1 and 2 hidden rows, the register-path
tensor cores at 3 to 16, tcgen05 at 32, NVFP4 and FP8 heads), each head on
two calls in a row, and each result is checked against the CPU oracle by
the parity rule -- which also shows that one call leaves the shared scratch
usable for the next.  A d2t entry outside the vocabulary that wins is
reported through dvl_noalloc_status, and the bit survives later calls until
it is read.  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest

import synthetic as S
from parity import check_argmax

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

OUT_OF_RANGE_BIT = 1 << 2  # 1 << DVL_ERR_OUT_OF_RANGE


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


def noalloc(dvl, head, h):
    """One dvl_draft_argmax_noalloc call on the current stream."""
    from draft_vocab_lm_gb300._native import lib
    L = lib()
    M = h.shape[0]
    ids = torch.full((M,), -9, dtype=torch.int32, device="cuda")
    vals = torch.zeros(M, dtype=torch.float32, device="cuda")
    rc = L.dvl_draft_argmax_noalloc(ctypes.byref(head.struct()), h.data_ptr(), M,
                                    ids.data_ptr(), vals.data_ptr(),
                                    torch.cuda.current_stream().cuda_stream)
    assert rc == 0, L.dvl_last_error()
    return ids, vals


def status(dvl):
    from draft_vocab_lm_gb300._native import lib
    bits = ctypes.c_uint32(0xdead)
    assert lib().dvl_noalloc_status(ctypes.byref(bits),
                                    torch.cuda.current_stream().cuda_stream) == 0
    return int(bits.value)


def test_noalloc_argmax_matches_the_oracle_on_every_kernel_family(dvl, oracle_mod):
    status(dvl)  # start from a read (and so cleared) status word
    N, K, V = 20_000, 2560, 248_320
    w = S.normal_bf16_rows(12, N, K, 0.02)
    rng = np.random.default_rng(12)
    d2t = np.sort(rng.choice(V, size=N, replace=False)).astype(np.int32)
    head = dvl.Head(dev(w), V=V, d2t=dev(d2t))
    # 1, 2 rows: CUDA cores; 3, 5, 16: register-path tensor cores (20,000
    # rows is a long enough head on a 152-SM GB300); 32: tcgen05
    for M in (1, 2, 3, 5, 16, 32):
        for call in range(2):
            h = S.hidden_bf16(100 + 2 * M + call, M, K)
            ids, vals = noalloc(dvl, head, dev(h))
            torch.cuda.synchronize()
            L, _ = oracle_mod.logits_bf16(w, h)
            check_argmax(oracle_mod, L, d2t, ids.cpu().numpy(), vals.cpu().numpy())

    # the NVFP4 and FP8 heads (the low-bit tensor-core kernel)
    Nq, Kq = 4099, 5120
    wq = S.normal_bf16_rows(13, Nq, Kq, 0.02)
    q, sc, g = S.quantize_nvfp4(wq)
    dq = rng.permutation(V)[:Nq].astype(np.int32)
    h4 = dvl.Head(dev(q), scales=dev(sc), global_scale=g, V=V, d2t=dev(dq))
    q8, g8 = S.quantize_fp8(wq)
    h8 = dvl.Head(dev(q8), fmt="fp8", global_scale=g8, V=V, d2t=dev(dq))
    for M in (1, 3):
        for call in range(2):
            h = S.hidden_bf16(200 + 2 * M + call, M, Kq)
            ids, vals = noalloc(dvl, h4, dev(h))
            ids8, vals8 = noalloc(dvl, h8, dev(h))
            torch.cuda.synchronize()
            L, _ = oracle_mod.logits_nvfp4(q, sc, g, h)
            check_argmax(oracle_mod, L, dq, ids.cpu().numpy(), vals.cpu().numpy())
            L8, _ = oracle_mod.logits_fp8(q8, g8, h)
            check_argmax(oracle_mod, L8, dq, ids8.cpu().numpy(), vals8.cpu().numpy())
    assert status(dvl) == 0

    # beyond the fixed scratch: a clear error, nothing enqueued
    from draft_vocab_lm_gb300._native import lib
    h33 = torch.zeros((33, K), dtype=torch.int16, device="cuda")
    out = torch.zeros(33, dtype=torch.int32, device="cuda")
    assert lib().dvl_draft_argmax_noalloc(ctypes.byref(head.struct()), h33.data_ptr(), 33,
                                          out.data_ptr(), out.data_ptr(),
                                          torch.cuda.current_stream().cuda_stream) == 1


def test_noalloc_reports_an_out_of_range_d2t_entry_until_read(dvl, oracle_mod):
    status(dvl)
    N, K, V = 3001, 256, 50_000
    w = S.normal_bf16_rows(14, N, K, 0.02)
    h = S.hidden_bf16(14, 1, K)
    L, _ = oracle_mod.logits_bf16(w, h)
    win = int(np.argmax(L[0]))
    d2t = np.random.default_rng(14).permutation(V)[:N].astype(np.int32)
    bad = d2t.copy()
    bad[win] = V + 5  # the winning row's entry lies outside [0, V)
    ids, _ = noalloc(dvl, dvl.Head(dev(w), V=V, d2t=dev(bad)), dev(h))
    torch.cuda.synchronize()
    assert int(ids[0]) == V + 5  # returned as it is
    # a clean call afterwards leaves the bit in place
    ids, vals = noalloc(dvl, dvl.Head(dev(w), V=V, d2t=dev(d2t)), dev(h))
    torch.cuda.synchronize()
    check_argmax(oracle_mod, L, d2t, ids.cpu().numpy(), vals.cpu().numpy())
    assert status(dvl) == OUT_OF_RANGE_BIT
    assert status(dvl) == 0  # read and cleared
