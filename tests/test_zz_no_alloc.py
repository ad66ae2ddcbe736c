"""dvl_draft_argmax_noalloc, called through the C ABI: for callers that
cannot allocate device memory (plugins inside an engine that owns every
allocation; decode loops that cannot afford cudaMalloc's stall) the library
keeps the argmax's reduction scratch in its own static device array.  Its
results must equal dvl_draft_argmax's (same kernel, caller-owned workspace)
on two calls in a row, which also shows that the shared scratch is left
usable by the first call.  This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest

import synthetic as S
from parity import LOGIT_REL

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
    return torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).cuda()


def test_noalloc_argmax_matches_the_workspace_entry_point_twice(dvl):
    from draft_vocab_lm_gb300._native import DvlHead, lib
    L = lib()
    fn = L.dvl_draft_argmax_noalloc
    fn.argtypes = [ctypes.POINTER(DvlHead), ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p,
                   ctypes.c_void_p, ctypes.c_void_p]
    fn.restype = ctypes.c_int

    N, K, V = 20_000, 2560, 248_320
    w = S.normal_bf16_rows(12, N, K, 0.02)
    rng = np.random.default_rng(12)
    d2t = np.sort(rng.choice(V, size=N, replace=False)).astype(np.int32)
    head = dvl.Head(dev(w), V=V, d2t=dev(d2t))
    st = head.struct()
    stream = torch.cuda.current_stream().cuda_stream

    # 3, 5 and 16 rows run on the register-path tensor cores (20,000 rows is
    # a long enough head on a 152-SM GB300), 32 on tcgen05
    for call, M in enumerate((3, 5, 16, 32)):
        h = dev(S.hidden_bf16(100 + call, M, K))
        ids = torch.full((M,), -9, dtype=torch.int32, device="cuda")
        vals = torch.zeros(M, dtype=torch.float32, device="cuda")
        rc = fn(ctypes.byref(st), h.data_ptr(), M, ids.data_ptr(), vals.data_ptr(), stream)
        assert rc == 0, L.dvl_last_error()
        ref_ids, ref_vals = dvl.draft_argmax(head, h)
        torch.cuda.synchronize()
        assert np.array_equal(ids.cpu().numpy(), ref_ids.cpu().numpy()), call
        got, ref = vals.cpu().numpy(), ref_vals.cpu().numpy()
        assert np.all(np.abs(got - ref) <= LOGIT_REL * np.maximum(np.abs(ref), 1e-6)), call

    # beyond the fixed scratch: a clear error, nothing enqueued
    h33 = torch.zeros((33, K), dtype=torch.int16, device="cuda")
    out = torch.zeros(33, dtype=torch.int32, device="cuda")
    assert fn(ctypes.byref(st), h33.data_ptr(), 33, out.data_ptr(), out.data_ptr(), stream) == 1
