"""CPU-side checks of the C-ABI library: it loads, exports every symbol the
header declares, its host-only ranks builder matches the oracle's, and the
argument checks reject bad calls before touching the GPU."""
import ctypes
import os
import re

import numpy as np
import pytest

from conftest import ROOT
import synthetic as S


@pytest.fixture(scope="session")
def dvl():
    from draft_vocab_lm_gb300 import build
    build.build()
    import draft_vocab_lm_gb300 as d
    return d


def _declared_symbols():
    text = open(os.path.join(ROOT, "include", "dvl.h")).read()
    return sorted(set(re.findall(r"\b(dvl_[a-z_0-9]+)\s*\(", text)))


def test_exports_every_declared_symbol(dvl):
    from draft_vocab_lm_gb300 import _native
    lib = _native.lib()
    declared = _declared_symbols()
    assert set(declared) == set(_native.EXPORTS)
    for name in declared:
        assert hasattr(lib, name), name
    assert dvl.version() == 101
    assert lib.dvl_last_error() == b"no error"
    assert lib.dvl_status_string(0) == b"ok"
    assert lib.dvl_status_string(4) == b"workspace missing or too small"


def test_workspace_bytes(dvl):
    assert dvl.workspace_bytes(1, 1) == 512
    assert dvl.workspace_bytes(32, 1) == 512
    # per-block lists for up to 1,024 blocks, 64 group lists, 64 group tickets
    assert dvl.workspace_bytes(3, 4) == 512 + (1024 + 64) * 3 * 4 * 8 + 64 * 4
    assert dvl.workspace_bytes(0, 1) == 0
    assert dvl.workspace_bytes(33, 1) == 0
    assert dvl.workspace_bytes(1, 5) == 0


@pytest.mark.parametrize("seed", range(4))
def test_build_ranks_matches_oracle(dvl, oracle_mod, seed):
    rng = np.random.default_rng(seed)
    V = 5000
    tokens = S.zipf_tokens(seed, V, 40_000)
    c_lib = dvl.histogram(tokens, V)
    c_or = oracle_mod.histogram(tokens, V)
    assert np.array_equal(c_lib, c_or)
    forced = rng.integers(0, V, size=300).astype(np.int32)
    for N in (1, 100, 2500, V, V + 10):
        for srt in (False, True):
            a = dvl.build_ranks(c_lib, N, forced, sorted_ids=srt)
            b = oracle_mod.build_ranks(c_or, N, forced, sorted_ids=srt)
            assert np.array_equal(a, b), (N, srt)


def test_union_matches_oracle_and_printed_counts(dvl, oracle_mod):
    A, B = S.union_sets(3, S.V_FULL, 47149, 9749, 9749 - 5606)
    u = dvl.union_sorted(A, B)
    assert np.array_equal(u, oracle_mod.union_sorted(A, B))
    assert u.shape[0] == 52755
    assert dvl.union_sorted([], []).shape[0] == 0
    assert list(dvl.union_sorted([3, 1, 3], [2, 1])) == [1, 2, 3]


def test_frspec_ranks_from_zipf_stream(dvl, oracle_mod):
    # the trim list of the 32,768-row workload: top ranks of a Zipf stream
    tokens = S.zipf_tokens(2, S.V_FULL, 1_000_000)
    counts = dvl.histogram(tokens, S.V_FULL)
    ranks = dvl.build_ranks(counts, 32768)
    assert np.array_equal(ranks, oracle_mod.build_ranks(counts, 32768))
    assert len(set(ranks.tolist())) == 32768
    assert np.all(np.diff(counts[ranks]) <= 0)  # rank order


def test_host_builder_errors(dvl):
    with pytest.raises(dvl.DvlError) as e:
        dvl.histogram(np.array([0, 7], np.int32), 5)
    assert e.value.status == 2
    with pytest.raises(dvl.DvlError) as e:
        dvl.build_ranks(np.zeros(5, np.int64), 3, forced=[9])
    assert e.value.status == 2


def test_ranks_txt_roundtrip(dvl, tmp_path):
    ids = np.array([5, 0, 248319, 77], np.int32)
    p = tmp_path / "ranks.txt"
    dvl.write_ranks_txt(str(p), ids)
    assert p.read_text() == "5\n0\n248319\n77\n"
    assert np.array_equal(dvl.read_ranks_txt(str(p)), ids)


def _head(**kw):
    from draft_vocab_lm_gb300._native import DvlHead
    h = DvlHead()
    h.dtype, h.N, h.K, h.V = 0, 100, 256, 100
    h.w = 0x1000
    for k, v in kw.items():
        setattr(h, k, v)
    return h


@pytest.mark.parametrize("bad", [
    dict(dtype=7), dict(N=0), dict(K=100), dict(K=0), dict(K=24576 + 64), dict(flags=2), dict(reserved2=1),
    dict(w=None), dict(w=0x1004), dict(dtype=1), dict(V=50), dict(id_base=1),
])
def test_argument_checks_reject_before_any_launch(dvl, bad):
    # pointer values are never dereferenced: the checks fail first
    from draft_vocab_lm_gb300._native import lib
    L = lib()
    h = _head(**bad)
    ids = ctypes.c_void_p(0x2000)
    st = L.dvl_draft_argmax(ctypes.byref(h), 0x3000, 1, ids, 0x4000, 0x5000, 1 << 20, None)
    assert st == 1


def test_workspace_and_shape_checks(dvl):
    from draft_vocab_lm_gb300._native import lib
    L = lib()
    h = _head()
    assert L.dvl_draft_argmax(ctypes.byref(h), 0x3000, 0, 0x2000, 0x4000, 0x5000, 1 << 20, None) == 1
    assert L.dvl_draft_argmax(ctypes.byref(h), 0x3000, 33, 0x2000, 0x4000, 0x5000, 1 << 20, None) == 1
    assert L.dvl_draft_argmax(ctypes.byref(h), 0x3008, 1, 0x2000, 0x4000, 0x5000, 1 << 20, None) == 1
    assert L.dvl_draft_argmax(ctypes.byref(h), 0x3000, 1, 0x2000, 0x4000, 0x5000, 100, None) == 4
    assert L.dvl_draft_argmax(ctypes.byref(h), 0x3000, 1, 0x2000, 0x4000, None, 1 << 20, None) == 4
    assert L.dvl_draft_topk(ctypes.byref(h), 0x3000, 2, 5, 0x2000, 0x4000, 0x5000, 1 << 20, None) == 1
    small = _head(N=3)
    assert L.dvl_draft_topk(ctypes.byref(small), 0x3000, 1, 4, 0x2000, 0x4000, 0x5000, 1 << 20, None) == 1
    assert L.dvl_draft_topk(ctypes.byref(h), 0x3000, 2, 4, 0x2000, 0x4000, 0x5000, 1000, None) == 4


def test_trim_checks_reject_bad_ranks_before_any_launch(dvl):
    from draft_vocab_lm_gb300._native import lib
    L = lib()
    h = _head()
    ranks = (ctypes.c_int32 * 3)(1, 100, 2)  # 100 is outside [0, V)
    st = L.dvl_trim_head(ctypes.byref(h), ranks, 3, 0x1000, None, 0x2000, None, None)
    assert st == 2
    neg = (ctypes.c_int32 * 1)(-1)
    assert L.dvl_trim_head(ctypes.byref(h), neg, 1, 0x1000, None, 0x2000, None, None) == 2
    sliced = _head(N=50)  # not a full head
    assert L.dvl_trim_head(ctypes.byref(sliced), ranks, 1, 0x1000, None, 0x2000, None, None) == 1


@pytest.mark.parametrize("bad", [
    dict(dtype=7), dict(N=0), dict(K=100), dict(flags=2), dict(w=None), dict(dtype=1),
    dict(d2t=0x6000),
])
def test_score_checks_reject_bad_heads_before_any_launch(dvl, bad):
    # a head with d2t has no row for an arbitrary full id: refused
    from draft_vocab_lm_gb300._native import lib
    L = lib()
    h = _head(**bad)
    assert L.dvl_score_ids(ctypes.byref(h), 0x3000, 1, 0x2000, 4, 0x4000, None) == 1


def test_score_shape_and_pointer_checks(dvl):
    from draft_vocab_lm_gb300._native import lib
    L = lib()
    h = _head()
    assert L.dvl_score_ids(ctypes.byref(h), 0x3000, 0, 0x2000, 4, 0x4000, None) == 1
    assert L.dvl_score_ids(ctypes.byref(h), 0x3000, 33, 0x2000, 4, 0x4000, None) == 1
    assert L.dvl_score_ids(ctypes.byref(h), 0x3000, 1, 0x2000, 0, 0x4000, None) == 1
    assert L.dvl_score_ids(ctypes.byref(h), 0x3000, 32, 0x2000, 0x7fffffff, 0x4000, None) == 1
    assert L.dvl_score_ids(ctypes.byref(h), 0x3008, 1, 0x2000, 4, 0x4000, None) == 1
    assert L.dvl_score_ids(ctypes.byref(h), 0x3000, 1, None, 4, 0x4000, None) == 1
    assert L.dvl_score_ids(ctypes.byref(h), 0x3000, 1, 0x2002, 4, 0x4000, None) == 1
    assert L.dvl_score_ids(ctypes.byref(h), 0x3000, 1, 0x2000, 4, None, None) == 1


def test_learn_checks_reject_before_any_launch(dvl):
    from draft_vocab_lm_gb300._native import lib
    L = lib()
    h = _head()
    ids = (ctypes.c_int32 * 3)(4, 100, 7)  # 100 is outside [0, V)
    assert L.dvl_learn_rows(ctypes.byref(h), ids, 3, 10, 0x1000, None, 0x2000, None) == 2
    ok = (ctypes.c_int32 * 2)(4, 7)
    assert L.dvl_learn_rows(ctypes.byref(h), ok, 0, 10, 0x1000, None, 0x2000, None) == 1
    assert L.dvl_learn_rows(ctypes.byref(h), ok, 2, -1, 0x1000, None, 0x2000, None) == 1
    assert L.dvl_learn_rows(ctypes.byref(h), ok, 2, 0x7fffffff, 0x1000, None, 0x2000, None) == 1
    assert L.dvl_learn_rows(ctypes.byref(h), None, 2, 0, 0x1000, None, 0x2000, None) == 1
    assert L.dvl_learn_rows(ctypes.byref(h), ok, 2, 0, 0x1008, None, 0x2000, None) == 1
    assert L.dvl_learn_rows(ctypes.byref(h), ok, 2, 0, 0x1000, None, 0x2002, None) == 1
    sliced = _head(N=50)  # not a full head
    assert L.dvl_learn_rows(ctypes.byref(sliced), ok, 2, 0, 0x1000, None, 0x2000, None) == 1
    nv = _head(dtype=1, scales=None)  # NVFP4 without scales
    assert L.dvl_learn_rows(ctypes.byref(nv), ok, 2, 0, 0x1000, None, 0x2000, None) == 1


def test_learn_missing_selects_on_the_host(dvl):
    # the repair step's decision: ids the list holds, repeats and ids past
    # the capacity are not learned; a call that learns nothing enqueues
    # nothing (so this runs without a GPU); an id outside [0, V) changes
    # nothing
    from draft_vocab_lm_gb300._native import lib
    L = lib()
    h = _head()
    row_of = np.full(100, -1, dtype=np.int32)
    row_of[[4, 7, 50]] = [0, 1, 2]
    learned = np.zeros(8, dtype=np.int32)
    rows, nl = ctypes.c_int32(3), ctypes.c_int32(-1)

    def call(ids, cap):
        ids = np.ascontiguousarray(ids, dtype=np.int32)
        return L.dvl_learn_missing(ctypes.byref(h), ids.ctypes.data if ids.size else None,
                                   ids.size, row_of.ctypes.data, ctypes.byref(rows), cap,
                                   0x1000, None, 0x2000, learned.ctypes.data, ctypes.byref(nl),
                                   None)
    assert call([7, 4, 50, 7], 10) == 0 and nl.value == 0 and rows.value == 3
    assert call([], 10) == 0 and nl.value == 0
    assert call([8, 8, 9], 3) == 0 and nl.value == 0 and rows.value == 3  # no spare row
    before = row_of.copy()
    assert call([8, 100], 10) == 2 and rows.value == 3  # 100 is outside [0, V)
    assert np.array_equal(row_of, before)
    assert call([8], 2) == 1  # capacity below the rows in use
    nv = _head(dtype=1, scales=None)
    assert L.dvl_learn_missing(ctypes.byref(nv), None, 0, row_of.ctypes.data, ctypes.byref(rows),
                               10, 0x1000, None, 0x2000, learned.ctypes.data, ctypes.byref(nl),
                               None) == 1


def test_fp8_head_checks(dvl):
    # FP8 heads take no per-block scales; a valid FP8 head passes the head
    # checks (the out-of-range id is what a trim then refuses)
    from draft_vocab_lm_gb300._native import lib, DVL_FP8
    L = lib()
    ids = (ctypes.c_int32 * 2)(4, 100)
    fp8 = _head(dtype=DVL_FP8)
    assert L.dvl_learn_rows(ctypes.byref(fp8), ids, 2, 0, 0x1000, None, 0x2000, None) == 2
    with_scales = _head(dtype=DVL_FP8, scales=0x7000)
    assert L.dvl_learn_rows(ctypes.byref(with_scales), ids, 2, 0, 0x1000, None, 0x2000, None) == 1
    assert L.dvl_score_ids(ctypes.byref(with_scales), 0x3000, 1, 0x2000, 4, 0x4000, None) == 1
    bf16_scales = _head(scales=0x7000)
    assert L.dvl_score_ids(ctypes.byref(bf16_scales), 0x3000, 1, 0x2000, 4, 0x4000, None) == 1
    unknown = _head(dtype=3)
    assert L.dvl_score_ids(ctypes.byref(unknown), 0x3000, 1, 0x2000, 4, 0x4000, None) == 1


def test_quantize_checks_reject_before_any_launch(dvl):
    from draft_vocab_lm_gb300._native import lib, DVL_NVFP4, DVL_FP8
    L = lib()
    g = ctypes.c_float(0.0)
    h = _head()
    ok_ws = 0x5000
    # target format, source format, pointers, scales presence, workspace
    assert L.dvl_quantize_head(ctypes.byref(h), 0, 0x1000, None, ctypes.byref(g), ok_ws, 512, None) == 1
    assert L.dvl_quantize_head(ctypes.byref(_head(dtype=DVL_FP8)), DVL_FP8, 0x1000, None,
                               ctypes.byref(g), ok_ws, 512, None) == 1
    assert L.dvl_quantize_head(ctypes.byref(h), DVL_FP8, 0x1008, None, ctypes.byref(g), ok_ws, 512, None) == 1
    assert L.dvl_quantize_head(ctypes.byref(h), DVL_FP8, 0x1000, 0x2000, ctypes.byref(g), ok_ws, 512, None) == 1
    assert L.dvl_quantize_head(ctypes.byref(h), DVL_NVFP4, 0x1000, None, ctypes.byref(g), ok_ws, 512, None) == 1
    assert L.dvl_quantize_head(ctypes.byref(h), DVL_NVFP4, 0x1000, 0x2000, None, ok_ws, 512, None) == 1
    assert L.dvl_quantize_head(ctypes.byref(h), DVL_FP8, 0x1000, None, ctypes.byref(g), None, 512, None) == 4
    assert L.dvl_quantize_head(ctypes.byref(h), DVL_FP8, 0x1000, None, ctypes.byref(g), ok_ws, 100, None) == 4


def test_plan_without_a_device(dvl):
    # argument checks first; low-bit plans need no device; bf16 plans for
    # three or more rows read the SM count (DVL_ERR_CUDA without a device)
    from draft_vocab_lm_gb300._native import lib, DVL_FP8, DVL_NVFP4
    L = lib()
    name, n = ctypes.c_char_p(), ctypes.c_int32()
    h = _head()
    assert L.dvl_draft_plan(ctypes.byref(h), 0, 1, ctypes.byref(name), ctypes.byref(n)) == 1
    assert L.dvl_draft_plan(ctypes.byref(h), 1, 5, ctypes.byref(name), ctypes.byref(n)) == 1
    assert L.dvl_draft_plan(ctypes.byref(h), 1, 1, None, ctypes.byref(n)) == 1
    assert L.dvl_draft_plan(ctypes.byref(_head(K=100)), 1, 1, ctypes.byref(name), ctypes.byref(n)) == 1
    st = L.dvl_draft_plan(ctypes.byref(h), 5, 4, ctypes.byref(name), ctypes.byref(n))
    assert st in (0, 5)
    if st == 0:  # a 100-row head is below the register-path threshold
        assert (name.value, n.value) == (b"bf16-tcgen05", 1)
    assert L.dvl_draft_plan(ctypes.byref(_head(dtype=DVL_FP8)), 3, 1, ctypes.byref(name),
                            ctypes.byref(n)) == 0
    assert (name.value, n.value) == (b"fp8-mma", 1)
    nv = _head(dtype=DVL_NVFP4, scales=0x7000, K=5120)
    assert L.dvl_draft_plan(ctypes.byref(nv), 32, 4, ctypes.byref(name), ctypes.byref(n)) == 0
    # one launch per 16 hidden rows at width 5,120
    assert name.value == b"nvfp4-mma" and n.value == 2


def test_call_stream_handle_without_a_device(dvl, monkeypatch):
    # an explicit stream (object or raw handle) is passed through unchanged;
    # the current stream is read as a raw handle when torch offers that
    import types
    import draft_vocab_lm_gb300 as d
    torch = pytest.importorskip("torch")
    t = torch.zeros(1)
    assert d._call_stream(types.SimpleNamespace(cuda_stream=1234), t) == 1234
    assert d._call_stream(77, t) == 77
    monkeypatch.setattr(d, "_raw_stream_fn", lambda dev_index: 4242 + dev_index)
    t.get_device = lambda: 0  # a CPU tensor reports -1
    assert d._call_stream(None, t) == 4242


def test_noalloc_checks_reject_before_any_launch(dvl):
    # the fixed scratch holds at most DVL_MAX_M rows; bad heads and pointers
    # fail before the scratch is looked up (no device needed)
    from draft_vocab_lm_gb300._native import lib
    L = lib()
    good, bad = _head(), _head(K=100)
    for M in (0, -1, 33):
        assert L.dvl_draft_argmax_noalloc(ctypes.byref(good), 0x3000, M, 0x2000, 0x4000, None) == 1
    assert L.dvl_draft_argmax_noalloc(ctypes.byref(bad), 0x3000, 1, 0x2000, 0x4000, None) == 1
    assert L.dvl_draft_argmax_noalloc(ctypes.byref(good), None, 1, 0x2000, 0x4000, None) == 1
    assert L.dvl_draft_argmax_noalloc(ctypes.byref(good), 0x3008, 1, 0x2000, 0x4000, None) == 1
    assert L.dvl_draft_argmax_noalloc(ctypes.byref(good), 0x3000, 1, None, 0x4000, None) == 1
    assert L.dvl_draft_argmax_noalloc(ctypes.byref(good), 0x3000, 1, 0x2000, 0x4002, None) == 1
    assert L.dvl_noalloc_status(None, None) == 1
