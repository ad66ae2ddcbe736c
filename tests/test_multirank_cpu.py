"""The vocabulary-split path on CPU ranks: two gloo ranks each hold a row
slice of a head, take the slice's argmax (the oracle stands in for the GPU
kernel here) and combine with one MAX all-reduce of packed keys; the result
must equal the whole head's argmax, including ties across ranks."""
import os
import socket

import numpy as np
import pytest

import synthetic as S
from draft_vocab_lm_gb300 import shard


def test_pack_keys_order_matches_result_order():
    logits = np.array([1.0, 1.0, -0.0, 0.0, -5.0, np.nan, np.inf, -np.inf, 3.5], np.float32)
    ids = np.array([7, 3, 9, 2, 0, 1, 40, 41, 5], np.int32)
    keys = shard.pack_keys(ids, logits)
    order = np.argsort(-keys, kind="stable")
    # inf, 3.5, 1.0 (id 3 then 7), +-0 (id 2 then 9), -5, -inf, NaN
    assert [int(ids[i]) for i in order] == [40, 5, 3, 7, 2, 9, 0, 41, 1]
    back_ids, back_lg = shard.unpack_keys(keys)
    assert np.array_equal(back_ids, ids)
    fin = ~np.isnan(logits)
    assert np.array_equal(back_lg[fin], np.where(logits[fin] == 0, 0.0, logits[fin]))
    assert np.isnan(back_lg[~fin]).all()


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    import oracle
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        N, K, M = 3000, 128, 4
        w = S.normal_bf16_rows(5, N, K, 0.02)
        h = S.hidden_bf16(5, M, K)
        # plant a cross-rank tie for row 0: the same row in both halves
        w[N - 1] = w[10]
        n0, n1 = N * rank // world, N * (rank + 1) // world
        L, _ = oracle.logits_bf16(w[n0:n1], h, nthreads=1)
        ids, vals = oracle.argmax(L)
        ids = ids + n0  # the slice's rows keep their full ids
        gi, gv = shard.allreduce_argmax(ids, vals)
        Lf, _ = oracle.logits_bf16(w, h, nthreads=1)
        wi, wv = oracle.argmax(Lf)
        out.put((rank, gi.tolist(), gv.tolist(), wi.tolist(), wv.tolist()))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_combine_to_the_whole_head_argmax():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, gi, gv, wi, wv in results:
        assert gi == wi and gv == wv


def test_combine_on_host_with_a_tie_picks_the_lower_id():
    parts = [(np.array([100, 5]), np.array([2.0, 1.0], np.float32)),
             (np.array([40, 6]), np.array([2.0, 1.5], np.float32))]
    ids, vals = shard.combine(parts)
    assert ids.tolist() == [40, 6] and vals.tolist() == [2.0, 1.5]
