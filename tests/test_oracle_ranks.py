"""Pins of the oracle's ranks builder (histogram, top-N after a forced set,
set union) to brute force with Python's own sort and set operations and to
the counts the pages print."""
import numpy as np
import pytest

from conftest import read_kv
import synthetic as S


def _brute_ranks(counts, forced, N, sorted_ids):
    forced_set = []
    for f in forced:
        if f not in forced_set:
            forced_set.append(int(f))
    key = lambda t: (-int(counts[t]), t)
    first = sorted(forced_set, key=key)
    rest = sorted((t for t in range(len(counts)) if t not in set(forced_set)), key=key)
    out = (first + rest)[:min(N, len(counts))]
    return sorted(out) if sorted_ids else out


@pytest.mark.parametrize("seed", range(5))
def test_build_ranks_bruteforce(oracle_mod, seed):
    rng = np.random.default_rng(seed)
    V = 60
    tokens = rng.integers(0, V, size=200).astype(np.int32)
    counts = oracle_mod.histogram(tokens, V)
    assert np.array_equal(counts, np.bincount(tokens, minlength=V))
    forced = rng.integers(0, V, size=7).astype(np.int32)  # may repeat
    for N in (0, 5, 20, V, V + 3):
        for srt in (False, True):
            got = oracle_mod.build_ranks(counts, N, forced, srt)
            assert list(got) == _brute_ranks(counts, forced, N, srt)


def test_histogram_accumulates_and_rejects_out_of_range(oracle_mod):
    c = oracle_mod.histogram(np.array([1, 1, 2], np.int32), 4)
    c = oracle_mod.histogram(np.array([2, 3], np.int32), 4, c)
    assert list(c) == [0, 2, 2, 1]
    with pytest.raises(ValueError):
        oracle_mod.histogram(np.array([4], np.int32), 4)
    with pytest.raises(ValueError):
        oracle_mod.build_ranks(np.zeros(4, np.int64), 2, np.array([9], np.int32))


@pytest.mark.parametrize("seed", range(4))
def test_union_bruteforce(oracle_mod, seed):
    rng = np.random.default_rng(seed)
    a = rng.integers(0, 50, size=30).astype(np.int32)
    b = rng.integers(0, 50, size=17).astype(np.int32)
    assert list(oracle_mod.union_sorted(a, b)) == sorted(set(a.tolist()) | set(b.tolist()))
    assert list(oracle_mod.union_sorted(a[:0], b[:0])) == []


def test_union_reproduces_printed_merge_counts(oracle_mod):
    p = read_kv("page_numbers.txt")
    na, nb = int(p["union_a"]), int(p["union_b"])
    n_new, n_union = int(p["union_b_new"]), int(p["union_size"])
    assert na + n_new == n_union
    A, B = S.union_sets(3, S.V_FULL, na, nb, nb - n_new)
    U = oracle_mod.union_sorted(A, B)
    assert len(set(A.tolist())) == na and len(set(B.tolist())) == nb
    assert len(set(B.tolist()) - set(A.tolist())) == n_new
    assert U.shape[0] == n_union
    assert np.all(np.diff(U) > 0)


def test_16k_composition_counts(oracle_mod):
    # every id below 8,192 + a structural core (3,531 of its 4,152 ids above
    # 8,192) + the most frequent remaining ids until 16,000
    p = read_kv("page_numbers.txt")
    low, core, above, total = (int(p[k]) for k in ("sl_low", "sl_core", "sl_core_above",
                                                  "sl_total"))
    low_ids, core_ids = S.structural_forced_set(0, S.V_FULL, low, core, above)
    forced = np.concatenate([low_ids, core_ids])
    tokens = S.zipf_tokens(0, S.V_FULL, 200_000)
    counts = oracle_mod.histogram(tokens, S.V_FULL)
    ranks = oracle_mod.build_ranks(counts, total, forced, sorted_ids=False)
    assert ranks.shape[0] == total
    n_forced = len(set(forced.tolist()))
    assert n_forced == low + above
    fill = ranks[n_forced:]
    assert fill.shape[0] == total - low - above == 4277
    assert set(forced.tolist()) <= set(ranks.tolist())
    # the fill is the most frequent non-forced ids, by (count desc, id asc)
    rest = np.setdiff1d(np.arange(S.V_FULL), forced)
    order = rest[np.lexsort((rest, -counts[rest]))]
    assert np.array_equal(fill, order[:fill.shape[0]])
