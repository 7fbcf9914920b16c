"""Pins for the oracle's budgeted Top-K and gather-compaction.

Top-K keeps the k - R best tokens of [0, T - R) by (z descending, position
ascending) plus the protected recent window [T - R, T) (H2O page, 双缓冲), each
head on its own (按头独立驱逐).  Compaction is the "real drop" of the evicted
rows (两套代码) into a preallocated slot cache (FlexGen 改造).
"""
import itertools

import numpy as np
import pytest


def _brute_best(z, k, R):
    """Exhaustive: the (k-R)-subset of [0, T-R) with the largest sum; among equal
    sums the one whose sorted (z desc, pos asc) sequence is lexicographically first."""
    T = len(z)
    best = None
    for sub in itertools.combinations(range(T - R), k - R):
        key = (-sum(z[i] for i in sub), sorted((-z[i], i) for i in sub))
        if best is None or key < best[0]:
            best = (key, sub)
    return sorted(list(best[1]) + list(range(T - R, T)))


@pytest.mark.parametrize("seed", range(6))
def test_exhaustive_small(oracle_mod, seed):
    rng = np.random.default_rng(seed)
    for T in range(1, 10):
        for k in range(1, T + 1):
            for R in range(0, k):
                z = rng.integers(0, 4, size=T).astype(np.float64)  # many ties
                idx = oracle_mod.select_topk(z[None, None], k, R)[0, 0]
                assert list(idx) == _brute_best(list(z), k, R), (T, k, R, z)


def test_exhaustive_small_signed_scores(oracle_mod):
    """Negative scores and -0.0 beside +0.0 (equal: the lower position wins)."""
    rng = np.random.default_rng(99)
    values = np.array([-3.0, -1.0, -0.0, 0.0, 2.0])
    for T in range(1, 9):
        for k in range(1, T + 1):
            for R in range(0, k):
                z = values[rng.integers(0, len(values), size=T)]
                idx = oracle_mod.select_topk(z[None, None], k, R)[0, 0]
                assert list(idx) == _brute_best(list(z), k, R), (T, k, R, z)


def test_order_characterisation_and_library_sort(oracle_mod):
    rng = np.random.default_rng(20)
    B, H, T, k, R = 2, 3, 500, 60, 17
    z = np.round(rng.random((B, H, T)) * 50) / 7  # ties
    idx = oracle_mod.select_topk(z, k, R)
    for b in range(B):
        for h in range(H):
            got = idx[b, h]
            assert len(got) == k and np.all(np.diff(got) > 0)
            assert set(range(T - R, T)) <= set(got)
            heavy = set(got) - set(range(T - R, T))
            out = set(range(T - R)) - heavy
            for i in heavy:
                for j in out:
                    assert z[b, h, i] > z[b, h, j] or (z[b, h, i] == z[b, h, j] and i < j)
            order = np.lexsort((np.arange(T - R), -z[b, h, :T - R]))
            np.testing.assert_array_equal(np.sort(order[:k - R]), sorted(heavy))


def test_keep_all_when_budget_is_prompt(oracle_mod):
    z = np.random.default_rng(21).random((1, 2, 40))
    np.testing.assert_array_equal(oracle_mod.select_topk(z, 40, 5)[0, 1], np.arange(40))


def test_rejects_bad_budget(oracle_mod):
    z = np.zeros((1, 1, 10))
    for k, R in ((5, 5), (11, 0), (0, 0)):
        with pytest.raises(ValueError):
            oracle_mod.select_topk(z, k, R)


@pytest.mark.parametrize("bits", [True, False])
def test_compact_is_fancy_indexing(oracle_mod, bits):
    rng = np.random.default_rng(22)
    B, H, T, d, k, cap = 2, 3, 50, 8, 11, 13
    if bits:
        K = rng.integers(0, 2 ** 16, size=(B, H, T, d), dtype=np.uint16)
        V = rng.integers(0, 2 ** 16, size=(B, H, T, d), dtype=np.uint16)
    else:
        K = rng.standard_normal((B, H, T, d)).astype(np.float32)
        V = rng.standard_normal((B, H, T, d)).astype(np.float32)
    s = rng.random((B, H, T))
    idx = np.sort(np.stack([np.stack([rng.choice(T, k, replace=False) for _ in range(H)])
                            for _ in range(B)]), axis=-1).astype(np.int32)
    Ko, Vo, pos, acc, ln = oracle_mod.compact(K, V, s, idx, cap)
    bi = np.arange(B)[:, None, None]
    hi = np.arange(H)[None, :, None]
    np.testing.assert_array_equal(Ko[:, :, :k], K[bi, hi, idx])
    np.testing.assert_array_equal(Vo[:, :, :k], V[bi, hi, idx])
    np.testing.assert_array_equal(pos[:, :, :k], idx)
    np.testing.assert_array_equal(acc[:, :, :k], s[bi, hi, idx].astype(np.float32))
    np.testing.assert_array_equal(ln, k)
    assert not Ko[:, :, k:].any() and not pos[:, :, k:].any()


def test_kv_cache_bytes_worked_examples(oracle_mod):
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "kv_cache_bytes.txt")
    n = 0
    for line in open(path):
        if line.startswith("#") or not line.strip():
            continue
        name, L, H, d, T, eb, want, *_ = line.split()
        assert oracle_mod.kv_cache_bytes(int(L), int(H), int(d), int(T), int(eb)) == int(want), name
        n += 1
    assert n == 3
