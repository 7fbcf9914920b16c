"""Pins for the layer-level competitive budget and the ragged compaction.

NestedKV technical summary, 3. Hoofd-gewijze Geheugentoewijzing: the heads of a
layer compete for one budget; the (token, head) pairs with the highest scores
win, and every head keeps a minimum.  KV-cache survey blog §4.4 (PyramidKV): the
budget is set per layer rather than per head.

What fixes the oracle here, apart from its own steps:
  * brute force on tiny rows: the kept set has the largest score sum among all
    sets that keep the protected positions, at least `floor` per head and
    `budget` in all; ties go to the lexicographically first (z desc, head asc,
    position asc) sequence;
  * exchange optimality at larger sizes (no swap of a kept and a dropped pair
    that keeps the set feasible raises the sum);
  * special cases: budget = H * floor is the per-head Top-K with k = floor;
    a single head is the per-head Top-K with k = budget;
  * the ragged compaction equals the uniform one head by head.
"""
import itertools

import numpy as np
import pytest


def _brute_budget(z, budget, floor, R, S):
    """z [H][T] -> list of per-head sorted kept positions, by exhaustive search."""
    H, T = z.shape
    middle = [(h, p) for h in range(H) for p in range(S, T - R)]
    free = budget - H * (S + R)
    best = None
    for sub in itertools.combinations(middle, free):
        counts = [0] * H
        for h, _ in sub:
            counts[h] += 1
        if min(counts) < floor - S - R:
            continue
        key = (-sum(z[h, p] for h, p in sub), sorted((-z[h, p], h, p) for h, p in sub))
        if best is None or key < best[0]:
            best = (key, sub)
    out = []
    for h in range(H):
        kept = set(range(S)) | set(range(T - R, T)) | {p for hh, p in best[1] if hh == h}
        out.append(sorted(kept))
    return out


def _split(idx, off):
    return [list(idx[off[h]:off[h + 1]]) for h in range(len(off) - 1)]


@pytest.mark.parametrize("seed", range(3))
def test_budget_matches_brute_force_on_tiny_rows(oracle_mod, seed):
    rng = np.random.default_rng(200 + seed)
    cases = 0
    for H in (1, 2, 3):
        for T in range(1, 6 if H < 3 else 5):
            for S in range(0, T + 1):
                for R in range(0, T + 1 - S):
                    for floor in range(max(1, S + R), T + 1):
                        for budget in range(H * floor, H * T + 1):
                            z = rng.integers(0, 3, size=(H, T)).astype(np.float64)  # many ties
                            idx, off = oracle_mod.select_budget(z[None], budget, floor, R, S)
                            got = _split(idx[0], off[0])
                            assert got == _brute_budget(z, budget, floor, R, S), (H, T, S, R, floor, budget, z)
                            cases += 1
    assert cases > 300


def test_budget_matches_brute_force_with_signed_scores(oracle_mod):
    """Negative scores, and -0.0 beside +0.0 (equal scores: the tie goes to the
    lower head, then the lower position)."""
    rng = np.random.default_rng(321)
    values = np.array([-2.0, -1.0, -0.0, 0.0, 1.0])
    cases = 0
    for H in (1, 2, 3):
        for T in range(1, 5):
            for S in range(0, T + 1):
                for R in range(0, T + 1 - S):
                    for floor in range(max(1, S + R), T + 1):
                        for budget in range(H * floor, H * T + 1):
                            z = values[rng.integers(0, len(values), size=(H, T))]
                            idx, off = oracle_mod.select_budget(z[None], budget, floor, R, S)
                            got = _split(idx[0], off[0])
                            assert got == _brute_budget(z, budget, floor, R, S), (H, T, S, R, floor, budget, z)
                            cases += 1
    assert cases > 200


def _check_exchange_optimal(z, kept, floor, R, S):
    """No feasible swap of a kept middle pair x for a dropped middle pair y
    raises the sum: within a head always feasible, across heads when x's head
    keeps more than `floor`."""
    H, T = z.shape
    in_mid = lambda p: S <= p < T - R  # noqa: E731
    counts = [len(k) for k in kept]
    kept_sets = [set(k) for k in kept]
    for h in range(H):
        kmid = [z[h, p] for p in kept_sets[h] if in_mid(p)]
        dmid = [z[h, p] for p in range(S, T - R) if p not in kept_sets[h]]
        if kmid and dmid:
            assert max(dmid) <= min(kmid)  # a head keeps a prefix of its own order
    lo_surplus = min((z[h, p] for h in range(H) if counts[h] > floor
                      for p in kept_sets[h] if in_mid(p)), default=np.inf)
    hi_dropped = max((z[h, p] for h in range(H) for p in range(S, T - R)
                      if p not in kept_sets[h]), default=-np.inf)
    assert hi_dropped <= lo_surplus


@pytest.mark.parametrize("H,T,budget,floor,R,S", [
    (8, 300, 8 * 40, 20, 8, 4),
    (8, 300, 8 * 40, 12, 8, 4),      # floor = sinks + recent: all heavy slots compete
    (5, 97, 5 * 30, 29, 0, 0),
    (32, 64, 32 * 10, 3, 2, 1),
    (3, 1000, 1200, 150, 64, 0),
])
def test_budget_invariants_and_exchange_optimality(oracle_mod, H, T, budget, floor, R, S):
    rng = np.random.default_rng(H * 1000 + T)
    scale = rng.lognormal(0.0, 1.5, size=(1, H, 1))   # heads on different scales
    z = rng.random((2, H, T)) ** 3 * scale
    idx, off = oracle_mod.select_budget(z, budget, floor, R, S)
    for b in range(2):
        assert off[b, 0] == 0 and off[b, H] == budget and np.all(np.diff(off[b]) >= floor)
        kept = _split(idx[b], off[b])
        for h, kh in enumerate(kept):
            assert np.all(np.diff(kh) > 0)
            assert set(range(S)) <= set(kh) and set(range(T - R, T)) <= set(kh)
        _check_exchange_optimal(z[b], kept, floor, R, S)


def test_budget_with_floor_filling_it_is_per_head_topk(oracle_mod):
    rng = np.random.default_rng(210)
    z = rng.random((3, 6, 250))
    z[..., 10:20] = 0.5                       # ties
    for k, R, S in [(40, 8, 0), (40, 8, 4), (25, 0, 3), (250, 10, 0)]:
        idx, off = oracle_mod.select_budget(z, 6 * k, k, R, S)
        np.testing.assert_array_equal(off, np.tile(np.arange(7) * k, (3, 1)))
        np.testing.assert_array_equal(idx.reshape(3, 6, k), oracle_mod.select_topk(z, k, R, sink=S))


def test_budget_single_head_is_per_head_topk(oracle_mod):
    rng = np.random.default_rng(211)
    z = rng.random((4, 1, 180))
    for k, floor, R, S in [(50, 10, 10, 0), (50, 12, 8, 4), (50, 50, 8, 4), (51, 1, 0, 0)]:
        idx, off = oracle_mod.select_budget(z, k, floor, R, S)
        np.testing.assert_array_equal(idx[:, None, :], oracle_mod.select_topk(z, k, R, sink=S))
        assert np.all(off[:, 1] == k)


def test_budget_moves_slots_to_the_heads_with_the_mass(oracle_mod):
    # head 0 holds all the large scores: it takes everything above the floors
    z = np.zeros((1, 4, 100))
    z[0, 0] = np.linspace(10, 20, 100)
    z[0, 1:] = np.linspace(0, 1, 100)
    idx, off = oracle_mod.select_budget(z, 4 * 20, 5, 2, 1)
    np.testing.assert_array_equal(np.diff(off[0]), [65, 5, 5, 5])
    # equal scores across heads: the tie goes to the lower head index
    z = np.ones((1, 3, 10))
    idx, off = oracle_mod.select_budget(z, 12, 2, 0, 0)
    np.testing.assert_array_equal(np.diff(off[0]), [8, 2, 2])
    np.testing.assert_array_equal(idx[0, :8], np.arange(8))


def test_budget_rejects_bad_arguments(oracle_mod):
    z = np.zeros((1, 2, 10))
    for budget, floor, R, S in [(3, 2, 0, 0),      # budget < H * floor
                                (21, 2, 0, 0),     # budget > H * T
                                (10, 2, 2, 1),     # floor < sinks + recent
                                (10, 0, 0, 0),     # floor < 1
                                (10, 11, 0, 0),    # floor > T
                                (10, 3, -1, 0), (10, 3, 0, -1)]:
        with pytest.raises(ValueError):
            oracle_mod.select_budget(z, budget, floor, R, S)


# ---------------------------------------------------------------- ragged compaction
def test_compact_ragged_equals_uniform_compaction_head_by_head(oracle_mod):
    rng = np.random.default_rng(220)
    B, H, T, d = 2, 4, 90, 16
    K = rng.integers(0, 1 << 16, size=(B, H, T, d), dtype=np.uint16)
    V = rng.integers(0, 1 << 16, size=(B, H, T, d), dtype=np.uint16)
    s = rng.random((B, H, T))
    z = rng.random((B, H, T)) ** 4 * rng.lognormal(0, 1, size=(1, H, 1))
    budget, floor, R, S, cap = 4 * 20, 6, 4, 2, 70
    idx, off = oracle_mod.select_budget(z, budget, floor, R, S)
    K_out, V_out, pos, acc, ln = oracle_mod.compact_ragged(K, V, s, idx, off, cap)
    for b in range(B):
        for h in range(H):
            n = off[b, h + 1] - off[b, h]
            rows = idx[b, off[b, h]:off[b, h + 1]]
            assert ln[b, h] == n
            Ku, Vu, pu, au, lu = oracle_mod.compact(K[b:b + 1, h:h + 1], V[b:b + 1, h:h + 1],
                                                    s[b:b + 1, h:h + 1], rows[None, None], cap)
            np.testing.assert_array_equal(K_out[b, h], Ku[0, 0])
            np.testing.assert_array_equal(V_out[b, h], Vu[0, 0])
            np.testing.assert_array_equal(pos[b, h], pu[0, 0])
            np.testing.assert_array_equal(acc[b, h], au[0, 0])
            np.testing.assert_array_equal(K_out[b, h, :n], K[b, h, rows])


def test_compact_ragged_leaves_spare_slots_and_rejects_overfull_heads(oracle_mod):
    rng = np.random.default_rng(221)
    K = rng.standard_normal((1, 2, 12, 8)).astype(np.float32)
    idx = np.array([[1, 5, 7, 0, 2, 3, 4, 11]], np.int32)
    off = np.array([[0, 3, 8]], np.int32)
    sentinel = tuple(np.full(shape, fill, dtype) for shape, fill, dtype in [
        ((1, 2, 6, 8), 7.0, np.float32), ((1, 2, 6, 8), 7.0, np.float32),
        ((1, 2, 6), -9, np.int32), ((1, 2, 6), 3.0, np.float32), ((1, 2), -1, np.int32)])
    K_out, V_out, pos, acc, ln = oracle_mod.compact_ragged(K, K, None, idx, off, 6, out=sentinel)
    np.testing.assert_array_equal(ln, [[3, 5]])
    np.testing.assert_array_equal(pos[0, 0], [1, 5, 7, -9, -9, -9])
    np.testing.assert_array_equal(pos[0, 1], [0, 2, 3, 4, 11, -9])
    assert np.all(K_out[0, 0, 3:] == 7.0) and np.all(acc == 3.0)   # s = None: acc untouched
    with pytest.raises(ValueError):
        oracle_mod.compact_ragged(K, K, None, idx, off, 4)           # head 1 keeps 5 > cap
    with pytest.raises(ValueError):
        oracle_mod.compact_ragged(K, K, None, idx, np.array([[0, 5, 3]], np.int32), 6)


@pytest.mark.parametrize("H,T,budget,floor,R,S,signed", [
    (8, 300, 8 * 40, 20, 8, 4, False),
    (8, 300, 8 * 40, 12, 8, 4, True),
    (5, 97, 5 * 30, 29, 0, 0, False),
    (3, 64, 3 * 64, 10, 2, 1, True),      # everything kept
    (4, 200, 4 * 30, 30, 5, 3, False),    # budget = H * floor: no competition
])
def test_threshold_decomposition_equals_the_oracle(oracle_mod, H, T, budget, floor, R, S, signed):
    """The identity the GPU kernel is built on, checked against the oracle's own
    selection: with the order (z desc, head asc, position asc) over a row's
    middle pairs, theta_h the (floor-S-R)-th best pair of head h and tau the
    (budget - H*floor)-th best pair among those below their head's theta_h,
    head h keeps exactly its middle pairs at or above min(theta_h, tau)."""
    rng = np.random.default_rng(H * T + budget)
    z = rng.standard_normal((H, T)) if signed else np.round(rng.random((H, T)) * 40) / 40
    n, nf = T - R - S, floor - R - S
    extra = budget - H * floor
    # rank of every middle pair in the row order (0 = best)
    hs, ps = np.meshgrid(np.arange(H), np.arange(S, T - R), indexing="ij")
    hs, ps = hs.ravel(), ps.ravel()
    order = np.lexsort((ps, hs, -z[hs, ps]))
    rank = np.empty(len(order), dtype=np.int64)
    rank[order] = np.arange(len(order))
    rank = rank.reshape(H, n)
    # -1: no floor / no competition ("selects nothing": no rank is <= -1)
    theta = np.array([np.sort(rank[h])[nf - 1] if nf > 0 else -1 for h in range(H)])
    below = np.concatenate([rank[h][rank[h] > theta[h]] for h in range(H)])
    tau = np.sort(below)[extra - 1] if extra > 0 else -1
    idx, off = oracle_mod.select_budget(z[None], budget, floor, R, S)
    for h in range(H):
        lam = max(theta[h], tau)  # ranks: smaller is better, so min over keys is max over ranks
        mid = [S + i for i in range(n) if rank[h, i] <= lam]
        want = list(range(S)) + mid + list(range(T - R, T))
        assert list(idx[0, off[0, h]:off[0, h + 1]]) == want, h
