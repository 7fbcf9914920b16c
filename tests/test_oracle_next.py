"""Pins for the oracle's variants beyond the five core steps.

* Attention sinks (KV-cache survey blog §4.1-4.2: the first few tokens are kept
  as sinks; StreamingLLM keeps sinks plus the recent window): Top-K keeps the
  first S positions as well as the recent window, and a decode step never evicts
  a position below S.
* HubKV's weaker variants (HubKV walkthrough, 尝试路线：效果一般的可能原因):
  average-pool smoothing ("CommunitySmooth") in place of the local-hub step, and
  a fixed head weight (beta = 1) in place of head calibration.
"""
import itertools

import numpy as np
import pytest

from test_oracle_decode import _expected_step, _full_state


# ---------------------------------------------------------------- Top-K sinks
def _brute_best_sink(z, k, R, S):
    """Exhaustive: [0, S) and [T-R, T) kept; among all (k-R-S)-subsets of
    [S, T-R), the one with the largest sum, ties broken by the lexicographically
    first sorted (z desc, pos asc) sequence."""
    T = len(z)
    best = None
    for sub in itertools.combinations(range(S, T - R), k - R - S):
        key = (-sum(z[i] for i in sub), sorted((-z[i], i) for i in sub))
        if best is None or key < best[0]:
            best = (key, sub)
    return sorted(list(range(S)) + list(best[1]) + list(range(T - R, T)))


@pytest.mark.parametrize("seed", range(4))
def test_select_sinks_exhaustive_small(oracle_mod, seed):
    rng = np.random.default_rng(100 + seed)
    for T in range(2, 10):
        for k in range(2, T + 1):
            for R in range(0, k):
                for S in range(0, k - R):
                    z = rng.integers(0, 4, size=T).astype(np.float64)  # many ties
                    idx = oracle_mod.select_topk(z[None, None], k, R, sink=S)[0, 0]
                    assert list(idx) == _brute_best_sink(list(z), k, R, S), (T, k, R, S, z)


def test_select_sinks_zero_is_plain_select_and_sinks_always_kept(oracle_mod):
    rng = np.random.default_rng(110)
    z = rng.standard_normal((2, 3, 300))
    z[..., :4] = -10.0  # sinks the scores would drop
    np.testing.assert_array_equal(oracle_mod.select_topk(z, 40, 8, sink=0),
                                  oracle_mod.select_topk(z, 40, 8))
    idx = oracle_mod.select_topk(z, 40, 8, sink=4)
    for row in idx.reshape(-1, 40):
        assert set(range(4)) <= set(row) and set(range(292, 300)) <= set(row)
        assert np.all(np.diff(row) > 0)


def test_select_sinks_rejects_overfull_protection(oracle_mod):
    z = np.zeros((1, 1, 20))
    with pytest.raises(ValueError):
        oracle_mod.select_topk(z, 8, 4, sink=4)   # S + R must stay below k
    with pytest.raises(ValueError):
        oracle_mod.select_topk(z, 8, 2, sink=-1)


# ---------------------------------------------------------------- decode sinks
def test_decode_sinks_never_evicted_and_greedy_among_the_rest(oracle_mod):
    rng = np.random.default_rng(120)
    B, Hkv, G, cap, d, R, S, T0 = 2, 2, 2, 10, 8, 2, 3, 40
    Hq = Hkv * G
    K, V, pos, acc, ln = _full_state(rng, B, Hkv, cap, d, T0)
    pos[:, :, :S] = np.arange(S)        # the sinks are cached, with the lowest scores
    acc[:, :, :S] = 0.0
    scale = d ** -0.5
    for step in range(30):
        new_pos = T0 + step
        q = rng.standard_normal((B, Hq, d)).astype(np.float32)
        kn = rng.standard_normal((B, Hkv, d)).astype(np.float32)
        vn = rng.standard_normal((B, Hkv, d)).astype(np.float32)
        before = (K.copy(), V.copy(), pos.copy(), acc.copy(), ln.copy())
        _, ev = oracle_mod.decode_step(q, kn, vn, K, V, pos, acc, ln, R, new_pos, scale, sink=S)
        for b in range(B):
            for h in range(Hkv):
                Kb, Vb, pb, ab, lb = (x[b, h] for x in before)
                _, P, _ = _expected_step(q[b, h * G:(h + 1) * G], kn[b, h], vn[b, h],
                                         Kb, Vb, pb, ab, lb, R, new_pos, scale, G)
                acc_upd = (ab.astype(np.float64) + P).astype(np.float32)
                cand = [j for j in range(cap) if S <= pb[j] <= new_pos - R]
                best = min(cand, key=lambda j: (acc_upd[j], pb[j]))
                assert ev[b, h] == pb[best]
                assert set(range(S)) <= set(pos[b, h].tolist())      # the sinks stay
                old, new = set(pb.tolist()), set(pos[b, h].tolist())
                assert old - new == {pb[best]} and new - old == {new_pos}


def test_decode_sinks_zero_is_plain_decode(oracle_mod):
    rng = np.random.default_rng(121)
    B, Hkv, G, cap, d, R = 1, 2, 4, 9, 8, 3
    state_a = list(_full_state(rng, B, Hkv, cap, d, 30))
    state_b = [x.copy() for x in state_a]
    for step in range(10):
        q = rng.standard_normal((B, Hkv * G, d)).astype(np.float32)
        kn = rng.standard_normal((B, Hkv, d)).astype(np.float32)
        vn = rng.standard_normal((B, Hkv, d)).astype(np.float32)
        oa, ea = oracle_mod.decode_step(q, kn, vn, *state_a, R, 30 + step, 0.3, sink=0)
        ob, eb = oracle_mod.decode_step(q, kn, vn, *state_b, R, 30 + step, 0.3)
        np.testing.assert_array_equal(oa, ob)
        np.testing.assert_array_equal(ea, eb)
    for x, y in zip(state_a, state_b):
        np.testing.assert_array_equal(x, y)


def test_decode_sink_with_lowest_score_is_skipped(oracle_mod):
    rng = np.random.default_rng(122)
    K, V, pos, acc, ln = _full_state(rng, 1, 1, 5, 4, 8)
    pos[0, 0] = np.array([0, 1, 3, 5, 6])
    acc[0, 0] = np.array([0.0, 0.5, 2.0, 1.0, 7.0], np.float32)
    args = [rng.standard_normal((1, 1, 4)).astype(np.float32) for _ in range(3)]
    _, ev = oracle_mod.decode_step(*args, K, V, pos, acc, ln, 2, 9, 0.5, sink=1)
    # candidates: positions 1..7 (pos <= 9 - 2, pos >= 1): {1, 3, 5, 6}; 1 scores lowest
    assert ev[0, 0] == 1 and 0 in pos[0, 0]


# ---------------------------------------------------------------- HubKV variants
def _window_mean(s, half):
    """Mean of s over [i - half, i + half] cut at the ends, by prefix sums."""
    T = len(s)
    c = np.concatenate([[0.0], np.cumsum(s)])
    lo = np.maximum(np.arange(T) - half, 0)
    hi = np.minimum(np.arange(T) + half, T - 1)
    return (c[hi + 1] - c[lo]) / (hi - lo + 1)


def test_avgpool_variant_is_window_mean_in_the_gate(oracle_mod):
    rng = np.random.default_rng(130)
    s = rng.random((2, 3, 57)) ** 3
    r = 0.7
    z, beta, _ = oracle_mod.hubkv_refine(s, r, flags=oracle_mod.HUB_AVGPOOL)
    _, beta_plain, _ = oracle_mod.hubkv_refine(s, r)
    np.testing.assert_array_equal(beta, beta_plain)   # head calibration untouched
    for b in range(2):
        for h in range(3):
            q = _window_mean(s[b, h], 2)
            want = s[b, h] + r * r * (beta[b, h] * q - s[b, h])
            np.testing.assert_allclose(z[b, h], want, rtol=1e-13, atol=1e-15)


def test_avgpool_constant_scores_are_fixed_points_of_smoothing(oracle_mod):
    s = np.full((1, 2, 11), 0.25)
    z, beta, _ = oracle_mod.hubkv_refine(s, 0.9, flags=oracle_mod.HUB_AVGPOOL)
    np.testing.assert_allclose(z, s[0][None] + 0.81 * (beta[..., None] * s - s), rtol=1e-14)


def test_fixed_head_variant_equals_unit_clip_range(oracle_mod):
    rng = np.random.default_rng(131)
    s = rng.random((3, 4, 40)) ** 2
    z, beta, _ = oracle_mod.hubkv_refine(s, 0.8, flags=oracle_mod.HUB_FIXED_HEAD)
    z1, beta1, _ = oracle_mod.hubkv_refine(s, 0.8, beta_lo=1.0, beta_hi=1.0)
    np.testing.assert_array_equal(beta, np.ones_like(beta))
    np.testing.assert_array_equal(beta1, np.ones_like(beta1))
    np.testing.assert_allclose(z, z1, rtol=0, atol=0)


def test_both_variants_compose(oracle_mod):
    rng = np.random.default_rng(132)
    s = rng.random((1, 2, 30))
    z, beta, _ = oracle_mod.hubkv_refine(s, 0.5, flags=oracle_mod.HUB_AVGPOOL | oracle_mod.HUB_FIXED_HEAD)
    np.testing.assert_array_equal(beta, np.ones_like(beta))
    for h in range(2):
        np.testing.assert_allclose(z[0, h], s[0, h] + 0.25 * (_window_mean(s[0, h], 2) - s[0, h]),
                                   rtol=1e-13, atol=1e-15)


def test_variant_flags_rejected_when_unknown(oracle_mod):
    with pytest.raises(ValueError):
        oracle_mod.hubkv_refine(np.ones((1, 1, 4)), 0.5, flags=8)
