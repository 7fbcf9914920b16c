"""Pins for the oracle's H2O decode step.

Sources: H2O page, 问题形式化 (|S_i| = k, at most one eviction per step,
attention renormalised over the kept keys), 贪心驱逐算法 (Algorithm 1: evicting
the lowest accumulated score maximises the kept set's score), 双缓冲 (a
protected recent window), FlexGen 改造 (preallocated slots overwritten in place).
"""
import numpy as np
import pytest
from scipy.special import softmax

from oracle.alg1 import h2o_greedy_literal


def _empty_state(B, Hkv, cap, d, dtype=np.float32):
    return (np.zeros((B, Hkv, cap, d), dtype), np.zeros((B, Hkv, cap, d), dtype),
            np.zeros((B, Hkv, cap), np.int32), np.zeros((B, Hkv, cap), np.float32),
            np.zeros((B, Hkv), np.int32))


def _full_state(rng, B, Hkv, cap, d, T0):
    K, V, pos, acc, ln = _empty_state(B, Hkv, cap, d)
    for b in range(B):
        for h in range(Hkv):
            pos[b, h] = np.sort(rng.choice(T0, cap, replace=False))
    K[:] = rng.standard_normal(K.shape)
    V[:] = rng.standard_normal(V.shape)
    acc[:] = rng.random(acc.shape).astype(np.float32) * 3
    ln[:] = cap
    return K, V, pos, acc, ln


@pytest.mark.parametrize("budget", [1, 3, 8])
def test_alg1_matches_literal_loop(oracle_mod, budget):
    rng = np.random.default_rng(budget)
    n, d = 30, 16
    Q = rng.standard_normal((n, d)).astype(np.float32)
    Kt = rng.standard_normal((n, d)).astype(np.float32)
    Vt = rng.standard_normal((n, d)).astype(np.float32)
    cache, evicted, acc_lit = h2o_greedy_literal(Q, Kt, budget)
    K, V, pos, acc, ln = _empty_state(1, 1, budget, d)
    got_ev = []
    for i in range(n):
        _, ev = oracle_mod.decode_step(Q[i][None, None], Kt[i][None, None], Vt[i][None, None],
                                       K, V, pos, acc, ln, recent=0, new_pos=i, scale=1.0,
                                       flags=oracle_mod.FLAG_ALG1)
        got_ev.append(int(ev[0, 0]))
    assert got_ev == evicted
    assert sorted(pos[0, 0, :ln[0, 0]]) == sorted(cache)
    for slot in range(ln[0, 0]):
        np.testing.assert_allclose(acc[0, 0, slot], acc_lit[int(pos[0, 0, slot])], rtol=2e-6, atol=1e-7)
        np.testing.assert_array_equal(K[0, 0, slot], Kt[pos[0, 0, slot]])


def _expected_step(q, kn, vn, K, V, pos, acc, ln, R, new_pos, scale, G):
    """Float64 restatement for one unit with library softmax: returns (o, P_slots, P_new)."""
    n = int(ln)
    Kall = np.concatenate([K[:n], kn[None]]).astype(np.float64)
    Vall = np.concatenate([V[:n], vn[None]]).astype(np.float64)
    P = np.zeros(n + 1)
    o = np.zeros((G, K.shape[-1]))
    for g in range(G):
        p = softmax(scale * Kall @ q[g].astype(np.float64))
        P += p
        o[g] = p @ Vall
    return o, P[:n], P[n]


def test_default_mode_invariants_and_greedy_optimality(oracle_mod):
    rng = np.random.default_rng(30)
    B, Hkv, G, cap, d, R, T0 = 2, 2, 2, 10, 8, 3, 40
    Hq = Hkv * G
    K, V, pos, acc, ln = _full_state(rng, B, Hkv, cap, d, T0)
    scale = d ** -0.5
    for step in range(40):
        new_pos = T0 + step
        q = rng.standard_normal((B, Hq, d)).astype(np.float32)
        kn = rng.standard_normal((B, Hkv, d)).astype(np.float32)
        vn = rng.standard_normal((B, Hkv, d)).astype(np.float32)
        before = (K.copy(), V.copy(), pos.copy(), acc.copy(), ln.copy())
        o, ev = oracle_mod.decode_step(q, kn, vn, K, V, pos, acc, ln, R, new_pos, scale)
        for b in range(B):
            for h in range(Hkv):
                Kb, Vb, pb, ab, lb = (x[b, h] for x in before)
                o_want, P, P_new = _expected_step(q[b, h * G:(h + 1) * G], kn[b, h], vn[b, h],
                                                  Kb, Vb, pb, ab, lb, R, new_pos, scale, G)
                np.testing.assert_allclose(o[b, h * G:(h + 1) * G], o_want, rtol=1e-12, atol=1e-12)
                assert ln[b, h] == cap                                   # |S_i| = k
                old, new = set(pb.tolist()), set(pos[b, h].tolist())
                assert len(new - old) == 1 and new - old == {new_pos}    # <= 1 eviction, new kept
                gone = (old - new).pop()
                assert ev[b, h] == gone and gone <= new_pos - R
                acc_upd = (ab.astype(np.float64) + P).astype(np.float32)
                # greedy: the evicted candidate has the lowest (acc, pos) among the candidates
                cand = [j for j in range(cap) if pb[j] <= new_pos - R]
                best = min(cand, key=lambda j: (acc_upd[j], pb[j]))
                assert pb[best] == gone
                kept_sum = acc_upd.astype(np.float64).sum() - acc_upd[best]
                for j in cand:
                    assert kept_sum >= acc_upd.astype(np.float64).sum() - acc_upd[j] - 1e-12
                # mass conservation: every query head hands out probability 1
                np.testing.assert_allclose(P.sum() + P_new, G, rtol=1e-12)
                slot = list(pos[b, h]).index(new_pos)
                np.testing.assert_allclose(acc[b, h, slot], np.float32(P_new), rtol=0, atol=0)
                np.testing.assert_array_equal(K[b, h, slot], kn[b, h])
                np.testing.assert_array_equal(V[b, h, slot], vn[b, h])


def test_append_phase(oracle_mod):
    rng = np.random.default_rng(31)
    B, Hkv, cap, d = 1, 2, 6, 4
    K, V, pos, acc, ln = _empty_state(B, Hkv, cap, d)
    for i in range(cap):
        q = rng.standard_normal((B, Hkv, d)).astype(np.float32)
        kn = rng.standard_normal((B, Hkv, d)).astype(np.float32)
        _, ev = oracle_mod.decode_step(q, kn, kn, K, V, pos, acc, ln, 2, i, 0.5)
        assert (ev == -1).all() and (ln == i + 1).all()
        np.testing.assert_array_equal(pos[0, :, : i + 1], np.tile(np.arange(i + 1), (Hkv, 1)))
    # the first token attended only to itself: its accumulator starts at 1
    # (one query head per KV head) and grows by its later probabilities
    assert (acc[0, :, 0] >= 1.0).all()


def test_uniform_attention_closed_form(oracle_mod):
    """All keys (cached and new) equal: attention is uniform over the n+1 tokens,
    o is the mean value row and each accumulator gains G / (n+1)."""
    rng = np.random.default_rng(32)
    B, Hkv, G, cap, d = 1, 1, 3, 5, 8
    K, V, pos, acc, ln = _full_state(rng, B, Hkv, cap, d, 20)
    key = rng.standard_normal(d).astype(np.float32)
    K[:] = key
    acc0 = acc.copy()
    q = rng.standard_normal((B, G, d)).astype(np.float32)
    vn = rng.standard_normal((B, Hkv, d)).astype(np.float32)
    V_old = V.copy()
    o, ev = oracle_mod.decode_step(q, key[None, None].copy(), vn, K, V, pos, acc, ln, 1, 20, 1.0)
    mean_v = (V_old[0, 0].astype(np.float64).sum(0) + vn[0, 0]) / (cap + 1)
    for g in range(G):
        np.testing.assert_allclose(o[0, g], mean_v, rtol=1e-12)
    kept = pos[0, 0] != 20
    want = (acc0[0, 0].astype(np.float64) + G / (cap + 1)).astype(np.float32)
    np.testing.assert_array_equal(acc[0, 0][kept], want[kept])
    assert ev[0, 0] >= 0 and kept.sum() == cap - 1


def test_new_token_can_be_victim_without_window(oracle_mod):
    rng = np.random.default_rng(33)
    B, Hkv, cap, d = 1, 1, 4, 8
    K, V, pos, acc, ln = _full_state(rng, B, Hkv, cap, d, 10)
    acc[:] = 50.0
    K0, pos0 = K.copy(), pos.copy()
    q = rng.standard_normal((B, 1, d)).astype(np.float32)
    kn = rng.standard_normal((B, 1, d)).astype(np.float32)
    _, ev = oracle_mod.decode_step(q, kn, kn, K, V, pos, acc, ln, 0, 10, 0.3)
    assert ev[0, 0] == 10
    np.testing.assert_array_equal(pos, pos0)
    np.testing.assert_array_equal(K, K0)


def test_ties_evict_oldest(oracle_mod):
    rng = np.random.default_rng(34)
    B, Hkv, cap, d, R = 1, 1, 6, 4, 2
    K, V, pos, acc, ln = _full_state(rng, B, Hkv, cap, d, 30)
    K[:] = 1.0
    acc[:] = 2.0
    pos[0, 0] = np.array([17, 3, 25, 9, 28, 29])
    q = np.ones((B, 1, d), np.float32)
    _, ev = oracle_mod.decode_step(q, np.ones((B, 1, d), np.float32), np.ones((B, 1, d), np.float32),
                                   K, V, pos, acc, ln, R, 30, 0.5)
    assert ev[0, 0] == 3 and pos[0, 0, 1] == 30


def test_protected_window_never_evicted(oracle_mod):
    rng = np.random.default_rng(35)
    B, Hkv, cap, d, R = 1, 1, 5, 4, 4
    K, V, pos, acc, ln = _full_state(rng, B, Hkv, cap, d, 8)
    pos[0, 0] = np.array([2, 5, 6, 7, 4])
    acc[0, 0] = np.array([9.0, 0.0, 0.0, 0.0, 1.0], np.float32)   # recent ones have acc 0
    _, ev = oracle_mod.decode_step(rng.standard_normal((B, 1, d)).astype(np.float32),
                                   rng.standard_normal((B, 1, d)).astype(np.float32),
                                   rng.standard_normal((B, 1, d)).astype(np.float32),
                                   K, V, pos, acc, ln, R, 8, 0.5)
    # candidates: positions <= 8 - 4 = 4 -> {2, 4}; 4 has the lower accumulator
    assert ev[0, 0] == 4


def test_rejects_bad_arguments(oracle_mod):
    K, V, pos, acc, ln = _empty_state(1, 1, 4, 4)
    z = np.zeros((1, 1, 4), np.float32)
    with pytest.raises(ValueError):   # ALG1 requires recent = 0
        oracle_mod.decode_step(z, z, z, K, V, pos, acc, ln, 1, 0, 1.0, flags=oracle_mod.FLAG_ALG1)
    with pytest.raises(ValueError):   # recent must be < cap
        oracle_mod.decode_step(z, z, z, K, V, pos, acc, ln, 4, 0, 1.0)
