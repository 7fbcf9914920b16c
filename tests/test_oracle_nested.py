"""Pins for the oracle's NestedKV key-only scorer (NestedKV technical summary,
1. Continuum Geheugentoestand: stable / episodic (b ~ N/32) / current (W = 64)
anchors and a_k(i) = -cos(k_i, mu_k); 2. Buitenste Leraar: softmax blending
with a fixed log-prior, surprise = std of the three scores, routing to the max).

Closed forms fix every step independently of the oracle's code:
  * keys along one direction: every anchor is that direction, a = -1, surprise
    0, weights = softmax(log-prior);
  * orthogonal keys: a_s = -1/sqrt(T), a_e = -1/sqrt(block size), a_c =
    -1/sqrt(window length at i), so the block size (ceil(T/32)), the causal
    window (i included) and the sign are all pinned; the discriminative power,
    the softmax weights, the surprise and the routing follow by hand.
"""
import math

import numpy as np
import pytest


def _softmax(x):
    e = np.exp(np.asarray(x) - np.max(x))
    return e / e.sum()


def test_one_direction_keys_give_minus_one_and_prior_weights(oracle_mod):
    rng = np.random.default_rng(300)
    T, d = 200, 16
    u = rng.standard_normal(d)
    K = (rng.uniform(0.1, 5.0, size=(1, 1, T, 1)) * u).astype(np.float32)
    lp = (0.0, math.log(2.0), math.log(3.0))
    r = oracle_mod.nested_score(K, n_disc=20, thresh=0.05, log_prior=lp)
    np.testing.assert_allclose(r["a"], -1.0, rtol=0, atol=1e-6)   # float32 keys: direction to ~1e-7
    np.testing.assert_allclose(r["sigma"], 0.0, atol=1e-6)
    np.testing.assert_allclose(r["w"][0, 0], [1 / 6, 2 / 6, 3 / 6], rtol=1e-5)
    np.testing.assert_allclose(r["score"], -1.0, atol=1e-6)


def _orthogonal_case(T, d, window, n_blocks, n_disc, lp, thresh, seed):
    rng = np.random.default_rng(seed)
    K = np.zeros((1, 1, T, d), dtype=np.float32)
    K[0, 0, np.arange(T), rng.permutation(d)[:T]] = rng.uniform(0.5, 3.0, size=T)
    blk = -(-T // n_blocks)
    a_s = np.full(T, -1 / math.sqrt(T))
    sizes = np.array([min(blk, T - (i // blk) * blk) for i in range(T)])
    a_e = -1 / np.sqrt(sizes)
    wl = np.minimum(np.arange(T) + 1, window)
    a_c = -1 / np.sqrt(wl)
    A = np.stack([a_s, a_e, a_c])
    D = [np.mean(np.sort(x)[-n_disc:]) - np.mean(np.sort(x)[:n_disc]) for x in A]
    w = _softmax(np.array(D) + np.array(lp))
    blend = w @ A
    sig = A.std(axis=0)
    if thresh is None:  # between the smallest and the largest surprise: both routes occur
        thresh = 0.5 * (sig.min() + sig.max())
    score = np.where(sig > thresh, A.max(axis=0), blend)
    return K, A, w, sig, score, thresh


@pytest.mark.parametrize("T,d,window,n_blocks,n_disc", [
    (64, 64, 16, 32, 8),     # blocks of 2
    (70, 72, 64, 32, 7),     # ceil(70/32) = 3: 23 blocks of 3 and one of 1
    (100, 128, 64, 32, 1),   # n_disc = 1: max - min
    (33, 40, 5, 4, 33),      # n_disc = T: the two means coincide, D = 0
])
def test_orthogonal_keys_closed_form(oracle_mod, T, d, window, n_blocks, n_disc):
    lp = (0.3, -0.2, 0.1)
    K, A, w, sig, score, thresh = _orthogonal_case(T, d, window, n_blocks, n_disc, lp, None, seed=T)
    r = oracle_mod.nested_score(K, n_disc=n_disc, thresh=thresh, log_prior=lp, window=window,
                                n_blocks=n_blocks)
    np.testing.assert_allclose(r["a"][0, 0], A, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(r["w"][0, 0], w, rtol=1e-12)
    np.testing.assert_allclose(r["sigma"][0, 0], sig, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(r["score"][0, 0], score, rtol=1e-12, atol=1e-14)
    # both routes occur in these cases, so the routing itself is exercised
    assert (sig > thresh).any() and (sig <= thresh).any()


def test_zero_key_scores_zero_and_does_not_move_the_anchors(oracle_mod):
    rng = np.random.default_rng(301)
    K = rng.standard_normal((1, 1, 50, 8)).astype(np.float32)
    K0 = K.copy()
    K0[0, 0, 17] = 0.0
    r = oracle_mod.nested_score(K0, n_disc=5, thresh=0.2)
    np.testing.assert_array_equal(r["a"][0, 0, :, 17], 0.0)
    # the stable anchor is the mean of unit vectors: a zero key only rescales it
    ref = oracle_mod.nested_score(np.delete(K0, 17, axis=2), n_disc=5, thresh=0.2)
    np.testing.assert_allclose(np.delete(r["a"][0, 0, 0], 17), ref["a"][0, 0, 0], rtol=1e-12)


def test_positive_rescaling_of_keys_changes_nothing(oracle_mod):
    rng = np.random.default_rng(302)
    K = rng.standard_normal((2, 3, 400, 32))
    c = rng.uniform(0.01, 100.0, size=(2, 3, 400, 1))
    r1 = oracle_mod.nested_score(K.astype(np.float32), n_disc=40, thresh=0.1)
    r2 = oracle_mod.nested_score((K * c).astype(np.float32), n_disc=40, thresh=0.1)
    for key in ("a", "w", "sigma"):
        np.testing.assert_allclose(r1[key], r2[key], rtol=1e-5, atol=1e-6)


def test_bf16_bits_read_as_their_values(oracle_mod):
    rng = np.random.default_rng(303)
    bits = rng.integers(0, 1 << 16, size=(1, 2, 90, 16), dtype=np.uint16)
    bits &= np.uint16(0xBFFF)   # keep exponents small: finite values only
    vals = oracle_mod.bf16_bits_to_f64(bits).astype(np.float32)
    r1 = oracle_mod.nested_score(bits, n_disc=9, thresh=0.1)
    r2 = oracle_mod.nested_score(vals, n_disc=9, thresh=0.1)
    for key in ("a", "w", "sigma", "score"):
        np.testing.assert_array_equal(r1[key], r2[key])


def test_rejects_bad_arguments(oracle_mod):
    K = np.ones((1, 1, 10, 4), np.float32)
    for kw in (dict(n_disc=11), dict(n_disc=0), dict(n_disc=2, window=0), dict(n_disc=2, n_blocks=0)):
        with pytest.raises(ValueError):
            oracle_mod.nested_score(K, thresh=0.1, **kw)
    K[0, 0, 3, 1] = np.inf
    with pytest.raises(ValueError):
        oracle_mod.nested_score(K, n_disc=2, thresh=0.1)
