"""Pins for the oracle's HubKV refinement (HubKV walkthrough, Method: 最终算法).

The steps are: local hubs by width-5 max-pooling, hubs keep their score and
non-hubs are multiplied by gamma, a head weight beta_h clipped to [0.8, 1.2],
and the ratio gate z_i = s_i + r^2 (beta_h q_i - s_i).  The gate is the
bounded perturbation z = (1 - lambda) s + lambda u with lambda = r^2 and
u = beta_h q (局部理论保证).  The selectivity behind beta_h is this
implementation's reading (normalised entropy); only its clip range, its
monotonicity in sharpness and the identical-heads case are pinned.
"""
import math
import os

import numpy as np
import pytest
from scipy.ndimage import maximum_filter1d
from scipy.stats import entropy

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand_scores(rng, B, H, T, clustered=True):
    s = rng.gamma(0.5, 1.0, size=(B, H, T))
    if clustered:
        s = maximum_filter1d(s, size=3, axis=-1) + 1e-3 * rng.random((B, H, T))
    return s


def _hubs_from_r1(oracle_mod, s, gamma=0.5):
    """With r = 1 the gate returns beta * q, so q = z / beta reveals the hub mask."""
    z, beta, _ = oracle_mod.hubkv_refine(s, r=1.0, gamma=gamma)
    q = z / beta[..., None]
    return np.isclose(q, s, rtol=1e-12, atol=0), q, beta


def test_worked_example_hubs():
    rows = {}
    for line in open(os.path.join(GOLDEN, "hubkv_worked_example.txt")):
        if line.strip() and not line.startswith("#"):
            name, *vals = line.split()
            rows[name] = np.array([float(v) for v in vals])
    import oracle
    s = rows["s"][None, None, :]
    hub, q, beta = _hubs_from_r1(oracle, s)
    pos = rows["s"] > 0  # a zero score is its own discount: the hub flag is invisible there
    np.testing.assert_array_equal(hub[0, 0][pos], rows["hub"].astype(bool)[pos])
    np.testing.assert_allclose(q[0, 0], rows["q"], rtol=1e-12)


def test_pool_window_matches_library_max_filter(oracle_mod):
    rng = np.random.default_rng(10)
    for T in (1, 2, 3, 4, 5, 6, 17, 200):
        s = _rand_scores(rng, 2, 3, T)
        s[0, 0, : min(T, 4)] = 1.0  # a tied plateau: every member is a hub
        hub, _, _ = _hubs_from_r1(oracle_mod, s)
        M = maximum_filter1d(s, size=5, axis=-1, mode="constant", cval=-np.inf)
        np.testing.assert_array_equal(hub, s == M)


def test_hub_dominance(oracle_mod):
    """Every non-hub has a strictly larger score within distance 2, and after the
    discount that neighbour's q is larger than the non-hub's q (s_h > gamma s_i)."""
    rng = np.random.default_rng(11)
    s = _rand_scores(rng, 2, 4, 300)
    hub, q, _ = _hubs_from_r1(oracle_mod, s)
    T = s.shape[-1]
    for b, h, i in zip(*np.nonzero(~hub)):
        win = slice(max(0, i - 2), min(T, i + 3))
        assert s[b, h, win].max() > s[b, h, i]
        if s[b, h, i] > 0:
            assert q[b, h, win].max() > q[b, h, i]


def test_beta_clip_range_and_identities(oracle_mod):
    rng = np.random.default_rng(12)
    s = _rand_scores(rng, 3, 8, 257)
    s[1, 2] = rng.random(257) * 1e-3 + 1.0     # flat head
    s[1, 3] = 0.0
    s[1, 3, 100] = 5.0                           # one-hot head
    for r in (0.0, 0.1, 0.5, 1.0):
        z, beta, _ = oracle_mod.hubkv_refine(s, r=r)
        assert (beta >= 0.8 - 1e-15).all() and (beta <= 1.2 + 1e-15).all()
        if r == 0.0:
            np.testing.assert_array_equal(z, s)
    _, q, beta = _hubs_from_r1(oracle_mod, s)
    for r in (0.1, 0.3, 0.9):
        z, beta_r, _ = oracle_mod.hubkv_refine(s, r=r)
        lam = r * r
        np.testing.assert_allclose(beta_r, beta, rtol=0, atol=0)
        np.testing.assert_allclose(z, (1 - lam) * s + lam * beta[..., None] * q, rtol=1e-13)


def test_gamma_one_identical_heads_is_identity(oracle_mod):
    rng = np.random.default_rng(13)
    one = _rand_scores(rng, 1, 1, 123)
    s = np.repeat(one, 5, axis=1)
    z, beta, _ = oracle_mod.hubkv_refine(s, r=0.7, gamma=1.0)
    np.testing.assert_allclose(beta, 1.0, rtol=0, atol=1e-15)
    np.testing.assert_allclose(z, s, rtol=1e-14)


def test_selectivity_entropy_and_extremes(oracle_mod):
    rng = np.random.default_rng(14)
    T = 64
    s = rng.random((1, 4, T)) + 0.01
    s[0, 0] = 1.0                 # uniform: sel = 0
    s[0, 1] = 0.0
    s[0, 1, 7] = 3.0              # one-hot: sel = 1
    _, beta, sel = oracle_mod.hubkv_refine(s, r=0.1)
    want = 1 - entropy(s[0], axis=-1) / math.log(T)
    np.testing.assert_allclose(sel[0], want, rtol=1e-12, atol=1e-12)
    assert abs(sel[0, 0]) < 1e-12 and abs(sel[0, 1] - 1.0) < 1e-12
    # two heads: uniform and one-hot -> mean 0.5 -> betas clipped to 0.8 and 1.2
    _, beta2, _ = oracle_mod.hubkv_refine(s[:, :2], r=0.1)
    np.testing.assert_allclose(beta2[0], [0.8, 1.2], rtol=1e-12)


def test_sharper_head_gets_larger_beta(oracle_mod):
    T = 200
    x = np.linspace(-3, 3, T)
    heads = [np.exp(-x ** 2 / (2 * w ** 2)) for w in (0.3, 0.6, 1.0, 2.0)]
    s = np.stack(heads)[None]
    _, beta, sel = oracle_mod.hubkv_refine(s, r=0.1, beta_lo=0.0, beta_hi=10.0)
    assert np.all(np.diff(sel[0]) < 0)
    assert np.all(np.diff(beta[0]) < 0)


def test_all_zero_unit_gives_beta_one(oracle_mod):
    s = np.zeros((2, 3, 16))
    s[1] = np.random.default_rng(15).random((3, 16))
    z, beta, sel = oracle_mod.hubkv_refine(s, r=0.5)
    np.testing.assert_array_equal(beta[0], 1.0)
    np.testing.assert_array_equal(z[0], 0.0)


def test_head_mean_is_per_batch_row(oracle_mod):
    """beta of a batch row does not depend on the other batch rows."""
    rng = np.random.default_rng(16)
    s = _rand_scores(rng, 3, 4, 90)
    _, beta_all, _ = oracle_mod.hubkv_refine(s, r=0.2)
    for b in range(3):
        _, beta_one, _ = oracle_mod.hubkv_refine(s[b:b + 1], r=0.2)
        np.testing.assert_array_equal(beta_one[0], beta_all[b])
