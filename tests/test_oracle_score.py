"""Pins for the oracle's observation-window scoring (closed forms and invariants).

Scoring follows the H2O page (观察二: accumulated attention o_s, the sum of the
attention probabilities a token receives) applied to SnapKV's observation
window (KV-cache blog §4.3), with softmax(q.k / sqrt(d_head)) from blog §1.1.
"""
import math

import numpy as np
import pytest

from kv_cache_compression_obs_gb300 import gen

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _bf16(x):
    """Round float32 to bf16 bit patterns (nearest-even) via the generator module."""
    import torch
    return gen.to_numpy_bits(torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.bfloat16))


def test_rows_sum_to_one_and_nonnegative(oracle_mod):
    rng = np.random.default_rng(0)
    B, Hq, Hkv, W, T, d = 2, 4, 2, 5, 37, 16
    for dt in ("f32", "bf16"):
        Q = rng.standard_normal((B, Hq, W, d)).astype(np.float32)
        K = rng.standard_normal((B, Hkv, T, d)).astype(np.float32)
        if dt == "bf16":
            Q, K = _bf16(Q), _bf16(K)
        s = oracle_mod.score_obs(Q, K, 1 / math.sqrt(d))
        G = Hq // Hkv
        assert s.shape == (B, Hkv, T)
        assert (s >= 0).all()
        np.testing.assert_allclose(s.sum(-1), G * W, rtol=1e-12)


def test_equal_keys_closed_form(oracle_mod):
    """All keys equal: each row spreads mass 1/(p+1) over keys 0..p (p = T-W+w)."""
    rng = np.random.default_rng(1)
    B, Hq, Hkv, W, T, d = 1, 6, 3, 7, 20, 8
    G = Hq // Hkv
    Q = rng.standard_normal((B, Hq, W, d)).astype(np.float32)
    K = np.broadcast_to(rng.standard_normal(d).astype(np.float32), (B, Hkv, T, d)).copy()
    s = oracle_mod.score_obs(Q, K, 0.3)
    want = np.zeros(T)
    for w in range(W):
        p = T - W + w
        want[: p + 1] += 1.0 / (p + 1)
    for h in range(Hkv):
        np.testing.assert_allclose(s[0, h], G * want, rtol=1e-12)
    s0 = oracle_mod.score_obs(np.zeros_like(Q), rng.standard_normal((B, Hkv, T, d)).astype(np.float32), 1.0)
    np.testing.assert_allclose(s0[0, 0], G * want, rtol=1e-12)


def test_two_keys_scale(oracle_mod):
    """One window row at position 1 sees keys 0 and 1: p_0 = 1 / (1 + exp(scale (b - a)))."""
    d = 4
    Q = np.array([[[[1.0, 0, 0, 0]]]], dtype=np.float32)
    K = np.array([[[[2.0, 1, 0, 0], [0.5, 0, 3, 0]]]], dtype=np.float32)
    for scale in (1.0, 0.5, 1 / math.sqrt(d)):
        s = oracle_mod.score_obs(Q, K, scale)
        p0 = 1.0 / (1.0 + math.exp(scale * (0.5 - 2.0)))
        np.testing.assert_allclose(s[0, 0], [p0, 1 - p0], rtol=1e-14)


def test_bf16_decoding(oracle_mod):
    """bf16 bit patterns 0x3F80 = 1.0 and 0x4000 = 2.0 give the same logits as float32."""
    Qf = np.array([[[[1.0, 2.0]]]], dtype=np.float32)
    Kf = np.array([[[[1.0, 1.0], [2.0, 1.0]]]], dtype=np.float32)
    Qb = np.array([[[[0x3F80, 0x4000]]]], dtype=np.uint16)
    Kb = np.array([[[[0x3F80, 0x3F80], [0x4000, 0x3F80]]]], dtype=np.uint16)
    np.testing.assert_array_equal(oracle_mod.score_obs(Qf, Kf, 1.0), oracle_mod.score_obs(Qb, Kb, 1.0))
    p0 = 1 / (1 + math.exp(1.0))
    np.testing.assert_allclose(oracle_mod.score_obs(Qb, Kb, 1.0)[0, 0], [p0, 1 - p0], rtol=1e-14)


def test_gqa_grouping_point_masses(oracle_mod):
    """Each query row points sharply at one key; the mass must land on the KV head
    that serves its query head (query head hq belongs to KV head hq // G)."""
    B, Hkv, G, W, d = 2, 3, 2, 4, 32
    Hq = Hkv * G
    T = d
    K = np.zeros((B, Hkv, T, d), dtype=np.float32)
    for j in range(T):
        K[:, :, j, j] = 40.0
    Q = np.zeros((B, Hq, W, d), dtype=np.float32)
    want = np.zeros((B, Hkv, T))
    rng = np.random.default_rng(3)
    for b in range(B):
        for hq in range(Hq):
            for w in range(W):
                p = T - W + w
                tgt = int(rng.integers(0, p + 1))
                Q[b, hq, w, tgt] = 40.0
                want[b, hq // G, tgt] += 1.0
    s = oracle_mod.score_obs(Q, K, 1 / math.sqrt(d))
    np.testing.assert_allclose(s, want, atol=1e-9)


def test_causal_mask(oracle_mod):
    """The last key is visible only to the last window row.  Give it a dominant
    logit: the last row puts (almost) all its mass there, the earlier rows none."""
    rng = np.random.default_rng(4)
    B, H, W, T, d = 1, 1, 3, 10, 8
    Q = np.zeros((B, H, W, d), dtype=np.float32)
    Q[..., 0] = 1.0
    Q[..., 1:] = 0.01 * rng.standard_normal((B, H, W, d - 1))
    K = (0.01 * rng.standard_normal((B, H, T, d))).astype(np.float32)
    K[0, 0, T - 1, 0] = 200.0
    s = oracle_mod.score_obs(Q, K, 1.0)
    assert abs(s[0, 0, T - 1] - 1.0) < 1e-12
    np.testing.assert_allclose(s[0, 0, :T - 1].sum(), 2.0, rtol=1e-12)
    # key T-2 is seen by rows at T-2 and T-1 only: without the last key it gets
    # its share from the row at T-2 (spread over keys 0..T-2) plus ~0 from the last row
    assert s[0, 0, T - 2] < 0.2


def test_matches_library_softmax_columns(oracle_mod):
    """Cross-check against column sums of scipy's float64 softmax with a causal mask."""
    from scipy.special import softmax
    rng = np.random.default_rng(5)
    B, Hq, Hkv, W, T, d = 1, 4, 2, 6, 25, 16
    Q = rng.standard_normal((B, Hq, W, d)).astype(np.float32)
    K = rng.standard_normal((B, Hkv, T, d)).astype(np.float32)
    scale = 1 / math.sqrt(d)
    s = oracle_mod.score_obs(Q, K, scale)
    G = Hq // Hkv
    for h in range(Hkv):
        want = np.zeros(T)
        for g in range(G):
            logits = scale * Q[0, h * G + g].astype(np.float64) @ K[0, h].astype(np.float64).T
            mask = np.arange(T)[None, :] > (T - W + np.arange(W))[:, None]
            logits[mask] = -np.inf
            want += softmax(logits, axis=1).sum(0)
        np.testing.assert_allclose(s[0, h], want, rtol=1e-12, atol=1e-15)
