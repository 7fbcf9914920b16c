"""Stage-isolated parity of each CUDA entry point against the float64 oracle.

Each GPU call gets exactly the bytes the oracle gets, so index work must match
bit for bit and floating-point results within the stated tolerance.
"""
import math

import numpy as np
import pytest
import torch

from _parity import RTOL, assert_close, decode_lockstep
from kv_cache_compression_obs_gb300 import gen
from kv_cache_compression_obs_gb300.configs import Workload

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _wl(B, Hq, Hkv, T, W, d, dtype, keys="segments", n_segments=0, n_sinks=0, R=0, seed=11):
    k = max(R + 1, T // 10)
    return Workload("case", B=B, L=1, Hq=Hq, Hkv=Hkv, d=d, T=T, W=W, dtype=dtype, r=0.1, k=k, R=R,
                    n_decode=0, seed=seed, keys=keys, n_segments=n_segments, n_sinks=n_sinks)


SCORE_CASES = [
    # B, Hq, Hkv, T, W, d, dtype, recipe
    (1, 4, 4, 512, 16, 64, "f32", dict(keys="sinks", n_sinks=4)),          # the tiny workload
    (1, 2, 1, 1, 1, 64, "bf16", {}),                                      # T = 1
    (1, 1, 1, 5, 5, 64, "f32", {}),                                       # W = T, tiny
    (2, 8, 2, 2085, 64, 128, "bf16", dict(n_segments=12, R=64)),          # GQA, ragged T
    (1, 4, 2, 777, 777, 128, "bf16", dict(keys="zipf")),                  # W = T: full causal
    (3, 2, 2, 130, 1, 64, "f32", {}),                                     # W = 1
    (1, 8, 1, 300, 40, 128, "f32", {}),                                   # MQA-like group of 8
    (1, 32, 32, 4096, 32, 128, "bf16", dict(n_segments=40, R=32)),        # Llama-2-7B layer
    # tensor-core path boundaries: G*W = 256 (two M-tiles, N = 256), 129 (second
    # M-tile with one row), 200 (N padded to 208), 128; d = 64; ragged T
    (2, 8, 2, 5000, 64, 128, "bf16", dict(n_segments=30, n_sinks=4, R=64)),
    (1, 3, 1, 1000, 43, 128, "bf16", dict(keys="zipf")),
    (1, 8, 2, 3333, 50, 64, "bf16", dict(n_segments=10, R=50)),
    (3, 4, 4, 700, 128, 128, "bf16", dict(keys="zipf")),
    (1, 1, 1, 130, 1, 128, "bf16", {}),
]


@pytest.mark.parametrize("case", SCORE_CASES, ids=lambda c: f"B{c[0]}Hq{c[1]}Hkv{c[2]}T{c[3]}W{c[4]}d{c[5]}{c[6]}")
def test_score_obs(kvc, oracle_mod, case):
    B, Hq, Hkv, T, W, d, dt, recipe = case
    wl = _wl(B, Hq, Hkv, T, W, d, dt, **recipe)
    Q, K, _ = gen.prefill_inputs(wl, device=DEV)
    s = kvc.kv_score_obs(Q, K)
    torch.cuda.synchronize()
    ref = oracle_mod.score_obs(gen.to_numpy_bits(Q), gen.to_numpy_bits(K), d ** -0.5)
    assert_close(s.cpu().numpy(), ref, what="s")
    # rows sum to one: every unit hands out G * W in total
    np.testing.assert_allclose(s.double().sum(-1).cpu().numpy(), (Hq // Hkv) * W, rtol=1e-5)
    # deterministic: a second run gives the same bits
    s2 = kvc.kv_score_obs(Q, K)
    assert torch.equal(s, s2)


def _scores_like(B, H, T, seed):
    g = torch.Generator(device=DEV)
    g.manual_seed(seed)
    s = torch.rand(B, H, T, generator=g, device=DEV) ** 4
    s = torch.nn.functional.max_pool1d(s.reshape(B * H, 1, T), 3, 1, 1).reshape(B, H, T)
    s = s + 1e-3 * torch.rand(B, H, T, generator=g, device=DEV)
    s[..., :4] += 5.0  # sinks
    return s.contiguous()


@pytest.mark.parametrize("shape", [(1, 1, 1), (1, 2, 2), (2, 3, 5), (1, 32, 4096), (2, 8, 32768),
                                   (1, 4, 10001)])
@pytest.mark.parametrize("r", [0.0, 0.1, 0.9])
def test_hubkv_refine(kvc, oracle_mod, shape, r):
    B, H, T = shape
    s = _scores_like(B, H, T, seed=T + H)
    s[0, 0, T // 2:T // 2 + min(T // 2, 7)] = 2.5  # a tied plateau
    if H > 1:
        s[-1, 1] = 0.0  # an all-zero head
    z, beta = kvc.hubkv_refine(s, r)
    torch.cuda.synchronize()
    s_np = s.cpu().numpy().astype(np.float64)
    z_ref, beta_ref, _ = oracle_mod.hubkv_refine(s_np, r)
    assert_close(beta.cpu().numpy(), beta_ref, rtol=1e-6, atol=0, what="beta")
    assert_close(z.cpu().numpy(), z_ref, rtol=RTOL, atol=1e-30, what="z")
    if r == 0.0:
        assert torch.equal(z, s)


def test_hubkv_gamma_one_identical_heads(kvc):
    one = _scores_like(1, 1, 999, seed=3)
    s = one.repeat(2, 6, 1).contiguous()
    z, beta = kvc.hubkv_refine(s, 0.7, gamma=1.0)
    assert torch.all(beta == 1.0)
    torch.testing.assert_close(z, s, rtol=1e-6, atol=0)


@pytest.mark.parametrize("T,k,R", [(10, 3, 0), (10, 10, 2), (4096, 409, 32), (8192, 1638, 819),
                                   (32768, 3276, 64), (131072, 6553, 64), (1000, 999, 998),
                                   (2049, 100, 1),
                                   (16385, 1000, 0),      # two CTAs per head, ragged slices
                                   (50000, 5000, 17),     # a cluster of 4
                                   (300000, 15000, 64),   # 8 CTAs with large slices
                                   (400000, 20000, 64)])  # beyond the resident limit: streaming kernel
@pytest.mark.parametrize("ties", [False, True, "signed"])
def test_select_topk_bit_exact(kvc, oracle_mod, T, k, R, ties):
    B, H = 2, 3
    g = torch.Generator(device=DEV)
    g.manual_seed(T + k)
    z = torch.rand(B, H, T, generator=g, device=DEV)
    if ties == "signed":                  # negative scores beside positive ones
        z = torch.randn(B, H, T, generator=g, device=DEV)
        z[1, 2] = -z[1, 2].abs()          # a head with no positive score
        z[0, 1, ::9] = -0.0
        z[0, 1, 4::9] = 0.0
    elif ties:
        z = torch.floor(z * 7) / 7        # heavy ties: the position rule decides
        z[0, 0, ::5] = -0.0               # signed zeros compare equal
        z[0, 0, 1::5] = 0.0
    idx = kvc.kv_select_topk(z, k, R)
    torch.cuda.synchronize()
    ref = oracle_mod.select_topk(z.cpu().numpy().astype(np.float64), k, R)
    np.testing.assert_array_equal(idx.cpu().numpy(), ref)


@pytest.mark.parametrize("dt,d", [("bf16", 128), ("bf16", 64), ("f32", 64), ("f32", 128)])
def test_compact_bit_exact(kvc, oracle_mod, dt, d):
    B, H, T, k, cap = 2, 3, 1500, 150, 170
    tdt = torch.bfloat16 if dt == "bf16" else torch.float32
    g = torch.Generator(device=DEV)
    g.manual_seed(d)
    K = torch.randn(B, H, T, d, generator=g, device=DEV).to(tdt)
    V = torch.randn(B, H, T, d, generator=g, device=DEV).to(tdt)
    s = torch.rand(B, H, T, generator=g, device=DEV)
    idx = torch.sort(torch.stack([torch.randperm(T, generator=g, device=DEV)[:k] for _ in range(B * H)]),
                     dim=-1).values.reshape(B, H, k).to(torch.int32).contiguous()
    sentinel = torch.full((B, H, cap, d), 7, dtype=tdt, device=DEV)
    Ko, Vo, pos, acc, ln = kvc.kv_compact(K, V, s, idx, cap, K_out=sentinel.clone(),
                                          V_out=sentinel.clone())
    torch.cuda.synchronize()
    Kr, Vr, pr, ar, lr = oracle_mod.compact(gen.to_numpy_bits(K), gen.to_numpy_bits(V),
                                            s.cpu().numpy().astype(np.float64), idx.cpu().numpy(), cap)
    np.testing.assert_array_equal(gen.to_numpy_bits(Ko)[:, :, :k], Kr[:, :, :k])
    np.testing.assert_array_equal(gen.to_numpy_bits(Vo)[:, :, :k], Vr[:, :, :k])
    np.testing.assert_array_equal(pos.cpu().numpy()[:, :, :k], pr[:, :, :k])
    np.testing.assert_array_equal(acc.cpu().numpy()[:, :, :k], ar[:, :, :k])
    np.testing.assert_array_equal(ln.cpu().numpy(), lr)
    assert torch.all(Ko[:, :, k:] == 7) and torch.all(Vo[:, :, k:] == 7)  # slots >= k untouched


def _decode_lockstep(kvc, oracle_mod, *args, **kw):
    return decode_lockstep(kvc, oracle_mod, *args, **kw)


@pytest.mark.parametrize("budget", [1, 4, 16])
def test_decode_alg1_matches_literal_loop(kvc, oracle_mod, budget):
    from oracle.alg1 import h2o_greedy_literal
    n, d = 48, 64
    g = torch.Generator(device=DEV)
    g.manual_seed(budget)
    Q = torch.randn(n, d, generator=g, device=DEV)
    Kt = torch.randn(n, d, generator=g, device=DEV)
    Vt = torch.randn(n, d, generator=g, device=DEV)
    cache, evicted, acc_lit = h2o_greedy_literal(Q.cpu().numpy(), Kt.cpu().numpy(), budget)
    Kc = torch.zeros(1, 1, budget, d, device=DEV)
    Vc = torch.zeros_like(Kc)
    pos = torch.zeros(1, 1, budget, dtype=torch.int32, device=DEV)
    acc = torch.zeros(1, 1, budget, device=DEV)
    ln = torch.zeros(1, 1, dtype=torch.int32, device=DEV)
    got = []
    for i in range(n):
        _, ev = kvc.h2o_decode_step(Q[i].reshape(1, 1, d), Kt[i].reshape(1, 1, d), Vt[i].reshape(1, 1, d),
                                    Kc, Vc, pos, acc, ln, 0, i, 1.0, kvc.KV_H2O_ALG1)
        got.append(int(ev.item()))
    assert got == evicted
    kept = pos[0, 0, :int(ln.item())].cpu().numpy()
    assert sorted(kept.tolist()) == sorted(cache)
    for slot, p in enumerate(kept):
        assert abs(acc[0, 0, slot].item() - acc_lit[int(p)]) <= 2e-5 * max(1.0, acc_lit[int(p)])


@pytest.mark.parametrize("G,dt,d,R", [(1, "bf16", 128, 8), (4, "bf16", 128, 8), (2, "f32", 64, 3),
                                      (8, "bf16", 64, 1), (4, "bf16", 128, 0)])
def test_decode_lockstep(kvc, oracle_mod, G, dt, d, R):
    B, Hkv, cap, T0, steps = 2, 3, 40, 200, 30
    Hq = G * Hkv
    tdt = torch.bfloat16 if dt == "bf16" else torch.float32
    g = torch.Generator(device=DEV)
    g.manual_seed(G * 100 + d + R)
    Kc = torch.randn(B, Hkv, cap, d, generator=g, device=DEV).to(tdt)
    Vc = torch.randn(B, Hkv, cap, d, generator=g, device=DEV).to(tdt)
    pos = torch.stack([torch.sort(torch.randperm(T0, generator=g, device=DEV)[:cap]).values
                       for _ in range(B * Hkv)]).reshape(B, Hkv, cap).to(torch.int32).contiguous()
    acc = (torch.rand(B, Hkv, cap, generator=g, device=DEV) * 2).contiguous()
    ln = torch.full((B, Hkv), cap - 5, dtype=torch.int32, device=DEV)  # 5 appends, then evictions
    scale = d ** -0.5
    exact = 0
    for step in range(steps):
        q = torch.randn(B, Hq, d, generator=g, device=DEV).to(tdt)
        kn = torch.randn(B, Hkv, d, generator=g, device=DEV).to(tdt)
        vn = torch.randn(B, Hkv, d, generator=g, device=DEV).to(tdt)
        exact += _decode_lockstep(kvc, oracle_mod, q, kn, vn, Kc, Vc, pos, acc, ln, R, T0 + step, scale)
    assert exact >= steps - 2  # near-tie victims are rare


def test_decode_new_token_victim_and_append(kvc, oracle_mod):
    B, Hkv, cap, d = 1, 2, 6, 64
    g = torch.Generator(device=DEV)
    g.manual_seed(5)
    Kc = torch.randn(B, Hkv, cap, d, generator=g, device=DEV)
    Vc = torch.randn_like(Kc)
    pos = torch.arange(cap, dtype=torch.int32, device=DEV).repeat(B, Hkv, 1).contiguous()
    acc = torch.full((B, Hkv, cap), 50.0, device=DEV)
    ln = torch.full((B, Hkv), cap, dtype=torch.int32, device=DEV)
    q = torch.randn(B, Hkv, d, generator=g, device=DEV)
    kn = torch.randn(B, Hkv, d, generator=g, device=DEV)
    K0 = Kc.clone()
    _, ev = kvc.h2o_decode_step(q, kn, kn, Kc, Vc, pos, acc, ln, 0, cap, 0.125)
    assert torch.all(ev == cap) and torch.equal(Kc, K0)
    ln.fill_(2)
    _, ev = kvc.h2o_decode_step(q, kn, kn, Kc, Vc, pos, acc, ln, 1, cap + 1, 0.125)
    assert torch.all(ev == -1) and torch.all(ln == 3) and torch.all(pos[:, :, 2] == cap + 1)
    assert torch.equal(Kc[:, :, 2], kn)


def test_decode_device_status_on_corrupt_length(kvc):
    B, Hkv, cap, d = 1, 1, 4, 64
    Kc = torch.zeros(B, Hkv, cap, d, device=DEV)
    pos = torch.zeros(B, Hkv, cap, dtype=torch.int32, device=DEV)
    acc = torch.zeros(B, Hkv, cap, device=DEV)
    ln = torch.full((B, Hkv), cap + 3, dtype=torch.int32, device=DEV)  # corrupt state
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    q = torch.zeros(B, Hkv, d, device=DEV)
    kvc.h2o_decode_step(q, q, q, Kc, Kc.clone(), pos, acc, ln, 0, 9, 0.1, dev_status=status)
    torch.cuda.synchronize()
    assert status.item() == kvc.KV_ERR_INVALID_ARG
    assert ln.item() == cap + 3  # nothing was written
