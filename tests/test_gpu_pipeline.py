"""End-to-end parity of the eviction path on the five workloads.

Small and reduced workloads run the whole chain on both sides (end to end);
the full-size workloads (32-layer GQA prefill, 128K context, batch-8 H2O
decode) run on the GPU in full and are checked on sampled units the oracle can
afford, stage by stage, plus invariants that hold at any size.
"""
import numpy as np
import pytest
import torch

from _parity import RTOL, assert_close, assert_kept_sets_equivalent, decode_lockstep
from kv_cache_compression_obs_gb300 import configs, gen

pytestmark = pytest.mark.gpu
DEV = "cuda"

REDUCED = [
    configs.TINY,
    configs.LLAMA2_LAYER,
    configs.H2O_DECODE.scaled(B=2, Hq=4, Hkv=4, T=1024, W=1024, k=204, R=102, n_decode=24),
    configs.GQA_PREFILL.scaled(B=1, L=2, T=4096, k=409, n_segments=40),
    configs.LONG_CONTEXT.scaled(L=1, T=16384, k=819, n_segments=150, n_decode=24),
]


def _np(t):
    return gen.to_numpy_bits(t)


def _decode_steps(kvc, oracle_mod, wl, out, steps, rows=None):
    """Run decode steps on the GPU for all units; lockstep-check the units of `rows`."""
    Kc, Vc, pos, acc, ln = out["K"], out["V"], out["pos"], out["acc"], out["len"]
    exact = 0
    for step in range(steps):
        q, kn, vn = gen.decode_inputs(wl, step, device=DEV)
        exact += decode_lockstep(kvc, oracle_mod, q, kn, vn, Kc, Vc, pos, acc, ln, wl.R,
                                 wl.T + step, wl.scale, rows=rows)
        # |S_i| = k and the recent window never loses a token
        assert torch.all(ln == wl.cap)
    return exact


@pytest.mark.parametrize("wl", REDUCED, ids=lambda w: f"{w.name}-T{w.T}")
def test_end_to_end_reduced(kvc, oracle_mod, wl):
    Q, K, V = gen.prefill_inputs(wl, device=DEV)
    out = kvc.compress_prefill(Q, K, V, wl.k, wl.R, wl.r, wl.gamma, wl.pool_width, wl.beta_lo,
                               wl.beta_hi, cap=wl.cap)
    torch.cuda.synchronize()
    Qh, Kh, Vh = _np(Q), _np(K), _np(V)
    s_ref = oracle_mod.score_obs(Qh, Kh, wl.scale)
    s_gpu = out["s"].cpu().numpy().astype(np.float64)
    assert_close(s_gpu, s_ref, what="s")
    if wl.r is not None:
        z_iso, beta_iso, _ = oracle_mod.hubkv_refine(s_gpu, wl.r, wl.gamma, wl.pool_width,
                                                     wl.beta_lo, wl.beta_hi)
        assert_close(out["z"].cpu().numpy(), z_iso, what="z (stage)")
        z_e2e, _, _ = oracle_mod.hubkv_refine(s_ref, wl.r, wl.gamma, wl.pool_width, wl.beta_lo,
                                              wl.beta_hi)
    else:
        z_e2e = s_ref
    z_gpu = out["z"].cpu().numpy().astype(np.float64)
    idx_gpu = out["idx"].cpu().numpy()
    np.testing.assert_array_equal(idx_gpu, oracle_mod.select_topk(z_gpu, wl.k, wl.R))
    assert_kept_sets_equivalent(idx_gpu, oracle_mod.select_topk(z_e2e, wl.k, wl.R), z_e2e, wl.k, wl.R)
    Kr, Vr, pr, ar, lr = oracle_mod.compact(Kh, Vh, s_gpu, idx_gpu, wl.cap)
    np.testing.assert_array_equal(_np(out["K"]), Kr)
    np.testing.assert_array_equal(_np(out["V"]), Vr)
    np.testing.assert_array_equal(out["pos"].cpu().numpy(), pr)
    np.testing.assert_array_equal(out["acc"].cpu().numpy(), ar)
    if wl.n_decode:
        steps = min(wl.n_decode, 64)
        assert _decode_steps(kvc, oracle_mod, wl, out, steps) >= steps - 2


def _sample_rows(wl, n=2):
    return sorted({0, wl.rows - 1} if n >= 2 else {0})


@pytest.mark.parametrize("wl", [configs.GQA_PREFILL, configs.LONG_CONTEXT], ids=lambda w: w.name)
def test_full_size_sampled(kvc, oracle_mod, wl):
    """All units on the GPU at the full size; the oracle checks two batch rows."""
    Q, K, V = gen.prefill_inputs(wl, device=DEV)
    out = kvc.compress_prefill(Q, K, V, wl.k, wl.R, wl.r, wl.gamma, wl.pool_width, wl.beta_lo,
                               wl.beta_hi, cap=wl.cap)
    torch.cuda.synchronize()
    # invariants at full size: every unit hands out G * W of attention mass
    tot = out["s"].double().sum(-1)
    torch.testing.assert_close(tot, torch.full_like(tot, wl.G * wl.W), rtol=1e-5, atol=0)
    rows = _sample_rows(wl)
    sl = lambda t: t[rows]
    s_gpu = out["s"][rows].cpu().numpy().astype(np.float64)
    s_ref = oracle_mod.score_obs(_np(sl(Q)), _np(sl(K)), wl.scale)
    assert_close(s_gpu, s_ref, what="s (sampled rows)")
    z_iso, _, _ = oracle_mod.hubkv_refine(s_gpu, wl.r, wl.gamma, wl.pool_width, wl.beta_lo, wl.beta_hi)
    assert_close(out["z"][rows].cpu().numpy(), z_iso, what="z (sampled rows)")
    z_gpu = out["z"][rows].cpu().numpy().astype(np.float64)
    idx_gpu = out["idx"][rows].cpu().numpy()
    np.testing.assert_array_equal(idx_gpu, oracle_mod.select_topk(z_gpu, wl.k, wl.R))
    Kr, Vr, pr, ar, _ = oracle_mod.compact(_np(sl(K)), _np(sl(V)), s_gpu, idx_gpu, wl.cap)
    np.testing.assert_array_equal(_np(out["K"][rows]), Kr)
    np.testing.assert_array_equal(_np(out["V"][rows]), Vr)
    np.testing.assert_array_equal(out["acc"][rows].cpu().numpy(), ar)
    if wl.n_decode:
        steps = 8
        assert _decode_steps(kvc, oracle_mod, wl, out, steps, rows) >= steps - 1


def test_h2o_decode_full_size_sampled(kvc, oracle_mod):
    """Batch-8 H2O decode at full size: prefill scores over all prompt queries
    (W = T = 8192), heavy + recent split, 256 steps with one eviction per head."""
    wl = configs.H2O_DECODE
    Q, K, V = gen.prefill_inputs(wl, device=DEV)
    out = kvc.compress_prefill(Q, K, V, wl.k, wl.R, None, cap=wl.cap)
    torch.cuda.synchronize()
    tot = out["s"].double().sum(-1)
    torch.testing.assert_close(tot, torch.full_like(tot, float(wl.W)), rtol=1e-5, atol=0)
    u = (3, 17)  # one unit checked against the oracle (the full causal 8192 x 8192 pattern)
    s_ref = oracle_mod.score_obs(_np(Q[u[0]:u[0] + 1, u[1]:u[1] + 1]),
                                 _np(K[u[0]:u[0] + 1, u[1]:u[1] + 1]), wl.scale)
    assert_close(out["s"][u[0], u[1]].cpu().numpy(), s_ref[0, 0], what="s (unit)")
    idx_gpu = out["idx"].cpu().numpy()
    np.testing.assert_array_equal(
        idx_gpu, oracle_mod.select_topk(out["s"].cpu().numpy().astype(np.float64), wl.k, wl.R))
    Kc, Vc, pos, acc, ln = out["K"], out["V"], out["pos"], out["acc"], out["len"]
    rows = [0, 7]
    exact = 0
    for step in range(wl.n_decode):
        q, kn, vn = gen.decode_inputs(wl, step, device=DEV)
        before = pos.clone()
        if step < 16:
            exact += decode_lockstep(kvc, oracle_mod, q, kn, vn, Kc, Vc, pos, acc, ln, wl.R,
                                     wl.T + step, wl.scale, rows=rows)
        else:
            _, ev = kvc.h2o_decode_step(q, kn, vn, Kc, Vc, pos, acc, ln, wl.R, wl.T + step)
            # exactly one eviction per head, never from the recent window
            assert torch.all(ev >= 0) and torch.all(ev <= wl.T + step - wl.R)
            changed = (pos != before).sum(-1)
            assert torch.all(changed == 1)
    assert exact >= 15


@pytest.mark.parametrize("wl", [configs.GQA_PREFILL.scaled(B=1, L=3, T=4096, k=409, n_segments=40),
                                configs.LONG_CONTEXT.scaled(L=2, T=16384, k=819, n_segments=150),
                                configs.TINY],
                         ids=lambda w: w.name)
def test_host_input_prefill_matches_the_device_path(kvc, wl):
    """compress_prefill_host (keys streamed per batch row on a copy stream, kept V
    rows gathered from pinned host memory) gives, bit for bit, what
    compress_prefill gives on the same rows with the inputs already on the GPU."""
    Q, K, V = gen.prefill_inputs(wl, device=DEV)
    hQ, hK, hV = (t.cpu().pin_memory() for t in (Q, K, V))
    got = kvc.compress_prefill_host(hQ, hK, hV, wl.k, wl.R, wl.r, wl.gamma, wl.pool_width,
                                    wl.beta_lo, wl.beta_hi, wl.scale)
    torch.cuda.synchronize()
    for b in range(wl.rows):  # one batch row per call, as the host path chunks it
        ref = kvc.compress_prefill(Q[b:b + 1], K[b:b + 1], V[b:b + 1], wl.k, wl.R, wl.r, wl.gamma,
                                   wl.pool_width, wl.beta_lo, wl.beta_hi, scale=wl.scale)
        torch.cuda.synchronize()
        for key in ("s", "idx", "K", "V", "pos", "acc", "len", "beta"):
            if ref[key] is not None:
                assert torch.equal(got[key][b:b + 1], ref[key]), (key, b)
        assert got["z"] is None if wl.r is not None else torch.equal(got["z"][b:b + 1], ref["z"])


def test_host_input_prefill_reuses_buffers_across_steps(kvc):
    """Two steps over the same buffers in row groups, with different inputs and
    other work queued on the stream between the calls: every result equals the
    device path's on that step's inputs (the copies never overwrite rows that an
    earlier call's chain still reads)."""
    wl = configs.LONG_CONTEXT.scaled(L=4, T=8192, k=409, n_segments=60)
    groups = [(0, 2), (2, 4)]
    steps = []
    for seed_shift in (0, 1):
        Q, K, V = gen.prefill_inputs(wl.scaled(seed=wl.seed + seed_shift), device=DEV)
        steps.append((Q, K, V, *(t.cpu().pin_memory() for t in (Q, K, V))))
    bufs = kvc.prefill_host_buffers(steps[0][3], steps[0][4], wl.k, wl.r)
    busy = torch.empty(64 << 20, device=DEV)
    for Q, K, V, hQ, hK, hV in steps:
        outs = []
        for r0, r1 in groups:
            got = kvc.compress_prefill_host(hQ, hK, hV, wl.k, wl.R, wl.r, wl.gamma, wl.pool_width,
                                            wl.beta_lo, wl.beta_hi, wl.scale, buffers=bufs,
                                            rows=(r0, r1))
            outs.append({key: got[key][r0:r1].clone() for key in ("idx", "K", "V", "len")})
            for _ in range(20):  # unrelated work queued between the calls
                busy.mul_(1.0)
        torch.cuda.synchronize()
        for (r0, r1), out in zip(groups, outs):
            ref = kvc.compress_prefill(Q[r0:r1], K[r0:r1], V[r0:r1], wl.k, wl.R, wl.r, wl.gamma,
                                       wl.pool_width, wl.beta_lo, wl.beta_hi, scale=wl.scale)
            torch.cuda.synchronize()
            for key in out:
                assert torch.equal(out[key], ref[key]), (key, r0)
