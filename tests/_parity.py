"""Comparison helpers shared by the GPU parity tests.

Tolerances (fp32 GPU arithmetic against the float64 oracle):
  * scores and attention outputs: |gpu - ref| <= RTOL |ref| + ATOL with RTOL = 1e-5
    (the stated parity bar for fp32 scores computed from bf16 inputs) and an
    absolute floor far below any value that matters (fp32 flushes probabilities
    below ~1e-38 that the float64 oracle still resolves);
  * index work (Top-K, compaction, eviction) is compared bit for bit when both
    sides start from the same bytes; end to end, kept sets may differ only by
    swaps between tokens whose scores lie within RTOL of the selection threshold.
"""
from __future__ import annotations

import numpy as np

RTOL = 1e-5
ATOL_SCORE = 1e-30


def assert_close(gpu, ref, rtol=RTOL, atol=ATOL_SCORE, what="value"):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert gpu.shape == ref.shape, (what, gpu.shape, ref.shape)
    err = np.abs(gpu - ref)
    bound = rtol * np.abs(ref) + atol
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err / np.maximum(bound, 1e-300)), err.shape)
        raise AssertionError(
            f"{what}: {int(bad.sum())}/{bad.size} elements outside rtol={rtol} atol={atol}; "
            f"worst at {i}: gpu={gpu[i]!r} ref={ref[i]!r} rel={err[i] / max(abs(ref[i]), 1e-300):.3e}")


def max_rel_err(gpu, ref, floor=1e-30):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    return float(np.max(np.abs(gpu - ref) / np.maximum(np.abs(ref), floor)))


def assert_kept_sets_equivalent(idx_gpu, idx_ref, z_ref, k, R, rtol=RTOL):
    """Per head: same recent window; heavy sets may differ only by near-threshold swaps."""
    idx_gpu = np.asarray(idx_gpu)
    idx_ref = np.asarray(idx_ref)
    z_ref = np.asarray(z_ref, dtype=np.float64)
    T = z_ref.shape[-1]
    heads = idx_ref.reshape(-1, k)
    got = idx_gpu.reshape(-1, k)
    zz = z_ref.reshape(-1, T)
    n_swaps = 0
    for hh in range(heads.shape[0]):
        g, r = got[hh], heads[hh]
        assert np.all(np.diff(g) > 0), f"head {hh}: positions not ascending"
        assert np.array_equal(g[k - R:], np.arange(T - R, T)) or R == 0, f"head {hh}: recent window"
        if np.array_equal(g, r):
            continue
        cand = zz[hh, :T - R]
        thr = np.sort(cand)[::-1][k - R - 1]
        extra = np.setdiff1d(g, r)
        missing = np.setdiff1d(r, g)
        assert len(extra) == len(missing)
        for j in np.concatenate([extra, missing]):
            assert abs(cand[j] - thr) <= rtol * abs(thr) + 1e-30, (
                f"head {hh}: position {j} (z={cand[j]!r}) differs but threshold is {thr!r}")
        n_swaps += len(extra)
    return n_swaps


def _acc_of(pos_after, acc_after, u, p):
    """Updated accumulator of the token at position p in one side's post-step state."""
    hit = np.nonzero(pos_after[u] == p)[0]
    assert hit.size == 1, (u, p)
    return float(acc_after[u][hit[0]])


def decode_lockstep(kvc, oracle_mod, q, kn, vn, Kc, Vc, pos, acc, ln, R, new_pos, scale, flags=0,
                    rows=None, sink=0):
    """One GPU decode step over all units and one oracle step over the batch rows
    `rows` (all when None), both from the same state.

    Returns True when both evicted the same tokens.  A different victim is
    accepted only when the two victims' updated accumulators agree within the
    fp32 tolerance (a near tie: both choices are valid greedy steps); the
    caller then continues from the GPU state."""
    from kv_cache_compression_obs_gb300 import gen
    import torch

    sel = (lambda t: t) if rows is None else (lambda t: t[rows])
    st = [gen.to_numpy_bits(sel(t)).copy() for t in (Kc, Vc, pos, acc, ln)]
    qs, kns, vns = (gen.to_numpy_bits(sel(t)) for t in (q, kn, vn))
    o, ev = kvc.h2o_decode_step(q, kn, vn, Kc, Vc, pos, acc, ln, R, new_pos, scale, flags, sink=sink)
    torch.cuda.synchronize()
    o_ref, ev_ref = oracle_mod.decode_step(qs, kns, vns, *st, R, new_pos, scale, flags, sink=sink)
    Kr, Vr, pr, ar, lr = st  # updated in place by the oracle
    assert_close(sel(o).cpu().numpy(), o_ref, rtol=RTOL, atol=1e-6, what="o")
    ev_g = sel(ev).cpu().numpy()
    pos_g, acc_g = sel(pos).cpu().numpy(), sel(acc).cpu().numpy()
    np.testing.assert_array_equal(sel(ln).cpu().numpy(), lr)
    same = ev_g == ev_ref
    for u in zip(*np.nonzero(~same)):
        assert ev_g[u] >= 0 and ev_ref[u] >= 0, (u, ev_g[u], ev_ref[u])
        a_g = _acc_of(pr, ar, u, ev_g[u])          # GPU's victim, as the oracle updated it
        a_r = _acc_of(pos_g, acc_g, u, ev_ref[u])  # oracle's victim, as the GPU updated it
        assert abs(a_g - a_r) <= 2 * RTOL * max(abs(a_g), abs(a_r)), (u, a_g, a_r)
    if same.all():
        np.testing.assert_array_equal(pos_g, pr)
        np.testing.assert_array_equal(gen.to_numpy_bits(sel(Kc)), Kr)
        np.testing.assert_array_equal(gen.to_numpy_bits(sel(Vc)), Vr)
        assert_close(acc_g, ar, rtol=RTOL, atol=1e-30, what="acc")
    return bool(same.all())
