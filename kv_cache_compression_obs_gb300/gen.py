"""Seeded synthetic inputs for the eviction path (shared by the CUDA path's tests,
the oracle's tests and the benchmark).

This module holds none of the method's arithmetic: it only draws random
queries, keys and values and plants the structure the pages' workloads have
(attention sinks, clusters of similar keys, power-law key norms).  Every unit
(batch row, KV head) draws from its own seeded torch generator, so any subset of
units can be regenerated bit-identically on the same device type.  bf16 values
are rounded from float32 with round-to-nearest-even (torch's conversion).

Recipes (dimensions per unit: G query heads x W window rows, T keys):
  * queries, keys, values ~ N(0, 1);
  * "sinks": the first n_sinks keys become 4 x their norm along the mean
    observation query direction q_hat;
  * "segments": n_segments non-overlapping runs of 20..60 tokens placed
    uniformly in [4, T - R); run s has direction
    u_s = normalise(0.5 q_hat + sqrt(0.75) n_s) with n_s a random unit vector, and
    each key in it becomes |k_j| normalise(0.8 u_s + 0.6 e_j) with e_j a random
    unit vector orthogonal to u_s (cosine 0.8 to u_s);
  * "zipf": key j is scaled by 1 + 3 r_j^(-1.1), r_j a random permutation of
    1..T (a Zipf s = 1.1 norm profile whose largest key is 4x).
Decode steps draw fresh N(0, 1) q, k, v per step; under "zipf" the new key is
scaled by 1 + 3 r^(-1.1) with r uniform in 1..T.
"""
from __future__ import annotations

import math

import numpy as np
import torch

from .configs import Workload

SEGMENT_ALIGN = 0.5           # weight of the mean query direction in a segment direction
SEGMENT_COS = 0.8             # cosine between a segment key and its segment direction
SINK_SCALE = 4.0
ZIPF_S = 1.1
ZIPF_TOP = 3.0
SEG_MIN, SEG_MAX = 20, 60
SEG_START = 4


def torch_dtype(wl: Workload):
    return torch.bfloat16 if wl.dtype == "bf16" else torch.float32


def _gen(device, *key: int) -> torch.Generator:
    g = torch.Generator(device=device)
    h = 0x9E3779B97F4A7C15
    for k in key:
        h = (h * 0x100000001B3 + (k & 0xFFFFFFFFFFFF) + 0x5851F42D) & 0x7FFFFFFFFFFFFFFF
    g.manual_seed(h)
    return g


def _unit_rows(n: int, d: int, g, device) -> torch.Tensor:
    return torch.randn(n, d, generator=g, device=device, dtype=torch.float32)


def _normalise(x: torch.Tensor) -> torch.Tensor:
    return x / x.norm(dim=-1, keepdim=True).clamp_min(1e-30)


def segment_layout(wl: Workload, unit: int, T: int | None = None) -> list[tuple[int, int]]:
    """(start, length) of the planted key clusters of one unit, non-overlapping in [4, T-R)."""
    T = wl.T if T is None else T
    if wl.keys != "segments" or wl.n_segments == 0:
        return []
    rng = np.random.default_rng([wl.seed, unit, 7])
    n = wl.n_segments
    lens = rng.integers(SEG_MIN, SEG_MAX + 1, size=n)
    room = (T - wl.R) - SEG_START - int(lens.sum())
    if room < 0:
        raise ValueError(f"{n} segments do not fit in T={T}")
    gaps = np.sort(rng.integers(0, room + 1, size=n))
    out, cursor = [], SEG_START
    prev = 0
    for g_, ln in zip(gaps, lens):
        cursor += int(g_ - prev)
        prev = int(g_)
        out.append((cursor, int(ln)))
        cursor += int(ln)
    return out


def _plant_unit(wl: Workload, unit: int, q: torch.Tensor, k: torch.Tensor, g) -> None:
    """Plant sinks / segments / zipf structure into one unit's keys (in place, f32)."""
    T, d = k.shape
    device = k.device
    qhat = _normalise(q.reshape(-1, d).mean(0))
    if wl.keys == "zipf":
        ranks = torch.randperm(T, generator=g, device=device).to(torch.float32) + 1.0
        k.mul_((1.0 + ZIPF_TOP * ranks.pow(-ZIPF_S)).unsqueeze(1))
    if wl.keys == "segments":
        segs = segment_layout(wl, unit, T)
        if segs:
            n = len(segs)
            ns = _normalise(torch.randn(n, d, generator=g, device=device))
            us = _normalise(SEGMENT_ALIGN * qhat + math.sqrt(1 - SEGMENT_ALIGN ** 2) * ns)
            starts = np.array([s_ for s_, _ in segs], dtype=np.int64)
            lens = np.array([ln for _, ln in segs], dtype=np.int64)
            sid_np = np.repeat(np.arange(n, dtype=np.int64), lens)
            pos_np = starts[sid_np] + (np.arange(lens.sum()) - np.repeat(np.cumsum(lens) - lens, lens))
            pos = torch.from_numpy(pos_np).to(device)
            sid = torch.from_numpy(sid_np).to(device)
            u = us[sid]
            e = torch.randn(pos.numel(), d, generator=g, device=device)
            e = _normalise(e - (e * u).sum(-1, keepdim=True) * u)
            norm = k[pos].norm(dim=-1, keepdim=True)
            k[pos] = norm * _normalise(SEGMENT_COS * u + math.sqrt(1 - SEGMENT_COS ** 2) * e)
    if wl.n_sinks:
        ns_ = min(wl.n_sinks, T)
        k[:ns_] = SINK_SCALE * k[:ns_].norm(dim=-1, keepdim=True) * qhat


def unit_tensors(wl: Workload, unit: int, device="cpu"):
    """(q [G][W][d], k [T][d], v [T][d]) of one unit, float32, structure planted."""
    g = _gen(device, wl.seed, unit, 1)
    q = _unit_rows(wl.G * wl.W, wl.d, g, device).reshape(wl.G, wl.W, wl.d)
    k = _unit_rows(wl.T, wl.d, g, device)
    v = _unit_rows(wl.T, wl.d, g, device)
    _plant_unit(wl, unit, q, k, g)
    return q, k, v


def prefill_inputs(wl: Workload, device="cpu", units=None):
    """Q [rows][Hq][W][d], K, V [rows][Hkv][T][d] in the workload dtype.

    With ``units`` (a list of unit indices) only those units are generated and the
    result has shape [len(units)][G][W][d] / [len(units)][T][d] per tensor, each
    bit-identical to the same unit of the full generation on the same device.
    """
    dt = torch_dtype(wl)
    if units is not None:
        qs, ks, vs = [], [], []
        for u in units:
            q, k, v = unit_tensors(wl, u, device)
            qs.append(q.to(dt))
            ks.append(k.to(dt))
            vs.append(v.to(dt))
        return torch.stack(qs), torch.stack(ks), torch.stack(vs)
    Q = torch.empty(wl.rows, wl.Hq, wl.W, wl.d, dtype=dt, device=device)
    K = torch.empty(wl.rows, wl.Hkv, wl.T, wl.d, dtype=dt, device=device)
    V = torch.empty_like(K)
    G = wl.G
    for u in range(wl.units):
        row, h = divmod(u, wl.Hkv)
        q, k, v = unit_tensors(wl, u, device)
        Q[row, h * G:(h + 1) * G].copy_(q.to(dt))
        K[row, h].copy_(k.to(dt))
        V[row, h].copy_(v.to(dt))
    return Q, K, V


def decode_inputs(wl: Workload, step: int, device="cpu"):
    """(q [rows][Hq][d], k_new, v_new [rows][Hkv][d]) for one decode step."""
    dt = torch_dtype(wl)
    g = _gen(device, wl.seed, step, 2)
    q = torch.randn(wl.rows, wl.Hq, wl.d, generator=g, device=device)
    k = torch.randn(wl.rows, wl.Hkv, wl.d, generator=g, device=device)
    v = torch.randn(wl.rows, wl.Hkv, wl.d, generator=g, device=device)
    if wl.keys == "zipf":
        r = torch.randint(1, wl.T + 1, (wl.rows, wl.Hkv, 1), generator=g, device=device)
        k.mul_(1.0 + ZIPF_TOP * r.to(torch.float32).pow(-ZIPF_S))
    return q.to(dt), k.to(dt), v.to(dt)


def to_numpy_bits(t: torch.Tensor) -> np.ndarray:
    """Host numpy copy of a tensor: uint16 bit patterns for bf16, the same dtype otherwise."""
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype in (torch.float32, torch.int32):
        return t.numpy()
    raise TypeError(t.dtype)


def from_numpy_bits(a: np.ndarray) -> torch.Tensor:
    """Inverse of to_numpy_bits (host tensor)."""
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16).copy()).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a))
