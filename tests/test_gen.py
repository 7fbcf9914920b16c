"""The seeded input generator: determinism, unit independence and planted structure."""
import math

import numpy as np
import pytest
import torch

from kv_cache_compression_obs_gb300 import configs, gen


def _small(wl, **kw):
    return wl.scaled(**kw)


def test_deterministic_and_subset_identical():
    wl = _small(configs.GQA_PREFILL, B=1, L=2, T=2048, W=16, k=205, R=16, n_segments=20)
    Q1, K1, V1 = gen.prefill_inputs(wl)
    Q2, K2, V2 = gen.prefill_inputs(wl)
    assert torch.equal(Q1, Q2) and torch.equal(K1, K2) and torch.equal(V1, V2)
    units = [3, 0, 12]
    q, k, v = gen.prefill_inputs(wl, units=units)
    for i, u in enumerate(units):
        row, h = divmod(u, wl.Hkv)
        assert torch.equal(q[i], Q1[row, h * wl.G:(h + 1) * wl.G])
        assert torch.equal(k[i], K1[row, h]) and torch.equal(v[i], V1[row, h])


def test_segments_are_disjoint_and_placed():
    wl = configs.LONG_CONTEXT
    for unit in (0, 77, 255):
        segs = gen.segment_layout(wl, unit)
        assert len(segs) == wl.n_segments
        end = gen.SEG_START
        for s, ln in segs:
            assert gen.SEG_MIN <= ln <= gen.SEG_MAX and s >= end
            end = s + ln
        assert end <= wl.T - wl.R


def test_segment_keys_cosine_and_sinks():
    wl = _small(configs.LONG_CONTEXT, L=1, Hkv=2, Hq=8, T=4096, k=205, R=64, n_segments=30)
    q, k, _ = gen.unit_tensors(wl, 1)
    qhat = q.reshape(-1, wl.d).mean(0)
    qhat = qhat / qhat.norm()
    for s, ln in gen.segment_layout(wl, 1):
        ks = k[s:s + ln]
        kn = ks / ks.norm(dim=-1, keepdim=True)
        # all keys of a run share a direction u with cosine 0.8: pairwise cosine 0.64 on average
        c = (kn @ kn.T)[~torch.eye(ln, dtype=bool)]
        assert abs(c.mean().item() - 0.64) < 0.08
    sink = k[:wl.n_sinks] / k[:wl.n_sinks].norm(dim=-1, keepdim=True)
    assert torch.allclose(sink @ qhat, torch.ones(wl.n_sinks), atol=1e-5)


def test_zipf_norm_profile():
    wl = _small(configs.H2O_DECODE, B=1, Hq=1, Hkv=1, T=4096, W=8, k=819, R=409)
    _, k, _ = gen.unit_tensors(wl, 0)
    norms = k.norm(dim=-1) / math.sqrt(wl.d)
    assert norms.max().item() > 3.0      # the rank-1 key is scaled by 4
    assert abs(norms.median().item() - 1.0) < 0.05


def test_bf16_is_round_to_nearest_even():
    x = torch.tensor([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -(1.0 + 2 ** -8)], dtype=torch.float32)
    bits = gen.to_numpy_bits(x.to(torch.bfloat16))
    # halfway cases round to the even mantissa
    assert list(bits) == [0x3F80, 0x3F82, 0xBF80]
    assert torch.equal(gen.from_numpy_bits(bits).to(torch.float32),
                       torch.tensor([1.0, 1.0 + 2 ** -6, -1.0]))


def test_decode_inputs_shapes():
    wl = configs.TINY
    q, k, v = gen.decode_inputs(wl, 0)
    assert q.shape == (1, 4, 64) and k.shape == (1, 4, 64) and q.dtype == torch.float32
    q2, _, _ = gen.decode_inputs(wl, 0)
    assert torch.equal(q, q2)
