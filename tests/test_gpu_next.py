"""GPU parity for the variants beyond the five core steps: attention sinks in
Top-K and the decode step (KV-cache survey blog §4.1-4.2), and the HubKV
comparison variants (HubKV walkthrough, 尝试路线：效果一般的可能原因)."""
import numpy as np
import pytest
import torch

from _parity import RTOL, assert_close, decode_lockstep
from kv_cache_compression_obs_gb300 import gen

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.mark.parametrize("T,k,R,S", [(10, 5, 2, 2), (10, 10, 2, 3), (4096, 409, 32, 4),
                                     (8192, 1638, 819, 16), (3001, 300, 0, 5), (131072, 6553, 64, 4),
                                     (777, 100, 1, 98)])
@pytest.mark.parametrize("ties", [False, True])
def test_select_topk_sinks_bit_exact(kvc, oracle_mod, T, k, R, S, ties):
    B, H = 2, 3
    g = torch.Generator(device=DEV)
    g.manual_seed(T + k + S)
    z = torch.rand(B, H, T, generator=g, device=DEV)
    if ties:
        z = torch.floor(z * 7) / 7
        z[0, 0, ::5] = -0.0
        z[0, 0, 1::5] = 0.0
    z[..., :S] = -1.0  # sinks the scores alone would drop
    idx = kvc.kv_select_topk(z, k, R, sink=S)
    torch.cuda.synchronize()
    ref = oracle_mod.select_topk(z.cpu().numpy().astype(np.float64), k, R, sink=S)
    np.testing.assert_array_equal(idx.cpu().numpy(), ref)
    assert (idx[..., :S].cpu() == torch.arange(S, dtype=torch.int32)).all()


def _scores(B, H, T, seed):
    g = torch.Generator(device=DEV)
    g.manual_seed(seed)
    s = torch.rand(B, H, T, generator=g, device=DEV) ** 4
    return (s / s.sum(-1, keepdim=True) * 8).contiguous()


@pytest.mark.parametrize("flags", [1, 2, 3])
@pytest.mark.parametrize("shape", [(1, 1, 1), (1, 2, 3), (2, 8, 32768), (1, 4, 10001)])
@pytest.mark.parametrize("r", [0.1, 0.9])
def test_hubkv_variants(kvc, oracle_mod, flags, shape, r):
    B, H, T = shape
    s = _scores(B, H, T, seed=T + H + flags)
    z, beta = kvc.hubkv_refine(s, r, flags=flags)
    torch.cuda.synchronize()
    z_ref, beta_ref, _ = oracle_mod.hubkv_refine(s.cpu().numpy().astype(np.float64), r, flags=flags)
    assert_close(beta.cpu().numpy(), beta_ref, rtol=1e-6, atol=0, what="beta")
    assert_close(z.cpu().numpy(), z_ref, rtol=RTOL, atol=1e-30, what="z")
    if flags & kvc.KV_HUB_FIXED_HEAD:
        assert torch.all(beta == 1.0)


def test_hubkv_variant_flags_rejected(kvc):
    s = _scores(1, 2, 64, seed=1)
    with pytest.raises(kvc.KvcError):
        kvc.hubkv_refine(s, 0.5, flags=4)


@pytest.mark.parametrize("G,dt,d,R,S", [(4, "bf16", 128, 8, 4), (1, "f32", 64, 0, 2), (8, "bf16", 64, 3, 1),
                                        (2, "bf16", 128, 0, 6)])
def test_decode_lockstep_sinks(kvc, oracle_mod, G, dt, d, R, S):
    B, Hkv, cap, T0, steps = 2, 3, 40, 200, 30
    Hq = G * Hkv
    tdt = torch.bfloat16 if dt == "bf16" else torch.float32
    g = torch.Generator(device=DEV)
    g.manual_seed(G * 100 + d + R + S)
    Kc = torch.randn(B, Hkv, cap, d, generator=g, device=DEV).to(tdt)
    Vc = torch.randn(B, Hkv, cap, d, generator=g, device=DEV).to(tdt)
    pos = torch.stack([torch.sort(torch.randperm(T0 - S, generator=g, device=DEV)[:cap - S] + S).values
                       for _ in range(B * Hkv)]).reshape(B, Hkv, cap - S).to(torch.int32)
    pos = torch.cat([torch.arange(S, dtype=torch.int32, device=DEV).expand(B, Hkv, S), pos], -1).contiguous()
    acc = (torch.rand(B, Hkv, cap, generator=g, device=DEV) * 2).contiguous()
    acc[..., :S] = 0.0   # the sinks score lowest: only the protection keeps them
    ln = torch.full((B, Hkv), cap, dtype=torch.int32, device=DEV)
    scale = d ** -0.5
    exact = 0
    for step in range(steps):
        q = torch.randn(B, Hq, d, generator=g, device=DEV).to(tdt)
        kn = torch.randn(B, Hkv, d, generator=g, device=DEV).to(tdt)
        vn = torch.randn(B, Hkv, d, generator=g, device=DEV).to(tdt)
        exact += decode_lockstep(kvc, oracle_mod, q, kn, vn, Kc, Vc, pos, acc, ln, R, T0 + step, scale,
                                 sink=S)
        for s in range(S):
            assert bool((pos == s).any(-1).all()), "a sink was evicted"
    assert exact >= steps - 2


@pytest.mark.parametrize("G,sink,R,fill", [(4, 0, 16, 1.0), (2, 3, 0, 1.0), (1, 2, 8, 0.6)])
def test_multi_step_decode_equals_single_steps(kvc, G, sink, R, fill):
    """h2o_decode_steps is, bit for bit, the same single steps enqueued one by one
    (full caches evicting, and a partly filled cache appending first)."""
    g = torch.Generator(device=DEV)
    g.manual_seed(G * 10 + sink)
    B, Hkv, cap, d, n = 2, 3, 300, 128, 20
    Hq = Hkv * G
    K = torch.randn(B, Hkv, cap, d, generator=g, device=DEV).to(torch.bfloat16)
    V = torch.randn(B, Hkv, cap, d, generator=g, device=DEV).to(torch.bfloat16)
    pos = torch.arange(cap, dtype=torch.int32, device=DEV).repeat(B, Hkv, 1).contiguous()
    acc = torch.rand(B, Hkv, cap, generator=g, device=DEV)
    ln = torch.full((B, Hkv), int(cap * fill), dtype=torch.int32, device=DEV)
    q = torch.randn(n, B, Hq, d, generator=g, device=DEV).to(torch.bfloat16)
    kn = torch.randn(n, B, Hkv, d, generator=g, device=DEV).to(torch.bfloat16)
    vn = torch.randn(n, B, Hkv, d, generator=g, device=DEV).to(torch.bfloat16)
    one = [t.clone() for t in (K, V, pos, acc, ln)]
    many = [t.clone() for t in (K, V, pos, acc, ln)]
    o1, e1 = [], []
    for t in range(n):
        o, ev = kvc.h2o_decode_step(q[t], kn[t], vn[t], *one, R, cap + t, sink=sink)
        o1.append(o)
        e1.append(ev)
    o2, e2 = kvc.h2o_decode_steps(q, kn, vn, *many, R, cap, sink=sink)
    torch.cuda.synchronize()
    assert torch.equal(torch.stack(o1), o2) and torch.equal(torch.stack(e1), e2)
    for a, b in zip(one, many):
        assert torch.equal(a, b)


def test_multi_step_decode_alg1_and_zero_steps(kvc):
    g = torch.Generator(device=DEV)
    g.manual_seed(77)
    B, Hkv, G, cap, d, n = 1, 2, 4, 64, 64, 9
    K = torch.randn(B, Hkv, cap, d, generator=g, device=DEV)
    V = torch.randn(B, Hkv, cap, d, generator=g, device=DEV)
    pos = torch.arange(cap, dtype=torch.int32, device=DEV).repeat(B, Hkv, 1).contiguous()
    acc = torch.rand(B, Hkv, cap, generator=g, device=DEV)
    ln = torch.full((B, Hkv), cap, dtype=torch.int32, device=DEV)
    q = torch.randn(n, B, Hkv * G, d, generator=g, device=DEV)
    kn = torch.randn(n, B, Hkv, d, generator=g, device=DEV)
    vn = torch.randn(n, B, Hkv, d, generator=g, device=DEV)
    one = [t.clone() for t in (K, V, pos, acc, ln)]
    many = [t.clone() for t in (K, V, pos, acc, ln)]
    o1, e1 = zip(*[kvc.h2o_decode_step(q[t], kn[t], vn[t], *one, 0, cap + t, flags=kvc.KV_H2O_ALG1)
                   for t in range(n)])
    o2, e2 = kvc.h2o_decode_steps(q, kn, vn, *many, 0, cap, flags=kvc.KV_H2O_ALG1)
    torch.cuda.synchronize()
    assert torch.equal(torch.stack(o1), o2) and torch.equal(torch.stack(e1), e2)
    for a, b in zip(one, many):
        assert torch.equal(a, b)
    # zero steps: nothing changes
    before = [t.clone() for t in many]
    kvc.h2o_decode_steps(q[:0], kn[:0], vn[:0], *many, 0, cap + n, flags=kvc.KV_H2O_ALG1)
    torch.cuda.synchronize()
    for a, b in zip(before, many):
        assert torch.equal(a, b)


def test_decode_and_chain_graph_replay_equal_eager(kvc):
    """The library is safe to capture in a CUDA graph: the prefill chain and a
    multi-step decode (two row halves, the second on the library's side stream,
    joined through events) replayed from a graph give, bit for bit, what the
    same calls enqueued from the host give."""
    g = torch.Generator(device=DEV)
    g.manual_seed(2024)
    B, Hq, Hkv, T, d, W, k, R, n = 4, 8, 2, 2048, 128, 32, 256, 32, 12
    cap = k + 8
    Q = torch.randn(B, Hq, W, d, generator=g, device=DEV).to(torch.bfloat16)
    K = torch.randn(B, Hkv, T, d, generator=g, device=DEV).to(torch.bfloat16)
    V = torch.randn(B, Hkv, T, d, generator=g, device=DEV).to(torch.bfloat16)
    q = torch.randn(n, B, Hq, d, generator=g, device=DEV).to(torch.bfloat16)
    kn = torch.randn(n, B, Hkv, d, generator=g, device=DEV).to(torch.bfloat16)
    vn = torch.randn(n, B, Hkv, d, generator=g, device=DEV).to(torch.bfloat16)

    def buffers():
        f32, i32 = torch.float32, torch.int32
        return dict(s=torch.empty(B, Hkv, T, dtype=f32, device=DEV),
                    z=torch.empty(B, Hkv, T, dtype=f32, device=DEV),
                    idx=torch.empty(B, Hkv, k, dtype=i32, device=DEV),
                    Kc=torch.empty(B, Hkv, cap, d, dtype=K.dtype, device=DEV),
                    Vc=torch.empty(B, Hkv, cap, d, dtype=K.dtype, device=DEV),
                    pos=torch.empty(B, Hkv, cap, dtype=i32, device=DEV),
                    acc=torch.empty(B, Hkv, cap, dtype=f32, device=DEV),
                    ln=torch.empty(B, Hkv, dtype=i32, device=DEV),
                    o=torch.empty(n, B, Hq, d, dtype=f32, device=DEV),
                    ev=torch.empty(n, B, Hkv, dtype=i32, device=DEV),
                    ws=torch.empty(max(kvc.kv_workspace_size(kvc.KV_OP_SCORE_OBS, B, Hq, Hkv, T, d, W),
                                       kvc.kv_workspace_size(kvc.KV_OP_HUBKV_REFINE, B, Hkv, Hkv, T)),
                                   dtype=torch.uint8, device=DEV),
                    dws=torch.empty(kvc.kv_workspace_size(kvc.KV_OP_DECODE, B, Hq, Hkv, cap, d),
                                    dtype=torch.uint8, device=DEV))

    def run(b):
        kvc.kv_score_obs(Q, K, out=b["s"], workspace=b["ws"])
        kvc.hubkv_refine(b["s"], 0.1, out=b["z"], workspace=b["ws"])
        kvc.kv_select_topk(b["z"], k, R, out=b["idx"])
        kvc.kv_compact(K, V, b["s"], b["idx"], cap, K_out=b["Kc"], V_out=b["Vc"], pos_out=b["pos"],
                       acc_out=b["acc"], len_out=b["ln"])
        kvc.h2o_decode_steps(q, kn, vn, b["Kc"], b["Vc"], b["pos"], b["acc"], b["ln"], R, T,
                             o_out=b["o"], evicted_out=b["ev"], workspace=b["dws"])

    eager, graphed = buffers(), buffers()
    run(eager)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        run(graphed)  # warm-up on a non-default stream, then capture and replay once
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    for t in graphed.values():
        t.zero_()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        run(graphed)
    graph.replay()
    torch.cuda.synchronize()
    for name in ("s", "z", "idx", "Kc", "Vc", "pos", "acc", "ln", "o", "ev"):
        assert torch.equal(eager[name], graphed[name]), name


def test_select_topk_many_heads(kvc, oracle_mod):
    """Thousands of single-CTA heads and a few 2-CTA clusters in one launch."""
    g = torch.Generator(device=DEV)
    g.manual_seed(3001)
    for B, H, T, k, R in [(3, 1000, 1000, 100, 10), (1, 40, 17000, 1700, 64)]:
        z = torch.rand(B, H, T, generator=g, device=DEV)
        z = torch.floor(z * 50) / 50
        idx = kvc.kv_select_topk(z, k, R)
        torch.cuda.synchronize()
        ref = oracle_mod.select_topk(z.cpu().numpy().astype(np.float64), k, R)
        np.testing.assert_array_equal(idx.cpu().numpy(), ref)
