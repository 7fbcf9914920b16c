"""GPU parity of the layer-level competitive budget (NestedKV technical summary,
3. Hoofd-gewijze Geheugentoewijzing; KV-cache survey blog §4.4, PyramidKV) and
of the ragged compaction that follows it.  Index work: bit-exact against the
oracle on the same float32 scores."""
import numpy as np
import pytest
import torch

from _parity import decode_lockstep
from kv_cache_compression_obs_gb300 import gen

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _z(B, H, T, seed, ties=False, spread=True):
    g = torch.Generator(device=DEV)
    g.manual_seed(seed)
    z = torch.rand(B, H, T, generator=g, device=DEV) ** 3
    if spread:  # heads on different scales, so the competition moves slots
        z = z * torch.exp(2 * torch.rand(1, H, 1, generator=g, device=DEV))
    if ties:
        z = torch.floor(z * 5) / 5
        z[0, 0, ::7] = -0.0
        z[0, 0, 3::7] = 0.0
    return z.contiguous()


CASES = [
    # B, H, T, budget, floor, R, S
    (1, 1, 10, 5, 3, 1, 1),            # one head: per-head Top-K with k = budget
    (2, 3, 10, 15, 3, 1, 1),           # cluster of 3
    (2, 3, 10, 30, 10, 2, 3),          # everything kept
    (2, 4, 700, 4 * 70, 70, 8, 4),     # budget = H * floor: no competition
    (2, 4, 700, 4 * 70, 12, 8, 4),     # floor = sinks + recent: all heavy slots compete
    (3, 8, 5000, 8 * 500, 125, 64, 4),  # ragged tail (T not a multiple of 1024)
    (1, 12, 3001, 12 * 300, 40, 0, 0),  # 12 heads on 8 CTAs: uneven ownership
    (1, 32, 4096, 32 * 409, 100, 32, 0),  # Llama-2-7B layer shape, 4 heads per CTA
    (2, 8, 131072, 8 * 6553, 1638, 64, 4),  # long-context layers
    (1, 5, 1, 5, 1, 0, 0),             # T = 1
    (1, 2, 2048, 2 * 2048 - 1, 2000, 16, 0),  # all but one kept
    (1, 4, 300000, 4 * 15000, 4000, 64, 4),   # heads too long for the on-chip bitmask
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}H{}T{}b{}f{}R{}S{}".format(*c))
@pytest.mark.parametrize("ties", [False, True])
def test_select_budget_bit_exact(kvc, oracle_mod, case, ties):
    B, H, T, budget, floor, R, S = case
    z = _z(B, H, T, seed=sum(case) + ties, ties=ties)
    idx, off = kvc.kv_select_budget(z, budget, floor, R, S)
    torch.cuda.synchronize()
    ref_idx, ref_off = oracle_mod.select_budget(z.cpu().numpy().astype(np.float64), budget, floor, R, S)
    np.testing.assert_array_equal(off.cpu().numpy(), ref_off)
    np.testing.assert_array_equal(idx.cpu().numpy(), ref_idx)
    # deterministic
    idx2, off2 = kvc.kv_select_budget(z, budget, floor, R, S)
    assert torch.equal(idx, idx2) and torch.equal(off, off2)


def test_select_budget_equals_per_head_topk_when_floor_fills_it(kvc):
    z = _z(3, 8, 8192, seed=5)
    k, R, S = 819, 64, 4
    idx, off = kvc.kv_select_budget(z, 8 * k, k, R, S)
    ref = kvc.kv_select_topk(z, k, R, sink=S)
    assert torch.equal(idx.view(3, 8, k), ref)
    assert torch.equal(off, (torch.arange(9, device=DEV, dtype=torch.int32) * k).expand(3, 9))


def test_select_budget_many_rows(kvc, oracle_mod):
    """More clusters than SMs can hold at once (64 rows x 8 CTAs)."""
    B, H, T, budget, floor, R, S = 64, 8, 2000, 8 * 200, 50, 16, 2
    z = _z(B, H, T, seed=77)
    idx, off = kvc.kv_select_budget(z, budget, floor, R, S)
    torch.cuda.synchronize()
    ref_idx, ref_off = oracle_mod.select_budget(z.cpu().numpy().astype(np.float64), budget, floor, R, S)
    np.testing.assert_array_equal(off.cpu().numpy(), ref_off)
    np.testing.assert_array_equal(idx.cpu().numpy(), ref_idx)


@pytest.mark.parametrize("levels", [0, 40, 3000])
@pytest.mark.parametrize("case", [(2, 4, 700, 4 * 120, 40, 8, 4), (1, 8, 4096, 8 * 400, 150, 32, 4),
                                  (1, 12, 3001, 12 * 300, 100, 16, 0)],
                         ids=lambda c: "B{}H{}T{}b{}f{}R{}S{}".format(*c))
def test_select_budget_thresholds_share_a_bin(kvc, oracle_mod, case, levels):
    """Scores in [1, 1.12): every pair has the same top 12 key bits, so each
    head's floor threshold and the competition's lie in one bin, the
    competition's second digits come from the floor's, and with few distinct
    values (`levels`) the two thresholds often share one 20-bit bucket too."""
    B, H, T, budget, floor, R, S = case
    g = torch.Generator(device=DEV)
    g.manual_seed(levels + T)
    u = torch.rand(B, H, T, generator=g, device=DEV)
    if levels:
        u = torch.floor(u * levels) / levels
    z = (1.0 + 0.12 * u).contiguous()
    idx, off = kvc.kv_select_budget(z, budget, floor, R, S)
    torch.cuda.synchronize()
    ref_idx, ref_off = oracle_mod.select_budget(z.cpu().numpy().astype(np.float64), budget, floor, R, S)
    np.testing.assert_array_equal(off.cpu().numpy(), ref_off)
    np.testing.assert_array_equal(idx.cpu().numpy(), ref_idx)


@pytest.mark.parametrize("which", ["all", "one_head"])
@pytest.mark.parametrize("case", [(2, 4, 700, 4 * 120, 40, 8, 4), (1, 8, 4096, 8 * 400, 150, 32, 4),
                                  (1, 12, 3001, 12 * 300, 100, 16, 0)],
                         ids=lambda c: "B{}H{}T{}b{}f{}R{}S{}".format(*c))
def test_select_budget_signed_scores(kvc, oracle_mod, case, which):
    """Negative scores (every head, or one head of each row beside non-negative
    ones, with -0.0 and +0.0 among them): the order keys of signed floats."""
    B, H, T, budget, floor, R, S = case
    g = torch.Generator(device=DEV)
    g.manual_seed(T + len(which))
    if which == "all":
        z = torch.randn(B, H, T, generator=g, device=DEV)
    else:
        z = torch.rand(B, H, T, generator=g, device=DEV) ** 2
        z[:, 1] -= 0.5
    z[:, :, 5::11] = -0.0
    z[:, :, 7::13] = 0.0
    z = z.contiguous()
    idx, off = kvc.kv_select_budget(z, budget, floor, R, S)
    torch.cuda.synchronize()
    ref_idx, ref_off = oracle_mod.select_budget(z.cpu().numpy().astype(np.float64), budget, floor, R, S)
    np.testing.assert_array_equal(off.cpu().numpy(), ref_off)
    np.testing.assert_array_equal(idx.cpu().numpy(), ref_idx)


# ---------------------------------------------------------------- ragged compaction
@pytest.mark.parametrize("dt,d", [("bf16", 128), ("f32", 64), ("bf16", 64)])
def test_compact_ragged_bit_exact(kvc, oracle_mod, dt, d):
    B, H, T = 2, 8, 3000
    budget, floor, R, S = 8 * 300, 60, 16, 4
    z = _z(B, H, T, seed=d)
    g = torch.Generator(device=DEV)
    g.manual_seed(9)
    tdt = torch.bfloat16 if dt == "bf16" else torch.float32
    K = torch.randn(B, H, T, d, generator=g, device=DEV).to(tdt)
    V = torch.randn(B, H, T, d, generator=g, device=DEV).to(tdt)
    s = torch.rand(B, H, T, generator=g, device=DEV)
    idx, off = kvc.kv_select_budget(z, budget, floor, R, S)
    cap = int((off[:, 1:] - off[:, :-1]).max()) + 5
    sent = dict(K_out=torch.full((B, H, cap, d), 3.0, device=DEV).to(tdt),
                V_out=torch.full((B, H, cap, d), -2.0, device=DEV).to(tdt),
                pos_out=torch.full((B, H, cap), -7, dtype=torch.int32, device=DEV),
                acc_out=torch.full((B, H, cap), 9.0, device=DEV),
                len_out=torch.full((B, H), -1, dtype=torch.int32, device=DEV))
    out = kvc.kv_compact_ragged(K, V, s, idx, off, cap, **sent)
    torch.cuda.synchronize()
    bits = gen.to_numpy_bits
    ref_out = tuple(bits(t).copy() if t.dtype == torch.bfloat16 else t.cpu().numpy().copy()
                    for t in (sent["K_out"], sent["V_out"], sent["pos_out"], sent["acc_out"],
                              sent["len_out"]))
    # the oracle writes into copies of the same sentinel-filled buffers
    ref = oracle_mod.compact_ragged(bits(K), bits(V), s.cpu().numpy().astype(np.float64),
                                    idx.cpu().numpy(), off.cpu().numpy(), cap, out=ref_out)
    for got, want in zip(out, ref):
        got_np = bits(got) if got.dtype == torch.bfloat16 else got.cpu().numpy()
        np.testing.assert_array_equal(got_np, want)


def test_compact_ragged_device_status(kvc):
    """An overfull head and malformed offsets are reported on the device and
    leave their head / row untouched; the rest is still written."""
    B, H, T, d = 2, 2, 50, 64
    K = torch.randn(B, H, T, d, device=DEV)
    idx = torch.arange(10, dtype=torch.int32, device=DEV).repeat(B, 1).contiguous()
    off = torch.tensor([[0, 3, 10], [0, 6, 4]], dtype=torch.int32, device=DEV)  # row 1 decreasing
    cap = 5
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    Ko = torch.full((B, H, cap, d), 7.0, device=DEV)
    pos = torch.full((B, H, cap), -9, dtype=torch.int32, device=DEV)
    ln = torch.full((B, H), -1, dtype=torch.int32, device=DEV)
    kvc.kv_compact_ragged(K, K, None, idx, off, cap, K_out=Ko, V_out=Ko.clone(), pos_out=pos,
                          len_out=ln, dev_status=status)
    torch.cuda.synchronize()
    assert int(status) == kvc.KV_ERR_INVALID_ARG
    assert ln.cpu().tolist() == [[3, -1], [-1, -1]]
    assert pos[0, 0].cpu().tolist() == [0, 1, 2, -9, -9]
    assert torch.equal(Ko[0, 0, :3], K[0, 0, :3])
    assert (pos[0, 1] == -9).all() and (pos[1] == -9).all() and (Ko[1] == 7.0).all()


def test_budget_chain_then_decode_appends(kvc, oracle_mod):
    """Budget, ragged compaction, then decode steps over the per-head lengths:
    heads below capacity append, the others evict (lock-step with the oracle)."""
    B, Hkv, G, T, d = 1, 4, 2, 600, 64
    budget, floor, R, S = 4 * 60, 20, 8, 2
    z = _z(B, Hkv, T, seed=31)
    g = torch.Generator(device=DEV)
    g.manual_seed(32)
    K = torch.randn(B, Hkv, T, d, generator=g, device=DEV).to(torch.bfloat16)
    V = torch.randn(B, Hkv, T, d, generator=g, device=DEV).to(torch.bfloat16)
    s = torch.rand(B, Hkv, T, generator=g, device=DEV)
    idx, off = kvc.kv_select_budget(z, budget, floor, R, S)
    counts = (off[:, 1:] - off[:, :-1]).cpu()
    cap = int(counts.max()) + 3
    Kc, Vc, pos, acc, ln = kvc.kv_compact_ragged(K, V, s, idx, off, cap)
    torch.cuda.synchronize()
    assert torch.equal(ln.cpu(), counts)
    scale = d ** -0.5
    for step in range(12):
        q = torch.randn(B, Hkv * G, d, generator=g, device=DEV).to(torch.bfloat16)
        kn = torch.randn(B, Hkv, d, generator=g, device=DEV).to(torch.bfloat16)
        vn = torch.randn(B, Hkv, d, generator=g, device=DEV).to(torch.bfloat16)
        decode_lockstep(kvc, oracle_mod, q, kn, vn, Kc, Vc, pos, acc, ln, R, T + step, scale, sink=S)
    torch.cuda.synchronize()
    assert torch.equal(ln.cpu(), torch.clamp(counts + 12, max=cap))


def test_select_budget_max_heads(kvc, oracle_mod):
    """256 heads: 32 heads per CTA of an 8-CTA cluster."""
    B, H, T = 2, 256, 300
    z = _z(B, H, T, seed=256, ties=True)
    budget, floor, R, S = H * 40, 20, 4, 2
    idx, off = kvc.kv_select_budget(z, budget, floor, R, S)
    torch.cuda.synchronize()
    ref_idx, ref_off = oracle_mod.select_budget(z.cpu().numpy().astype(np.float64), budget, floor, R, S)
    np.testing.assert_array_equal(off.cpu().numpy(), ref_off)
    np.testing.assert_array_equal(idx.cpu().numpy(), ref_idx)


def test_compact_ragged_empty_heads_and_zero_budget(kvc, oracle_mod):
    B, H, T, d, cap = 1, 4, 40, 64, 6
    K = torch.randn(B, H, T, d, device=DEV)
    idx = torch.tensor([[3, 9, 1, 0, 5]], dtype=torch.int32, device=DEV)
    off = torch.tensor([[0, 0, 2, 2, 5]], dtype=torch.int32, device=DEV)  # heads 0 and 2 keep nothing
    outs = dict(K_out=torch.full((B, H, cap, d), 5.0, device=DEV),
                V_out=torch.full((B, H, cap, d), 5.0, device=DEV),
                pos_out=torch.full((B, H, cap), -3, dtype=torch.int32, device=DEV),
                len_out=torch.full((B, H), -1, dtype=torch.int32, device=DEV))
    kvc.kv_compact_ragged(K, K, None, idx, off, cap, **outs)
    torch.cuda.synchronize()
    ref = oracle_mod.compact_ragged(K.cpu().numpy(), K.cpu().numpy(), None, idx.cpu().numpy(),
                                    off.cpu().numpy(), cap,
                                    out=tuple(t.cpu().numpy().copy() for t in (
                                        outs["K_out"], outs["V_out"], outs["pos_out"],
                                        torch.zeros(B, H, cap), outs["len_out"])))
    np.testing.assert_array_equal(outs["len_out"].cpu().numpy(), [[0, 2, 0, 3]])
    np.testing.assert_array_equal(outs["pos_out"].cpu().numpy(), ref[2])
    np.testing.assert_array_equal(outs["K_out"].cpu().numpy(), ref[0])
    # a zero budget writes only the lengths
    idx0 = torch.zeros(B, 0, dtype=torch.int32, device=DEV)
    off0 = torch.zeros(B, H + 1, dtype=torch.int32, device=DEV)
    kvc.kv_compact_ragged(K, K, None, idx0, off0, cap, **outs)
    torch.cuda.synchronize()
    assert (outs["len_out"] == 0).all()
    np.testing.assert_array_equal(outs["pos_out"].cpu().numpy(), ref[2])
