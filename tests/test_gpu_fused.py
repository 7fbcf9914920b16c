"""hubkv_select_topk: the HubKV refinement folded into the Top-K selection.

The fused call must return exactly what the two separate calls return
(hubkv_refine_ex, then kv_select_topk_ex on its z): the kept positions, and
z / beta when asked for, bit for bit, and its kept positions must equal the
float64 oracle's selection on those same z bits.  Shapes cover the on-chip path
(heads of up to 393216 candidates, z formed while the selection loads its
slice), the long-head path (z first, then the streaming selection), k = T,
sinks, both discount variants and the fixed head weight.
"""
import numpy as np
import pytest
import torch

from _parity import assert_close

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _scores(B, H, T, seed):
    g = torch.Generator(device=DEV)
    g.manual_seed(seed)
    s = torch.rand(B, H, T, generator=g, device=DEV) ** 6
    s = torch.nn.functional.max_pool1d(s.reshape(B * H, 1, T), 3, 1, 1).reshape(B, H, T)
    s = s + 1e-4 * torch.rand(B, H, T, generator=g, device=DEV)
    s[..., :4] += 3.0  # sinks
    s[..., T // 3: T // 3 + min(9, T // 3)] = 0.5  # a tied plateau
    return s.contiguous()


CASES = [
    # B, H, T, k, recent, sink, r, flags
    (1, 1, 1, 1, 0, 0, 0.1, 0),             # T = 1 (k = T)
    (2, 3, 777, 80, 5, 0, 0.9, 0),          # strong gate
    (1, 4, 5000, 500, 17, 3, 0.2, 2),       # fixed head weight, sinks
    (2, 4, 32768, 3276, 64, 0, 0.1, 1),     # average-pool variant, GQA-prefill head length
    (1, 8, 131072, 6553, 64, 4, 0.05, 0),   # one long-context layer
    (1, 2, 1000, 1000, 10, 0, 0.3, 0),      # k = T: everything kept
    (1, 2, 400000, 20000, 64, 0, 0.1, 0),   # too long to hold on chip
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}H{}T{}k{}R{}S{}r{}f{}".format(*c))
def test_fused_equals_separate_calls(kvc, oracle_mod, case):
    B, H, T, k, R, S, r, flags = case
    s = _scores(B, H, T, seed=T + k)
    z = torch.full_like(s, float("nan"))
    beta = torch.full((B, H), float("nan"), device=DEV)
    idx = kvc.hubkv_select_topk(s, k, R, r, sink=S, flags=flags, z_out=z, beta_out=beta)
    idx_plain = kvc.hubkv_select_topk(s, k, R, r, sink=S, flags=flags)  # z never written
    z_ref, beta_ref = kvc.hubkv_refine(s, r, flags=flags)
    idx_ref = kvc.kv_select_topk(z_ref, k, R, sink=S)
    torch.cuda.synchronize()
    assert torch.equal(z, z_ref)
    assert torch.equal(beta, beta_ref)
    assert torch.equal(idx, idx_ref)
    assert torch.equal(idx_plain, idx_ref)
    # against the oracle: the selection on the same z bits, and z itself
    z_np = z.cpu().numpy().astype(np.float64)
    np.testing.assert_array_equal(idx.cpu().numpy(), oracle_mod.select_topk(z_np, k, R, S))
    if T <= 131072:
        z_or, beta_or, _ = oracle_mod.hubkv_refine(s.cpu().numpy().astype(np.float64), r,
                                                    flags=flags)
        assert_close(z.cpu().numpy(), z_or, rtol=1e-5, atol=1e-30, what="z")


@pytest.mark.parametrize("pool_width,flags", [(1, 0), (3, 0), (9, 0), (129, 0), (7, 1), (5, 1)])
def test_fused_pool_widths(kvc, oracle_mod, pool_width, flags):
    """Pooling windows other than the default 5 (which has its own four-candidate
    path in the selection kernel) take the generic per-candidate gate: the same
    bits as the separate refinement, and the oracle's selection on them."""
    B, H, T, k, R, S, r = 2, 3, 20000, 2000, 32, 2, 0.3
    s = _scores(B, H, T, seed=pool_width + 17)
    z = torch.full_like(s, float("nan"))
    idx = kvc.hubkv_select_topk(s, k, R, r, pool_width=pool_width, sink=S, flags=flags, z_out=z)
    z_ref, _ = kvc.hubkv_refine(s, r, pool_width=pool_width, flags=flags)
    idx_ref = kvc.kv_select_topk(z_ref, k, R, sink=S)
    torch.cuda.synchronize()
    assert torch.equal(z, z_ref)
    assert torch.equal(idx, idx_ref)
    z_np = z.cpu().numpy().astype(np.float64)
    np.testing.assert_array_equal(idx.cpu().numpy(), oracle_mod.select_topk(z_np, k, R, S))
    z_or, _, _ = oracle_mod.hubkv_refine(s.cpu().numpy().astype(np.float64), r, pool_width=pool_width,
                                         flags=flags)
    assert_close(z.cpu().numpy(), z_or, rtol=1e-5, atol=1e-30, what="z")
