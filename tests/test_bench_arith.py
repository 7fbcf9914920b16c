"""The benchmark's roofline arithmetic on CPU: the algorithmic bytes and flops
`bench.py` divides by its event times, checked against the per-unit figures
worked out by hand for the long-context workload (32 layers x 8 KV heads,
G = 4 query heads per KV head, W = 64, d = 128, T = 131072, k = cap = 6553, bf16)."""
import pytest

import bench
from kv_cache_compression_obs_gb300 import configs

WL = configs.LONG_CONTEXT
UNITS = 32 * 8          # (layer, KV head) pairs of the one batch row
G, W, D, T, K = 4, 64, 128, 131072, 6553
ROW = D * 2             # one bf16 K or V row


def test_workload_shape():
    assert (WL.units, WL.Hq // WL.Hkv, WL.W, WL.d, WL.T, WL.k, WL.cap, WL.elem_bytes) == \
        (UNITS, G, W, D, T, K, K, 2)


def test_prefill_bytes_per_unit():
    a = bench.algorithmic_bytes(WL)
    # scoring: the unit's G x W query rows and its T keys read once, the scores written
    assert a["kv_score_obs"] == UNITS * (G * W * ROW + T * ROW + 4 * T)
    # refinement + Top-K (one call): the scores read twice (the head weights need
    # every score of a head before any refined score), k positions written
    assert a["hubkv_select_topk"] == UNITS * (2 * 4 * T + 4 * K)
    # compaction: k K rows and k V rows read and written, and per kept slot its
    # index, score, position and accumulator
    assert a["kv_compact"] == UNITS * K * (4 * ROW + 16)
    assert sum(a[n] for n in ("kv_score_obs", "hubkv_select_topk", "kv_compact")) \
        == 10_760_745_984


def test_decode_bytes_per_step():
    a = bench.algorithmic_bytes(WL)
    # every slot's K and V row, accumulator (read + write) and position; per unit
    # the G query rows (bf16 in, fp32 out) and the new token's K and V rows
    assert a["h2o_decode_step"] == UNITS * (K * (2 * ROW + 12) + G * D * 6 + 2 * ROW)
    assert a["h2o_decode_step"] == 879_963_136
    # the measured DRAM traffic the bench reports beside it is that, plus a few percent
    traffic = bench.DECODE_TRAFFIC_PER_UNIT["long-context"] * WL.units
    assert 1.0 <= traffic / a["h2o_decode_step"] <= 1.1
    # kept per unit: a run on fewer layers gets the same traffic per unit
    assert bench.DECODE_TRAFFIC_PER_UNIT["long-context"] * WL.scaled(L=2).units == traffic / 16


def test_score_flops_one_contraction_over_visible_pairs():
    # one Q K^T, 2 d flops per (query row, key) pair the window sees: row w of a
    # query head sits at position T - W + w and sees keys 0 .. T - W + w
    pairs = G * sum(T - W + w + 1 for w in range(W))
    assert bench.score_pairs(WL) == pairs == 33_546_368
    assert bench.score_flops(WL) == 2 * D * pairs * UNITS == 2_198_494_773_248
    # the two-pass kernels issue twice that (statistics, then column mass)
    assert bench.score_flops_executed(WL) == 2 * bench.score_flops(WL)


def test_score_pairs_full_causal():
    # every prompt position observed (W = T, the H2O decode workload's scoring):
    # the causal triangle, T (T + 1) / 2 pairs per query head
    wl = configs.H2O_DECODE
    assert wl.W == wl.T and wl.Hq == wl.Hkv
    assert bench.score_pairs(wl) == wl.T * (wl.T + 1) // 2


def test_whole_job_rate_counts_every_rank():
    # value = KV tokens (rows x T) of all ranks over the slowest rank's step time
    assert bench.whole_job_rate(WL.rows * WL.T, 1, 0.02338) == WL.rows * WL.T / 0.02338
    assert bench.whole_job_rate(100, 4, 2.0) == 200.0


def test_sfu_fraction_counts_one_exp_per_visible_pair():
    """The scoring's SFU fraction: one exponential per causally visible (row, key)
    pair (two as executed), against ex2/clock/SM x SMs x the sampled clock."""
    wl = configs.LONG_CONTEXT
    f = bench.sfu_fraction(wl, 2.0e-3, {"sm_mhz": 2000.0, "sm_max_mhz": 2070.0}, 152)
    exps = bench.score_pairs(wl) * wl.units
    peak = bench.SFU_EX2_PER_CLK_SM * 152 * 2000.0e6
    assert f["sfu_peak"] == pytest.approx(peak)
    assert f["sfu_exp_per_s"] == pytest.approx(exps / 2.0e-3)
    assert f["sfu_frac"] == pytest.approx(exps / 2.0e-3 / peak)
    assert f["sfu_executed_frac"] == pytest.approx(2 * f["sfu_frac"])
    assert bench.sfu_fraction(wl, 1.0, {}, 152) == {}
