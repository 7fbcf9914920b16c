"""Benchmark of the KV-cache eviction path on one GB300 (or N, one process each).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl ours|reference]

One step is the whole path over one batch of synthetic input: observation-window
scoring, HubKV refinement, Top-K and compaction of every (batch row x layer x KV
head), then the workload's H2O decode steps on the compacted cache.  The default
workload is the 128K long-context one (1 x 32 layers, 32 query / 8 KV heads,
d = 128, T = 131072, bf16, 5% budget incl. 64 recent, then 128 decode steps); it
is the workload that exercises all five operations at full size.

Prints one JSON line (rank 0).  `value` is KV tokens (batch rows x layers x
prompt tokens) scored + selected + compacted per second over whole steps, summed
over ranks; `decode` reports H2O decode steps per second; `roofline` is the
dominant kernel's achieved bandwidth against the measured HBM copy peak;
`cpu_baseline` times the float64 oracle on a bounded sample on the host cores;
`next_rows` times the rows built beyond the five-step path (layer-level budget,
ragged compaction, NestedKV key-only scoring) on the same workload, outside the
timed step.
Under torchrun every rank runs its own full workload (weak scaling, no
collective on the data path); rank 0 reports the max time over ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "KV tokens scored+selected+compacted/s; H2O decode steps/s; % HBM roofline"
UNIT = "KV tokens/s"
L2_BYTES = 129 * 2 ** 20


def _env_int(name, default):
    try:
        return int(os.environ.get(name, default))
    except ValueError:
        return default


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)  # ~0.8 s timed: several clock samples
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--config", default="long-context")
    ap.add_argument("--layers", type=int, default=None,
                    help="override the workload's layer count (smaller profiling cases)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--eager", action="store_true",
                    help="enqueue every launch from the host in the timed region (no CUDA graphs)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-groups", type=int, default=None,
                    help="layer-row groups of the end-to-end path (default E2E_GROUPS)")
    ap.add_argument("--no-next-rows", action="store_true",
                    help="skip the separate timing of the rows beyond the five-step path")
    ap.add_argument("--no-other-workloads", action="store_true",
                    help="skip the separate timing of the other workloads (single layer, H2O "
                         "decode, GQA prefill)")
    return ap.parse_args()


# ---------------------------------------------------------------------------
# algorithmic work per step (bytes that any implementation must move)
# ---------------------------------------------------------------------------
def algorithmic_bytes(wl):
    eb = wl.elem_bytes
    units = wl.units
    q_bytes = wl.rows * wl.Hq * wl.W * wl.d * eb
    k_bytes = units * wl.T * wl.d * eb
    s_bytes = units * wl.T * 4
    score = q_bytes + k_bytes + s_bytes                    # read Q, K; write s
    # refinement + Top-K (one fused call): the head weights need each head's whole
    # score vector before any refined score exists, so s is read twice (entropy,
    # then the selection, which forms z as it loads); the kept positions written
    select = (2 * s_bytes if wl.r is not None else s_bytes) + units * wl.k * 4
    row = wl.d * eb
    compact = units * wl.k * (4 * row + 4 + 4 + 4 + 4)     # K,V rows read+written; idx, s, pos, acc
    decode_step = units * wl.cap * (2 * row + 4 + 4 + 4) + wl.rows * (wl.Hq * wl.d * (eb + 4)
                                                                    + 2 * wl.Hkv * row)
    return {"kv_score_obs": score, "hubkv_select_topk": select,
            "kv_compact": compact, "h2o_decode_step": decode_step}


def score_pairs(wl):
    """(query row, key) pairs the observation window sees per (batch row, KV head):
    each of the G query heads' W rows at prompt position p = T - W + w sees the
    keys 0..p (causal), G * (W (T - W) + W (W + 1) / 2) in all."""
    G = wl.Hq // wl.Hkv
    return G * (wl.W * (wl.T - wl.W) + wl.W * (wl.W + 1) // 2)


def score_flops(wl):
    """Algorithmic flops of the observation-window contraction: one Q K^T over the
    visible (row, key) pairs, 2 d per pair (multiply + add), for every unit.  The
    exact column mass needs every row's softmax normaliser first, so the kernels
    form each logit twice; that recompute is reported as executed work, not
    counted here."""
    return 2 * wl.d * score_pairs(wl) * wl.units


# ex2 results per clock per SM of this GPU's special-function units, measured with a
# register-only probe (a dependent-free stream of ex2.approx.ftz.f32 on every SM)
SFU_EX2_PER_CLK_SM = 31.4


def sfu_fraction(wl, score_s, clocks, sms):
    """Exponentials per second of the scoring against the SFU rate of `sms` SMs at the
    sampled SM clock: one exp per visible (row, key) pair algorithmically, two as
    executed."""
    mhz = clocks.get("sm_mhz") or clocks.get("sm_max_mhz")
    if not mhz:
        return {}
    peak = SFU_EX2_PER_CLK_SM * sms * mhz * 1e6
    exps = score_pairs(wl) * wl.units
    return {"sfu_exp_per_s": exps / score_s, "sfu_peak": peak,
            "sfu_peak_kind": f"probe-measured {SFU_EX2_PER_CLK_SM} ex2/clock/SM x {sms} SMs x "
                             f"{mhz:.0f} MHz (sampled)",
            "sfu_frac": exps / score_s / peak, "sfu_executed_frac": 2 * exps / score_s / peak}


def score_flops_executed(wl):
    """Flops the two-pass kernels issue: both passes over every visible pair."""
    return 2 * score_flops(wl)


# DRAM bytes per decode step and unit (all the step's launches: the two row halves'
# stream and finalize kernels) from `ncu --metrics dram__bytes_read.sum,
# dram__bytes_write.sum`, captured on 8 of the 32 layers of the long-context
# workload (mean over four row halves of 32 units each; the traffic is
# proportional to the units, so a run on fewer layers scales it), with the
# SHA-256 of the decode kernel source it was taken on.  When the source has
# changed since, the figure no longer describes the kernel and is reported as null.
DECODE_TRAFFIC_PER_UNIT = {"long-context": (107470016 + 897536 + 5472576) / 32}
DECODE_TRAFFIC_SOURCE = "kv_cache_compression_obs_gb300/csrc/h2o_decode.cu"
DECODE_TRAFFIC_SOURCE_SHA256 = "20c1313e366e778898cf19320ffdbee6ee33b6b3d030d9bb99bdd90496642201"


def _source_sha256(rel):
    import hashlib
    try:
        with open(os.path.join(ROOT, rel), "rb") as f:
            return hashlib.sha256(f.read()).hexdigest()
    except OSError:
        return None


def measured_peaks():
    """(HBM GB/s, bf16 dense TFLOP/s burst, kind): MEASURED_PEAKS.json, else the fallback."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


class ClockSampler:
    """nvidia-smi clock/throttle samples while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                self.out = ""

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in (self.out or "").splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# the GPU path
# ---------------------------------------------------------------------------
class Pipeline:
    """Preallocated buffers for one workload; step() enqueues the whole path."""

    def __init__(self, wl, device):
        import torch

        from kv_cache_compression_obs_gb300 import api, gen

        self.api, self.wl, self.dev = api, wl, device
        self.Q, self.K, self.V = gen.prefill_inputs(wl, device=device)
        units_shape = (wl.rows, wl.Hkv)
        f32, i32 = torch.float32, torch.int32
        self.s = torch.empty(*units_shape, wl.T, dtype=f32, device=device)
        self.z = torch.empty_like(self.s) if wl.r is not None else self.s
        self.beta = torch.empty(*units_shape, dtype=f32, device=device)
        self.idx = torch.empty(*units_shape, wl.k, dtype=i32, device=device)
        dt = self.K.dtype
        self.Kc = torch.empty(*units_shape, wl.cap, wl.d, dtype=dt, device=device)
        self.Vc = torch.empty_like(self.Kc)
        self.pos = torch.empty(*units_shape, wl.cap, dtype=i32, device=device)
        self.acc = torch.empty(*units_shape, wl.cap, dtype=f32, device=device)
        self.len = torch.empty(*units_shape, dtype=i32, device=device)
        nd = max(wl.n_decode, 1)
        self.O = torch.empty(nd, wl.rows, wl.Hq, wl.d, dtype=f32, device=device)  # every step's output
        self.EV = torch.empty(nd, *units_shape, dtype=i32, device=device)
        self.o, self.ev = self.O[-1], self.EV[-1]
        ws = max(api.kv_workspace_size(api.KV_OP_SCORE_OBS, wl.rows, wl.Hq, wl.Hkv, wl.T, wl.d, wl.W),
                 api.kv_workspace_size(api.KV_OP_HUBKV_SELECT, wl.rows, wl.Hkv, wl.Hkv, wl.T, 0,
                                       wl.R, wl.k), 256)
        self.ws = torch.empty(ws, dtype=torch.uint8, device=device)
        dws = api.kv_workspace_size(api.KV_OP_DECODE, wl.rows, wl.Hq, wl.Hkv, wl.cap, wl.d)
        self.dws = torch.empty(max(dws, 256), dtype=torch.uint8, device=device)
        steps = [gen.decode_inputs(wl, t, device=device) for t in range(wl.n_decode)]
        if steps:  # [n_decode][rows][heads][d], one tensor per input
            self.DQ, self.DK, self.DV = (torch.stack([x[i] for x in steps]) for i in range(3))
        self.dq = [self.DQ[t] for t in range(wl.n_decode)]
        self.dk = [self.DK[t] for t in range(wl.n_decode)]
        self.dv = [self.DV[t] for t in range(wl.n_decode)]

    def select(self, stream=None):
        """HubKV refinement + Top-K (one fused call), or Top-K on s without refinement."""
        a, wl = self.api, self.wl
        if wl.r is not None:
            a.hubkv_select_topk(self.s, wl.k, wl.R, wl.r, wl.gamma, wl.pool_width, wl.beta_lo,
                                wl.beta_hi, out=self.idx, beta_out=self.beta, workspace=self.ws,
                                stream=stream)
        else:
            a.kv_select_topk(self.s, wl.k, wl.R, out=self.idx, stream=stream)

    def prefill(self, stream=None):
        a, wl = self.api, self.wl
        a.kv_score_obs(self.Q, self.K, wl.scale, out=self.s, workspace=self.ws, stream=stream)
        self.select(stream)
        a.kv_compact(self.K, self.V, self.s, self.idx, wl.cap, K_out=self.Kc, V_out=self.Vc,
                     pos_out=self.pos, acc_out=self.acc, len_out=self.len, stream=stream)

    def decode_all(self, stream=None):
        """All the workload's decode steps, one library call."""
        wl = self.wl
        if wl.n_decode:
            self.api.h2o_decode_steps(self.DQ, self.DK, self.DV, self.Kc, self.Vc, self.pos,
                                      self.acc, self.len, wl.R, wl.T, wl.scale, o_out=self.O,
                                      evicted_out=self.EV, workspace=self.dws, stream=stream)

    def step(self, stream=None):
        if self.graphs is not None:
            self.graphs[0].replay()
            if self.graphs[1] is not None:
                self.graphs[1].replay()
            return
        self.prefill(stream)
        self.decode_all(stream)

    graphs = None  # (prefill, decode) CUDA graphs once captured
    launches_per_step = None

    def capture(self):
        """The step as two CUDA graphs (the prefill chain, then every decode step),
        captured once after warm-up and replayed: the 128 x 4 decode launches then
        cost no host round trip each.  The library's own side stream joins the
        capture through its fork / join events."""
        import torch
        side = torch.cuda.Stream(device=self.dev)
        side.wait_stream(torch.cuda.current_stream(self.dev))
        with torch.cuda.stream(side):  # one eager pass on a non-default stream first
            self.prefill()
            self.decode_all()
        torch.cuda.current_stream(self.dev).wait_stream(side)
        torch.cuda.synchronize(self.dev)
        gp = torch.cuda.CUDAGraph()
        gd = torch.cuda.CUDAGraph() if self.wl.n_decode else None
        n0 = launch_count()
        with torch.cuda.graph(gp):
            self.prefill()
        n1 = launch_count()
        if gd is not None:  # a workload without decode steps has no decode graph
            with torch.cuda.graph(gd):
                self.decode_all()
        n2 = launch_count()
        torch.cuda.synchronize(self.dev)
        self.graphs = (gp, gd)
        self.launches_per_step = n2 - n0
        self.launches_decode = n2 - n1

    def timed_phases(self):
        """One step with events between the phases: ms per phase."""
        import torch
        a, wl = self.api, self.wl
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
        ev[0].record()
        a.kv_score_obs(self.Q, self.K, wl.scale, out=self.s, workspace=self.ws)
        ev[1].record()
        self.select()
        ev[2].record()
        a.kv_compact(self.K, self.V, self.s, self.idx, wl.cap, K_out=self.Kc, V_out=self.Vc,
                     pos_out=self.pos, acc_out=self.acc, len_out=self.len)
        ev[3].record()
        if self.graphs is not None:
            if self.graphs[1] is not None:
                self.graphs[1].replay()
        else:
            self.decode_all()
        ev[4].record()
        torch.cuda.synchronize()
        names = ["kv_score_obs", "hubkv_select_topk", "kv_compact", "h2o_decode_step"]
        ms = {n: ev[i].elapsed_time(ev[i + 1]) for i, n in enumerate(names)}
        if wl.n_decode:
            ms["h2o_decode_step"] /= wl.n_decode  # per decode step
        return ms


NESTED_THRESH = 0.1  # surprise threshold of the NestedKV timing (the pages leave it open)


def nested_bytes(wl):
    """Bytes any NestedKV scorer must move: the keys twice (the stable anchor needs
    every key before any score, and a head's keys do not fit on chip), the three
    anomaly scores written once and read twice (the discriminative powers need all
    of them before the final pass), and the score written."""
    k_bytes = wl.units * wl.T * wl.d * wl.elem_bytes
    return 2 * k_bytes + wl.units * wl.T * (12 + 12 + 12 + 4)


def budget_floor(wl):
    """Per-head minimum for the layer-level budget on a workload: the recent window
    plus a quarter of the head's heavy share, k_heavy = k - R."""
    return wl.R + (wl.k - wl.R) // 4


def time_next_rows(pipe, reps=5, warmup=3):
    """Event timing of the rows built beyond the five-step path, on the same
    workload's buffers, outside the timed step: the layer-level budget
    (kv_select_budget on z with the same total, Hkv x k per layer) and the ragged
    compaction that follows it.  L2 is flushed before every repetition."""
    import torch
    a, wl = pipe.api, pipe.wl
    dev = pipe.dev
    budget, floor = wl.Hkv * wl.k, budget_floor(wl)
    idx = torch.empty(wl.rows, budget, dtype=torch.int32, device=dev)
    off = torch.empty(wl.rows, wl.Hkv + 1, dtype=torch.int32, device=dev)
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    cap = budget - (wl.Hkv - 1) * floor  # the most one head can keep
    dt = pipe.K.dtype
    Kc = torch.empty(wl.rows, wl.Hkv, cap, wl.d, dtype=dt, device=dev)
    Vc = torch.empty_like(Kc)
    pos = torch.empty(wl.rows, wl.Hkv, cap, dtype=torch.int32, device=dev)
    acc = torch.empty(wl.rows, wl.Hkv, cap, dtype=torch.float32, device=dev)
    ln = torch.empty(wl.rows, wl.Hkv, dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)

    def sel():
        a.kv_select_budget(pipe.z, budget, floor, wl.R, 0, idx_out=idx, off_out=off)

    def comp():
        a.kv_compact_ragged(pipe.K, pipe.V, pipe.s, idx, off, cap, K_out=Kc, V_out=Vc, pos_out=pos,
                            acc_out=acc, len_out=ln, dev_status=status)

    def timed(fn):
        for _ in range(warmup):
            fn()
        ts = []
        for _ in range(reps):
            flush.fill_(1.0)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
        return statistics.median(ts)

    out = {}
    peak, _, kind = measured_peaks()
    if wl.r is not None:  # the refined scores the layer budget ranks (not kept by the step)
        a.hubkv_refine(pipe.s, wl.r, wl.gamma, wl.pool_width, wl.beta_lo, wl.beta_hi, out=pipe.z,
                       workspace=pipe.ws)
    ms = timed(sel)
    counts = (off[:, 1:] - off[:, :-1])
    nbytes = wl.units * wl.T * 4 + wl.rows * (budget + wl.Hkv + 1) * 4
    gbs = nbytes / (ms / 1e3) / 1e9
    out["kv_select_budget"] = {"ms": ms, "budget_per_layer": budget, "floor": floor,
                               "algorithmic_bytes": nbytes, "achieved_gbs": gbs,
                               "frac": gbs / peak, "peak_kind": kind,
                               "per_head_kept": {"min": int(counts.min()), "max": int(counts.max())}}
    ms = timed(comp)
    if int(status.item()) != 0:
        raise RuntimeError("ragged compaction reported a device status")
    row = wl.d * pipe.K.element_size()
    nbytes = wl.rows * budget * (4 * row + 4 + 4 + 4 + 4) + wl.rows * (wl.Hkv + 1) * 4
    gbs = nbytes / (ms / 1e3) / 1e9
    out["kv_compact_ragged"] = {"ms": ms, "cap": cap, "algorithmic_bytes": nbytes,
                                "achieved_gbs": gbs, "frac": gbs / peak, "peak_kind": kind}
    # NestedKV key-only scoring of the same keys
    n_disc = -(-wl.T // 10)
    nscore = torch.empty(wl.rows, wl.Hkv, wl.T, dtype=torch.float32, device=dev)
    nw = torch.empty(wl.rows, wl.Hkv, 3, dtype=torch.float32, device=dev)
    nws = torch.empty(a.kv_workspace_size(a.KV_OP_SCORE_NESTED, wl.rows, 0, wl.Hkv, wl.T, wl.d, 32),
                      dtype=torch.uint8, device=dev)
    launches0 = launch_count()
    ms = timed(lambda: a.kv_score_nested(pipe.K, n_disc, NESTED_THRESH, (0.0, 0.0, 0.0), 64, 32,
                                         out=nscore, w_out=nw, workspace=nws))
    per_call = (launch_count() - launches0) // (warmup + reps)
    k_bytes = wl.units * wl.T * wl.d * pipe.K.element_size()
    nbytes = nested_bytes(wl)
    gbs = nbytes / (ms / 1e3) / 1e9
    out["kv_score_nested"] = {"ms": ms, "window": 64, "n_blocks": 32, "n_disc": n_disc,
                              "surprise_thresh": NESTED_THRESH, "launches": per_call,
                              "algorithmic_bytes": nbytes, "k_bytes": k_bytes,
                              "achieved_gbs": gbs, "frac": gbs / peak, "peak_kind": kind,
                              "tokens_per_s": wl.units * wl.T / (ms / 1e3)}
    return out


OTHER_WORKLOADS = ("llama2-7b-layer", "h2o-decode", "gqa-prefill")


def time_workload(name, reps=5, clocks=None):
    """One of the pages' other workloads on its own buffers, outside the timed step:
    the prefill chain (and the decode steps, where the workload has them) captured
    as CUDA graphs and replayed, each replay timed with events on the launching
    stream; L2 is flushed before every replay when the workload's keys fit in it.
    Per-phase times come from one eager pass with events between the phases."""
    import torch
    from kv_cache_compression_obs_gb300 import configs

    wl = configs.BY_NAME[name]
    dev = torch.device("cuda", torch.cuda.current_device())
    pipe = Pipeline(wl, dev)
    for _ in range(3):
        pipe.step()
    torch.cuda.synchronize()
    pipe.capture()
    phases = pipe.timed_phases()
    gp, gd = pipe.graphs
    k_bytes = wl.units * wl.T * wl.d * wl.elem_bytes
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev) if k_bytes < L2_BYTES else None
    tp, td = [], []
    for _ in range(reps + 1):  # the first replay is untimed
        if flush is not None:
            flush.fill_(1.0)
        e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        e[0].record()
        gp.replay()
        e[1].record()
        if gd is not None:
            gd.replay()
        e[2].record()
        torch.cuda.synchronize()
        tp.append(e[0].elapsed_time(e[1]))
        td.append(e[1].elapsed_time(e[2]))
    tp, td = tp[1:], td[1:]
    peak, peak_tf, kind = measured_peaks()
    alg = algorithmic_bytes(wl)
    names = ("kv_score_obs", "hubkv_select_topk", "kv_compact")
    pre_bytes = sum(alg[n] for n in names)
    ms = statistics.median(tp)
    score_s = phases["kv_score_obs"] / 1e3
    out = {"workload": wl.name, "units": wl.units, "prompt": wl.T, "obs_window": wl.W,
           "budget_k": wl.k, "recent": wl.R, "hubkv": wl.r is not None,
           "l2": "flushed before every replay" if flush is not None else "inputs larger than L2",
           "prefill": {"ms": ms, "kv_tokens_per_s": wl.rows * wl.T / (ms / 1e3),
                       "head_tokens_per_s": wl.units * wl.T / (ms / 1e3),
                       "algorithmic_bytes": pre_bytes,
                       "hbm_frac": pre_bytes / (ms / 1e3) / 1e9 / peak, "peak_kind": kind,
                       "graph": "a1-a4 replayed as one CUDA graph"},
           "phases_ms_eager": phases,
           "score": {"ms": phases["kv_score_obs"], "algorithmic_flops": score_flops(wl),
                     "tflops": score_flops(wl) / score_s / 1e12,
                     "tensor_frac": score_flops(wl) / score_s / 1e12 / peak_tf,
                     "hbm_frac": alg["kv_score_obs"] / score_s / 1e9 / peak}}
    sfu = sfu_fraction(wl, score_s, clocks or {},
                       torch.cuda.get_device_properties(0).multi_processor_count)
    if sfu:
        out["score"]["sfu_frac"] = sfu["sfu_frac"]
        out["score"]["sfu_executed_frac"] = sfu["sfu_executed_frac"]
    if wl.n_decode:
        step_ms = statistics.median(td) / wl.n_decode
        out["decode"] = {"steps": wl.n_decode, "ms_per_step": step_ms,
                         "steps_per_s": 1e3 / step_ms,
                         "algorithmic_bytes_per_step": alg["h2o_decode_step"],
                         "hbm_frac": alg["h2o_decode_step"] / (step_ms / 1e3) / 1e9 / peak,
                         "cap": wl.cap, "kv_heads": wl.units, "group": wl.G}
    del pipe, flush
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return out


def launch_count():
    from kv_cache_compression_obs_gb300 import api
    return int(api.library_handle().kv_launch_count())


E2E_GROUPS = 4  # layer-row groups of the end-to-end path (decode of one overlaps the next's keys)


def run_e2e(wl, pipe, steps, n_groups):
    """Same metric through the public API from pinned host inputs, copies inside the
    timed region.  Layer rows are independent through the whole path, so they run
    in n_groups groups: compress_prefill_host streams a group's Q and K to the
    device one layer row at a time on a copy stream (the compaction gathers the
    kept V rows straight from host memory), then the group's decode steps run as
    one h2o_decode_steps call while the next group's keys stream.  The kept
    positions and every decode step's evictions and attention outputs are copied
    back."""
    import torch
    a = pipe.api
    groups = [(g * wl.rows // n_groups, (g + 1) * wl.rows // n_groups) for g in range(n_groups)]
    groups = [gr for gr in groups if gr[1] > gr[0]]
    hQ = pipe.Q.cpu().pin_memory()
    hK = pipe.K.cpu().pin_memory()
    hV = pipe.V.cpu().pin_memory()
    # decode inputs held group-major on the host, so that each group's are contiguous
    hD = [[X[:, r0:r1].contiguous().cpu().pin_memory() for X in (pipe.DQ, pipe.DK, pipe.DV)]
          for r0, r1 in groups] if wl.n_decode else []
    dD = [[torch.empty_like(h, device=pipe.dev) for h in hg] for hg in hD]
    dO = [torch.empty(wl.n_decode, r1 - r0, wl.Hq, wl.d, dtype=torch.float32, device=pipe.dev)
          for r0, r1 in groups]
    dE = [torch.empty(wl.n_decode, r1 - r0, wl.Hkv, dtype=torch.int32, device=pipe.dev)
          for r0, r1 in groups]
    out_idx = torch.empty(pipe.idx.shape, dtype=torch.int32).pin_memory()
    out_o = [torch.empty(o.shape, dtype=torch.float32).pin_memory() for o in dO]  # every step's
    out_ev = [torch.empty(e.shape, dtype=torch.int32).pin_memory() for e in dE]
    bufs = {"Q": pipe.Q, "K": pipe.K, "s": pipe.s, "z": pipe.z, "beta": pipe.beta, "idx": pipe.idx,
            "Kc": pipe.Kc, "Vc": pipe.Vc, "pos": pipe.pos, "acc": pipe.acc, "len": pipe.len,
            "ws": pipe.ws, "copy_stream": torch.cuda.Stream(), "rows_per_chunk": 1, "cap": wl.cap}
    row = wl.d * wl.elem_bytes
    h2d = (hQ.numel() * hQ.element_size() + hK.numel() * hK.element_size()
           + wl.units * wl.k * row  # the kept V rows, gathered from host memory
           + sum(h.numel() * h.element_size() for hg in hD for h in hg))
    d2h = out_idx.numel() * 4 + sum(o.numel() * 4 for o in out_o) + sum(e.numel() * 4 for e in out_ev)

    def one():
        for dg, hg in zip(dD, hD):  # decode inputs first: small
            for d_, h_ in zip(dg, hg):
                d_.copy_(h_, non_blocking=True)
        for gi, (r0, r1) in enumerate(groups):
            a.compress_prefill_host(hQ, hK, hV, wl.k, wl.R, wl.r, wl.gamma, wl.pool_width,
                                    wl.beta_lo, wl.beta_hi, wl.scale, buffers=bufs, rows=(r0, r1),
                                    wait=(gi == 0))
            out_idx[r0:r1].copy_(pipe.idx[r0:r1], non_blocking=True)
            if wl.n_decode:
                sl = slice(r0, r1)
                a.h2o_decode_steps(*dD[gi], pipe.Kc[sl], pipe.Vc[sl], pipe.pos[sl], pipe.acc[sl],
                                   pipe.len[sl], wl.R, wl.T, wl.scale, o_out=dO[gi],
                                   evicted_out=dE[gi], workspace=pipe.dws)
                out_ev[gi].copy_(dE[gi], non_blocking=True)
                out_o[gi].copy_(dO[gi], non_blocking=True)

    one()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(steps):
        one()
    torch.cuda.synchronize()
    dt = (time.perf_counter() - t0) / steps
    return dt, h2d, d2h


def host_cpu_model():
    """The host CPU's model name (lscpu / /proc/cpuinfo), or the machine type."""
    import platform
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu part")):
                    return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return platform.machine()


def cpu_baseline(wl, pipe, budget_s=20.0):
    """The float64 oracle as it stands, on one batch row of the workload, on the host cores."""
    import numpy as np

    import oracle
    from kv_cache_compression_obs_gb300 import gen

    cores = os.cpu_count() or 1
    row = slice(0, 1)
    Qh = gen.to_numpy_bits(pipe.Q[row])
    Kh = gen.to_numpy_bits(pipe.K[row])
    Vh = gen.to_numpy_bits(pipe.V[row])
    t0 = time.perf_counter()
    s = oracle.score_obs(Qh, Kh, wl.scale)
    z = oracle.hubkv_refine(s, wl.r, wl.gamma, wl.pool_width, wl.beta_lo, wl.beta_hi)[0] \
        if wl.r is not None else s
    idx = oracle.select_topk(z, wl.k, wl.R)
    Kc, Vc, pos, acc, ln = oracle.compact(Kh, Vh, s, idx, wl.cap)
    t_prefill = time.perf_counter() - t0
    n_dec = 0
    t1 = time.perf_counter()
    for t in range(wl.n_decode):
        if time.perf_counter() - t0 > budget_s:
            break
        q, kn, vn = (gen.to_numpy_bits(x[row]) for x in (pipe.dq[t], pipe.dk[t], pipe.dv[t]))
        oracle.decode_step(q, kn, vn, Kc, Vc, pos, acc, ln, wl.R, wl.T + t, wl.scale)
        n_dec += 1
    t_dec = time.perf_counter() - t1
    per_step_dec = t_dec / max(n_dec, 1)
    # a whole step for this row: prefill + all decode steps (decode time extrapolated per step)
    t_row = t_prefill + per_step_dec * wl.n_decode
    tokens = 1 * wl.T
    return {"value": tokens / t_row, "unit": UNIT, "cores": int(os.environ.get("OMP_NUM_THREADS", cores)),
            "cpu": host_cpu_model(), "kind": "oracle",
            "sample": (f"batch row 0 of {wl.rows} ({wl.Hkv} KV heads, T={wl.T}): score+refine+Top-K+"
                       f"compact in {t_prefill:.2f} s, {n_dec} of {wl.n_decode} decode steps timed "
                       f"({per_step_dec * 1e3:.1f} ms each)"),
            "decode_steps_per_s": 1.0 / per_step_dec if n_dec else None}


def oracle_single_thread(names=("tiny", "llama2-7b-layer")):
    """The oracle's prefill chain (score, refine, Top-K, compaction) on one OpenMP
    thread, on the small workloads' first batch row: seconds per call and KV
    tokens/s, beside the multi-core baseline."""
    import ctypes

    import oracle
    from kv_cache_compression_obs_gb300 import configs, gen

    try:
        gomp = ctypes.CDLL("libgomp.so.1")
    except OSError:
        return None
    before = gomp.omp_get_max_threads()
    out = {}
    try:
        gomp.omp_set_num_threads(1)
        for nm in names:
            wl = configs.BY_NAME[nm]
            Q, K, V = gen.prefill_inputs(wl, units=list(range(wl.Hkv)))
            Qh, Kh, Vh = (gen.to_numpy_bits(x) for x in (Q, K, V))
            Qh = Qh.reshape(1, wl.Hq, wl.W, wl.d)
            Kh, Vh = Kh.reshape(1, wl.Hkv, wl.T, wl.d), Vh.reshape(1, wl.Hkv, wl.T, wl.d)
            t0 = time.perf_counter()
            s = oracle.score_obs(Qh, Kh, wl.scale)
            z = oracle.hubkv_refine(s, wl.r, wl.gamma, wl.pool_width, wl.beta_lo, wl.beta_hi)[0] \
                if wl.r is not None else s
            idx = oracle.select_topk(z, wl.k, wl.R)
            oracle.compact(Kh, Vh, s, idx, wl.cap)
            dt = time.perf_counter() - t0
            out[nm] = {"s": dt, "kv_tokens_per_s": wl.T / dt, "threads": 1}
    finally:
        gomp.omp_set_num_threads(before)
    return out


def max_over_ranks(x: float, world: int, device) -> float:
    """The largest of every rank's x: the job is as slow as its slowest rank."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: float, world: int, seconds: float) -> float:
    """Units all ranks processed (each rank runs its own full workload) per second
    of the slowest rank."""
    return world * units_per_rank / seconds


def run_ours(args, wl, rank, world):
    import torch
    import torch.distributed as dist

    local = _env_int("LOCAL_RANK", 0)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pipe = Pipeline(wl, dev)
    torch.cuda.synchronize()
    for _ in range(max(args.warmup, 0)):
        pipe.step()
    torch.cuda.synchronize()
    if not args.eager:
        pipe.capture()
        for _ in range(2):  # the graphs' own first replays, untimed
            pipe.step()
        torch.cuda.synchronize()
    phases = pipe.timed_phases()

    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    launches0 = launch_count()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        e0.record()
        for _ in range(args.steps):
            pipe.step()
        e1.record()
        torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    launches = launch_count() - launches0
    if pipe.graphs is not None:  # replays count no launches on the host: the captured ones, per step
        launches = pipe.launches_per_step * args.steps
    ms = e0.elapsed_time(e1) / args.steps
    ms_max = max_over_ranks(ms, world, dev)

    tokens = wl.rows * wl.T
    value = whole_job_rate(tokens, world, ms_max / 1e3)
    PREFILL = ("kv_score_obs", "hubkv_select_topk", "kv_compact")
    prefill_ms = sum(phases[n] for n in PREFILL)
    peak, peak_tf, peak_kind = measured_peaks()
    alg = algorithmic_bytes(wl)
    prefill_bytes = sum(alg[n] for n in PREFILL)
    per_launch = {k: alg[k] for k in alg}
    dom = max(phases, key=lambda n: phases[n] * (wl.n_decode if n == "h2o_decode_step" else 1))
    achieved = per_launch[dom] / (phases[dom] / 1e3) / 1e9
    traffic, traffic_source = None, None
    if dom == "h2o_decode_step" and wl.name in DECODE_TRAFFIC_PER_UNIT:
        if _source_sha256(DECODE_TRAFFIC_SOURCE) == DECODE_TRAFFIC_SOURCE_SHA256:
            traffic = round(DECODE_TRAFFIC_PER_UNIT[wl.name] * wl.units)
            traffic_source = ("ncu dram__bytes_read.sum + dram__bytes_write.sum of the decode "
                              "launches, taken on this decode source (sha256 "
                              f"{DECODE_TRAFFIC_SOURCE_SHA256[:12]})")
        else:
            traffic_source = "stale: the decode source changed since the ncu capture"
    score_s = phases["kv_score_obs"] / 1e3
    score_tf = score_flops(wl) / score_s / 1e12
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": wl.dtype, "data": "synthetic",
        "config": {"workload": wl.name, "batch": wl.B, "layers": wl.L, "q_heads": wl.Hq,
                   "kv_heads": wl.Hkv, "d_head": wl.d, "prompt": wl.T, "obs_window": wl.W,
                   "budget_k": wl.k, "recent": wl.R, "r": wl.r, "gamma": wl.gamma,
                   "decode_steps": wl.n_decode, "parallelism": f"replica x{world}",
                   "l2": f"inputs larger than L2 (K+V {2 * wl.units * wl.T * wl.d * wl.elem_bytes / 1e9:.1f} GB)"},
        "prefill": {"ms": prefill_ms, "tokens_per_s": whole_job_rate(tokens, world, prefill_ms / 1e3),
                    "head_tokens_per_s": whole_job_rate(tokens * wl.Hkv, world, prefill_ms / 1e3),
                    "algorithmic_bytes": prefill_bytes,
                    "hbm_frac": prefill_bytes / (prefill_ms / 1e3) / 1e9 / peak,
                    "note": "score + refine + Top-K + compaction (one phase-timed step); the "
                            "scoring share is bound by its two MMA + exp passes, see roofline_score"},
        "decode": {"steps_per_s": (1e3 / phases["h2o_decode_step"]) if wl.n_decode else None,
                   "ms_per_decode_step": phases["h2o_decode_step"] if wl.n_decode else None},
        "phases_ms": phases,
        "gpu_launches": launches,
        "roofline": {"kernel": dom, "bound": "hbm", "achieved": achieved, "peak": peak,
                     "peak_kind": peak_kind, "unit": "GB/s", "frac": achieved / peak,
                     "algorithmic_bytes": per_launch[dom], "traffic": traffic,
                     "traffic_source": traffic_source,
                     "note": ("one decode step = its stream and finalize launches (two row halves on two streams), timed together"
                              if dom == "h2o_decode_step" else None)},
        "roofline_score": {"kernel": "kv_score_obs", "bound": "tensor", "achieved": score_tf,
                           "peak": peak_tf, "peak_kind": peak_kind + " bf16 dense (burst)",
                           "unit": "TFLOP/s", "frac": score_tf / peak_tf,
                           "algorithmic_flops": score_flops(wl),
                           "executed_flops": score_flops_executed(wl),
                           "executed_frac": score_flops_executed(wl) / score_s / 1e12 / peak_tf,
                           "hbm_gbs": per_launch["kv_score_obs"] / score_s / 1e9,
                           "hbm_frac": per_launch["kv_score_obs"] / score_s / 1e9 / peak,
                           "note": "algorithmic = one Q K^T over the causally visible pairs; "
                                   "executed = both passes (statistics, column mass)"},
        "clocks": clk.summary(),
    }
    line["roofline_score"].update(sfu_fraction(
        wl, score_s, line["clocks"], torch.cuda.get_device_properties(dev).multi_processor_count))
    if not args.no_next_rows:
        line["next_rows"] = time_next_rows(pipe)
    if not args.no_other_workloads and world == 1:
        # the pages' other workloads, each on its own buffers (about 20 GB beside the
        # headline workload's, far below the GPU's memory)
        line["other_workloads"] = {nm: time_workload(nm, clocks=line["clocks"]) for nm in OTHER_WORKLOADS
                                   if nm != wl.name}
    if not args.no_e2e:
        if world > 1:
            dist.barrier()
        dt, h2d, d2h = run_e2e(wl, pipe, min(args.steps, 3), args.e2e_groups or E2E_GROUPS)
        dt = max_over_ranks(dt, world, dev)
        line["e2e"] = {"value": whole_job_rate(tokens, world, dt), "unit": UNIT,
                       "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, pipe)
        st = oracle_single_thread()
        if st:
            line["cpu_baseline"]["single_thread_prefill"] = st
    return line


def run_reference(args, wl):
    """The oracle as the reference arm: a bounded sample per step on the host cores."""
    import torch

    from kv_cache_compression_obs_gb300 import gen

    class HostPipe:
        pass

    p = HostPipe()
    p.Q, p.K, p.V = gen.prefill_inputs(wl.scaled(B=1, L=1), device="cpu")
    steps_in = [gen.decode_inputs(wl.scaled(B=1, L=1), t, device="cpu") for t in range(wl.n_decode)]
    p.dq = [x[0] for x in steps_in]
    p.dk = [x[1] for x in steps_in]
    p.dv = [x[2] for x in steps_in]
    for _ in range(max(args.warmup, 0)):
        cpu_baseline(wl.scaled(B=1, L=1), p, budget_s=0.0)
    vals = []
    t0 = time.perf_counter()
    for _ in range(args.steps):
        vals.append(cpu_baseline(wl.scaled(B=1, L=1), p, budget_s=10.0))
    dt = time.perf_counter() - t0
    v = statistics.median(x["value"] for x in vals)
    cb = dict(vals[-1])
    cb["value"] = v
    return {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": wl.name, "batch": wl.B, "layers": wl.L, "q_heads": wl.Hq,
                       "kv_heads": wl.Hkv, "d_head": wl.d, "prompt": wl.T, "obs_window": wl.W,
                       "budget_k": wl.k, "recent": wl.R, "decode_steps": wl.n_decode},
            "cpu_baseline": cb,
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    args = parse()
    from kv_cache_compression_obs_gb300 import configs

    wl = configs.BY_NAME[args.config]
    if args.layers is not None:
        wl = wl.scaled(L=args.layers)
    rank, world = _env_int("RANK", 0), _env_int("WORLD_SIZE", 1)
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, wl)), flush=True)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(_env_int("LOCAL_RANK", 0))
        dist.init_process_group("nccl")
    line = run_ours(args, wl, rank, world)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
