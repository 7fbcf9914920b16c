"""The five synthetic workloads the eviction path is measured and checked on.

Shapes follow the pages' workloads: Llama-2-7B-like heads (d_head = 128, 32
heads; KV-cache blog §1.3), GQA-8 (32 query / 8 KV heads; blog §3.3), 4K-128K
prompts and 5-20% budgets (H2O page, 精度 section: 20% budget).  Layers are
independent and are folded into the batch dimension: a workload with B batch
rows and L layers runs as B*L rows.

Budget readings: k = floor(budget * T); "x% heavy + y% recent" gives
R = floor(y * T); "split heavy/recent" gives R = floor(k / 2) (H2O page,
双缓冲: half each); "incl. N recent" gives R = N; the GQA prefill workload has
no stated window and uses R = W = 64.
"""
from __future__ import annotations

from dataclasses import dataclass, replace


@dataclass(frozen=True)
class Workload:
    name: str
    B: int            # batch rows
    L: int            # layers, folded into the batch: rows = B * L
    Hq: int           # query heads
    Hkv: int          # KV heads
    d: int            # head dimension
    T: int            # prompt length
    W: int            # observation window (queries = last W prompt positions)
    dtype: str        # "f32" or "bf16"
    r: float | None   # HubKV compression ratio; None = no refinement step
    k: int            # budget (kept slots per KV head)
    R: int            # protected recent window
    n_decode: int     # H2O decode steps after compaction
    seed: int
    keys: str         # key recipe: "sinks", "segments", "zipf"
    n_segments: int = 0
    n_sinks: int = 0
    gamma: float = 0.5
    pool_width: int = 5
    beta_lo: float = 0.8
    beta_hi: float = 1.2

    @property
    def rows(self) -> int:
        return self.B * self.L

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def units(self) -> int:
        return self.rows * self.Hkv

    @property
    def cap(self) -> int:
        return self.k

    @property
    def scale(self) -> float:
        return self.d ** -0.5

    @property
    def elem_bytes(self) -> int:
        return 2 if self.dtype == "bf16" else 4

    def scaled(self, **kw) -> "Workload":
        """A smaller variant with the same recipe (for parity tests)."""
        return replace(self, **kw)


TINY = Workload("tiny", B=1, L=1, Hq=4, Hkv=4, d=64, T=512, W=16, dtype="f32", r=0.2,
                k=102, R=51, n_decode=64, seed=1, keys="sinks", n_sinks=4)
LLAMA2_LAYER = Workload("llama2-7b-layer", B=1, L=1, Hq=32, Hkv=32, d=128, T=4096, W=32,
                        dtype="bf16", r=0.1, k=409, R=32, n_decode=0, seed=2,
                        keys="segments", n_segments=40)
H2O_DECODE = Workload("h2o-decode", B=8, L=1, Hq=32, Hkv=32, d=128, T=8192, W=8192,
                      dtype="bf16", r=None, k=1638, R=819, n_decode=256, seed=3, keys="zipf")
GQA_PREFILL = Workload("gqa-prefill", B=4, L=32, Hq=32, Hkv=8, d=128, T=32768, W=64,
                       dtype="bf16", r=0.1, k=3276, R=64, n_decode=0, seed=4,
                       keys="segments", n_segments=200)
LONG_CONTEXT = Workload("long-context", B=1, L=32, Hq=32, Hkv=8, d=128, T=131072, W=64,
                        dtype="bf16", r=0.05, k=6553, R=64, n_decode=128, seed=5,
                        keys="segments", n_segments=1000, n_sinks=4)

ALL = [TINY, LLAMA2_LAYER, H2O_DECODE, GQA_PREFILL, LONG_CONTEXT]
BY_NAME = {w.name: w for w in ALL}
