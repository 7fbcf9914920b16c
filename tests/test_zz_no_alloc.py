"""kv_score_obs_noalloc: scoring for callers that cannot allocate device memory.

Some callers of this library are handed only their input and output buffers by
a host framework, or must not call cudaMalloc because it can synchronise the
device; they cannot provide kv_score_obs's scratch workspace.  The no-alloc
entry point takes its scratch from a fixed array inside the library instead.
This test calls it through the C ABI and checks, on two calls in a row with
different shapes (so the second call runs on the first call's leftovers), that
it returns bit for bit what kv_score_obs returns (both run the same kernels with
the same plan), and that a device status word passed to it stays 0.  The file
is named so that pytest collects it last: a failure in the shared-array path
then cannot stop a run with -x before every other test has run.
"""
import ctypes

import pytest
import torch

from kv_cache_compression_obs_gb300 import gen
from kv_cache_compression_obs_gb300.configs import Workload

pytestmark = pytest.mark.gpu


def _c_noalloc(lib, Q, K, s, scale, status=None):
    fn = lib.kv_score_obs_noalloc
    P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    fn.restype = I
    fn.argtypes = [P, P, I, I, I, I, I, I, F, I, P, P, P]
    B, Hq, W, d = Q.shape
    _, Hkv, T, _ = K.shape
    dt = 0 if K.dtype == torch.bfloat16 else 1
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return fn(ctypes.c_void_p(Q.data_ptr()), ctypes.c_void_p(K.data_ptr()), B, Hq, Hkv, T, d, W,
              float(scale), dt, ctypes.c_void_p(s.data_ptr()),
              None if status is None else ctypes.c_void_p(status.data_ptr()), stream)


WORKLOADS = [
    Workload("noalloc-a", B=2, L=1, Hq=8, Hkv=2, d=128, T=3000, W=64, dtype="bf16", r=0.1, k=300,
             R=64, n_decode=0, seed=41, keys="segments", n_segments=20),
    Workload("noalloc-b", B=1, L=1, Hq=4, Hkv=4, d=64, T=777, W=16, dtype="f32", r=0.2, k=100,
             R=20, n_decode=0, seed=42, keys="sinks", n_sinks=4),
]


def test_noalloc_matches_workspace_entry_point(kvc):
    lib = kvc.library_handle()
    for i, wl in enumerate(WORKLOADS):  # two calls in a row, different shapes and dtypes
        Q, K, _ = gen.prefill_inputs(wl, device="cuda")
        ref = kvc.kv_score_obs(Q, K)
        s = torch.full_like(ref, float("nan"))
        status = torch.zeros(1, dtype=torch.int32, device="cuda") if i == 0 else None
        assert _c_noalloc(lib, Q, K, s, wl.scale, status) == kvc.KV_OK
        torch.cuda.synchronize()
        assert torch.equal(s, ref), f"noalloc vs workspace ({wl.name}): bits differ"
        if status is not None:
            assert int(status.item()) == 0  # no device-side wait gave up


def test_noalloc_rejects_shapes_beyond_its_scratch(kvc):
    lib = kvc.library_handle()
    # full-prompt scoring (every prompt query observed) of 8 x 32 heads x 8192
    # tokens needs more scratch than the fixed array holds
    B, H, T, d = 8, 32, 8192, 128
    need = kvc.kv_workspace_size(kvc.KV_OP_SCORE_OBS, B, H, H, T, d, T)
    assert need > (16 << 20)
    Q = torch.zeros(B, H, T, d, dtype=torch.bfloat16, device="cuda")
    s = torch.zeros(B, H, T, device="cuda")
    assert _c_noalloc(lib, Q, Q, s, 0.1) == kvc.KV_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.all(s == 0)  # nothing was launched
