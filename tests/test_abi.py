"""The C ABI without a GPU: the library loads, exports every declared symbol, and
rejects bad arguments on the host before touching CUDA."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kvc.h")


@pytest.fixture(scope="module")
def lib():
    from kv_cache_compression_obs_gb300.build import build
    path = build()
    lib = ctypes.CDLL(path)
    P, I, F, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.kv_score_obs.argtypes = [P, P, I, I, I, I, I, I, F, I, P, P, Z, P, P]
    lib.hubkv_refine.argtypes = [P, I, I, I, I, F, F, F, F, P, P, P, Z, P]
    lib.kv_select_topk.argtypes = [P, I, I, I, I, I, P, P, Z, P]
    lib.kv_compact.argtypes = [P, P, P, P, I, I, I, I, I, I, P, P, I, P, P, P, P]
    lib.h2o_decode_step.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, F, I, I, P, P, P, Z, P,
                                    P]
    lib.kv_workspace_size.restype = Z
    lib.kv_workspace_size.argtypes = [I, I, I, I, I, I, I, I]
    lib.kv_status_string.restype = ctypes.c_char_p
    lib.kv_last_error_detail.restype = ctypes.c_char_p
    lib.hubkv_refine_ex.argtypes = [P, I, I, I, I, F, F, F, F, I, P, P, P, Z, P]
    lib.kv_select_topk_ex.argtypes = [P, I, I, I, I, I, I, P, P, Z, P]
    lib.h2o_decode_step_ex.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, I, F, I, I, P, P,
                                       P, Z, P, P]
    lib.kv_select_budget.argtypes = [P, I, I, I, I, I, I, I, P, P, P]
    lib.kv_score_nested.argtypes = [P, I, I, I, I, I, I, I, I, F, F, F, F, P, P, P, P, Z, P]
    lib.h2o_decode_steps.argtypes = [P, P, P, I, P, P, P, P, P, I, I, I, I, I, I, I, I, F, I, I, P, P,
                                     P, Z, P, P]
    lib.kv_compact_ragged.argtypes = [P, P, P, P, P, I, I, I, I, I, I, P, P, I, P, P, P, P, P]
    lib.hubkv_select_topk.argtypes = [P, I, I, I, I, F, F, F, F, I, I, I, I, P, P, P, P, Z, P]
    return lib


def declared_functions():
    text = open(HEADER).read()
    return re.findall(r"KVC_API\s+[\w\s\*]+?\b(\w+)\s*\(", text)


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert set(names) >= {"kv_score_obs", "hubkv_refine", "kv_select_topk", "kv_compact",
                          "h2o_decode_step", "kv_workspace_size", "kv_status_string", "kv_version"}
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings_and_version(lib):
    assert lib.kv_status_string(0) == b"ok"
    assert b"invalid" in lib.kv_status_string(-1)
    assert lib.kv_status_string(-4) == b"device-side wait timed out"
    assert lib.kv_version() >= 100


def test_error_detail_is_empty_before_any_cuda_failure(lib):
    assert lib.kv_last_error_detail() == b""


def test_workspace_size(lib):
    assert lib.kv_workspace_size(1, 4, 32, 8, 32768, 128, 64, 3276) > 0
    assert lib.kv_workspace_size(1, 1, 32, 8, 100, 128, 101, 1) == 0   # W > T: invalid
    assert lib.kv_workspace_size(2, 4, 8, 8, 32768, 128, 64, 0) > 0
    assert lib.kv_workspace_size(3, 4, 8, 8, 32768, 128, 64, 100) == 0
    assert lib.kv_workspace_size(99, 4, 8, 8, 32768, 128, 64, 100) == 0
    assert lib.kv_workspace_size(4, 1, 32, 8, 6553, 128, 0, 0) > 32 * 6554 * 4


NULL = None


def test_host_validation_rejects_before_cuda(lib):
    # score: W > T, Hq % Hkv, d unsupported, null pointers
    assert lib.kv_score_obs(NULL, NULL, 1, 4, 2, 10, 64, 11, 0.1, 0, NULL, NULL, 0, NULL, NULL) == -1
    assert lib.kv_score_obs(NULL, NULL, 1, 3, 2, 10, 64, 4, 0.1, 0, NULL, NULL, 0, NULL, NULL) == -1
    assert lib.kv_score_obs(NULL, NULL, 1, 4, 2, 10, 96, 4, 0.1, 0, NULL, NULL, 0, NULL, NULL) == -2
    assert lib.kv_score_obs(NULL, NULL, 1, 4, 2, 10, 64, 4, 0.1, 7, NULL, NULL, 0, NULL, NULL) == -1
    assert lib.kv_score_obs(NULL, NULL, 1, 4, 2, 10, 64, 4, 0.1, 0, NULL, NULL, 0, NULL, NULL) == -1
    # refine: even pool width, bad clip range
    assert lib.hubkv_refine(NULL, 1, 2, 10, 4, 0.5, 0.1, 0.8, 1.2, NULL, NULL, NULL, 0, NULL) == -1
    assert lib.hubkv_refine(NULL, 1, 2, 10, 5, 0.5, 0.1, 1.3, 1.2, NULL, NULL, NULL, 0, NULL) == -1
    # select: k <= recent, k > T
    assert lib.kv_select_topk(NULL, 1, 2, 10, 3, 3, NULL, NULL, 0, NULL) == -1
    assert lib.kv_select_topk(NULL, 1, 2, 10, 11, 3, NULL, NULL, 0, NULL) == -1
    # compact: cap < k
    assert lib.kv_compact(NULL, NULL, NULL, NULL, 1, 2, 10, 5, 64, 0, NULL, NULL, 4, NULL, NULL,
                          NULL, NULL) == -1
    # decode: ALG1 with a recent window, recent >= cap, unsupported group size
    assert lib.h2o_decode_step(NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, 1, 4, 4, 8, 64, 1, 9,
                               0.1, 1, 0, NULL, NULL, NULL, 0, NULL, NULL) == -1
    assert lib.h2o_decode_step(NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, 1, 4, 4, 8, 64, 8, 9,
                               0.1, 0, 0, NULL, NULL, NULL, 0, NULL, NULL) == -1
    p = ctypes.c_void_p(16)  # a dummy aligned pointer: never dereferenced, the call is rejected first
    assert lib.h2o_decode_step(p, p, p, p, p, p, p, p, 1, 12, 4, 8, 64, 1, 9, 0.1, 0, 0, p, p, NULL,
                               0, NULL, NULL) == -2


def test_extended_entry_points_validate_on_the_host(lib):
    # refine: an unknown variant flag
    assert lib.hubkv_refine_ex(NULL, 1, 2, 10, 5, 0.5, 0.1, 0.8, 1.2, 4, NULL, NULL, NULL, 0, NULL) == -1
    # select: negative sink, sinks + recent filling the budget
    assert lib.kv_select_topk_ex(NULL, 1, 2, 10, 5, 1, -1, NULL, NULL, 0, NULL) == -1
    assert lib.kv_select_topk_ex(NULL, 1, 2, 10, 5, 2, 3, NULL, NULL, 0, NULL) == -1
    # decode: negative sink
    assert lib.h2o_decode_step_ex(NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, 1, 4, 4, 8, 64, 1, -1,
                                  9, 0.1, 0, 0, NULL, NULL, NULL, 0, NULL, NULL) == -1
    # empty batches are no-ops
    assert lib.hubkv_refine_ex(NULL, 0, 2, 10, 5, 0.5, 0.1, 0.8, 1.2, 3, NULL, NULL, NULL, 0, NULL) == 0
    assert lib.kv_select_topk_ex(NULL, 0, 2, 10, 5, 1, 2, NULL, NULL, 0, NULL) == 0


def test_fused_refine_select_validates_on_the_host(lib):
    sel = lambda B, T, pw, flags, k, R, S, ws=0: lib.hubkv_select_topk(  # noqa: E731
        NULL, B, 2, T, pw, 0.5, 0.1, 0.8, 1.2, flags, k, R, S, NULL, NULL, NULL, NULL, ws, NULL)
    assert sel(1, 10, 4, 0, 5, 1, 0) == -1     # even pool width
    assert sel(1, 10, 5, 4, 5, 1, 0) == -1     # unknown variant flag
    assert sel(1, 10, 5, 0, 5, 2, 3) == -1     # sinks + recent fill the budget
    assert sel(1, 10, 5, 0, 11, 1, 0) == -1    # k > T
    assert sel(1, 10, 131, 0, 5, 1, 0) == -2   # pooling window beyond 129
    assert sel(0, 10, 5, 3, 5, 1, 2) == 0      # empty batch: nothing to do
    p = ctypes.c_void_p(256)  # dummy aligned pointers: rejected before any use
    assert lib.hubkv_select_topk(p, 1, 2, 10, 5, 0.5, 0.1, 0.8, 1.2, 0, 5, 1, 0, p, NULL, NULL,
                                 NULL, 0, NULL) == -5  # no workspace
    # workspace: the refinement's partials and head weights; a z buffer only for
    # heads too long to hold on chip
    short = lib.kv_workspace_size(6, 4, 8, 8, 131072, 0, 64, 6553)
    assert short == lib.kv_workspace_size(6, 4, 8, 8, 1000, 0, 64, 100) or short > 0
    assert short < 4 * 8 * 131072 * 4
    long_ = lib.kv_workspace_size(6, 1, 2, 2, 400000, 0, 64, 20000)
    assert long_ >= 1 * 2 * 400000 * 4
    assert lib.kv_workspace_size(6, 1, 2, 2, 100, 0, 64, 64) == 0  # k <= recent + sink


def test_layer_budget_entry_points_validate_on_the_host(lib):
    sel = lambda B, H, T, budget, floor, R, S: lib.kv_select_budget(  # noqa: E731
        NULL, B, H, T, budget, floor, R, S, NULL, NULL, NULL)
    assert sel(1, 2, 10, 3, 2, 0, 0) == -1      # budget < H * floor
    assert sel(1, 2, 10, 21, 2, 0, 0) == -1     # budget > H * T
    assert sel(1, 2, 10, 10, 2, 2, 1) == -1     # floor < sinks + recent
    assert sel(1, 2, 10, 10, 0, 0, 0) == -1     # floor < 1
    assert sel(1, 2, 10, 10, 11, 0, 0) == -1    # floor > T
    assert sel(1, 2, 10, 10, 3, -1, 0) == -1
    assert sel(1, 257, 10, 2570, 10, 0, 0) == -2   # more heads than one cluster serves
    assert sel(1, 2, 10, 10, 3, 1, 0) == -1     # null pointers
    assert sel(0, 2, 10, 10, 3, 1, 1) == 0      # empty batch
    rag = lambda B, H, budget, d, cap: lib.kv_compact_ragged(  # noqa: E731
        NULL, NULL, NULL, NULL, NULL, B, H, 10, budget, d, 0, NULL, NULL, cap, NULL, NULL, NULL,
        NULL, NULL)
    assert rag(1, 2, 8, 64, -1) == -1
    assert rag(1, 2, -1, 64, 4) == -1
    assert rag(1, 2, 8, 96, 4) == -2
    assert rag(1, 2, 8, 64, 4) == -1            # null pointers
    assert rag(0, 2, 8, 64, 4) == 0


def test_nested_scorer_validates_on_the_host(lib):
    def call(B=1, H=2, T=100, d=128, dt=0, window=64, nb=32, nd=10, lp=(0.0, 0.0, 0.0), th=0.1,
             ws=NULL, wsb=0):
        return lib.kv_score_nested(NULL, B, H, T, d, dt, window, nb, nd, lp[0], lp[1], lp[2], th,
                                   NULL, NULL, NULL, ws, wsb, NULL)
    assert call(nd=101) == -1                 # n_disc > T
    assert call(nd=0) == -1
    assert call(window=0) == -1
    assert call(nb=0) == -1
    assert call(th=float("nan")) == -1
    assert call(lp=(float("inf"), 0.0, 0.0)) == -1
    assert call(d=96) == -2
    assert call(window=5000) == -2
    assert call() == -1                       # null pointers
    assert call(B=0) == 0
    assert lib.kv_workspace_size(5, 1, 0, 8, 131072, 128, 32, 0) >= 8 * 3 * 131072 * 4
    assert lib.kv_workspace_size(5, 1, 0, 8, 131072, 96, 32, 0) == 0


def test_multi_step_decode_validates_on_the_host(lib):
    def call(n=4, B=1, Hq=4, Hkv=4, cap=8, d=64, R=1, S=0, first=9, flags=0):
        return lib.h2o_decode_steps(NULL, NULL, NULL, n, NULL, NULL, NULL, NULL, NULL, B, Hq, Hkv, cap,
                                    d, R, S, first, 0.1, flags, 0, NULL, NULL, NULL, 0, NULL, NULL)
    assert call(n=-1) == -1
    assert call(first=2 ** 31 - 2, n=4) == -1   # positions past int32
    assert call(R=8) == -1                       # recent >= cap, caught on the first step
    assert call(flags=1) == -1                   # ALG1 with a recent window
    assert call(d=96) == -2
    assert call() == -1                          # null pointers
    assert call(n=0) == 0 and call(B=0) == 0     # nothing to do


def test_empty_batch_is_a_no_op(lib):
    assert lib.kv_score_obs(NULL, NULL, 0, 4, 2, 10, 64, 4, 0.1, 0, NULL, NULL, 0, NULL, NULL) == 0
    assert lib.hubkv_refine(NULL, 0, 2, 10, 5, 0.5, 0.1, 0.8, 1.2, NULL, NULL, NULL, 0, NULL) == 0
    assert lib.kv_select_topk(NULL, 0, 2, 10, 5, 3, NULL, NULL, 0, NULL) == 0
    assert lib.kv_compact(NULL, NULL, NULL, NULL, 0, 2, 10, 5, 64, 0, NULL, NULL, 5, NULL, NULL,
                          NULL, NULL) == 0
    assert lib.h2o_decode_step(NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, 0, 4, 4, 8, 64, 1, 9,
                               0.1, 0, 0, NULL, NULL, NULL, 0, NULL, NULL) == 0


def test_no_product_module_imports_the_oracle():
    """The CUDA path and its binding never import or load the oracle."""
    pkg = os.path.join(ROOT, "kv_cache_compression_obs_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f), encoding="utf-8").read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "liboracle" not in text and "kvc_oracle" not in text, f
