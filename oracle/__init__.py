"""CPU oracle of the KV-cache eviction path -- TEST INFRASTRUCTURE ONLY.

Only the tests, the smoke check and the benchmark's CPU-baseline leg may import
this package.  The product path (the CUDA library and its Python binding) never
imports, links or calls it, and it never imports the product path.

Thin ctypes wrappers over ``liboracle.so`` (float64 C, see kvc_oracle.c) plus the
literal greedy-eviction loop in ``alg1.py``.  Array arguments are numpy arrays:
bf16 tensors are passed as their uint16 bit patterns, float32 as float32.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from .build import build_oracle

BF16, F32 = 0, 1
FLAG_ALG1 = 1
HUB_AVGPOOL, HUB_FIXED_HEAD = 1, 2

_lib = None


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build_oracle())
        P, I, D, LL = ctypes.c_void_p, ctypes.c_int, ctypes.c_double, ctypes.c_longlong
        lib.oracle_kv_cache_bytes.restype = LL
        lib.oracle_kv_cache_bytes.argtypes = [LL, LL, LL, LL, LL]
        lib.oracle_score_obs.restype = I
        lib.oracle_score_obs.argtypes = [P, P, I, I, I, I, I, I, D, I, P]
        lib.oracle_hubkv_refine_ex.restype = I
        lib.oracle_hubkv_refine_ex.argtypes = [P, I, I, I, I, D, D, D, D, I, P, P, P]
        lib.oracle_select_topk_ex.restype = I
        lib.oracle_select_topk_ex.argtypes = [P, I, I, I, I, I, I, P]
        lib.oracle_compact.restype = I
        lib.oracle_compact.argtypes = [P, P, P, P, I, I, I, I, I, I, P, P, I, P, P, P]
        lib.oracle_select_budget.restype = I
        lib.oracle_select_budget.argtypes = [P, I, I, I, I, I, I, I, P, P]
        lib.oracle_nested_score.restype = I
        lib.oracle_nested_score.argtypes = [P, I, I, I, I, I, I, I, I, P, D, P, P, P, P]
        lib.oracle_compact_ragged.restype = I
        lib.oracle_compact_ragged.argtypes = [P, P, P, P, P, I, I, I, I, I, I, P, P, I, P, P, P]
        lib.oracle_decode_step_ex.restype = I
        lib.oracle_decode_step_ex.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, I, D, I, I, P, P]
        _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _dtype_code(a: np.ndarray) -> int:
    if a.dtype == np.uint16:
        return BF16
    if a.dtype == np.float32:
        return F32
    raise TypeError(f"oracle inputs are bf16 bits (uint16) or float32, got {a.dtype}")


def kv_cache_bytes(L: int, Hkv: int, d: int, T: int, elem_bytes: int) -> int:
    return int(_load().oracle_kv_cache_bytes(L, Hkv, d, T, elem_bytes))


def score_obs(Q: np.ndarray, K: np.ndarray, scale: float) -> np.ndarray:
    """Q [B][Hq][W][d], K [B][Hkv][T][d] -> s [B][Hkv][T] float64."""
    B, Hq, W, d = Q.shape
    B2, Hkv, T, d2 = K.shape
    assert B == B2 and d == d2 and Q.dtype == K.dtype
    Q = np.ascontiguousarray(Q)
    K = np.ascontiguousarray(K)
    s = np.zeros((B, Hkv, T), dtype=np.float64)
    rc = _load().oracle_score_obs(_ptr(Q), _ptr(K), B, Hq, Hkv, T, d, W, float(scale), _dtype_code(Q), _ptr(s))
    if rc != 0:
        raise ValueError("oracle_score_obs rejected its inputs")
    return s


def hubkv_refine(s: np.ndarray, r: float, gamma: float = 0.5, pool_width: int = 5,
                 beta_lo: float = 0.8, beta_hi: float = 1.2, flags: int = 0):
    """s [B][H][T] (any float dtype, read as float64) -> (z, beta, sel), all float64.

    flags: HUB_AVGPOOL (average-pool smoothing in place of hubs), HUB_FIXED_HEAD (beta = 1)."""
    s = np.ascontiguousarray(s, dtype=np.float64)
    B, H, T = s.shape
    z = np.zeros_like(s)
    beta = np.zeros((B, H), dtype=np.float64)
    sel = np.zeros((B, H), dtype=np.float64)
    rc = _load().oracle_hubkv_refine_ex(_ptr(s), B, H, T, pool_width, float(gamma), float(r),
                                        float(beta_lo), float(beta_hi), int(flags), _ptr(z), _ptr(beta),
                                        _ptr(sel))
    if rc != 0:
        raise ValueError("oracle_hubkv_refine rejected its inputs")
    return z, beta, sel


def select_topk(z: np.ndarray, k: int, recent: int, sink: int = 0) -> np.ndarray:
    """z [B][H][T] (read as float64) -> idx [B][H][k] int32, ascending per head.

    sink: the first `sink` positions are always kept (attention sinks)."""
    z = np.ascontiguousarray(z, dtype=np.float64)
    B, H, T = z.shape
    idx = np.zeros((B, H, k), dtype=np.int32)
    rc = _load().oracle_select_topk_ex(_ptr(z), B, H, T, int(k), int(recent), int(sink), _ptr(idx))
    if rc != 0:
        raise ValueError("oracle_select_topk rejected its inputs")
    return idx


def compact(K: np.ndarray, V: np.ndarray, s, idx: np.ndarray, cap: int):
    """Gather kept rows. Returns (K_out, V_out, pos, acc, len); slots >= k are zero."""
    B, H, T, d = K.shape
    k = idx.shape[-1]
    K = np.ascontiguousarray(K)
    V = np.ascontiguousarray(V)
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    K_out = np.zeros((B, H, cap, d), dtype=K.dtype)
    V_out = np.zeros((B, H, cap, d), dtype=V.dtype)
    pos = np.zeros((B, H, cap), dtype=np.int32)
    acc = np.zeros((B, H, cap), dtype=np.float32)
    ln = np.zeros((B, H), dtype=np.int32)
    s_arr = None if s is None else np.ascontiguousarray(s, dtype=np.float64)
    rc = _load().oracle_compact(_ptr(K), _ptr(V), None if s_arr is None else _ptr(s_arr), _ptr(idx),
                                B, H, T, k, d, _dtype_code(K), _ptr(K_out), _ptr(V_out), int(cap),
                                _ptr(pos), _ptr(acc), _ptr(ln))
    if rc != 0:
        raise ValueError("oracle_compact rejected its inputs")
    return K_out, V_out, pos, acc, ln


def select_budget(z: np.ndarray, budget: int, floor: int, recent: int, sink: int = 0):
    """Layer-level competitive budget: z [B][H][T] (read as float64), one layer per
    batch row -> (idx [B][budget] int32, off [B][H+1] int32), CSR per head."""
    z = np.ascontiguousarray(z, dtype=np.float64)
    B, H, T = z.shape
    idx = np.zeros((B, budget), dtype=np.int32)
    off = np.zeros((B, H + 1), dtype=np.int32)
    rc = _load().oracle_select_budget(_ptr(z), B, H, T, int(budget), int(floor), int(recent),
                                      int(sink), _ptr(idx), _ptr(off))
    if rc != 0:
        raise ValueError("oracle_select_budget rejected its inputs")
    return idx, off


def compact_ragged(K: np.ndarray, V: np.ndarray, s, idx: np.ndarray, off: np.ndarray, cap: int,
                   out=None):
    """Gather head h's rows idx[b][off[b][h]:off[b][h+1]] into slots 0..n-1.

    Returns (K_out, V_out, pos, acc, len); `out` (the same five arrays) is written
    in place when given, so untouched slots keep their contents."""
    B, H, T, d = K.shape
    budget = idx.shape[-1]
    K = np.ascontiguousarray(K)
    V = np.ascontiguousarray(V)
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    off = np.ascontiguousarray(off, dtype=np.int32)
    if out is None:
        out = (np.zeros((B, H, cap, d), dtype=K.dtype), np.zeros((B, H, cap, d), dtype=V.dtype),
               np.zeros((B, H, cap), dtype=np.int32), np.zeros((B, H, cap), dtype=np.float32),
               np.zeros((B, H), dtype=np.int32))
    K_out, V_out, pos, acc, ln = out
    s_arr = None if s is None else np.ascontiguousarray(s, dtype=np.float64)
    rc = _load().oracle_compact_ragged(_ptr(K), _ptr(V), None if s_arr is None else _ptr(s_arr),
                                       _ptr(idx), _ptr(off), B, H, T, budget, d, _dtype_code(K),
                                       _ptr(K_out), _ptr(V_out), int(cap), _ptr(pos), _ptr(acc),
                                       _ptr(ln))
    if rc != 0:
        raise ValueError("oracle_compact_ragged rejected its inputs")
    return K_out, V_out, pos, acc, ln


def nested_score(K: np.ndarray, n_disc: int, thresh: float, log_prior=(0.0, 0.0, 0.0),
                 window: int = 64, n_blocks: int = 32):
    """NestedKV key-only scores: K [B][H][T][d] (bf16 bits or float32) ->
    dict(score [B][H][T], a [B][H][3][T] (stable, episodic, current),
    sigma [B][H][T], w [B][H][3]), all float64."""
    B, H, T, d = K.shape
    K = np.ascontiguousarray(K)
    lp = np.ascontiguousarray(log_prior, dtype=np.float64)
    assert lp.shape == (3,)
    score = np.zeros((B, H, T), dtype=np.float64)
    a = np.zeros((B, H, 3, T), dtype=np.float64)
    sig = np.zeros((B, H, T), dtype=np.float64)
    w = np.zeros((B, H, 3), dtype=np.float64)
    rc = _load().oracle_nested_score(_ptr(K), B, H, T, d, _dtype_code(K), int(window), int(n_blocks),
                                     int(n_disc), _ptr(lp), float(thresh), _ptr(score), _ptr(a),
                                     _ptr(sig), _ptr(w))
    if rc != 0:
        raise ValueError("oracle_nested_score rejected its inputs")
    return {"score": score, "a": a, "sigma": sig, "w": w}


def decode_step(q, k_new, v_new, K_cache, V_cache, pos, acc, ln, recent: int, new_pos: int,
                scale: float, flags: int = 0, sink: int = 0):
    """One decode step; K_cache, V_cache, pos, acc, ln are updated IN PLACE.
    Positions below `sink` are never evicted.

    Returns (o [B][Hq][d] float64, evicted [B][Hkv] int32).
    """
    B, Hq, d = q.shape
    _, Hkv, cap, _ = K_cache.shape
    for a in (K_cache, V_cache, pos, acc, ln):
        assert a.flags["C_CONTIGUOUS"]
    assert pos.dtype == np.int32 and acc.dtype == np.float32 and ln.dtype == np.int32
    q = np.ascontiguousarray(q)
    k_new = np.ascontiguousarray(k_new)
    v_new = np.ascontiguousarray(v_new)
    o = np.zeros((B, Hq, d), dtype=np.float64)
    ev = np.zeros((B, Hkv), dtype=np.int32)
    rc = _load().oracle_decode_step_ex(_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(K_cache), _ptr(V_cache),
                                       _ptr(pos), _ptr(acc), _ptr(ln), B, Hq, Hkv, cap, d, int(recent),
                                       int(sink), int(new_pos), float(scale), int(flags), _dtype_code(q),
                                       _ptr(o), _ptr(ev))
    if rc != 0:
        raise ValueError("oracle_decode_step rejected its inputs")
    return o, ev


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact float value of bf16 bit patterns (for tests that need the values)."""
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


__all__ = ["BF16", "F32", "FLAG_ALG1", "kv_cache_bytes", "score_obs", "hubkv_refine",
           "select_topk", "compact", "select_budget", "compact_ragged", "nested_score", "decode_step",
           "bf16_bits_to_f64"]

from .alg1 import h2o_greedy_literal  # noqa: E402

__all__.append("h2o_greedy_literal")
del os
