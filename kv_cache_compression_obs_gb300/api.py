"""Python binding of libkvc.so: the same calls, argument marshalling only.

Every function takes CUDA torch tensors, checks dtype/shape/contiguity, passes
raw device pointers and the current CUDA stream to the C ABI, and raises
``KvcError`` on a non-zero status.  All arithmetic runs in the library's CUDA
kernels; importing this module raises if ``libkvc.so`` has not been built.
Output tensors may be passed in (``out=...``) to avoid allocation; otherwise they
are allocated with torch on the input's device.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkvc.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build the CUDA library first "
        "(python -m kv_cache_compression_obs_gb300.build)")

_lib = ctypes.CDLL(LIB_PATH)

KV_OK, KV_ERR_INVALID_ARG, KV_ERR_UNSUPPORTED, KV_ERR_CUDA, KV_ERR_TIMEOUT, KV_ERR_WORKSPACE = (
    0, -1, -2, -3, -4, -5)
KV_BF16, KV_F32 = 0, 1
KV_H2O_ALG1 = 1
KV_HUB_AVGPOOL, KV_HUB_FIXED_HEAD = 1, 2
KV_OP_SCORE_OBS, KV_OP_HUBKV_REFINE, KV_OP_SELECT_TOPK, KV_OP_DECODE, KV_OP_SCORE_NESTED = 1, 2, 3, 4, 5
KV_OP_HUBKV_SELECT = 6

_P, _I, _F, _Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
_lib.kv_score_obs.restype = _I
_lib.kv_score_obs.argtypes = [_P, _P, _I, _I, _I, _I, _I, _I, _F, _I, _P, _P, _Z, _P, _P]
_lib.hubkv_refine.restype = _I
_lib.hubkv_refine.argtypes = [_P, _I, _I, _I, _I, _F, _F, _F, _F, _P, _P, _P, _Z, _P]
_lib.hubkv_refine_ex.restype = _I
_lib.hubkv_refine_ex.argtypes = [_P, _I, _I, _I, _I, _F, _F, _F, _F, _I, _P, _P, _P, _Z, _P]
_lib.kv_select_topk.restype = _I
_lib.kv_select_topk.argtypes = [_P, _I, _I, _I, _I, _I, _P, _P, _Z, _P]
_lib.kv_select_topk_ex.restype = _I
_lib.kv_select_topk_ex.argtypes = [_P, _I, _I, _I, _I, _I, _I, _P, _P, _Z, _P]
_lib.hubkv_select_topk.restype = _I
_lib.hubkv_select_topk.argtypes = [_P, _I, _I, _I, _I, _F, _F, _F, _F, _I, _I, _I, _I, _P, _P, _P, _P,
                                   _Z, _P]
_lib.kv_compact.restype = _I
_lib.kv_compact.argtypes = [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P, _I, _P, _P, _P, _P]
_lib.kv_score_nested.restype = _I
_lib.kv_score_nested.argtypes = [_P, _I, _I, _I, _I, _I, _I, _I, _I, _F, _F, _F, _F, _P, _P, _P, _P,
                                 _Z, _P]
_lib.kv_select_budget.restype = _I
_lib.kv_select_budget.argtypes = [_P, _I, _I, _I, _I, _I, _I, _I, _P, _P, _P]
_lib.kv_compact_ragged.restype = _I
_lib.kv_compact_ragged.argtypes = [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P, _I, _P, _P,
                                   _P, _P, _P]
_lib.h2o_decode_step.restype = _I
_lib.h2o_decode_step.argtypes = [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F,
                                 _I, _I, _P, _P, _P, _Z, _P, _P]
_lib.h2o_decode_step_ex.restype = _I
_lib.h2o_decode_step_ex.argtypes = [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I,
                                    _F, _I, _I, _P, _P, _P, _Z, _P, _P]
_lib.h2o_decode_steps.restype = _I
_lib.h2o_decode_steps.argtypes = [_P, _P, _P, _I, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I,
                                  _F, _I, _I, _P, _P, _P, _Z, _P, _P]
_lib.kv_score_obs_noalloc.restype = _I
_lib.kv_score_obs_noalloc.argtypes = [_P, _P, _I, _I, _I, _I, _I, _I, _F, _I, _P, _P, _P]
_lib.kv_workspace_size.restype = _Z
_lib.kv_workspace_size.argtypes = [_I, _I, _I, _I, _I, _I, _I, _I]
_lib.kv_status_string.restype = ctypes.c_char_p
_lib.kv_status_string.argtypes = [_I]
_lib.kv_version.restype = _I
_lib.kv_last_error_detail.restype = ctypes.c_char_p
_lib.kv_last_error_detail.argtypes = []


class KvcError(RuntimeError):
    def __init__(self, call: str, status: int):
        msg = f"{call}: {_lib.kv_status_string(status).decode()} (status {status})"
        if status == KV_ERR_CUDA:
            detail = _lib.kv_last_error_detail().decode()
            if detail:
                msg += f": {detail}"
        super().__init__(msg)
        self.status = status


def _check(call: str, status: int) -> None:
    if status != KV_OK:
        raise KvcError(call, status)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return KV_BF16
    if t.dtype == torch.float32:
        return KV_F32
    raise TypeError(f"expected bfloat16 or float32, got {t.dtype}")


def _on_current_device(t):
    """The library launches on the current CUDA device (and takes its scratch and
    side stream from it), so a tensor on another device would be handed to the
    wrong GPU."""
    if t.device.index != torch.cuda.current_device():
        raise ValueError(f"tensor on {t.device} but the current CUDA device is "
                         f"cuda:{torch.cuda.current_device()}: call inside "
                         f"`with torch.cuda.device({t.device})`")


def _dev(*ts):
    for t in ts:
        if t is not None:
            if not t.is_cuda or not t.is_contiguous():
                raise ValueError("tensors must be contiguous CUDA tensors")
            _on_current_device(t)


def _dev_or_pinned(*ts):
    """Gather sources may also be pinned host tensors (read by the kernel over the
    host link, only the rows it keeps)."""
    for t in ts:
        if t is not None:
            if not t.is_contiguous() or not (t.is_cuda or t.is_pinned()):
                raise ValueError("tensors must be contiguous CUDA tensors or pinned host tensors")
            if t.is_cuda:
                _on_current_device(t)


def kv_workspace_size(op: int, B: int, Hq: int, Hkv: int, T: int, d: int = 128, W: int = 1,
                      k: int = 1) -> int:
    return int(_lib.kv_workspace_size(op, B, Hq, Hkv, T, d, W, k))


def _workspace(nbytes: int, device, given):
    if nbytes == 0:
        return None, 0
    if given is not None:
        return given, given.numel() * given.element_size()
    return torch.empty(nbytes, dtype=torch.uint8, device=device), nbytes


def kv_score_obs(Q_obs: torch.Tensor, K: torch.Tensor, scale: float | None = None, out=None,
                 workspace=None, dev_status=None, stream=None) -> torch.Tensor:
    """Q_obs [B][Hq][W][d], K [B][Hkv][T][d] -> s [B][Hkv][T] float32."""
    B, Hq, W, d = Q_obs.shape
    B2, Hkv, T, d2 = K.shape
    if B2 != B or d2 != d or Q_obs.dtype != K.dtype:
        raise ValueError("Q_obs and K disagree in batch, head dim or dtype")
    _dev(Q_obs, K, out)
    if scale is None:
        scale = d ** -0.5
    s = out if out is not None else torch.empty(B, Hkv, T, dtype=torch.float32, device=K.device)
    ws, nbytes = _workspace(kv_workspace_size(KV_OP_SCORE_OBS, B, Hq, Hkv, T, d, W), K.device,
                            workspace)
    _dev(dev_status)
    _check("kv_score_obs", _lib.kv_score_obs(_ptr(Q_obs), _ptr(K), B, Hq, Hkv, T, d, W,
                                             float(scale), _dtype_code(K), _ptr(s), _ptr(ws),
                                             nbytes, _ptr(dev_status), _stream(stream)))
    return s


def kv_score_obs_noalloc(Q_obs: torch.Tensor, K: torch.Tensor, scale: float | None = None,
                         out=None, dev_status=None, stream=None) -> torch.Tensor:
    """kv_score_obs with the library's built-in scratch array instead of a workspace."""
    B, Hq, W, d = Q_obs.shape
    B2, Hkv, T, d2 = K.shape
    if B2 != B or d2 != d or Q_obs.dtype != K.dtype:
        raise ValueError("Q_obs and K disagree in batch, head dim or dtype")
    _dev(Q_obs, K, out)
    if scale is None:
        scale = d ** -0.5
    s = out if out is not None else torch.empty(B, Hkv, T, dtype=torch.float32, device=K.device)
    _dev(dev_status)
    _check("kv_score_obs_noalloc", _lib.kv_score_obs_noalloc(
        _ptr(Q_obs), _ptr(K), B, Hq, Hkv, T, d, W, float(scale), _dtype_code(K), _ptr(s),
        _ptr(dev_status), _stream(stream)))
    return s


def hubkv_refine(s: torch.Tensor, r: float, gamma: float = 0.5, pool_width: int = 5,
                 beta_lo: float = 0.8, beta_hi: float = 1.2, out=None, beta_out=None,
                 workspace=None, stream=None, flags: int = 0):
    """s [B][H][T] float32 -> (z [B][H][T], beta [B][H]) float32.

    flags: KV_HUB_AVGPOOL and/or KV_HUB_FIXED_HEAD select the comparison variants."""
    B, H, T = s.shape
    if s.dtype != torch.float32:
        raise TypeError("s must be float32")
    _dev(s, out, beta_out)
    z = out if out is not None else torch.empty_like(s)
    beta = beta_out if beta_out is not None else torch.empty(B, H, dtype=torch.float32,
                                                             device=s.device)
    ws, nbytes = _workspace(kv_workspace_size(KV_OP_HUBKV_REFINE, B, H, H, T), s.device, workspace)
    _check("hubkv_refine", _lib.hubkv_refine_ex(_ptr(s), B, H, T, pool_width, float(gamma), float(r),
                                                float(beta_lo), float(beta_hi), int(flags), _ptr(z),
                                                _ptr(beta), _ptr(ws), nbytes, _stream(stream)))
    return z, beta


def kv_select_topk(z: torch.Tensor, k: int, recent: int, out=None, stream=None,
                   sink: int = 0) -> torch.Tensor:
    """z [B][H][T] float32 -> idx [B][H][k] int32 (ascending positions); the first
    `sink` positions are kept as attention sinks."""
    B, H, T = z.shape
    if z.dtype != torch.float32:
        raise TypeError("z must be float32")
    _dev(z, out)
    idx = out if out is not None else torch.empty(B, H, k, dtype=torch.int32, device=z.device)
    _check("kv_select_topk", _lib.kv_select_topk_ex(_ptr(z), B, H, T, int(k), int(recent), int(sink),
                                                    _ptr(idx), None, 0, _stream(stream)))
    return idx


def hubkv_select_topk(s: torch.Tensor, k: int, recent: int, r: float, gamma: float = 0.5,
                      pool_width: int = 5, beta_lo: float = 0.8, beta_hi: float = 1.2,
                      sink: int = 0, flags: int = 0, out=None, z_out=None, beta_out=None,
                      workspace=None, stream=None) -> torch.Tensor:
    """hubkv_refine then kv_select_topk in one call: s [B][H][T] float32 ->
    idx [B][H][k] int32 (ascending).  z_out [B][H][T] and beta_out [B][H] are
    filled when given."""
    B, H, T = s.shape
    if s.dtype != torch.float32:
        raise TypeError("s must be float32")
    _dev(s, out, z_out, beta_out)
    idx = out if out is not None else torch.empty(B, H, k, dtype=torch.int32, device=s.device)
    ws, nbytes = _workspace(kv_workspace_size(KV_OP_HUBKV_SELECT, B, H, H, T, 0, recent + sink, k),
                            s.device, workspace)
    _check("hubkv_select_topk", _lib.hubkv_select_topk(
        _ptr(s), B, H, T, int(pool_width), float(gamma), float(r), float(beta_lo), float(beta_hi),
        int(flags), int(k), int(recent), int(sink), _ptr(idx), _ptr(z_out), _ptr(beta_out),
        _ptr(ws), nbytes, _stream(stream)))
    return idx


def kv_compact(K: torch.Tensor, V: torch.Tensor, s, idx: torch.Tensor, cap: int | None = None,
               K_out=None, V_out=None, pos_out=None, acc_out=None, len_out=None, stream=None):
    """Gather the kept rows into a slot cache; returns (K_out, V_out, pos, acc, len)."""
    B, H, T, d = K.shape
    k = idx.shape[-1]
    cap = k if cap is None else cap
    if idx.dtype != torch.int32 or V.shape != K.shape or V.dtype != K.dtype:
        raise ValueError("idx must be int32 and V must match K")
    _dev(s, idx, K_out, V_out, pos_out, acc_out, len_out)
    _dev_or_pinned(K, V)
    dev = idx.device
    K_out = K_out if K_out is not None else torch.empty(B, H, cap, d, dtype=K.dtype, device=dev)
    V_out = V_out if V_out is not None else torch.empty(B, H, cap, d, dtype=K.dtype, device=dev)
    pos = pos_out if pos_out is not None else torch.zeros(B, H, cap, dtype=torch.int32, device=dev)
    acc = acc_out if acc_out is not None else torch.zeros(B, H, cap, dtype=torch.float32, device=dev)
    ln = len_out if len_out is not None else torch.empty(B, H, dtype=torch.int32, device=dev)
    _check("kv_compact", _lib.kv_compact(_ptr(K), _ptr(V), _ptr(s), _ptr(idx), B, H, T, k, d,
                                         _dtype_code(K), _ptr(K_out), _ptr(V_out), int(cap),
                                         _ptr(pos), _ptr(acc if s is not None else None), _ptr(ln),
                                         _stream(stream)))
    return K_out, V_out, pos, acc, ln


def h2o_decode_steps(q, k_new, v_new, K_cache, V_cache, pos, acc, len_, recent: int,
                     first_pos: int, scale: float | None = None, flags: int = 0, o_out=None,
                     evicted_out=None, workspace=None, dev_status=None, stream=None,
                     sink: int = 0):
    """n consecutive decode steps in one call: q [n][B][Hq][d], k_new, v_new [n][B][Hkv][d];
    step t uses position first_pos + t.  Returns (o [n][B][Hq][d] f32, evicted [n][B][Hkv])."""
    n, B, Hq, d = q.shape
    _, Hkv, cap, _ = K_cache.shape
    _dev(q, k_new, v_new, K_cache, V_cache, pos, acc, len_, o_out, evicted_out, dev_status)
    if scale is None:
        scale = d ** -0.5
    o = o_out if o_out is not None else torch.empty(n, B, Hq, d, dtype=torch.float32,
                                                    device=q.device)
    ev = evicted_out if evicted_out is not None else torch.empty(n, B, Hkv, dtype=torch.int32,
                                                                 device=q.device)
    ws, nbytes = _workspace(kv_workspace_size(KV_OP_DECODE, B, Hq, Hkv, cap, d), q.device, workspace)
    _check("h2o_decode_steps", _lib.h2o_decode_steps(
        _ptr(q), _ptr(k_new), _ptr(v_new), int(n), _ptr(K_cache), _ptr(V_cache), _ptr(pos),
        _ptr(acc), _ptr(len_), B, Hq, Hkv, cap, d, int(recent), int(sink), int(first_pos),
        float(scale), int(flags), _dtype_code(q), _ptr(o), _ptr(ev), _ptr(ws), nbytes,
        _ptr(dev_status), _stream(stream)))
    return o, ev


def kv_score_nested(K: torch.Tensor, n_disc: int, thresh: float, log_prior=(0.0, 0.0, 0.0),
                    window: int = 64, n_blocks: int = 32, out=None, w_out=None, a_out=None,
                    workspace=None, stream=None):
    """NestedKV key-only scores: K [B][H][T][d] -> (score [B][H][T], w [B][H][3]) float32.
    a_out ([B][H][3][T] float32), when given, receives the three anomaly scores."""
    B, H, T, d = K.shape
    _dev(K, out, w_out, a_out)
    dev = K.device
    score = out if out is not None else torch.empty(B, H, T, dtype=torch.float32, device=dev)
    w = w_out if w_out is not None else torch.empty(B, H, 3, dtype=torch.float32, device=dev)
    ws, nbytes = _workspace(kv_workspace_size(KV_OP_SCORE_NESTED, B, 0, H, T, d, n_blocks), dev,
                            workspace)
    lp = [float(x) for x in log_prior]
    _check("kv_score_nested", _lib.kv_score_nested(
        _ptr(K), B, H, T, d, _dtype_code(K), int(window), int(n_blocks), int(n_disc), lp[0], lp[1],
        lp[2], float(thresh), _ptr(score), _ptr(w), _ptr(a_out), _ptr(ws), nbytes, _stream(stream)))
    return score, w


def kv_select_budget(z: torch.Tensor, budget: int, floor: int, recent: int, sink: int = 0,
                     idx_out=None, off_out=None, stream=None):
    """Layer-level competitive budget: z [B][H][T] float32, one layer per batch row
    -> (idx [B][budget] int32, off [B][H+1] int32): head h's kept positions,
    ascending, are idx[b][off[b][h]:off[b][h+1]]."""
    B, H, T = z.shape
    if z.dtype != torch.float32:
        raise TypeError("z must be float32")
    _dev(z, idx_out, off_out)
    dev = z.device
    idx = idx_out if idx_out is not None else torch.empty(B, budget, dtype=torch.int32, device=dev)
    off = off_out if off_out is not None else torch.empty(B, H + 1, dtype=torch.int32, device=dev)
    _check("kv_select_budget", _lib.kv_select_budget(_ptr(z), B, H, T, int(budget), int(floor),
                                                     int(recent), int(sink), _ptr(idx), _ptr(off),
                                                     _stream(stream)))
    return idx, off


def kv_compact_ragged(K: torch.Tensor, V: torch.Tensor, s, idx: torch.Tensor, off: torch.Tensor,
                      cap: int, K_out=None, V_out=None, pos_out=None, acc_out=None, len_out=None,
                      dev_status=None, stream=None):
    """Gather each head's CSR rows (kv_select_budget's output) into its slots
    0..n-1 of a slot cache; returns (K_out, V_out, pos, acc, len)."""
    B, H, T, d = K.shape
    budget = idx.shape[-1]
    if idx.dtype != torch.int32 or off.dtype != torch.int32 or V.shape != K.shape or V.dtype != K.dtype:
        raise ValueError("idx and off must be int32 and V must match K")
    if tuple(off.shape) != (B, H + 1) or idx.shape[0] != B:
        raise ValueError("idx must be [B][budget] and off [B][H+1]")
    _dev(s, idx, off, K_out, V_out, pos_out, acc_out, len_out, dev_status)
    _dev_or_pinned(K, V)
    dev = idx.device
    K_out = K_out if K_out is not None else torch.empty(B, H, cap, d, dtype=K.dtype, device=dev)
    V_out = V_out if V_out is not None else torch.empty(B, H, cap, d, dtype=K.dtype, device=dev)
    pos = pos_out if pos_out is not None else torch.zeros(B, H, cap, dtype=torch.int32, device=dev)
    acc = acc_out if acc_out is not None else torch.zeros(B, H, cap, dtype=torch.float32, device=dev)
    ln = len_out if len_out is not None else torch.empty(B, H, dtype=torch.int32, device=dev)
    _check("kv_compact_ragged", _lib.kv_compact_ragged(
        _ptr(K), _ptr(V), _ptr(s), _ptr(idx), _ptr(off), B, H, T, budget, d, _dtype_code(K),
        _ptr(K_out), _ptr(V_out), int(cap), _ptr(pos), _ptr(acc if s is not None else None),
        _ptr(ln), _ptr(dev_status), _stream(stream)))
    return K_out, V_out, pos, acc, ln


def h2o_decode_step(q, k_new, v_new, K_cache, V_cache, pos, acc, len_, recent: int, new_pos: int,
                    scale: float | None = None, flags: int = 0, o_out=None, evicted_out=None,
                    workspace=None, dev_status=None, stream=None, sink: int = 0):
    """One decode step, cache state updated in place; returns (o [B][Hq][d] f32, evicted [B][Hkv]).
    Positions below `sink` are never evicted (attention sinks)."""
    B, Hq, d = q.shape
    _, Hkv, cap, _ = K_cache.shape
    _dev(q, k_new, v_new, K_cache, V_cache, pos, acc, len_, o_out, evicted_out, dev_status)
    if scale is None:
        scale = d ** -0.5
    o = o_out if o_out is not None else torch.empty(B, Hq, d, dtype=torch.float32, device=q.device)
    ev = evicted_out if evicted_out is not None else torch.empty(B, Hkv, dtype=torch.int32,
                                                                 device=q.device)
    ws, nbytes = _workspace(kv_workspace_size(KV_OP_DECODE, B, Hq, Hkv, cap, d), q.device, workspace)
    _check("h2o_decode_step", _lib.h2o_decode_step_ex(
        _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(K_cache), _ptr(V_cache), _ptr(pos), _ptr(acc),
        _ptr(len_), B, Hq, Hkv, cap, d, int(recent), int(sink), int(new_pos), float(scale), int(flags),
        _dtype_code(q), _ptr(o), _ptr(ev), _ptr(ws), nbytes, _ptr(dev_status), _stream(stream)))
    return o, ev


def compress_prefill(Q_obs, K, V, k: int, recent: int, r: float | None, gamma: float = 0.5,
                     pool_width: int = 5, beta_lo: float = 0.8, beta_hi: float = 1.2,
                     cap: int | None = None, scale: float | None = None, stream=None):
    """The prefill eviction chain: score -> (HubKV refine) -> Top-K -> compact.

    Returns a dict with the base scores s, the refined scores z (s itself when
    r is None), the kept positions idx and the slot cache (K, V, pos, acc, len).
    """
    s = kv_score_obs(Q_obs, K, scale, stream=stream)
    if r is None:
        z = s
        beta = None
        idx = kv_select_topk(z, k, recent, stream=stream)
    else:
        z = torch.empty_like(s)
        beta = torch.empty(s.shape[:2], dtype=torch.float32, device=s.device)
        idx = hubkv_select_topk(s, k, recent, r, gamma, pool_width, beta_lo, beta_hi, z_out=z,
                                beta_out=beta, stream=stream)
    Kc, Vc, pos, acc, ln = kv_compact(K, V, s, idx, cap, stream=stream)
    return {"s": s, "z": z, "beta": beta, "idx": idx, "K": Kc, "V": Vc, "pos": pos, "acc": acc,
            "len": ln}


def prefill_host_buffers(hQ: torch.Tensor, hK: torch.Tensor, k: int, r: float | None,
                         cap: int | None = None, device=None, rows_per_chunk: int = 1):
    """Device buffers for compress_prefill_host (reusable across calls)."""
    B, Hq, W, d = hQ.shape
    _, Hkv, T, _ = hK.shape
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    cap = k if cap is None else cap
    f32, i32 = torch.float32, torch.int32
    rc = min(rows_per_chunk, B)
    ws = max(kv_workspace_size(KV_OP_SCORE_OBS, rc, Hq, Hkv, T, d, W),
             kv_workspace_size(KV_OP_HUBKV_REFINE, rc, Hkv, Hkv, T),
             kv_workspace_size(KV_OP_HUBKV_SELECT, rc, Hkv, Hkv, T, 0, 0, k), 256)
    s = torch.empty(B, Hkv, T, dtype=f32, device=dev)
    return {
        "Q": torch.empty(hQ.shape, dtype=hQ.dtype, device=dev),
        "K": torch.empty(hK.shape, dtype=hK.dtype, device=dev),
        "s": s,
        "z": torch.empty_like(s) if r is not None else s,
        "beta": torch.empty(B, Hkv, dtype=f32, device=dev),
        "idx": torch.empty(B, Hkv, k, dtype=i32, device=dev),
        "Kc": torch.empty(B, Hkv, cap, d, dtype=hK.dtype, device=dev),
        "Vc": torch.empty(B, Hkv, cap, d, dtype=hK.dtype, device=dev),
        "pos": torch.zeros(B, Hkv, cap, dtype=i32, device=dev),
        "acc": torch.zeros(B, Hkv, cap, dtype=f32, device=dev),
        "len": torch.empty(B, Hkv, dtype=i32, device=dev),
        "ws": torch.empty(ws, dtype=torch.uint8, device=dev),
        "copy_stream": torch.cuda.Stream(device=dev),
        "rows_per_chunk": rc,
        "cap": cap,
    }


def compress_prefill_host(hQ: torch.Tensor, hK: torch.Tensor, hV: torch.Tensor, k: int, recent: int,
                          r: float | None, gamma: float = 0.5, pool_width: int = 5,
                          beta_lo: float = 0.8, beta_hi: float = 1.2, scale: float | None = None,
                          buffers=None, stream=None, rows=None, wait=True):
    """The prefill chain of compress_prefill on host-resident inputs.

    hQ [B][Hq][W][d], hK, hV [B][Hkv][T][d]: pinned host tensors.  Q and K move to
    the device one chunk of batch rows at a time on a copy stream; each chunk's
    chain (score, refine, Top-K, compact) runs on `stream` as soon as its keys
    have landed, so the copies of later chunks overlap the work on earlier ones.
    V never moves in full: the compaction gathers the kept rows straight from the
    pinned host memory over the host link.  `buffers` comes from
    prefill_host_buffers; the result dict holds the same entries as
    compress_prefill's (views of the buffers).  hV must stay alive until the
    stream has passed the call.  `rows` = (r0, r1) restricts the call to those
    batch rows (independent of the others); wait=False skips the copy stream's
    wait for the work already on `stream`, for a caller that knows those rows'
    buffers are free (e.g. the later row groups of one step).  With HubKV
    refinement the refined scores z are formed inside the selection and not
    written (the result's "z" is None).
    """
    for t in (hQ, hK, hV):
        if t.is_cuda or not t.is_pinned() or not t.is_contiguous():
            raise ValueError("host inputs must be contiguous pinned CPU tensors")
    B = hK.shape[0]
    lo, hi = (0, B) if rows is None else rows
    bf = buffers if buffers is not None else prefill_host_buffers(hQ, hK, k, r)
    cs = torch.cuda.current_stream() if stream is None else stream
    cp = bf["copy_stream"]
    if wait:
        cp.wait_stream(cs)  # the buffers' previous readers are done
    with torch.cuda.stream(cp):
        bf["Q"][lo:hi].copy_(hQ[lo:hi], non_blocking=True)
    step = bf["rows_per_chunk"]
    for r0 in range(lo, hi, step):
        r1 = min(hi, r0 + step)
        with torch.cuda.stream(cp):
            bf["K"][r0:r1].copy_(hK[r0:r1], non_blocking=True)
            landed = torch.cuda.Event()
            landed.record(cp)
        cs.wait_event(landed)
        Q, K, sc = bf["Q"][r0:r1], bf["K"][r0:r1], bf["s"][r0:r1]
        kv_score_obs(Q, K, scale, out=sc, workspace=bf["ws"], stream=cs)
        if r is None:
            idx = kv_select_topk(sc, k, recent, out=bf["idx"][r0:r1], stream=cs)
        else:  # refinement folded into the selection: z is not written
            idx = hubkv_select_topk(sc, k, recent, r, gamma, pool_width, beta_lo, beta_hi,
                                    out=bf["idx"][r0:r1], beta_out=bf["beta"][r0:r1],
                                    workspace=bf["ws"], stream=cs)
        kv_compact(K, hV[r0:r1], sc, idx, bf["cap"], K_out=bf["Kc"][r0:r1], V_out=bf["Vc"][r0:r1],
                   pos_out=bf["pos"][r0:r1], acc_out=bf["acc"][r0:r1], len_out=bf["len"][r0:r1],
                   stream=cs)
    return {"s": bf["s"], "z": None if r is not None else bf["s"],
            "beta": bf["beta"] if r is not None else None,
            "idx": bf["idx"], "K": bf["Kc"], "V": bf["Vc"], "pos": bf["pos"], "acc": bf["acc"],
            "len": bf["len"]}


def library_handle():
    """The loaded ctypes library (for tests that check exported symbols)."""
    return _lib
