"""ctypes binding of libkda.so (C ABI in include/kda.h).

Argument marshalling only: torch tensors are turned into device pointers and
sizes, the state tensors' dtype into the ABI's state-dtype code.  Every step of
the computation runs in the library's CUDA kernels; if the library is missing
or fails to load this module raises, it never falls back to anything else.

The Python signature mirrors flash_kda.fwd from the FlashKDA README "Kernel
API" section: ``kda_fwd(q, k, v, g, beta, scale, out, A_log, dt_bias,
lower_bound, initial_state=None, final_state=None, cu_seqlens=None)``; it
returns nothing and writes ``out`` (and ``final_state``) in place.  ``lower_bound=None``
selects the gate without a lower bound (the C entry point kda_fwd_unbounded).
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libkda.so")

KDA_OK = 0
KDA_ERR_NULL = 1
KDA_ERR_DTYPE = 2
KDA_ERR_SHAPE = 3
KDA_ERR_UNSUPPORTED = 4
KDA_ERR_ALIGN = 5
KDA_ERR_VALUE = 6
KDA_ERR_CUDA = 7
KDA_ERR_TIMEOUT = 8
KDA_ERR_LIMIT = 9
KDA_ERR_RANGE = 10

KDA_STATE_NONE = 0
KDA_STATE_BF16 = 1
KDA_STATE_FP32 = 2

# Every symbol include/kda.h declares.
EXPORTED = ("kda_fwd", "kda_fwd_ws", "kda_fwd_unbounded", "kda_workspace_size", "kda_workspace_size_pool",
            "kda_status_string", "kda_get_device_status", "kda_version", "kda_fwd_static",
            "kda_bwd")

# Workspace bytes per (sequence, head) of kda_fwd_ws (KDA_WORKSPACE_BYTES_PER_UNIT).
WORKSPACE_BYTES_PER_UNIT = 99328
# Most (sequence, head) units of one kda_fwd_static call (KDA_STATIC_MAX_UNITS).
STATIC_MAX_UNITS = 128

_lock = threading.Lock()
_lib = None


class KDAError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(msg)
        self.status = status


def lib() -> ctypes.CDLL:
    """Open libkda.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                                   "`python -m gated_delta_rule_52_gb300.build`")
            L = ctypes.CDLL(LIB_PATH)
            vp, f, i64, ci = ctypes.c_void_p, ctypes.c_float, ctypes.c_int64, ctypes.c_int
            L.kda_fwd.argtypes = [vp, vp, vp, vp, vp, f, vp, vp, vp, f, vp, vp, ci, vp, i64,
                                  i64, i64, i64, i64, i64, vp]
            L.kda_fwd.restype = ci
            L.kda_fwd_ws.argtypes = [vp, vp, vp, vp, vp, f, vp, vp, vp, f, vp, vp, ci, vp, i64,
                                     i64, i64, i64, i64, i64, vp, ctypes.c_size_t, vp]
            L.kda_fwd_ws.restype = ci
            L.kda_fwd_unbounded.argtypes = [vp, vp, vp, vp, vp, f, vp, vp, vp, vp, vp, ci, vp, i64,
                                            i64, i64, i64, i64, i64, vp]
            L.kda_fwd_unbounded.restype = ci
            L.kda_fwd_static.argtypes = [vp, vp, vp, vp, vp, f, vp, vp, vp, f, vp, vp, ci, vp,
                                         i64, i64, i64, i64, i64, i64, vp]
            L.kda_fwd_static.restype = ci
            L.kda_bwd.argtypes = [vp, vp, vp, vp, vp, f, vp, vp, f, ci, vp, ci, vp, vp, vp, i64,
                                  i64, i64, i64, i64, i64, vp, vp, vp, vp, vp, vp, vp, vp, vp]
            L.kda_bwd.restype = ci
            L.kda_workspace_size.argtypes = [i64, i64]
            L.kda_workspace_size.restype = ctypes.c_size_t
            L.kda_workspace_size_pool.argtypes = [i64, i64]
            L.kda_workspace_size_pool.restype = ctypes.c_size_t
            L.kda_status_string.argtypes = [ci]
            L.kda_status_string.restype = ctypes.c_char_p
            L.kda_get_device_status.argtypes = [vp]
            L.kda_get_device_status.restype = ci
            L.kda_version.argtypes = []
            L.kda_version.restype = ci
            _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().kda_status_string(int(status)).decode()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check_tensor(name, t, dtype, shape=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def state_dtype_code(initial_state, final_state) -> int:
    dts = {t.dtype for t in (initial_state, final_state) if t is not None}
    if not dts:
        return KDA_STATE_NONE
    if len(dts) != 1:
        raise ValueError("initial_state and final_state must have the same dtype")
    dt = dts.pop()
    if dt == torch.bfloat16:
        return KDA_STATE_BF16
    if dt == torch.float32:
        return KDA_STATE_FP32
    raise ValueError(f"state dtype must be bf16 or fp32, got {dt}")


def workspace_bytes(num_seqs: int, H: int) -> int:
    """Size of the workspace kda_fwd_ws needs for N sequences of H heads."""
    return int(num_seqs) * int(H) * WORKSPACE_BYTES_PER_UNIT


def workspace_bytes_pool(num_seqs: int, H: int) -> int:
    """Size of a kda_fwd_ws workspace with which fixed-length calls of more than 64 rows
    run the persistent pool kernel (kda_workspace_size_pool; on the current device)."""
    return int(lib().kda_workspace_size_pool(int(num_seqs), int(H)))


def kda_fwd(q, k, v, g, beta, scale, out, A_log, dt_bias, lower_bound, initial_state=None,
            final_state=None, cu_seqlens=None, stream=None, workspace=None) -> None:
    """KDA forward through libkda.so.  Writes ``out`` [B,T,H,V] (and ``final_state``)
    in place, asynchronously on ``stream`` (default: the current torch stream).
    With ``workspace`` (a CUDA uint8 tensor of at least ``workspace_bytes(N, H)``
    bytes) the call goes to kda_fwd_ws and allocates nothing.  ``lower_bound=None``
    selects the gate without a lower bound (kda_fwd_unbounded: -exp(A_log) softplus(g +
    dt_bias); the chunked form above 64 rows, each token's decay floored at 2^-14)."""
    if q.dim() != 4:
        raise ValueError("q must be [B, T, H, K]")
    B, T, H, K = q.shape
    V = v.shape[-1] if v.dim() == 4 else -1
    _check_tensor("q", q, torch.bfloat16)
    _check_tensor("k", k, torch.bfloat16, (B, T, H, K))
    _check_tensor("g", g, torch.bfloat16, (B, T, H, K))
    _check_tensor("v", v, torch.bfloat16, (B, T, H, V))
    _check_tensor("beta", beta, torch.bfloat16, (B, T, H))
    _check_tensor("out", out, torch.bfloat16, (B, T, H, V))
    _check_tensor("A_log", A_log, torch.float32, (H,))
    _check_tensor("dt_bias", dt_bias, torch.float32, (H, K))
    num_seqs = 0
    if cu_seqlens is not None:
        _check_tensor("cu_seqlens", cu_seqlens, torch.int64)
        if cu_seqlens.dim() != 1 or cu_seqlens.numel() < 2:
            raise ValueError("cu_seqlens must be 1-D with at least 2 entries")
        num_seqs = cu_seqlens.numel() - 1
    N = num_seqs if cu_seqlens is not None else B
    code = state_dtype_code(initial_state, final_state)
    for name, s in (("initial_state", initial_state), ("final_state", final_state)):
        if s is not None:
            _check_tensor(name, s, s.dtype, (N, H, V, K))
    if lower_bound is None:
        if workspace is not None:
            raise ValueError("the gate without a lower bound takes no workspace")
        st = lib().kda_fwd_unbounded(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale),
                                     _ptr(out), _ptr(A_log), _ptr(dt_bias), _ptr(initial_state),
                                     _ptr(final_state), code, _ptr(cu_seqlens), num_seqs, B, T, H,
                                     K, V, _stream_handle(stream))
        if st != KDA_OK:
            raise KDAError(st, status_string(st))
        return
    args = (_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale), _ptr(out), _ptr(A_log),
            _ptr(dt_bias), float(lower_bound), _ptr(initial_state), _ptr(final_state), code,
            _ptr(cu_seqlens), num_seqs, B, T, H, K, V)
    if workspace is None:
        st = lib().kda_fwd(*args, _stream_handle(stream))
    else:
        _check_tensor("workspace", workspace, torch.uint8)
        st = lib().kda_fwd_ws(*args, _ptr(workspace), workspace.numel(), _stream_handle(stream))
    if st != KDA_OK:
        raise KDAError(st, status_string(st))


def kda_fwd_static(q, k, v, g, beta, scale, out, A_log, dt_bias, lower_bound,
                   initial_state=None, final_state=None, cu_seqlens=None, stream=None) -> None:
    """kda_fwd through the C entry point kda_fwd_static, which allocates nothing: for
    callers that cannot allocate device memory (an engine that owns all of it, a
    plug-in host that hands over only the inputs and outputs).  Its scratch is a fixed
    array inside libkda.so, so a call holds at most ``STATIC_MAX_UNITS`` (sequence,
    head) units, and calls that may overlap on the GPU race on that array.  Same
    arguments and results as ``kda_fwd`` with a lower bound."""
    if q.dim() != 4:
        raise ValueError("q must be [B, T, H, K]")
    B, T, H, K = q.shape
    V = v.shape[-1] if v.dim() == 4 else -1
    for name, t, shape in (("q", q, None), ("k", k, (B, T, H, K)), ("g", g, (B, T, H, K)),
                           ("v", v, (B, T, H, V)), ("beta", beta, (B, T, H)),
                           ("out", out, (B, T, H, V))):
        _check_tensor(name, t, torch.bfloat16, shape)
    _check_tensor("A_log", A_log, torch.float32, (H,))
    _check_tensor("dt_bias", dt_bias, torch.float32, (H, K))
    num_seqs = 0
    if cu_seqlens is not None:
        _check_tensor("cu_seqlens", cu_seqlens, torch.int64)
        if cu_seqlens.dim() != 1 or cu_seqlens.numel() < 2:
            raise ValueError("cu_seqlens must be 1-D with at least 2 entries")
        num_seqs = cu_seqlens.numel() - 1
    N = num_seqs if cu_seqlens is not None else B
    code = state_dtype_code(initial_state, final_state)
    for name, s in (("initial_state", initial_state), ("final_state", final_state)):
        if s is not None:
            _check_tensor(name, s, s.dtype, (N, H, V, K))
    st = lib().kda_fwd_static(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale),
                              _ptr(out), _ptr(A_log), _ptr(dt_bias), float(lower_bound),
                              _ptr(initial_state), _ptr(final_state), code, _ptr(cu_seqlens),
                              num_seqs, B, T, H, K, V, _stream_handle(stream))
    if st != KDA_OK:
        raise KDAError(st, status_string(st))


def kda_bwd(q, k, v, g, beta, scale, A_log, dt_bias, lower_bound, dout, initial_state=None,
            dfinal=None, cu_seqlens=None, want_dinit=True, stream=None) -> dict:
    """Gradients of L = sum(dout * out) + sum(dfinal * final_state) through libkda.so's
    kda_bwd, with respect to the inputs of ``kda_fwd`` (``lower_bound=None``: the gate
    without a lower bound).  ``dout`` bf16 [B,T,H,V]; ``dfinal`` fp32 [N,H,V,K] or None.
    Returns a dict of new fp32 CUDA tensors: dq, dk, dv, dg, dbeta (of the beta logits),
    dA_log, ddt_bias and dinit (None unless ``want_dinit``); asynchronous on ``stream``."""
    if q.dim() != 4:
        raise ValueError("q must be [B, T, H, K]")
    B, T, H, K = q.shape
    V = v.shape[-1] if v.dim() == 4 else -1
    for name, t, shape in (("q", q, None), ("k", k, (B, T, H, K)), ("g", g, (B, T, H, K)),
                           ("v", v, (B, T, H, V)), ("beta", beta, (B, T, H)),
                           ("dout", dout, (B, T, H, V))):
        _check_tensor(name, t, torch.bfloat16, shape)
    _check_tensor("A_log", A_log, torch.float32, (H,))
    _check_tensor("dt_bias", dt_bias, torch.float32, (H, K))
    num_seqs = 0
    if cu_seqlens is not None:
        _check_tensor("cu_seqlens", cu_seqlens, torch.int64)
        if cu_seqlens.dim() != 1 or cu_seqlens.numel() < 2:
            raise ValueError("cu_seqlens must be 1-D with at least 2 entries")
        num_seqs = cu_seqlens.numel() - 1
    N = num_seqs if cu_seqlens is not None else B
    code = state_dtype_code(initial_state, None)
    if initial_state is not None:
        _check_tensor("initial_state", initial_state, initial_state.dtype, (N, H, V, K))
    if dfinal is not None:
        _check_tensor("dfinal", dfinal, torch.float32, (N, H, V, K))
    dev = q.device
    r = {"dq": torch.empty((B, T, H, K), dtype=torch.float32, device=dev),
         "dk": torch.empty((B, T, H, K), dtype=torch.float32, device=dev),
         "dv": torch.empty((B, T, H, V), dtype=torch.float32, device=dev),
         "dg": torch.empty((B, T, H, K), dtype=torch.float32, device=dev),
         "dbeta": torch.empty((B, T, H), dtype=torch.float32, device=dev),
         "dA_log": torch.empty((H,), dtype=torch.float32, device=dev),
         "ddt_bias": torch.empty((H, K), dtype=torch.float32, device=dev),
         "dinit": torch.empty((N, H, V, K), dtype=torch.float32, device=dev) if want_dinit else None}
    unb = lower_bound is None
    st = lib().kda_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale), _ptr(A_log),
                       _ptr(dt_bias), 0.0 if unb else float(lower_bound), 1 if unb else 0,
                       _ptr(initial_state), code, _ptr(dout), _ptr(dfinal), _ptr(cu_seqlens),
                       num_seqs, B, T, H, K, V, _ptr(r["dq"]), _ptr(r["dk"]), _ptr(r["dv"]),
                       _ptr(r["dg"]), _ptr(r["dbeta"]), _ptr(r["dA_log"]), _ptr(r["ddt_bias"]),
                       _ptr(r["dinit"]), _stream_handle(stream))
    if st != KDA_OK:
        raise KDAError(st, status_string(st))
    return r


def get_device_status(stream=None) -> int:
    """Synchronise ``stream`` and return (and clear) the device error word."""
    return int(lib().kda_get_device_status(_stream_handle(stream)))


def raw_call(*args):
    """Direct call of the C entry point with already-marshalled arguments (checks of
    the validation path use this with host-side fake pointers; nothing is launched
    when validation fails)."""
    return int(lib().kda_fwd(*args))


def raw_call_ws(*args):
    """Direct call of kda_fwd_ws with already-marshalled arguments (validation checks)."""
    return int(lib().kda_fwd_ws(*args))
