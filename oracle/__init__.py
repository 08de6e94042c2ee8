"""fp64 CPU oracle for the KDA forward pass and its gradient.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this package.  The CUDA library never
imports, links or runs anything here, and this package imports nothing from the
CUDA path.

``kda_oracle.c`` holds the arithmetic (a token-by-token recurrence in fp64) and
``kda_oracle_bwd.c`` its gradient (reverse-mode differentiation of the same loop,
written out); this module compiles them with gcc and marshals numpy arrays to them.
See the files' headers for what is computed and which readings of the FlashKDA pages
they take.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_SRCS = [_SRC, os.path.join(_HERE, "kda_oracle_bwd.c")]
_LIB = os.path.join(_HERE, "libkda_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle into ``oracle/libkda_oracle.so`` (gcc, -O2, OpenMP,
    no fast-math).  Returns the library path."""
    with _lock:
        if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < max(map(os.path.getmtime, _SRCS)):
            tmp = _LIB + f".tmp{os.getpid()}"
            cmd = ["gcc", "-O2", "-fno-fast-math", "-fopenmp", "-fPIC", "-shared",
                   "-o", tmp] + _SRCS + ["-lm"]
            subprocess.run(cmd, check=True)
            os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        d, i64, ip = ctypes.c_double, ctypes.c_int64, ctypes.c_void_p
        lib.kda_oracle_fwd.argtypes = [ip, ip, ip, ip, ip, d, ip, ip, d, ip, ip, ip, ip, i64,
                                       i64, i64, i64, i64, i64, ip, i64, ctypes.c_int]
        lib.kda_oracle_fwd.restype = ctypes.c_int
        lib.kda_oracle_recurrence.argtypes = [ip, ip, ip, ip, ip, d, ip, ip, ip, ip, i64,
                                              i64, i64, i64, i64, i64, ctypes.c_int]
        lib.kda_oracle_recurrence.restype = ctypes.c_int
        lib.kda_oracle_activations.argtypes = [ip, ip, ip, ip, ip, ip, d, i64, i64, i64, i64,
                                               ip, ip, ip, ip]
        lib.kda_oracle_activations.restype = ctypes.c_int
        lib.kda_oracle_max_threads.restype = ctypes.c_int
        lib.kda_oracle_bwd.argtypes = [ip, ip, ip, ip, ip, d, ip, ip, d, ip, ip, ip, ip, i64,
                                       i64, i64, i64, i64, i64, ip, ip, ip, ip, ip, ip, ip, ip,
                                       ctypes.c_int]
        lib.kda_oracle_bwd.restype = ctypes.c_int
        _lib = lib
    return _lib


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor: exact widening of bf16/fp32 values
        import torch
        x = x.detach().to("cpu", torch.float64).numpy()
    return np.ascontiguousarray(x, dtype=np.float64)


def _i64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):
        x = x.detach().cpu().numpy()
    return np.ascontiguousarray(x, dtype=np.int64)


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _lb(lower_bound):
    """None (no lower bound: the softplus gate) travels to the C code as NaN."""
    return float("nan") if lower_bound is None else float(lower_bound)


def max_threads() -> int:
    return int(_load().kda_oracle_max_threads())


def kda_fwd(q, k, v, g, beta, scale, A_log, dt_bias, lower_bound, initial_state=None,
            cu_seqlens=None, want_final=True, pairs=None, nthreads=0):
    """Full KDA forward in fp64 from raw inputs (numpy arrays or torch tensors in the
    Kernel API layouts).  Returns ``(out, final_state)`` as fp64 numpy arrays;
    ``final_state`` is None when ``want_final`` is false.  ``pairs`` (optional, a list
    of (sequence, head)) restricts the work; other outputs stay NaN.  ``lower_bound``
    None selects the gate without a lower bound (softplus; see kda_oracle.c)."""
    lib = _load()
    q, k, v, g, beta = _f64(q), _f64(k), _f64(v), _f64(g), _f64(beta)
    A_log, dt_bias, init = _f64(A_log), _f64(dt_bias), _f64(initial_state)
    cu = _i64(cu_seqlens)
    B, T, H, K = q.shape
    V = v.shape[-1]
    N = (cu.shape[0] - 1) if cu is not None else B
    out = np.full((B, T, H, V), np.nan)
    fin = np.full((N, H, V, K), np.nan) if want_final else None
    pr = None
    if pairs is not None:
        pr = np.ascontiguousarray(np.asarray(pairs, dtype=np.int64).reshape(-1, 2))
    rc = lib.kda_oracle_fwd(_p(q), _p(k), _p(v), _p(g), _p(beta), float(scale), _p(A_log),
                            _p(dt_bias), _lb(lower_bound), _p(init), _p(fin), _p(out), _p(cu),
                            N if cu is not None else 0, B, T, H, K, V, _p(pr),
                            0 if pr is None else pr.shape[0], int(nthreads))
    if rc:
        raise ValueError(f"oracle rejected the sizes or cu_seqlens (code {rc})")
    return out, fin


def recurrence(q, k, v, gk, beta, scale, initial_state=None, cu_seqlens=None, want_final=True,
               nthreads=0):
    """The recurrence alone on activated inputs: q, k used as given (no norm), gk the
    per-channel log decay [B,T,H,K], beta the post-sigmoid beta [B,T,H]."""
    lib = _load()
    q, k, v, gk, beta, init = _f64(q), _f64(k), _f64(v), _f64(gk), _f64(beta), _f64(initial_state)
    cu = _i64(cu_seqlens)
    B, T, H, K = q.shape
    V = v.shape[-1]
    N = (cu.shape[0] - 1) if cu is not None else B
    out = np.full((B, T, H, V), np.nan)
    fin = np.full((N, H, V, K), np.nan) if want_final else None
    rc = lib.kda_oracle_recurrence(_p(q), _p(k), _p(v), _p(gk), _p(beta), float(scale), _p(init),
                                   _p(fin), _p(out), _p(cu), N if cu is not None else 0,
                                   B, T, H, K, V, int(nthreads))
    if rc:
        raise ValueError(f"oracle rejected the sizes or cu_seqlens (code {rc})")
    return out, fin


def activations(q, k, g, beta, A_log, dt_bias, lower_bound):
    """The prologue alone: returns (q_hat, k_hat, gk, beta) in fp64."""
    lib = _load()
    q, k, g, beta, A_log, dt_bias = _f64(q), _f64(k), _f64(g), _f64(beta), _f64(A_log), _f64(dt_bias)
    B, T, H, K = q.shape
    qn, kn, gk = np.empty_like(q), np.empty_like(k), np.empty_like(g)
    bo = np.empty_like(beta)
    rc = lib.kda_oracle_activations(_p(q), _p(k), _p(g), _p(beta), _p(A_log), _p(dt_bias),
                                    _lb(lower_bound), B, T, H, K, _p(qn), _p(kn), _p(gk), _p(bo))
    if rc:
        raise ValueError("oracle rejected the sizes")
    return qn, kn, gk, bo


def kda_bwd(q, k, v, g, beta, scale, A_log, dt_bias, lower_bound, dout, initial_state=None,
            dfinal=None, cu_seqlens=None, want_dinit=True, nthreads=0):
    """Gradients of L = sum(dout * out) + sum(dfinal * final_state) with respect to the
    inputs of ``kda_fwd`` (same layouts), fp64.  Returns a dict with dq, dk, dv, dg,
    dbeta (of the beta logits), dA_log, ddt_bias and dinit (the initial state's gradient,
    None unless ``want_dinit``)."""
    lib = _load()
    q, k, v, g, beta = _f64(q), _f64(k), _f64(v), _f64(g), _f64(beta)
    A_log, dt_bias, init = _f64(A_log), _f64(dt_bias), _f64(initial_state)
    dout, dfin, cu = _f64(dout), _f64(dfinal), _i64(cu_seqlens)
    B, T, H, K = q.shape
    V = v.shape[-1]
    N = (cu.shape[0] - 1) if cu is not None else B
    r = {"dq": np.zeros((B, T, H, K)), "dk": np.zeros((B, T, H, K)), "dv": np.zeros((B, T, H, V)),
         "dg": np.zeros((B, T, H, K)), "dbeta": np.zeros((B, T, H)), "dA_log": np.zeros(H),
         "ddt_bias": np.zeros((H, K)), "dinit": np.zeros((N, H, V, K)) if want_dinit else None}
    rc = lib.kda_oracle_bwd(_p(q), _p(k), _p(v), _p(g), _p(beta), float(scale), _p(A_log),
                            _p(dt_bias), _lb(lower_bound), _p(init), _p(dout), _p(dfin), _p(cu),
                            N if cu is not None else 0, B, T, H, K, V, _p(r["dq"]), _p(r["dk"]),
                            _p(r["dv"]), _p(r["dg"]), _p(r["dbeta"]), _p(r["dA_log"]),
                            _p(r["ddt_bias"]), _p(r["dinit"]), int(nthreads))
    if rc:
        raise ValueError(f"oracle rejected the sizes or cu_seqlens (code {rc})")
    return r
