"""Naive chunked (UT/WY) form of the KDA recurrence in numpy fp64.

An independent route to the same result as the oracle's token loop, used only to
pin the oracle.  Per chunk of C tokens with entering state S0 (K x V), cumulative
log decay G_r = sum_{s<=r} gk_s (per channel):

  A[t,i] = beta_t * sum_c k[t,c] k[i,c] exp(G[t,c]-G[i,c])      (i < t)
  M[t,i] =          sum_c q[t,c] k[i,c] exp(G[t,c]-G[i,c])      (i <= t)
  Tinv   = (I + A)^-1
  W      = Tinv @ (beta * k * exp(G)),   Ut = Tinv @ (beta * v)
  U      = Ut - W @ S0
  O      = scale * ((q * exp(G)) @ S0 + M @ U)
  S_C    = exp(G_C) * S0 + (k * exp(G_C - G)).T @ U

Derived by unrolling S_r = (I - b k k^T) Diag(exp(gk_r)) S_{r-1} + b k v^T inside
the chunk (u_r = beta_r (v_r - S_{r-1}^T (alpha_r * k_r)) satisfies (I+A)U =
beta V - beta (K*Gamma) S0).  Every exponent used is <= 0, so nothing overflows.
"""
import numpy as np


def chunked_pair(q, k, v, gk, beta, scale, S0, C):
    """One (sequence, head): q,k,gk [L,K], v [L,V], beta [L]; S0 [K,V].
    Returns (out [L,V], S_final [K,V])."""
    L = q.shape[0]
    S = S0.copy()
    out = np.zeros((L, v.shape[1]))
    for s in range(0, L, C):
        e = min(s + C, L)
        qc, kc, vc, gc, bc = q[s:e], k[s:e], v[s:e], gk[s:e], beta[s:e]
        n = e - s
        G = np.cumsum(gc, axis=0)
        A = np.zeros((n, n))
        M = np.zeros((n, n))
        for t in range(n):
            for i in range(t + 1):
                dec = np.exp(G[t] - G[i])
                M[t, i] = np.sum(qc[t] * kc[i] * dec)
                if i < t:
                    A[t, i] = bc[t] * np.sum(kc[t] * kc[i] * dec)
        Tinv = np.linalg.inv(np.eye(n) + A)
        W = Tinv @ (bc[:, None] * kc * np.exp(G))
        Ut = Tinv @ (bc[:, None] * vc)
        U = Ut - W @ S
        out[s:e] = scale * ((qc * np.exp(G)) @ S + M @ U)
        S = np.exp(G[-1])[:, None] * S + (kc * np.exp(G[-1][None, :] - G)).T @ U
    return out, S
