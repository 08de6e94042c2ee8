"""A numpy model of the decay-factor arithmetic of the pool kernel's front (CPU only).

The front forms A and M of a 64-token chunk as bf16 GEMMs of factored operands: the
rows k 2^(H - mu), q 2^(H - mu), the key variants 2^(mu - H) k for the diagonal 16-token
block and, for a later row block bt, 2^(mu - H) k times 2^mu (giving 2^(Gs[b+1] - G) k,
at most 1) times the table entry 2^(Gs[bt] - Gs[b+1] + mu[bt]).  mu is half a block's
total decay for the gate without a lower bound and 0 with it.  This model rounds where
the kernel rounds (fp32 exponentials and products, bf16 operands, fp32 sums) and
checks the products against the exact exp(G_t - G_i) sums:
  - the kernel's form keeps A and M at bf16 level (below 1e-2 relative) for both gates,
    with each token's log2 decay floored at -14 for the gate without a lower bound;
  - putting the later-block variant in one table entry, 2^(Gs[bt] - Gs[b] + mu[bt] -
    mu[b]), underflows where two blocks both decay strongly, although the product does
    not: it fails for the gate without a lower bound.
"""
import numpy as np
import pytest
import torch

from gated_delta_rule_52_gb300 import workloads as W

L2E = 1.0 / np.log(2.0)


def _bf16(x):
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).to(torch.float64).numpy()


def _f32(x):
    return np.asarray(x, dtype=np.float32).astype(np.float64)


def _chunk_errors(qc, kc, gk2, unbounded, two_step):
    n = qc.shape[0]
    G = np.cumsum(gk2, 0)                       # exact cumulative decay (log2)
    H = np.zeros_like(gk2)
    btot = np.zeros((4, gk2.shape[1]))
    for b in range(4):
        H[16 * b:16 * b + 16] = np.cumsum(gk2[16 * b:16 * b + 16], 0)
        btot[b] = gk2[16 * b:16 * b + 16].sum(0)
    Gs = np.concatenate([np.zeros((1, gk2.shape[1])), np.cumsum(btot, 0)[:-1]], 0)
    mu = 0.5 * btot if unbounded else np.zeros_like(btot)
    blk = np.arange(n) // 16
    Hs = H - mu[blk]
    e1, e2 = _f32(np.exp2(Hs)), _f32(np.exp2(-Hs))
    Kp, Qp, kn = _bf16(kc * e1), _bf16(qc * e1), _f32(kc * e2)
    A, M = np.zeros((n, n)), np.zeros((n, n))
    for bt in range(4):
        rows = slice(16 * bt, 16 * bt + 16)
        cols = np.zeros((16 * bt + 16, kc.shape[1]))
        for bi in range(bt + 1):
            ci = slice(16 * bi, 16 * bi + 16)
            if bi == bt:
                cols[ci] = _bf16(kn[ci])
            elif two_step:
                t2 = _f32(np.exp2(Gs[bt] - (Gs[bi] + 2 * mu[bi]) + mu[bt]))
                cols[ci] = _bf16(_f32(_f32(kn[ci] * _f32(np.exp2(mu[bi]))) * t2))
            else:
                fac = _f32(np.exp2(Gs[bt] - Gs[bi] + mu[bt] - mu[bi]))
                cols[ci] = _bf16(_f32(kn[ci] * fac))
        A[rows, :16 * bt + 16] = Kp[rows] @ cols.T
        M[rows, :16 * bt + 16] = Qp[rows] @ cols.T
    dec = np.exp2(G[:, None, :] - G[None, :, :])            # [t, i, c], used for i <= t only
    Ax = np.einsum("tc,ic,tic->ti", kc, kc, np.where(np.tril(np.ones((n, n)), -1)[..., None] > 0, dec, 0.0))
    Mx = np.einsum("tc,ic,tic->ti", qc, kc, np.where(np.tril(np.ones((n, n)))[..., None] > 0, dec, 0.0))
    A = np.tril(A, -1)
    M = np.tril(M)
    return (np.linalg.norm(A - Ax) / np.linalg.norm(Ax), np.linalg.norm(M - Mx) / np.linalg.norm(Mx))


def _worst(unbounded, two_step):
    d = W.make_inputs(W.get("tiny", B=2, T=256, H=3, state_dtype="fp32", initial_state="normal",
                            g_std=1.0, lower_bound=None if unbounded else -5.0, seed=340))
    q, k, g = d["q"].double().numpy(), d["k"].double().numpy(), d["g"].double().numpy()
    A_log, dtb = d["A_log"].double().numpy(), d["dt_bias"].double().numpy()
    worst = 0.0
    for b in range(2):
        for h in range(3):
            for ch in range(4):
                sl = slice(64 * ch, 64 * ch + 64)
                x = g[b, sl, h] + dtb[h]
                if unbounded:   # -exp(A_log) softplus, in log2 units, floored at -14 per token
                    sp2 = np.maximum(x * L2E, 0) + np.log2(1 + np.exp2(-np.abs(x * L2E)))
                    gk2 = np.maximum(-np.exp(A_log[h]) * sp2, -14.0)
                else:
                    gk2 = -5.0 * L2E / (1 + np.exp(-np.exp(A_log[h]) * x))
                ea, em = _chunk_errors(q[b, sl, h], k[b, sl, h], _f32(gk2), unbounded, two_step)
                worst = max(worst, ea, em)
    return worst


@pytest.mark.parametrize("unbounded", [False, True])
def test_kernel_factor_form_keeps_bf16_accuracy(unbounded):
    assert _worst(unbounded, two_step=True) < 1e-2


def test_single_entry_variants_fail_without_a_lower_bound():
    assert _worst(False, two_step=False) < 1e-2    # with the lower bound both forms hold
    assert _worst(True, two_step=False) > 1e-1     # the underflowing entry loses terms
