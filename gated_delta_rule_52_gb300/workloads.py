"""Seeded synthetic inputs for the KDA forward workloads.

This module only draws random numbers and lays them out; it holds none of the
method's arithmetic (no gate, no normalisation, no recurrence).  Both the fp64
reference and the CUDA path take their inputs from here, so the two sides see
identical bf16/fp32 values.

Shapes and dtypes follow the FlashKDA README's Kernel API table ("Kernel API",
flash_kda.fwd parameter list): q, k, g bf16 [B,T,H,K]; v bf16 [B,T,H,V]; beta
logits bf16 [B,T,H]; A_log fp32 [H]; dt_bias fp32 [H,K]; optional recurrent state
[B|N,H,V,K] in bf16 or fp32; cu_seqlens int64 [N+1] with B=1.

Draw order for one workload, all from one CPU ``torch.Generator`` seeded with the
workload's seed: sequence lengths (ragged varlen only), q, k, v, g, beta, A_log,
dt_bias, initial_state, lower_bound.  Normal draws are fp32 ``randn`` scaled by the
standard deviation and shifted by the mean, then rounded to bf16 where the tensor
is bf16.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace
from typing import Optional

import torch

HEAD_DIM = 128


@dataclass(frozen=True)
class Workload:
    """One synthetic KDA forward problem (sizes and input distributions)."""

    name: str
    B: int
    T: int
    H: int
    K: int = HEAD_DIM
    V: int = HEAD_DIM
    seed: int = 0
    # varlen: "uniform" -> n_seqs equal lengths; "ragged" -> log-uniform lengths
    varlen: Optional[str] = None
    n_seqs: int = 0
    seqlens: Optional[tuple] = None          # explicit lengths (overrides varlen draw)
    lower_bound: Optional[float] = -5.0      # None: the gate without a lower bound (softplus)
    lower_bound_range: Optional[tuple] = None  # draw lb ~ U[lo, hi] if set
    state_dtype: Optional[str] = None        # None | "fp32" | "bf16"
    initial_state: str = "none"              # "none" | "normal" | "alternate" (zeros on even seqs)
    state_std: float = 0.02
    g_std: float = 1.0
    beta_mean: float = 0.0
    ragged_total: Optional[tuple] = None     # accepted total-token window for ragged draws
    ragged_len_range: tuple = (17, 16384)
    description: str = ""

    @property
    def n_states(self) -> int:
        return self.n_seqs if self.varlen else self.B


# The five workloads: tiny, carried-state batch, long prefill (throughput
# workload), uniform varlen, ragged varlen.
WORKLOADS = {
    "tiny": Workload(
        name="tiny", B=1, T=256, H=2, seed=0, state_dtype="fp32", initial_state="none",
        description="B=1 T=256 H=2; no initial state; fp32 final state"),
    "batch_state": Workload(
        name="batch_state", B=4, T=2048, H=16, seed=1, state_dtype="fp32", initial_state="normal",
        description="B=4 T=2048 H=16; fp32 initial/final state N(0,0.02)"),
    "prefill_8k": Workload(
        name="prefill_8k", B=1, T=8192, H=64, seed=2, state_dtype="bf16", initial_state="normal",
        description="B=1 T=8192 H=64; bf16 initial/final state N(0,0.02)"),
    "varlen_uniform": Workload(
        name="varlen_uniform", B=1, T=8192, H=64, seed=3, varlen="uniform", n_seqs=8,
        lower_bound_range=(-5.0, -0.5), state_dtype="fp32", initial_state="normal",
        description="cu_seqlens 8 x 1024 (T=8192) H=64; fp32 state; lb ~ U[-5,-0.5]"),
    "varlen_ragged": Workload(
        name="varlen_ragged", B=1, T=0, H=32, seed=4, varlen="ragged", n_seqs=32,
        state_dtype="fp32", initial_state="alternate", g_std=2.0, beta_mean=2.0,
        ragged_total=(117965, 144179),
        description="32 log-uniform lengths in [17,16384] (~131K tokens) H=32; fp32 state; "
                    "zeros/N(0,0.02) alternating initial state; g~N(0,2); beta~N(2,1)"),
    # Short steps (the token-recurrence kernel): one decode token for 64 sequences with
    # their fp32 recurrent states, and a 16-token step.
    "decode": Workload(
        name="decode", B=64, T=1, H=64, seed=5, state_dtype="fp32", initial_state="normal",
        description="B=64 T=1 H=64 (one decode token per sequence); fp32 state N(0,0.02)"),
    "decode_16": Workload(
        name="decode_16", B=64, T=16, H=64, seed=6, state_dtype="bf16", initial_state="normal",
        description="B=64 T=16 H=64 (16-token step); bf16 state N(0,0.02)"),
    # A 64-token step (e.g. verifying a speculative draft, or a small prefill chunk) for
    # 64 sequences: the 16-row-block kernel, four blocks per (sequence, head).
    "step_64": Workload(
        name="step_64", B=64, T=64, H=64, seed=8, state_dtype="bf16", initial_state="normal",
        description="B=64 T=64 H=64 (64-token step); bf16 state N(0,0.02)"),
    # A serving batch of short prompts: 512 sequences of 1..64 tokens (log-uniform), the
    # 16-row-block kernel for every one of them.
    "varlen_short": Workload(
        name="varlen_short", B=1, T=0, H=32, seed=9, varlen="ragged", n_seqs=512,
        ragged_len_range=(1, 64), state_dtype="fp32", initial_state="normal",
        description="512 log-uniform lengths in [1,64] H=32; fp32 state N(0,0.02)"),
    # A long prefill with few heads (e.g. 8 heads on one GPU of a tensor-parallel group):
    # 8 (sequence, head) units, the sequence-parallel path.
    "prefill_64k_h8": Workload(
        name="prefill_64k_h8", B=1, T=65536, H=8, seed=7, state_dtype="bf16", initial_state="normal",
        description="B=1 T=65536 H=8; bf16 initial/final state N(0,0.02)"),
    # The long prefill with the gate that has no lower bound (softplus), which runs the
    # token recurrence instead of the chunked kernel.
    "prefill_8k_unbounded": Workload(
        name="prefill_8k_unbounded", B=1, T=8192, H=64, seed=10, lower_bound=None,
        state_dtype="bf16", initial_state="normal",
        description="B=1 T=8192 H=64, gate without a lower bound; bf16 state N(0,0.02)"),
}

# The throughput workload timed by bench.py.
HEADLINE = "prefill_8k"


def get(name: str, **overrides) -> Workload:
    """Return a named workload, optionally with fields replaced (e.g. smaller T or H)."""
    w = WORKLOADS[name]
    return replace(w, **overrides) if overrides else w


def _normal(gen, shape, std=1.0, mean=0.0):
    x = torch.randn(shape, generator=gen, dtype=torch.float32)
    if std != 1.0:
        x = x * std
    if mean != 0.0:
        x = x + mean
    return x


def _ragged_lengths(gen, n, lo, hi, window):
    """Log-uniform integer lengths in [lo, hi], none a multiple of 64; the whole set is
    redrawn from the continuing generator until its total falls inside ``window``."""
    for _ in range(100000):
        u = torch.rand((n,), generator=gen, dtype=torch.float64)
        lens = torch.floor(torch.exp(math.log(lo) + u * (math.log(hi) - math.log(lo)))).long()
        lens = lens.clamp(lo, hi)
        out = []
        for L in lens.tolist():
            if L % 64 == 0:
                L = L - 1 if L + 1 > hi else L + 1
            out.append(int(L))
        if window is None or window[0] <= sum(out) <= window[1]:
            return out
    raise RuntimeError("could not draw ragged lengths inside the requested window")


def seqlens_of(w: Workload, gen=None) -> Optional[list]:
    if not w.varlen:
        return None
    if w.seqlens is not None:
        return list(w.seqlens)
    if w.varlen == "uniform":
        assert w.T % w.n_seqs == 0
        return [w.T // w.n_seqs] * w.n_seqs
    assert gen is not None
    return _ragged_lengths(gen, w.n_seqs, w.ragged_len_range[0], w.ragged_len_range[1], w.ragged_total)


def make_inputs(w: Workload, device="cpu") -> dict:
    """Draw every input of workload ``w``.  Returns a dict with keys q, k, v, g, beta
    (bf16), A_log, dt_bias (fp32), scale, lower_bound (python floats),
    initial_state (tensor or None), state_dtype (None/"fp32"/"bf16"),
    cu_seqlens (int64 tensor or None), seqlens (list or None), B, T, H, K, V, N."""
    gen = torch.Generator(device="cpu")
    gen.manual_seed(w.seed)
    lens = seqlens_of(w, gen)
    if lens is not None:
        B, T = 1, int(sum(lens))
        cu = torch.zeros(len(lens) + 1, dtype=torch.int64)
        cu[1:] = torch.cumsum(torch.tensor(lens, dtype=torch.int64), 0)
    else:
        B, T, cu = w.B, w.T, None
    H, K, V = w.H, w.K, w.V
    q = _normal(gen, (B, T, H, K)).to(torch.bfloat16)
    k = _normal(gen, (B, T, H, K)).to(torch.bfloat16)
    v = _normal(gen, (B, T, H, V)).to(torch.bfloat16)
    g = _normal(gen, (B, T, H, K), std=w.g_std).to(torch.bfloat16)
    beta = _normal(gen, (B, T, H), mean=w.beta_mean).to(torch.bfloat16)
    A_log = torch.log(1.0 + 15.0 * torch.rand((H,), generator=gen, dtype=torch.float32))
    dt_bias = _normal(gen, (H, K), std=0.1)
    N = len(lens) if lens is not None else B
    init = None
    if w.initial_state != "none":
        s = _normal(gen, (N, H, V, K), std=w.state_std)
        if w.initial_state == "alternate":
            s[0::2] = 0.0
        init = s.to(torch.bfloat16) if w.state_dtype == "bf16" else s
    if w.lower_bound_range is not None:
        lo, hi = w.lower_bound_range
        lb = float(lo + (hi - lo) * torch.rand((), generator=gen, dtype=torch.float64).item())
    else:
        lb = None if w.lower_bound is None else float(w.lower_bound)
    d = dict(q=q, k=k, v=v, g=g, beta=beta, A_log=A_log, dt_bias=dt_bias,
             scale=1.0 / math.sqrt(K), lower_bound=lb, initial_state=init,
             state_dtype=w.state_dtype, cu_seqlens=cu, seqlens=lens,
             B=B, T=T, H=H, K=K, V=V, N=N)
    if device != "cpu":
        for key in ("q", "k", "v", "g", "beta", "A_log", "dt_bias", "initial_state", "cu_seqlens"):
            if d[key] is not None:
                d[key] = d[key].to(device)
    return d


def token_heads(d: dict) -> int:
    """Number of (token, head) pairs in an input set."""
    return int(d["B"] * d["T"] * d["H"])
