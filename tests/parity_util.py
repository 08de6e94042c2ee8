"""Helpers for GPU-vs-oracle parity tests: run the CUDA path through the C ABI,
run the oracle on the same inputs, compare with the stated tolerances.

Tolerances (fp32 accumulation, bf16 operands and bf16 output):
  out          max |err| <= 2e-2  and  ||err||_2 / ||ref||_2 <= 5e-3
  final_state  ||err||_2 / ||ref||_2 <= 1e-3 (fp32 state), <= 1e-2 (bf16 state)
"""
import numpy as np
import torch

import oracle
from gated_delta_rule_52_gb300 import kda

OUT_MAX_ABS = 2e-2
OUT_REL_L2 = 5e-3
STATE_REL_L2 = {"fp32": 1e-3, "bf16": 1e-2}


def to_device(d, device="cuda"):
    e = dict(d)
    for key in ("q", "k", "v", "g", "beta", "A_log", "dt_bias", "initial_state", "cu_seqlens"):
        if e[key] is not None:
            e[key] = e[key].to(device)
    return e


def state_torch_dtype(sd):
    return {"fp32": torch.float32, "bf16": torch.bfloat16}[sd]


def run_gpu(d, want_final=True, stream=None, fill=float("nan")):
    """Runs libkda on the inputs in ``d`` (CPU tensors); returns (out, final) on CPU."""
    e = to_device(d)
    out = torch.full((d["B"], d["T"], d["H"], d["V"]), fill, dtype=torch.bfloat16, device="cuda")
    fin = None
    if want_final and d["state_dtype"] is not None:
        fin = torch.full((d["N"], d["H"], d["V"], d["K"]), fill,
                         dtype=state_torch_dtype(d["state_dtype"]), device="cuda")
    kda.kda_fwd(e["q"], e["k"], e["v"], e["g"], e["beta"], d["scale"], out, e["A_log"],
                e["dt_bias"], d["lower_bound"], initial_state=e["initial_state"],
                final_state=fin, cu_seqlens=e["cu_seqlens"], stream=stream)
    assert kda.get_device_status(stream) == kda.KDA_OK
    return out.cpu(), (fin.cpu() if fin is not None else None)


def run_oracle(d, pairs=None, want_final=True):
    return oracle.kda_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["scale"], d["A_log"],
                          d["dt_bias"], d["lower_bound"], initial_state=d["initial_state"],
                          cu_seqlens=d["cu_seqlens"], want_final=want_final, pairs=pairs)


def errors(got, ref):
    got = np.asarray(got, dtype=np.float64).ravel()
    ref = np.asarray(ref, dtype=np.float64).ravel()
    diff = got - ref
    nref = np.linalg.norm(ref)
    return float(np.max(np.abs(diff))) if diff.size else 0.0, \
        float(np.linalg.norm(diff) / nref) if nref > 0 else float(np.linalg.norm(diff))


def token_slices(d):
    """(batch row, token slice) of every sequence."""
    if d["cu_seqlens"] is None:
        return [(b, slice(0, d["T"])) for b in range(d["B"])]
    cu = d["cu_seqlens"].tolist()
    return [(0, slice(cu[n], cu[n + 1])) for n in range(len(cu) - 1)]


def gather_pairs(arr_out, arr_fin, d, pairs):
    """Concatenate the outputs (and final states) of the listed (sequence, head) pairs."""
    sl = token_slices(d)
    outs, fins = [], []
    for n, h in pairs:
        b, s = sl[n]
        outs.append(np.asarray(arr_out[b, s, h], dtype=np.float64).reshape(-1))
        if arr_fin is not None:
            fins.append(np.asarray(arr_fin[n, h], dtype=np.float64).reshape(-1))
    return np.concatenate(outs), (np.concatenate(fins) if fins else None)


def check(d, got_out, got_fin, ref_out, ref_fin, pairs=None, label=""):
    """Asserts the tolerances; returns the error figures."""
    go, gf = got_out.float().numpy(), (got_fin.float().numpy() if got_fin is not None else None)
    if pairs is not None:
        go, gf = gather_pairs(go, gf, d, pairs)
        ro, rf = gather_pairs(ref_out, ref_fin if gf is not None else None, d, pairs)
    else:
        ro, rf = ref_out, ref_fin
    assert np.all(np.isfinite(go)), f"{label}: non-finite output"
    mx, rl = errors(go, ro)
    res = {"out_max_abs": mx, "out_rel_l2": rl}
    assert mx <= OUT_MAX_ABS, f"{label}: out max-abs {mx:.3e} > {OUT_MAX_ABS}"
    assert rl <= OUT_REL_L2, f"{label}: out rel-L2 {rl:.3e} > {OUT_REL_L2}"
    if gf is not None:
        assert np.all(np.isfinite(gf)), f"{label}: non-finite final state"
        _, srl = errors(gf, rf)
        res["state_rel_l2"] = srl
        tol = STATE_REL_L2[d["state_dtype"]]
        assert srl <= tol, f"{label}: final_state rel-L2 {srl:.3e} > {tol}"
    return res


def check_full(d, got_out, got_fin, label="", max_tokens=16384):
    """Compares every element of a full-size call with the oracle, one batch row (or a
    group of whole varlen sequences of at most ``max_tokens`` packed tokens) at a time, so
    that the fp64 copies stay small; the error figures are those of the whole tensors."""
    go = got_out.float()
    gf = got_fin.float() if got_fin is not None else None
    acc = {"d_out": 0.0, "r_out": 0.0, "max": 0.0, "d_fin": 0.0, "r_fin": 0.0}

    def compare(sub, o_slice, f_slice):
        ro, rf = run_oracle(sub, want_final=f_slice is not None)
        o = o_slice.numpy().astype(np.float64)
        assert np.all(np.isfinite(o)), f"{label}: non-finite output"
        diff = o - ro
        acc["d_out"] += float(np.sum(diff * diff))
        acc["r_out"] += float(np.sum(ro * ro))
        if diff.size:
            acc["max"] = max(acc["max"], float(np.max(np.abs(diff))))
        if f_slice is not None:
            f = f_slice.numpy().astype(np.float64)
            assert np.all(np.isfinite(f)), f"{label}: non-finite final state"
            acc["d_fin"] += float(np.sum((f - rf) ** 2))
            acc["r_fin"] += float(np.sum(rf * rf))

    def sub_inputs(**over):
        e = dict(d)
        e.update(over)
        return e

    if d["cu_seqlens"] is None:
        for b in range(d["B"]):
            sl = slice(b, b + 1)
            sub = sub_inputs(B=1, N=1, q=d["q"][sl], k=d["k"][sl], v=d["v"][sl], g=d["g"][sl],
                             beta=d["beta"][sl],
                             initial_state=None if d["initial_state"] is None else d["initial_state"][sl])
            compare(sub, go[sl], None if gf is None else gf[sl])
    else:
        cu = d["cu_seqlens"].tolist()
        n = 0
        N = len(cu) - 1
        while n < N:
            m = n + 1
            while m < N and cu[m + 1] - cu[n] <= max_tokens:
                m += 1
            t0, t1 = cu[n], cu[m]
            ts = slice(t0, t1)
            sub = sub_inputs(T=t1 - t0, N=m - n, q=d["q"][:, ts], k=d["k"][:, ts], v=d["v"][:, ts],
                             g=d["g"][:, ts], beta=d["beta"][:, ts],
                             cu_seqlens=d["cu_seqlens"][n:m + 1] - t0,
                             initial_state=None if d["initial_state"] is None else d["initial_state"][n:m])
            compare(sub, go[:, ts], None if gf is None else gf[n:m])
            n = m
    rl = (acc["d_out"] ** 0.5) / (acc["r_out"] ** 0.5) if acc["r_out"] > 0 else acc["d_out"] ** 0.5
    res = {"out_max_abs": acc["max"], "out_rel_l2": rl}
    assert acc["max"] <= OUT_MAX_ABS, f"{label}: out max-abs {acc['max']:.3e} > {OUT_MAX_ABS}"
    assert rl <= OUT_REL_L2, f"{label}: out rel-L2 {rl:.3e} > {OUT_REL_L2}"
    if gf is not None:
        srl = (acc["d_fin"] ** 0.5) / (acc["r_fin"] ** 0.5) if acc["r_fin"] > 0 else acc["d_fin"] ** 0.5
        res["state_rel_l2"] = srl
        tol = STATE_REL_L2[d["state_dtype"]]
        assert srl <= tol, f"{label}: final_state rel-L2 {srl:.3e} > {tol}"
    return res
