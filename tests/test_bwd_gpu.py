"""kda_bwd (the gradients of the forward) against the fp64 backward oracle, element by
element, through the C ABI.

Bars: every gradient tensor within a relative L2 error of 2e-5 of the oracle's, and
dA_log / ddt_bias (sums over every token of a head, where terms cancel) within 1e-4.
The kernel runs the recurrence and its reverse in fp32 on exactly the oracle's inputs
(bf16 values widen exactly), so its error is fp32 rounding accumulated over the tokens:
1e-7 to 4e-7 on these cases on a GB300; the bars leave room for longer sequences.
"""
import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_52_gb300 import kda
from gated_delta_rule_52_gb300 import workloads as W

pytestmark = pytest.mark.gpu

TOL = 2e-5
TOL_SUM = 1e-4


def _upstream(d, seed, with_dfinal=True):
    g = torch.Generator().manual_seed(seed)
    dout = torch.randn(d["v"].shape, generator=g).to(torch.bfloat16)
    dfin = torch.randn((d["N"], d["H"], 128, 128), generator=g) if with_dfinal else None
    return dout, dfin


def _run(d, dout, dfin):
    e = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in d.items()}
    r = kda.kda_bwd(e["q"], e["k"], e["v"], e["g"], e["beta"], d["scale"], e["A_log"], e["dt_bias"],
                    d["lower_bound"], dout.cuda(), initial_state=e["initial_state"],
                    dfinal=None if dfin is None else dfin.cuda(), cu_seqlens=e["cu_seqlens"])
    torch.cuda.synchronize()
    assert kda.get_device_status() == kda.KDA_OK
    return {k: (None if v is None else v.cpu().double().numpy()) for k, v in r.items()}


def _ref(d, dout, dfin):
    return oracle.kda_bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["scale"], d["A_log"],
                          d["dt_bias"], d["lower_bound"], dout, initial_state=d["initial_state"],
                          dfinal=dfin, cu_seqlens=d["cu_seqlens"])


def _check(got, ref, label):
    errs = {}
    for name, r in ref.items():
        if r is None:
            continue
        gv = got[name]
        assert np.all(np.isfinite(gv)), f"{label}: {name} not finite"
        den = np.linalg.norm(r)
        rel = np.linalg.norm(gv - r) / den if den > 0 else np.linalg.norm(gv)
        errs[name] = rel
        bar = TOL_SUM if name in ("dA_log", "ddt_bias") else TOL
        assert rel <= bar, f"{label}: {name} rel-L2 {rel:.3e} > {bar}"
    return errs


@pytest.mark.parametrize("B,T,H,sd,init,unbounded", [(2, 300, 3, "fp32", "normal", False),
                                                      (1, 129, 2, "bf16", "normal", False),
                                                      (2, 64, 2, None, "none", False),
                                                      (1, 1, 2, "fp32", "normal", False),
                                                      (2, 300, 2, "fp32", "normal", True),
                                                      (3, 70, 2, "bf16", "normal", True)])
def test_bwd_all_elements(B, T, H, sd, init, unbounded):
    d = W.make_inputs(W.get("tiny", B=B, T=T, H=H, state_dtype=sd, initial_state=init, g_std=1.5,
                            lower_bound=None if unbounded else -5.0, seed=120 + T + H))
    dout, dfin = _upstream(d, 7 + T, with_dfinal=sd is not None)
    got, ref = _run(d, dout, dfin), _ref(d, dout, dfin)
    print("bwd", B, T, H, sd, unbounded, _check(got, ref, f"bwd T={T}"))


def test_bwd_varlen_with_empty_sequences():
    seqlens = (0, 65, 1, 200, 0, 64, 130)
    for lb in (-3.0, None):
        d = W.make_inputs(W.get("varlen_ragged", H=2, seqlens=seqlens, lower_bound=lb, seed=131))
        dout, dfin = _upstream(d, 11)
        got, ref = _run(d, dout, dfin), _ref(d, dout, dfin)
        print("bwd varlen", lb, _check(got, ref, f"bwd varlen lb={lb}"))
        # an empty sequence passes the final-state gradient straight to the initial state
        for n in (0, 4):
            np.testing.assert_allclose(got["dinit"][n], dfin[n].double().numpy(), rtol=0, atol=0)


def test_bwd_longer_sequence_more_heads():
    # many chunks (checkpoints, recomputation, the reverse sweep) and a ragged tail
    d = W.make_inputs(W.get("prefill_8k", T=2100, H=4, state_dtype="fp32", seed=133))
    dout, dfin = _upstream(d, 13)
    got, ref = _run(d, dout, dfin), _ref(d, dout, dfin)
    print("bwd T=2100", _check(got, ref, "bwd T=2100"))


def test_bwd_more_units_than_sms():
    # the state kernel is persistent over the units: 160 units on 152 SMs
    d = W.make_inputs(W.get("batch_state", B=40, T=70, H=4, seed=134))
    dout, dfin = _upstream(d, 14)
    got, ref = _run(d, dout, dfin), _ref(d, dout, dfin)
    print("bwd 160 units", _check(got, ref, "bwd 160 units"))
