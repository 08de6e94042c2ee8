"""kda_fwd_static, the entry point for callers that cannot allocate device memory
(an engine that reserves all of it for its own pool, a plug-in host that hands over
only the inputs and outputs).  Its scratch is a fixed array inside libkda.so, so two
calls in a row reuse what the first one left there: both must still give what
kda_fwd gives on the same inputs, within the parity tolerances.

The file name sorts last, so a run that stops at the first failure has run every
other test before this one."""
import pytest
import torch

from gated_delta_rule_52_gb300 import build as kbuild
from gated_delta_rule_52_gb300 import kda
from gated_delta_rule_52_gb300 import workloads as W
from tests.parity_util import OUT_MAX_ABS, OUT_REL_L2, STATE_REL_L2, errors, to_device

pytestmark = pytest.mark.gpu


def _outputs(d):
    out = torch.full((d["B"], d["T"], d["H"], d["V"]), float("nan"), dtype=torch.bfloat16,
                     device="cuda")
    dt = torch.bfloat16 if d["state_dtype"] == "bf16" else torch.float32
    fin = torch.full((d["N"], d["H"], d["V"], d["K"]), float("nan"), dtype=dt, device="cuda")
    return out, fin


def _call(fn, e, d, out, fin):
    fn(e["q"], e["k"], e["v"], e["g"], e["beta"], d["scale"], out, e["A_log"], e["dt_bias"],
       d["lower_bound"], initial_state=e["initial_state"], final_state=fin,
       cu_seqlens=e["cu_seqlens"])


def _close(d, got, ref):
    (go, gf), (ro, rf) = got, ref
    assert torch.isfinite(go.float()).all() and torch.isfinite(gf.float()).all()
    mx, rl = errors(go.float().cpu().numpy(), ro.float().cpu().numpy())
    assert mx <= OUT_MAX_ABS and rl <= OUT_REL_L2, (mx, rl)
    _, srl = errors(gf.float().cpu().numpy(), rf.float().cpu().numpy())
    assert srl <= STATE_REL_L2[d["state_dtype"]], srl


def test_static_scratch_entry_point_matches_kda_fwd_on_two_calls_in_a_row():
    kbuild.build_library()
    # Two different problems, both on the chunked prefill kernel (the one with
    # scratch): the second call finds the first one's data in the shared array.
    cases = [W.get("batch_state", B=2, T=700, H=8),                    # 16 units, fp32 state
             W.get("prefill_8k", T=1000, H=kda.STATIC_MAX_UNITS)]      # the unit limit, bf16 state
    results = []
    for wl in cases:
        d = W.make_inputs(wl)
        e = to_device(d)
        got = _outputs(d)
        _call(kda.kda_fwd_static, e, d, *got)
        results.append((d, e, got))
    assert kda.get_device_status() == kda.KDA_OK
    for d, e, got in results:
        ref = _outputs(d)
        _call(kda.kda_fwd, e, d, *ref)
        assert kda.get_device_status() == kda.KDA_OK
        _close(d, got, ref)


def test_static_scratch_entry_point_rejects_calls_above_its_limit():
    d = W.make_inputs(W.get("prefill_8k", T=80, H=kda.STATIC_MAX_UNITS + 1))
    e = to_device(d)
    out, fin = _outputs(d)
    with pytest.raises(kda.KDAError) as ei:
        _call(kda.kda_fwd_static, e, d, out, fin)
    assert ei.value.status == kda.KDA_ERR_LIMIT
    torch.cuda.synchronize()
    assert torch.isnan(out.float()).all()   # nothing was enqueued
