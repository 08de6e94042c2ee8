"""Runs kda_fwd on a seeded synthetic workload (for profiling and quick checks).

  python -m gated_delta_rule_52_gb300.run [--workload prefill_8k] [--T 2048] [--H 64]
                                          [--iters 3] [--bwd]

Builds libkda.so if needed, draws the workload's inputs on the GPU, calls
kda_fwd (with --bwd: kda_bwd, on a random upstream gradient) `iters` times and prints
the CUDA-event time of the last call and the device status.  It checks no numbers: a profiling and timing runner only.
"""
import argparse
import os
import sys

import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from gated_delta_rule_52_gb300 import build, kda  # noqa: E402
from gated_delta_rule_52_gb300 import workloads as W  # noqa: E402


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="prefill_8k")
    ap.add_argument("--T", type=int, default=None)
    ap.add_argument("--H", type=int, default=None)
    ap.add_argument("--iters", type=int, default=3)
    ap.add_argument("--bwd", action="store_true", help="run kda_bwd instead of kda_fwd")
    a = ap.parse_args(argv)
    over = {}
    if a.T is not None:
        over["T"] = a.T
    if a.H is not None:
        over["H"] = a.H
    build.build_library()
    d = W.make_inputs(W.get(a.workload, **over))
    e = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in d.items()}
    out = torch.empty((d["B"], d["T"], d["H"], 128), dtype=torch.bfloat16, device="cuda")
    fin = None
    if d["state_dtype"]:
        fin = torch.empty((d["N"], d["H"], 128, 128), device="cuda",
                          dtype=torch.bfloat16 if d["state_dtype"] == "bf16" else torch.float32)
    s, t = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    dout = None
    if a.bwd:
        gen = torch.Generator().manual_seed(1)
        dout = torch.randn(d["v"].shape, generator=gen).to(torch.bfloat16).cuda()
    for _ in range(a.iters):
        s.record()
        if a.bwd:
            kda.kda_bwd(e["q"], e["k"], e["v"], e["g"], e["beta"], e["scale"], e["A_log"],
                        e["dt_bias"], e["lower_bound"], dout, initial_state=e["initial_state"],
                        cu_seqlens=e["cu_seqlens"])
        else:
            kda.kda_fwd(e["q"], e["k"], e["v"], e["g"], e["beta"], e["scale"], out, e["A_log"],
                        e["dt_bias"], e["lower_bound"], initial_state=e["initial_state"],
                        final_state=fin, cu_seqlens=e["cu_seqlens"])
        t.record()
    torch.cuda.synchronize()
    st = kda.get_device_status()
    print(f"{a.workload} B={d['B']} T={d['T']} H={d['H']}: {s.elapsed_time(t):.3f} ms "
          f"(last call), device status {st}")
    return 0 if st == kda.KDA_OK else 1


if __name__ == "__main__":
    sys.exit(main())
