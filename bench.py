"""KDA forward prefill throughput on GB300.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME]

One step = one kda_fwd call (the whole hot path: prologue, intra-chunk UT/WY,
chunk-sequential state pass, state load/store) over the long-prefill workload
B=1, T=8192, H=64, K=V=128 with bf16 initial/final state.  Inputs are seeded
synthetic data resident in HBM; out/final_state are preallocated.  The working
set (676 MB of algorithmic traffic) is larger than L2 (129 MB) and a 256 MB
L2-flush write runs between timed steps (outside the timed kernel).  Each step is timed
with CUDA events on the launching stream; rank 0 prints one JSON line.

--workload picks another named workload (gated_delta_rule_52_gb300/workloads.py): the
other prefill/varlen shapes, the decode and short-step batches (decode, decode_16, step_64,
varlen_short), the few-head long prefill (prefill_64k_h8, sequence-parallel path) and the
gate without a lower bound (prefill_8k_unbounded, token recurrence, roofline on the fp32
lanes).  Every kernel's time is the whole kda_fwd call.

--impl reference times the fp64 CPU oracle (the baseline, on the host cores) on
a bounded sample of the same workload.

Under torchrun (N > 1) every rank processes its own copy of the workload with a
different seed (weak scaling, no data-path collective); the timed region is
bracketed by barriers and the max over ranks is reported.
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "KDA fwd prefill tokens/s on 1 GB300 (T=8192,H=64,K=V=128) + % of roofline"
UNIT = "tokens/s"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
# Algorithmic work per (token, head): q,k,v,g,out bf16 (5 x 256 B) + beta (2 B);
# FLOPs of the chunked form with C=64, K=V=128 (A, M, W, U~, M U dense; W S, Q S, K^T U).
BYTES_PER_TOKEN_HEAD = 5 * 128 * 2 + 2
FLOPS_PER_TOKEN_HEAD = 2 * 64 * (3 * 128 + 2 * 128) + 2 * 3 * 128 * 128
# Source files each kernel is built from (a stored ncu traffic figure is valid only
# while these are unchanged).
KERNEL_SOURCES = {
    "pool": ("kda_pool.cu", "kda_chunk.cuh", "sm103.cuh", "kda_internal.h"),
    "cluster": ("kda_cluster.cu", "kda_chunk.cuh", "sm103.cuh", "kda_internal.h"),
    "decode": ("kda_decode.cu", "sm103.cuh", "kda_internal.h"),
    "short": ("kda_short.cu", "sm103.cuh", "kda_internal.h"),
    "recur": ("kda_recur.cu", "sm103.cuh", "kda_internal.h"),
}
KERNEL_NAMES = {"pool": "kda_pool_kernel", "cluster": "kda_cluster_kernel", "decode": "kda_decode1_kernel", "short": "kda_short_kernel",
                "recur": "kda_recur_kernel"}
CSRC = os.path.join("gated_delta_rule_52_gb300", "csrc")
DECODE_MAX_T = 64   # calls with at most this many token rows run a kernel without workspace
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")


# --------------------------------------------------------------------------- helpers
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def shard_seed(base_seed: int, rank: int) -> int:
    """Each rank draws an independent problem of the same shape."""
    return base_seed + 1000 * rank


def aggregate(tokens_per_rank: int, world: int, times_ms):
    """Whole-job throughput from the per-rank timed-region durations (ms): the
    slowest rank bounds the job."""
    t = max(times_ms)
    return world * tokens_per_rank / (t / 1e3), t


def max_over_ranks(ms: float, device=None) -> float:
    """Max of a per-rank duration over all ranks (identity without a process group).
    Works with gloo (CPU tensors) and nccl (device tensors)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return ms
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def algorithmic_bytes(d) -> int:
    th = d["B"] * d["T"] * d["H"]
    sb = {"fp32": 4, "bf16": 2, None: 0}[d["state_dtype"]]
    n_state = (1 if d["initial_state"] is not None else 0) + (1 if d["state_dtype"] else 0)
    return th * BYTES_PER_TOKEN_HEAD + d["N"] * d["H"] * 128 * 128 * sb * n_state


# The token recurrence (the gate without a lower bound): per token-head, the decay,
# k^T S, the rank-1 update and q^T S, each K x V multiply-adds, 2 flops each.
RECUR_FLOPS_PER_TOKEN_HEAD = 4 * 128 * 128 * 2
SM_MAX_MHZ = 2070   # GB300 maximum SM clock, used when nvidia-smi reports none
SMS_DEFAULT = 152   # GB300 SM count, for host-side dispatch figures without a device


def algorithmic_flops(d) -> int:
    return d["B"] * d["T"] * d["H"] * FLOPS_PER_TOKEN_HEAD


def workload_config(name: str, d) -> dict:
    """The `config` keys both arms report for a workload."""
    return {"workload": name, "B": d["B"], "T": d["T"], "H": d["H"], "K": 128, "V": 128,
            "state": d["state_dtype"], "lower_bound": d["lower_bound"],
            "gate": ("-exp(A_log) softplus(g + dt_bias), no lower bound"
                     if d["lower_bound"] is None else "lower_bound sigmoid(exp(A_log) (g + dt_bias))")}


POOL_MAX_SEQS = 4096   # kda_internal.h kPoolMaxSeqs: larger varlen batches run the cluster kernel


def kernel_of(T: int, unbounded: bool = False, varlen: bool = False, n_seqs: int = 1) -> str:
    """The kernel libkda runs for a call of T packed token rows: calls of more than 64
    rows run the persistent pool kernel, except varlen calls of more than POOL_MAX_SEQS
    sequences (the cluster kernel; the token recurrence for the gate without a lower
    bound); calls of at most 64 rows the one-token or 16-row-block kernels (the token
    recurrence for the gate without a lower bound)."""
    big_varlen = varlen and n_seqs > POOL_MAX_SEQS
    if unbounded:
        return "recur" if T <= DECODE_MAX_T or big_varlen else "pool"
    if T == 1:
        return "decode"
    if T <= DECODE_MAX_T:
        return "short"
    return "cluster" if big_varlen else "pool"


def kernel_for(d, sms: int = SMS_DEFAULT) -> str:
    """The dominant kernel of a kda_fwd call on these inputs (the sequence-parallel
    path's state-only and output runs are pool-kernel launches)."""
    varlen = d["cu_seqlens"] is not None
    if not varlen and tsplit_segments(d["N"], d["T"], d["H"], False, sms):
        return "pool"
    return kernel_of(d["T"], d["lower_bound"] is None, varlen, d["N"])


# The dispatch rule of kda_fwd for the sequence-parallel path (kda_internal.h,
# tsplit_segments): fixed-length calls of at most sms / 8 (sequence, head) units run
# each sequence as P >= 4 segments of at least 2048 tokens, P units near 3/8 of the SMs.
TSPLIT_MIN_SEG, TSPLIT_MAX_SEG = 2048, 32


def tsplit_segments(N: int, T: int, H: int, varlen: bool, sms: int) -> int:
    if varlen or N <= 0 or T < 4 * TSPLIT_MIN_SEG or N * H <= 0:
        return 0
    P = (sms * 3 // 8) // (N * H)
    if P < 4 and (sms // 2) // (N * H) >= 4:
        P = 4
    P = min(P, T // TSPLIT_MIN_SEG, TSPLIT_MAX_SEG)
    return P if P >= 4 else 0


MIXED_MAX_AVG = 256   # kda_internal.h kMixedMaxAvg


def mixed_dispatch(d) -> bool:
    """A varlen call of more than 64 rows with at most 256 per sequence on average (bounded
    gate): the short-step kernel and the chunked kernel each take their own sequences."""
    return (d["lower_bound"] is not None and d["cu_seqlens"] is not None
            and DECODE_MAX_T < d["T"] <= MIXED_MAX_AVG * d["N"])


def launches_per_call(d, sms: int) -> int:
    """libkda kernel launches of one kda_fwd call on these inputs."""
    P = tsplit_segments(d["N"], d["T"], d["H"], d["cu_seqlens"] is not None, sms)
    if P:   # segment bounds, segment states, one plan, 2 pool runs, scan (+ final copy)
        return 6 + (d["state_dtype"] is not None)
    if d["lower_bound"] is None:
        return 2 if d["cu_seqlens"] is not None and kernel_for(d, sms) == "pool" else 1
    if d["T"] <= DECODE_MAX_T:
        return 1
    pool_varlen = d["cu_seqlens"] is not None and kernel_for(d, sms) == "pool"   # plan + pool
    return (2 if pool_varlen else 1) + (1 if mixed_dispatch(d) else 0)


def kernel_source_hash(kernel: str = "cluster") -> str:
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, CSRC, name), "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), float(j.get("bf16_tflops", FALLBACK_BF16_TFLOPS)), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


def stored_traffic(workload: str, kernel: str = "cluster"):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on the
    current sources of the kernel (else None)."""
    try:
        with open(TRAFFIC_FILE) as f:
            j = json.load(f)
        e = j.get(workload)
        if e and e.get("source_hash") == kernel_source_hash(kernel):
            return float(e["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.tmp = None

    def start(self):
        try:
            self.tmp = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.tmp, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.tmp.flush()
        self.tmp.seek(0)
        rows = [r for r in csv.reader(io.StringIO(self.tmp.read())) if len(r) >= 9]
        self.tmp.close()
        os.unlink(self.tmp.name)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].strip().replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in rows:
            for i, nm in enumerate(names):
                if r[5 + i].strip() == "Active":
                    reasons.add(nm)
        loaded = [s for s in sm if mx and s >= 0.5 * max(mx)] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(rows)}


# --------------------------------------------------------------------------- oracle
def oracle_sample(d, pairs_per_call: int, tokens: int, nthreads: int):
    """Runs the fp64 oracle on the first `tokens` tokens of `pairs_per_call`
    (batch row, head) pairs of the workload, heads first, at most B*H of them;
    returns (seconds, token-heads)."""
    import oracle
    T = min(tokens, d["T"])
    H, B = d["H"], d["q"].shape[0]
    pairs = [((i // H) % B, i % H) for i in range(min(pairs_per_call, B * H))]
    sub = {key: d[key][:, :T].contiguous() for key in ("q", "k", "v", "g", "beta")}
    t0 = time.perf_counter()
    oracle.kda_fwd(sub["q"], sub["k"], sub["v"], sub["g"], sub["beta"], d["scale"], d["A_log"],
                   d["dt_bias"], d["lower_bound"], initial_state=d["initial_state"],
                   want_final=True, pairs=pairs, nthreads=nthreads)
    return time.perf_counter() - t0, len(pairs) * T


def cpu_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def cpu_baseline(d, budget_s: float = 12.0):
    """The oracle, as it stands, timed on the host cores on a bounded sample of the
    workload: full-length (batch row, head) pairs, `cores` of them first, grown toward
    ~budget_s of wall time; a workload whose every pair runs in well under that is
    timed whole, a few times over."""
    import oracle
    cores = cpu_cores()
    nthreads = min(cores, oracle.max_threads()) or cores
    total = d["q"].shape[0] * d["H"]
    pairs = min(total, nthreads)
    secs, th = oracle_sample(d, pairs, d["T"], nthreads)
    if secs < budget_s / 4 and pairs < total:
        pairs = min(total, pairs * max(1, int(budget_s / max(secs, 1e-3))))
        secs, th = oracle_sample(d, pairs, d["T"], nthreads)
    reps = 1
    if secs < 1.0:
        reps = max(1, min(20, int(2.0 / max(secs, 1e-3))))
        secs, th = 0.0, 0
        for _ in range(reps):
            s, t = oracle_sample(d, pairs, d["T"], nthreads)
            secs += s
            th += t
    value = (th / d["H"]) / secs
    return {"value": value, "unit": UNIT, "cores": nthreads, "kind": "oracle",
            "sample": f"{pairs} of {total} (batch row, head) pairs x {d['T']} tokens"
                      f"{f', {reps} times' if reps > 1 else ''}, fp64, {secs:.1f} s wall; "
                      "tokens/s = token-heads / H / s"}


# --------------------------------------------------------------------------- arms
def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    from gated_delta_rule_52_gb300 import workloads as W
    import oracle
    oracle.build()
    w = W.get(args.workload)
    d = W.make_inputs(w)
    cores = cpu_cores()
    nthreads = min(cores, oracle.max_threads()) or cores
    # size one step so that warmup + steps fit in ~150 s
    per_step = max(0.05, 150.0 / max(1, args.steps + args.warmup))
    secs, _ = oracle_sample(d, nthreads, 128, nthreads)
    tokens = int(max(16, min(d["T"], 128 * per_step / max(secs, 1e-4))))
    for _ in range(args.warmup):
        oracle_sample(d, nthreads, tokens, nthreads)
    tot_s, tot_th = 0.0, 0
    for _ in range(args.steps):
        s, th = oracle_sample(d, nthreads, tokens, nthreads)
        tot_s += s
        tot_th += th
    value = (tot_th / d["H"]) / tot_s
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * tot_s / max(1, args.steps),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference",
            "config": workload_config(w.name, d),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": nthreads, "kind": "oracle",
                             "sample": f"per step {nthreads} (sequence, head) pairs x {tokens} "
                                       f"tokens, fp64"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args):
    import torch
    import torch.distributed as dist
    from gated_delta_rule_52_gb300 import build as kbuild
    from gated_delta_rule_52_gb300 import kda
    from gated_delta_rule_52_gb300 import workloads as W

    ws, rank, local = dist_env()
    if ws > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0 or ws == 1:
        kbuild.build_library()
    if ws > 1:
        dist.barrier()
    kda.lib()

    w = W.get(args.workload)
    if args.split == "heads":   # one problem, its heads split over the ranks (strong scaling)
        from gated_delta_rule_52_gb300 import shard
        d_cfg = W.make_inputs(w)
        d_cpu = shard.shard(d_cfg, rank, ws)
    else:                       # an independent problem per rank (weak scaling)
        w = W.get(args.workload, seed=shard_seed(w.seed, rank))
        d_cpu = d_cfg = W.make_inputs(w)
    e = {key: (val.to(dev) if torch.is_tensor(val) else val) for key, val in d_cpu.items()}
    B, T, H, N = d_cpu["B"], d_cpu["T"], d_cpu["H"], d_cpu["N"]
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    lpc = launches_per_call(d_cpu, sms)
    kern = kernel_for(d_cpu, sms)
    out = torch.empty((B, T, H, 128), dtype=torch.bfloat16, device=dev)
    fin = None
    if d_cpu["state_dtype"]:
        sdt = torch.bfloat16 if d_cpu["state_dtype"] == "bf16" else torch.float32
        fin = torch.empty((N, H, 128, 128), dtype=sdt, device=dev)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        kda.kda_fwd(e["q"], e["k"], e["v"], e["g"], e["beta"], e["scale"], out, e["A_log"],
                    e["dt_bias"], e["lower_bound"], initial_state=e["initial_state"],
                    final_state=fin, cu_seqlens=e["cu_seqlens"], stream=stream)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    if kda.get_device_status(stream) != kda.KDA_OK:
        raise RuntimeError("device reported an error during warm-up")

    clocks = ClockSampler(local)
    clocks.start()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    for i in range(args.steps):
        flush.zero_()
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    if ws > 1:
        dist.barrier()
    clk = clocks.stop()
    if kda.get_device_status(stream) != kda.KDA_OK:
        raise RuntimeError("device reported an error during the timed region")
    per_step = [s.elapsed_time(t) for s, t in zip(starts, ends)]
    kernel_ms = sum(per_step)
    times = [max_over_ranks(kernel_ms, dev)]
    # with a head split every rank covers the whole call's tokens for its heads: the job
    # processes B T tokens (of all H heads) per step
    tokens_per_rank = B * T * args.steps / (ws if args.split == "heads" else 1)
    value, tmax = aggregate(tokens_per_rank, ws, times)
    ms_per_step = tmax / args.steps
    avg_launch_ms = kernel_ms / args.steps

    # End to end through the public API: every step copies its inputs from pinned host
    # memory to the device, runs kda_fwd and copies its result (out, final state) back
    # to pinned host memory.  Steps are pipelined the way a serving loop streams
    # batches: two buffer sets, inputs on one copy stream, results on another, so step
    # i+1's upload and step i-1's download overlap step i's kernel.  The serial form
    # (one stream, no overlap) is reported beside it.
    e2e = None
    if rank == 0:
        names = ["q", "k", "v", "g", "beta", "A_log", "dt_bias", "initial_state"]
        host = {nm: d_cpu[nm].pin_memory() for nm in names if d_cpu[nm] is not None}
        dev_in = [{nm: torch.empty_like(host[nm], device=dev) for nm in host} for _ in range(2)]
        outs = [out, torch.empty_like(out)]
        fins = [fin, torch.empty_like(fin)] if fin is not None else [None, None]
        h_out = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
        h_fin = [torch.empty(fin.shape, dtype=fin.dtype).pin_memory() for _ in range(2)] \
            if fin is not None else [None, None]
        h2d = sum(t.numel() * t.element_size() for t in host.values())
        d2h = out.numel() * out.element_size() + (fin.numel() * fin.element_size() if fin is not None else 0)
        up, down = torch.cuda.Stream(), torch.cuda.Stream()
        ev_in = [torch.cuda.Event() for _ in range(2)]
        ev_k = [torch.cuda.Event() for _ in range(2)]
        ev_out = [torch.cuda.Event() for _ in range(2)]

        def e2e_steps(n, serial):
            for i in range(n):
                b = 0 if serial else i % 2
                cin = stream if serial else up
                cout = stream if serial else down
                if not serial and i >= 2:
                    up.wait_event(ev_k[b])          # the kernel of step i-2 has read buffer b
                with torch.cuda.stream(cin):
                    for nm, t in host.items():
                        dev_in[b][nm].copy_(t, non_blocking=True)
                    ev_in[b].record(cin)
                stream.wait_event(ev_in[b])
                if not serial and i >= 2:
                    stream.wait_event(ev_out[b])    # step i-2's result has left out/fin buffer b
                kda.kda_fwd(dev_in[b]["q"], dev_in[b]["k"], dev_in[b]["v"], dev_in[b]["g"],
                            dev_in[b]["beta"], e["scale"], outs[b], dev_in[b]["A_log"],
                            dev_in[b]["dt_bias"], e["lower_bound"],
                            initial_state=dev_in[b].get("initial_state"), final_state=fins[b],
                            cu_seqlens=e["cu_seqlens"], stream=stream)
                ev_k[b].record(stream)
                cout.wait_event(ev_k[b])
                with torch.cuda.stream(cout):
                    h_out[b].copy_(outs[b], non_blocking=True)
                    if h_fin[b] is not None:
                        h_fin[b].copy_(fins[b], non_blocking=True)
                    ev_out[b].record(cout)

        def timed(serial):
            e2e_steps(2, serial)
            torch.cuda.synchronize()
            n_e2e = max(3, min(args.steps, 20))
            s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s0.record(stream if serial else up)
            e2e_steps(n_e2e, serial)
            (stream if serial else down).wait_event(ev_k[(n_e2e - 1) % 2])
            s1.record(stream if serial else down)
            torch.cuda.synchronize()
            return s0.elapsed_time(s1) / n_e2e, n_e2e

        serial_ms, _ = timed(True)
        e2e_ms, n_e2e = timed(False)
        e2e = {"value": B * T / (e2e_ms / 1e3), "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms, "steps": n_e2e,
               "pipelined": "2 buffer sets; uploads, kernels and downloads on three streams",
               "serial_ms_per_step": serial_ms}

    if rank != 0:
        if ws > 1:
            dist.destroy_process_group()
        return 0

    hbm, tflops, src = measured_peaks()
    abytes = algorithmic_bytes(d_cpu)
    achieved = abytes / (avg_launch_ms / 1e3) / 1e9
    roof = {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
            "frac": achieved / hbm, "traffic": stored_traffic(w.name, kern),
            "peak_source": f"{src} (MEASURED_PEAKS.json hbm_gbs)" if src == "measured"
            else f"{src} {hbm} GB/s",
            "kernel": (f"kda_short_kernel + {KERNEL_NAMES[kern]} (kda_fwd: each on its own sequences, "
                       f"{lpc} launches per step, the time of the whole call)") if mixed_dispatch(d_cpu) else
                      KERNEL_NAMES[kern] + (
                " (kda_fwd: one launch per step)" if lpc == 1 else
                f" (kda_fwd: sequence-parallel path, {lpc} launches per step, the time of the whole call)"
                if tsplit_segments(d_cpu["N"], d_cpu["T"], d_cpu["H"], d_cpu["cu_seqlens"] is not None, sms)
                else
                " (kda_fwd: a one-CTA plan and the pool, 2 launches per step, the time of the whole call)"),
            "algorithmic_bytes_per_launch": abytes,
            "algorithmic_flops_per_launch": algorithmic_flops(d_cpu),
            "tensor_frac": algorithmic_flops(d_cpu) / (avg_launch_ms / 1e3) / (tflops * 1e12)}
    if kern == "recur":
        # `frac` stays the HBM roofline of the method (the same definition as every other
        # workload).  The token recurrence itself runs on the fp32 CUDA cores: 4 K V
        # multiply-adds per token-head (decay, k^T S, the rank-1 update, q^T S), against
        # 128 fp32 lanes per SM at the maximum SM clock; that fraction is `alu_view`.
        mhz = (clk or {}).get("sm_max_mhz") or SM_MAX_MHZ
        peak_alu = sms * 128 * 2 * mhz * 1e6 / 1e12
        rflops = B * T * H * RECUR_FLOPS_PER_TOKEN_HEAD
        ach = rflops / (avg_launch_ms / 1e3) / 1e12
        roof["alu_view"] = {"bound": "alu", "achieved": ach, "peak": peak_alu, "unit": "TFLOP/s",
                            "frac": ach / peak_alu, "flops_per_launch": rflops,
                            "peak_source": f"derived: {sms} SMs x 128 fp32 lanes x 2 flops x {mhz:.0f} MHz"}
    cpu = cpu_baseline(d_cpu) if ws == 1 else None
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
            "scaling": "strong" if args.split == "heads" else "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic",
            "config": dict(workload_config(w.name, d_cfg), **({"split": f"heads over {ws} ranks"}
                                                             if args.split == "heads" else {})),
            "l2": f"algorithmic traffic {abytes / 1e6:.0f} MB per step "
                  f"({'larger' if abytes > 129e6 else 'smaller'} than the 129 MB L2); "
                  "a 256 MB flush write between timed steps",
            "timing": "CUDA events around each kda_fwd call",
            "roofline": roof, "cpu_baseline": cpu, "e2e": e2e, "clocks": clk,
            "gpu_launches": args.steps * lpc,
            "wall_s_timed_region": wall}
    print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()
    return 0


def free_port() -> int:
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def relaunch_cmd(args, argv) -> list:
    """The torchrun command that runs this bench on `--gpus` ranks of this node."""
    return [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
            f"--nproc-per-node={args.gpus}", "--master-addr", "127.0.0.1",
            "--master-port", str(free_port()), os.path.abspath(__file__)] + list(argv)


def check_world(args) -> str | None:
    """--gpus must agree with the launcher's world size (None when it does)."""
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if args.gpus < 1:
        return f"--gpus {args.gpus}: at least one GPU"
    if "WORLD_SIZE" in os.environ and ws != args.gpus:
        return f"--gpus {args.gpus} but the launcher started {ws} ranks"
    return None


# The backward per (token, head): q, k, v, g, dout read (5 x 256 B) and beta (2 B);
# dq, dk, dv, dg written in fp32 (4 x 512 B) and dbeta (4 B).  Its arithmetic on the fp32
# lanes: the forward recurrence twice (the checkpoint sweep and the per-chunk
# recomputation, 3 K V multiply-adds each) and the reverse step (about 9 K V).
BWD_BYTES_PER_TOKEN_HEAD = 5 * 256 + 2 + 4 * 512 + 4
BWD_ALU_FLOPS_PER_TOKEN_HEAD = 2 * (3 + 3 + 9) * 128 * 128


def run_ours_bwd(args):
    """Times kda_bwd (the gradients of every forward input) on a workload: inputs and the
    upstream gradient resident, fp32 outputs allocated per call by the binding."""
    import torch
    from gated_delta_rule_52_gb300 import build as kbuild
    from gated_delta_rule_52_gb300 import kda
    from gated_delta_rule_52_gb300 import workloads as W
    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    kbuild.build_library()
    kda.lib()
    w = W.get(args.workload)
    d_cpu = W.make_inputs(w)
    e = {key: (val.to(dev) if torch.is_tensor(val) else val) for key, val in d_cpu.items()}
    B, T, H, N = d_cpu["B"], d_cpu["T"], d_cpu["H"], d_cpu["N"]
    gen = torch.Generator().manual_seed(1)
    dout = torch.randn(d_cpu["v"].shape, generator=gen).to(torch.bfloat16).to(dev)
    dfin = torch.randn((N, H, 128, 128), generator=gen).to(dev) if d_cpu["state_dtype"] else None
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        return kda.kda_bwd(e["q"], e["k"], e["v"], e["g"], e["beta"], e["scale"], e["A_log"],
                           e["dt_bias"], e["lower_bound"], dout, initial_state=e["initial_state"],
                           dfinal=dfin, cu_seqlens=e["cu_seqlens"], stream=stream)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    if kda.get_device_status(stream) != kda.KDA_OK:
        raise RuntimeError("device reported an error during warm-up")
    clocks = ClockSampler(local)
    clocks.start()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    torch.cuda.synchronize()
    for i in range(args.steps):
        flush.zero_()
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    if kda.get_device_status(stream) != kda.KDA_OK:
        raise RuntimeError("device reported an error during the timed region")
    ms = sum(s.elapsed_time(t) for s, t in zip(starts, ends)) / args.steps
    th = B * T * H
    sb = {"fp32": 4, "bf16": 2, None: 0}[d_cpu["state_dtype"]]
    abytes = th * BWD_BYTES_PER_TOKEN_HEAD + N * H * 128 * 128 * (sb + (8 if sb else 4))
    hbm, _, src = measured_peaks()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    mhz = (clk or {}).get("sm_max_mhz") or SM_MAX_MHZ
    peak_alu = sms * 128 * 2 * mhz * 1e6 / 1e12
    ach = abytes / (ms / 1e3) / 1e9
    alu = th * BWD_ALU_FLOPS_PER_TOKEN_HEAD / (ms / 1e3) / 1e12
    line = {"metric": "KDA bwd tokens/s on 1 GB300 (gradients of every forward input)",
            "value": B * T / (ms / 1e3), "unit": UNIT, "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic", "pass": "bwd",
            "config": workload_config(w.name, d_cpu),
            "l2": "a 256 MB flush write between timed steps", "timing": "CUDA events around each kda_bwd call",
            "roofline": {"bound": "hbm", "achieved": ach, "peak": hbm, "unit": "GB/s", "frac": ach / hbm,
                         "traffic": None, "peak_source": src,
                         "kernel": "kda_bwd_state_kernel + kda_bwd_act_kernel (the time of the whole call)",
                         "algorithmic_bytes_per_launch": abytes,
                         "alu_view": {"bound": "alu", "achieved": alu, "peak": peak_alu, "unit": "TFLOP/s",
                                      "frac": alu / peak_alu,
                                      "flops_per_launch": th * BWD_ALU_FLOPS_PER_TOKEN_HEAD}},
            "clocks": clk, "gpu_launches": args.steps * 2,
            "cpu_baseline": bwd_cpu_baseline(d_cpu, dout.cpu(), None if dfin is None else dfin.cpu())}
    print(json.dumps(line), flush=True)
    return 0


def bwd_cpu_baseline(d, dout, dfin, tokens=512):
    """The backward oracle, as it stands, on the host cores: the first `tokens` tokens of
    as many heads as cores (fixed-length workloads; None for varlen ones)."""
    import oracle
    if d["cu_seqlens"] is not None:
        return None
    cores = cpu_cores()
    nthreads = min(cores, oracle.max_threads()) or cores
    T, nh, B = min(tokens, d["T"]), min(nthreads, d["H"]), d["B"]
    sl = lambda x: x[:, :T, :nh].contiguous()
    init = None if d["initial_state"] is None else d["initial_state"][:, :nh].contiguous()
    t0 = time.perf_counter()
    oracle.kda_bwd(sl(d["q"]), sl(d["k"]), sl(d["v"]), sl(d["g"]), sl(d["beta"]), d["scale"],
                   d["A_log"][:nh].contiguous(), d["dt_bias"][:nh].contiguous(), d["lower_bound"],
                   sl(dout), initial_state=init, dfinal=None if dfin is None else dfin[:, :nh].contiguous(),
                   nthreads=nthreads)
    secs = time.perf_counter() - t0
    return {"value": (B * T * nh / d["H"]) / secs, "unit": UNIT, "cores": nthreads, "kind": "oracle",
            "sample": f"{B} x {T} tokens x {nh} of {d['H']} heads, fp64 backward, {secs:.1f} s; "
                      "tokens/s = token-heads / H / s"}


def main(argv=None):
    argv = sys.argv[1:] if argv is None else argv
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1,
                    help="ranks (one per GPU); more than 1 without torchrun relaunches under it")
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="prefill_8k")
    ap.add_argument("--split", choices=["problems", "heads"], default="problems",
                    help="N > 1: an independent problem per rank (weak), or one problem's heads split")
    ap.add_argument("--pass", dest="pass_", choices=["fwd", "bwd"], default="fwd",
                    help="bwd times kda_bwd (the gradients) instead of the forward")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        return subprocess.call(relaunch_cmd(args, argv))
    bad = check_world(args)
    if bad:
        print(bad, file=sys.stderr)
        return 2
    if args.impl == "reference":
        return run_reference(args)
    if args.pass_ == "bwd":
        return run_ours_bwd(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
