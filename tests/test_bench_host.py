"""Host-side logic of bench.py without a GPU: the roofline byte/FLOP model, the
weak-scaling shard seeds and aggregation, and the cross-rank max reduction over
world_size-2 gloo process groups."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from gated_delta_rule_52_gb300 import workloads as W


def test_roofline_model_prefill():
    d = W.make_inputs(W.get("prefill_8k", T=64, H=2))   # small draw, then scale the sizes
    d = dict(d, T=8192, H=64, N=1)
    # 524,288 token-heads x 1,282 B + 64 heads x bf16 state in and out
    assert bench.algorithmic_bytes(d) == 524288 * 1282 + 64 * 128 * 128 * 2 * 2 == 676331520
    assert bench.algorithmic_flops(d) == 524288 * 180224


def test_roofline_model_state_variants():
    base = dict(B=1, T=64, H=2, N=1)
    d = dict(base, state_dtype=None, initial_state=None)
    assert bench.algorithmic_bytes(d) == 128 * 1282
    d = dict(base, state_dtype="fp32", initial_state=None)        # final only
    assert bench.algorithmic_bytes(d) == 128 * 1282 + 2 * 128 * 128 * 4
    d = dict(base, state_dtype="fp32", initial_state=object())    # in and out
    assert bench.algorithmic_bytes(d) == 128 * 1282 + 2 * 2 * 128 * 128 * 4


def test_shard_seeds_distinct_and_aggregate():
    seeds = {bench.shard_seed(2, r) for r in range(8)}
    assert len(seeds) == 8
    value, t = bench.aggregate(8192, 4, [10.0, 12.5, 11.0, 9.0])
    assert t == 12.5 and value == pytest.approx(4 * 8192 / 0.0125)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank_main(rank, world, port, ms_list, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        m = bench.max_over_ranks(ms_list[rank])
        value, t = bench.aggregate(1000, world, [m])
        out[rank] = (m, value)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    ms = [3.0, 7.5]
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, ms, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    for r in range(2):
        m, value = out[r]
        assert m == 7.5
        assert value == pytest.approx(2 * 1000 / 0.0075)


def test_max_over_ranks_without_group_is_identity():
    assert bench.max_over_ranks(4.25) == 4.25


def test_kernel_of_follows_the_packed_token_count():
    # the kernel label and stored-traffic lookup follow the dispatch of kda_fwd:
    # one row -> token recurrence, up to 64 -> 16-row blocks, more -> the pool kernel
    # (varlen batches of more than 4096 sequences: the cluster kernel)
    import bench
    from gated_delta_rule_52_gb300 import workloads as W
    assert bench.kernel_of(1) == "decode"
    assert bench.kernel_of(2) == "short" and bench.kernel_of(64) == "short"
    assert bench.kernel_of(65) == "pool" and bench.kernel_of(65, varlen=True) == "pool"
    assert bench.kernel_of(10**5, varlen=True, n_seqs=5000) == "cluster"
    d = W.make_inputs(W.get("varlen_ragged", H=1, seqlens=(40, 30)))
    assert bench.kernel_for(d) == "pool"   # the ragged workload's T is the packed total
    dl = W.make_inputs(W.get("varlen_ragged", H=1, seqlens=(600, 300)))
    assert not bench.mixed_dispatch(dl) and bench.launches_per_call(dl, 152) == 2   # the plan and the pool
    assert bench.kernel_for(W.make_inputs(W.get("tiny"))) == "pool"
    assert bench.launches_per_call(W.make_inputs(W.get("tiny")), 152) == 1
    # few units on a long fixed-length call: the sequence-parallel path (one plan, two
    # pool runs, the segment bounds and states, the scan, the final state)
    d8 = W.make_inputs(W.get("tiny", T=8192, H=1))
    assert bench.kernel_for(d8) == "pool" and bench.launches_per_call(d8, 152) == 7
    for k in bench.KERNEL_SOURCES:
        assert len(bench.kernel_source_hash(k)) == 16 and k in bench.KERNEL_NAMES


def test_tsplit_rule_mirror():
    # the few-units rule of kda_fwd's sequence-parallel path, as bench.py mirrors it
    import bench
    assert bench.tsplit_segments(1, 65536, 8, False, 152) == 7      # 57 chains (3/8 of 152) / 8 units
    assert bench.tsplit_segments(1, 65536, 16, False, 152) == 4
    assert bench.tsplit_segments(1, 65536, 19, False, 152) == 4     # 4 segments up to 152 / 8 units
    assert bench.tsplit_segments(1, 65536, 20, False, 152) == 0
    assert bench.tsplit_segments(1, 8192, 64, False, 152) == 0      # the headline: units fill the GPU
    assert bench.tsplit_segments(1, 8192, 2, False, 152) == 4       # capped by 2048-token segments
    assert bench.tsplit_segments(1, 65536, 1, False, 152) == 32     # capped at 32 segments
    assert bench.tsplit_segments(1, 65536, 8, True, 152) == 0       # varlen calls never split
    assert bench.tsplit_segments(1, 4096, 1, False, 152) == 0       # too short


def test_mixed_dispatch_rule_mirror():
    # varlen calls of more than 64 rows with at most 256 per sequence on average run the
    # short-step kernel beside the cluster kernel (kda_api.cu), as bench.py mirrors it
    import bench
    from gated_delta_rule_52_gb300 import workloads as W
    dm = W.make_inputs(W.get("varlen_ragged", H=1, seqlens=(40, 30, 20)))
    assert bench.mixed_dispatch(dm) and bench.launches_per_call(dm, 152) == 3   # short, plan, pool
    assert not bench.mixed_dispatch(W.make_inputs(W.get("varlen_ragged", H=1, seqlens=(40, 20))))   # 60 rows
    assert not bench.mixed_dispatch(W.make_inputs(W.get("varlen_ragged", H=1, seqlens=(600, 20))))  # avg 310
    assert not bench.mixed_dispatch(W.make_inputs(W.get("tiny")))                                   # fixed length


def test_gate_without_lower_bound_dispatch():
    # the gate without a lower bound: the pool kernel above 64 rows (every sequence on it,
    # no mixed split), the token recurrence for short calls and huge varlen batches
    d = W.make_inputs(W.get("varlen_ragged", H=1, seqlens=(40, 30, 20), lower_bound=None))
    assert d["lower_bound"] is None
    assert bench.kernel_for(d) == "pool" and not bench.mixed_dispatch(d)
    assert bench.launches_per_call(d, 152) == 2
    ds = W.make_inputs(W.get("varlen_ragged", H=1, seqlens=(40, 20), lower_bound=None))
    assert bench.kernel_for(ds) == "recur" and bench.launches_per_call(ds, 152) == 1
    assert bench.kernel_of(8192, unbounded=True) == "pool" and bench.kernel_of(8192) == "pool"
    assert bench.kernel_of(10**6, unbounded=True, varlen=True, n_seqs=5000) == "recur"
    assert "recur" in bench.KERNEL_NAMES and len(bench.kernel_source_hash("recur")) == 16
    # long fixed-length calls with few units: the sequence-parallel path, both gates
    du = W.make_inputs(W.get("tiny", T=8192, H=1, lower_bound=None))
    assert bench.kernel_for(du) == "pool" and bench.launches_per_call(du, 152) == 7


def test_both_arms_report_the_same_workload_config():
    d = W.make_inputs(W.get("tiny"))
    c = bench.workload_config("tiny", d)
    assert c["workload"] == "tiny" and c["T"] == 256 and c["lower_bound"] == -5.0
    assert "sigmoid" in c["gate"]
    du = W.make_inputs(W.get("tiny", lower_bound=None))
    cu = bench.workload_config("tiny", du)
    assert cu["lower_bound"] is None and "softplus" in cu["gate"]


def test_gpus_flag_is_checked_against_the_launcher(monkeypatch):
    import argparse
    args = argparse.Namespace(gpus=2, steps=3, warmup=3, impl="ours", workload="tiny")
    monkeypatch.setenv("WORLD_SIZE", "2")
    assert bench.check_world(args) is None
    monkeypatch.setenv("WORLD_SIZE", "4")
    assert "4 ranks" in bench.check_world(args)
    monkeypatch.delenv("WORLD_SIZE")
    cmd = bench.relaunch_cmd(args, ["--gpus", "2", "--steps", "3"])
    assert "torch.distributed.run" in cmd and "--nproc-per-node=2" in cmd
    assert cmd[cmd.index("--master-addr") + 1] == "127.0.0.1"
    assert cmd[-3:] == ["--gpus", "2", "--steps", "3"][-3:]
    assert bench.check_world(argparse.Namespace(gpus=0)) is not None


def test_head_ranges_cover_every_head_once():
    from gated_delta_rule_52_gb300 import shard
    for H in (1, 2, 5, 64, 67):
        for world in (1, 2, 3, 8):
            rs = [shard.head_range(r, world, H) for r in range(world)]
            assert rs[0][0] == 0 and rs[-1][1] == H
            assert all(a[1] == b[0] for a, b in zip(rs, rs[1:]))
            sizes = [h1 - h0 for h0, h1 in rs]
            assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        shard.head_range(2, 2, 4)


def _head_split_rank(rank, world, port, out):
    # one problem, its heads split over the ranks: each rank runs its slice (the oracle
    # stands in for a GPU here), the slices are gathered and joined
    import oracle
    from gated_delta_rule_52_gb300 import shard
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        d = W.make_inputs(W.get("varlen_ragged", H=5, seqlens=(40, 0, 70), seed=61))
        s = shard.shard(d, rank, world)
        o, f = oracle.kda_fwd(s["q"], s["k"], s["v"], s["g"], s["beta"], s["scale"], s["A_log"],
                              s["dt_bias"], s["lower_bound"], initial_state=s["initial_state"],
                              cu_seqlens=s["cu_seqlens"], nthreads=1)
        o, f = torch.from_numpy(o), torch.from_numpy(f)
        outs = [None] * world
        fins = [None] * world
        dist.all_gather_object(outs, o)
        dist.all_gather_object(fins, f)
        if rank == 0:
            full_o, full_f = oracle.kda_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["scale"],
                                            d["A_log"], d["dt_bias"], d["lower_bound"],
                                            initial_state=d["initial_state"],
                                            cu_seqlens=d["cu_seqlens"], nthreads=1)
            out["same"] = bool(torch.equal(shard.join(outs, "out"), torch.from_numpy(full_o)) and
                               torch.equal(shard.join(fins, "final_state"), torch.from_numpy(full_f)))
    finally:
        dist.destroy_process_group()


def test_head_split_of_one_problem_gloo_world2():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_head_split_rank, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(180)
        assert p.exitcode == 0
    assert out["same"]   # every (sequence, head) is computed by exactly one rank, exactly
