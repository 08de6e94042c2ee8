"""GPU parity: libkda (through the C ABI) against the fp64 oracle on the same
seeded inputs, element by element.  Reduced sizes span several 64-token chunks and
ragged tails; the full workload sizes are compared in full too, the oracle running
one batch row (or a group of varlen sequences) at a time."""
import numpy as np
import pytest
import torch

from gated_delta_rule_52_gb300 import kda
from gated_delta_rule_52_gb300 import workloads as W
from tests import parity_util as pu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from gated_delta_rule_52_gb300 import build
    build.build_library()
    kda.lib()


REDUCED = {
    "tiny": W.get("tiny"),
    "batch_state": W.get("batch_state", T=200, H=4),
    "prefill_8k": W.get("prefill_8k", T=1000, H=4),
    "varlen_uniform": W.get("varlen_uniform", T=8 * 130, H=4),
    "varlen_ragged": W.get("varlen_ragged", H=4, seqlens=(1, 17, 63, 64, 65, 0, 129, 300, 2, 191)),
}


@pytest.mark.parametrize("name", list(REDUCED))
def test_reduced_all_elements(name):
    d = W.make_inputs(REDUCED[name])
    out, fin = pu.run_gpu(d)
    ref_out, ref_fin = pu.run_oracle(d)
    res = pu.check(d, out, fin, ref_out, ref_fin, label=name)
    print(name, res)


@pytest.mark.parametrize("name", ["batch_state", "prefill_8k", "varlen_uniform", "varlen_ragged"])
def test_full_size_all_elements(name):
    d = W.make_inputs(W.get(name))
    out, fin = pu.run_gpu(d)
    res = pu.check_full(d, out, fin, label=name)
    print(name, res)


def test_chained_calls_match_single_call():
    # Two T=1024 calls chained through final_state -> initial_state equal one T=2048 call.
    d = W.make_inputs(W.get("batch_state"))
    out, fin = pu.run_gpu(d)
    T1 = 1024
    d1 = dict(d, T=T1, q=d["q"][:, :T1], k=d["k"][:, :T1], v=d["v"][:, :T1], g=d["g"][:, :T1],
              beta=d["beta"][:, :T1])
    d1 = {kk: (vv.contiguous() if torch.is_tensor(vv) else vv) for kk, vv in d1.items()}
    o1, f1 = pu.run_gpu(d1)
    d2 = dict(d, T=d["T"] - T1, q=d["q"][:, T1:], k=d["k"][:, T1:], v=d["v"][:, T1:],
              g=d["g"][:, T1:], beta=d["beta"][:, T1:], initial_state=f1)
    d2 = {kk: (vv.contiguous() if torch.is_tensor(vv) else vv) for kk, vv in d2.items()}
    o2, f2 = pu.run_gpu(d2)
    chained = torch.cat([o1, o2], 1).float().numpy()
    mx, rl = pu.errors(chained, out.float().numpy())
    assert mx <= pu.OUT_MAX_ABS and rl <= pu.OUT_REL_L2, (mx, rl)
    _, srl = pu.errors(f2.numpy(), fin.numpy())
    assert srl <= pu.STATE_REL_L2["fp32"], srl
    # and the chained result against the oracle on sampled pairs
    pairs = [(0, 0), (1, 5), (3, 15)]
    ref_out, ref_fin = pu.run_oracle(d, pairs=pairs)
    pu.check(d, torch.cat([o1, o2], 1), f2, ref_out, ref_fin, pairs=pairs, label="chained")


def test_zero_length_tokens_pass_state_through():
    d = W.make_inputs(W.get("batch_state", B=2, T=0, H=3))
    out, fin = pu.run_gpu(d)
    assert out.numel() == 0
    torch.testing.assert_close(fin, d["initial_state"], rtol=0, atol=0)


def test_state_variants():
    base = W.get("batch_state", B=2, T=130, H=2)
    for sd, init in (("fp32", "none"), ("bf16", "normal"), ("bf16", "none")):
        d = W.make_inputs(W.get("batch_state", B=2, T=130, H=2, state_dtype=sd, initial_state=init))
        out, fin = pu.run_gpu(d)
        ref_out, ref_fin = pu.run_oracle(d)
        pu.check(d, out, fin, ref_out, ref_fin, label=f"{sd}/{init}")
    # initial state given, final state not requested
    d = W.make_inputs(base)
    out, _ = pu.run_gpu(d, want_final=False)
    ref_out, _ = pu.run_oracle(d, want_final=False)
    pu.check(d, out, None, ref_out, None, label="no-final")
    # no state at all
    d = W.make_inputs(W.get("tiny", state_dtype=None))
    out, fin = pu.run_gpu(d)
    assert fin is None
    ref_out, _ = pu.run_oracle(d, want_final=False)
    pu.check(d, out, None, ref_out, None, label="stateless")


@pytest.mark.parametrize("lb", [0.0, -0.5, -5.0])
def test_lower_bound_extremes(lb):
    # lb = 0: no decay (pure delta rule); lb = -5 with large gates: decay saturates.
    d = W.make_inputs(W.get("varlen_ragged", H=2, seqlens=(70, 129, 5), lower_bound=lb))
    out, fin = pu.run_gpu(d)
    ref_out, ref_fin = pu.run_oracle(d)
    print("lb", lb, pu.check(d, out, fin, ref_out, ref_fin, label=f"lb={lb}"))


def test_out_guard_region_untouched():
    # Varlen tails must not write outside [0, T): surround `out` with guard rows.
    d = W.make_inputs(W.get("varlen_ragged", H=3, seqlens=(65, 1, 130, 63)))
    e = pu.to_device(d)
    T, H = d["T"], d["H"]
    buf = torch.full((T + 128, H, 128), 7.0, dtype=torch.bfloat16, device="cuda")
    out = buf[64:64 + T].view(1, T, H, 128)
    fin = torch.empty((d["N"], H, 128, 128), dtype=torch.float32, device="cuda")
    kda.kda_fwd(e["q"], e["k"], e["v"], e["g"], e["beta"], d["scale"], out, e["A_log"],
                e["dt_bias"], d["lower_bound"], initial_state=e["initial_state"], final_state=fin,
                cu_seqlens=e["cu_seqlens"])
    torch.cuda.synchronize()
    assert (buf[:64] == 7.0).all() and (buf[64 + T:] == 7.0).all()
    ref_out, ref_fin = pu.run_oracle(d)
    pu.check(d, out.cpu(), fin.cpu(), ref_out, ref_fin, label="guard")


@pytest.mark.parametrize("B,T,H,lb", [(3, 200, 64, -5.0), (2, 130, 65, -2.0), (3, 200, 64, None),
                                      (1, 300, 3, -5.0), (1, 200, 1, None), (1, 1000, 5, None)])
def test_fixed_length_more_units_than_chains(B, T, H, lb):
    # more (sequence, head) units than the pool runs chains (192 units on 64 chains, 130 on
    # 65): each chain takes its units one after another, its state leaving TMEM between
    # them; and small odd unit counts (3, 1 and 5 units, one chain each); ragged last
    # chunks; both gates
    d = W.make_inputs(W.get("prefill_8k", B=B, T=T, H=H, seed=90 + H, state_dtype="fp32",
                            lower_bound=lb))
    out, fin = pu.run_gpu(d)
    ref_out, ref_fin = pu.run_oracle(d)
    print(B, T, H, lb, pu.check(d, out, fin, ref_out, ref_fin, label=f"{B * H} units"))


def test_deterministic():
    d = W.make_inputs(W.get("prefill_8k", T=700, H=3))
    a, fa = pu.run_gpu(d)
    b, fb = pu.run_gpu(d)
    assert torch.equal(a, b) and torch.equal(fa, fb)


def test_runs_on_a_side_stream():
    d = W.make_inputs(W.get("tiny"))
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        out, fin = pu.run_gpu(d, stream=s)
    ref_out, ref_fin = pu.run_oracle(d)
    pu.check(d, out, fin, ref_out, ref_fin, label="stream")


def test_binding_rejects_bad_tensors():
    d = pu.to_device(W.make_inputs(W.get("tiny")))
    out = torch.empty_like(d["v"])
    args = [d["q"], d["k"], d["v"], d["g"], d["beta"], d["scale"], out, d["A_log"], d["dt_bias"],
            d["lower_bound"]]
    bad = list(args); bad[0] = d["q"].float()
    with pytest.raises(ValueError):
        kda.kda_fwd(*bad)
    bad = list(args); bad[2] = d["v"][:, :, :, :64]
    with pytest.raises(ValueError):
        kda.kda_fwd(*bad)
    with pytest.raises(kda.KDAError) as ei:
        kda.kda_fwd(*args[:9], -7.0)
    assert ei.value.status == kda.KDA_ERR_VALUE
    with pytest.raises(ValueError):
        kda.kda_fwd(*args, initial_state=torch.zeros(1, 2, 128, 128, device="cuda"),
                    final_state=torch.zeros(1, 2, 128, 128, device="cuda", dtype=torch.bfloat16))


def test_many_short_sequences_longest_first_order():
    # More clusters than SMs, zero-length and single-token sequences mixed in:
    # every sequence must land on exactly one cluster whatever the order.  Three long
    # sequences keep the average above 256 rows, so the cluster kernel takes them all.
    r = np.random.default_rng(7)
    lens = [int(x) for x in r.integers(0, 90, 300)]
    lens[0], lens[5], lens[-1] = 0, 1, 200
    lens[-2], lens[-3], lens[-4] = 30000, 30000, 20000
    d = W.make_inputs(W.get("varlen_ragged", H=1, seqlens=tuple(lens)))
    out, fin = pu.run_gpu(d)
    ref_out, ref_fin = pu.run_oracle(d)
    print("many-seqs", pu.check(d, out, fin, ref_out, ref_fin, label="many-seqs"))


def test_more_sequences_than_the_pool_plans():
    # Varlen calls of more than 4096 sequences skip the pool's one-CTA plan and run one
    # two-CTA cluster per (sequence, head) instead; zero-length sequences in between
    r = np.random.default_rng(11)
    lens = [int(x) for x in r.integers(65, 90, 4100)]
    lens[3], lens[4000] = 0, 0
    d = W.make_inputs(W.get("varlen_ragged", H=1, seqlens=tuple(lens), seed=91))
    assert d["N"] > 4096
    out, fin = pu.run_gpu(d)
    ref_out, ref_fin = pu.run_oracle(d)
    print("4100 seqs", pu.check(d, out, fin, ref_out, ref_fin, label="4100 sequences"))


def test_the_most_sequences_the_pool_plans():
    # 4096 sequences, the plan's limit (a full bitonic sort of 4096 keys), lengths from 0 to
    # 600 with the average above 256 rows, so the pool takes every one of them (empty ones
    # pass their state through)
    r = np.random.default_rng(12)
    lens = [int(x) for x in r.integers(0, 600, 4096)]
    lens[0], lens[17], lens[4095] = 0, 1, 64
    d = W.make_inputs(W.get("varlen_ragged", H=1, seqlens=tuple(lens), seed=92))
    assert d["N"] == 4096 and d["T"] > 256 * d["N"]
    out, fin = pu.run_gpu(d)
    ref_out, ref_fin = pu.run_oracle(d)
    print("4096 seqs", pu.check(d, out, fin, ref_out, ref_fin, label="4096 sequences"))
    torch.testing.assert_close(fin[0], d["initial_state"][0].to(fin.dtype), rtol=0, atol=0)


def test_caller_workspace_entry_point():
    # kda_fwd_ws (the cluster kernel on a caller buffer) matches the oracle, and a buffer
    # full of garbage gives the result of a zeroed one bit for bit
    d = W.make_inputs(W.get("varlen_ragged", H=3, seqlens=(65, 1, 130, 63, 200)))
    e = pu.to_device(d)
    ref_out, ref_fin = pu.run_gpu(d)
    outs = []
    for fill in (0x00, 0xFF):
        out = torch.empty_like(ref_out, device="cuda")
        fin = torch.empty_like(ref_fin, device="cuda")
        ws = torch.full((kda.workspace_bytes(d["N"], d["H"]),), fill, dtype=torch.uint8, device="cuda")
        kda.kda_fwd(e["q"], e["k"], e["v"], e["g"], e["beta"], d["scale"], out, e["A_log"],
                    e["dt_bias"], d["lower_bound"], initial_state=e["initial_state"], final_state=fin,
                    cu_seqlens=e["cu_seqlens"], workspace=ws)
        torch.cuda.synchronize()
        assert kda.get_device_status() == kda.KDA_OK
        outs.append((out.cpu(), fin.cpu()))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
    o_ref, f_ref = pu.run_oracle(d)
    pu.check(d, outs[1][0], outs[1][1], o_ref, f_ref, label="kda_fwd_ws")
    pu.check(d, ref_out, ref_fin, o_ref, f_ref, label="kda_fwd")
    with pytest.raises(kda.KDAError) as ei:
        kda.kda_fwd(e["q"], e["k"], e["v"], e["g"], e["beta"], d["scale"], out, e["A_log"],
                    e["dt_bias"], d["lower_bound"], initial_state=e["initial_state"],
                    final_state=fin, cu_seqlens=e["cu_seqlens"], workspace=ws[:-16])
    assert ei.value.status == kda.KDA_ERR_VALUE


def test_caller_workspace_pool_path():
    # a fixed-length kda_fwd_ws call whose workspace holds kda_workspace_size_pool bytes
    # runs the pool kernel (one with the cluster kernel's size runs the cluster kernel):
    # both match the oracle, and garbage in the workspace gives the result of zeros
    d = W.make_inputs(W.get("prefill_8k", B=2, T=300, H=3, seed=96, state_dtype="fp32"))
    e = pu.to_device(d)
    n_pool, n_cluster = kda.workspace_bytes_pool(d["N"], d["H"]), kda.workspace_bytes(d["N"], d["H"])
    assert n_pool >= n_cluster > 0
    ref_out, ref_fin = pu.run_oracle(d)
    res = []
    for size, fill in ((n_pool, 0x00), (n_pool, 0xFF), (n_cluster, 0xFF)):
        out = torch.empty((d["B"], d["T"], d["H"], 128), dtype=torch.bfloat16, device="cuda")
        fin = torch.empty((d["N"], d["H"], 128, 128), dtype=torch.float32, device="cuda")
        ws = torch.full((size,), fill, dtype=torch.uint8, device="cuda")
        kda.kda_fwd(e["q"], e["k"], e["v"], e["g"], e["beta"], d["scale"], out, e["A_log"],
                    e["dt_bias"], d["lower_bound"], initial_state=e["initial_state"], final_state=fin,
                    workspace=ws)
        torch.cuda.synchronize()
        assert kda.get_device_status() == kda.KDA_OK
        pu.check(d, out.cpu(), fin.cpu(), ref_out, ref_fin, label=f"kda_fwd_ws {size} bytes")
        res.append((out.cpu(), fin.cpu()))
    assert torch.equal(res[0][0], res[1][0]) and torch.equal(res[0][1], res[1][1])
    # the pool path gives kda_fwd's results bit for bit (same kernel, same inputs)
    out2, fin2 = pu.run_gpu(d)
    assert torch.equal(out2, res[0][0]) and torch.equal(fin2.float(), res[0][1].float())


# ---- short steps (T <= 64 token rows): the token recurrence (T = 1) and the 16-row-block kernel

@pytest.mark.parametrize("T,sd,init", [(1, "fp32", "normal"), (1, "bf16", "none"), (1, None, "normal"),
                                       (3, "bf16", "normal"), (16, "fp32", "none"),
                                       (16, "bf16", "normal"), (5, None, "none")])
def test_short_step_all_elements(T, sd, init):
    d = W.make_inputs(W.get("decode", B=5, T=T, H=3, state_dtype=sd, initial_state=init))
    out, fin = pu.run_gpu(d, want_final=sd is not None)
    ref_out, ref_fin = pu.run_oracle(d, want_final=sd is not None)
    print("short", T, sd, init, pu.check(d, out, fin, ref_out, ref_fin, label=f"short T={T}"))


@pytest.mark.parametrize("seqlens", [(1, 0, 5, 10, 0), (0, 1, 0, 0, 0)])
def test_short_step_varlen_with_empty_sequences(seqlens):
    # (0, 1, 0, 0, 0): one packed token, so the one-token kernel with cu_seqlens
    d = W.make_inputs(W.get("varlen_ragged", H=2, seqlens=seqlens))
    assert d["T"] <= 16
    out, fin = pu.run_gpu(d)
    ref_out, ref_fin = pu.run_oracle(d)
    pu.check(d, out, fin, ref_out, ref_fin, label="short varlen")
    # zero-length sequences pass their state through unchanged
    for n in [i for i, L in enumerate(seqlens) if L == 0]:
        torch.testing.assert_close(fin[n], d["initial_state"][n].to(fin.dtype), rtol=0, atol=0)


@pytest.mark.parametrize("name", ["decode", "decode_16", "step_64", "varlen_short"])
def test_short_step_full_size_all_elements(name):
    d = W.make_inputs(W.get(name))
    out, fin = pu.run_gpu(d)
    print(name, pu.check_full(d, out, fin, label=name))


def test_short_and_chunked_paths_agree_at_the_threshold():
    # T = 64 runs the 16-row-block kernel, T = 65 the chunked kernel; their first 64
    # outputs must agree within the parity tolerances.
    d65 = W.make_inputs(W.get("decode", B=3, T=65, H=2))
    d64 = dict(d65, T=64, q=d65["q"][:, :64], k=d65["k"][:, :64], v=d65["v"][:, :64],
               g=d65["g"][:, :64], beta=d65["beta"][:, :64])
    d64 = {kk: (vv.contiguous() if torch.is_tensor(vv) else vv) for kk, vv in d64.items()}
    o65, _ = pu.run_gpu(d65)
    o64, _ = pu.run_gpu(d64)
    mx, rl = pu.errors(o64.float().numpy(), o65[:, :64].float().numpy())
    assert mx <= pu.OUT_MAX_ABS and rl <= pu.OUT_REL_L2, (mx, rl)


@pytest.mark.parametrize("T,sd,init", [(17, "fp32", "normal"), (33, "bf16", "normal"),
                                       (64, "fp32", "none"), (48, None, "none")])
def test_multi_block_steps_all_elements(T, sd, init):
    # 17..64 token rows: the state stays in registers across the 16-row blocks
    d = W.make_inputs(W.get("decode", B=4, T=T, H=3, state_dtype=sd, initial_state=init, seed=30 + T))
    out, fin = pu.run_gpu(d, want_final=sd is not None)
    ref_out, ref_fin = pu.run_oracle(d, want_final=sd is not None)
    print("multi-block", T, sd, init, pu.check(d, out, fin, ref_out, ref_fin, label=f"multi-block T={T}"))


def test_multi_block_varlen_with_empty_sequences():
    d = W.make_inputs(W.get("varlen_ragged", H=2, seqlens=(30, 0, 1, 17, 0, 16)))
    assert 16 < d["T"] <= 64
    out, fin = pu.run_gpu(d)
    ref_out, ref_fin = pu.run_oracle(d)
    pu.check(d, out, fin, ref_out, ref_fin, label="multi-block varlen")
    for n in (1, 4):
        torch.testing.assert_close(fin[n], d["initial_state"][n].to(fin.dtype), rtol=0, atol=0)


# ---- seeded random configurations: shapes, lengths (empty, short, chunk-crossing),
# state types, gate lower bounds and input spreads drawn per case; both kernels

def _random_case(i):
    r = np.random.default_rng(9000 + i)
    H = int(r.integers(1, 6))
    sd = [None, "fp32", "bf16"][int(r.integers(3))]
    init = ["none", "normal", "alternate"][int(r.integers(3))]
    common = dict(H=H, seed=9000 + i, state_dtype=sd, initial_state=init,
                  lower_bound=float(r.uniform(-5.0, 0.0)),
                  g_std=float(r.choice([0.5, 1.0, 2.0, 3.0])),
                  beta_mean=float(r.choice([-2.0, 0.0, 2.0])),
                  state_std=float(r.choice([0.02, 0.3])))
    short = i % 3 == 0
    if i % 2 == 0:
        T = int(r.integers(1, 17)) if short else int(r.integers(17, 400))
        return W.Workload(name=f"rand{i}", B=int(r.integers(1, 4)), T=T, **common)
    n = int(r.integers(1, 7))
    if short:
        lens = [int(x) for x in r.integers(0, 4, size=n)]
    else:
        lens = [int(r.choice([0, int(r.integers(1, 17)), int(r.integers(17, 300))])) for _ in range(n)]
    return W.Workload(name=f"rand{i}", B=1, T=0, varlen="ragged", n_seqs=n,
                      seqlens=tuple(lens), **common)


@pytest.mark.parametrize("i", range(12))
def test_random_configurations_without_a_lower_bound(i):
    # the same random shapes with the gate without a lower bound (the pool kernel's
    # chunked form above 64 rows, the token recurrence below)
    w = _random_case(100 + i)
    w = W.Workload(**{**w.__dict__, "lower_bound": None, "name": f"urand{i}"})
    d = W.make_inputs(w)
    assert d["lower_bound"] is None
    want = w.state_dtype is not None
    out, fin = pu.run_gpu(d, want_final=want)
    ref_out, ref_fin = pu.run_oracle(d, want_final=want)
    print(w.name, pu.check(d, out, fin, ref_out, ref_fin, label=w.name))


@pytest.mark.parametrize("i", range(18))
def test_random_configurations(i):
    w = _random_case(i)
    d = W.make_inputs(w)
    want = w.state_dtype is not None
    out, fin = pu.run_gpu(d, want_final=want)
    ref_out, ref_fin = pu.run_oracle(d, want_final=want)
    print(w, pu.check(d, out, fin, ref_out, ref_fin, label=w.name))


# ---- sequence-parallel prefill: fixed-length calls with few (sequence, head) units and
# T >= 8192 run the T-split path (segments, their affine state maps, a scan, a re-run)

@pytest.mark.parametrize("B,T,H,sd,init", [(1, 8192, 2, "bf16", "normal"),
                                           (2, 8200, 1, "fp32", "alternate"),
                                           (1, 8192, 3, None, "none")])
def test_sequence_parallel_prefill_all_elements(B, T, H, sd, init):
    d = W.make_inputs(W.get("prefill_8k", B=B, T=T, H=H, seed=11 + T + H, state_dtype=sd,
                            initial_state=init, state_std=0.3))
    want = sd is not None
    out, fin = pu.run_gpu(d, want_final=want)
    ref_out, ref_fin = pu.run_oracle(d, want_final=want)
    print("tsplit", B, T, H, sd, pu.check(d, out, fin, ref_out, ref_fin, label=f"tsplit B={B} T={T} H={H}"))


def test_sequence_parallel_and_plain_paths_agree():
    # kda_fwd runs the segmented path at this size; kda_fwd_ws (caller workspace) always
    # runs the plain one.  Both must agree within the parity tolerances.
    d = W.make_inputs(W.get("prefill_8k", B=1, T=8192, H=2, seed=21, state_dtype="fp32"))
    e = pu.to_device(d)
    o_seg, f_seg = pu.run_gpu(d)
    out = torch.empty_like(e["q"])
    fin = torch.empty((d["N"], d["H"], 128, 128), dtype=torch.float32, device="cuda")
    ws = torch.empty(kda.workspace_bytes(d["N"], d["H"]), dtype=torch.uint8, device="cuda")
    kda.kda_fwd(e["q"], e["k"], e["v"], e["g"], e["beta"], d["scale"], out, e["A_log"], e["dt_bias"],
                d["lower_bound"], initial_state=e["initial_state"], final_state=fin, workspace=ws)
    torch.cuda.synchronize()
    assert kda.get_device_status() == kda.KDA_OK
    mx, rl = pu.errors(o_seg.float().numpy(), out.cpu().float().numpy())
    assert mx <= pu.OUT_MAX_ABS and rl <= pu.OUT_REL_L2, (mx, rl)
    _, srl = pu.errors(f_seg.numpy(), fin.cpu().numpy())
    assert srl <= pu.STATE_REL_L2["fp32"], srl


@pytest.mark.parametrize("init,want_final", [("none", True), ("normal", False)])
def test_sequence_parallel_state_options(init, want_final):
    d = W.make_inputs(W.get("prefill_8k", B=1, T=8192, H=2, seed=22, state_dtype="fp32",
                            initial_state=init))
    out, fin = pu.run_gpu(d, want_final=want_final)
    ref_out, ref_fin = pu.run_oracle(d, want_final=want_final)
    pu.check(d, out, fin, ref_out, ref_fin, label=f"tsplit init={init} final={want_final}")


# ---- varlen batches of mostly short sequences (packed T > 64, at most 256 rows per
# sequence on average): the 16-row-block kernel takes the sequences of at most 64 tokens,
# the cluster kernel the rest

@pytest.mark.parametrize("seqlens,sd", [((3, 40, 64, 65, 0, 200, 17, 1, 50, 16, 33), "bf16"),
                                        (tuple(range(1, 65, 3)), "fp32")])
def test_mixed_length_batches(seqlens, sd):
    d = W.make_inputs(W.get("varlen_ragged", H=3, seqlens=seqlens, state_dtype=sd, seed=40 + len(seqlens)))
    assert d["T"] > 64 and d["T"] <= 256 * len(seqlens)
    out, fin = pu.run_gpu(d)
    ref_out, ref_fin = pu.run_oracle(d)
    print("mixed", seqlens[:4], sd, pu.check(d, out, fin, ref_out, ref_fin, label="mixed-length varlen"))
    n0 = seqlens.index(0) if 0 in seqlens else None
    if n0 is not None:   # a zero-length sequence passes its state through
        torch.testing.assert_close(fin[n0], d["initial_state"][n0].to(fin.dtype), rtol=0, atol=0)


@pytest.mark.parametrize("name,wl", [("decode", dict(B=2, T=1, H=2)), ("short", dict(B=2, T=8, H=2)),
                                     ("prefill", dict(B=1, T=300, H=2)),
                                     ("sequence_parallel", dict(B=1, T=8192, H=2))])
def test_cuda_graph_capture_replays_the_call(name, wl):
    # A serving loop captures kda_fwd in a CUDA graph: the workspace is stream-ordered
    # pool memory and every launch goes to the capturing stream, so a replay must give
    # the direct call's results exactly.  T=8192 with 2 units takes the sequence-parallel
    # path (segment kernels, two plan + pool runs with their flag clears, the scan).
    d = W.make_inputs(W.get("decode", state_dtype="fp32", seed=50, **wl))
    e = pu.to_device(d)
    out = torch.empty((d["B"], d["T"], d["H"], 128), dtype=torch.bfloat16, device="cuda")
    fin = torch.empty((d["N"], d["H"], 128, 128), dtype=torch.float32, device="cuda")

    def call():
        kda.kda_fwd(e["q"], e["k"], e["v"], e["g"], e["beta"], d["scale"], out, e["A_log"], e["dt_bias"],
                    d["lower_bound"], initial_state=e["initial_state"], final_state=fin)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        call()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    ref_out, ref_fin = out.clone(), fin.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    out.zero_()
    fin.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert kda.get_device_status() == kda.KDA_OK
    assert torch.equal(out, ref_out) and torch.equal(fin, ref_fin)
    # A serving loop replays the graph on new inputs written into the same buffers: every
    # replay must see only its own data (no state carried between replays of the call)
    d2 = W.make_inputs(W.get("decode", state_dtype="fp32", seed=51, **wl))
    for key in ("q", "k", "v", "g", "beta", "initial_state"):
        e[key].copy_(d2[key].to(e[key].device))
    call()
    torch.cuda.synchronize()
    ref_out2, ref_fin2 = out.clone(), fin.clone()
    assert not torch.equal(ref_out2, ref_out)
    for _ in range(2):
        out.zero_()
        fin.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert kda.get_device_status() == kda.KDA_OK
        assert torch.equal(out, ref_out2) and torch.equal(fin, ref_fin2)


# ---- the gate without a lower bound (kda_fwd_unbounded: the pool kernel's chunked form above
# 64 rows, the token recurrence for short calls)

@pytest.mark.parametrize("B,T,H,sd,init,g_std", [(2, 300, 3, "fp32", "normal", 1.0),
                                                 (1, 1, 4, "bf16", "normal", 1.0),
                                                 (3, 70, 2, None, "none", 1.0),
                                                 (2, 17, 2, "bf16", "none", 1.0),
                                                 (1, 200, 2, "fp32", "alternate", 3.0),
                                                 (40, 33, 2, "bf16", "normal", 1.0)])
def test_unbounded_gate_all_elements(B, T, H, sd, init, g_std):
    # up to 76 (sequence, head) units the kernel sums k^T S and q^T S in one reduction;
    # the 80-unit case (160 CTAs on 152 SMs) takes the two-reduction form
    d = W.make_inputs(W.get("tiny", B=B, T=T, H=H, state_dtype=sd, initial_state=init, g_std=g_std,
                            lower_bound=None, seed=40 + T))
    assert d["lower_bound"] is None
    out, fin = pu.run_gpu(d, want_final=sd is not None)
    ref_out, ref_fin = pu.run_oracle(d, want_final=sd is not None)
    print("unbounded", B, T, H, sd, init, pu.check(d, out, fin, ref_out, ref_fin, label=f"unbounded T={T}"))


@pytest.mark.parametrize("case", ["all", "half", "varlen"])
def test_unbounded_gate_extreme_decays(case):
    # softplus(g + dt_bias) near 30 gives per-token decays of e^-30 to e^-480 (past e^-60
    # wherever exp(A_log) > 2); the chunked form raises each token's log2 decay to -14
    # (a factor 2^-14 where the exact one is smaller), so the parity bars still hold
    w = W.get("tiny", B=2, T=300, H=3, state_dtype="fp32", initial_state="normal", lower_bound=None, seed=93)
    if case == "varlen":
        w = W.get("varlen_ragged", H=3, seqlens=(300, 1, 129, 0, 70), lower_bound=None, seed=94)
    d = W.make_inputs(w)
    g = d["g"].float()
    if case == "half":
        mask = torch.rand(g.shape[:-1], generator=torch.Generator().manual_seed(5)) < 0.5
        g[mask] = 30.0
    else:
        g[:] = 30.0
    d["g"] = g.to(torch.bfloat16)
    out, fin = pu.run_gpu(d)
    ref_out, ref_fin = pu.run_oracle(d)
    print("unbounded extreme", case, pu.check(d, out, fin, ref_out, ref_fin, label=f"unbounded extreme {case}"))


def test_unbounded_gate_varlen_with_empty_sequences():
    seqlens = (0, 5, 130, 0, 1, 64)
    d = W.make_inputs(W.get("varlen_ragged", H=2, seqlens=seqlens, lower_bound=None))
    out, fin = pu.run_gpu(d)
    ref_out, ref_fin = pu.run_oracle(d)
    pu.check(d, out, fin, ref_out, ref_fin, label="unbounded varlen")
    for n in [i for i, L in enumerate(seqlens) if L == 0]:
        torch.testing.assert_close(fin[n], d["initial_state"][n].to(fin.dtype), rtol=0, atol=0)


def test_unbounded_gate_full_size_all_elements():
    d = W.make_inputs(W.get("prefill_8k_unbounded"))
    out, fin = pu.run_gpu(d)
    print("prefill_8k_unbounded", pu.check_full(d, out, fin, label="prefill_8k_unbounded"))


def test_unbounded_and_bounded_gates_differ():
    # the two entry points compute different gates on the same inputs
    d = W.make_inputs(W.get("tiny", T=64, H=2))
    du = dict(d, lower_bound=None)
    o_b, _ = pu.run_gpu(d)
    o_u, _ = pu.run_gpu(du)
    assert (o_b.float() - o_u.float()).abs().max() > 1e-2


@pytest.mark.parametrize("sd", ["fp32", "bf16"])
def test_unbounded_gate_zero_length_passes_state_through(sd):
    d = W.make_inputs(W.get("batch_state", B=2, T=0, H=3, state_dtype=sd, lower_bound=None))
    out, fin = pu.run_gpu(d)
    assert out.numel() == 0
    torch.testing.assert_close(fin, d["initial_state"].to(fin.dtype), rtol=0, atol=0)
    # and a varlen call whose sequences are all empty
    dv = W.make_inputs(W.get("varlen_ragged", H=2, seqlens=(0, 0, 0), lower_bound=None))
    assert dv["T"] == 0
    out, fin = pu.run_gpu(dv)
    torch.testing.assert_close(fin, dv["initial_state"].to(fin.dtype), rtol=0, atol=0)


# ---- corners: long sequence-parallel splits, saturated gates, the fp16 operand range

@pytest.mark.parametrize("name,over,segments", [("prefill_64k_h8", {}, 7),
                                                ("prefill_8k", dict(T=65536, H=1, seed=77), 32)])
def test_sequence_parallel_prefill_long_splits(name, over, segments):
    # T = 65536 with 8 (sequence, head) units runs 7 segments per sequence, with one unit
    # 32 (the most the path takes): the fp32 scan over 7 and 32 segment maps
    d = W.make_inputs(W.get(name, **over))
    out, fin = pu.run_gpu(d)
    print(name, segments, pu.check_full(d, out, fin, label=f"{name} ({segments} segments)"))


@pytest.mark.parametrize("T,H", [(8192, 2), (65536, 8)])
def test_sequence_parallel_unbounded_gate(T, H):
    # the gate without a lower bound takes the sequence-parallel path too (4 and 8
    # segments): the floored per-token decays make the same affine segment maps
    d = W.make_inputs(W.get("prefill_8k", B=1, T=T, H=H, seed=95 + H, state_dtype="fp32",
                            lower_bound=None, g_std=1.5))
    out, fin = pu.run_gpu(d)
    print(T, H, pu.check_full(d, out, fin, label=f"unbounded sequence-parallel T={T} H={H}"))


@pytest.mark.parametrize("g_value", [30.0, -30.0])
@pytest.mark.parametrize("case", ["fixed", "varlen", "short"])
def test_saturated_gate(case, g_value):
    # g = +30: the gate sits at lower_bound = -5 on every token and channel (the 16-token
    # blocks span e^-80, the largest range the factored operands meet); g = -30: no decay
    wl = {"fixed": W.get("prefill_8k", T=1000, H=4, seed=81),
          "varlen": W.get("varlen_ragged", H=3, seqlens=(65, 1, 130, 63, 200), seed=82),
          "short": W.get("decode", B=3, T=40, H=2, seed=83)}[case]
    d = W.make_inputs(wl)
    d["g"] = torch.full_like(d["g"], g_value)
    out, fin = pu.run_gpu(d)
    ref_out, ref_fin = pu.run_oracle(d)
    print(case, g_value, pu.check(d, out, fin, ref_out, ref_fin, label=f"saturated {case} g={g_value}"))


def _call_status(d):
    e = pu.to_device(d)
    out = torch.empty((d["B"], d["T"], d["H"], 128), dtype=torch.bfloat16, device="cuda")
    fin = torch.empty((d["N"], d["H"], 128, 128), dtype=pu.state_torch_dtype(d["state_dtype"]),
                      device="cuda")
    kda.kda_fwd(e["q"], e["k"], e["v"], e["g"], e["beta"], d["scale"], out, e["A_log"],
                e["dt_bias"], d["lower_bound"], initial_state=e["initial_state"], final_state=fin,
                cu_seqlens=e["cu_seqlens"])
    return kda.get_device_status()


@pytest.mark.parametrize("case", ["fixed", "varlen", "short", "unbounded", "sequence_parallel"])
@pytest.mark.parametrize("where", ["v", "state"])
def test_fp16_operand_range_is_reported(case, where):
    # a value beyond +-65504 where the tensor-core paths keep fp16 operands sets
    # KDA_ERR_RANGE in the device status word, which the next status read clears (the
    # gate without a lower bound in its chunked form, and the sequence-parallel runs,
    # included)
    wl = {"fixed": W.get("prefill_8k", T=300, H=2, seed=84, state_dtype="fp32"),
          "varlen": W.get("varlen_ragged", H=2, seqlens=(70, 130), seed=85),
          "short": W.get("decode", B=2, T=8, H=2, seed=86),
          "unbounded": W.get("prefill_8k", T=300, H=2, seed=88, state_dtype="fp32", lower_bound=None),
          "sequence_parallel": W.get("prefill_8k", T=8192, H=2, seed=89, state_dtype="fp32")}[case]
    d = W.make_inputs(wl)
    assert _call_status(d) == kda.KDA_OK
    if where == "v":
        d["v"] = d["v"].clone()
        d["v"][0, 3, 1, 5] = 1.0e5
    else:
        d["initial_state"] = d["initial_state"].clone()
        d["initial_state"][-1, 1, 7, 9] = 1.0e5
    assert _call_status(d) == kda.KDA_ERR_RANGE
    assert kda.get_device_status() == kda.KDA_OK   # cleared by the read


def test_one_token_step_has_no_fp16_limit():
    # T = 1 runs the fp32 token recurrence: values far beyond the fp16 range are fine
    d = W.make_inputs(W.get("decode", B=2, T=1, H=2, seed=87))
    d["v"] = d["v"] * 1.0e5
    d["initial_state"] = d["initial_state"] * 1.0e5
    out, fin = pu.run_gpu(d)
    ref_out, ref_fin = pu.run_oracle(d)
    pu.check(d, out.float() / 1.0e5, fin / 1.0e5, ref_out / 1.0e5, ref_fin / 1.0e5,
             label="decode large values")
