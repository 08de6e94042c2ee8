"""Head partition of one KDA problem across ranks (one GPU each).

Every (sequence, head) recurrence is independent, so a call splits over the head axis
with no collective on the data path: rank r takes a contiguous block of heads, runs
kda_fwd on its slice of every per-head tensor, and owns the same slice of `out` and of
the final state.  Nothing here computes any part of the method; it only cuts and joins
tensors in the Kernel API layouts (q, k, v, g, out [B,T,H,*]; beta [B,T,H]; A_log [H];
dt_bias [H,K]; states [N,H,V,K]).
"""
from __future__ import annotations


def head_range(rank: int, world: int, H: int) -> tuple[int, int]:
    """Heads [h0, h1) of `rank`: contiguous blocks whose sizes differ by at most one."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError(f"rank {rank} of {world}")
    base, extra = divmod(H, world)
    h0 = rank * base + min(rank, extra)
    return h0, h0 + base + (1 if rank < extra else 0)


# the head axis of each per-head tensor of a call
HEAD_AXIS = {"q": 2, "k": 2, "v": 2, "g": 2, "beta": 2, "out": 2, "A_log": 0, "dt_bias": 0,
             "initial_state": 1, "final_state": 1}


def shard(inputs: dict, rank: int, world: int) -> dict:
    """The rank's slice of a call's inputs (contiguous copies of the per-head tensors;
    every other entry as it is, with "H" set to the slice's head count)."""
    H = int(inputs["H"]) if "H" in inputs else int(inputs["q"].shape[2])
    h0, h1 = head_range(rank, world, H)
    out = {}
    for key, val in inputs.items():
        ax = HEAD_AXIS.get(key)
        if ax is None or val is None:
            out[key] = val
        else:
            out[key] = val.narrow(ax, h0, h1 - h0).contiguous()
    out["H"] = h1 - h0
    return out


def join(parts: list, key: str):
    """The whole tensor `key` from the ranks' slices, in rank order."""
    import torch
    return torch.cat([p for p in parts], dim=HEAD_AXIS[key])
