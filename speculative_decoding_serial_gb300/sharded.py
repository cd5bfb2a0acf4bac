"""A vocabulary sharded over GPUs, one process per GPU (torch.distributed).

Each rank holds rows [lo, hi) of W (cut on 16-row group boundaries) and the base logits of those rows. It
walks them one step at a time through the C ABI (whead_walk_keys with gamma = 1). The ranks agree on each
step's winner as the largest packed key over all ranks: Fig. 8's packed selection, taken across GPUs by an
all-reduce MAX. Every rank then advances the state from that winner on its own GPU (whead_advance), so only
B packed keys cross between GPUs per step.

The packed keys are uint64 (ord(key) << 32 | (2^32 - 1 - row)). torch.distributed reduces int64, so the
keys travel with their top bit flipped, which maps uint64 order onto int64 order.

This is host plumbing around the library's kernels: the projection, selection and advance all run on the
GPU, and a rank's only collective is the all-reduce of B int64 per step.
"""
from __future__ import annotations

from typing import Callable

GROUP_ROWS = 16
_FLIP = -(1 << 63)  # int64 with only the top bit set


def shard_bounds(V: int, world: int, rank: int) -> tuple[int, int]:
    """Rows [lo, hi) of rank `rank` out of `world`: whole 16-row groups, as even as possible, in rank order."""
    groups = (V + GROUP_ROWS - 1) // GROUP_ROWS
    per = groups // world
    extra = groups % world
    g0 = rank * per + min(rank, extra)
    g1 = g0 + per + (1 if rank < extra else 0)
    return min(V, g0 * GROUP_ROWS), min(V, g1 * GROUP_ROWS)


def to_ordered(keys):
    """uint64 keys (held as int64 bits) to int64 values with the same order (flip the top bit)."""
    return keys ^ _FLIP


def from_ordered(vals):
    return vals ^ _FLIP


def row_of_key(keys):
    """Global row of each packed key (the low 32 bits hold 2^32 - 1 - row)."""
    import torch
    return (0xFFFFFFFF - (keys & 0xFFFFFFFF)).to(torch.int32)


class ShardedWalk:
    """The per-step protocol. step(t, s) -> this rank's winning packed keys (B,) int64 for step t from state s;
    merge(ordered keys) -> their maximum over all ranks (in place or returned); advance(x, s) -> next state."""

    def __init__(self, step: Callable, merge: Callable, advance: Callable):
        self.step, self.merge, self.advance = step, merge, advance

    def walk(self, s0, gamma: int):
        """Returns (tokens (B, gamma) int32 global rows, states (B, gamma, r): the state after each step)."""
        import torch
        s = s0
        toks, states = [], []
        for t in range(gamma):
            keys = self.step(t, s)
            merged = from_ordered(self.merge(to_ordered(keys)))
            x = row_of_key(merged)
            s = self.advance(x, s)
            toks.append(x)
            states.append(s)
        return torch.stack(toks, dim=1), torch.stack(states, dim=1)


def allreduce_max(group=None):
    """merge() over a torch.distributed process group (NCCL for CUDA tensors, gloo for CPU ones)."""
    import torch.distributed as dist

    def merge(v):
        dist.all_reduce(v, op=dist.ReduceOp.MAX, group=group)
        return v
    return merge


class ShardedHead:
    """One rank's shard on its GPU. W_shard: rows [lo, hi) of W (hi - lo rows, bf16, contiguous). E: every row of
    E (bf16, V x r). A, c: the recurrent head's, on every rank. base_shard: (B, gamma, hi - lo) fp32."""

    def __init__(self, W_shard, E, lo: int, *, kind=0, A=None, c=None, max_B=1, T=0.0, seed=0, group=None,
                 merge: Callable | None = None, **head_kwargs):
        from . import whead as wh
        if W_shard.shape[0] == 0:
            raise ValueError("empty shard: more ranks than 16-row groups of the vocabulary")
        self.head = wh.Head(W_shard, E, kind=kind, A=A, c=c, max_B=max_B, max_gamma=1, v_offset=lo,
                            e_rows=int(E.shape[0]), **head_kwargs)
        self.lo, self.T, self.seed = lo, float(T), int(seed)
        self.merge = merge if merge is not None else allreduce_max(group)

    def walk(self, base_shard, s0):
        import torch
        B, gamma, _ = base_shard.shape
        steps = [base_shard[:, t:t + 1].contiguous() for t in range(gamma)]
        tok = torch.empty((B, 1), dtype=torch.int32, device=s0.device)
        keys = torch.empty((B, 1), dtype=torch.int64, device=s0.device)

        def step(t, s):
            self.head.walk_keys(steps[t], s.contiguous(), T=self.T, seed=self.seed, t0=t, out_tokens=tok,
                                out_keys=keys)
            return keys[:, 0].clone()

        def advance(x, s):
            nxt = torch.empty_like(s)
            return self.head.advance(x.contiguous(), s.contiguous(), nxt)

        return ShardedWalk(step, self.merge, advance).walk(s0, gamma)

    def close(self):
        self.head.close()
