"""Head sharding across GPUs (host logic only).

Heads are independent ("xLSTM", part 17/30: multiple heads are multiple cells
with no memory mixing), so a batch of B*H sequences splits across ranks with
no exchange: each rank runs the parallel forward (or the recurrent step) on a
contiguous block of (b, h) sequences and owns that block of the output.  An
all-gather is needed only if one consumer wants the whole output.
"""
from __future__ import annotations

from typing import Dict, Tuple

import torch


def head_range(num_heads: int, rank: int, world: int) -> Tuple[int, int]:
    """Contiguous block [start, stop) of num_heads flattened (b, h) sequences
    for `rank` of `world`; block sizes differ by at most one."""
    if world <= 0 or not 0 <= rank < world:
        raise ValueError("bad rank/world")
    base, extra = divmod(num_heads, world)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)


def shard_sequences(x: Dict[str, torch.Tensor], rank: int, world: int) -> Dict[str, torch.Tensor]:
    """The rank's block of every [B, H, ...] tensor, flattened to [1, n, ...]."""
    out = {}
    for k, t in x.items():
        flat = t.reshape(t.shape[0] * t.shape[1], *t.shape[2:])
        s, e = head_range(flat.shape[0], rank, world)
        out[k] = flat[s:e].unsqueeze(0).contiguous()
    return out
