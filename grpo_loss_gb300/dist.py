"""Data-parallel bookkeeping for the GRPO loss over several ranks.

The loss is token-local apart from two normalisations: advantages are taken
over each group of G generations, and the loss averages over the B
sequences. Sharding whole groups across ranks therefore keeps every row's
arithmetic local. Ranks only need the global sequence count, plus one
scalar all-reduce to form the global loss and KL mean. dH rows need no
exchange at all, and dW needs a sum over ranks like any data-parallel
weight gradient.

Host-side logic only; the per-rank loss itself is computed by the library.
"""
from __future__ import annotations

from typing import Tuple

import torch


def group_shard(num_seqs: int, group_size: int, world_size: int, rank: int) -> Tuple[int, int]:
    """(first sequence, sequence count) of ``rank``'s share, in whole groups.

    Groups are dealt out contiguously and as evenly as possible; a rank may
    receive zero groups when there are fewer groups than ranks.
    """
    if group_size < 1 or num_seqs % group_size:
        raise ValueError("group_size must divide num_seqs")
    if not 0 <= rank < world_size:
        raise ValueError("rank out of range")
    groups = num_seqs // group_size
    base, extra = divmod(groups, world_size)
    g0 = rank * base + min(rank, extra)
    ng = base + (1 if rank < extra else 0)
    return g0 * group_size, ng * group_size


def grad_scale(num_seqs_local: int, num_seqs_global: int) -> float:
    """Upstream gradient to pass to the local backward so that dH equals the
    gradient of the global loss: the local loss averages over its own B
    sequences, the global one over all of them."""
    return num_seqs_local / float(num_seqs_global)


def global_loss(loss_local: float, kl_mean_local: float, num_seqs_local: int,
                valid_local: int, num_seqs_global: int, group=None) -> Tuple[float, float]:
    """Combine per-rank (loss, kl_mean) into the global values with one
    all-reduce of three float64 scalars."""
    import torch.distributed as dist
    t = torch.tensor([loss_local * num_seqs_local / float(num_seqs_global),
                      kl_mean_local * valid_local, float(valid_local)], dtype=torch.float64)
    if dist.is_available() and dist.is_initialized():
        dist.all_reduce(t, op=dist.ReduceOp.SUM, group=group)
    loss = float(t[0])
    kl = float(t[1] / t[2]) if t[2] > 0 else 0.0
    return loss, kl


def reduce_timing(ms_local: float, tokens_local: float, device=None, group=None):
    """(max step time over ranks, total tokens over ranks): the whole-job
    throughput is the second over the first."""
    import torch.distributed as dist
    t = torch.tensor([ms_local], dtype=torch.float64, device=device)
    n = torch.tensor([tokens_local], dtype=torch.float64, device=device)
    if dist.is_available() and dist.is_initialized() and dist.get_world_size(group) > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
        dist.all_reduce(n, op=dist.ReduceOp.SUM, group=group)
    return float(t.item()), float(n.item())
