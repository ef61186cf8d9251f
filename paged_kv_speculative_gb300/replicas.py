"""Host-side logic for running the path on several GPUs of one node.

Verify attention needs no exchange between ranks: every (sequence, KV head)
is independent. Ranks either run their own batch (replicas, weak scaling) or
take disjoint blocks of one batch's sequences (shards). The only collectives
are host-level: a barrier around the timed region and the maximum of the
ranks' times.
"""
from __future__ import annotations

import numpy as np

from .synth import shard_sequences  # noqa: F401  (re-exported)


def max_over_ranks(value: float, device=None) -> float:
    """Maximum of `value` over the default process group (identity without one)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(value: float, device=None) -> float:
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def job_throughput(bytes_all_ranks: float, steps: int, max_total_ms: float) -> float:
    """Whole-job GB/s: every rank's bytes over the slowest rank's time."""
    return bytes_all_ranks * steps / (max_total_ms * 1e-3) / 1e9


def sub_batch(context_lens, query_lens, world: int, rank: int):
    """(context_lens, query_lens, sequence indices) of this rank's shard."""
    idx = shard_sequences(len(context_lens), world, rank)
    cl = np.asarray(context_lens)[idx]
    ql = np.asarray(query_lens)[idx]
    return cl.tolist(), ql.tolist(), idx
