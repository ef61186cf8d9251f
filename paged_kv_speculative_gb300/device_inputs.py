"""Copies a host batch (``synth.Problem``) to device tensors for the binding."""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np
import torch

from . import synth


@dataclasses.dataclass
class DeviceProblem:
    q: torch.Tensor
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    k_scale: Optional[torch.Tensor]
    v_scale: Optional[torch.Tensor]
    block_table: torch.Tensor
    context_lens: torch.Tensor
    query_lens: torch.Tensor

    def args(self):
        return (self.q, self.k_cache, self.v_cache, self.k_scale, self.v_scale, self.block_table,
                self.context_lens, self.query_lens)


def host_tensors(prob: synth.Problem, pin: bool = False) -> DeviceProblem:
    """The problem as CPU torch tensors (optionally in pinned memory)."""
    def t(a: Optional[np.ndarray], dtype=None):
        if a is None:
            return None
        x = torch.from_numpy(np.ascontiguousarray(a))
        if dtype is not None:
            x = x.view(dtype)
        return x.pin_memory() if pin else x
    kv_dt = torch.bfloat16 if prob.kv_dtype == synth.KV_BF16 else torch.uint8
    kc = prob.k_cache.view(np.int16) if prob.kv_dtype == synth.KV_BF16 else prob.k_cache
    vc = prob.v_cache.view(np.int16) if prob.kv_dtype == synth.KV_BF16 else prob.v_cache
    return DeviceProblem(q=t(prob.q.view(np.int16), torch.bfloat16), k_cache=t(kc, kv_dt), v_cache=t(vc, kv_dt),
                         k_scale=t(prob.k_scale), v_scale=t(prob.v_scale),
                         block_table=t(prob.block_table.astype(np.int32)),
                         context_lens=t(prob.context_lens.astype(np.int32)),
                         query_lens=t(prob.query_lens.astype(np.int32)))


def to_device(prob: synth.Problem, device="cuda") -> DeviceProblem:
    h = host_tensors(prob)
    mv = lambda x: None if x is None else x.to(device, non_blocking=False)
    return DeviceProblem(*(mv(getattr(h, f.name)) for f in dataclasses.fields(DeviceProblem)))
