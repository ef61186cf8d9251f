"""Seeded synthetic inputs for paged verify attention.

This module only draws random numbers and lays them out; it holds none of the
attention arithmetic, so the CPU oracle and the CUDA path can both consume
the exact same bytes.

Layouts (all host numpy arrays, C-contiguous):

* ``q``            uint16 ``[T, Hq, D]``   bf16 bit patterns, sequences packed in order
* ``k_cache``      uint16 ``[N_pg, Hkv, 16, D]`` (bf16 bits) or uint8 (OCP E4M3 bytes)
* ``v_cache``      same as ``k_cache``
* ``k_scale``      float32 ``[N_pg, Hkv, 16]`` per-token, per-head scales (FP8 only)
* ``v_scale``      same
* ``block_table``  int32 ``[B, stride]``, entry ``p`` of row ``b`` is the pool page
                   holding tokens ``16p .. 16p+15`` of sequence ``b``
* ``context_lens`` int32 ``[B]``: all cached tokens, the verify tokens included
* ``query_lens``   int32 ``[B]``: 1..8 verify tokens; they sit at the end of the context

The page-16, head-major-per-page cache and the per-token scales follow the
DSpark P/D page ("page-16 views", "head-major per page") and the MTP-5
routing page (per-token FP8 KV scales with a trailing singleton dimension).

Random draws: K/V/q values are N(0, 1) drawn in fp32 from a seeded torch CPU
generator, then rounded to bf16 (RNE) or quantised per (token, head) to E4M3
with ``s = amax / 448`` (``s = 1`` when ``amax == 0``), clamped to +-448 and
cast with torch's round-to-nearest-even E4M3 conversion. Pool pages are a
seeded permutation handed out to sequences in order, so pages are disjoint
across sequences and scattered in the pool. Unused slots of a sequence's last
page, pool pages no sequence references and block-table entries past a
sequence's last page are poisoned (NaN values, NaN scales, page id -1) when
``poison=True``, so any read of them shows up in the result.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence, Tuple

import numpy as np
import torch

PAGE = 16
KV_BF16 = 0
KV_FP8 = 1
BF16_NAN = 0x7FC0
E4M3_NAN = 0x7F
E4M3_MAX = 448.0


@dataclasses.dataclass
class Problem:
    """One batch of verify-attention inputs (host arrays)."""

    name: str
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    kv_dtype: int
    q: np.ndarray
    k_cache: np.ndarray
    v_cache: np.ndarray
    k_scale: Optional[np.ndarray]
    v_scale: Optional[np.ndarray]
    block_table: np.ndarray
    context_lens: np.ndarray
    query_lens: np.ndarray
    softmax_scale: float
    seed: int

    @property
    def num_seqs(self) -> int:
        return int(self.context_lens.shape[0])

    @property
    def num_pages(self) -> int:
        return int(self.k_cache.shape[0])

    @property
    def num_tokens(self) -> int:
        return int(self.query_lens.sum())

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def kv_bytes(self) -> int:
        """Algorithmic K+V bytes of one call: every cached token of every KV
        head read once (data, plus both fp32 scales for FP8)."""
        per_elem = 2 if self.kv_dtype == KV_BF16 else 1
        per_token_head = 2 * self.head_dim * per_elem + (8 if self.kv_dtype == KV_FP8 else 0)
        return int(self.context_lens.astype(np.int64).sum()) * self.num_kv_heads * per_token_head

    def q_offsets(self) -> np.ndarray:
        off = np.zeros(self.num_seqs + 1, dtype=np.int64)
        off[1:] = np.cumsum(self.query_lens.astype(np.int64))
        return off


def _bf16_bits(x: torch.Tensor) -> np.ndarray:
    return x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _quantise_e4m3(x: torch.Tensor):
    """x: [..., D] fp32 -> (E4M3 bytes [..., D], fp32 scales [...])."""
    amax = x.abs().amax(dim=-1)
    s = torch.where(amax > 0, amax / E4M3_MAX, torch.ones_like(amax))
    y = (x / s.unsqueeze(-1)).clamp(-E4M3_MAX, E4M3_MAX)
    q8 = y.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    return q8, s.numpy().astype(np.float32)


def make_problem(
    context_lens: Sequence[int],
    query_lens: Sequence[int],
    num_q_heads: int,
    num_kv_heads: int,
    head_dim: int,
    kv_dtype: int = KV_BF16,
    seed: int = 0,
    pool_pages: Optional[int] = None,
    extra_pages: int = 2,
    stride_extra: int = 1,
    poison: bool = True,
    softmax_scale: Optional[float] = None,
    name: str = "custom",
    contiguous: bool = False,
    q_row_log2: Optional[Tuple[float, float]] = None,
    k_ramp_log2: float = 0.0,
    v_tok_log2: Optional[Tuple[float, float]] = None,
    zero_frac: float = 0.0,
    tiny_v_frac: float = 0.0,
) -> Problem:
    """Draw one batch. ``pool_pages`` defaults to the pages the batch needs
    plus ``extra_pages`` unreferenced ones. ``contiguous`` hands pages out in
    pool order (block table = identity runs) instead of a random permutation.

    Value-distribution knobs (all off by default; when on, their random
    numbers come from a second generator, so the default draws are unchanged).
    Each multiplies the fp32 draw before rounding to bf16 or quantising:

    * ``q_row_log2 = (lo, hi)``: every (token, q head) row of q times 2^u,
      u ~ U[lo, hi] (rows of widely different norms).
    * ``k_ramp_log2 = a``: the K row of position t of a sequence of L tokens
      times 2^(a t / (L - 1)) (key norms, hence scores, growing along the
      context, so that later tiles beat earlier maxima).
    * ``v_tok_log2 = (lo, hi)``: every (token, KV head) V row times 2^u,
      u ~ U[lo, hi] (FP8: per-token scales spread over several decades).
    * ``zero_frac``: that fraction of (token, KV head) rows has K and V all
      zero (FP8: amax = 0, so both scales are 1).
    * ``tiny_v_frac``: that fraction of (token, KV head) V rows times 2^-104
      (FP8: a V scale far below 2^-100).
    """
    ctx = np.asarray(context_lens, dtype=np.int32)
    ql = np.asarray(query_lens, dtype=np.int32)
    assert ctx.shape == ql.shape and ctx.ndim == 1
    B = ctx.shape[0]
    D = head_dim
    Hq, Hkv = num_q_heads, num_kv_heads
    g = torch.Generator().manual_seed(int(seed))
    pages_per_seq = [(int(L) + PAGE - 1) // PAGE for L in ctx]
    need = sum(pages_per_seq)
    n_pg = need + extra_pages if pool_pages is None else int(pool_pages)
    assert n_pg >= need, "pool smaller than the batch needs"
    perm = torch.arange(n_pg) if contiguous else torch.randperm(n_pg, generator=g)
    perm = perm.numpy().astype(np.int32)
    stride = max(pages_per_seq + [1]) + stride_extra
    table = np.full((B, stride), -1 if poison else 0, dtype=np.int32)
    pos = 0
    for b, npg in enumerate(pages_per_seq):
        table[b, :npg] = perm[pos:pos + npg]
        pos += npg

    T = int(ql.sum())
    qf = torch.randn((T, Hq, D), generator=g, dtype=torch.float32)
    knobs = q_row_log2 is not None or k_ramp_log2 != 0.0 or v_tok_log2 is not None or zero_frac > 0 or tiny_v_frac > 0
    g2 = torch.Generator().manual_seed(int(seed) * 7919 + 17) if knobs else None
    if q_row_log2 is not None:
        lo, hi = q_row_log2
        qf = qf * torch.exp2(lo + (hi - lo) * torch.rand((T, Hq, 1), generator=g2, dtype=torch.float32))
    q = _bf16_bits(qf)

    # position of every pool slot in its sequence (-1: not referenced) and that sequence's length
    slot_pos = np.full((n_pg, PAGE), -1, dtype=np.int64)
    slot_len = np.ones((n_pg, PAGE), dtype=np.int64)
    for b, npg in enumerate(pages_per_seq):
        for j in range(npg):
            slot_pos[table[b, j]] = 16 * j + np.arange(PAGE)
            slot_len[table[b, j]] = int(ctx[b])

    def token_factor(which: int, p0: int, p1: int) -> Optional[torch.Tensor]:
        """[p1 - p0, Hkv, 16, 1] multiplier of pool slots for K (which 0) or V (1), or None."""
        if not knobs:
            return None
        f = torch.ones((p1 - p0, Hkv, PAGE), dtype=torch.float32)
        if which == 0 and k_ramp_log2 != 0.0:
            pos = torch.from_numpy(np.maximum(slot_pos[p0:p1], 0)).float()
            span = torch.from_numpy(np.maximum(slot_len[p0:p1] - 1, 1)).float()
            f = f * torch.exp2(k_ramp_log2 * pos / span).unsqueeze(1)
        if which == 1 and v_tok_log2 is not None:
            lo, hi = v_tok_log2
            f = f * torch.exp2(lo + (hi - lo) * torch.rand(f.shape, generator=g2, dtype=torch.float32))
        if zero_frac > 0:
            # the same rows for K and V: the draw for K is kept and reused for V
            if which == 0:
                token_factor.zero = torch.rand(f.shape, generator=g2) < zero_frac
            f = torch.where(token_factor.zero, torch.zeros_like(f), f)
        if which == 1 and tiny_v_frac > 0:
            f = torch.where(torch.rand(f.shape, generator=g2) < tiny_v_frac, f * 2.0 ** -104, f)
        return f.unsqueeze(-1)

    # K/V for the whole pool, drawn page block by page block to bound memory.
    if kv_dtype == KV_BF16:
        k_cache = np.empty((n_pg, Hkv, PAGE, D), dtype=np.uint16)
        v_cache = np.empty((n_pg, Hkv, PAGE, D), dtype=np.uint16)
        k_scale = v_scale = None
    else:
        k_cache = np.empty((n_pg, Hkv, PAGE, D), dtype=np.uint8)
        v_cache = np.empty((n_pg, Hkv, PAGE, D), dtype=np.uint8)
        k_scale = np.empty((n_pg, Hkv, PAGE), dtype=np.float32)
        v_scale = np.empty((n_pg, Hkv, PAGE), dtype=np.float32)
    blk = max(1, (1 << 22) // max(1, Hkv * PAGE * D))
    zero_rows = {}
    for which, (dst, sc) in enumerate(((k_cache, k_scale), (v_cache, v_scale))):
        for p0 in range(0, n_pg, blk):
            p1 = min(n_pg, p0 + blk)
            x = torch.randn((p1 - p0, Hkv, PAGE, D), generator=g, dtype=torch.float32)
            if knobs:
                if zero_frac > 0 and which == 1:
                    token_factor.zero = zero_rows[p0]
                f = token_factor(which, p0, p1)
                if zero_frac > 0 and which == 0:
                    zero_rows[p0] = token_factor.zero
                x = x * f
            if kv_dtype == KV_BF16:
                dst[p0:p1] = _bf16_bits(x)
            else:
                q8, s = _quantise_e4m3(x)
                dst[p0:p1] = q8
                sc[p0:p1] = s

    if poison:
        nan_val = BF16_NAN if kv_dtype == KV_BF16 else E4M3_NAN
        used = np.zeros(n_pg, dtype=bool)
        for b, npg in enumerate(pages_per_seq):
            pages = table[b, :npg]
            used[pages] = True
            tail = int(ctx[b]) - (npg - 1) * PAGE  # valid slots in the last page
            if npg > 0 and tail < PAGE:
                last = pages[-1]
                k_cache[last, :, tail:, :] = nan_val
                v_cache[last, :, tail:, :] = nan_val
                if k_scale is not None:
                    k_scale[last, :, tail:] = np.nan
                    v_scale[last, :, tail:] = np.nan
        k_cache[~used] = nan_val
        v_cache[~used] = nan_val
        if k_scale is not None:
            k_scale[~used] = np.nan
            v_scale[~used] = np.nan

    sm = 1.0 / math.sqrt(D) if softmax_scale is None else float(softmax_scale)
    return Problem(name=name, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D, kv_dtype=kv_dtype,
                   q=q, k_cache=k_cache, v_cache=v_cache, k_scale=k_scale, v_scale=v_scale,
                   block_table=table, context_lens=ctx, query_lens=ql, softmax_scale=sm, seed=int(seed))


# --------------------------------------------------------------------------
# The five workloads. Lengths are drawn from their own generator (seeded with
# the workload's seed) before any value is drawn.
# --------------------------------------------------------------------------

CONFIG_NAMES = ("tiny", "mtp5_bf16", "mtp5_fp8", "mixed_fp8", "ctx1mi_bf16")
# The head_dim-256 FP8 shape of the aiter follow-up on the MTP-5 routing page:
# GQA 8 x query length 6 = 48 rows over one KV head, context 150,000 tokens,
# batch 1, 2, 4 or 8.
EXTRA_NAMES = ("d256_fp8_bs1", "d256_fp8_bs2", "d256_fp8_bs4", "d256_fp8_bs8", "d256_bf16_bs8")
ALL_NAMES = CONFIG_NAMES + EXTRA_NAMES


def config_lengths(name: str):
    """(context_lens, query_lens, Hq, Hkv, D, kv_dtype, seed) of a workload."""
    if name == "tiny":
        return [37, 100], [1, 6], 4, 1, 64, KV_BF16, 0
    if name == "mtp5_bf16":
        g = torch.Generator().manual_seed(2)
        ctx = torch.randint(4096, 32768 + 1, (8,), generator=g).tolist()
        return ctx, [6] * 8, 32, 4, 128, KV_BF16, 2
    if name == "mtp5_fp8":
        return [131072] * 4, [6] * 4, 32, 4, 128, KV_FP8, 3
    if name == "mixed_fp8":
        g = torch.Generator().manual_seed(4)
        ql = torch.randint(1, 9, (64,), generator=g)
        z = torch.randn((64,), generator=g, dtype=torch.float64)
        raw = torch.round(torch.exp(math.log(8192.0) + 1.0 * z)).to(torch.int64)
        ctx = torch.clamp(torch.maximum(raw, ql), max=131072)
        return ctx.tolist(), ql.tolist(), 16, 2, 128, KV_FP8, 4
    if name == "ctx1mi_bf16":
        return [1 << 20], [6], 8, 1, 128, KV_BF16, 5
    if name in EXTRA_NAMES:
        bs = int(name.rsplit("bs", 1)[1])
        return [150000] * bs, [6] * bs, 8, 1, 256, (KV_BF16 if "bf16" in name else KV_FP8), 6
    raise KeyError(name)


def make_config(name: str, poison: bool = True, **kw) -> Problem:
    ctx, ql, hq, hkv, d, kvd, seed = config_lengths(name)
    if name == "tiny":
        kw.setdefault("pool_pages", 32)
    return make_problem(ctx, ql, hq, hkv, d, kv_dtype=kvd, seed=seed, poison=poison, name=name, **kw)


def shard_sequences(num_seqs: int, world_size: int, rank: int) -> np.ndarray:
    """Sequences of a batch that rank ``rank`` of ``world_size`` processes:
    a contiguous, balanced block (the path needs no exchange between ranks)."""
    base, rem = divmod(num_seqs, world_size)
    start = rank * base + min(rank, rem)
    count = base + (1 if rank < rem else 0)
    return np.arange(start, start + count, dtype=np.int64)
