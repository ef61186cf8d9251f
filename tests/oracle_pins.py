"""Independent checks the oracle is pinned to (CPU only).

Each pin returns ``(ok, detail)`` so the same battery can be run against the
normal oracle build and against builds with a planted mistake. None of them
re-types the oracle's loop: they use a dense masked brute force over gathered
contiguous tensors with torch's own bf16/E4M3 decoders, torch's SDPA for the
decode special case, closed forms, and invariants of the definition.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from paged_kv_speculative_gb300 import synth


def _dec_cache(prob, which: str) -> torch.Tensor:
    cache = prob.k_cache if which == "k" else prob.v_cache
    if prob.kv_dtype == synth.KV_BF16:
        return torch.from_numpy(cache.view(np.int16).copy()).view(torch.bfloat16).double()
    scale = prob.k_scale if which == "k" else prob.v_scale
    x = torch.from_numpy(cache.copy()).view(torch.float8_e4m3fn).double()
    return x * torch.from_numpy(scale.astype(np.float64)).unsqueeze(-1)


def brute_force(prob) -> np.ndarray:
    """Dense fp64 masked softmax attention per sequence and q head."""
    q = torch.from_numpy(prob.q.view(np.int16).copy()).view(torch.bfloat16).double()
    K = _dec_cache(prob, "k")
    V = _dec_cache(prob, "v")
    G = prob.group
    out = torch.zeros_like(q)
    off = prob.q_offsets()
    for b in range(prob.num_seqs):
        L = int(prob.context_lens[b])
        ql = int(prob.query_lens[b])
        npg = (L + 15) // 16
        pages = torch.from_numpy(prob.block_table[b, :npg].astype(np.int64))
        Kc = K[pages].permute(1, 0, 2, 3).reshape(prob.num_kv_heads, npg * 16, -1)[:, :L]
        Vc = V[pages].permute(1, 0, 2, 3).reshape(prob.num_kv_heads, npg * 16, -1)[:, :L]
        i = torch.arange(ql).unsqueeze(1)
        t = torch.arange(L).unsqueeze(0)
        visible = t <= (L - ql + i)
        Qb = q[off[b]:off[b + 1]]
        for h in range(prob.num_q_heads):
            g = h // G
            S = (Qb[:, h] @ Kc[g].T) * prob.softmax_scale
            S = S.masked_fill(~visible, float("-inf"))
            P = torch.softmax(S, dim=-1)
            out[off[b]:off[b + 1], h] = P @ Vc[g]
    return out.numpy()


def pin_brute_force(prob, mutant=0, tol=1e-11):
    got = oracle.verify_attention(prob, mutant=mutant)
    ref = brute_force(prob)
    err = float(np.nanmax(np.abs(got - ref))) if np.isfinite(got).all() else float("inf")
    return err <= tol, f"max|oracle-brute|={err:.3e}"


def pin_sdpa_decode(prob, mutant=0, tol=1e-11):
    """query_len 1 everywhere: ordinary decode over the whole context."""
    assert (prob.query_lens == 1).all()
    got = oracle.verify_attention(prob, mutant=mutant)
    q = torch.from_numpy(prob.q.view(np.int16).copy()).view(torch.bfloat16).double()
    K = _dec_cache(prob, "k")
    V = _dec_cache(prob, "v")
    G = prob.group
    err = 0.0
    for b in range(prob.num_seqs):
        L = int(prob.context_lens[b])
        npg = (L + 15) // 16
        pages = torch.from_numpy(prob.block_table[b, :npg].astype(np.int64))
        Kc = K[pages].permute(1, 0, 2, 3).reshape(prob.num_kv_heads, npg * 16, -1)[:, :L]
        Vc = V[pages].permute(1, 0, 2, 3).reshape(prob.num_kv_heads, npg * 16, -1)[:, :L]
        Kh = Kc.repeat_interleave(G, dim=0).unsqueeze(0)  # [1, Hq, L, D]
        Vh = Vc.repeat_interleave(G, dim=0).unsqueeze(0)
        qb = q[b].unsqueeze(0).unsqueeze(2)  # [1, Hq, 1, D]
        ref = torch.nn.functional.scaled_dot_product_attention(qb, Kh, Vh, scale=prob.softmax_scale)
        ref = ref[0, :, 0].numpy()
        d = np.abs(got[b] - ref)
        err = max(err, float(np.max(d)) if np.isfinite(d).all() else float("inf"))
    return err <= tol, f"max|oracle-sdpa|={err:.3e}"


def pin_causal_prefix(prob, mutant=0):
    """Row i of a verify call equals a query-length-1 call whose context ends
    at the last key row i may see (context L - q + i + 1)."""
    got = oracle.verify_attention(prob, mutant=mutant)
    off = prob.q_offsets()
    worst = 0.0
    for b in range(prob.num_seqs):
        L = int(prob.context_lens[b])
        ql = int(prob.query_lens[b])
        for i in range(ql):
            one = synth.Problem(name="prefix", num_q_heads=prob.num_q_heads, num_kv_heads=prob.num_kv_heads,
                                head_dim=prob.head_dim, kv_dtype=prob.kv_dtype,
                                q=prob.q[off[b] + i:off[b] + i + 1].copy(), k_cache=prob.k_cache,
                                v_cache=prob.v_cache, k_scale=prob.k_scale, v_scale=prob.v_scale,
                                block_table=prob.block_table[b:b + 1].copy(),
                                context_lens=np.array([L - ql + i + 1], dtype=np.int32),
                                query_lens=np.array([1], dtype=np.int32),
                                softmax_scale=prob.softmax_scale, seed=prob.seed)
            ref = oracle.verify_attention(one, mutant=mutant)[0]
            d = np.abs(got[off[b] + i] - ref)
            worst = max(worst, float(np.max(d)) if np.isfinite(d).all() else float("inf"))
    return worst == 0.0, f"max|row - prefix call|={worst:.3e}"


def permute_pool(prob, seed=123):
    """Same problem with the pool pages relabelled by a random permutation."""
    n = prob.num_pages
    perm = np.random.default_rng(seed).permutation(n).astype(np.int32)  # old page p -> new page perm[p]
    inv = np.empty_like(perm)
    inv[perm] = np.arange(n, dtype=np.int32)
    bt = prob.block_table.copy()
    valid = bt >= 0
    bt[valid] = perm[bt[valid]]
    return synth.Problem(name=prob.name + "_perm", num_q_heads=prob.num_q_heads, num_kv_heads=prob.num_kv_heads,
                         head_dim=prob.head_dim, kv_dtype=prob.kv_dtype, q=prob.q,
                         k_cache=prob.k_cache[inv].copy(), v_cache=prob.v_cache[inv].copy(),
                         k_scale=None if prob.k_scale is None else prob.k_scale[inv].copy(),
                         v_scale=None if prob.v_scale is None else prob.v_scale[inv].copy(),
                         block_table=bt, context_lens=prob.context_lens, query_lens=prob.query_lens,
                         softmax_scale=prob.softmax_scale, seed=prob.seed)


def pin_page_permutation(prob, mutant=0):
    a = oracle.verify_attention(prob, mutant=mutant)
    b = oracle.verify_attention(permute_pool(prob), mutant=mutant)
    same = np.array_equal(a, b, equal_nan=False)
    return same, "identical under page relabelling" if same else "differs under page relabelling"


def pin_closed_forms(prob, mutant=0):
    """Constant V -> that constant; equal keys -> mean of the visible V rows;
    one dominant key (logit ~ 800) -> that key's V row."""
    msgs = []
    ok = True
    D = prob.head_dim
    off = prob.q_offsets()
    bf = synth.KV_BF16
    # (1) constant V
    if prob.kv_dtype == bf:
        c = 0.75
        pv = synth.Problem(**{**prob.__dict__, "v_cache": np.full_like(prob.v_cache, 0x3F40)})  # bf16 0.75
        o = oracle.verify_attention(pv, mutant=mutant)
        e = float(np.max(np.abs(o - c))) if np.isfinite(o).all() else float("inf")
        ok &= e < 1e-13
        msgs.append(f"constV err {e:.2e}")
    # (2) equal keys: every key row = 1.0 -> uniform weights
    if prob.kv_dtype == bf:
        pk = synth.Problem(**{**prob.__dict__, "k_cache": np.full_like(prob.k_cache, 0x3F80)})
        o = oracle.verify_attention(pk, mutant=mutant)
        V = _dec_cache(prob, "v").numpy()
        worst = 0.0
        for b in range(prob.num_seqs):
            L = int(prob.context_lens[b])
            ql = int(prob.query_lens[b])
            npg = (L + 15) // 16
            Vc = V[prob.block_table[b, :npg]].transpose(1, 0, 2, 3).reshape(prob.num_kv_heads, npg * 16, D)
            for i in range(ql):
                for h in range(prob.num_q_heads):
                    ref = Vc[h // prob.group, :L - ql + i + 1].mean(axis=0)
                    d = np.abs(o[off[b] + i, h] - ref)
                    worst = max(worst, float(d.max()) if np.isfinite(d).all() else float("inf"))
        ok &= worst < 1e-12
        msgs.append(f"equalK err {worst:.2e}")
    # (3) one dominant key for the first row of sequence 0
    if prob.kv_dtype == bf:
        qv = torch.from_numpy(prob.q[0, 0].view(np.int16).copy()).view(torch.bfloat16).double()
        big = (qv * 100.0).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        kc = np.zeros_like(prob.k_cache)  # all-zero keys -> logit 0
        t_star = 0
        pg = prob.block_table[0, t_star // 16]
        kc[pg, 0, t_star % 16] = big
        pd = synth.Problem(**{**prob.__dict__, "k_cache": kc})
        o = oracle.verify_attention(pd, rows=np.array([[0, 0]]), mutant=mutant)[0]
        vref = _dec_cache(prob, "v").numpy()[pg, 0, t_star % 16]
        d = np.abs(o - vref)
        e = float(d.max()) if np.isfinite(d).all() else float("inf")
        ok &= e < 1e-12
        msgs.append(f"dominant err {e:.2e}")
    return bool(ok), "; ".join(msgs)


def tiny_problems():
    """A small, varied set: the tiny workload, GQA with two KV heads, FP8,
    query lengths 1..8, ragged last pages, contiguous pages."""
    ps = [synth.make_config("tiny")]
    ps.append(synth.make_problem([33, 70, 16], [3, 8, 1], 4, 2, 64, seed=11, name="gqa2"))
    ps.append(synth.make_problem([45, 29], [6, 2], 4, 2, 64, kv_dtype=synth.KV_FP8, seed=12, name="fp8"))
    ps.append(synth.make_problem([17, 64], [4, 5], 2, 1, 128, seed=13, name="d128", contiguous=True))
    return ps


def decode_problem(kv_dtype=synth.KV_BF16):
    return synth.make_problem([23, 50, 8], [1, 1, 1], 4, 2, 64, kv_dtype=kv_dtype, seed=21, name="decode")


def run_battery(mutant=0):
    """All pins; returns a list of (name, ok, detail)."""
    res = []
    for p in tiny_problems():
        ok, det = pin_brute_force(p, mutant)
        res.append((f"brute:{p.name}", ok, det))
    for kvd in (synth.KV_BF16, synth.KV_FP8):
        ok, det = pin_sdpa_decode(decode_problem(kvd), mutant)
        res.append((f"sdpa:{kvd}", ok, det))
    for p in tiny_problems()[:2]:
        ok, det = pin_causal_prefix(p, mutant)
        res.append((f"prefix:{p.name}", ok, det))
        ok, det = pin_page_permutation(p, mutant)
        res.append((f"perm:{p.name}", ok, det))
        ok, det = pin_closed_forms(p, mutant)
        res.append((f"closed:{p.name}", ok, det))
    return res
