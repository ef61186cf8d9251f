"""Batches of more than 64 sequences (up to 1024, the batch the pages' reducer
is sized for: MTP-5 routing page, Motivation), through the C ABI, against the
fp64 oracle on every row.

Above 64 sequences a plan's work table no longer fits the kernel parameters:
each run builds it on the device from the device lengths (the planner of the
capacity plans). Capacity plans of 128 sequences (the pages' largest CUDA-graph
capture width: DeepSeek-V4.1 page, launch flags) are captured once and
replayed over padded batches.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_speculative_gb300 import _build, pa_verify as pv, synth
from paged_kv_speculative_gb300.device_inputs import to_device

pytestmark = pytest.mark.gpu

TOL = {synth.KV_BF16: 1e-2, synth.KV_FP8: 2e-2}


@pytest.fixture(scope="module", autouse=True)
def built():
    _build.build()
    yield


def lengths(B, seed, lo=6, hi=3000):
    rng = np.random.default_rng(seed)
    ql = rng.integers(1, 9, B)
    ctx = np.maximum(rng.integers(lo, hi + 1, B), ql)
    return ctx.tolist(), ql.tolist()


def max_err(a, b):
    d = np.abs(a.astype(np.float64) - b)
    assert np.isfinite(d).all(), "non-finite output"
    return float(d.max())


@pytest.mark.parametrize("B", [65, 128, 256])
@pytest.mark.parametrize("kv,d,hq,hkv,kernel", [
    (synth.KV_BF16, 128, 16, 2, pv.KERNEL_AUTO),
    (synth.KV_FP8, 128, 16, 2, pv.KERNEL_AUTO),
    (synth.KV_FP8, 256, 8, 1, pv.KERNEL_AUTO),
    (synth.KV_BF16, 128, 16, 1, pv.KERNEL_AUTO),       # up to 128 rows: row halves on the tcgen05 kernel
    (synth.KV_FP8, 128, 16, 1, pv.KERNEL_AUTO),
    (synth.KV_BF16, 128, 16, 1, pv.KERNEL_WARP_MMA),   # the same on the warp-MMA kernel
    (synth.KV_BF16, 64, 8, 2, pv.KERNEL_AUTO),
], ids=["bf16", "fp8", "fp8_d256", "bf16_rows128", "fp8_rows128", "bf16_rows128_mma", "bf16_d64"])
def test_large_batch_every_row(B, kv, d, hq, hkv, kernel):
    ctx, ql = lengths(B, seed=B + d + hkv)
    prob = synth.make_problem(ctx, ql, hq, hkv, d, kv_dtype=kv, seed=70 + B)
    dev = to_device(prob)
    va = pv.VerifyAttention(hq, hkv, d, kv, prob.num_pages, prob.block_table.shape[1], ctx, ql, kernel=kernel)
    assert va.info["device_table"] == 1
    assert va.info["kernel"] == (pv.KERNEL_WARP_MMA if kernel == pv.KERNEL_WARP_MMA else pv.KERNEL_TCGEN05)
    out = va(*dev.args(), prob.softmax_scale)
    torch.cuda.synchronize()
    assert va.device_errors() == 0
    assert max_err(out.cpu().numpy(), oracle.verify_attention(prob)) <= TOL[kv]


def test_batch_of_1024():
    ctx, ql = lengths(1024, seed=5, hi=900)
    prob = synth.make_problem(ctx, ql, 8, 1, 128, seed=77)
    dev = to_device(prob)
    va = pv.VerifyAttention(8, 1, 128, synth.KV_BF16, prob.num_pages, prob.block_table.shape[1], ctx, ql)
    out = va(*dev.args(), prob.softmax_scale)
    torch.cuda.synchronize()
    assert va.device_errors() == 0
    assert max_err(out.cpu().numpy(), oracle.verify_attention(prob)) <= TOL[synth.KV_BF16]


def _scenario(base, ctx, ql, seed):
    g = torch.Generator().manual_seed(seed)
    T = int(sum(ql))
    q = torch.randn((T, base.num_q_heads, base.head_dim), generator=g).to(torch.bfloat16)
    q = q.view(torch.int16).numpy().view(np.uint16)
    return synth.Problem(**{**base.__dict__, "q": q, "context_lens": np.array(ctx, dtype=np.int32),
                            "query_lens": np.array(ql, dtype=np.int32)})


@pytest.mark.parametrize("kvd", [synth.KV_BF16, synth.KV_FP8], ids=["bf16", "fp8"])
def test_capture_width_128_graph_replays_padded_batches(kvd):
    cap, max_len, max_q = 128, 2500, 8
    base = synth.make_problem([max_len] * cap, [max_q] * cap, 16, 2, 128, kv_dtype=kvd, seed=64)
    dev = to_device(base)
    plan = pv.plan_dynamic(16, 2, 128, kvd, pv.OUT_F32, base.num_pages, base.block_table.shape[1], capacity=cap,
                           max_context_len=max_len, max_query_len=max_q)
    assert plan.info.device_table == 1 and plan.info.dynamic == 1
    ws = torch.zeros(plan.workspace_bytes, dtype=torch.uint8, device="cuda")
    q_buf = torch.zeros((cap * max_q, 16, 128), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros((cap * max_q, 16, 128), dtype=torch.float32, device="cuda")
    rng = np.random.default_rng(9)
    scenarios = []
    for live in (128, 100, 37, 1):  # full width, then fewer live sequences (the rest padded, query length 0)
        ql = np.zeros(cap, dtype=np.int64)
        slots = rng.choice(cap, live, replace=False)
        ql[slots] = rng.integers(1, max_q + 1, live)
        ctx = np.where(ql > 0, np.maximum(rng.integers(1, max_len + 1, cap), ql), rng.integers(0, max_len + 1, cap))
        scenarios.append((ctx.tolist(), ql.tolist()))
    ctx_d = torch.tensor(scenarios[0][0], dtype=torch.int32, device="cuda")
    ql_d = torch.tensor(scenarios[0][1], dtype=torch.int32, device="cuda")
    args = (q_buf, dev.k_cache, dev.v_cache, dev.k_scale, dev.v_scale, dev.block_table, ctx_d, ql_d,
            base.softmax_scale, out, ws)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        pv.run(plan, *args)  # warm-up outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        pv.run(plan, *args)
    for k, (ctx, ql) in enumerate(scenarios):
        prob = _scenario(base, ctx, ql, seed=300 + k)
        T = int(sum(ql))
        q_buf[:T].copy_(torch.from_numpy(prob.q.view(np.int16)).view(torch.bfloat16))
        ctx_d.copy_(torch.tensor(ctx, dtype=torch.int32))
        ql_d.copy_(torch.tensor(ql, dtype=torch.int32))
        out.fill_(7.0)
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        live = [b for b in range(cap) if ql[b] > 0]
        sub = synth.Problem(**{**prob.__dict__, "context_lens": np.array([ctx[b] for b in live], dtype=np.int32),
                               "query_lens": np.array([ql[b] for b in live], dtype=np.int32),
                               "block_table": prob.block_table[live]})
        ref = oracle.verify_attention(sub)
        got = out[:T].cpu().numpy().astype(np.float64)
        assert max_err(got, ref) <= TOL[kvd], k
        assert bool((out[T:] == 7.0).all())  # rows past the batch are untouched
    assert pv.device_errors(ws) == 0
