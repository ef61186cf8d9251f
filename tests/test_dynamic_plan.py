"""Dynamic (capacity) plans: lengths read on the device at every run, padded
sequences (query length 0) writing nothing, and one captured CUDA graph
replayed over different batches."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_speculative_gb300 import _build, pa_verify as pv, synth
from paged_kv_speculative_gb300.device_inputs import to_device

TOL = {synth.KV_BF16: 1e-2, synth.KV_FP8: 2e-2}


@pytest.fixture(scope="module", autouse=True)
def built():
    _build.build()


def test_capacity_figures():
    p = pv.plan_dynamic(32, 4, 128, pv.KV_BF16, pv.OUT_F32, 4096, 2048, capacity=8, max_context_len=32768,
                        max_query_len=6, sm_count=152)
    i = p.info
    assert i.dynamic == 1 and i.needs_combine == 1
    assert i.rows_max == 6 * 8 and i.num_tokens == 8 * 6
    assert i.num_units >= 152  # the split grid covers one wave at least
    assert p.workspace_bytes >= 256 + i.num_units * 48 * 129 * 4


@pytest.mark.parametrize("kw,status", [
    (dict(capacity=0), pv.ERR_INVALID),
    (dict(max_query_len=9), pv.ERR_INVALID),
    (dict(max_context_len=3, max_query_len=6), pv.ERR_INVALID),
    (dict(max_context_len=1 << 20), pv.ERR_INVALID),  # more pages than the block-table stride
    (dict(capacity=1025), pv.ERR_UNSUPPORTED),
])
def test_dynamic_plan_refusals(kw, status):
    args = dict(capacity=8, max_context_len=4096, max_query_len=6)
    args.update(kw)
    with pytest.raises(pv.PaVerifyError) as e:
        pv.plan_dynamic(32, 4, 128, pv.KV_BF16, pv.OUT_F32, 4096, 256, sm_count=152, **args)
    assert e.value.status == status


def _scenario(base, ctx, ql, seed):
    """The pool and block table of `base` with new lengths and new query rows."""
    g = torch.Generator().manual_seed(seed)
    T = int(sum(ql))
    q = torch.randn((T, base.num_q_heads, base.head_dim), generator=g).to(torch.bfloat16)
    q = q.view(torch.int16).numpy().view(np.uint16)
    return synth.Problem(**{**base.__dict__, "q": q, "context_lens": np.array(ctx, dtype=np.int32),
                            "query_lens": np.array(ql, dtype=np.int32)})


SCENARIOS = [
    ([3000, 1200, 700, 4000], [6, 6, 3, 1]),
    ([4000, 5, 4000, 900], [8, 0, 2, 6]),       # a padded slot
    ([100, 0, 0, 2500], [6, 0, 0, 4]),          # two padded slots
    ([4000, 4000, 4000, 4000], [1, 1, 1, 1]),   # draft-step shape
]


@pytest.mark.gpu
@pytest.mark.parametrize("kvd", [synth.KV_BF16, synth.KV_FP8])
@pytest.mark.parametrize("kernel", [pv.KERNEL_AUTO, pv.KERNEL_WARP_MMA])
def test_dynamic_runs_match_oracle(kvd, kernel):
    base = synth.make_problem([4000] * 4, [8] * 4, 16, 2, 128, kv_dtype=kvd, seed=61)
    dev = to_device(base)
    cap_rows = 4 * 8
    plan = pv.plan_dynamic(16, 2, 128, kvd, pv.OUT_F32, base.num_pages, base.block_table.shape[1], capacity=4,
                           max_context_len=4000, max_query_len=8, kernel=kernel)
    ws = torch.zeros(plan.workspace_bytes, dtype=torch.uint8, device="cuda")
    q_buf = torch.zeros((cap_rows, 16, 128), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros((cap_rows, 16, 128), dtype=torch.float32, device="cuda")
    for k, (ctx, ql) in enumerate(SCENARIOS):
        prob = _scenario(base, ctx, ql, seed=100 + k)
        T = int(sum(ql))
        q_buf[:T].copy_(torch.from_numpy(prob.q.view(np.int16)).view(torch.bfloat16))
        out.fill_(7.0)
        ctx_d = torch.tensor(ctx, dtype=torch.int32, device="cuda")
        ql_d = torch.tensor(ql, dtype=torch.int32, device="cuda")
        pv.run(plan, q_buf, dev.k_cache, dev.v_cache, dev.k_scale, dev.v_scale, dev.block_table, ctx_d, ql_d,
               base.softmax_scale, out, ws)
        torch.cuda.synchronize()
        assert pv.device_errors(ws) == 0
        ref = oracle.verify_attention(prob)
        got = out[:T].cpu().numpy().astype(np.float64)
        assert np.isfinite(got).all()
        assert float(np.abs(got - ref).max()) <= TOL[kvd], (ctx, ql)
        assert bool((out[T:] == 7.0).all())  # rows past the batch are untouched


@pytest.mark.gpu
def test_dynamic_fp8_head_dim_256_matches_oracle():
    """A capacity plan at the head-256 FP8 shape (GQA 8 over one KV head), over the padded scenarios."""
    base = synth.make_problem([4000] * 4, [8] * 4, 8, 1, 256, kv_dtype=synth.KV_FP8, seed=62)
    dev = to_device(base)
    cap_rows = 4 * 8
    plan = pv.plan_dynamic(8, 1, 256, synth.KV_FP8, pv.OUT_F32, base.num_pages, base.block_table.shape[1], capacity=4,
                           max_context_len=4000, max_query_len=8)
    assert plan.info.kernel == pv.KERNEL_TCGEN05
    ws = torch.zeros(plan.workspace_bytes, dtype=torch.uint8, device="cuda")
    q_buf = torch.zeros((cap_rows, 8, 256), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros((cap_rows, 8, 256), dtype=torch.float32, device="cuda")
    for k, (ctx, ql) in enumerate(SCENARIOS[:3]):
        prob = _scenario(base, ctx, ql, seed=200 + k)
        T = int(sum(ql))
        q_buf[:T].copy_(torch.from_numpy(prob.q.view(np.int16)).view(torch.bfloat16))
        out.fill_(7.0)
        ctx_d = torch.tensor(ctx, dtype=torch.int32, device="cuda")
        ql_d = torch.tensor(ql, dtype=torch.int32, device="cuda")
        pv.run(plan, q_buf, dev.k_cache, dev.v_cache, dev.k_scale, dev.v_scale, dev.block_table, ctx_d, ql_d,
               base.softmax_scale, out, ws)
        torch.cuda.synchronize()
        assert pv.device_errors(ws) == 0
        ref = oracle.verify_attention(prob)
        got = out[:T].cpu().numpy().astype(np.float64)
        assert np.isfinite(got).all()
        assert float(np.abs(got - ref).max()) <= TOL[synth.KV_FP8], (ctx, ql)
        assert bool((out[T:] == 7.0).all())


@pytest.mark.gpu
@pytest.mark.parametrize("kvd", [synth.KV_BF16, synth.KV_FP8])
def test_one_captured_graph_serves_every_batch(kvd):
    base = synth.make_problem([4000] * 4, [8] * 4, 16, 2, 128, kv_dtype=kvd, seed=62)
    dev = to_device(base)
    cap_rows = 4 * 8
    plan = pv.plan_dynamic(16, 2, 128, kvd, pv.OUT_F32, base.num_pages, base.block_table.shape[1], capacity=4,
                           max_context_len=4000, max_query_len=8)
    ws = torch.zeros(plan.workspace_bytes, dtype=torch.uint8, device="cuda")
    q_buf = torch.zeros((cap_rows, 16, 128), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros((cap_rows, 16, 128), dtype=torch.float32, device="cuda")
    ctx_d = torch.tensor(SCENARIOS[0][0], dtype=torch.int32, device="cuda")
    ql_d = torch.tensor(SCENARIOS[0][1], dtype=torch.int32, device="cuda")
    args = (q_buf, dev.k_cache, dev.v_cache, dev.k_scale, dev.v_scale, dev.block_table, ctx_d, ql_d,
            base.softmax_scale, out, ws)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        pv.run(plan, *args)  # warm-up outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        pv.run(plan, *args)
    for k, (ctx, ql) in enumerate(SCENARIOS[::-1]):
        prob = _scenario(base, ctx, ql, seed=200 + k)
        T = int(sum(ql))
        q_buf[:T].copy_(torch.from_numpy(prob.q.view(np.int16)).view(torch.bfloat16))
        ctx_d.copy_(torch.tensor(ctx, dtype=torch.int32))
        ql_d.copy_(torch.tensor(ql, dtype=torch.int32))
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        ref = oracle.verify_attention(prob)
        got = out[:T].cpu().numpy().astype(np.float64)
        assert np.isfinite(got).all()
        assert float(np.abs(got - ref).max()) <= TOL[kvd], (ctx, ql)
    assert pv.device_errors(ws) == 0


@pytest.mark.gpu
def test_out_of_capacity_lengths_are_flagged_and_padded():
    base = synth.make_problem([2000] * 2, [6] * 2, 8, 1, 128, seed=63)
    dev = to_device(base)
    plan = pv.plan_dynamic(8, 1, 128, pv.KV_BF16, pv.OUT_F32, base.num_pages, base.block_table.shape[1], capacity=2,
                           max_context_len=2000, max_query_len=6)
    ws = torch.zeros(plan.workspace_bytes, dtype=torch.uint8, device="cuda")
    q_buf = torch.from_numpy(base.q.view(np.int16)).cuda().view(torch.bfloat16)
    out = torch.full((12, 8, 128), 7.0, dtype=torch.float32, device="cuda")
    ctx_d = torch.tensor([2000, 2000], dtype=torch.int32, device="cuda")
    ql_d = torch.tensor([6, 9], dtype=torch.int32, device="cuda")  # 9 > max_query_len
    pv.run(plan, q_buf, dev.k_cache, dev.v_cache, None, None, dev.block_table, ctx_d, ql_d, base.softmax_scale,
           out, ws)
    torch.cuda.synchronize()
    assert pv.device_errors(ws) & pv.DEVERR_LENGTHS
    prob = _scenario(base, [2000, 2000], [6, 0], seed=0)
    prob = synth.Problem(**{**prob.__dict__, "q": base.q[:6].copy()})
    ref = oracle.verify_attention(prob)
    assert float(np.abs(out[:6].cpu().numpy() - ref).max()) <= 1e-2
    assert bool((out[6:] == 7.0).all())


@pytest.mark.gpu
@pytest.mark.parametrize("kvd,d", [(synth.KV_BF16, 128), (synth.KV_FP8, 128), (synth.KV_FP8, 256)],
                         ids=["bf16", "fp8", "fp8_d256"])
def test_dynamic_row_halves_match_oracle(kvd, d):
    """Capacity plans of up to 128 rows (group 16 x query 8) on the tcgen05 kernel: the device planner makes a
    pair of more than 64 rows two virtual pairs, and the combine finds a row's half without a host table."""
    base = synth.make_problem([4000] * 4, [8] * 4, 16, 1, d, kv_dtype=kvd, seed=65)
    dev = to_device(base)
    cap_rows = 4 * 8
    plan = pv.plan_dynamic(16, 1, d, kvd, pv.OUT_F32, base.num_pages, base.block_table.shape[1], capacity=4,
                           max_context_len=4000, max_query_len=8)
    assert plan.info.kernel == pv.KERNEL_TCGEN05 and plan.info.rows_max == 128
    ws = torch.zeros(plan.workspace_bytes, dtype=torch.uint8, device="cuda")
    q_buf = torch.zeros((cap_rows, 16, d), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros((cap_rows, 16, d), dtype=torch.float32, device="cuda")
    for k, (ctx, ql) in enumerate(SCENARIOS):
        prob = _scenario(base, ctx, ql, seed=200 + k)
        T = int(sum(ql))
        q_buf[:T].copy_(torch.from_numpy(prob.q.view(np.int16)).view(torch.bfloat16))
        out.fill_(7.0)
        ctx_d = torch.tensor(ctx, dtype=torch.int32, device="cuda")
        ql_d = torch.tensor(ql, dtype=torch.int32, device="cuda")
        pv.run(plan, q_buf, dev.k_cache, dev.v_cache, dev.k_scale, dev.v_scale, dev.block_table, ctx_d, ql_d,
               base.softmax_scale, out, ws)
        torch.cuda.synchronize()
        assert pv.device_errors(ws) == 0
        ref = oracle.verify_attention(prob)
        got = out[:T].cpu().numpy().astype(np.float64)
        assert np.isfinite(got).all()
        assert float(np.abs(got - ref).max()) <= TOL[kvd], (ctx, ql)
        assert bool((out[T:] == 7.0).all())
