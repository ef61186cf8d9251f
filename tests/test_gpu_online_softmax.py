"""The online softmax under scores that rise inside a segment, and the inputs
that stress the FP8 arithmetic, against the fp64 oracle through the C ABI.

With q, K, V ~ N(0, 1) a later K/V tile never beats the first tile's
row maximum by 2^8 (the tensor-core kernel's lazy-reference threshold), so the
kernel's in-segment rescale of the output accumulator in tensor memory would
never run. Here the K rows grow along the context (2^(a t / L)) and the q rows
have norms spread over several octaves, so the row maxima keep rising and
rows rise at different tiles. Workspace word 1 counts the rescales: each
tensor-core test asserts it is non-zero, so the branch provably ran.

The FP8 cases also spread the per-token V scales over three decades, zero
whole K/V rows (amax = 0, both scales 1) and shrink some V rows to 2^-104
(scales far below the kernel's 2^-100 floor of s_v).

Tolerances: max |GPU - oracle| 1e-2 for bf16 KV and 2e-2 for FP8 KV on fp32
output, the bar of the verify-attention workloads.
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


def run(prob, split=0, kernel=pv.KERNEL_AUTO):
    dev = to_device(prob)
    va = pv.VerifyAttention(prob.num_q_heads, prob.num_kv_heads, prob.head_dim, prob.kv_dtype, prob.num_pages,
                            prob.block_table.shape[1], prob.context_lens.tolist(), prob.query_lens.tolist(),
                            out_dtype=pv.OUT_F32, split_override=split, kernel=kernel)
    out = va(*dev.args(), prob.softmax_scale)
    torch.cuda.synchronize()
    assert va.device_errors() == 0
    return out.cpu().numpy().astype(np.float64), va


def max_err(a, b):
    d = np.abs(a - b)
    assert np.isfinite(d).all(), "non-finite output"
    return float(d.max())


# (kv, head_dim, Hq, Hkv, query lengths): the row counts pick the kernel instance
# (q_len x group padded to 16 / 48 / 64; up to 48 rows the reference maxima sit in
# registers, at 64 in shared memory; head_dim 256 at 48 rows runs three warpgroups)
SHAPES = [
    ("bf16_r16", synth.KV_BF16, 128, 16, 2, [2, 1]),
    ("bf16_r48", synth.KV_BF16, 128, 16, 2, [6, 4]),
    ("bf16_r64", synth.KV_BF16, 128, 16, 2, [8, 7]),
    ("bf16_d64_r48", synth.KV_BF16, 64, 16, 2, [6, 4]),
    ("bf16_d64_r64", synth.KV_BF16, 64, 16, 2, [8, 5]),
    ("fp8_r32", synth.KV_FP8, 128, 16, 2, [4, 3]),
    ("fp8_r48", synth.KV_FP8, 128, 16, 2, [6, 4]),
    ("fp8_r64", synth.KV_FP8, 128, 16, 2, [8, 7]),
    ("fp8_d256_r16", synth.KV_FP8, 256, 8, 1, [2, 1]),
    ("fp8_d256_r48", synth.KV_FP8, 256, 8, 1, [6, 5]),
    ("fp8_d256_r64", synth.KV_FP8, 256, 16, 2, [8, 7]),
    ("bf16_d256_r48", synth.KV_BF16, 256, 8, 1, [6, 5]),
    ("bf16_d256_r64", synth.KV_BF16, 256, 16, 2, [8, 7]),
]


def ramp_problem(kv, d, hq, hkv, ql, seed, ctx=(3000, 1700), ramp=4.0, **kw):
    return synth.make_problem(list(ctx), ql, hq, hkv, d, kv_dtype=kv, seed=seed, q_row_log2=(-2.0, 2.0),
                              k_ramp_log2=ramp, **kw)


@pytest.mark.parametrize("split", [0, 1, 5], ids=["planner", "one_segment", "five_way"])
@pytest.mark.parametrize("name,kv,d,hq,hkv,ql", SHAPES, ids=[s[0] for s in SHAPES])
def test_rising_scores_rescale_inside_segments(name, kv, d, hq, hkv, ql, split):
    # The planner spreads the pairs' tiles over every SM: contexts of a few thousand tokens would
    # leave one tile per CTA (no second tile in any segment), so its case takes 65 k tokens.
    if split == 0:
        prob = ramp_problem(kv, d, hq, hkv, ql, seed=51, ctx=(40000, 25000), ramp=6.0)
    else:
        prob = ramp_problem(kv, d, hq, hkv, ql, seed=51)
    ref = oracle.verify_attention(prob)
    got, va = run(prob, split=split, kernel=pv.KERNEL_TCGEN05)
    assert va.info["kernel"] == pv.KERNEL_TCGEN05
    assert pv.rescale_count(va.workspace) > 0, "the in-segment rescale did not run"
    assert max_err(got, ref) <= TOL[kv], name


@pytest.mark.parametrize("kv", [synth.KV_BF16, synth.KV_FP8], ids=["bf16", "fp8"])
def test_rising_scores_on_the_warp_mma_kernel(kv):
    prob = ramp_problem(kv, 128, 16, 2, [8, 7], seed=52)
    ref = oracle.verify_attention(prob)
    got, va = run(prob, split=3, kernel=pv.KERNEL_WARP_MMA)
    assert va.info["kernel"] == pv.KERNEL_WARP_MMA
    assert max_err(got, ref) <= TOL[kv]


def test_plain_inputs_do_not_rescale():
    # N(0, 1) inputs stay under the 2^8 threshold after the first tile: the counter is a real signal
    prob = synth.make_problem([3000, 1700], [6, 4], 16, 2, 128, seed=53)
    _, va = run(prob, split=1, kernel=pv.KERNEL_TCGEN05)
    assert pv.rescale_count(va.workspace) == 0


@pytest.mark.parametrize("d,hq,hkv,ql", [(128, 16, 2, [6, 4, 8]), (256, 8, 1, [6, 5, 2])], ids=["d128", "d256"])
@pytest.mark.parametrize("split", [0, 4])
def test_fp8_scales_over_decades_zero_and_tiny_rows(d, hq, hkv, ql, split):
    prob = synth.make_problem([2500, 1300, 700], ql, hq, hkv, d, kv_dtype=synth.KV_FP8, seed=54,
                              q_row_log2=(-6.0, 6.0), k_ramp_log2=2.0, v_tok_log2=(-10.0, 0.0), zero_frac=0.03,
                              tiny_v_frac=0.03)
    ks, vs = prob.k_scale[np.isfinite(prob.k_scale)], prob.v_scale[np.isfinite(prob.v_scale)]
    assert (ks == 1.0).any() and (vs == 1.0).any()   # amax = 0 rows
    assert (vs < 2.0 ** -100).any()                   # below the s_v floor
    assert vs.max() / vs[vs > 2.0 ** -90].min() > 500  # spread over decades
    ref = oracle.verify_attention(prob)
    for kernel in (pv.KERNEL_TCGEN05, pv.KERNEL_WARP_MMA):
        if kernel == pv.KERNEL_WARP_MMA and d == 256:
            continue
        got, _ = run(prob, split=split, kernel=kernel)
        assert max_err(got, ref) <= TOL[synth.KV_FP8], kernel


@pytest.mark.parametrize("kv", [synth.KV_BF16, synth.KV_FP8], ids=["bf16", "fp8"])
def test_wide_q_row_range_and_zero_rows(kv):
    prob = synth.make_problem([1800, 900], [6, 3], 16, 2, 128, kv_dtype=kv, seed=55, q_row_log2=(-8.0, 8.0),
                              zero_frac=0.05)
    ref = oracle.verify_attention(prob)
    for kernel in (pv.KERNEL_TCGEN05, pv.KERNEL_WARP_MMA):
        got, _ = run(prob, split=2, kernel=kernel)
        assert max_err(got, ref) <= TOL[kv], kernel


# ------------------------------------------------------------ bounded waits
@pytest.mark.parametrize("kv,d,hq,hkv", [(synth.KV_BF16, 128, 16, 2), (synth.KV_FP8, 128, 16, 2),
                                         (synth.KV_FP8, 256, 8, 1)], ids=["bf16", "fp8", "fp8_d256"])
def test_a_wait_that_runs_out_sets_the_timeout_bit(kv, d, hq, hkv):
    """CTA 0's MMA issuer waits on a barrier that nothing completes; its bounded
    wait (20 ms here) runs out, the CTA's other roles run out theirs, drain and
    return, and the error word says so. The next run without the hook is clean
    and matches the oracle."""
    prob = synth.make_problem([3000, 1200], [6, 6], hq, hkv, d, kv_dtype=kv, seed=56)
    ref = oracle.verify_attention(prob)
    dev = to_device(prob)
    va = pv.VerifyAttention(hq, hkv, d, kv, prob.num_pages, prob.block_table.shape[1], prob.context_lens.tolist(),
                            prob.query_lens.tolist(), split_override=3, kernel=pv.KERNEL_TCGEN05)
    pv.debug_stall(va.plan, 0, 20000)
    va(*dev.args(), prob.softmax_scale)
    torch.cuda.synchronize()
    assert va.device_errors(clear=True) & pv.DEVERR_TIMEOUT
    pv.debug_stall(va.plan, -1, 0)
    out = va(*dev.args(), prob.softmax_scale)
    torch.cuda.synchronize()
    assert va.device_errors() == 0
    assert max_err(out.cpu().numpy().astype(np.float64), ref) <= TOL[kv]
