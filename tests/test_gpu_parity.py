"""CUDA path against the fp64 oracle, element by element, through the C ABI.

Tolerances (max |GPU - oracle| on fp32 output): 1e-2 for bf16 KV and 2e-2 for
FP8 KV, the bar the verify-attention workloads set. bf16 output adds its own
rounding (2^-9 relative), so those comparisons allow 1e-2 on top.
Full-size workloads are checked on every output row.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_speculative_gb300 import pa_verify as pv, synth
from paged_kv_speculative_gb300.device_inputs import to_device
from tests import oracle_pins

pytestmark = pytest.mark.gpu

TOL = {synth.KV_BF16: 1e-2, synth.KV_FP8: 2e-2}


@pytest.fixture(scope="module", autouse=True)
def built():
    from paged_kv_speculative_gb300 import _build
    _build.build()
    yield


def tc_applies(prob):
    # every head_dim and up to 128 rows (65-128 rows as two row halves)
    return int(prob.query_lens.max()) * prob.group <= 128


def mma_applies(prob):
    return prob.head_dim != 256  # head_dim 256 runs on the tcgen05 kernel only


KERNELS = [pv.KERNEL_WARP_MMA, pv.KERNEL_TCGEN05]
KID = {pv.KERNEL_WARP_MMA: "mma", pv.KERNEL_TCGEN05: "tc"}


def gpu_run(prob, out_dtype=pv.OUT_F32, split_override=0, dev=None, check_errors=True, kernel=pv.KERNEL_AUTO):
    dev = dev or to_device(prob)
    va = pv.VerifyAttention(prob.num_q_heads, prob.num_kv_heads, prob.head_dim, prob.kv_dtype, prob.num_pages,
                            prob.block_table.shape[1], prob.context_lens.tolist(), prob.query_lens.tolist(),
                            out_dtype=out_dtype, split_override=split_override, kernel=kernel)
    out = va(*dev.args(), prob.softmax_scale)
    torch.cuda.synchronize()
    if check_errors:
        assert va.device_errors() == 0
    return out.float().cpu().numpy(), va


def max_err(a, b):
    d = np.abs(a.astype(np.float64) - b)
    assert np.isfinite(d).all(), "non-finite output"
    return float(d.max())


SMALL = [
    ("tiny", lambda: synth.make_config("tiny")),
    ("gqa2_ragged", lambda: synth.make_problem([33, 70, 16, 1], [3, 8, 1, 1], 4, 2, 64, seed=11)),
    ("d128_multi_tile", lambda: synth.make_problem([1000, 333, 2049], [6, 3, 8], 16, 2, 128, seed=31)),
    ("d64_multi_tile", lambda: synth.make_problem([700, 129, 1500], [6, 1, 4], 8, 1, 64, seed=32)),
    ("q_equals_ctx", lambda: synth.make_problem([6, 1, 8, 64], [6, 1, 8, 5], 8, 2, 128, seed=33)),
    ("rows128", lambda: synth.make_problem([500, 77], [8, 5], 16, 1, 128, seed=34)),
    ("fp8_small", lambda: synth.make_problem([45, 29, 300], [6, 2, 8], 8, 1, 128, kv_dtype=synth.KV_FP8, seed=12)),
    ("fp8_multi_tile", lambda: synth.make_problem([1500, 257, 4099], [6, 1, 7], 16, 2, 128,
                                                  kv_dtype=synth.KV_FP8, seed=35)),
    ("fp8_d256_small", lambda: synth.make_problem([45, 29, 300, 6], [6, 2, 8, 6], 8, 1, 256,
                                                  kv_dtype=synth.KV_FP8, seed=13)),
    ("fp8_d256_multi_tile", lambda: synth.make_problem([1500, 257, 4099, 128], [6, 1, 7, 3], 16, 2, 256,
                                                       kv_dtype=synth.KV_FP8, seed=37)),
    ("fp8_d256_rows16", lambda: synth.make_problem([700, 129], [2, 1], 8, 1, 256, kv_dtype=synth.KV_FP8, seed=38)),
    ("bf16_d256_small", lambda: synth.make_problem([45, 29, 300, 6], [6, 2, 8, 6], 8, 1, 256, seed=14)),
    ("bf16_d256_multi_tile", lambda: synth.make_problem([1500, 257, 4099, 128], [6, 1, 7, 3], 16, 2, 256, seed=15)),
]


@pytest.mark.parametrize("name,make", SMALL, ids=[s[0] for s in SMALL])
@pytest.mark.parametrize("split", [0, 1, 3])
@pytest.mark.parametrize("kernel", KERNELS, ids=[KID[k] for k in KERNELS])
def test_small_against_oracle(name, make, split, kernel):
    prob = make()
    if kernel == pv.KERNEL_TCGEN05 and not tc_applies(prob):
        pytest.skip("outside the tcgen05 kernel's envelope")
    if kernel == pv.KERNEL_WARP_MMA and not mma_applies(prob):
        pytest.skip("outside the warp-MMA kernel's envelope")
    ref = oracle.verify_attention(prob)
    got, va = gpu_run(prob, split_override=split, kernel=kernel)
    assert va.info["kernel"] == kernel
    assert max_err(got, ref) <= TOL[prob.kv_dtype], name


# Flat plans: a few tiles per CTA (split_override = ceil(longest pair's tiles / per)) put segment
# boundaries everywhere, one-tile segments and CTAs spanning several sequences included. The lengths
# end on, just after and just before 128-token tile edges.
SEG_CTX = [1, 17, 128, 129, 255, 300, 640, 1000, 5, 2049, 16, 383, 256, 513]
SEG_Q = [1, 6, 8, 2, 3, 6, 7, 1, 4, 6, 5, 8, 2, 7]


@pytest.mark.parametrize("split", [17, 9, 6, 4, 0])
@pytest.mark.parametrize("kv,d", [(synth.KV_BF16, 128), (synth.KV_FP8, 128), (synth.KV_FP8, 256),
                                  (synth.KV_BF16, 256)], ids=["bf16", "fp8", "fp8_d256", "bf16_d256"])
def test_flat_segments_against_oracle(kv, d, split):
    prob = synth.make_problem(SEG_CTX, SEG_Q, 16, 2, d, kv_dtype=kv, seed=36)
    ref = oracle.verify_attention(prob)
    got, va = gpu_run(prob, split_override=split, kernel=pv.KERNEL_TCGEN05)
    assert va.info["flat"] == 1
    assert max_err(got, ref) <= TOL[kv]


BF16_OUT = SMALL[:3] + SMALL[6:7] + SMALL[8:9]


@pytest.mark.parametrize("name,make", BF16_OUT, ids=[s[0] for s in BF16_OUT])
def test_bf16_output(name, make):
    prob = make()
    ref = oracle.verify_attention(prob)
    got, _ = gpu_run(prob, out_dtype=pv.OUT_BF16)
    assert max_err(got, ref) <= TOL[prob.kv_dtype] + 1e-2


@pytest.mark.parametrize("kernel", KERNELS, ids=[KID[k] for k in KERNELS])
def test_split_count_does_not_change_the_result(kernel):
    prob = synth.make_problem([3000, 1200], [6, 6], 16, 2, 128, seed=41)
    outs = [gpu_run(prob, split_override=k, kernel=kernel)[0] for k in (1, 2, 5, 1000)]
    for o in outs[1:]:
        # P is rounded to bf16 against a split-dependent running max: 2^-8 relative per weight
        assert max_err(o, outs[0]) <= 2e-3


def test_fp8_d256_split_count_does_not_change_the_result():
    prob = synth.make_problem([3000, 1200], [6, 6], 8, 1, 256, kv_dtype=synth.KV_FP8, seed=47)
    outs = [gpu_run(prob, split_override=k)[0] for k in (1, 2, 5, 1000)]
    for o in outs[1:]:
        # P's hi/lo E4M3 terms carry about 7 bits against a split-dependent running max
        assert max_err(o, outs[0]) <= 4e-3


@pytest.mark.parametrize("kernel", KERNELS, ids=[KID[k] for k in KERNELS])
def test_repeat_runs_are_bit_identical(kernel):
    prob = synth.make_problem([3000, 1200], [6, 6], 16, 2, 128, seed=42)
    dev = to_device(prob)
    a, va = gpu_run(prob, dev=dev, kernel=kernel)
    b = va(*dev.args(), prob.softmax_scale).cpu().numpy()
    assert np.array_equal(a, b)


def test_page_relabelling_is_bit_identical():
    prob = synth.make_problem([900, 400], [6, 3], 8, 1, 128, seed=43)
    a, _ = gpu_run(prob)
    b, _ = gpu_run(oracle_pins.permute_pool(prob, seed=5))
    assert np.array_equal(a, b)


def test_draft_row_matches_prefix_decode_on_gpu():
    prob = synth.make_problem([777], [6], 8, 1, 128, seed=44)
    full, _ = gpu_run(prob)
    for i in range(6):
        one = synth.Problem(**{**prob.__dict__, "q": prob.q[i:i + 1].copy(),
                               "context_lens": np.array([777 - 6 + i + 1], dtype=np.int32),
                               "query_lens": np.array([1], dtype=np.int32)})
        row, _ = gpu_run(one)
        assert max_err(full[i], row[0].astype(np.float64)) <= 2e-3


def test_empty_batch_is_a_no_op():
    va = pv.VerifyAttention(8, 1, 128, pv.KV_BF16, 4, 4, [], [], out_dtype=pv.OUT_F32)
    z = torch.zeros(16, device="cuda")
    t = torch.zeros(1, dtype=torch.int32, device="cuda")
    q = torch.zeros(1, 8, 128, dtype=torch.bfloat16, device="cuda")
    pv.run(va.plan, q, z, z, None, None, t, t, t, 0.1, z, va.workspace)
    torch.cuda.synchronize()


def test_out_of_range_page_is_flagged_not_faulted():
    prob = synth.make_problem([200], [6], 8, 1, 128, seed=45)
    prob.block_table[0, 3] = prob.num_pages + 1000  # not a pool page
    _, va = gpu_run(prob, check_errors=False)
    assert va.device_errors(clear=True) & pv.DEVERR_PAGE_RANGE
    assert va.device_errors() == 0


def test_device_length_mismatch_is_flagged():
    prob = synth.make_problem([200, 100], [6, 6], 8, 1, 128, seed=46)
    dev = to_device(prob)
    va = pv.VerifyAttention(8, 1, 128, pv.KV_BF16, prob.num_pages, prob.block_table.shape[1], [200, 100], [6, 6])
    dev.context_lens[1] = 99  # differs from the planned 100 (still a valid length)
    va(*dev.args(), prob.softmax_scale)
    torch.cuda.synchronize()
    assert va.device_errors() & pv.DEVERR_LENGTHS


# --------------------------------------------------------------- full-size workloads
_cache = {}


def _workload(name):
    if name not in _cache:
        _cache[name] = synth.make_config(name)
    return _cache[name]


def _workload_dev(name):
    key = name + ":dev"
    if key not in _cache:
        _cache[key] = to_device(_workload(name))
    return _cache[key]


def _workload_ref(name):
    key = name + ":ref"
    if key not in _cache:
        _cache[key] = oracle.verify_attention(_workload(name))  # every row (a few seconds on the host's threads)
    return _cache[key]


@pytest.mark.parametrize("name", ["mtp5_bf16", "mtp5_fp8", "mixed_fp8", "ctx1mi_bf16", "d256_fp8_bs8"])
@pytest.mark.parametrize("kernel", KERNELS, ids=[KID[k] for k in KERNELS])
def test_full_workload_every_row(name, kernel):
    if kernel == pv.KERNEL_WARP_MMA and name.startswith("d256"):
        pytest.skip("head_dim 256 runs on the tcgen05 kernel only")
    prob = _workload(name)
    got, va = gpu_run(prob, dev=_workload_dev(name), kernel=kernel)
    assert va.info["kernel"] == kernel
    assert max_err(got, _workload_ref(name)) <= TOL[prob.kv_dtype], name


def test_tiny_workload_runs_on_the_tcgen05_kernel():
    prob = synth.make_config("tiny")
    got, va = gpu_run(prob)
    assert va.info["kernel"] == pv.KERNEL_TCGEN05
    assert max_err(got, oracle.verify_attention(prob)) <= TOL[synth.KV_BF16]


@pytest.mark.parametrize("split", [0, 1, 4, 17])
def test_head_dim_64_flat_segments(split):
    # every segment layout of the flat plans at head_dim 64, mixed row counts (8 .. 64) in the 64-row instance
    prob = synth.make_problem(SEG_CTX, SEG_Q, 16, 2, 64, seed=39)
    got, va = gpu_run(prob, split_override=split, kernel=pv.KERNEL_TCGEN05)
    assert max_err(got, oracle.verify_attention(prob)) <= TOL[synth.KV_BF16]


# --------------------------------------------------------------- plans beyond one wave
@pytest.mark.parametrize("kv,d,hq,hkv", [(synth.KV_BF16, 128, 16, 2), (synth.KV_FP8, 256, 8, 1)], ids=["bf16", "fp8_d256"])
def test_flat_plans_beyond_one_wave(kv, d, hq, hkv):
    # one tile per CTA over more tiles than SMs: the split kernel runs several waves, the combine merges them
    prob = synth.make_problem([20000, 10000], [6, 3], hq, hkv, d, kv_dtype=kv, seed=49)
    ref = oracle.verify_attention(prob)
    got, va = gpu_run(prob, split_override=100000, kernel=pv.KERNEL_TCGEN05)
    assert va.info["num_units"] > torch.cuda.get_device_properties(0).multi_processor_count
    assert va.info["needs_combine"] == 1
    assert max_err(got, ref) <= TOL[kv]


# --------------------------------------------------------------- two-launch plans
@pytest.mark.parametrize("out_dtype", [pv.OUT_F32, pv.OUT_BF16], ids=["f32", "bf16"])
def test_two_launch_plan_against_oracle(out_dtype):
    """FP8 pairs of up to 48 rows and pairs of more, long enough that both classes split over several CTAs:
    two split launches (256-token tiles, then the 64-row instance) into one workspace, one combine."""
    prob = synth.make_problem([90000, 300, 50000, 70, 120000, 2500, 33], [6, 8, 2, 7, 8, 1, 8], 16, 2, 128,
                              kv_dtype=synth.KV_FP8, seed=57)
    ref = oracle.verify_attention(prob)
    got, va = gpu_run(prob, out_dtype=out_dtype)
    assert va.info["launches"] == 2 and va.info["needs_combine"] == 1
    second = va.plan.second()
    assert second.info.max_splits > 1 and va.info["max_splits"] > 1
    assert max_err(got, ref) <= TOL[synth.KV_FP8] + (1e-2 if out_dtype == pv.OUT_BF16 else 0.0)


def test_two_launch_plan_static_entry_point_matches():
    """The entry point without a workspace runs both launches too, bit for bit the same output."""
    prob = synth.make_problem([40000, 700, 25000, 9000], [7, 3, 8, 5], 16, 2, 128, kv_dtype=synth.KV_FP8, seed=58)
    dev = to_device(prob)
    va = pv.VerifyAttention(16, 2, 128, synth.KV_FP8, prob.num_pages, prob.block_table.shape[1],
                            prob.context_lens.tolist(), prob.query_lens.tolist())
    assert va.info["launches"] == 2
    a = va(*dev.args(), prob.softmax_scale)
    b = torch.empty_like(a)
    pv.run_static(va.plan, *dev.args(), prob.softmax_scale, b)
    torch.cuda.synchronize()
    assert pv.device_errors(None) == 0
    assert torch.equal(a, b)


# --------------------------------------------------------------- 65-128 rows: row halves
ROW_HALF_CASES = [
    ("bf16_d128", synth.KV_BF16, 128, 16, 1, [3000, 130, 8000, 600], [8, 5, 1, 7]),
    ("fp8_d128", synth.KV_FP8, 128, 16, 1, [3000, 130, 8000, 600], [8, 5, 1, 7]),
    ("bf16_d64", synth.KV_BF16, 64, 16, 1, [2000, 257, 4100], [8, 6, 3]),
    ("bf16_d256", synth.KV_BF16, 256, 16, 1, [2000, 257, 4100], [8, 6, 3]),
    ("fp8_d256", synth.KV_FP8, 256, 16, 1, [2000, 257, 4100], [8, 6, 3]),
    ("fp8_hkv2_group12", synth.KV_FP8, 128, 24, 2, [5000, 1000, 77], [7, 8, 2]),
]


@pytest.mark.parametrize("split", [0, 1, 4], ids=["planner", "one_segment", "four_way"])
@pytest.mark.parametrize("name,kv,d,hq,hkv,ctx,ql", ROW_HALF_CASES, ids=[c[0] for c in ROW_HALF_CASES])
def test_row_halves_against_oracle(name, kv, d, hq, hkv, ctx, ql, split):
    """Pairs of 65-128 rows on the tcgen05 kernel: two virtual pairs of the 64-row instance, rows 0-63 and
    the rest, each a pass over the context; every output row against the oracle."""
    prob = synth.make_problem(ctx, ql, hq, hkv, d, kv_dtype=kv, seed=59)
    ref = oracle.verify_attention(prob)
    got, va = gpu_run(prob, split_override=split, kernel=pv.KERNEL_AUTO)
    assert va.info["kernel"] == pv.KERNEL_TCGEN05 and va.info["rows_max"] > 64
    assert max_err(got, ref) <= TOL[kv], name


def test_row_halves_match_the_warp_mma_kernel():
    prob = synth.make_problem([9000, 3100], [8, 8], 16, 1, 128, seed=60)
    a, va = gpu_run(prob, kernel=pv.KERNEL_TCGEN05)
    b, vb = gpu_run(prob, kernel=pv.KERNEL_WARP_MMA)
    assert va.info["kernel"] == pv.KERNEL_TCGEN05 and vb.info["kernel"] == pv.KERNEL_WARP_MMA
    assert max_err(a, b.astype(np.float64)) <= 1e-2


def test_row_halves_without_the_combine_table():
    """320 split virtual pairs: more than the combine's table holds, so the combine finds each row's half and
    partials from the plan's work table."""
    ctx = [2000 + 37 * i for i in range(40)]
    ql = [8 - (i % 3) for i in range(40)]  # 128, 112 and 96 rows
    prob = synth.make_problem(ctx, ql, 64, 4, 128, seed=61)
    got, va = gpu_run(prob, split_override=4)
    assert va.info["kernel"] == pv.KERNEL_TCGEN05 and va.info["split_pairs"] == -1
    assert max_err(got, oracle.verify_attention(prob)) <= TOL[synth.KV_BF16]
