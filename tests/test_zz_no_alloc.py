"""pa_verify_run_static, the entry point for callers that cannot allocate
device memory (no workspace argument; the library's fixed device scratch is
used instead). Called through the C ABI and checked against pa_verify_run on
the same inputs, on two calls in a row: the two share the plan and the
kernels, so their outputs must be bit-identical. Its device error word is read
back through pa_verify_device_errors with a NULL workspace. This file is
collected last."""
import ctypes

import numpy as np
import pytest
import torch

from paged_kv_speculative_gb300 import _build, pa_verify as pv, synth
from paged_kv_speculative_gb300.device_inputs import to_device

pytestmark = pytest.mark.gpu

def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _static_call(lib, plan, dev, softmax_scale, out):
    stream = torch.cuda.current_stream()
    return lib.pa_verify_run_static(
        ctypes.c_void_p(plan.handle), _ptr(dev.q), _ptr(dev.k_cache), _ptr(dev.v_cache), _ptr(dev.k_scale),
        _ptr(dev.v_scale), _ptr(dev.block_table), _ptr(dev.context_lens), _ptr(dev.query_lens),
        ctypes.c_float(softmax_scale), _ptr(out), ctypes.c_void_p(stream.cuda_stream))


@pytest.mark.parametrize("kv", [synth.KV_BF16, synth.KV_FP8])
@pytest.mark.parametrize("kernel", [pv.KERNEL_AUTO, pv.KERNEL_WARP_MMA])
def test_static_scratch_matches_workspace_entry(kv, kernel):
    _build.build()
    lib = pv.lib()
    prob = synth.make_problem([3000, 777, 5000], [6, 3, 8], 16, 2, 128, kv_dtype=kv, seed=91)
    dev = to_device(prob)
    va = pv.VerifyAttention(prob.num_q_heads, prob.num_kv_heads, 128, kv, prob.num_pages, prob.block_table.shape[1],
                            prob.context_lens.tolist(), prob.query_lens.tolist(), split_override=5, kernel=kernel)
    assert va.info["needs_combine"] == 1  # the split partials live in the scratch
    ref = va(*dev.args(), prob.softmax_scale)
    torch.cuda.synchronize()
    for _ in range(2):
        out = torch.full_like(ref, float("nan"))
        rc = _static_call(lib, va.plan, dev, prob.softmax_scale, out)
        assert rc == pv.OK, pv.last_error()
        torch.cuda.synchronize()
        assert torch.equal(out, ref)
        assert pv.device_errors(None) == 0


def test_static_scratch_fp8_head_dim_256():
    _build.build()
    lib = pv.lib()
    prob = synth.make_problem([3000, 777, 5000], [6, 3, 8], 8, 1, 256, kv_dtype=synth.KV_FP8, seed=92)
    dev = to_device(prob)
    va = pv.VerifyAttention(8, 1, 256, synth.KV_FP8, prob.num_pages, prob.block_table.shape[1],
                            prob.context_lens.tolist(), prob.query_lens.tolist(), split_override=5)
    assert va.info["needs_combine"] == 1 and va.info["kernel"] == pv.KERNEL_TCGEN05
    ref = va(*dev.args(), prob.softmax_scale)
    torch.cuda.synchronize()
    for _ in range(2):
        out = torch.full_like(ref, float("nan"))
        rc = _static_call(lib, va.plan, dev, prob.softmax_scale, out)
        assert rc == pv.OK, pv.last_error()
        torch.cuda.synchronize()
        assert torch.equal(out, ref)


def test_static_scratch_with_a_dynamic_plan():
    """A capacity plan keeps its device-written work table in the scratch too."""
    _build.build()
    lib = pv.lib()
    prob = synth.make_problem([3000, 5, 2200, 900], [6, 1, 8, 3], 16, 2, 128, seed=93)
    dev = to_device(prob)
    plan = pv.plan_dynamic(16, 2, 128, synth.KV_BF16, pv.OUT_F32, prob.num_pages, prob.block_table.shape[1],
                           capacity=4, max_context_len=3000, max_query_len=8)
    assert plan.workspace_bytes <= (16 << 20)
    ws = torch.zeros(plan.workspace_bytes, dtype=torch.uint8, device="cuda")
    ref = torch.empty((int(prob.query_lens.sum()), 16, 128), dtype=torch.float32, device="cuda")
    pv.run(plan, *dev.args(), prob.softmax_scale, ref, ws)
    torch.cuda.synchronize()
    assert pv.device_errors(ws) == 0
    for _ in range(2):
        out = torch.full_like(ref, float("nan"))
        rc = _static_call(lib, plan, dev, prob.softmax_scale, out)
        assert rc == pv.OK, pv.last_error()
        torch.cuda.synchronize()
        assert torch.equal(out, ref)
        assert pv.device_errors(None) == 0


def test_static_scratch_error_word_reads_back():
    """An out-of-range page id, then device lengths that differ from the plan's,
    are flagged in the fixed scratch's error word; each call starts from a
    cleared word."""
    _build.build()
    lib = pv.lib()
    prob = synth.make_problem([900, 400], [6, 3], 16, 2, 128, seed=94)
    dev = to_device(prob)
    va = pv.VerifyAttention(16, 2, 128, synth.KV_BF16, prob.num_pages, prob.block_table.shape[1],
                            prob.context_lens.tolist(), prob.query_lens.tolist(), split_override=3)
    ref = va(*dev.args(), prob.softmax_scale)
    out = torch.empty_like(ref)
    bad = dev.block_table.clone()
    bad[0, 2] = prob.num_pages + 77  # not a pool page: zeros are read instead, and the word says so
    dev_bad = type(dev)(**{**dev.__dict__, "block_table": bad})
    assert _static_call(lib, va.plan, dev_bad, prob.softmax_scale, out) == pv.OK, pv.last_error()
    assert pv.device_errors(None) & pv.DEVERR_PAGE_RANGE
    # device lengths that differ from the plan's: the kernel follows the plan and the word says so
    ctx_bad = dev.context_lens.clone()
    ctx_bad[1] += 5
    dev_len = type(dev)(**{**dev.__dict__, "context_lens": ctx_bad})
    assert _static_call(lib, va.plan, dev_len, prob.softmax_scale, out) == pv.OK, pv.last_error()
    flags = pv.device_errors(None)
    assert flags & pv.DEVERR_LENGTHS and not flags & pv.DEVERR_PAGE_RANGE
    assert _static_call(lib, va.plan, dev, prob.softmax_scale, out) == pv.OK, pv.last_error()
    assert pv.device_errors(None) == 0
    torch.cuda.synchronize()
    assert torch.equal(out, ref)


def test_static_scratch_refuses_plans_that_do_not_fit():
    _build.build()
    lib = pv.lib()
    # 64 sequences x 8 KV heads split into many chunks: partials far above the fixed scratch
    p = pv.plan(64, 8, 128, pv.KV_BF16, pv.OUT_F32, 64 * 2048, 2048, [32768] * 64, [8] * 64,
                split_override=200, kernel=pv.KERNEL_WARP_MMA)
    assert p.workspace_bytes > (16 << 20)
    buf = torch.zeros(16, dtype=torch.uint8, device="cuda")
    rc = lib.pa_verify_run_static(ctypes.c_void_p(p.handle), *([_ptr(buf)] * 8), ctypes.c_float(0.1), _ptr(buf),
                                  None)
    assert rc == pv.ERR_WORKSPACE
    assert "scratch" in pv.last_error()
