"""pa_verify_run_static, the entry point for callers that cannot allocate
device memory (no workspace argument; the library's fixed device scratch is
used instead). Called through the C ABI and checked against pa_verify_run on
the same inputs, on two calls in a row. This file is collected last."""
import ctypes

import numpy as np
import pytest
import torch

from paged_kv_speculative_gb300 import _build, pa_verify as pv, synth
from paged_kv_speculative_gb300.device_inputs import to_device

pytestmark = pytest.mark.gpu

TOL = {synth.KV_BF16: 1e-2, synth.KV_FP8: 2e-2}


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


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
    stream = torch.cuda.current_stream()
    for _ in range(2):
        out = torch.full_like(ref, float("nan"))
        rc = lib.pa_verify_run_static(
            ctypes.c_void_p(va.plan.handle), _ptr(dev.q), _ptr(dev.k_cache), _ptr(dev.v_cache), _ptr(dev.k_scale),
            _ptr(dev.v_scale), _ptr(dev.block_table), _ptr(dev.context_lens), _ptr(dev.query_lens),
            ctypes.c_float(prob.softmax_scale), _ptr(out), ctypes.c_void_p(stream.cuda_stream))
        assert rc == pv.OK, pv.last_error()
        torch.cuda.synchronize()
        d = (out - ref).abs()
        assert torch.isfinite(out).all()
        assert float(d.max()) <= TOL[kv]


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
    out = torch.full_like(ref, float("nan"))
    stream = torch.cuda.current_stream()
    rc = lib.pa_verify_run_static(
        ctypes.c_void_p(va.plan.handle), _ptr(dev.q), _ptr(dev.k_cache), _ptr(dev.v_cache), _ptr(dev.k_scale),
        _ptr(dev.v_scale), _ptr(dev.block_table), _ptr(dev.context_lens), _ptr(dev.query_lens),
        ctypes.c_float(prob.softmax_scale), _ptr(out), ctypes.c_void_p(stream.cuda_stream))
    assert rc == pv.OK, pv.last_error()
    torch.cuda.synchronize()
    assert torch.isfinite(out).all()
    assert float((out - ref).abs().max()) <= TOL[synth.KV_FP8]


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
