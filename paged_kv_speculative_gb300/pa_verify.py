"""Python binding of the C ABI in ``include/pa_verify.h``.

Argument marshalling only: every step of the attention runs in the CUDA
library ``_lib/libpa_verify.so``. There is no fallback; if the library is
missing or fails to load, every entry point raises.

Functions keep the C names without the ``pa_verify_`` prefix: ``plan``,
``run``, ``free``, ``device_errors``, ``last_error``. ``VerifyAttention``
bundles a plan with its device workspace.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import torch

from . import _build

KV_BF16 = 0
KV_FP8_E4M3 = 1
OUT_BF16 = 0
OUT_F32 = 1

OK = 0
ERR_INVALID = -1
ERR_UNSUPPORTED = -2
ERR_WORKSPACE = -3
ERR_CUDA = -4
ERR_NOMEM = -5

KERNEL_AUTO = 0
KERNEL_WARP_MMA = 1
KERNEL_TCGEN05 = 2

DEVERR_PAGE_RANGE = 1
DEVERR_LENGTHS = 2
DEVERR_TIMEOUT = 4

# every symbol include/pa_verify.h declares
EXPORTED = ("pa_verify_plan", "pa_verify_plan_get_info", "pa_verify_run", "pa_verify_free",
            "pa_verify_device_errors", "pa_verify_last_error", "pa_verify_profile_enable",
            "pa_verify_profile_read", "pa_kv_write", "pa_greedy_verdict_workspace_bytes",
            "pa_greedy_verdict", "pa_verify_run_static", "pa_verify_plan_dynamic", "pa_verify_plan_get_cta_starts",
            "pa_verify_debug_stall", "pa_verify_plan_get_second")


class PaVerifyError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"pa_verify status {status}: {message}")
        self.status = status


class Desc(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "num_seqs", "num_q_heads", "num_kv_heads", "head_dim", "page_size", "kv_dtype", "out_dtype",
        "num_pages", "block_table_stride", "split_override", "sm_count", "kernel")]


class KvWriteDesc(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("num_tokens", "num_kv_heads", "head_dim", "kv_dtype", "num_pages")]


class PlanInfo(ctypes.Structure):
    _fields_ = [
        ("num_units", ctypes.c_int32), ("chunk_tokens", ctypes.c_int32), ("tile_tokens", ctypes.c_int32),
        ("rows_max", ctypes.c_int32), ("warps", ctypes.c_int32), ("max_splits", ctypes.c_int32),
        ("needs_combine", ctypes.c_int32), ("num_tokens", ctypes.c_int32), ("kv_bytes", ctypes.c_int64),
        ("workspace_bytes", ctypes.c_size_t), ("kernel", ctypes.c_int32), ("dynamic", ctypes.c_int32),
        ("flat", ctypes.c_int32), ("total_tiles", ctypes.c_int32), ("device_table", ctypes.c_int32),
        ("launches", ctypes.c_int32), ("split_pairs", ctypes.c_int32)]

    def as_dict(self) -> dict:
        return {k: getattr(self, k) for k, _ in self._fields_}


_lib = None


def lib(path: Optional[str] = None):
    """Loads the library (it must have been built: ``__graft_entry__.build()``)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or _build.LIB
    if not os.path.exists(p):
        raise RuntimeError(f"CUDA library {p} is not built; run __graft_entry__.build() first")
    L = ctypes.CDLL(p)
    vp, sz, i32p = ctypes.c_void_p, ctypes.c_size_t, ctypes.POINTER(ctypes.c_int32)
    L.pa_verify_plan.argtypes = [ctypes.POINTER(Desc), i32p, i32p, ctypes.POINTER(vp), ctypes.POINTER(sz)]
    L.pa_verify_plan.restype = ctypes.c_int
    L.pa_verify_plan_dynamic.argtypes = [ctypes.POINTER(Desc), ctypes.c_int32, ctypes.c_int32, ctypes.POINTER(vp),
                                         ctypes.POINTER(sz)]
    L.pa_verify_plan_dynamic.restype = ctypes.c_int
    L.pa_verify_plan_get_info.argtypes = [vp, ctypes.POINTER(PlanInfo)]
    L.pa_verify_plan_get_info.restype = ctypes.c_int
    L.pa_verify_plan_get_cta_starts.argtypes = [vp, i32p, ctypes.c_int32]
    L.pa_verify_plan_get_cta_starts.restype = ctypes.c_int
    L.pa_verify_plan_get_second.argtypes = [vp]
    L.pa_verify_plan_get_second.restype = vp
    L.pa_verify_run.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_float, vp, vp, sz, vp]
    L.pa_verify_run.restype = ctypes.c_int
    L.pa_verify_run_static.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_float, vp, vp]
    L.pa_verify_run_static.restype = ctypes.c_int
    L.pa_verify_debug_stall.argtypes = [vp, ctypes.c_int32, ctypes.c_uint32]
    L.pa_verify_debug_stall.restype = ctypes.c_int
    L.pa_verify_free.argtypes = [vp]
    L.pa_verify_free.restype = None
    L.pa_verify_device_errors.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32), ctypes.c_int, vp]
    L.pa_verify_device_errors.restype = ctypes.c_int
    L.pa_verify_profile_enable.argtypes = [vp, ctypes.c_int]
    L.pa_verify_profile_enable.restype = ctypes.c_int
    L.pa_verify_profile_read.argtypes = [vp, ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_float)]
    L.pa_verify_profile_read.restype = ctypes.c_int
    L.pa_kv_write.argtypes = [ctypes.POINTER(KvWriteDesc), vp, vp, vp, vp, vp, vp, vp, vp, vp]
    L.pa_kv_write.restype = ctypes.c_int
    L.pa_greedy_verdict_workspace_bytes.argtypes = [ctypes.c_int32, ctypes.c_int32]
    L.pa_greedy_verdict_workspace_bytes.restype = ctypes.c_size_t
    L.pa_greedy_verdict.argtypes = [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32] + [vp] * 7 + [sz, vp]
    L.pa_greedy_verdict.restype = ctypes.c_int
    L.pa_verify_last_error.argtypes = []
    L.pa_verify_last_error.restype = ctypes.c_char_p
    if path is None:
        _lib = L
    return L


def last_error() -> str:
    return lib().pa_verify_last_error().decode()


def _check(status: int):
    if status != OK:
        raise PaVerifyError(status, last_error())


class Plan:
    """A host-side plan (owns the C handle)."""

    def __init__(self, handle: int, desc: Desc, workspace_bytes: int, owned: bool = True):
        self.handle = handle
        self.desc = desc
        self.workspace_bytes = workspace_bytes
        self.owned = owned
        info = PlanInfo()
        _check(lib().pa_verify_plan_get_info(handle, ctypes.byref(info)))
        self.info = info

    def second(self) -> Optional["Plan"]:
        """The second launch of a two-launch plan (a view owned by this plan), or None."""
        h = lib().pa_verify_plan_get_second(self.handle)
        if not h:
            return None
        v = Plan(h, self.desc, self.workspace_bytes, owned=False)
        v.parent = self  # keeps the owner alive while the view is used
        return v

    def cta_starts(self) -> list:
        """A static flat plan's CTA ranges: CTA c covers flat tiles [s[c], s[c + 1])."""
        buf = (ctypes.c_int32 * (self.info.num_units + 1))()
        n = lib().pa_verify_plan_get_cta_starts(self.handle, buf, len(buf))
        _check(min(n, 0))
        return list(buf[:n])

    def free(self):
        if self.handle and self.owned:
            lib().pa_verify_free(self.handle)
        self.handle = None

    def __del__(self):
        try:
            self.free()
        except Exception:
            pass


def _runnable(p: Plan):
    if not p.owned:
        raise ValueError("the second launch of a two-launch plan runs only as part of its plan")


def plan(num_q_heads: int, num_kv_heads: int, head_dim: int, kv_dtype: int, out_dtype: int, num_pages: int,
         block_table_stride: int, context_lens: Sequence[int], query_lens: Sequence[int],
         split_override: int = 0, sm_count: int = 0, page_size: int = 16, kernel: int = KERNEL_AUTO) -> Plan:
    """pa_verify_plan with host lengths; raises PaVerifyError on refusal."""
    n = len(context_lens)
    d = Desc(num_seqs=n, num_q_heads=num_q_heads, num_kv_heads=num_kv_heads, head_dim=head_dim,
             page_size=page_size, kv_dtype=kv_dtype, out_dtype=out_dtype, num_pages=num_pages,
             block_table_stride=block_table_stride, split_override=split_override, sm_count=sm_count,
             kernel=kernel)
    arr = ctypes.c_int32 * max(1, n)
    cl = arr(*[int(x) for x in context_lens])
    ql = arr(*[int(x) for x in query_lens])
    h = ctypes.c_void_p()
    ws = ctypes.c_size_t()
    _check(lib().pa_verify_plan(ctypes.byref(d), cl, ql, ctypes.byref(h), ctypes.byref(ws)))
    return Plan(h.value, d, ws.value)


def plan_dynamic(num_q_heads: int, num_kv_heads: int, head_dim: int, kv_dtype: int, out_dtype: int, num_pages: int,
                 block_table_stride: int, capacity: int, max_context_len: int, max_query_len: int,
                 sm_count: int = 0, kernel: int = KERNEL_AUTO) -> Plan:
    """pa_verify_plan_dynamic: a capacity plan whose lengths are read on the device each run."""
    d = Desc(num_seqs=capacity, num_q_heads=num_q_heads, num_kv_heads=num_kv_heads, head_dim=head_dim, page_size=16,
             kv_dtype=kv_dtype, out_dtype=out_dtype, num_pages=num_pages, block_table_stride=block_table_stride,
             split_override=0, sm_count=sm_count, kernel=kernel)
    h = ctypes.c_void_p()
    ws = ctypes.c_size_t()
    _check(lib().pa_verify_plan_dynamic(ctypes.byref(d), int(max_context_len), int(max_query_len), ctypes.byref(h),
                                        ctypes.byref(ws)))
    return Plan(h.value, d, ws.value)


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _need(t: torch.Tensor, name: str, dtype=None):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")


def run(p: Plan, q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, k_scale: Optional[torch.Tensor],
        v_scale: Optional[torch.Tensor], block_table: torch.Tensor, context_lens: torch.Tensor,
        query_lens: torch.Tensor, softmax_scale: float, out: torch.Tensor, workspace: torch.Tensor,
        stream: Optional[torch.cuda.Stream] = None):
    """pa_verify_run on device tensors (enqueued on ``stream`` or torch's current stream)."""
    _runnable(p)
    _need(q, "q", torch.bfloat16)
    for t, nm in ((k_cache, "k_cache"), (v_cache, "v_cache"), (out, "out"), (workspace, "workspace")):
        _need(t, nm)
    for t, nm in ((block_table, "block_table"), (context_lens, "context_lens"), (query_lens, "query_lens")):
        _need(t, nm, torch.int32)
    for t, nm in ((k_scale, "k_scale"), (v_scale, "v_scale")):
        if t is not None:
            _need(t, nm, torch.float32)
    s = stream if stream is not None else torch.cuda.current_stream(q.device)
    _check(lib().pa_verify_run(p.handle, _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
                               _ptr(block_table), _ptr(context_lens), _ptr(query_lens), float(softmax_scale),
                               _ptr(out), _ptr(workspace), workspace.numel() * workspace.element_size(),
                               s.cuda_stream))


def run_static(p: Plan, q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
               k_scale: Optional[torch.Tensor], v_scale: Optional[torch.Tensor], block_table: torch.Tensor,
               context_lens: torch.Tensor, query_lens: torch.Tensor, softmax_scale: float, out: torch.Tensor,
               stream: Optional[torch.cuda.Stream] = None):
    """pa_verify_run_static: like ``run`` but with the library's fixed device
    scratch instead of a workspace, for callers that cannot allocate."""
    _runnable(p)
    _need(q, "q", torch.bfloat16)
    for t, nm in ((k_cache, "k_cache"), (v_cache, "v_cache"), (out, "out")):
        _need(t, nm)
    s = stream if stream is not None else torch.cuda.current_stream(q.device)
    _check(lib().pa_verify_run_static(p.handle, _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale),
                                      _ptr(v_scale), _ptr(block_table), _ptr(context_lens), _ptr(query_lens),
                                      float(softmax_scale), _ptr(out), s.cuda_stream))


def device_errors(workspace: Optional[torch.Tensor], clear: bool = False,
                  stream: Optional[torch.cuda.Stream] = None) -> int:
    """The device error word of ``workspace``; ``None`` reads the fixed scratch of ``run_static``."""
    s = stream if stream is not None else torch.cuda.current_stream(
        workspace.device if workspace is not None else None)
    flags = ctypes.c_uint32()
    _check(lib().pa_verify_device_errors(_ptr(workspace), ctypes.byref(flags), int(bool(clear)), s.cuda_stream))
    return int(flags.value)


def rescale_count(workspace: torch.Tensor) -> int:
    """Word 1 of a workspace header: in-segment rescales of the output accumulator so far."""
    return int(workspace[4:8].view(torch.int32).item())


def debug_stall(p: Plan, stall_cta: int, wait_limit_us: int = 0):
    """pa_verify_debug_stall: bounded-wait test hook (stall_cta = -1 and 0 restore the defaults)."""
    _check(lib().pa_verify_debug_stall(p.handle, int(stall_cta), int(wait_limit_us)))


def profile_enable(p: Plan, enable: bool = True):
    _check(lib().pa_verify_profile_enable(p.handle, int(bool(enable))))


def profile_read(p: Plan):
    """(split kernel ms, combine kernel ms) of the last profiled run."""
    a, b = ctypes.c_float(), ctypes.c_float()
    _check(lib().pa_verify_profile_read(p.handle, ctypes.byref(a), ctypes.byref(b)))
    return float(a.value), float(b.value)


def free(p: Plan):
    p.free()


def kv_write(k_new: torch.Tensor, v_new: torch.Tensor, slot_mapping: torch.Tensor, k_cache: torch.Tensor,
             v_cache: torch.Tensor, k_scale: Optional[torch.Tensor], v_scale: Optional[torch.Tensor],
             kv_dtype: int, error_flags: Optional[torch.Tensor] = None, stream: Optional[torch.cuda.Stream] = None):
    """pa_kv_write: stores new tokens' K/V rows [n, Hkv, D] into their slots."""
    _need(k_new, "k_new", torch.bfloat16)
    _need(v_new, "v_new", torch.bfloat16)
    _need(slot_mapping, "slot_mapping", torch.int64)
    _need(k_cache, "k_cache")
    _need(v_cache, "v_cache")
    n, hkv, d = k_new.shape
    desc = KvWriteDesc(num_tokens=n, num_kv_heads=hkv, head_dim=d, kv_dtype=kv_dtype, num_pages=k_cache.shape[0])
    s = stream if stream is not None else torch.cuda.current_stream(k_new.device)
    _check(lib().pa_kv_write(ctypes.byref(desc), _ptr(k_new), _ptr(v_new), _ptr(slot_mapping), _ptr(k_cache),
                             _ptr(v_cache), _ptr(k_scale), _ptr(v_scale), _ptr(error_flags), s.cuda_stream))


class VerifyAttention:
    """A plan plus a zero-initialised device workspace for one batch shape."""

    def __init__(self, num_q_heads: int, num_kv_heads: int, head_dim: int, kv_dtype: int, num_pages: int,
                 block_table_stride: int, context_lens: Sequence[int], query_lens: Sequence[int],
                 out_dtype: int = OUT_F32, split_override: int = 0, device: Optional[torch.device] = None,
                 kernel: int = KERNEL_AUTO):
        self.device = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
        with torch.cuda.device(self.device):
            self.plan = plan(num_q_heads, num_kv_heads, head_dim, kv_dtype, out_dtype, num_pages, block_table_stride,
                             context_lens, query_lens, split_override=split_override, kernel=kernel)
        self.out_dtype = out_dtype
        self.num_q_heads = num_q_heads
        self.head_dim = head_dim
        self.workspace = torch.zeros(max(256, self.plan.workspace_bytes), dtype=torch.uint8, device=self.device)

    @property
    def info(self) -> dict:
        return self.plan.info.as_dict()

    def new_out(self) -> torch.Tensor:
        T = self.plan.info.num_tokens
        dt = torch.float32 if self.out_dtype == OUT_F32 else torch.bfloat16
        return torch.empty((T, self.num_q_heads, self.head_dim), dtype=dt, device=self.device)

    def __call__(self, q, k_cache, v_cache, k_scale, v_scale, block_table, context_lens, query_lens,
                 softmax_scale: float, out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
        if out is None:
            out = self.new_out()
        run(self.plan, q, k_cache, v_cache, k_scale, v_scale, block_table, context_lens, query_lens,
            softmax_scale, out, self.workspace, stream)
        return out

    def device_errors(self, clear: bool = False) -> int:
        return device_errors(self.workspace, clear=clear)


def greedy_verdict(logits: torch.Tensor, input_ids: torch.Tensor, query_lens: torch.Tensor,
                   workspace: Optional[torch.Tensor] = None, stream: Optional[torch.cuda.Stream] = None):
    """pa_greedy_verdict: (target_ids [T], accepted [B], next_token [B]) int32 device tensors."""
    _need(logits, "logits", torch.bfloat16)
    _need(input_ids, "input_ids", torch.int32)
    _need(query_lens, "query_lens", torch.int32)
    T, V = logits.shape
    B = query_lens.shape[0]
    dev = logits.device
    need = lib().pa_greedy_verdict_workspace_bytes(T, V)
    if workspace is None:
        workspace = torch.zeros(max(256, need), dtype=torch.uint8, device=dev)
    tgt = torch.empty(T, dtype=torch.int32, device=dev)
    acc = torch.empty(B, dtype=torch.int32, device=dev)
    nxt = torch.empty(B, dtype=torch.int32, device=dev)
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    _check(lib().pa_greedy_verdict(B, T, V, _ptr(logits), _ptr(input_ids), _ptr(query_lens), _ptr(tgt), _ptr(acc),
                                   _ptr(nxt), _ptr(workspace), workspace.numel(), s.cuda_stream))
    return tgt, acc, nxt
