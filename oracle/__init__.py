"""CPU fp64 oracle for paged verify attention: TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
legs of ``bench.py`` may import this package. It shares no code with the CUDA
library (``paged_kv_speculative_gb300``) and imports nothing from it; the two
meet only in the seeded input generator, which holds none of the method's
arithmetic.

The arithmetic lives in ``pa_oracle.c`` (plain C, fp64, two-pass softmax);
this module compiles it with gcc and calls it through ctypes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pa_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_lock = threading.Lock()
_libs: dict = {}


class _Problem(ctypes.Structure):
    _fields_ = [
        ("num_seqs", ctypes.c_int32),
        ("num_q_heads", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("kv_dtype", ctypes.c_int32),
        ("num_pages", ctypes.c_int32),
        ("block_table_stride", ctypes.c_int32),
        ("pad_", ctypes.c_int32),
        ("q", ctypes.c_void_p),
        ("k_cache", ctypes.c_void_p),
        ("v_cache", ctypes.c_void_p),
        ("k_scale", ctypes.c_void_p),
        ("v_scale", ctypes.c_void_p),
        ("block_table", ctypes.c_void_p),
        ("context_lens", ctypes.c_void_p),
        ("query_lens", ctypes.c_void_p),
        ("softmax_scale", ctypes.c_double),
    ]


def lib_path(mutant: int = 0) -> str:
    return os.path.join(_BUILD, f"libpa_oracle_m{int(mutant)}.so")


def build(mutant: int = 0, force: bool = False) -> str:
    """Compile the oracle (gcc, -O2, no fast-math: IEEE fp64 throughout)."""
    out = lib_path(mutant)
    with _lock:
        if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(_SRC):
            return out
        os.makedirs(_BUILD, exist_ok=True)
        tmp = out + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-fno-fast-math",
               "-ffp-contract=off", f"-DORACLE_MUTANT={int(mutant)}", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, out)
        return out


def _load(mutant: int = 0):
    if mutant in _libs:
        return _libs[mutant]
    lib = ctypes.CDLL(build(mutant))
    lib.oracle_verify_attention.argtypes = [ctypes.POINTER(_Problem), ctypes.c_void_p, ctypes.c_int64,
                                            ctypes.c_void_p, ctypes.c_int]
    lib.oracle_verify_attention.restype = ctypes.c_int
    lib.oracle_decode_e4m3.argtypes = [ctypes.c_uint8]
    lib.oracle_decode_e4m3.restype = ctypes.c_double
    lib.oracle_decode_bf16.argtypes = [ctypes.c_uint16]
    lib.oracle_decode_bf16.restype = ctypes.c_double
    lib.oracle_encode_e4m3.argtypes = [ctypes.c_float]
    lib.oracle_encode_e4m3.restype = ctypes.c_uint8
    vp = ctypes.c_void_p
    lib.oracle_kv_write.argtypes = [ctypes.c_int32] * 5 + [vp] * 7
    lib.oracle_kv_write.restype = ctypes.c_int
    lib.oracle_greedy_verdict.argtypes = [ctypes.c_int32, vp, ctypes.c_int32, vp, vp, vp, vp, vp]
    lib.oracle_greedy_verdict.restype = ctypes.c_int
    _libs[mutant] = lib
    return lib


def decode_e4m3(codes) -> np.ndarray:
    lib = _load()
    return np.array([lib.oracle_decode_e4m3(int(c)) for c in np.asarray(codes).ravel()], dtype=np.float64)


def decode_bf16(bits) -> np.ndarray:
    lib = _load()
    return np.array([lib.oracle_decode_bf16(int(c)) for c in np.asarray(bits).ravel()], dtype=np.float64)


def encode_e4m3(values) -> np.ndarray:
    lib = _load()
    return np.array([lib.oracle_encode_e4m3(float(v)) for v in np.asarray(values, dtype=np.float32).ravel()],
                    dtype=np.uint8)


def kv_write(k_new: np.ndarray, v_new: np.ndarray, slot_mapping: np.ndarray, k_cache: np.ndarray,
             v_cache: np.ndarray, k_scale: Optional[np.ndarray], v_scale: Optional[np.ndarray],
             kv_dtype: int) -> int:
    """Paged KV write (in place on the given host arrays). k_new/v_new: uint16
    bf16 bits [n, Hkv, D]; slot_mapping int64 [n] (-1 skips the token).
    Returns the oracle's status (0, or -1 if a slot was out of range)."""
    lib = _load()
    n, hkv, d = k_new.shape
    for a in (k_new, v_new, k_cache, v_cache):
        assert a.flags.c_contiguous
    sm = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    return lib.oracle_kv_write(n, hkv, d, kv_dtype, k_cache.shape[0], k_new.ctypes.data, v_new.ctypes.data,
                               sm.ctypes.data, k_cache.ctypes.data, v_cache.ctypes.data,
                               None if k_scale is None else k_scale.ctypes.data,
                               None if v_scale is None else v_scale.ctypes.data)


def greedy_verdict(query_lens: np.ndarray, logits_bf16: np.ndarray, input_ids: np.ndarray):
    """(target_ids [T], accepted [B], next_token [B]) of a greedy verify step.
    logits_bf16: uint16 [T, V]; input_ids: int32 [T] (per sequence: last
    committed token, then the drafts)."""
    lib = _load()
    ql = np.ascontiguousarray(query_lens, dtype=np.int32)
    lg = np.ascontiguousarray(logits_bf16, dtype=np.uint16)
    ids = np.ascontiguousarray(input_ids, dtype=np.int32)
    T, V = lg.shape
    tgt = np.empty(T, dtype=np.int32)
    acc = np.empty(ql.shape[0], dtype=np.int32)
    nxt = np.empty(ql.shape[0], dtype=np.int32)
    rc = lib.oracle_greedy_verdict(ql.shape[0], ql.ctypes.data, V, lg.ctypes.data, ids.ctypes.data,
                                   tgt.ctypes.data, acc.ctypes.data, nxt.ctypes.data)
    if rc != 0:
        raise RuntimeError(f"oracle_greedy_verdict failed with status {rc}")
    return tgt, acc, nxt


def _ptr(a: Optional[np.ndarray]) -> Optional[int]:
    return None if a is None else a.ctypes.data


def verify_attention(prob, rows: Optional[np.ndarray] = None, threads: Optional[int] = None,
                     mutant: int = 0) -> np.ndarray:
    """fp64 verify attention of ``prob`` (a ``synth.Problem``).

    ``rows``: optional int64 array [n, 2] of (token, q head) pairs; the result
    is then [n, D]. Without it the result is [T, Hq, D]."""
    lib = _load(mutant)
    arrs = dict(q=np.ascontiguousarray(prob.q), k=np.ascontiguousarray(prob.k_cache),
                v=np.ascontiguousarray(prob.v_cache), bt=np.ascontiguousarray(prob.block_table, dtype=np.int32),
                cl=np.ascontiguousarray(prob.context_lens, dtype=np.int32),
                ql=np.ascontiguousarray(prob.query_lens, dtype=np.int32))
    ks = None if prob.k_scale is None else np.ascontiguousarray(prob.k_scale, dtype=np.float32)
    vs = None if prob.v_scale is None else np.ascontiguousarray(prob.v_scale, dtype=np.float32)
    p = _Problem(num_seqs=prob.num_seqs, num_q_heads=prob.num_q_heads, num_kv_heads=prob.num_kv_heads,
                 head_dim=prob.head_dim, kv_dtype=prob.kv_dtype, num_pages=prob.num_pages,
                 block_table_stride=arrs["bt"].shape[1], pad_=0,
                 q=_ptr(arrs["q"]), k_cache=_ptr(arrs["k"]), v_cache=_ptr(arrs["v"]),
                 k_scale=_ptr(ks), v_scale=_ptr(vs), block_table=_ptr(arrs["bt"]),
                 context_lens=_ptr(arrs["cl"]), query_lens=_ptr(arrs["ql"]),
                 softmax_scale=float(prob.softmax_scale))
    T, Hq, D = prob.num_tokens, prob.num_q_heads, prob.head_dim
    if rows is None:
        n = T * Hq
        rows_arr = None
    else:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1, 2))
        n = rows_arr.shape[0]
    out = np.empty((n, D), dtype=np.float64)
    nthr = threads if threads is not None else (os.cpu_count() or 1)
    rc = lib.oracle_verify_attention(ctypes.byref(p), _ptr(rows_arr), n, _ptr(out), int(nthr))
    if rc != 0:
        raise RuntimeError(f"oracle_verify_attention failed with status {rc}")
    return out.reshape(T, Hq, D) if rows is None else out
