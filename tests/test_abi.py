"""The C ABI on the CPU: the library loads, exports what the header declares,
plans and refuses without a GPU (no compute call is made here)."""
import ctypes
import os
import re

import numpy as np
import pytest

from paged_kv_speculative_gb300 import _build, pa_verify as pv

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="session", autouse=True)
def built():
    _build.build()


def header_symbols():
    txt = open(os.path.join(ROOT, "include", "pa_verify.h")).read()
    return sorted(set(re.findall(r"^(?:int|void|size_t|const char\*|pa_verify_plan_t)\s+(pa_\w+)\s*\(", txt, flags=re.M)))


def test_header_symbols_exported():
    syms = header_symbols()
    assert set(syms) == set(pv.EXPORTED)
    lib = ctypes.CDLL(_build.LIB)
    for s in syms:
        assert hasattr(lib, s), s


def mk(ctx, ql, hq=8, hkv=1, d=128, kv=pv.KV_BF16, sms=152, stride=None, pages=None, **kw):
    stride = stride or max(1, max((c + 15) // 16 for c in ctx) if ctx else 1)
    pages = pages or max(1, sum((c + 15) // 16 for c in ctx))
    return pv.plan(hq, hkv, d, kv, pv.OUT_F32, pages, stride, ctx, ql, sm_count=sms, **kw)


def test_rows_follow_the_pages_shape_facts():
    with open(os.path.join(ROOT, "tests", "golden", "shape_facts.txt")) as f:
        facts = [tuple(int(x) for x in ln.split("#")[0].split()) for ln in f if ln.split("#")[0].strip()]
    assert facts
    for qlen, group, rows in facts:
        p = mk([4096], [qlen], hq=group, hkv=1)
        assert p.info.rows_max == rows
        assert p.info.warps == (rows + 15) // 16


CASES = [([37, 100], [1, 6], 1), ([4096 + 7 * i for i in range(8)], [6] * 8, 4),
         ([1 << 20], [6], 1), ([5, 9000, 131072, 64], [3, 8, 1, 2], 2)]


def tc_tile(kv, d, rows_max):
    """Tokens per K/V tile of the tensor-core kernel: 256 for FP8 K/V at head_dim 128 with up to 48 rows
    (two 128-token MMA sub-tiles), 128 elsewhere."""
    return 256 if kv == pv.KV_FP8_E4M3 and d == 128 and rows_max <= 48 else 128


# The planner's cost model, in 1/32 of the instance's tile: a tile costs 32 (64-row instances: 32 + rows // 10,
# since they skip the P work of empty column chunks); a pair switch costs the measured number of tiles below,
# in half tiles by (K/V type, head_dim) and N = 16, 32, 48, 64.
SWITCH_HALF_TILES = {(pv.KV_BF16, 64): (4, 10, 20, 26), (pv.KV_BF16, 128): (4, 10, 20, 26),
                     (pv.KV_BF16, 256): (4, 6, 7, 14), (pv.KV_FP8_E4M3, 128): (4, 11, 20, 26),
                     (pv.KV_FP8_E4M3, 256): (4, 8, 16, 40)}


def costs(rows_max, rows, kv=pv.KV_BF16, d=128):
    np_ = 16 if rows_max <= 16 else 32 if rows_max <= 32 else 48 if rows_max <= 48 else 64
    return (32 + rows // 10 if np_ == 64 else 32), SWITCH_HALF_TILES[(kv, d)][np_ // 16 - 1] * 16


def pack(nt, w, sw, tau):
    """Greedy cut of the tiles into CTA ranges of cost (tile costs + sw per pair switch) <= tau."""
    starts, ctas, load, pos, open_ = [], 0, 0, 0, False
    for n, wk in zip(nt, w):
        rem = n
        while rem > 0:
            if not open_:
                starts.append(pos)
                open_, load = True, 0
            enter = sw if load > 0 else 0
            room = tau - load - enter
            if room < wk:
                ctas, open_ = ctas + 1, False
                continue
            take = min(rem, room // wk)
            load, rem, pos = load + enter + take * wk, rem - take, pos + take
    ctas += open_
    return ctas, starts + [pos]


def flat_model(ctx, ql, hkv, sms, split_override=0, group=8, tile=128, kv=pv.KV_BF16, d=128):
    """Independent model of a flat plan: pairs (longest sequence first, then KV
    head; a pair of more than 64 rows as two row halves, rows 0-63 then the
    rest) end to end as `tile`-token tiles, cut into CTA ranges. Returns (CTA
    starts, every (virtual) pair's (first tile, tiles), the cost bound)."""
    order = sorted(range(len(ctx)), key=lambda b: -ctx[b])  # stable: ties keep batch order
    halves = lambda b: [ql[b] * group] if ql[b] * group <= 64 else [64, ql[b] * group - 64]
    nt = [-(-ctx[b] // tile) for b in order for _ in range(hkv) for _ in halves(b)]
    rows_max = max(ql) * group
    w = [costs(rows_max, r, kv, d)[0] for b in order for _ in range(hkv) for r in halves(b)]
    sw = costs(rows_max, 0, kv, d)[1]
    total = sum(nt)
    pairs, t = [], 0
    for n in nt:
        pairs.append((t, n))
        t += n
    if split_override:
        per = max(1, -(-max(nt) // split_override))
        return [min(c * per, total) for c in range(-(-total // per) + 1)], pairs, None
    cost = sum(n * wk for n, wk in zip(nt, w))
    lo, hi = max(-(-cost // sms), max(w)), cost + sw * len(nt)
    while lo < hi:
        mid = (lo + hi) // 2
        if pack(nt, w, sw, mid)[0] <= sms:
            hi = mid
        else:
            lo = mid + 1
    return pack(nt, w, sw, lo)[1], pairs, (lo, w, sw)


def check_launch(starts, chunk_tokens, ctx, ql, hkv, split, sms, kv, group=8):
    """One launch's CTA ranges equal the model's and keep the invariants the kernels rely on; returns the
    (virtual) pairs' CTA spans."""
    T = tc_tile(kv, 128, group * max(ql))
    m_starts, pairs, bound = flat_model(ctx, ql, hkv, sms, split, group=group, tile=T, kv=kv)
    assert starts == m_starts
    assert starts[-1] == hkv * sum(-(-c // T) * (2 if q * group > 64 else 1) for c, q in zip(ctx, ql))
    # the ranges tile the flat space once, without empty CTAs
    assert starts[0] == 0 and all(a < b for a, b in zip(starts, starts[1:]))
    n = len(starts) - 1
    cta_of = lambda f: max(c for c in range(n) if starts[c] <= f)
    spans = [(cta_of(t0), cta_of(t0 + nt - 1)) for t0, nt in pairs]
    if split == 0:
        assert n <= sms
        # no CTA costs more than the bound, which the plan reports in whole tiles as the chunk
        tau, w, sw = bound
        assert chunk_tokens // T == -(-tau // 32)
        for c in range(n):
            cost = sw * (sum(1 for a, b in spans if a <= c <= b) - 1)
            for k, (t0, nt) in enumerate(pairs):
                cost += w[k] * max(0, min(t0 + nt, starts[c + 1]) - max(t0, starts[c]))
            assert cost <= tau
    return spans


def check_flat_plan(ctx, ql, hkv, split, sms=152, kv=pv.KV_BF16, group=8):
    """The library's flat plan equals the model's ranges and keeps every invariant the kernels rely on. A batch
    of FP8 pairs with up to 48 rows and pairs with more is planned as two launches, one per class."""
    p = mk(ctx, ql, hq=group * hkv, hkv=hkv, split_override=split, sms=sms, kv=kv)
    i = p.info
    assert i.flat == 1 and i.kernel == pv.KERNEL_TCGEN05
    lo = [b for b in range(len(ctx)) if group * ql[b] <= 48]
    two = kv == pv.KV_FP8_E4M3 and split == 0 and 0 < len(lo) < len(ctx)
    assert i.launches == (2 if two else 1)
    parts = [(p, list(range(len(ctx))))] if not two else [(p, lo), (p.second(), [b for b in range(len(ctx)) if b not in lo])]
    slots, base, units, tiles, splits, n_split = [], 0, 0, 0, 0, 0
    for part, mem in parts:
        c_ctx, c_ql = [ctx[b] for b in mem], [ql[b] for b in mem]
        starts = part.cta_starts()
        T = tc_tile(kv, 128, group * max(c_ql))
        assert part.info.tile_tokens == T
        spans = check_launch(starts, part.info.chunk_tokens, c_ctx, c_ql, hkv, split, sms, kv, group)
        n = len(starts) - 1
        # slot base + c + pair of each CTA's piece of a pair: unique over both launches
        slots += [base + c + k for k, (a, b) in enumerate(spans) for c in range(a, b + 1)]
        base += n + len(spans)
        units, tiles = units + n, tiles + starts[-1]
        splits = max(splits, max(b - a + 1 for a, b in spans))
        n_split += sum(1 for a, b in spans if b > a)
    assert len(slots) == len(set(slots)) and max(slots) < base
    assert i.split_pairs == n_split  # the combine's table lists every split pair of both launches
    assert i.num_units == units and i.total_tiles == tiles
    assert i.max_splits == splits and i.needs_combine == (splits > 1)
    assert i.rows_max == group * max(ql)
    assert i.kv_bytes == sum(ctx) * hkv * (128 * 4 if kv == pv.KV_BF16 else 128 * 2 + 8)
    if two:
        q = p.second()
        assert q.info.launches == 1 and q.second() is None and q.info.workspace_bytes == i.workspace_bytes


@pytest.mark.parametrize("kv", [pv.KV_BF16, pv.KV_FP8_E4M3], ids=["bf16", "fp8"])
@pytest.mark.parametrize("ctx,ql,hkv", CASES)
@pytest.mark.parametrize("split", [0, 1, 4, 1000])
def test_flat_plan_ranges(ctx, ql, hkv, split, kv):
    check_flat_plan(ctx, ql, hkv, split, kv=kv)


def test_flat_plan_ranges_on_random_batches():
    """Seeded random batches (1-64 sequences, lognormal lengths up to 200k, 1-4 KV heads, several SM counts)."""
    rng = np.random.default_rng(2024)
    for _ in range(120):
        B = int(rng.integers(1, 65))
        ql = [int(x) for x in rng.integers(1, 9, B)]
        ctx = [max(q, min(200000, int(np.exp(rng.normal(np.log(6000), 1.3))))) for q in ql]
        hkv = int(rng.choice([1, 2, 4]))
        sms = int(rng.choice([16, 132, 148, 152]))
        check_flat_plan(ctx, ql, hkv, 0, sms=sms, kv=int(rng.choice([pv.KV_BF16, pv.KV_FP8_E4M3])))


def test_flat_plan_does_not_cross_pairs_needlessly():
    # 8 equal pairs of 64 tiles on 16 SMs: two CTAs per pair, no CTA spanning two pairs
    p = mk([8192] * 8, [6] * 8, hq=8, hkv=1, sms=16)
    starts = p.cta_starts()
    assert starts == list(range(0, 8 * 64 + 1, 32))


@pytest.mark.parametrize("ctx,ql,hkv", CASES)
def test_chunk_plan_units_cover_every_token_once(ctx, ql, hkv):
    p = mk(ctx, ql, hq=8 * hkv, hkv=hkv, kernel=pv.KERNEL_WARP_MMA)
    i = p.info
    assert i.flat == 0
    assert i.chunk_tokens % i.tile_tokens == 0
    assert i.num_units == hkv * sum((c + i.chunk_tokens - 1) // i.chunk_tokens for c in ctx)
    assert i.max_splits == max((c + i.chunk_tokens - 1) // i.chunk_tokens for c in ctx)
    assert i.needs_combine == (i.max_splits > 1)
    assert i.kv_bytes == sum(ctx) * hkv * 128 * 4


def test_one_wave_when_possible():
    ctx = [4096 + 997 * i for i in range(8)]
    p = mk(ctx, [6] * 8, hq=32, hkv=4)
    assert p.info.num_units <= 152 * 2


def test_batch_one_gets_the_split_ceiling():
    p1 = mk([1 << 20], [6])
    assert p1.info.max_splits >= 152  # one sequence spreads over every SM
    p2 = mk([1 << 20] * 4, [6] * 4)
    assert p1.info.max_splits > p2.info.max_splits


def test_split_count_monotone_in_context():
    prev = 0
    for L in (64, 1000, 10000, 100000, 1 << 20):
        s = mk([L], [6]).info.max_splits
        assert s >= prev
        prev = s


def test_split_override():
    assert mk([10000], [6], split_override=1).info.max_splits == 1
    assert mk([10000], [6], split_override=4).info.max_splits == 4
    p = mk([10000], [6], split_override=100000)
    assert p.info.chunk_tokens == p.info.tile_tokens


def test_empty_batch_plans():
    p = mk([], [])
    assert p.info.num_units == 0 and p.workspace_bytes >= 0


@pytest.mark.parametrize("kw,status", [
    (dict(ctx=[10], ql=[0]), pv.ERR_INVALID),
    (dict(ctx=[10], ql=[9]), pv.ERR_INVALID),
    (dict(ctx=[3], ql=[6]), pv.ERR_INVALID),
    (dict(ctx=[10], ql=[1], d=96), pv.ERR_UNSUPPORTED),
    (dict(ctx=[10], ql=[1], d=64, kv=pv.KV_FP8_E4M3), pv.ERR_UNSUPPORTED),
    (dict(ctx=[100], ql=[8], hq=32, hkv=1), pv.ERR_UNSUPPORTED),
    (dict(ctx=[100], ql=[2], hq=6, hkv=4), pv.ERR_INVALID),
    (dict(ctx=[100], ql=[2], stride=3), pv.ERR_INVALID),
    (dict(ctx=[10] * 1025, ql=[1] * 1025), pv.ERR_UNSUPPORTED),
    (dict(ctx=[100], ql=[6], d=256, kernel=pv.KERNEL_WARP_MMA), pv.ERR_UNSUPPORTED),  # 256: tcgen05 only
    (dict(ctx=[100], ql=[8], hq=32, hkv=1, d=256), pv.ERR_UNSUPPORTED),  # 256 rows
    (dict(ctx=[100], ql=[6], d=32), pv.ERR_UNSUPPORTED),
    (dict(ctx=[100], ql=[8], hq=32, hkv=1, d=256, kv=pv.KV_FP8_E4M3), pv.ERR_UNSUPPORTED),  # 256 rows
    (dict(ctx=[100], ql=[6], d=256, kv=pv.KV_FP8_E4M3, kernel=pv.KERNEL_WARP_MMA), pv.ERR_UNSUPPORTED),
])
def test_plan_refusals(kw, status):
    with pytest.raises(pv.PaVerifyError) as e:
        mk(**kw)
    assert e.value.status == status
    assert pv.last_error()


@pytest.mark.parametrize("ql,hq", [(6, 8), (1, 8), (8, 8), (2, 16), (4, 16)])
def test_fp8_head_dim_256_plans_on_tensor_cores(ql, hq):
    """FP8 K/V with head_dim 256 (the aiter follow-up's shape: GQA 8 x query 6 = 48 rows) plans on the
    tcgen05 kernel, dynamic plans too; the workspace holds fp32 partials of 256 entries per row."""
    p = mk([150000, 40000], [ql, ql], hq=hq, hkv=1, d=256, kv=pv.KV_FP8_E4M3)
    assert p.info.kernel == pv.KERNEL_TCGEN05 and p.info.flat == 1
    assert p.info.rows_max == ql * hq
    assert p.info.tile_tokens == 128 and p.info.total_tiles == -(-150000 // 128) + -(-40000 // 128)
    q = mk([150000, 40000], [ql, ql], hq=hq, hkv=1, d=128, kv=pv.KV_FP8_E4M3)
    T = tc_tile(pv.KV_FP8_E4M3, 128, ql * hq)
    assert q.info.tile_tokens == T and q.info.total_tiles == -(-150000 // T) + -(-40000 // T)
    assert p.workspace_bytes > q.workspace_bytes
    dyn = pv.plan_dynamic(hq, 1, 256, pv.KV_FP8_E4M3, pv.OUT_BF16, 20000, 9400, 4, 150000, ql, sm_count=152)
    assert dyn.info.kernel == pv.KERNEL_TCGEN05


def test_page_size_must_be_16():
    with pytest.raises(pv.PaVerifyError) as e:
        pv.plan(8, 1, 128, pv.KV_BF16, pv.OUT_F32, 10, 10, [100], [6], sm_count=152, page_size=32)
    assert e.value.status == pv.ERR_UNSUPPORTED


def test_run_refusals_launch_nothing():
    """Argument checks of pa_verify_run happen before any CUDA call."""
    L = pv.lib()
    p = mk([100], [6])
    fake = ctypes.c_void_p(1 << 20)  # aligned, never dereferenced: each call below is refused first
    args = [p.handle] + [fake] * 8 + [ctypes.c_float(0.125), fake, fake, ctypes.c_size_t(p.workspace_bytes), None]
    a = list(args); a[1] = None
    assert L.pa_verify_run(*a) == pv.ERR_INVALID
    a = list(args); a[9] = ctypes.c_float(float("nan"))
    assert L.pa_verify_run(*a) == pv.ERR_INVALID
    a = list(args); a[9] = ctypes.c_float(-1.0)
    assert L.pa_verify_run(*a) == pv.ERR_INVALID
    a = list(args); a[12] = ctypes.c_size_t(p.workspace_bytes - 1)
    assert L.pa_verify_run(*a) == pv.ERR_WORKSPACE
    a = list(args); a[11] = ctypes.c_void_p((1 << 20) + 16)
    assert L.pa_verify_run(*a) == pv.ERR_INVALID  # workspace not 256-byte aligned
    a = list(args); a[2] = ctypes.c_void_p((1 << 20) + 8)
    assert L.pa_verify_run(*a) == pv.ERR_INVALID  # k_cache not 16-byte aligned
    assert L.pa_verify_run(None, *args[1:]) == pv.ERR_INVALID


def test_fp8_run_needs_scales():
    L = pv.lib()
    p = mk([100], [6], kv=pv.KV_FP8_E4M3)
    fake = ctypes.c_void_p(1 << 20)
    a = [p.handle, fake, fake, fake, None, None, fake, fake, fake, ctypes.c_float(0.1), fake, fake,
         ctypes.c_size_t(p.workspace_bytes), None]
    assert L.pa_verify_run(*a) == pv.ERR_INVALID


def test_free_accepts_null():
    pv.lib().pa_verify_free(None)


def test_batches_above_64_sequences_build_their_table_on_the_device():
    rng = np.random.default_rng(3)
    for B in (65, 128, 256, 1024):
        ctx = rng.integers(6, 5000, B).tolist()
        ql = rng.integers(1, 9, B).tolist()
        p = mk(ctx, ql, hq=16, hkv=2, sms=152)
        i = p.info
        assert i.device_table == 1 and i.dynamic == 0
        assert i.num_tokens == sum(ql)
        assert i.kv_bytes == sum(ctx) * 2 * 512
        assert i.rows_max == max(ql) * 8
        assert i.kernel == pv.KERNEL_TCGEN05 and i.flat == 1
        # header, the device table, then partials for one wave of CTAs plus one slot per (sequence, KV head)
        table = 32 + 40 * B
        assert p.workspace_bytes >= 256 + table + (152 + 2 * B) * max(ql) * 8 * 129 * 4
    with pytest.raises(pv.PaVerifyError) as e:
        mk([100] * 65, [6] * 65, split_override=2)
    assert e.value.status == pv.ERR_UNSUPPORTED
    small = mk([100] * 64, [6] * 64)
    assert small.info.device_table == 0


def test_bf16_head_dim_256_plans_on_tensor_cores():
    p = mk([150000, 40000], [6, 6], hq=8, hkv=1, d=256)
    assert p.info.kernel == pv.KERNEL_TCGEN05 and p.info.rows_max == 48
    assert p.info.kv_bytes == 190000 * 1024


@pytest.mark.parametrize("kv,d,ql,hq,T", [(pv.KV_FP8_E4M3, 128, 6, 8, 256), (pv.KV_FP8_E4M3, 128, 8, 8, 128),
                                          (pv.KV_FP8_E4M3, 128, 2, 8, 256), (pv.KV_BF16, 128, 6, 8, 128),
                                          (pv.KV_FP8_E4M3, 256, 6, 8, 128), (pv.KV_BF16, 64, 6, 8, 128)])
def test_tensor_core_tile_sizes(kv, d, ql, hq, T):
    """Static and capacity plans agree on the kernel's tile: 256 tokens for FP8 at head_dim 128 up to 48 rows."""
    assert mk([5000, 300], [ql, ql], hq=hq, d=d, kv=kv).info.tile_tokens == T
    dyn = pv.plan_dynamic(hq, 1, d, kv, pv.OUT_BF16, 20000, 9400, 4, 150000, ql, sm_count=152)
    assert dyn.info.tile_tokens == T


@pytest.mark.parametrize("kv,d,ql,split,launches", [
    (pv.KV_FP8_E4M3, 128, [6, 8, 2], 0, 2),   # FP8 rows 48 / 64 / 16: one launch per class
    (pv.KV_FP8_E4M3, 128, [6, 2, 1], 0, 1),   # every pair up to 48 rows
    (pv.KV_FP8_E4M3, 128, [7, 8, 8], 0, 1),   # every pair above 48 rows
    (pv.KV_FP8_E4M3, 128, [6, 8, 2], 3, 1),   # split_override keeps one launch
    (pv.KV_FP8_E4M3, 256, [6, 8, 2], 0, 1),   # head_dim 256: one instance family
    (pv.KV_BF16, 128, [6, 8, 2], 0, 1),       # bf16: one launch
])
def test_two_launch_plans_only_where_they_apply(kv, d, ql, split, launches):
    p = mk([20000, 9000, 300], ql, hq=8, d=d, kv=kv, split_override=split)
    assert p.info.launches == launches
    assert (p.second() is not None) == (launches == 2)
    if launches == 2:
        q = p.second()
        with pytest.raises(ValueError):  # a view: not runnable on its own, freed with its plan
            pv.run(q, *([None] * 9), 1.0, None, None)
        q.free()
        assert q.handle is None and p.second() is not None
        q = p.second()
        assert p.info.tile_tokens == 256 and q.info.tile_tokens == 128
        assert q.info.rows_max == 64 and p.info.rows_max == 64
        assert p.info.num_units == len(p.cta_starts()) - 1 + q.info.num_units


@pytest.mark.parametrize("kv", [pv.KV_BF16, pv.KV_FP8_E4M3], ids=["bf16", "fp8"])
@pytest.mark.parametrize("ctx,ql", [([30000, 5000, 9000], [8, 5, 2]), ([1 << 17], [7]), ([700, 64, 4000, 129], [6, 8, 3, 5])])
@pytest.mark.parametrize("split", [0, 3])
def test_flat_plan_row_halves(ctx, ql, kv, split):
    """Group 16: pairs of 80-128 rows run as two row halves (virtual pairs) of the 64-row instance."""
    check_flat_plan(ctx, ql, 1, split, kv=kv, group=16)
    assert mk(ctx, ql, hq=16, hkv=1, kv=kv, split_override=split).info.kernel == pv.KERNEL_TCGEN05


def test_row_halves_everywhere():
    # 65-128 rows run on the tensor-core kernel as row halves: static plans (with or without the combine's table)
    # and device-built tables alike; the warp-MMA kernel only when asked for
    assert mk([5000] * 64, [8] * 64, hq=16, hkv=1).info.kernel == pv.KERNEL_TCGEN05
    p = mk([5000] * 40, [8] * 40, hq=64, hkv=4, split_override=4)  # 320 split virtual pairs: no table, the
    assert p.info.kernel == pv.KERNEL_TCGEN05 and p.info.split_pairs == -1  # combine resolves every row itself
    q = mk([5000] * 65, [8] * 65, hq=16, hkv=1)
    assert q.info.kernel == pv.KERNEL_TCGEN05 and q.info.device_table == 1
    assert mk([5000] * 8, [8] * 8, hq=16, hkv=1, kernel=pv.KERNEL_WARP_MMA).info.kernel == pv.KERNEL_WARP_MMA
    dyn = pv.plan_dynamic(16, 1, 128, pv.KV_BF16, pv.OUT_BF16, 20000, 9400, 4, 150000, 8, sm_count=152)
    assert dyn.info.kernel == pv.KERNEL_TCGEN05 and dyn.info.rows_max == 128
