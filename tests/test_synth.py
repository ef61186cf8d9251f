"""The seeded input generator: determinism, layout, poison, workload shapes."""
import numpy as np
import pytest

from paged_kv_speculative_gb300 import synth


def test_same_seed_same_bytes():
    a = synth.make_problem([50, 20], [6, 2], 4, 1, 64, seed=7)
    b = synth.make_problem([50, 20], [6, 2], 4, 1, 64, seed=7)
    for f in ("q", "k_cache", "v_cache", "block_table"):
        assert np.array_equal(getattr(a, f), getattr(b, f))


def test_pages_are_disjoint_and_in_range():
    p = synth.make_problem([100, 33, 16, 1], [6, 6, 1, 1], 4, 2, 64, seed=1)
    used = []
    for b in range(p.num_seqs):
        npg = (int(p.context_lens[b]) + 15) // 16
        row = p.block_table[b]
        assert (row[:npg] >= 0).all() and (row[:npg] < p.num_pages).all()
        assert (row[npg:] == -1).all()
        used += row[:npg].tolist()
    assert len(used) == len(set(used))


def test_poison_marks_unused_slots_and_pages():
    p = synth.make_problem([20], [2], 2, 1, 64, seed=2, extra_pages=3)
    pg_last = p.block_table[0, 1]
    assert (p.k_cache[pg_last, :, 4:] == synth.BF16_NAN).all()
    assert (p.k_cache[pg_last, :, :4] != synth.BF16_NAN).any()
    used = set(p.block_table[0, :2].tolist())
    for pg in range(p.num_pages):
        if pg not in used:
            assert (p.v_cache[pg] == synth.BF16_NAN).all()


def test_fp8_quantisation_scales():
    p = synth.make_problem([32], [1], 2, 1, 64, kv_dtype=synth.KV_FP8, seed=4, poison=False)
    assert p.k_cache.dtype == np.uint8 and p.k_scale.shape == (p.num_pages, 1, 16)
    # every (token, head) row reaches the E4M3 maximum 448 in magnitude (code 0x7E / 0xFE)
    mag = p.k_cache & 0x7F
    assert (mag.max(axis=-1) == 0x7E).all()
    assert (p.k_scale > 0).all()


@pytest.mark.parametrize("name", synth.ALL_NAMES)
def test_workload_shapes(name):
    ctx, ql, hq, hkv, d, kvd, seed = synth.config_lengths(name)
    assert len(ctx) == len(ql)
    assert all(1 <= q <= 8 for q in ql)
    assert all(q <= c for q, c in zip(ql, ctx))
    if name == "tiny":
        assert ctx == [37, 100] and ql == [1, 6] and (hq, hkv, d) == (4, 1, 64)
    if name == "mtp5_bf16":
        assert len(ctx) == 8 and all(4096 <= c <= 32768 for c in ctx) and (hq, hkv, d) == (32, 4, 128)
    if name == "mtp5_fp8":
        assert ctx == [131072] * 4 and kvd == synth.KV_FP8
    if name == "mixed_fp8":
        assert len(ctx) == 64 and max(ctx) <= 131072 and (hq, hkv) == (16, 2)
    if name == "ctx1mi_bf16":
        assert ctx == [1 << 20] and (ctx[0] + 15) // 16 == 65536
    if name in synth.EXTRA_NAMES:
        kv = synth.KV_BF16 if "bf16" in name else synth.KV_FP8
        assert set(ctx) == {150000} and set(ql) == {6} and (hq, hkv, d, kvd) == (8, 1, 256, kv)
        assert len(ctx) == int(name[-1]) and ql[0] * hq // hkv == 48


def test_tiny_uses_a_32_page_pool():
    p = synth.make_config("tiny")
    assert p.num_pages == 32 and p.kv_bytes == (37 + 100) * 64 * 2 * 2


def test_shard_sequences_cover_batch():
    for n in (1, 7, 64):
        for w in (1, 2, 3, 8):
            parts = [synth.shard_sequences(n, w, r) for r in range(w)]
            allx = np.concatenate(parts)
            assert np.array_equal(np.sort(allx), np.arange(n))


def test_bench_describes_every_workload():
    import bench
    assert set(synth.ALL_NAMES) <= set(bench.WORKLOAD_DESC)
