"""The oracle against what the pages and the mathematics fix (CPU only)."""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from paged_kv_speculative_gb300 import synth
from tests import oracle_pins as pins

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def test_e4m3_decoder_matches_library_for_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    mine = oracle.decode_e4m3(codes)
    lib = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).double().numpy()
    assert np.array_equal(np.isnan(mine), np.isnan(lib))
    ok = ~np.isnan(lib)
    assert np.array_equal(mine[ok], lib[ok])
    assert np.array_equal(np.signbit(mine[ok]), np.signbit(lib[ok]))


def test_e4m3_decoder_matches_ocp_golden_values():
    rows = []
    with open(os.path.join(GOLDEN, "e4m3_ocp_values.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                code, val = line.split()[:2]
                rows.append((int(code, 16), float(val)))
    assert len(rows) == 10
    for code, val in rows:
        got = oracle.decode_e4m3([code])[0]
        if math.isnan(val):
            assert math.isnan(got)
        else:
            assert got == val and math.copysign(1, got) == math.copysign(1, val), hex(code)


def test_bf16_decoder_matches_library_for_all_codes():
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    mine = oracle.decode_bf16(codes)
    lib = torch.from_numpy(codes.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    assert np.array_equal(np.isnan(mine), np.isnan(lib))
    ok = ~np.isnan(lib)
    assert np.array_equal(mine[ok], lib[ok])


@pytest.mark.parametrize("idx", range(4))
def test_oracle_equals_dense_brute_force(idx):
    p = pins.tiny_problems()[idx]
    ok, det = pins.pin_brute_force(p)
    assert ok, det


@pytest.mark.parametrize("kvd", [synth.KV_BF16, synth.KV_FP8])
def test_query_length_one_is_ordinary_decode(kvd):
    ok, det = pins.pin_sdpa_decode(pins.decode_problem(kvd))
    assert ok, det


@pytest.mark.parametrize("idx", range(2))
def test_draft_row_equals_prefix_decode(idx):
    ok, det = pins.pin_causal_prefix(pins.tiny_problems()[idx])
    assert ok, det


@pytest.mark.parametrize("idx", range(4))
def test_block_table_permutation_invariance(idx):
    ok, det = pins.pin_page_permutation(pins.tiny_problems()[idx])
    assert ok, det


def test_contiguous_layout_equals_scattered_layout():
    a = synth.make_problem([40, 77], [6, 3], 4, 1, 64, seed=5, contiguous=True, poison=False)
    b = pins.permute_pool(a, seed=9)
    assert np.array_equal(oracle.verify_attention(a), oracle.verify_attention(b))


@pytest.mark.parametrize("idx", range(2))
def test_closed_forms(idx):
    ok, det = pins.pin_closed_forms(pins.tiny_problems()[idx])
    assert ok, det


def test_fp8_equals_attention_on_dequantised_tensors():
    p = synth.make_problem([45, 29], [6, 2], 4, 2, 64, kv_dtype=synth.KV_FP8, seed=12)
    ok, det = pins.pin_brute_force(p)
    assert ok, det


def test_fp8_head_dim_256_against_pins():
    """The head-256 FP8 shape (GQA 8 over one KV head, the aiter follow-up's): brute force on the dequantised tensors,
    ordinary decode at query length 1, and block-table permutation invariance."""
    p = synth.make_problem([45, 20], [6, 3], 8, 1, 256, kv_dtype=synth.KV_FP8, seed=14)
    for pin in (pins.pin_brute_force, pins.pin_page_permutation):
        ok, det = pin(p)
        assert ok, det
    d = synth.make_problem([23, 50, 8], [1, 1, 1], 8, 1, 256, kv_dtype=synth.KV_FP8, seed=22)
    ok, det = pins.pin_sdpa_decode(d)
    assert ok, det


def test_poisoned_slots_are_never_read():
    p = synth.make_config("tiny")
    out = oracle.verify_attention(p)
    assert np.isfinite(out).all()


def test_row_selection_matches_full_result():
    p = synth.make_config("tiny")
    full = oracle.verify_attention(p)
    rows = np.array([[0, 3], [5, 1], [6, 0]])
    sel = oracle.verify_attention(p, rows=rows)
    for k, (t, h) in enumerate(rows):
        assert np.array_equal(sel[k], full[t, h])


def test_thread_count_does_not_change_result():
    p = synth.make_problem([300, 41], [6, 6], 8, 2, 64, seed=3)
    assert np.array_equal(oracle.verify_attention(p, threads=1), oracle.verify_attention(p, threads=5))


@pytest.mark.parametrize("mutant", [1, 2, 3, 4, 5, 6])
def test_pins_catch_a_planted_mistake(mutant):
    """Each build with one planted mistake fails at least one pin."""
    res = pins.run_battery(mutant)
    failed = [name for name, ok, _ in res if not ok]
    assert failed, f"mutant {mutant} passed every pin"


def test_unmutated_oracle_passes_every_pin():
    res = pins.run_battery(0)
    bad = [(n, d) for n, ok, d in res if not ok]
    assert not bad, bad
