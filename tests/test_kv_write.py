"""Paged KV write with per-token FP8 quantisation: oracle pins (CPU) and the
CUDA kernel against the oracle, bit for bit (GPU)."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_speculative_gb300 import synth


def bf16_bits(x: torch.Tensor) -> np.ndarray:
    return x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def new_rows(n, hkv, d, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    k = bf16_bits(torch.randn((n, hkv, d), generator=g) * scale)
    v = bf16_bits(torch.randn((n, hkv, d), generator=g) * scale)
    return k, v


def empty_cache(n_pg, hkv, d, kvd):
    dt = np.uint16 if kvd == synth.KV_BF16 else np.uint8
    kc = np.full((n_pg, hkv, 16, d), 0x55, dtype=dt)
    vc = np.full((n_pg, hkv, 16, d), 0x33, dtype=dt)
    ks = vs = None
    if kvd == synth.KV_FP8:
        ks = np.full((n_pg, hkv, 16), -7.0, dtype=np.float32)
        vs = np.full((n_pg, hkv, 16), -7.0, dtype=np.float32)
    return kc, vc, ks, vs


def slots_for(n, n_pg, seed, dead=0.25):
    rng = np.random.default_rng(seed)
    s = rng.choice(n_pg * 16, size=n, replace=False).astype(np.int64)
    s[rng.random(n) < dead] = -1
    return s


# ------------------------------------------------------------------ CPU pins
def test_encoder_matches_library_rne():
    x = np.concatenate([np.linspace(-448, 448, 50001), np.linspace(-0.03, 0.03, 30001),
                        2.0 ** np.arange(-12, 8.8, 0.125)]).astype(np.float32)
    assert np.abs(x).max() <= 448.0  # torch's cast does not saturate: compare inside the range
    mine = oracle.encode_e4m3(x)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(mine, ref)


def test_encoder_saturates_and_keeps_nan():
    assert oracle.encode_e4m3([1e6, -1e6, 449.0, 464.0])[0] == 0x7E
    assert oracle.encode_e4m3([-1e6])[0] == 0xFE
    assert oracle.encode_e4m3([float("nan")])[0] == 0x7F


def test_quantiser_matches_the_generator_path():
    """On bf16-representable rows the oracle's quantiser gives the bytes of the
    torch-based quantiser the input generator uses (library division + RNE cast)."""
    k, v = new_rows(40, 2, 128, seed=1, scale=3.0)
    slots = np.arange(40, dtype=np.int64)
    kc, vc, ks, vs = empty_cache(3, 2, 128, synth.KV_FP8)
    assert oracle.kv_write(k, v, slots, kc, vc, ks, vs, synth.KV_FP8) == 0
    x = torch.from_numpy(k.view(np.int16).copy()).view(torch.bfloat16).float()  # [40, 2, 128]
    q8, s = synth._quantise_e4m3(x)
    page, off = slots // 16, slots % 16
    for t in range(40):
        assert np.array_equal(kc[page[t], :, off[t]], q8[t])
        assert np.array_equal(ks[page[t], :, off[t]], s[t])


def test_row_max_maps_to_448_and_dead_slots_write_nothing():
    k, v = new_rows(64, 1, 64, seed=2)
    slots = slots_for(64, 8, seed=3)
    kc, vc, ks, vs = empty_cache(8, 1, 64, synth.KV_FP8)
    kc0 = kc.copy()
    oracle.kv_write(k, v, slots, kc, vc, ks, vs, synth.KV_FP8)
    written = np.zeros((8, 16), dtype=bool)
    for t, sl in enumerate(slots):
        if sl >= 0:
            written[sl // 16, sl % 16] = True
            assert (kc[sl // 16, 0, sl % 16] & 0x7F).max() == 0x7E
            deq = oracle.decode_e4m3(kc[sl // 16, 0, sl % 16]) * ks[sl // 16, 0, sl % 16]
            x = torch.from_numpy(k[t, 0].view(np.int16).copy()).view(torch.bfloat16).double().numpy()
            assert np.all(np.abs(deq - x) <= np.abs(x) * 2.0 ** -4 + ks[sl // 16, 0, sl % 16] * 2.0 ** -10)
    assert np.array_equal(kc[:, 0][~written], kc0[:, 0][~written])
    assert (ks[:, 0][~written] == -7.0).all()


def test_bf16_write_is_a_copy():
    k, v = new_rows(10, 2, 128, seed=4)
    slots = np.arange(10, dtype=np.int64) * 3
    kc, vc, _, _ = empty_cache(2, 2, 128, synth.KV_BF16)
    oracle.kv_write(k, v, slots, kc, vc, None, None, synth.KV_BF16)
    for t, sl in enumerate(slots):
        assert np.array_equal(kc[sl // 16, :, sl % 16], k[t])
        assert np.array_equal(vc[sl // 16, :, sl % 16], v[t])


def test_out_of_range_slot_is_reported():
    k, v = new_rows(2, 1, 64, seed=5)
    kc, vc, ks, vs = empty_cache(1, 1, 64, synth.KV_FP8)
    assert oracle.kv_write(k, v, np.array([3, 16], dtype=np.int64), kc, vc, ks, vs, synth.KV_FP8) == -1


# ------------------------------------------------------------------ GPU parity
@pytest.mark.gpu
@pytest.mark.parametrize("kvd", [synth.KV_BF16, synth.KV_FP8])
@pytest.mark.parametrize("d", [64, 128, 256])
def test_gpu_kv_write_bit_exact(kvd, d):
    from paged_kv_speculative_gb300 import _build, pa_verify as pv
    _build.build()
    n, hkv, n_pg = 300, 4, 64
    k, v = new_rows(n, hkv, d, seed=10 + d, scale=2.5)
    k[0, 0, :] = 0  # an all-zero row: scale 1
    slots = slots_for(n, n_pg, seed=11)
    kc, vc, ks, vs = empty_cache(n_pg, hkv, d, kvd)
    dev = lambda a: None if a is None else torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).cuda()
    dkc, dvc, dks, dvs = dev(kc), dev(vc), dev(ks), dev(vs)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pv.kv_write(dev(k).view(torch.bfloat16), dev(v).view(torch.bfloat16), torch.from_numpy(slots).cuda(), dkc, dvc,
                dks, dvs, kvd, error_flags=err)
    torch.cuda.synchronize()
    oracle.kv_write(k, v, slots, kc, vc, ks, vs, kvd)
    assert int(err.item()) == 0
    back = lambda t, like: t.cpu().numpy().view(like.dtype)
    assert np.array_equal(back(dkc, kc), kc)
    assert np.array_equal(back(dvc, vc), vc)
    if kvd == synth.KV_FP8:
        assert np.array_equal(dks.cpu().numpy(), ks)
        assert np.array_equal(dvs.cpu().numpy(), vs)


@pytest.mark.gpu
def test_gpu_kv_write_then_verify_matches_oracle():
    """Write the verify tokens' K/V, then attend: the two steps compose."""
    from paged_kv_speculative_gb300 import _build, pa_verify as pv
    from paged_kv_speculative_gb300.device_inputs import to_device
    _build.build()
    prob = synth.make_problem([200, 90], [6, 4], 8, 2, 128, kv_dtype=synth.KV_FP8, seed=77, poison=False)
    # overwrite the verify tokens' rows with fresh values through the write path
    k, v = new_rows(10, 2, 128, seed=78)
    slots = []
    for b, (L, q) in enumerate(zip(prob.context_lens, prob.query_lens)):
        for t in range(L - q, L):
            slots.append(int(prob.block_table[b, t // 16]) * 16 + t % 16)
    slots = np.array(slots, dtype=np.int64)
    dp = to_device(prob)
    pv.kv_write(torch.from_numpy(k.view(np.int16)).cuda().view(torch.bfloat16),
                torch.from_numpy(v.view(np.int16)).cuda().view(torch.bfloat16), torch.from_numpy(slots).cuda(),
                dp.k_cache, dp.v_cache, dp.k_scale, dp.v_scale, synth.KV_FP8)
    oracle.kv_write(k, v, slots, prob.k_cache, prob.v_cache, prob.k_scale, prob.v_scale, synth.KV_FP8)
    va = pv.VerifyAttention(8, 2, 128, synth.KV_FP8, prob.num_pages, prob.block_table.shape[1], [200, 90], [6, 4])
    out = va(*dp.args(), prob.softmax_scale)
    ref = oracle.verify_attention(prob)
    assert float(np.abs(out.cpu().numpy() - ref).max()) <= 2e-2
