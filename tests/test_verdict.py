"""Greedy verify verdict: oracle pins (CPU) and the CUDA kernels against the
oracle, bit for bit (GPU)."""
import numpy as np
import pytest
import torch

import oracle


def bf16(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def make_case(qlens, vocab, seed, accept_prob=0.7, ties=False):
    rng = np.random.default_rng(seed)
    T = int(sum(qlens))
    x = rng.standard_normal((T, vocab)).astype(np.float32) * 3
    if ties:  # coarse values: many exact ties of the maximum
        x = np.round(x)
    lg = bf16(x)
    vals = torch.from_numpy(lg.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    picks = np.argmax(vals, axis=1)
    ids = np.empty(T, dtype=np.int32)
    off = 0
    for q in qlens:
        ids[off] = rng.integers(vocab)
        for i in range(1, q):  # draft i matches the target's pick at i-1 with probability accept_prob
            ids[off + i] = picks[off + i - 1] if rng.random() < accept_prob else (picks[off + i - 1] + 1) % vocab
        off += q
    return np.array(qlens, dtype=np.int32), lg, ids, vals


def numpy_verdict(qlens, vals, ids):
    tgt = np.argmax(vals, axis=1).astype(np.int32)  # first occurrence of the maximum; NaN wins
    acc, nxt, off = [], [], 0
    for q in qlens:
        a = 0
        while a < q - 1 and ids[off + a + 1] == tgt[off + a]:
            a += 1
        acc.append(a)
        nxt.append(tgt[off + a])
        off += q
    return tgt, np.array(acc), np.array(nxt)


@pytest.mark.parametrize("ties", [False, True])
def test_oracle_matches_numpy_argmax_rule(ties):
    ql, lg, ids, vals = make_case([6, 1, 8, 3, 6], 1000, seed=1, ties=ties)
    got = oracle.greedy_verdict(ql, lg, ids)
    ref = numpy_verdict(ql, vals, ids)
    for a, b in zip(got, ref):
        assert np.array_equal(a, b)


def test_oracle_nan_and_signed_zero():
    lg = bf16(np.array([[0.0, -0.0, -1.0], [-0.0, 0.0, -1.0], [1.0, np.nan, 5.0]], dtype=np.float32))
    tgt, acc, nxt = oracle.greedy_verdict(np.array([3]), lg, np.array([7, 0, 0], dtype=np.int32))
    assert tgt.tolist() == [0, 0, 1]
    assert acc[0] == 2 and nxt[0] == 1


def test_all_drafts_accepted_and_none_accepted():
    ql, lg, ids, vals = make_case([6, 6], 500, seed=2, accept_prob=1.0)
    _, acc, _ = oracle.greedy_verdict(ql, lg, ids)
    assert acc.tolist() == [5, 5]
    ql, lg, ids, vals = make_case([6, 6], 500, seed=3, accept_prob=0.0)
    _, acc, _ = oracle.greedy_verdict(ql, lg, ids)
    assert acc.tolist() == [0, 0]


@pytest.mark.gpu
@pytest.mark.parametrize("vocab", [7, 8192, 8193, 151936])
@pytest.mark.parametrize("ties", [False, True])
def test_gpu_verdict_bit_exact(vocab, ties):
    from paged_kv_speculative_gb300 import _build, pa_verify as pv
    _build.build()
    ql, lg, ids, _ = make_case([6, 1, 8, 3, 6, 2, 4, 6], vocab, seed=vocab + ties, ties=ties)
    if vocab > 100:
        lg[3, vocab // 2] = 0x7FC0  # a NaN row maximum
    ref = oracle.greedy_verdict(ql, lg, ids)
    d_lg = torch.from_numpy(lg.view(np.int16)).cuda().view(torch.bfloat16)
    tgt, acc, nxt = pv.greedy_verdict(d_lg, torch.from_numpy(ids).cuda(), torch.from_numpy(ql).cuda())
    torch.cuda.synchronize()
    for a, b in zip((tgt, acc, nxt), ref):
        assert np.array_equal(a.cpu().numpy(), b)
