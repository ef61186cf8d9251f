"""Model of the hand-offs inside the tcgen05 split kernel, checked for deadlock.

Each role of a CTA (K producer, V producer, MMA issuer, softmax warpgroups) is a
sequence of steps that wait for events and then post events, written in the
order the kernel takes them. The model runs the roles until every one has
finished or none can move. The kernel's MMA order (S(j+2) before PV(j), except
that a segment's first S goes after PV(j)) must finish for every layout of
segments; the plain order S(j+2)-before-PV(j) must get stuck on some layouts
(a segment of a single tile), which shows that the model can tell them apart.
"""
import random

import pytest


# ring depths (K, V) of the kernel's instances: bf16 head_dim 128; FP8 head_dim 128; FP8 head_dim 256
DEPTHS = {False: [(2, 3)], True: [(5, 5), (2, 2)]}


def run(seg_first, short_tile, fp8, slow, kernel_order=True, depths=None):
    n = len(seg_first)
    KS, VS = depths or DEPTHS[fp8][0]
    seg_last = [i == n - 1 or seg_first[i + 1] for i in range(n)]
    seg_of, s = [], -1
    for i in range(n):
        s += seg_first[i]
        seg_of.append(s)
    ev = set()

    def producer(kind, depth):
        for k in range(n):
            if k >= depth:  # the ring slot frees when S (K ring) or PV (V ring) of tile k - depth is done
                yield lambda k=k: (("S" if kind == "K" else "PV"), k - depth) in ev
            ev.add((kind + "full", k))

    def issuer():
        def S(i):
            return (lambda: ((not seg_first[i]) or ("qready", seg_of[i]) in ev) and ("Kfull", i) in ev
                    and (i < 2 or ("sfree", i - 2) in ev)), ("S", i)

        def PV(j):
            return (lambda: ("Vfull", j) in ev and ("pfull", j) in ev), ("PV", j)

        ops = [S(i) for i in range(min(2, n))]
        for j in range(n):
            nxt = j + 2 < n
            late = kernel_order and nxt and seg_first[j + 2]
            if nxt and not late:
                ops.append(S(j + 2))
            ops.append(PV(j))
            if late:
                ops.append(S(j + 2))
        for cond, e in ops:
            yield cond
            ev.add(e)

    def softmax():
        ev.add(("qready", 0))
        for i in range(n):
            yield lambda i=i: ("S", i) in ev
            ev.add(("sfree", i))
            if seg_last[i] and i + 1 < n:
                ev.add(("qready", seg_of[i] + 1))  # the next segment's Q, staged once S(i) is done
            if fp8:
                yield lambda i=i: ("Vfull", i) in ev  # scales ride in the V stage
            if slow[i] and not seg_first[i]:
                yield lambda i=i: ("PV", i - 1) in ev  # O rescale
            if i >= 2:
                yield lambda i=i: ("PV", i - 2) in ev  # P buffer reuse
            if short_tile[i] and not fp8:
                yield lambda i=i: ("Vfull", i) in ev  # zero the rows past the pair
            ev.add(("pfull", i))
            if seg_last[i]:
                yield lambda i=i: ("PV", i) in ev  # segment epilogue reads O

    roles = [producer("K", KS), producer("V", VS), issuer(), softmax()]
    pending = [None] * 4
    alive = [True] * 4
    while any(alive):
        moved = False
        for r in range(4):
            while alive[r]:
                if pending[r] is None:
                    moved = True
                    try:
                        pending[r] = next(roles[r])
                    except StopIteration:
                        alive[r] = False
                        break
                if pending[r]():
                    pending[r] = None
                    moved = True
                else:
                    break
        if not moved:
            return False
    return True


def layouts(count, seed):
    rng = random.Random(seed)
    for _ in range(count):
        n = rng.randint(1, 12)
        fp8 = rng.random() < 0.5
        yield ([True] + [rng.random() < 0.4 for _ in range(n - 1)], [rng.random() < 0.3 for _ in range(n)], fp8,
               [rng.random() < 0.3 for _ in range(n)])


def test_kernel_order_never_sticks():
    for seg_first, short, fp8, slow in layouts(4000, 1):
        for dep in DEPTHS[fp8]:
            assert run(seg_first, short, fp8, slow, depths=dep), (seg_first, short, fp8, slow, dep)


def test_plain_order_sticks_on_one_tile_segments():
    stuck = [lay for lay in layouts(4000, 1) if not run(*lay, kernel_order=False)]
    assert stuck
    # every stuck layout has a one-tile segment followed by another segment
    for seg_first, _, _, _ in stuck:
        n = len(seg_first)
        assert any(seg_first[j] and j + 1 < n and seg_first[j + 1] for j in range(n))


@pytest.mark.parametrize("fp8,dep", [(False, (2, 3)), (True, (5, 5)), (True, (2, 2))])
def test_single_tile_segments_back_to_back(fp8, dep):
    n = 9
    assert run([True] * n, [True] * n, fp8, [True] * n, depths=dep)
    assert not run([True] * n, [True] * n, fp8, [True] * n, kernel_order=False, depths=dep)
