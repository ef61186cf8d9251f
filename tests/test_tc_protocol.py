"""Model of the hand-offs inside the tcgen05 split kernel, checked for deadlock
and for the phase discipline of its mbarrier waits.

Each role of a CTA (K producer, V producer, MMA issuer, softmax warpgroups) is a
sequence of steps that wait for events and then post events, written in the
order the kernel takes them. An event is (kind, tile) and is posted on the
barrier slot tile % R of a ring of R barriers; a wait on it is a parity wait
on that slot. Such a wait is only sound if, when it starts, the slot has
completed the tile's previous phase (tile - R) and not yet the next one (tile +
R): otherwise the parity matches the wrong phase. The model runs the roles
until every one has finished or none can move, and records every unsound wait.

Checked: the kernel's MMA order (S(j+2) before PV(j), except that a segment's
first S goes after PV(j)) finishes for every layout of segments and makes no
unsound wait, for each instance's ring depths; the plain order
S(j+2)-before-PV(j) gets stuck on some layouts (a segment of a single tile),
which shows that the model tells them apart. The FP8 scale ring (KS + 2 slots,
refilled by the K producer without a wait of its own) never overwrites a slot
whose scales the softmax has not read; one slot fewer would. With three P
buffers and a two-deep V ring, the V slot of a short tile can still be a phase
behind when the softmax gets there, so its parity wait would be unsound; the
kernel first waits for PV of the slot's previous tile (waiting for that tile's
own V phase instead would be unsound too: the slot may already be past it).
"""
import random

import pytest

# (K ring, V ring, P buffers, FP8) of the kernel's instances
# (FP8 at head_dim 128: 256-token tiles up to 48 rows, 128-token tiles in the 64-row instance)
INSTANCES = {"bf16_d128": (2, 3, 2, False), "fp8_d128": (2, 2, 2, True), "fp8_d128_r64": (5, 5, 2, True),
             "fp8_d256": (2, 2, 3, True), "bf16_d64": (5, 5, 2, False), "bf16_d256": (1, 1, 3, False)}


def run(seg_first, short_tile, slow, ks, vs, pb, fp8, kernel_order=True, scale_slack=2, short_wait="pv", sched=None):
    """Returns (finished, unsound waits, scale-slot overwrites). Without `sched` each role runs as far as it
    can in turn (producers furthest ahead); with a random.Random, the roles take turns in random order and
    each moves a random number of steps, so producers may also lag."""
    n = len(seg_first)
    ss = ks + scale_slack
    seg_last = [i == n - 1 or seg_first[i + 1] for i in range(n)]
    seg_of, s = [], -1
    for i in range(n):
        s += seg_first[i]
        seg_of.append(s)
    ev = set()
    unsound, overwritten = [], []

    def producer(kind, depth):
        for k in range(n):
            if k >= depth:  # the slot frees when S (K ring) or PV (V ring) of tile k - depth is done
                yield ("S" if kind == "K" else "PV", k - depth, depth)
            if fp8 and kind == "K" and k >= ss and ("sread", k - ss) not in ev:
                overwritten.append(k)
            ev.add((kind + "full", k))
            if fp8 and kind == "K":
                ev.add(("SCfull", k))

    def issuer():
        def S(i):
            if seg_first[i]:
                yield ("qready", seg_of[i], 1)
            yield ("Kfull", i, ks)
            if i >= 2:
                yield ("sfree", i - 2, 2)
            ev.add(("S", i))

        def PV(j):
            yield ("Vfull", j, vs)
            yield ("pfull", j, pb)
            ev.add(("PV", j))

        for i in range(min(2, n)):
            yield from S(i)
        for j in range(n):
            nxt = j + 2 < n
            late = kernel_order and nxt and seg_first[j + 2]
            if nxt and not late:
                yield from S(j + 2)
            yield from PV(j)
            if late:
                yield from S(j + 2)

    def softmax():
        ev.add(("qready", 0))
        for i in range(n):
            yield ("S", i, 2)  # sfull
            if fp8:
                yield ("SCfull", i, ss)  # the tile's scales, read before S is released
                ev.add(("sread", i))
            ev.add(("sfree", i))
            if seg_last[i] and i + 1 < n:
                ev.add(("qready", seg_of[i] + 1))  # the next segment's Q, staged once S(i) is done
            if slow[i] and not seg_first[i]:
                yield ("PV", i - 1, pb)  # O rescale
            if i >= pb:
                yield ("PV", i - pb, pb)  # P buffer reuse
            if short_tile[i]:  # zero the rows past the pair in the V slot
                if short_wait == "pv" and vs < pb and i >= vs:
                    yield ("PV", i - vs, pb)  # the kernel's way
                if short_wait == "prev_v" and i >= vs:
                    yield ("Vfull", i - vs, vs)
                yield ("Vfull", i, vs)
            ev.add(("pfull", i))
            if seg_last[i]:
                yield ("PV", i, pb)  # segment epilogue reads O

    roles = [producer("K", ks), producer("V", vs), issuer(), softmax()]
    pending = [None] * 4
    alive = [True] * 4
    while any(alive):
        moved = False
        order = sched.sample(range(4), 4) if sched else range(4)
        for r in order:
            budget = sched.randint(1, 3) if sched else None
            while alive[r] and (budget is None or budget > 0):
                if budget is not None:
                    budget -= 1
                if pending[r] is None:
                    moved = True
                    try:
                        pending[r] = next(roles[r])
                    except StopIteration:
                        alive[r] = False
                        break
                    kind, t, ring = pending[r]
                    if (t - ring >= 0 and (kind, t - ring) not in ev) or (kind, t + ring) in ev:
                        unsound.append((r, kind, t))
                kind, t, _ = pending[r]
                if (kind, t) in ev:
                    pending[r] = None
                    moved = True
                else:
                    break
        if not moved:
            return False, unsound, overwritten
    return True, unsound, overwritten


def layouts(count, seed):
    rng = random.Random(seed)
    for _ in range(count):
        n = rng.randint(1, 12)
        yield ([True] + [rng.random() < 0.4 for _ in range(n - 1)], [rng.random() < 0.3 for _ in range(n)],
               [rng.random() < 0.3 for _ in range(n)])


@pytest.mark.parametrize("inst", list(INSTANCES))
def test_kernel_order_never_sticks_and_waits_soundly(inst):
    ks, vs, pb, fp8 = INSTANCES[inst]
    for lay in layouts(4000, 1):
        done, unsound, over = run(*lay, ks, vs, pb, fp8)
        assert done and not unsound and not over, (lay, unsound, over)


@pytest.mark.parametrize("inst", list(INSTANCES))
def test_random_schedules_wait_soundly(inst):
    ks, vs, pb, fp8 = INSTANCES[inst]
    sched = random.Random(7)
    for lay in layouts(1500, 4):
        for _ in range(3):
            done, unsound, over = run(*lay, ks, vs, pb, fp8, sched=sched)
            assert done and not unsound and not over, (lay, unsound, over)


@pytest.mark.parametrize("inst", list(INSTANCES))
def test_plain_order_sticks_on_one_tile_segments(inst):
    ks, vs, pb, fp8 = INSTANCES[inst]
    stuck = [lay for lay in layouts(4000, 1) if not run(*lay, ks, vs, pb, fp8, kernel_order=False)[0]]
    assert stuck
    # every stuck layout has a one-tile segment followed by another segment
    for seg_first, _, _ in stuck:
        n = len(seg_first)
        assert any(seg_first[j] and j + 1 < n and seg_first[j + 1] for j in range(n))


@pytest.mark.parametrize("inst", list(INSTANCES))
def test_single_tile_segments_back_to_back(inst):
    ks, vs, pb, fp8 = INSTANCES[inst]
    n = 9
    assert run([True] * n, [True] * n, [True] * n, ks, vs, pb, fp8)[0]
    assert not run([True] * n, [True] * n, [True] * n, ks, vs, pb, fp8, kernel_order=False)[0]


def test_a_shallower_scale_ring_would_be_overwritten():
    for inst in ("fp8_d128", "fp8_d256"):
        ks, vs, pb, fp8 = INSTANCES[inst]
        assert any(run(*lay, ks, vs, pb, fp8, scale_slack=1)[2] for lay in layouts(500, 2)), inst


@pytest.mark.parametrize("other", ["none", "prev_v"])
def test_short_tile_waits_for_pv_of_the_slots_previous_tile(other):
    ks, vs, pb, fp8 = INSTANCES["fp8_d256"]
    bad = [lay for lay in layouts(2000, 3) if run(*lay, ks, vs, pb, fp8, short_wait=other)[1]]
    assert bad  # a single parity wait meets the slot a phase behind; a wait on the previous phase, a phase ahead
    for lay in bad:
        assert run(*lay, ks, vs, pb, fp8)[0:2] == (True, [])
