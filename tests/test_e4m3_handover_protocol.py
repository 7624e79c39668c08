"""CPU model of the e4m3 decode kernel's softmax hand-over (mla_decode_e4m3_sm103a.cu).

The kernel's eight softmax warps ping-pong: warp (par, quad) takes the tiles j with
j % 2 == par of lane quadrant quad.  Each tile's running max goes to the other parity's warp
of the quadrant through a named barrier (bar.arrive by the sender, bar.sync by the
receiver), and named barriers have no timeout.  So the order of operations per tile is
modelled here and every combination of failing waits is run:

    fail = draining or a bounded wait of this tile failed
    if j >= 1:     receive the hand-over of tile j-1; a stop mark ends the warp
    if j + 1 < n:  hand over tile j, marked stop when draining
    if draining:   end the warp
    parity barrier (the 4 warps of the parity) ORs fail -> draining from the next tile on

Checked: nothing waits forever; no hand-over is sent while the previous one on the same
barrier is unreceived; every hand-over is received; the four warps of a parity leave at
the same tile (so the kernel's 128-thread parity barriers always see all four).
"""
import itertools
import random

import pytest


def _run(n, fail_at):
    warps = [(p, q) for p in range(2) for q in range(4)]
    st = {w: dict(j=w[0], ph=0, draining=False, fail=False, done=False, exit=None) for w in warps}
    arrives, syncs, stop = {}, {}, {}
    parity_bar = {0: {}, 1: {}}
    bar_index = {w: 0 for w in warps}
    progress = True
    while progress:
        progress = False
        for w in warps:
            s = st[w]
            if s["done"]:
                continue
            p, q = w
            j = s["j"]
            if j >= n:
                s.update(done=True, exit=("end", j))
                progress = True
                continue
            if s["ph"] == 0:  # this tile's bounded waits
                s["fail"] = s["draining"] or (fail_at[w] is not None and j >= fail_at[w])
                s["ph"] = 1
            elif s["ph"] == 1:  # receive tile j-1's hand-over
                if j >= 1:
                    bar = (q, p ^ 1)
                    if syncs.get(bar, 0) + 1 > arrives.get(bar, 0):
                        continue  # waits for the sender
                    syncs[bar] = syncs.get(bar, 0) + 1
                    if stop.get((p ^ 1, q), False):
                        s.update(done=True, exit=("stop", j))
                        progress = True
                        continue
                s["ph"] = 2
            elif s["ph"] == 2:  # hand over tile j
                if j + 1 < n:
                    bar = (q, p)
                    assert arrives.get(bar, 0) == syncs.get(bar, 0), f"second hand-over before the first was received {bar}"
                    stop[(p, q)] = s["draining"]
                    arrives[bar] = arrives.get(bar, 0) + 1
                if s["draining"]:
                    s.update(done=True, exit=("drain", j))
                    progress = True
                    continue
                s["ph"] = 3
            elif s["ph"] == 3:  # arrive at the parity barrier
                parity_bar[p].setdefault(bar_index[w], {})[q] = s["fail"]
                s["ph"] = 4
            else:  # leave it once all four have arrived
                inst = parity_bar[p][bar_index[w]]
                if len(inst) < 4:
                    continue
                bar_index[w] += 1
                if any(inst.values()):
                    s["draining"] = True
                s.update(j=j + 2, ph=0)
            progress = True
    stuck = [w for w in warps if not st[w]["done"]]
    assert not stuck, f"deadlock: n={n} fail_at={fail_at} stuck={stuck}"
    for bar in set(arrives) | set(syncs):
        assert arrives.get(bar, 0) == syncs.get(bar, 0), f"unreceived hand-over on {bar}"
    for p in range(2):
        assert len({st[(p, q)]["exit"] for q in range(4)}) == 1, f"parity {p} warps left at different tiles"


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5])
def test_handover_every_failure_pattern(n):
    warps = [(p, q) for p in range(2) for q in range(4)]
    options = [[None] + list(range(w[0], n, 2)) for w in warps]
    for combo in itertools.product(*options):
        _run(n, dict(zip(warps, combo)))


def test_handover_random_long_splits():
    rng = random.Random(7)
    warps = [(p, q) for p in range(2) for q in range(4)]
    for _ in range(3000):
        n = rng.randint(6, 60)
        fail_at = {w: (rng.choice(range(w[0], n, 2)) if rng.random() < 0.5 else None) for w in warps}
        _run(n, fail_at)


def test_handover_no_failure_runs_every_tile():
    for n in range(1, 20):
        _run(n, {(p, q): None for p in range(2) for q in range(4)})
