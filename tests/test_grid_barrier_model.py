"""A step-by-step model of the one-launch dispatch's grid barrier, run under
random interleavings on the CPU.

As the kernel does it: a CTA reads the generation word, then adds itself to
the arrival count; the CTA that completes the count resets it to zero and
then publishes generation + 1; the others spin until the generation moves.
The workspace (count, generation) carries over from one launch to the next
and from one barrier to the next inside a launch (the kernel has three).
Checks: no CTA leaves barrier i before every CTA has reached it, nobody
spins forever, and the count is zero again after every launch."""
import random

import pytest


class Ws:
    def __init__(self):
        self.count = 0
        self.gen = 12345          # any value left by earlier launches


def cta(ws, me, nblocks, nbar, arrived, left):
    for b in range(nbar):
        arrived[b].add(me)
        g = ws.gen                           # read the generation first
        yield
        old = ws.count                       # atomicAdd(count, 1)
        ws.count = old + 1
        yield
        if old == nblocks - 1:
            ws.count = 0                     # reset before releasing the others
            yield
            ws.gen = g + 1
            yield
        else:
            spins = 0
            while ws.gen == g:
                spins += 1
                assert spins < 200_000, "barrier wait never ends"
                yield
        # leaving barrier b: every CTA must have arrived at it
        assert len(arrived[b]) == nblocks, ("left barrier %d early" % b, me)
        left[b].add(me)
        yield


def run_launch(ws, nblocks, nbar, rng):
    arrived = [set() for _ in range(nbar)]
    left = [set() for _ in range(nbar)]
    gens = [cta(ws, i, nblocks, nbar, arrived, left) for i in range(nblocks)]
    alive = list(gens)
    while alive:
        g = rng.choice(alive)
        try:
            next(g)
        except StopIteration:
            alive.remove(g)
    assert all(len(s) == nblocks for s in left)
    assert ws.count == 0


@pytest.mark.parametrize("seed", range(8))
def test_grid_barrier_random_schedules(seed):
    rng = random.Random(seed)
    ws = Ws()
    for nblocks in (2, 3, 7, 16, 5, 2, 40):
        run_launch(ws, nblocks, 3, rng)
