"""A step-by-step model of the one-launch dispatch's grid barrier, run under
random interleavings on the CPU.

As the kernel does it: the workspace holds one 32-bit word, the arrival
count in its low 16 bits and a generation in its high 16.  Thread 0 of a CTA
adds 1 to the word (one atomic, which returns the old word); the CTA whose
add completes the count adds 0x10000 - n (count back to zero, generation + 1,
one more atomic); the others poll the word until its generation differs from
the one their add returned.  The word carries over from one barrier to the
next inside a launch (the kernel has up to three) and from one launch to
the next, whatever the grid size.
Checks: no CTA leaves barrier i before every CTA has reached it, nobody
spins forever, the word's count is zero after every launch, and the
generation wraps at 16 bits without losing a barrier."""
import random

import pytest

MASK = 0xFFFFFFFF


class Ws:
    def __init__(self, gen=0):
        self.word = (gen & 0xFFFF) << 16   # count 0; any generation left by earlier launches


def cta(ws, me, nblocks, nbar, arrived, left):
    for b in range(nbar):
        arrived[b].add(me)
        old = ws.word                            # atom.add: read and add in one step
        ws.word = (old + 1) & MASK
        yield
        gen = old >> 16
        if (old & 0xFFFF) == nblocks - 1:
            ws.word = (ws.word + 0x10000 - nblocks) & MASK   # red.add: count 0, gen + 1
            yield
        else:
            spins = 0
            while (ws.word >> 16) == gen:
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
    assert ws.word & 0xFFFF == 0


@pytest.mark.parametrize("seed", range(8))
def test_grid_barrier_random_schedules(seed):
    rng = random.Random(seed)
    ws = Ws(gen=rng.randrange(1 << 16))
    for nblocks in (2, 3, 7, 16, 5, 2, 40):
        for nbar in (3, 2):
            run_launch(ws, nblocks, nbar, rng)


def test_generation_wraps():
    rng = random.Random(5)
    ws = Ws(gen=0xFFFE)                 # the next barriers wrap the 16-bit generation
    for _ in range(4):
        run_launch(ws, 9, 3, rng)
    assert (ws.word >> 16) == (0xFFFE + 12) & 0xFFFF
