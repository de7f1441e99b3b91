"""A step-by-step model of the dispatch layout kernel's cross-CTA protocol,
run under random interleavings on the CPU (the GPU tests only see the
schedules the hardware happens to produce).

What is modelled, as the kernel does it: CTAs take tiles from a ticket
counter; a tile publishes its histogram (tile 0 of a source rank as an
inclusive prefix, the others as an aggregate) and then a status word tagged
with the launch epoch; a later tile of the same rank polls up to 32
predecessors at once, stops at the nearest inclusive prefix and adds the
vectors in between; with more than 33 tiles per rank a tile republishes its
own inclusive prefix once known; the last CTA out advances the epoch and
resets the counters.  Every memory access is a separate step that any other
CTA may interleave with.  Checks: every tile's exclusive prefix equals the
running sum of the earlier tiles' histograms, across several launches that
reuse one workspace with different tile counts (status words of an earlier
launch must never be taken for this launch's)."""
import random

import pytest

AGG, INC = 1, 2


class Workspace:
    def __init__(self, max_tiles, E):
        self.ticket = 0
        self.done = 0
        self.magic = 0
        self.status = [0] * max_tiles
        self.agg = [[0] * E for _ in range(max_tiles)]
        self.inc = [[0] * E for _ in range(max_tiles)]


def cta(ws, hist, tpr, num_tiles, E, out):
    """One CTA of one launch (a generator: each yield is a point where any
    other CTA may run)."""
    tile = ws.ticket
    ws.ticket += 1
    yield
    epoch = ws.magic % 0x3FFFFFFF + 1
    s, c = divmod(tile, tpr)
    tagg = hist[tile]
    vec = ws.inc if c == 0 else ws.agg
    for e in range(E):                       # the vector first ...
        vec[tile][e] = tagg[e]
        yield
    ws.status[tile] = (epoch << 2) | (INC if c == 0 else AGG)   # ... then its status
    yield
    excl = [0] * E
    if c > 0:
        first = tile - c
        hi = tile - 1
        while True:
            lanes = [hi - j for j in range(32) if hi - j >= first]
            seen = [0] * len(lanes)
            while not all(seen):             # lanes poll independently
                j = random.randrange(len(lanes))
                if not seen[j]:
                    v = ws.status[lanes[j]]
                    if (v >> 2) == epoch and (v & 3):
                        seen[j] = v & 3
                yield
            incs = [j for j, st in enumerate(seen) if st == INC]
            found = bool(incs)
            last = incs[0] if found else len(lanes) - 1
            for j in range(last + 1):        # vectors read one element at a time
                src = ws.inc if (found and j == last) else ws.agg
                for e in range(E):
                    excl[e] += src[lanes[j]][e]
                    yield
            if found:
                break
            hi -= 32
        if c < tpr - 1 and tpr > 33:         # republish as an inclusive prefix
            for e in range(E):
                ws.inc[tile][e] = excl[e] + tagg[e]
                yield
            ws.status[tile] = (epoch << 2) | INC
            yield
    out[tile] = excl
    d = ws.done
    ws.done += 1
    if d == num_tiles - 1:                   # the last CTA out
        ws.magic += 1
        ws.ticket = 0
        ws.done = 0
    yield


def run_launch(ws, R, tpr, E, rng):
    num_tiles = R * tpr
    hist = [[rng.randrange(0, 50) for _ in range(E)] for _ in range(num_tiles)]
    out = {}
    started, pending = [], num_tiles
    steps = 0
    while pending or started:
        steps += 1
        assert steps < 5_000_000
        # start a new CTA (takes the next ticket) or advance a started one
        if pending and (not started or rng.random() < 0.3):
            g = cta(ws, hist, tpr, num_tiles, E, out)
            started.append(g)
            pending -= 1
            continue
        g = rng.choice(started)
        try:
            next(g)
        except StopIteration:
            started.remove(g)
    for t in range(num_tiles):
        s, c = divmod(t, tpr)
        want = [sum(hist[s * tpr + u][e] for u in range(c)) for e in range(E)]
        assert out[t] == want, (t, out[t], want)
    assert ws.ticket == 0 and ws.done == 0


@pytest.mark.parametrize("seed", range(6))
def test_lookback_protocol_random_schedules(seed):
    rng = random.Random(seed)
    random.seed(seed)
    E = 3
    ws = Workspace(max_tiles=2 * 80, E=E)
    # several launches on one workspace, tile counts changing between them,
    # including ranks of more than 33 tiles (the republish path) and of
    # exactly 32 and 33 (window edges)
    for R, tpr in ((2, 5), (1, 40), (2, 33), (1, 32), (2, 70), (1, 2), (2, 34)):
        run_launch(ws, R, tpr, E, rng)
    assert ws.magic == 7
