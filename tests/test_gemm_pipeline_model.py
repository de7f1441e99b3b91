"""A step-by-step model of the grouped GEMM's mbarrier protocol (the TMA
producer, the MMA issuer and the epilogue warps of one CTA), run under random
interleavings on the CPU, with every main-loop wait given a short poll limit
so that it times out at random points.

As the kernel does it:

- the producer waits for a ring stage to be empty (parity trick: the first
  use of a stage passes at once), then issues the stage's TMA fill, which
  completes the stage's full barrier when it lands;
- the MMA issuer waits for a chunk accumulator to be free (tempty), then,
  per K block, for the stage to be full, issues the block's MMAs and commits
  them to the stage's empty barrier; after the chunk's last block it commits
  to the accumulator's tfull barrier (a commit arrives once every MMA issued
  before it has completed; MMAs complete in issue order);
- each epilogue warp waits for tfull, reads the accumulator, arrives on
  tempty, and after the tile's last chunk stores the tile (bulk stores it
  waits for before retiring);
- a wait that runs out sets the abort flag; a role that sees it stops
  issuing work and drains: the producer waits (full bound) for the last fill
  of each stage, the MMA issuer for its last stage release and its last
  chunk commit, and a chunk cut short is never committed; then all meet at
  the block barrier and TMEM is freed.

Checks: when the block barrier is passed (the CTA frees TMEM and may
retire) no TMA fill, MMA, commit arrive or store is still in flight; the
epilogue only ever reads a chunk whose MMAs are all complete; no drain wait
runs out; without timeouts every chunk of every tile is read and stored."""
import random

import pytest

DRAIN = 10 ** 6          # the drain waits' bound (never reached in the model)


class Bar:
    """mbarrier with a count of completed phases; try_wait(parity) is true
    once the phase of that parity has completed (the current phase's
    parity differs)."""

    def __init__(self, count=1):
        self.count = count
        self.pending = count
        self.done = 0

    def arrive(self):
        self.pending -= 1
        assert self.pending >= 0, "more arrivals than the barrier's count"
        if self.pending == 0:
            self.done += 1
            self.pending = self.count

    def try_wait(self, parity):
        return (self.done & 1) != parity


class Cta:
    def __init__(self, rng, S, tiles, nkb, chunk_blocks, epi_warps, main_limit):
        self.rng = rng
        self.S, self.tiles, self.nkb = S, tiles, nkb
        self.cb = chunk_blocks
        self.nchunks = (nkb + chunk_blocks - 1) // chunk_blocks
        self.E = epi_warps
        self.main_limit = main_limit
        self.full = [Bar() for _ in range(S)]
        self.empty = [Bar() for _ in range(S)]
        self.tfull = [Bar() for _ in range(2)]
        self.tempty = [Bar(epi_warps) for _ in range(2)]
        self.abort = False
        self.timeouts = 0
        # async engine
        self.fills = []            # (fill index, stage) in flight
        self.stage_fill = [None] * S   # fill index whose data sits in each stage
        self.mma_issued = 0
        self.mma_done = 0
        self.mma_chunk = []        # chunk id of MMA i
        self.commits = []          # (bar, mma count it waits for)
        self.stores = {}           # epilogue warp -> in-flight stores
        self.chunk_mmas = {}       # chunk id -> MMAs issued for it
        self.chunk_mmas_done = {}  # chunk id -> MMAs completed
        self.read = set()          # (warp, chunk id) reads
        self.stored = set()        # (warp, tile) stores completed
        self.at_barrier = 0

    # ---- waits -----------------------------------------------------------
    def wait(self, bar, parity, limit):
        for _ in range(limit):
            if bar.try_wait(parity):
                return True
            yield
        return False

    def drain_wait(self, bar, parity):
        ok = yield from self.wait(bar, parity, DRAIN)
        assert ok, "a drain wait ran out"

    # ---- roles -----------------------------------------------------------
    def producer(self):
        S = self.S
        stage = phase = nload = 0
        for t in range(self.tiles):
            if self.abort:
                break
            for kb in range(self.nkb):
                ok = yield from self.wait(self.empty[stage], phase ^ 1, self.main_limit)
                if not ok:
                    self.timeouts += 1
                    self.abort = True
                    break
                self.fills.append((nload, stage))     # arrive_expect_tx + two TMA loads
                nload += 1
                stage += 1
                if stage == S:
                    stage, phase = 0, phase ^ 1
                yield
        for _ in range(S):                            # last MMA read of every stage,
            if self.abort:                            # or until another role aborts
                break
            done = False
            for _ in range(DRAIN):
                done = self.empty[stage].try_wait(phase ^ 1)
                if done or self.abort:
                    break
                yield
            if not done and not self.abort:
                self.abort = True
            stage += 1
            if stage == S:
                stage, phase = 0, phase ^ 1
        if self.abort:                                # last fill of each stage lands
            for i in range(max(0, nload - S), nload):
                yield from self.drain_wait(self.full[i % S], (i // S) & 1)
        yield from self.block_barrier()

    def mma(self):
        S = self.S
        stage = phase = chunk_ctr = ncommit = 0
        last_tfull = None
        ok = True
        for t in range(self.tiles):
            if not ok:
                break
            for c in range(self.nchunks):
                b, use = chunk_ctr & 1, (chunk_ctr >> 1) & 1
                got = yield from self.wait(self.tempty[b], use ^ 1, self.main_limit)
                if not got or self.abort:
                    ok = False
                    break
                cid = (t, c)
                kb1 = min((c + 1) * self.cb, self.nkb)
                for kb in range(c * self.cb, kb1):
                    got = yield from self.wait(self.full[stage], phase, self.main_limit)
                    if not got or self.abort:
                        ok = False
                        break
                    assert self.stage_fill[stage] is not None, "MMA read an empty stage"
                    for _ in range(4):                # the block's MMAs
                        self.mma_issued += 1
                        self.mma_chunk.append(cid)
                        self.chunk_mmas[cid] = self.chunk_mmas.get(cid, 0) + 1
                    self.commits.append((self.empty[stage], self.mma_issued, ("stage", stage)))
                    ncommit += 1
                    stage += 1
                    if stage == S:
                        stage, phase = 0, phase ^ 1
                    yield
                if not ok:
                    break
                self.commits.append((self.tfull[b], self.mma_issued, ("chunk", cid)))
                last_tfull = (b, use)
                chunk_ctr += 1
        if not ok:
            self.timeouts += 1
            self.abort = True
        if self.abort and ncommit > 0:                # issued MMAs finish before TMEM goes
            k = ncommit - 1
            yield from self.drain_wait(self.empty[k % S], (k // S) & 1)
        if self.abort and last_tfull is not None:     # and the last chunk commit has landed
            yield from self.drain_wait(self.tfull[last_tfull[0]], last_tfull[1])
        yield from self.block_barrier()

    def epilogue(self, w):
        chunk_ctr = 0
        self.stores[w] = []
        for t in range(self.tiles):
            ok = True
            for c in range(self.nchunks):
                b, use = chunk_ctr & 1, (chunk_ctr >> 1) & 1
                got = yield from self.wait(self.tfull[b], use, self.main_limit)
                if not got or self.abort:
                    ok = False
                    break
                cid = (t, c)
                want = 4 * (min((c + 1) * self.cb, self.nkb) - c * self.cb)
                assert self.chunk_mmas.get(cid, 0) == want, "read a chunk cut short"
                assert self.chunk_mmas_done.get(cid, 0) == want, "read unfinished sums"
                self.read.add((w, cid))
                self.tempty[b].arrive()
                chunk_ctr += 1
                yield
            if not ok:
                self.timeouts += 1
                self.abort = True
                break
            self.stores[w].append(t)
            yield
        while self.stores[w]:                         # bulk wait_group 0
            yield
        yield from self.block_barrier()

    def block_barrier(self):
        self.at_barrier += 1
        while self.at_barrier < 2 + self.E:
            yield
        # past the barrier: TMEM is freed and the CTA may retire
        assert not self.fills, "a TMA fill is still in flight"
        assert self.mma_done == self.mma_issued, "an MMA is still running"
        assert not self.commits, "a commit arrive is still in flight"
        assert not any(self.stores.values()), "a store is still in flight"

    # ---- the asynchronous units --------------------------------------------
    def engine_step(self):
        choices = []
        if self.fills:
            choices.append("fill")
        if self.mma_done < self.mma_issued:
            choices.append("mma")
        if any(n <= self.mma_done for _, n, _ in self.commits):
            choices.append("commit")
        if any(self.stores.values()):
            choices.append("store")
        if not choices:
            return False
        kind = self.rng.choice(choices)
        if kind == "fill":
            i, s = self.fills.pop(self.rng.randrange(len(self.fills)))
            self.stage_fill[s] = i
            self.full[s].arrive()                     # the transaction bytes complete it
        elif kind == "mma":                           # in issue order
            cid = self.mma_chunk[self.mma_done]
            self.mma_done += 1
            self.chunk_mmas_done[cid] = self.chunk_mmas_done.get(cid, 0) + 1
        elif kind == "commit":                        # commits fire in issue order
            bar, n, what = self.commits[0]
            if n <= self.mma_done:
                self.commits.pop(0)
                if what[0] == "stage":
                    self.stage_fill[what[1]] = None   # the stage is free again
                bar.arrive()
        else:
            w = self.rng.choice([w for w, s in self.stores.items() if s])
            t = self.stores[w].pop(0)
            self.stored.add((w, t))
        return True


def run(seed, S, tiles, nkb, cb, E, main_limit, p_engine):
    rng = random.Random(seed)
    cta = Cta(rng, S, tiles, nkb, cb, E, main_limit)
    roles = [cta.producer(), cta.mma()] + [cta.epilogue(w) for w in range(E)]
    alive = list(roles)
    steps = 0
    while alive:
        steps += 1
        assert steps < 5_000_000, "the CTA never retires"
        if rng.random() < p_engine and cta.engine_step():
            continue
        g = rng.choice(alive)
        try:
            next(g)
        except StopIteration:
            alive.remove(g)
    return cta


@pytest.mark.parametrize("seed", range(40))
def test_timeouts_anywhere_leave_nothing_in_flight(seed):
    rng = random.Random(1000 + seed)
    S = rng.choice([3, 4])
    tiles = rng.randint(1, 4)
    nkb = rng.randint(1, 7)
    cb = rng.choice([1, 2, 3])
    E = rng.choice([1, 2, 4])
    limit = rng.choice([1, 1, 2, 3, 8, 40])
    p = rng.choice([0.05, 0.2, 0.5, 0.8])
    cta = run(seed, S, tiles, nkb, cb, E, limit, p)
    if cta.timeouts:
        assert cta.abort


@pytest.mark.parametrize("seed", range(12))
def test_without_timeouts_every_chunk_is_read_and_stored(seed):
    rng = random.Random(2000 + seed)
    S, tiles, nkb, cb, E = 4, rng.randint(1, 5), rng.randint(1, 9), 2, rng.choice([2, 4])
    cta = run(seed, S, tiles, nkb, cb, E, DRAIN, rng.choice([0.1, 0.5]))
    assert not cta.abort and cta.timeouts == 0
    nchunks = (nkb + cb - 1) // cb
    assert cta.read == {(w, (t, c)) for w in range(E) for t in range(tiles)
                        for c in range(nchunks)}
    assert cta.stored == {(w, t) for w in range(E) for t in range(tiles)}


def test_first_wait_times_out_at_once():
    """The smallest case with a one-poll limit, as the GPU test runs it: the
    MMA issuer's first stage wait cannot succeed before the engine runs."""
    cta = run(7, 4, 1, 2, 16, 8, 1, 0.0001)
    assert cta.abort and cta.timeouts >= 1
