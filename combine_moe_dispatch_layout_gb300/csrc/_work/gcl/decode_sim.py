"""Scratch: CPU model of the pair-tile decode of the clustered grouped GEMM."""
import random
BM, BN, RM = 128, 256, 8
def tables(counts, ntn, CL):
    goff, tpre = [0], [0]
    for c in counts:
        mt = (c + BM - 1) // BM
        goff.append(goff[-1] + c)
        tpre.append(tpre[-1] + ((mt + 1) // 2 if CL else mt) * ntn)
    return goff, tpre
def decode(t, goff, tpre, G, ntn, crank, CL):
    lo, hi = 0, G
    while hi - lo > 1:
        mid = (lo + hi) >> 1
        if tpre[mid] <= t: lo = mid
        else: hi = mid
    g = lo
    cnt = goff[g + 1] - goff[g]
    mt0 = (cnt + BM - 1) // BM
    mt = (mt0 + 1) // 2 if CL else mt0
    R = RM // 2 if CL else RM
    local = t - tpre[g]
    nblk = mt // R if mt // R > 0 else 1
    full = nblk - 1; per_full = R * ntn
    blk = local // per_full
    if blk < full:
        r = local - blk * per_full; m = blk * R + r % R; n = r // R
    else:
        rem = mt - full * R; r = local - full * per_full; m = full * R + r % rem; n = r // rem
    if CL: m = 2 * m + crank
    left = cnt - m * BM
    rows = BM if left >= BM else max(left, 0)
    return g, m, n, rows
random.seed(3)
cases = 0
for trial in range(400):
    G = random.randint(1, 40)
    counts = [random.choice([0, 1, 127, 128, 129, 700, 1024, 1030, 2049, random.randint(0, 5000)]) for _ in range(G)]
    N = random.choice([8, 136, 256, 4096, 7168])
    ntn = (N + BN - 1) // BN
    for CL in (False, True):
        goff, tpre = tables(counts, ntn, CL)
        seen = {}
        for t in range(tpre[G]):
            got = [decode(t, goff, tpre, G, ntn, cr, CL) for cr in ((0, 1) if CL else (0,))]
            if CL:
                assert got[0][0] == got[1][0] and got[0][2] == got[1][2], "pair shares expert and column tile"
                assert got[1][1] == got[0][1] + 1
            for g, m, n, rows in got:
                mt0 = (counts[g] + BM - 1) // BM
                if m < mt0:
                    assert rows == min(BM, counts[g] - m * BM) and rows > 0
                    key = (g, m, n)
                    assert key not in seen, ("dup", key)
                    seen[key] = 1
                else:
                    assert CL and rows == 0 and m == mt0, ("phantom", g, m, mt0, rows)
                assert 0 <= n < ntn
        want = sum(((c + BM - 1) // BM) * ntn for c in counts)
        assert len(seen) == want, (len(seen), want)
        cases += 1
print("ok", cases)
