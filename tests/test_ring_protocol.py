"""Host model of the all-laps ring launch's counter protocol (no GPU).

The cooperative GEMM launch of modes 6/7 orders ring refills with two
per-m-tile counters: producers wait for moved[gm] == 16 before loading an
m-tile, and the movers of lap L wait for consumed[gm'] == N/BN of the same
slot's previous tenant (lap L - 2). This model replays that protocol on
concrete schedules with every CTA walking its tiles and move items in the
kernel's order, and checks that it always makes progress (no wait cycle),
that the previous tenant is the same (expert, m-tile), and that every index
stays inside the buffers the host sizes, for 1, 2 and 4 mover warps per CTA.
"""
import numpy as np
import pytest

RING_BUFS = 2
MOVE_ITEMS = 16


def cdiv(a, b):
    return -(-a // b)


def lap_schedule(counts, E, S, C, T):
    """LAPTILES [Lb][Ep+1] and LAPBASE [Lb+1] as the schedule kernel defines them."""
    Ep = E + S
    Lb = cdiv(T, C)
    lt = np.zeros((Lb, Ep + 1), np.int64)
    for L in range(Lb):
        run = 0
        for e in range(Ep):
            lt[L, e] = run
            n = counts[e]
            ln = min(max(n - L * C, 0), C) if e < E else (n if L == 0 else 0)
            run += cdiv(ln, 128)
        lt[L, Ep] = run
    lapbase = np.concatenate([[0], np.cumsum(lt[:, Ep])])
    return lt, lapbase, Lb


def seg(v, n, x):
    lo, hi = 0, n
    while hi - lo > 1:
        mid = (lo + hi) // 2
        if v[mid] <= x:
            lo = mid
        else:
            hi = mid
    return lo


def replay(counts, E, S, T, C, grid, nt, mv=2):
    Ep = E + S
    lt, lapbase, Lb = lap_schedule(counts, E, S, C, T)
    A = int(sum(counts[:E]))
    Rmax = cdiv(A + S * T, 128) * 128 + 128 * Ep
    ntot = int(lapbase[-1])
    assert ntot <= Rmax // 128 + Ep * max(Lb, 1)          # counter buffers' size

    def decode(gm):
        L = seg(lapbase, Lb, gm)
        g = gm - lapbase[L]
        e = seg(lt[L], Ep, g)
        return L, g, e, g - lt[L, e]

    moved = np.zeros(ntot, int)
    consumed = np.zeros(ntot, int)
    prod = [list(range(c, ntot * nt, grid)) for c in range(grid)]
    movers = [list(range(mv * c + w, ntot * MOVE_ITEMS, mv * grid)) for c in range(grid) for w in range(mv)]
    pi = [0] * len(prod)
    mi = [0] * len(movers)
    while True:
        progressed = False
        for c, tiles in enumerate(prod):
            while pi[c] < len(tiles):
                gm = tiles[pi[c]] // nt
                L, g, e, mt = decode(gm)
                if e < E:
                    row = ((L % RING_BUFS) * E + e) * C + mt * 128
                    assert mt * 128 < C and row + 128 <= RING_BUFS * E * C
                    if moved[gm] < MOVE_ITEMS:
                        break
                    consumed[gm] += 1
                pi[c] += 1
                progressed = True
        for w, items in enumerate(movers):
            while mi[w] < len(items):
                gm = items[mi[w]] // MOVE_ITEMS
                L, g, e, mt = decode(gm)
                if g >= lt[L, E]:               # shared-expert tile: no move
                    mi[w] += 1
                    progressed = True
                    continue
                if L >= RING_BUFS:
                    gp = lapbase[L - RING_BUFS] + lt[L - RING_BUFS, e] + mt
                    assert decode(gp)[2:] == (e, mt)
                    if consumed[gp] < nt:
                        break
                moved[gm] += 1
                mi[w] += 1
                progressed = True
        if all(pi[c] == len(t) for c, t in enumerate(prod)) and all(mi[w] == len(i) for w, i in enumerate(movers)):
            break
        assert progressed, "wait cycle"
    assert (moved[[gm for gm in range(ntot) if decode(gm)[2] < E]] == MOVE_ITEMS).all()
    return ntot


def zipf_counts(E, T, k, s, seed):
    rng = np.random.default_rng(seed)
    p = 1.0 / np.arange(1, E + 1) ** s
    p /= p.sum()
    return [int(c) for c in np.minimum(rng.multinomial(T * k, rng.permutation(p)), T)]


@pytest.mark.parametrize("mv", [1, 2, 4])
@pytest.mark.parametrize("grid", [1, 3, 16, 152])
def test_zipf_wrap_schedule_progresses(grid, mv):
    counts = zipf_counts(64, 2048, 8, 1.1, 0) + [2048]
    assert max(counts[:64]) > 3 * 128                    # several laps of C=128
    replay(counts, 64, 1, 2048, 128, grid, 16, mv)


@pytest.mark.parametrize("mv", [1, 2, 4])
def test_benchmark_shape_schedule_progresses(mv):
    counts = zipf_counts(256, 16384, 8, 1.1, 1) + [16384]
    replay(counts, 256, 1, 16384, 640, 152, 16, mv)


@pytest.mark.parametrize("counts,E,S,T,C,nt", [
    ([300, 0, 5, 128, 129, 640, 1000, 20], 8, 0, 1000, 128, 2),   # empty expert, exact multiples, long tail
    ([515] * 8, 8, 0, 515, 128, 3),                             # every expert wraps
    ([515] * 8 + [515], 8, 1, 515, 128, 3),                     # plus the shared expert in lap 0
    ([0] * 4 + [0], 4, 1, 0, 128, 2),                           # no tokens
])
def test_edge_schedules_progress(counts, E, S, T, C, nt):
    for grid in (1, 2, 7):
        for mv in (1, 2, 4):
            replay(counts, E, S, T, C, grid, nt, mv)
