"""Host model of the all-laps ring launch's counter protocol (no GPU).

The cooperative GEMM launch of modes 6/7 orders ring refills with two
per-m-tile counters: producers wait for moved[gm] == 16 before loading an
m-tile, and the movers of lap L wait for consumed[gm'] == N/BN of the same
slot's previous tenant (lap L - 2). CTAs walk tiles and move items in the
schedule's walk order (LAPORDER: position -> lap-major m-tile gm). This model
restates that order from its definition, replays the protocol on concrete
schedules with every CTA walking its tiles and move items in that order, and
checks that it always makes progress (no wait cycle), that the previous
tenant is the same (expert, m-tile) at an earlier position, and that every
index stays inside the buffers the host sizes, for 1, 2 and 4 mover warps
per CTA. The lap-major order (identity walk) is replayed too.
"""
from fractions import Fraction

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


def walk_order(counts, E, S, C, T):
    """LAPORDER: lap-major m-tiles sorted by (key, expert, gm). An expert's unit is
    its lap pair P = L // 2; an expert with two or more pairs has key (2P+1) / (2 pairs),
    the experts with one pair take (2i+1) / (2 n_one) in expert order."""
    Ep = E + S
    lt, lapbase, Lb = lap_schedule(counts, E, S, C, T)
    laps = [cdiv(counts[e], C) if e < E else (1 if counts[e] > 0 else 0) for e in range(Ep)]
    pairs = [(n + 1) // 2 for n in laps]
    one_idx, n_one = {}, 0
    for e in range(Ep):
        if pairs[e] == 1:
            one_idx[e] = n_one
            n_one += 1
    keys = []
    for L in range(Lb):
        for e in range(Ep):
            for mt in range(lt[L, e + 1] - lt[L, e] if e + 1 <= Ep else 0):
                gm = int(lapbase[L] + lt[L, e] + mt)
                key = Fraction(2 * (L // 2) + 1, 2 * pairs[e]) if pairs[e] >= 2 else Fraction(2 * one_idx[e] + 1, 2 * n_one)
                keys.append((key, e, gm))
    keys.sort()
    order = [gm for _, _, gm in keys]
    assert sorted(order) == list(range(int(lapbase[-1])))
    return order


def decode_tables(counts, E, S, C, T):
    """The GEMMs' decode tables restated by searching the lap and expert prefix sums
    (the device builds them while it expands the walk order):
      ring[pos] = {gm, e | valid << 16 | ok << 24 | shared << 25, A row, padded rank row,
                   previous tenant's gm or -1, rank of the first row, count, poff[e]};
      push[g]   = e | valid << 16 for m-tile g of the padded rank rows;
      wg[r]     = {e, poff[e] / 128, tiles of e, 0} for the r-th expert by descending count."""
    Ep = E + S
    lt, lapbase, Lb = lap_schedule(counts, E, S, C, T)
    poff = np.concatenate([[0], np.cumsum([cdiv(c, 128) * 128 for c in counts])]).astype(np.int64)
    order = walk_order(counts, E, S, C, T)
    ring = np.zeros((len(order), 8), np.int64)
    for pos, gm in enumerate(order):
        L = seg(lapbase, Lb, gm)
        g = gm - lapbase[L]
        e = seg(lt[L], Ep, g)
        mt = g - lt[L, e]
        shared = e >= E
        rank0 = mt * 128 if shared else L * C + mt * 128
        a_row = mt * 128 if shared else ((L % RING_BUFS) * E + e) * C + mt * 128
        prow0 = poff[e] + rank0
        valid = min(max(counts[e] - rank0, 0), 128)
        ok = int(prow0 + 128 <= poff[e + 1] and valid > 0)
        gp = -1
        if not shared and L >= RING_BUFS:
            gp = lapbase[L - RING_BUFS] + lt[L - RING_BUFS, e] + mt
        ring[pos] = [gm, e | valid << 16 | ok << 24 | int(shared) << 25, a_row, prow0, gp, rank0, counts[e], poff[e]]
    push = np.zeros(int(poff[-1]) // 128, np.int64)
    for g in range(len(push)):
        e = seg(poff, Ep, g * 128)
        push[g] = e | min(max(counts[e] - (g * 128 - poff[e]), 0), 128) << 16
    by_count = sorted(range(Ep), key=lambda e: (-counts[e], e))
    wg = np.array([[e, poff[e] // 128, (poff[e + 1] - poff[e]) // 128, 0] for e in by_count], np.int64).reshape(-1, 4)
    return ring, push, wg


def replay(counts, E, S, T, C, grid, nt, mv=2, order=None):
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

    if order is None:
        order = walk_order(counts, E, S, C, T)
    position = {gm: i for i, gm in enumerate(order)}
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
                gm = order[tiles[pi[c]] // nt]
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
                gm = order[items[mi[w]] // MOVE_ITEMS]
                L, g, e, mt = decode(gm)
                if g >= lt[L, E]:               # shared-expert tile: no move
                    mi[w] += 1
                    progressed = True
                    continue
                if L >= RING_BUFS:
                    gp = lapbase[L - RING_BUFS] + lt[L - RING_BUFS, e] + mt
                    assert decode(gp)[2:] == (e, mt)
                    assert position[gp] < position[gm]     # the previous tenant is walked first
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
    replay(counts, 64, 1, 2048, 128, grid, 16, mv, order=list(range(replay(counts, 64, 1, 2048, 128, 1, 16, 1))))


def test_walk_order_pairs_and_spread():
    """The walk keeps an expert's laps 2P and 2P+1 side by side and spreads its pairs:
    every hot expert's pair P starts later than its pair P-1, and the hottest
    expert's pairs are not bunched at the end of the walk."""
    counts = zipf_counts(64, 2048, 8, 1.1, 0) + [2048]
    E, S, C, T = 64, 1, 128, 2048
    lt, lapbase, Lb = lap_schedule(counts, E, S, C, T)
    order = walk_order(counts, E, S, C, T)
    pos = {gm: i for i, gm in enumerate(order)}

    def tiles(e, L):
        return [int(lapbase[L] + lt[L, e] + mt) for mt in range(lt[L, e + 1] - lt[L, e])]
    hot = int(np.argmax(counts[:E]))
    laps = cdiv(counts[hot], C)
    first = []
    for P in range((laps + 1) // 2):
        span = [pos[g] for L in (2 * P, 2 * P + 1) if L < laps for g in tiles(hot, L)]
        assert max(span) - min(span) + 1 == len(span)    # the pair is contiguous in the walk
        first.append(min(span))
    assert first == sorted(first)
    assert first[0] < len(order) // 4 and first[-1] > len(order) // 2


@pytest.mark.parametrize("counts,E,S,T,C", [
    (zipf_counts(64, 2048, 8, 1.1, 0) + [2048], 64, 1, 2048, 128),
    ([300, 0, 5, 128, 129, 640, 1000, 20], 8, 0, 1000, 128),
    ([515] * 8 + [515], 8, 1, 515, 128),
])
def test_decode_tables_consistent(counts, E, S, T, C):
    """Every ring position decodes to an in-bounds ring slot whose previous tenant is the
    same (expert, m-tile) at an earlier position, the push table covers each expert's
    padded rows with its valid counts, and the weight-gradient table lists every expert."""
    Ep = E + S
    ring, push, wg = decode_tables(counts, E, S, C, T)
    order = walk_order(counts, E, S, C, T)
    pos = {gm: i for i, gm in enumerate(order)}
    assert list(ring[:, 0]) == order
    for r in ring:
        e, valid, ok, shared = r[1] & 0xFFFF, (r[1] >> 16) & 0xFF, (r[1] >> 24) & 1, (r[1] >> 25) & 1
        assert ok == 1 and 0 < valid <= 128 and shared == (e >= E)
        if not shared:
            assert r[2] + 128 <= RING_BUFS * E * C and r[5] % C + 128 <= C
        if r[4] >= 0:
            prev = ring[pos[int(r[4])]]
            assert pos[int(r[4])] < pos[int(r[0])] and prev[1] & 0xFFFF == e and prev[2] == r[2]
            assert prev[5] + RING_BUFS * C == r[5]
    assert sum(((v >> 16) & 0xFF) for v in push) == sum(counts)
    assert sorted(wg[:, 0]) == list(range(Ep)) and sum(wg[:, 2]) == len(push)


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
