"""Pins of the oracle's schedule against brute-force counting and invariants."""
import json
import os

import numpy as np

from oracle import schedule as S
from oracle import waves as W


def _brute(idx, E, C):
    seen = [0] * E
    rank = []
    for e in np.asarray(idx).reshape(-1):
        rank.append(seen[e])
        seen[e] += 1
    return np.array(seen), np.array(rank)


def test_schedule_brute_force_and_invariants():
    rng = np.random.default_rng(0)
    T, k, E, C = 300, 4, 16, 128
    idx = np.stack([rng.choice(E, k, replace=False) for _ in range(T)])
    idx[:40] = [0, 1, 2, 3]                       # make expert 0..3 overflow-prone
    sch = S.schedule(idx, E, C)
    counts, rank = _brute(idx, E, C)
    assert np.array_equal(sch["counts"], counts)
    assert np.array_equal(sch["rank"], rank)
    assert sch["counts"].sum() == T * k
    assert sorted(sch["pos"].tolist()) == list(range(T * k))          # bijection
    assert np.array_equal(sch["inv"][sch["pos"]], np.arange(T * k))
    assert np.array_equal(sch["lap"] * C + sch["slot"], sch["rank"])
    flat = idx.reshape(-1)
    # within one (expert, lap) no two assignments share a ring slot
    keys = set()
    for a in range(T * k):
        key = (flat[a], sch["lap"][a], sch["slot"][a])
        assert key not in keys
        keys.add(key)
    # ranks of an expert follow (t, j) order
    for e in range(E):
        rows = S.expert_rows(sch, e)
        assert np.all(np.diff(rows) > 0)
        assert np.all(flat[rows] == e)
    assert sch["n_laps"] == int(max((c + C - 1) // C for c in counts))


def test_empty_expert_and_empty_input():
    idx = np.array([[1, 2], [2, 1]])
    sch = S.schedule(idx, 4, 128)
    assert sch["counts"].tolist() == [0, 2, 2, 0]
    assert sch["offsets"].tolist() == [0, 0, 2, 4, 4]
    sch0 = S.schedule(np.zeros((0, 2), np.int64), 4, 128)
    assert sch0["counts"].sum() == 0 and sch0["n_laps"] == 0


def test_wave_threshold_worked_example():
    with open(os.path.join(os.path.dirname(__file__), "golden", "wave_threshold.json")) as f:
        g = json.load(f)
    i = g["inputs"]
    th = W.wave_threshold(i["sm_count"], i["tokens_per_sm_per_wave"], i["waves"])
    assert th == g["threshold"]
    for tok, hidden in g["decisions"].items():
        assert W.hides_communication(int(tok), th) == hidden


def test_grouped_gemm_waves():
    # 152 SMs; 256 experts with 128 rows each and N = 4096 at 256-wide tiles: 256*16/152
    assert abs(W.grouped_gemm_waves([128] * 256, 4096, 152) - 256 * 16 / 152) < 1e-12
    assert W.grouped_gemm_waves([129], 256, 1) == 2.0
