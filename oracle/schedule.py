"""Device-side schedule, stated plainly: counts, prefix sums, ranks, ring laps.

The write-ups: the schedule is built on the device with no CPU involvement,
it costs under 3 % of the MoE runtime, and backward reuses it with no
re-sort (Cursor blog summary, "method points", bullets on communication
direction and on removing CPU-GPU sync); tokens go into fixed-capacity ring
token buffers whose regions are reused once a batch is computed, without
dropping tokens (techlab report, section on the ring buffer; mlqm
commentary, section "signalling cut to 18 us").

Reading used here (the write-ups give no formulas):
  assignment a = t*k + j, taken in (t, j) lexicographic order;
  n_e       = #{a : idx[a] = e};
  offsets   = exclusive prefix sum of n_e (length E+1);
  rank r(a) = #{a' < a : idx[a'] = idx[a]}  (stable, (t,j) order);
  pos  p(a) = offsets[e] + r(a)             (a bijection onto [0, T*k));
  lap  = r // C, slot = r % C for ring capacity C per expert.
"""
from __future__ import annotations

import numpy as np


def schedule(idx, E: int, C: int) -> dict:
    flat = np.asarray(idx, dtype=np.int64).reshape(-1)
    A = flat.size
    counts = np.bincount(flat, minlength=E).astype(np.int64)
    offsets = np.zeros(E + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(counts)
    order = np.argsort(flat, kind="stable")          # assignments grouped by expert, (t,j) order inside
    rank = np.empty(A, dtype=np.int64)
    rank[order] = np.arange(A) - offsets[flat[order]]
    pos = offsets[flat] + rank
    inv = np.empty(A, dtype=np.int64)
    inv[pos] = np.arange(A)
    return {
        "counts": counts,
        "offsets": offsets,
        "rank": rank,
        "pos": pos,
        "inv": inv,
        "lap": rank // C,
        "slot": rank % C,
        "n_laps": int(((counts + C - 1) // C).max()) if A else 0,
    }


def expert_rows(sched: dict, e: int) -> np.ndarray:
    """Assignments a = t*k+j routed to expert e, in rank order."""
    o = sched["offsets"]
    return sched["inv"][o[e]:o[e + 1]]
