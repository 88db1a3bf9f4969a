"""SM-wave token threshold of the overlap-granularity heuristic.

The mlqm commentary (section "overlap granularity: the middle value is
optimal") states the rule that every per-expert grouped GEMM should cover at
least two full SM waves, and (section "a runnable snippet") restates it as
threshold = sm_count * tokens_per_sm_per_wave * waves, printing 2376 for
132 SMs, 9 tokens per SM per wave and 2 waves. The 2368-token figure quoted
for the Kimi 2.5 shape comes without its inputs, so only the product rule is
pinned here.

``grouped_gemm_waves`` is this layer's own measure of the same quantity:
output tiles of one grouped GEMM divided by the SM count.
"""
from __future__ import annotations

import numpy as np


def wave_threshold(sm_count: int, tokens_per_sm_per_wave: int, waves: int = 2) -> int:
    return sm_count * tokens_per_sm_per_wave * waves


def hides_communication(tokens: int, threshold: int) -> bool:
    return tokens >= threshold


def grouped_gemm_waves(counts, N: int, sm_count: int, BM: int = 128, BN: int = 256) -> float:
    counts = np.asarray(counts, dtype=np.int64)
    tiles = int(((counts + BM - 1) // BM).sum()) * (-(-N // BN))
    return tiles / float(sm_count)
