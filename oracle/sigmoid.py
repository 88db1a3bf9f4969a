"""The specified fp32 sigmoid of the router -- oracle side.

The write-ups describe a DeepSeek-V3-style router (Cursor blog summary,
"method points"): sigmoid scores, per-expert bias, group-limited top-k.
Which expert a token picks is an integer decision taken from floating-point
scores, so both implementations must compute the scores with the same
arithmetic. This module fixes that arithmetic; the CUDA kernel restates the
same definition independently.

Definition (IEEE binary32, round-to-nearest-even, no fused multiply-add):

  sigma(l) = 1 / (1 + E(-clamp(l, -80, 80)))

  E(z): Cody & Waite range reduction (W. J. Cody, W. Waite, "Software
  Manual for the Elementary Functions", 1980) followed by a Taylor
  polynomial:
    n  = rint(z * LOG2E)                    (ties to even)
    r  = (z - n*C1) - n*C2                  C1 = ln2 rounded to 9 significant
                                            bits, C2 = fp32(ln2 - C1)
    p  = Horner(r; 1/7!, 1/6!, ..., 1/1!, 1)   coefficients rounded to fp32
    E  = p * 2^n                            (2^n built from exponent bits)

With |r| <= ln2/2 the truncated Taylor term is below 6e-9, so E is within a
few ulp of exp (pinned against fp64 exp in the tests).
"""
from __future__ import annotations

import math

import numpy as np

f32 = np.float32

LOG2E = f32(1.0 / math.log(2.0))
C1 = f32(round(math.log(2.0) * 512.0) / 512.0)          # 355/512, exact in 9 bits
C2 = f32(math.log(2.0) - float(C1))
COEF = [f32(1.0 / math.factorial(i)) for i in range(8)]   # 1/0! .. 1/7!
CLAMP = f32(80.0)


def exp_spec(z) -> np.ndarray:
    """E(z) in fp32 for z in [-80, 80] (see module docstring)."""
    z = np.asarray(z, dtype=np.float32)
    n = np.rint(z * LOG2E).astype(np.float32)
    r = (z - n * C1) - n * C2
    p = COEF[7]
    for i in range(6, -1, -1):
        p = p * r + COEF[i]
    p = np.asarray(p, dtype=np.float32)
    two_n = ((n.astype(np.int32) + 127) << 23).astype(np.int32).view(np.float32)
    return (p * two_n).astype(np.float32)


def sigmoid_spec(l) -> np.ndarray:
    """sigma(l) in fp32, bit-for-bit the router's definition."""
    l = np.asarray(l, dtype=np.float32)
    lc = np.minimum(np.maximum(l, -CLAMP), CLAMP)
    e = exp_spec(-lc)
    return (f32(1.0) / (f32(1.0) + e)).astype(np.float32)
