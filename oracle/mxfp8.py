"""MXFP8 (E4M3 elements, E8M0 scale per 32-element block) -- oracle side.

The write-ups only name the format: the MoE layer runs "in MXFP8" (Cursor
blog summary, "method points"; mlqm commentary, section "two scorecards").
The plain reading is the OCP Microscaling Formats v1.0 MXFP8 type:

* element: FP8 E4M3 (bias 7, no infinities, S.1111.111 is NaN, largest
  finite 448, subnormals m * 2^-9);
* block: 32 consecutive elements along the quantisation axis share one
  E8M0 scale byte X = 2^(byte-127);
* scale choice: byte = floor(log2(amax)) - 8 + 127 (8 = exponent of the
  largest normal E4M3 value), clamped to [0, 254]; an all-zero block has
  byte 0;
* element conversion: round-to-nearest-even of v / X, saturating to +-448.

All arithmetic here is fp64, where v / X and the decoding are exact.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
BLOCK = 32


def e4m3_decode(codes) -> np.ndarray:
    """Decode E4M3 byte codes to float64 (NaN for the two NaN codes)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    mag = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2((e - 7).astype(np.float64)))
    mag = np.where((c & 0x7F) == 0x7F, np.nan, mag)
    return sign * mag


def e4m3_encode(v) -> np.ndarray:
    """Round float64 values to E4M3 codes: nearest, ties to even, saturate to 448.

    The sign bit always follows the input's sign (so -0.0 and negative values
    that round to zero give 0x80).
    """
    v = np.asarray(v, dtype=np.float64)
    neg = np.signbit(v)
    a = np.abs(v)
    out = np.zeros(a.shape, dtype=np.int64)
    # subnormal range (and values rounding up into the first normal binade):
    # multiples of 2^-9 below 2^-6.
    sub = a < 2.0 ** -6
    q = np.rint(a[sub] * 2.0 ** 9)          # 0..8; 8 is code 0x08 = 2^-6
    out[sub] = q.astype(np.int64)
    nrm = ~sub
    an = a[nrm]
    mant, ex = np.frexp(an)                 # an = mant * 2^ex, mant in [0.5, 1)
    e = ex - 1                              # floor(log2(an))
    frac = an / np.exp2(e.astype(np.float64))   # in [1, 2), exact
    qm = np.rint((frac - 1.0) * 8.0).astype(np.int64)   # 0..8, ties to even
    carry = qm == 8
    e = np.where(carry, e + 1, e)
    qm = np.where(carry, 0, qm)
    code = ((e + 7) << 3) | qm
    code = np.minimum(code, 0x7E)           # saturate (also catches e+7 > 15)
    out[nrm] = code
    out = np.where(neg, out | 0x80, out)
    return out.astype(np.uint8)


def scale_byte(amax) -> np.ndarray:
    """E8M0 scale byte of a block from its absolute maximum (0 for a zero block)."""
    amax = np.asarray(amax, dtype=np.float64)
    _, ex = np.frexp(amax)
    e = ex.astype(np.int64) - 1             # floor(log2(amax)), exact (subnormals too)
    b = np.clip(e - 8 + 127, 0, 254)
    return np.where(amax > 0, b, 0).astype(np.uint8)


def quantize(v, axis: int = -1):
    """MX-quantise ``v`` along ``axis`` (length a multiple of 32).

    Returns (codes uint8 same shape as v, scales uint8 with that axis / 32).
    """
    v = np.moveaxis(np.asarray(v, dtype=np.float64), axis, -1)
    n = v.shape[-1]
    if n % BLOCK:
        raise ValueError("quantisation axis must be a multiple of 32")
    blk = v.reshape(v.shape[:-1] + (n // BLOCK, BLOCK))
    amax = np.abs(blk).max(axis=-1)
    sb = scale_byte(amax)
    X = np.exp2(sb.astype(np.float64) - 127.0)
    codes = e4m3_encode(blk / X[..., None]).reshape(v.shape)
    return np.moveaxis(codes, -1, axis), np.moveaxis(sb, -1, axis)


def dequantize(codes, scales, axis: int = -1) -> np.ndarray:
    """Exact fp64 value of an MX-quantised tensor."""
    c = np.moveaxis(np.asarray(codes), axis, -1)
    s = np.moveaxis(np.asarray(scales), axis, -1)
    val = e4m3_decode(c)
    X = np.exp2(s.astype(np.float64) - 127.0)
    val = (val.reshape(val.shape[:-1] + (s.shape[-1], BLOCK)) * X[..., None]).reshape(c.shape)
    return np.moveaxis(val, -1, axis)


def roundtrip(v, axis: int = -1) -> np.ndarray:
    """dequantize(quantize(v)): the value an MXFP8 operand carries into a GEMM."""
    q, s = quantize(v, axis)
    return dequantize(q, s, axis)


def quantize_tokens(rows, axis_len_pad: int | None = None):
    """Token-axis quantisation of one expert's rank-ordered rows [n, K].

    Blocks are 32 consecutive ranks of one column; the rank axis is padded
    with zeros to a multiple of 32 (or to ``axis_len_pad``). Returns the
    transposed codes [K, n_pad] and scales [K, n_pad / 32].
    """
    rows = np.asarray(rows, dtype=np.float64)
    n = rows.shape[0]
    n_pad = axis_len_pad if axis_len_pad is not None else -(-n // BLOCK) * BLOCK
    padded = np.zeros((n_pad, rows.shape[1]), np.float64)
    padded[:n] = rows
    return quantize(padded.T, axis=-1)
