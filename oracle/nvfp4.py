"""NVFP4 (E2M1 elements, E4M3 scale per 16 elements, fp32 tensor scale) -- oracle side.

The write-ups name Cursor's earlier NVFP4 training kernels beside the MXFP8
ones (Cursor blog summary, the opening paragraph) and say nothing more. The
plain reading of "NVFP4" is NVIDIA's 4-bit format:

* element: FP4 E2M1 -- sign, 2 exponent bits (bias 1), 1 mantissa bit; the
  eight magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6; no infinities or NaN;
* block: 16 consecutive elements along the quantisation axis share one
  scale stored as an FP8 E4M3 value (not a power of two);
* tensor: one fp32 scale g for the whole operand, chosen so that the block
  scales fit the E4M3 range: g = amax(tensor) / (6 * 448) (g = 1 for an
  all-zero tensor).

The rounding points are fixed here, in fp32, so that both implementations
take every integer decision on identical fp32 values:

  denom = fp32(6 * g)
  sb    = E4M3_RNE_satfinite( fp32(amax(block) / denom) )   block scale code
  X     = fp32(decode(sb) * g)                                effective scale
  q_i   = E2M1_RNE_satfinite( fp32(v_i / X) )   (0 when X = 0)

The value a GEMM sees is decode(q_i) * decode(sb) * g; the tensor scale g of
each operand is applied once to the fp32 product (alpha = g_a * g_b).
"""
from __future__ import annotations

import numpy as np

from . import mxfp8

E2M1_MAX = 6.0
BLOCK = 16
_E2M1_MAG = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
f32 = np.float32


def e2m1_decode(codes) -> np.ndarray:
    """Decode 4-bit codes (low nibble of each byte) to float64."""
    c = np.asarray(codes, dtype=np.uint8) & 0xF
    mag = _E2M1_MAG[c & 7]
    return np.where(c & 8, -mag, mag)


def e2m1_encode(v) -> np.ndarray:
    """Nearest E2M1 code, ties to the even code (mantissa bit 0), saturating to +-6.
    The sign bit follows the sign of v (so -0.0 gives code 8)."""
    v = np.asarray(v, dtype=np.float64)
    a = np.minimum(np.abs(v), E2M1_MAX)
    # between neighbours m_i < a < m_{i+1}: the nearer; at a tie the even code
    dist = np.abs(a[..., None] - _E2M1_MAG)
    best = dist.min(axis=-1, keepdims=True)
    cand = dist == best
    even = cand & (np.arange(8) % 2 == 0)
    code = np.where(even.any(axis=-1), np.argmax(even, axis=-1), np.argmax(cand, axis=-1))
    return (code | np.where(np.signbit(v), 8, 0)).astype(np.uint8)


def tensor_scale(v) -> np.float32:
    """g = amax / (6 * 448) in fp32 (1 for an all-zero tensor)."""
    amax = f32(np.abs(np.asarray(v, dtype=np.float32)).max()) if np.size(v) else f32(0)
    return f32(amax / f32(E2M1_MAX * 448.0)) if amax > 0 else f32(1.0)


def quantize(v, g=None):
    """NVFP4 along the last axis (length a multiple of 16) of fp32-representable v.

    Returns (codes uint8 one 4-bit code per element, scale codes uint8 E4M3
    [..., K/16], g fp32)."""
    v = np.asarray(v, dtype=np.float32)
    if v.shape[-1] % BLOCK:
        raise ValueError("quantisation axis must be a multiple of 16")
    g = tensor_scale(v) if g is None else f32(g)
    blk = v.reshape(v.shape[:-1] + (v.shape[-1] // BLOCK, BLOCK))
    amax = np.abs(blk).max(axis=-1).astype(np.float32)
    denom = f32(f32(6.0) * g)
    sb = mxfp8.e4m3_encode((amax / denom).astype(np.float32).astype(np.float64))
    X = (mxfp8.e4m3_decode(sb).astype(np.float32) * g).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(X[..., None] > 0, (blk / X[..., None]).astype(np.float32), f32(0.0))
    codes = e2m1_encode(ratio.astype(np.float64)).reshape(v.shape)
    return codes, sb, g


def dequantize(codes, sb, g) -> np.ndarray:
    """Exact value of an NVFP4 operand (fp64)."""
    c = e2m1_decode(codes)
    X = mxfp8.e4m3_decode(sb) * float(g)
    return (c.reshape(c.shape[:-1] + (sb.shape[-1], BLOCK)) * X[..., None]).reshape(c.shape)


def pack(codes) -> np.ndarray:
    """Two 4-bit codes per byte along the last axis: element 2i in the low nibble."""
    c = np.asarray(codes, dtype=np.uint8)
    return (c[..., 0::2] & 0xF) | ((c[..., 1::2] & 0xF) << 4)


def unpack(packed) -> np.ndarray:
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (2 * p.shape[-1],), np.uint8)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = p >> 4
    return out
