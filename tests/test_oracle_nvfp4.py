"""Pins of the NVFP4 codec (numpy and C++ statements) against closed forms and brute force."""
import itertools

import numpy as np
import pytest

from oracle import cxx
from oracle import mxfp8
from oracle import nvfp4 as N


def _closed_form_value(code):
    """E2M1: sign, exponent e (2 bits, bias 1), mantissa m (1 bit); e = 0 is subnormal."""
    s = -1.0 if code & 8 else 1.0
    e, m = (code >> 1) & 3, code & 1
    return s * (m * 0.5 if e == 0 else 2.0 ** (e - 1) * (1 + m / 2))


def _brute_e2m1(x):
    """Nearest E2M1 magnitude by search over the 8 codes, ties to even mantissa, saturating."""
    a = min(abs(x), 6.0)
    vals = [abs(_closed_form_value(c)) for c in range(8)]
    d = [abs(a - v) for v in vals]
    best = [c for c in range(8) if d[c] == min(d)]
    c = [b for b in best if b % 2 == 0][0] if len(best) > 1 else best[0]
    return c | (8 if np.signbit(x) else 0)


def test_decode_closed_form():
    for c in range(16):
        assert N.e2m1_decode(np.uint8(c)) == _closed_form_value(c), c
    assert [abs(_closed_form_value(c)) for c in range(8)] == [0, 0.5, 1, 1.5, 2, 3, 4, 6]


@pytest.mark.parametrize("impl", ["numpy", "cxx"])
def test_encode_brute_force_ties_and_saturation(impl):
    enc = N.e2m1_encode if impl == "numpy" else cxx.e2m1_encode
    mags = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6.0])
    mids = (mags[:-1] + mags[1:]) / 2                       # every tie
    rng = np.random.default_rng(0)
    test = np.concatenate([mags, mids, -mids, rng.uniform(-8, 8, 3000), [6.5, 100.0, -0.0, 1e-30]])
    got = enc(test)
    assert [int(g) for g in got] == [_brute_e2m1(x) for x in test]


@pytest.mark.parametrize("impl", ["numpy", "cxx"])
def test_quantize_block_properties(impl):
    rng = np.random.default_rng(1)
    v = (rng.normal(0, 1, (32, 128)) * np.exp2(rng.integers(-6, 6, (32, 1)))).astype(np.float32)
    v[3, :16] = 0.0                                            # all-zero block
    q = N.quantize if impl == "numpy" else cxx.nvfp4_quantize
    codes, sb, g = q(v)
    assert g == np.float32(np.abs(v).max() / np.float32(6 * 448.0))
    assert sb[3, 0] == 0 and not (codes[3, :16] & 7).any()
    X = mxfp8.e4m3_decode(sb) * float(g)
    amax = np.abs(v.reshape(32, 8, 16)).max(-1).astype(np.float64)
    nz = amax > 0
    # the block scale is the E4M3 value nearest amax / (6 g): within half an E4M3 step
    assert np.all(np.abs(X[nz] * 6 - amax[nz]) <= amax[nz] * 2.0 ** -4 + 1e-30)
    assert mxfp8.e4m3_decode(sb).max() <= 448.0
    # every element: the brute-force nearest E2M1 of fp32(v / X)
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = (v.reshape(32, 8, 16) / X.astype(np.float32)[..., None]).astype(np.float32)
    for (r, b, i) in itertools.product(range(0, 32, 3), range(8), range(16)):
        if X[r, b] > 0:
            assert codes[r, b * 16 + i] == _brute_e2m1(float(ratio[r, b, i])), (r, b, i)
    # round trip: within half an E2M1 step of v / X, or saturated at 6 X
    deq = N.dequantize(codes, sb, g).reshape(32, 8, 16)
    a = np.abs(ratio.astype(np.float64))
    step = np.where(a < 2, 0.5, np.where(a < 4, 1.0, 2.0))
    err = np.abs(deq - v.reshape(32, 8, 16).astype(np.float64)) / np.where(X > 0, X, 1)[..., None]
    assert np.all(err[nz] <= (step / 2 + 1e-6)[nz] + np.maximum(a - 6, 0)[nz])


def test_numpy_and_cxx_agree_bit_for_bit():
    rng = np.random.default_rng(2)
    v = (rng.normal(0, 1, (64, 256)) * np.exp2(rng.integers(-10, 10, (64, 1)))).astype(np.float32)
    a = N.quantize(v)
    b = cxx.nvfp4_quantize(v)
    assert a[2] == b[2] and np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_pack_nibble_order():
    codes = np.arange(16, dtype=np.uint8)[None, :]
    p = N.pack(codes)
    assert p.tolist() == [[0x10, 0x32, 0x54, 0x76, 0x98, 0xBA, 0xDC, 0xFE]]
    assert np.array_equal(N.unpack(p), codes)
