"""Pins of the oracle's MXFP8 codec against the format's closed forms and brute force."""
import numpy as np
import pytest

from oracle import mxfp8

FINITE = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)


def test_decode_closed_form_values():
    # E4M3: bias 7, subnormal step 2^-9, largest finite 1.75 * 2^8, S.1111.111 NaN
    table = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6,
             0x38: 1.0, 0x3C: 1.5, 0x40: 2.0, 0x7E: 448.0, 0x77: 240.0,
             0xB8: -1.0, 0xFE: -448.0}
    for c, v in table.items():
        assert mxfp8.e4m3_decode(np.uint8(c)) == v, hex(c)
    assert np.isnan(mxfp8.e4m3_decode(np.uint8(0x7F)))
    assert np.isnan(mxfp8.e4m3_decode(np.uint8(0xFF)))
    assert np.signbit(mxfp8.e4m3_decode(np.uint8(0x80)))


def test_code_values_strictly_increasing():
    pos = np.arange(0, 0x7F, dtype=np.uint8)
    v = mxfp8.e4m3_decode(pos)
    assert np.all(np.diff(v) > 0)


def _brute_encode(v):
    """Nearest finite E4M3 value, ties to the code with even mantissa LSB, saturating."""
    pos = np.arange(0, 0x7F, dtype=np.uint8)
    vals = mxfp8.e4m3_decode(pos)
    out = []
    for x in np.atleast_1d(v):
        a = min(abs(x), 448.0)
        dist = np.abs(vals - a)
        best = np.flatnonzero(dist == dist.min())
        if len(best) > 1:
            best = [b for b in best if (pos[b] & 1) == 0]
        c = int(pos[best[0]])
        if np.signbit(x):
            c |= 0x80
        out.append(c)
    return np.array(out, dtype=np.uint8)


def test_encode_matches_brute_force_random():
    rng = np.random.default_rng(0)
    mags = np.exp2(rng.uniform(-12, 10, 4000)) * rng.choice([-1, 1], 4000)
    assert np.array_equal(mxfp8.e4m3_encode(mags), _brute_encode(mags))


def test_encode_ties_and_edges():
    vals = mxfp8.e4m3_decode(np.arange(0, 0x7F, dtype=np.uint8))
    mids = (vals[:-1] + vals[1:]) / 2            # every tie point between neighbours
    edges = np.array([0.0, -0.0, 2.0 ** -10, 2.0 ** -10 * 3, 447.9, 448.0, 456.0, 464.0,
                      465.0, 1e6, -1e6, 2.0 ** -6 - 2.0 ** -11])
    test = np.concatenate([mids, -mids, edges])
    assert np.array_equal(mxfp8.e4m3_encode(test), _brute_encode(test))


def test_encode_decode_roundtrip_all_codes():
    assert np.array_equal(mxfp8.e4m3_encode(mxfp8.e4m3_decode(FINITE)), FINITE)


def test_scale_byte_closed_form():
    # byte = floor(log2 amax) - 8 + 127, clamped to [0, 254]; zero block -> 0
    assert mxfp8.scale_byte(1.0) == 119
    assert mxfp8.scale_byte(448.0) == 127
    assert mxfp8.scale_byte(255.99) == 126
    assert mxfp8.scale_byte(256.0) == 127
    assert mxfp8.scale_byte(0.0) == 0
    assert mxfp8.scale_byte(2.0 ** -130) == 0
    assert mxfp8.scale_byte(2.0 ** -119) == 0
    assert mxfp8.scale_byte(2.0 ** -118) == 1
    assert mxfp8.scale_byte(3.0e38) == 127 + 127 - 8


def test_quantize_block_properties():
    rng = np.random.default_rng(1)
    v = rng.normal(0, 1, (64, 256)) * np.exp2(rng.integers(-20, 20, (64, 1)))
    q, s = mxfp8.quantize(v)
    assert q.shape == v.shape and s.shape == (64, 8)
    X = np.exp2(s.astype(np.float64) - 127)
    blk = v.reshape(64, 8, 32) / X[..., None]
    amax = np.abs(blk).max(-1)
    assert np.all((amax >= 256) & (amax < 512))          # scaled amax lands in [2^8, 2^9)
    # every element is the brute-force nearest E4M3 value of v / X
    assert np.array_equal(q.reshape(-1), _brute_encode(blk.reshape(-1)))
    # round-trip error: within half a grid step, or saturated to 448 X
    deq = mxfp8.dequantize(q, s)
    e = np.floor(np.log2(np.maximum(np.abs(blk), 2.0 ** -6)))
    half_ulp = np.exp2(e - 4) * X[..., None]
    err = np.abs(deq.reshape(64, 8, 32) - v.reshape(64, 8, 32))
    sat = np.abs(blk) > 448
    assert np.all(err[~sat] <= half_ulp[~sat] * (1 + 1e-12))
    assert np.all(np.abs(deq.reshape(64, 8, 32))[sat] == 448 * np.broadcast_to(X[..., None], sat.shape)[sat])


def test_zero_and_power_of_two_blocks():
    v = np.zeros((2, 64))
    v[1, 32:] = 2.0 ** np.arange(-8, 24)[:32].astype(np.float64) * 0 + 4.0
    q, s = mxfp8.quantize(v)
    assert np.all(q[0] == 0) and np.all(s[0] == 0) and np.all(q[1, :32] == 0) and s[1, 0] == 0
    # block of 4.0: byte = 2 - 8 + 127 = 121, 4 / 2^-6 = 256 -> code 0x78 (1.0 * 2^8)
    assert s[1, 1] == 121 and np.all(q[1, 32:] == 0x78)


def test_subnormal_elements():
    v = np.zeros(32)
    v[0] = 448.0
    v[1] = 2.0 ** -9 * 3     # 3 subnormal steps below scale 2^0
    v[2] = 2.0 ** -10        # tie between 0 and 2^-9 -> even (0)
    v[3] = 2.0 ** -10 * 3    # tie between 2^-9 and 2^-8 -> even (2 * 2^-9)
    q, s = mxfp8.quantize(v[None, :])
    assert s[0, 0] == 127
    assert q[0, 0] == 0x7E and q[0, 1] == 0x03 and q[0, 2] == 0x00 and q[0, 3] == 0x02


def test_quantize_axis0_equals_transpose():
    rng = np.random.default_rng(2)
    v = rng.normal(size=(64, 96))
    q0, s0 = mxfp8.quantize(v, axis=0)
    q1, s1 = mxfp8.quantize(v.T, axis=-1)
    assert np.array_equal(q0, q1.T) and np.array_equal(s0, s1.T)


def test_token_axis_zero_padding():
    rng = np.random.default_rng(3)
    rows = rng.normal(size=(45, 64))
    q, s = mxfp8.quantize_tokens(rows)
    assert q.shape == (64, 64) and s.shape == (64, 2)
    assert np.all(q[:, 45:] == 0)
    full = np.zeros((64, 64))
    full[:45] = rows
    q2, s2 = mxfp8.quantize(full.T)
    assert np.array_equal(q, q2) and np.array_equal(s, s2)


def test_rejects_ragged_axis():
    with pytest.raises(ValueError):
        mxfp8.quantize(np.ones((2, 33)))


def _block_closed_form(col):
    """One 32-element block by the format's closed form, element by element in
    Python scalars: scale byte from the exponent of amax, codes by nearest search."""
    import math
    amax = max(abs(float(v)) for v in col)
    if amax == 0.0:
        return np.zeros(32, np.uint8), 0
    e = math.frexp(amax)[1] - 1                     # floor(log2 amax)
    byte = min(max(e - 8 + 127, 0), 254)
    X = 2.0 ** (byte - 127)
    return _brute_encode(np.array([float(v) / X for v in col])), byte


@pytest.mark.parametrize("n", [1, 31, 32, 33, 45, 96])
def test_layer_token_axis_quantiser_against_closed_form(n):
    """oracle.layer.tokq -- the token-axis MX of one expert's rank-ordered rows that
    every weight-gradient reference uses -- against blocks of 32 consecutive ranks of
    one column, zero-padded past the last rank, each quantised by the closed form."""
    from oracle import layer as OL
    rng = np.random.default_rng(n)
    rows = rng.normal(size=(n, 64)) * np.exp2(rng.integers(-12, 12, (1, 64)))
    rows[:, 5] = 0.0                                 # an all-zero column
    q = OL.tokq(rows, exact=False)
    n_pad = -(-n // 32) * 32
    assert q.codes.shape == (64, n_pad) and q.scales.shape == (64, n_pad // 32)
    for c in range(64):
        col = np.zeros(n_pad)
        col[:n] = rows[:, c]
        for b in range(n_pad // 32):
            codes, byte = _block_closed_form(col[32 * b:32 * b + 32])
            assert np.array_equal(q.codes[c, 32 * b:32 * b + 32], codes), (c, b)
            assert q.scales[c, b] == byte, (c, b)
    assert not q.codes[:, n:].any()                  # padding ranks quantise to +0
    deq = mxfp8.e4m3_decode(q.codes) * np.exp2(np.repeat(q.scales.astype(np.float64), 32, axis=1) - 127)
    assert np.array_equal(q.val, deq)
    ex = OL.tokq(rows, exact=True)                   # exact mode: the padded transpose itself
    assert np.array_equal(ex.val[:, :n], rows.T) and not ex.val[:, n:].any()
