"""Pins of the C++ oracle (oracle/cpp/moe_oracle.cpp, via oracle.cxx).

The same closed forms, brute-force searches and invariants that pin the numpy
oracle pin the C++ statement here, piece by piece: the MX codec, the
specified sigmoid, the router's selection, the schedule, one expert's
forward and backward against plain loops, and the identity-expert invariant.
The whole layer is then checked against the numpy oracle (an independent
statement, itself pinned by finite differences): selections bit-exact, and
every bf16 output equal except where the two fp64 sums round to different
sides of a bf16 tie.
"""
import math

import numpy as np
import pytest

import gen
from oracle import cxx
from oracle import layer as OL
from oracle import mxfp8
from oracle import sigmoid as SG
from tests.test_oracle_mxfp8 import _block_closed_form, _brute_encode
from tests.test_oracle_route import _brute_select
from tests.test_oracle_schedule import _brute


# ---------------------------------------------------------------- MX codec
def test_decode_table_and_all_codes():
    table = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x38: 1.0, 0x3C: 1.5,
             0x40: 2.0, 0x7E: 448.0, 0x77: 240.0, 0xB8: -1.0, 0xFE: -448.0}
    for c, v in table.items():
        assert cxx.e4m3_decode(np.array([c], np.uint8))[0] == v, hex(c)
    assert np.isnan(cxx.e4m3_decode(np.array([0x7F, 0xFF], np.uint8))).all()
    finite = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    assert np.array_equal(cxx.e4m3_encode(cxx.e4m3_decode(finite)), finite)


def test_encode_against_brute_force():
    rng = np.random.default_rng(0)
    mags = np.exp2(rng.uniform(-12, 10, 4000)) * rng.choice([-1, 1], 4000)
    vals = mxfp8.e4m3_decode(np.arange(0, 0x7F, dtype=np.uint8))
    mids = (vals[:-1] + vals[1:]) / 2                  # every tie between neighbours
    edges = np.array([0.0, -0.0, 2.0 ** -10, 3 * 2.0 ** -10, 447.9, 448.0, 464.0, 465.0, 1e6, -1e6])
    test = np.concatenate([mags, mids, -mids, edges])
    assert np.array_equal(cxx.e4m3_encode(test), _brute_encode(test))


def test_scale_byte_closed_form():
    amax = np.array([1.0, 448.0, 255.99, 256.0, 0.0, 2.0 ** -130, 2.0 ** -119, 2.0 ** -118, 3.0e38])
    assert cxx.scale_byte(amax).tolist() == [119, 127, 126, 127, 0, 0, 0, 1, 246]


def test_quantize_blocks():
    rng = np.random.default_rng(1)
    v = rng.normal(0, 1, (64, 256)) * np.exp2(rng.integers(-20, 20, (64, 1)))
    v[0, :32] = 0.0
    q, s = cxx.quantize(v)
    X = np.exp2(s.astype(np.float64) - 127)
    blk = v.reshape(64, 8, 32) / X[..., None]
    amax = np.abs(blk).max(-1)
    nz = amax > 0
    assert np.all((amax[nz] >= 256) & (amax[nz] < 512)) and s[0, 0] == 0 and not q[0, :32].any()
    assert np.array_equal(q.reshape(-1), _brute_encode(blk.reshape(-1)))


@pytest.mark.parametrize("n", [1, 33, 45, 96])
def test_token_axis_quantiser(n):
    rng = np.random.default_rng(n)
    rows = rng.normal(size=(n, 64)) * np.exp2(rng.integers(-12, 12, (1, 64)))
    q, s = cxx.quantize_tokens(rows)
    n_pad = -(-n // 32) * 32
    for c in range(0, 64, 7):
        col = np.zeros(n_pad)
        col[:n] = rows[:, c]
        for b in range(n_pad // 32):
            codes, byte = _block_closed_form(col[32 * b:32 * b + 32])
            assert np.array_equal(q[c, 32 * b:32 * b + 32], codes) and s[c, b] == byte


# ---------------------------------------------------------------- router
def test_exp_spec_error_bound_and_sigmoid():
    z = np.linspace(-80, 80, 400001).astype(np.float32)
    ref = np.exp(z.astype(np.float64))
    ulp = np.spacing(ref.astype(np.float32)).astype(np.float64)
    assert (np.abs(cxx.exp_spec(z).astype(np.float64) - ref) / ulp).max() <= 2.0
    l = np.linspace(-30, 30, 20001).astype(np.float32)
    s = cxx.sigmoid_spec(l)
    assert cxx.sigmoid_spec(np.zeros(1, np.float32))[0] == np.float32(0.5)
    assert np.all(np.diff(s.astype(np.float64)) >= 0)
    assert np.max(np.abs(s + cxx.sigmoid_spec(-l) - 1.0)) < 2.5e-7
    # the specification is fixed bit for bit: the two statements agree on every input tried
    wide = np.concatenate([l, np.float32([1e4, -1e4, 80.0, -80.0, 0.5, -0.5])])
    assert np.array_equal(cxx.sigmoid_spec(wide).view(np.uint32), SG.sigmoid_spec(wide).view(np.uint32))


@pytest.mark.parametrize("E,k,G,g_top", [(8, 2, 1, 1), (16, 4, 4, 2)])
def test_select_against_brute_force(E, k, G, g_top):
    rng = np.random.default_rng(E)
    lg = rng.normal(0, 2, (150, E)).astype(np.float32)
    lg[:20, 3] = lg[:20, 5]                            # score ties
    b = rng.normal(0, 0.1, E).astype(np.float32)
    idx, w, s = cxx.select(lg, b, k, G, g_top)
    v = (cxx.sigmoid_spec(lg) + b).astype(np.float32)
    for t in range(150):
        assert list(idx[t]) == _brute_select(v[t], k, G, g_top)
    assert np.all(np.abs(w.astype(np.float64).sum(axis=1) - 1.0) <= k * 2.0 ** -24)
    assert np.array_equal(s, np.take_along_axis(cxx.sigmoid_spec(lg), idx, 1))


def test_all_ties_pick_lowest_indices():
    idx, w, _ = cxx.select(np.zeros((3, 16), np.float32), np.zeros(16, np.float32), 4, 4, 2)
    assert np.array_equal(idx, np.tile(np.arange(4), (3, 1))) and np.all(w == np.float32(0.25))


def test_router_logits_exact_sums():
    rng = np.random.default_rng(4)
    x = rng.normal(size=(6, 40)).astype(np.float32).astype(np.float64)
    wr = rng.normal(0, 0.02, (5, 40)).astype(np.float32).astype(np.float64)
    lg = cxx.router_logits(x, wr)
    for t in range(6):
        for e in range(5):
            assert lg[t, e] == np.float32(math.fsum(x[t, c] * wr[e, c] for c in range(40)))


# ---------------------------------------------------------------- schedule
def test_schedule_against_brute_force():
    rng = np.random.default_rng(0)
    T, k, E, C = 300, 4, 16, 128
    idx = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    idx[:40] = [0, 1, 2, 3]
    sch = cxx.schedule(idx, E, C)
    counts, rank = _brute(idx, E, C)
    assert np.array_equal(sch["counts"], counts) and np.array_equal(sch["rank"], rank)
    assert sorted(sch["pos"].tolist()) == list(range(T * k))
    assert np.array_equal(sch["inv"][sch["pos"]], np.arange(T * k))
    assert sch["offsets"][0] == 0 and np.array_equal(np.diff(sch["offsets"]), counts)


# ---------------------------------------------------------------- one expert against loops
def _mxv(a):
    return mxfp8.roundtrip(np.asarray(a, np.float64), 1)


def test_expert_against_loops():
    """Forward O, dgrad DX and both weight gradients of one expert, each element by plain
    Python loops over the MX values the definition names."""
    rng = np.random.default_rng(3)
    n, d, I = 5, 64, 32
    x = np.float32(rng.normal(size=(n, d))).astype(np.float64)
    dy = np.float32(rng.normal(size=(n, d))).astype(np.float64)
    gate = np.float32(rng.uniform(0.1, 0.9, n))
    w_gu = rng.normal(0, 0.1, (2 * I, d))
    w_d = rng.normal(0, 0.1, (d, I))
    r = cxx.expert(x, dy, gate, w_gu, w_d, nthreads=2)
    xv, wgu, wd = _mxv(x), _mxv(w_gu), _mxv(w_d)
    wdb, wgub = _mxv(w_d.T), _mxv(w_gu.T)
    dyv = _mxv(dy)
    h = np.zeros((n, I))
    gs = np.zeros((n, 2 * I))
    for t in range(n):
        g = np.array([math.fsum(xv[t, c] * wgu[i, c] for c in range(d)) for i in range(I)])
        u = np.array([math.fsum(xv[t, c] * wgu[I + i, c] for c in range(d)) for i in range(I)])
        h[t] = np.float32(g / (1 + np.exp(-g)) * u)
        gs[t] = OL.bf16(np.concatenate([g, u]))
        hq = _mxv(h[t:t + 1])[0]
        o = np.array([math.fsum(hq[i] * wd[c, i] for i in range(I)) for c in range(d)])
        assert np.array_equal(r["O"][t], OL.bf16(o)), t
    dgu = np.zeros((n, 2 * I))
    for t in range(n):
        dh = np.array([math.fsum(dyv[t, c] * wdb[i, c] for c in range(d)) for i in range(I)]) * float(gate[t])
        g, u = gs[t, :I], gs[t, I:]
        sg = 1 / (1 + np.exp(-g))
        dgu[t] = np.float32(np.concatenate([dh * u * sg * (1 + g * (1 - sg)), dh * (g * sg)]))
    dguv = _mxv(dgu)
    for t in range(n):
        dx = np.array([math.fsum(dguv[t, j] * wgub[c, j] for j in range(2 * I)) for c in range(d)])
        assert np.allclose(r["DX"][t], OL.bf16(dx), rtol=2.0 ** -8, atol=0), t
    dO = (gate[:, None] * np.float32(dy)).astype(np.float64)
    dOt, ht = OL.tokq(dO, False).val, OL.tokq(h, False).val
    dgt, xt = OL.tokq(dgu, False).val, OL.tokq(x, False).val
    for c in range(0, d, 9):
        for i in range(0, I, 5):
            assert np.isclose(r["dW_d"][c, i], OL.bf16(math.fsum(dOt[c, m] * ht[i, m] for m in range(dOt.shape[1]))),
                              rtol=2.0 ** -8, atol=0)
    for j in range(0, 2 * I, 7):
        for c in range(0, d, 11):
            assert np.isclose(r["dW_gu"][j, c], OL.bf16(math.fsum(dgt[j, m] * xt[c, m] for m in range(dgt.shape[1]))),
                              rtol=2.0 ** -8, atol=0)


# ---------------------------------------------------------------- whole layer
def _shape(name, T, d, E, k, G, g_top, I, S, C=128):
    return gen.make_shape(name, T, d, E, k, G, g_top, I, S, "zero", 0.05, C=C)


def _inputs(shape, seed=0):
    inp = gen.make_inputs(shape, seed=seed)
    out = {k: v.double().numpy() if v.dtype != np.float32 else v.numpy() for k, v in inp.items()}
    out["bias"] = np.random.default_rng(seed).normal(0, 0.1, shape.E).astype(np.float32)
    return out


def test_identity_experts_make_combine_the_gate_weighted_input():
    """With MX-exact inputs and experts that return their input, y = sum_j w_j x (routed only)."""
    T, d, E, k = 16, 64, 4, 2
    rng = np.random.default_rng(7)
    x = rng.integers(-4, 5, (T, d)).astype(np.float64)              # E4M3-exact, scale 2^0 blocks
    w = rng.dirichlet(np.ones(k), T).astype(np.float32)
    O = np.repeat(x[:, None, :], k, axis=1)
    assert np.array_equal(cxx.combine(w, O), OL.bf16((w.astype(np.float64)[:, :, None] * O).sum(axis=1)))
    assert np.allclose(cxx.combine(w, O), x, rtol=2.0 ** -8)


def _close_bf16(a, b):
    """Equal except where the two fp64 sums straddle a bf16 rounding tie (one bf16 step apart)."""
    a, b = np.asarray(a), np.asarray(b)
    diff = a != b
    if not diff.any():
        return True
    step = np.maximum(np.abs(a), np.abs(b)) * 2.0 ** -7
    return bool(np.all(np.abs(a - b)[diff] <= step[diff]) and diff.mean() < 1e-3)


@pytest.mark.parametrize("dims", [(64, 128, 8, 2, 4, 2, 64, 1), (96, 64, 6, 3, 1, 1, 32, 0)])
def test_layer_agrees_with_numpy_oracle(dims):
    shape = _shape("cx", *dims)
    inp = _inputs(shape, seed=dims[0])
    c = cxx.layer(inp, shape, nthreads=4)
    f = OL.layer_forward(inp, shape)
    b = OL.layer_backward(f, inp, shape)
    assert np.array_equal(c["idx"], f["idx"])
    assert np.array_equal(c["w"].view(np.uint32), f["w"].view(np.uint32))
    assert np.array_equal(c["logits"].view(np.uint32), np.asarray(f["logits"], np.float32).view(np.uint32))
    assert _close_bf16(c["y"], f["y"])
    for key in ("dx", "dW_gu", "dW_d", "dw_router"):
        assert _close_bf16(c[key], b[key]), key
    if shape.S:
        assert _close_bf16(c["dWs_gu"], b["dWs_gu"]) and _close_bf16(c["dWs_d"], b["dWs_d"])


def test_expert_q_on_prepared_weights_equals_expert():
    rng = np.random.default_rng(5)
    n, d, I = 40, 64, 32
    x = np.float32(rng.normal(size=(n, d))).astype(np.float64)
    dy = np.float32(rng.normal(size=(n, d))).astype(np.float64)
    w_gu, w_d = rng.normal(0, 0.1, (2 * I, d)), rng.normal(0, 0.1, (d, I))
    a = cxx.expert(x, dy, None, w_gu, w_d)
    W = cxx.ExpertWeights(w_gu, w_d)
    assert np.array_equal(W.W1, _mxv(w_gu)) and np.array_equal(W.W1b, _mxv(w_gu.T))
    assert np.array_equal(W.W2, _mxv(w_d)) and np.array_equal(W.W2b, _mxv(w_d.T))
    b = cxx.expert_q(x, dy, None, W)
    for key in a:
        assert np.array_equal(a[key], b[key]), key
