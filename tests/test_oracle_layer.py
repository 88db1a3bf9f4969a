"""Pins of the oracle's layer: brute-force loops, invariants, finite differences."""
import numpy as np
import torch

import gen
from oracle import layer as L
from oracle import mxfp8


def _tiny_shape(T=24, d=64, E=8, k=2, G=4, g_top=2, I=32, S=1, C=128):
    return gen.make_shape("pin", T, d, E, k, G, g_top, I, S, "zero", 0.05, C=C)


def _inputs(shape, seed=0, bias_std=0.0):
    inp = gen.make_inputs(shape, seed=seed)
    out = {k: v.to(torch.float64).numpy() for k, v in inp.items()}
    if bias_std:
        out["bias"] = np.random.default_rng(seed).normal(0, bias_std, shape.E).astype(np.float32)
    out["w_router"] = out["w_router"] * 10.0          # spread logits so routes are not near-ties
    return out


def test_expert_ffn_against_loops():
    rng = np.random.default_rng(0)
    n, d, I = 5, 64, 32
    x = rng.normal(size=(n, d))
    w_gu = rng.normal(0, 0.1, (2 * I, d))
    w_d = rng.normal(0, 0.1, (d, I))
    W = L.ExpertWeights(w_gu, w_d)
    xv = mxfp8.roundtrip(x, 1)
    r = L.expert_forward(xv, W)
    wgu = mxfp8.roundtrip(w_gu, 1)
    wd = mxfp8.roundtrip(w_d, 1)
    for t in range(n):
        g = [sum(xv[t, c] * wgu[i, c] for c in range(d)) for i in range(I)]
        u = [sum(xv[t, c] * wgu[I + i, c] for c in range(d)) for i in range(I)]
        h = np.array([np.float32(g[i] / (1 + np.exp(-g[i])) * u[i]) for i in range(I)], np.float64)
        assert np.allclose(r["gu"][t, :I], g, rtol=1e-12, atol=1e-14)
        assert np.allclose(r["gu"][t, I:], u, rtol=1e-12, atol=1e-14)
        assert np.array_equal(r["h"][t], h)
        hq = mxfp8.roundtrip(h[None, :], 1)[0]
        o = [sum(hq[i] * wd[c, i] for i in range(I)) for c in range(d)]
        assert np.allclose(r["o"][t], L.bf16(np.array(o)), rtol=0, atol=0)


def test_bf16_rounding_ties_to_even():
    one = 1.0
    ulp = 2.0 ** -7
    assert L.bf16(one + ulp / 2) == one                 # tie -> even (1.0)
    assert L.bf16(one + 1.5 * ulp) == one + 2 * ulp     # tie -> even (1 + 2 ulp)
    assert L.bf16(one + ulp / 2 + 1e-12) == one + ulp
    assert L.bf16(-3.0) == -3.0 and L.bf16(0.0) == 0.0
    x = np.float32(np.random.default_rng(1).normal(size=1000))
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(L.bf16(x.astype(np.float64)), ref)


def test_identity_experts_make_combine_the_gate_weighted_input():
    shape = _tiny_shape(S=0)
    inp = _inputs(shape)
    f = L.layer_forward(inp, shape)
    T, k = shape.T, shape.k
    O = np.repeat(inp["x"][:, None, :], k, axis=1)     # expert(x) = x for every expert
    y = L.combine(f["w"], O, np.zeros_like(inp["x"]), exact=True)
    assert np.allclose(y, inp["x"], rtol=1e-6, atol=1e-6)
    y2 = L.combine(f["w"], O, np.zeros_like(inp["x"]))  # with the bf16 output rounding
    assert np.max(np.abs(y2 - inp["x"])) <= 2.0 ** -7 * np.max(np.abs(inp["x"]))


def test_forward_structure_quantized():
    shape = _tiny_shape()
    inp = _inputs(shape)
    f = L.layer_forward(inp, shape)
    assert f["y"].shape == (shape.T, shape.d)
    assert np.array_equal(L.bf16(f["y"]), f["y"])
    sch = f["sched"]
    assert sch["counts"].sum() == shape.T * shape.k
    # routed output rows of each expert are the expert applied to its tokens
    e = int(np.argmax(sch["counts"]))
    a = sch["inv"][sch["offsets"][e]:sch["offsets"][e + 1]]
    r = L.expert_forward(f["xq"].val[a // shape.k], f["weights"][e])
    assert np.array_equal(f["O"].reshape(-1, shape.d)[a], r["o"])


def _directional(fn, params, name, direction, eps):
    p = params[name]
    params[name] = p + eps * direction
    lp = fn(params)
    params[name] = p - eps * direction
    lm = fn(params)
    params[name] = p
    return (lp - lm) / (2 * eps)


def test_backward_matches_finite_differences():
    shape = _tiny_shape(T=12, d=32, E=8, k=2, G=4, g_top=2, I=32, S=1)
    inp = _inputs(shape, seed=3, bias_std=0.05)
    f = L.layer_forward(inp, shape, exact=True)
    b = L.layer_backward(f, inp, shape, exact=True)
    idx0 = f["idx"].copy()

    def lossfn(p):
        ff = L.layer_forward(p, shape, exact=True)
        assert np.array_equal(ff["idx"], idx0), "route changed under perturbation"
        return L.loss(ff["y"], p["dy"])

    grads = {"x": b["dx"], "w_router": b["dw_router"], "w_gu": b["dW_gu"], "w_d": b["dW_d"],
             "ws_gu": b["dWs_gu"], "ws_d": b["dWs_d"]}
    rng = np.random.default_rng(7)
    params = dict(inp)
    for name, g in grads.items():
        for _ in range(2):
            dirn = rng.normal(size=g.shape)
            fd = _directional(lossfn, params, name, dirn, 1e-6)
            an = float((g * dirn).sum())
            assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (name, fd, an)
    # the bias only steers selection: a small change leaves the loss unchanged
    fd_b = _directional(lossfn, params, "bias", rng.normal(size=shape.E), 1e-9)
    assert abs(fd_b) < 1e-6


def test_quantized_backward_structure():
    shape = _tiny_shape(T=40, d=64, E=8, k=2, G=1, g_top=1, I=32, S=1)
    inp = _inputs(shape, seed=5)
    f = L.layer_forward(inp, shape)
    b = L.layer_backward(f, inp, shape)
    for key in ("dx", "dw_router", "dW_gu", "dW_d", "dWs_gu", "dWs_d"):
        assert np.array_equal(L.bf16(b[key]), b[key]), key
    # experts with no tokens get an exactly zero weight gradient
    empty = np.flatnonzero(f["sched"]["counts"] == 0)
    for e in empty:
        assert not b["dW_gu"][e].any() and not b["dW_d"][e].any()
    # quantized and exact gradients agree to the MXFP8 noise level
    fe = L.layer_forward(inp, shape, exact=True)
    assert np.array_equal(fe["idx"], f["idx"])
    be = L.layer_backward(fe, inp, shape, exact=True)
    for key in ("dx", "dW_gu", "dW_d"):
        rel = np.linalg.norm(b[key] - be[key]) / np.linalg.norm(be[key])
        assert rel < 0.1, (key, rel)


def test_gate_on_dh_equals_gate_on_dy_for_power_of_two_gates():
    # The expert dgrad quantises each token's dy once and scales dh by the
    # gate. A power-of-two gate moves only the E8M0 scale of MX(w dy), so then
    # MX(w dy) = w MX(dy) exactly and dh must equal the product of the
    # independently quantised w dy rows with W_d, row for row.
    shape = _tiny_shape(T=40, d=64, E=4, k=2, G=1, g_top=1, I=32, S=0)
    inp = _inputs(shape, seed=6)
    f = L.layer_forward(inp, shape)
    rng = np.random.default_rng(8)
    f = dict(f)
    f["w"] = 2.0 ** rng.integers(-3, 2, size=f["w"].shape).astype(np.float64)
    b = L.layer_backward(f, inp, shape)
    sch = f["sched"]
    k = shape.k
    for e in range(shape.E):
        a = sch["inv"][sch["offsets"][e]:sch["offsets"][e + 1]]
        if len(a) == 0:
            continue
        wdy = f["w"].reshape(-1)[a][:, None] * inp["dy"][a // k]
        dh = mxfp8.roundtrip(wdy, 1) @ mxfp8.roundtrip(inp["w_d"][e].T, 1).T    # W_d MX along d
        assert np.allclose(b["experts"][e]["dh"], dh, rtol=1e-12, atol=1e-300), e
    # a gate that is not a power of two moves the codes: the two rounding points differ
    f["w"] = f["w"] * 1.37
    b2 = L.layer_backward(f, inp, shape)
    e = int(np.argmax(sch["counts"]))
    a = sch["inv"][sch["offsets"][e]:sch["offsets"][e + 1]]
    wdy = f["w"].reshape(-1)[a][:, None] * inp["dy"][a // k]
    dh_other = mxfp8.roundtrip(wdy, 1) @ mxfp8.roundtrip(inp["w_d"][e].T, 1).T
    assert not np.allclose(b2["experts"][e]["dh"], dh_other, rtol=1e-9, atol=0)
