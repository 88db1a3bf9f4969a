"""The C++ oracle (oracle/cpp/moe_oracle.cpp) from Python -- TEST INFRASTRUCTURE ONLY.

Argument marshalling for the plain fp64 C++ statement of the layer, with the
same function names and results as the numpy modules beside it (mxfp8,
sigmoid, route, schedule, layer), so that the same pins check both. Only the
tests and the CPU-baseline leg of bench.py use it. Builds the library with
g++ on first use.
"""
from __future__ import annotations

import ctypes
import importlib.util
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))


def _load():
    spec = importlib.util.spec_from_file_location("moe_oracle_build", os.path.join(_HERE, "cpp", "build.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return ctypes.CDLL(mod.build())


_lib = _load()
_P = ctypes.c_void_p
_I = ctypes.c_int
_L = ctypes.c_int64
for _name, _args in {
    "orc_e4m3_encode": [_P, _L, _P], "orc_e4m3_decode": [_P, _L, _P], "orc_scale_byte": [_P, _L, _P],
    "orc_mx_quantize": [_P, _L, _L, _P, _P, _P], "orc_mx_quantize_tokens": [_P, _L, _L, _P, _P],
    "orc_exp_spec": [_P, _L, _P], "orc_sigmoid_spec": [_P, _L, _P],
    "orc_router_logits": [_P, _P, _I, _I, _I, _P, _I],
    "orc_select": [_P, _P, _I, _I, _I, _I, _I, _P, _P, _P],
    "orc_schedule": [_P, _L, _I, _P, _P, _P, _P, _P],
    "orc_expert": [_P, _P, _P, _L, _I, _I, _P, _P, _I, _P, _P, _P, _P],
    "orc_expert_weights": [_P, _P, _I, _I, _I, _P, _P, _P, _P],
    "orc_expert_q": [_P, _P, _P, _L, _I, _I, _P, _P, _P, _P, _I, _P, _P, _P, _P],
    "orc_combine": [_P, _P, _P, _I, _I, _I, _P],
    "orc_router_backward": [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _P],
    "orc_layer": [_I] * 8 + [_P] * 9 + [_I] + [_P] * 10,
    "orc_nvfp4_quantize": [_P, _L, _L, ctypes.c_float, _P, _P], "orc_e2m1_encode": [_P, _L, _P],
}.items():
    getattr(_lib, _name).argtypes = _args
    getattr(_lib, _name).restype = None


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


# ---------------------------------------------------------------- MX codec
def e4m3_encode(v) -> np.ndarray:
    v = _c(v, np.float64)
    out = np.empty(v.shape, np.uint8)
    _lib.orc_e4m3_encode(_p(v), v.size, _p(out))
    return out


def e4m3_decode(codes) -> np.ndarray:
    c = _c(codes, np.uint8)
    out = np.empty(c.shape, np.float64)
    _lib.orc_e4m3_decode(_p(c), c.size, _p(out))
    return out


def scale_byte(amax) -> np.ndarray:
    a = _c(amax, np.float64)
    out = np.empty(a.shape, np.uint8)
    _lib.orc_scale_byte(_p(a), a.size, _p(out))
    return out


def quantize(v, axis: int = -1):
    """MX along ``axis``: (codes, scales) as the numpy oracle returns them."""
    v = np.moveaxis(np.asarray(v, dtype=np.float64), axis, -1)
    if v.shape[-1] % 32:
        raise ValueError("quantisation axis must be a multiple of 32")
    flat = _c(v.reshape(-1, v.shape[-1]), np.float64)
    rows, K = flat.shape
    codes = np.empty((rows, K), np.uint8)
    scales = np.empty((rows, K // 32), np.uint8)
    _lib.orc_mx_quantize(_p(flat), rows, K, _p(codes), _p(scales), None)
    codes = codes.reshape(v.shape)
    scales = scales.reshape(v.shape[:-1] + (K // 32,))
    return np.moveaxis(codes, -1, axis), np.moveaxis(scales, -1, axis)


def quantize_tokens(rows):
    """Token-axis MX of rows [n, K]: codes [K, ceil32(n)], scales [K, ceil32(n) / 32]."""
    r = _c(rows, np.float64)
    n, K = r.shape
    n_pad = -(-n // 32) * 32
    codes = np.empty((K, n_pad), np.uint8)
    scales = np.empty((K, n_pad // 32), np.uint8)
    _lib.orc_mx_quantize_tokens(_p(r), n, K, _p(codes), _p(scales))
    return codes, scales


def e2m1_encode(v) -> np.ndarray:
    v = _c(v, np.float64)
    out = np.empty(v.shape, np.uint8)
    _lib.orc_e2m1_encode(_p(v), v.size, _p(out))
    return out


def nvfp4_quantize(v, g=None):
    """NVFP4 along the last axis: (4-bit codes, E4M3 block scales, tensor scale g)."""
    v = np.asarray(v, dtype=np.float32)
    if g is None:
        amax = np.float32(np.abs(v).max()) if v.size else np.float32(0)
        g = np.float32(amax / np.float32(6 * 448.0)) if amax > 0 else np.float32(1.0)
    flat = _c(v.reshape(-1, v.shape[-1]), np.float32)
    rows, K = flat.shape
    codes = np.empty((rows, K), np.uint8)
    sb = np.empty((rows, K // 16), np.uint8)
    _lib.orc_nvfp4_quantize(_p(flat), rows, K, float(g), _p(codes), _p(sb))
    return codes.reshape(v.shape), sb.reshape(v.shape[:-1] + (K // 16,)), np.float32(g)


# ---------------------------------------------------------------- router
def exp_spec(z) -> np.ndarray:
    z = _c(z, np.float32)
    out = np.empty(z.shape, np.float32)
    _lib.orc_exp_spec(_p(z), z.size, _p(out))
    return out


def sigmoid_spec(l) -> np.ndarray:
    l = _c(l, np.float32)
    out = np.empty(l.shape, np.float32)
    _lib.orc_sigmoid_spec(_p(l), l.size, _p(out))
    return out


def router_logits(x, w_router, nthreads: int = 0) -> np.ndarray:
    x = _c(x, np.float64)
    w = _c(w_router, np.float64)
    T, d = x.shape
    E = w.shape[0]
    out = np.empty((T, E), np.float32)
    _lib.orc_router_logits(_p(x), _p(w), T, d, E, _p(out), nthreads)
    return out


def select(logits, bias, k: int, G: int = 1, g_top: int = 1):
    lg = _c(logits, np.float32)
    b = _c(bias, np.float32)
    T, E = lg.shape
    idx = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float32)
    s = np.empty((T, k), np.float32)
    _lib.orc_select(_p(lg), _p(b), T, E, k, G, g_top, _p(idx), _p(w), _p(s))
    return idx, w, s


def route(x, w_router, bias, k: int, G: int = 1, g_top: int = 1, nthreads: int = 0):
    lg = router_logits(x, w_router, nthreads)
    idx, w, s = select(lg, bias, k, G, g_top)
    return idx, w, s, lg


# ---------------------------------------------------------------- schedule
def schedule(idx, E: int, C: int) -> dict:
    flat = _c(np.asarray(idx).reshape(-1), np.int32)
    A = flat.size
    counts = np.empty(E, np.int64)
    offsets = np.empty(E + 1, np.int64)
    rank = np.empty(A, np.int64)
    pos = np.empty(A, np.int64)
    inv = np.empty(A, np.int64)
    _lib.orc_schedule(_p(flat), A, E, _p(counts), _p(offsets), _p(rank), _p(pos), _p(inv))
    return {"counts": counts, "offsets": offsets, "rank": rank, "pos": pos, "inv": inv,
            "lap": rank // C, "slot": rank % C, "n_laps": int(((counts + C - 1) // C).max()) if A else 0}


# ---------------------------------------------------------------- expert, combine, router backward
def expert(x_rows, dy_rows, gate, w_gu, w_d, nthreads: int = 0) -> dict:
    """One expert's forward and backward on its rows (rank order). ``gate`` [n] fp32 or None (shared)."""
    x = _c(x_rows, np.float64)
    dy = _c(dy_rows, np.float64)
    n, d = x.shape
    wg = _c(w_gu, np.float64)
    wd = _c(w_d, np.float64)
    I = wd.shape[1]
    g = None if gate is None else _c(gate, np.float32)
    out = {"O": np.empty((n, d)), "DX": np.empty((n, d)), "dW_gu": np.empty((2 * I, d)), "dW_d": np.empty((d, I))}
    _lib.orc_expert(_p(x), _p(dy), _p(g), n, d, I, _p(wg), _p(wd), nthreads, _p(out["O"]), _p(out["DX"]),
                    _p(out["dW_gu"]), _p(out["dW_d"]))
    return out


class ExpertWeights:
    """One expert's weights in the four MX orientations (values), prepared once."""

    def __init__(self, w_gu, w_d, nthreads: int = 0):
        wg = _c(w_gu, np.float64)
        wd = _c(w_d, np.float64)
        self.d, self.I = wd.shape
        d, I = self.d, self.I
        self.W1, self.W2 = np.empty((2 * I, d)), np.empty((d, I))
        self.W2b, self.W1b = np.empty((I, d)), np.empty((d, 2 * I))
        _lib.orc_expert_weights(_p(wg), _p(wd), d, I, nthreads, _p(self.W1), _p(self.W2), _p(self.W2b),
                                _p(self.W1b))


def expert_q(x_rows, dy_rows, gate, W: ExpertWeights, nthreads: int = 0) -> dict:
    """expert() on weights prepared by ExpertWeights (the part of a layer step)."""
    x = _c(x_rows, np.float64)
    dy = _c(dy_rows, np.float64)
    n, d = x.shape
    I = W.I
    g = None if gate is None else _c(gate, np.float32)
    out = {"O": np.empty((n, d)), "DX": np.empty((n, d)), "dW_gu": np.empty((2 * I, d)), "dW_d": np.empty((d, I))}
    _lib.orc_expert_q(_p(x), _p(dy), _p(g), n, d, I, _p(W.W1), _p(W.W2), _p(W.W2b), _p(W.W1b), nthreads,
                      _p(out["O"]), _p(out["DX"]), _p(out["dW_gu"]), _p(out["dW_d"]))
    return out


def combine(w, O, S=None) -> np.ndarray:
    w = _c(w, np.float32)
    O = _c(O, np.float64)
    T, k, d = O.shape
    S = None if S is None else _c(S, np.float64)
    y = np.empty((T, d))
    _lib.orc_combine(_p(w), _p(O), _p(S), T, k, d, _p(y))
    return y


def router_backward(dw, w, s_sel, idx, x, w_router, E: int) -> dict:
    dw = _c(dw, np.float64)
    T, k = dw.shape
    x = _c(x, np.float64)
    wr = _c(w_router, np.float64)
    d = x.shape[1]
    out = {"dl": np.empty((T, k)), "dx_r": np.empty((T, d)), "dw_router": np.empty((E, d))}
    _lib.orc_router_backward(_p(dw), _p(_c(w, np.float32)), _p(_c(s_sel, np.float32)), _p(_c(idx, np.int32)),
                             _p(x), _p(wr), T, k, d, E, _p(out["dl"]), _p(out["dx_r"]), _p(out["dw_router"]))
    return out


# ---------------------------------------------------------------- whole layer
def layer(inp: dict, shape, logits=None, nthreads: int = 0) -> dict:
    """Forward and backward of the whole layer. ``inp`` holds the bf16 inputs
    as float arrays (x, dy, w_router, bias, w_gu, w_d, ws_gu, ws_d);
    ``logits`` (fp32 [T, E]) replaces the oracle's own router logits."""
    T, d, E, k, I, S = shape.T, shape.d, shape.E, shape.k, shape.I, shape.S
    f = lambda key: _c(np.asarray(inp[key], dtype=np.float64), np.float64)  # noqa: E731
    x, dy, wr = f("x"), f("dy"), f("w_router")
    w_gu, w_d = f("w_gu"), f("w_d")
    ws_gu = f("ws_gu") if S else np.zeros(1)
    ws_d = f("ws_d") if S else np.zeros(1)
    bias = _c(inp["bias"], np.float32)
    lg_in = None if logits is None else _c(logits, np.float32)
    out = {"idx": np.empty((T, k), np.int32), "w": np.empty((T, k), np.float32),
           "logits": np.empty((T, E), np.float32), "y": np.empty((T, d)), "dx": np.empty((T, d)),
           "dW_gu": np.empty((E, 2 * I, d)), "dW_d": np.empty((E, d, I)),
           "dWs_gu": np.empty((max(S, 1), 2 * I, d)), "dWs_d": np.empty((max(S, 1), d, I)),
           "dw_router": np.empty((E, d))}
    _lib.orc_layer(T, d, E, k, shape.G, shape.g_top, I, S, _p(x), _p(wr), _p(bias), _p(w_gu), _p(w_d), _p(ws_gu),
                   _p(ws_d), _p(dy), _p(lg_in), nthreads, _p(out["idx"]), _p(out["w"]), _p(out["logits"]),
                   _p(out["y"]), _p(out["dx"]), _p(out["dW_gu"]), _p(out["dW_d"]), _p(out["dWs_gu"]),
                   _p(out["dWs_d"]), _p(out["dw_router"]))
    if not S:
        out["dWs_gu"] = out["dWs_gu"][:0]
        out["dWs_d"] = out["dWs_d"][:0]
    return out
