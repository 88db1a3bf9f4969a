"""The MoE layer, forward and backward, stated plainly in fp64 -- oracle side.

What the layer is: a DeepSeek-V3-style MoE layer in MXFP8 whose forward
pass dispatches tokens to their experts, runs the expert feed-forward
networks and combines the results, and whose backward pass runs
reverse-combine and reverse-dispatch on the same schedule (Cursor blog
summary, "method points"; techlab report, section on MoK fusing compute and
communication). The write-ups give no formulas; this module takes the plain
reading, with every rounding point the layer materialises:

Forward, per assignment a = (t, j) routed to expert e = idx[t, j]:
  x_q      = MX(x[t]) along d                      (E4M3 + E8M0/32)
  [g | u]  = x_q . W_gu[e]^T,  W_gu MX along d     (fp64 sum of exact products)
  saved    = bf16(g), bf16(u)                      (kept for backward)
  h        = fp32(silu(g) * u)                     (from the unrounded g, u)
  h_q      = MX(h) along I
  O[t, j]  = bf16(h_q . W_d[e]^T),  W_d MX along I
  S[t]     = the same SwiGLU expert on every token with the shared weights
  y[t]     = bf16(sum_j w[t,j] * O[t,j] + S[t])    (fp64 sum)

Backward with upstream gradient dy:
  dw[t,j]  = <dy[t], O[t,j]>                        (fp32 result)
  dy_q     = MX(dy[t]) along d                      (once per token)
  dh       = w[t,j] * (dy_q . W_d[e])   (W_d MX along d; the gate is a per-row
             scalar of the gradient of O[t,j], so it is applied to dh rather
             than quantised into k copies of dy; the write-ups leave the
             rounding point open)
  dO[a]    = fp32(w[t,j] * dy[t]) ; MX along tokens (for dW_d)
  dg       = dh * u * sig(g) * (1 + g (1 - sig(g))),  du = dh * silu(g)
             (g, u the saved bf16 values)
  dGU      = fp32([dg | du]) ; MX along 2I and along tokens
  DX[t,j]  = bf16(dGU_q . W_gu[e])  (W_gu MX along 2I)
  dW_d[e]  = bf16(sum_r dO_tok[r]^T h_tok[r]),  dW_gu[e] = bf16(sum_r dGU_tok[r]^T x_tok[r])
             (token-axis MX: blocks of 32 consecutive ranks, zero-padded tail)
  router:  Z = sum_j s_j ; ds_j = (dw_j - sum_i dw_i w_i) / Z ; dl_j = ds_j s_j (1 - s_j)
           dx_r[t] = sum_j dl_j Wr[idx_j] ; dWr[e] = bf16(sum_{a->e} dl_a x[t_a]) ; no bias grad
  dx[t]    = bf16(sum_j DX[t,j] + DXs[t] + dx_r[t])

``exact=True`` drops every MX and bf16/fp32 rounding (pure fp64 algebra);
the finite-difference tests use it to pin the gradient formulas.
"""
from __future__ import annotations

import numpy as np

from . import mxfp8
from .route import route, select, select_f64, router_logits
from .schedule import schedule, expert_rows


# ---------------------------------------------------------------- roundings
def bf16(a) -> np.ndarray:
    """Round fp64 values to bf16 (nearest, ties to even), returned as fp64."""
    a = np.asarray(a, dtype=np.float64)
    m, e = np.frexp(a)                       # a = m 2^e, |m| in [0.5, 1)
    return np.ldexp(np.rint(m * 256.0) / 256.0, e)


def fp32(a) -> np.ndarray:
    return np.asarray(a, dtype=np.float64).astype(np.float32).astype(np.float64)


class Q:
    """MX quantisation of one operand; in exact mode a pass-through."""

    def __init__(self, v, axis: int, exact: bool):
        v = np.asarray(v, dtype=np.float64)
        if exact:
            self.codes = self.scales = None
            self.val = v
        else:
            self.codes, self.scales = mxfp8.quantize(v, axis)
            self.val = mxfp8.dequantize(self.codes, self.scales, axis)


def tokq(rows, exact: bool):
    """Token-axis MX of rank-ordered rows [n, K] -> object with val [K, n_pad]."""
    rows = np.asarray(rows, dtype=np.float64)
    n = rows.shape[0]
    n_pad = -(-n // 32) * 32
    padded = np.zeros((n_pad, rows.shape[1]))
    padded[:n] = rows
    return Q(padded.T, -1, exact)


def silu(g):
    return g / (1.0 + np.exp(-g))


# ---------------------------------------------------------------- weights
class ExpertWeights:
    """One SwiGLU expert's weights in the four MX orientations the layer uses."""

    def __init__(self, w_gu, w_d, exact: bool = False):
        w_gu = np.asarray(w_gu, dtype=np.float64)    # [2I, d]  rows: gate then up
        w_d = np.asarray(w_d, dtype=np.float64)      # [d, I]
        self.I = w_d.shape[1]
        self.gu_fwd = Q(w_gu, 1, exact)              # along d   (GEMM1, K = d)
        self.d_fwd = Q(w_d, 1, exact)                # along I   (GEMM2, K = I)
        self.d_bwd = Q(w_d.T, 1, exact)              # [I, d] along d   (dgrad of GEMM2, K = d)
        self.gu_bwd = Q(w_gu.T, 1, exact)            # [d, 2I] along 2I (dgrad of GEMM1, K = 2I)


# ---------------------------------------------------------------- expert fwd/bwd
def expert_gemm1(xv, W: ExpertWeights, exact: bool = False) -> dict:
    """GEMM1 + SwiGLU of rank-ordered rows (xv = values of the MX x rows)."""
    gu = xv @ W.gu_fwd.val.T                         # [n, 2I]
    I = W.I
    g, u = gu[:, :I], gu[:, I:]
    h = silu(g) * u
    if not exact:
        h = fp32(h)
    return {"gu": gu, "gu_saved": gu if exact else bf16(gu), "h": h}


def expert_gemm2(hv, W: ExpertWeights, exact: bool = False) -> np.ndarray:
    o = hv @ W.d_fwd.val.T                           # [n, d]
    return o if exact else bf16(o)


def expert_forward(xv, W: ExpertWeights, exact: bool = False) -> dict:
    r = expert_gemm1(xv, W, exact)
    hq = Q(r["h"], 1, exact)
    r["hq"] = hq
    r["o"] = expert_gemm2(hq.val, W, exact)
    return r


def swiglu_bwd(dh, g, u):
    sg = 1.0 / (1.0 + np.exp(-g))
    dg = dh * u * sg * (1.0 + g * (1.0 - sg))
    du = dh * (g * sg)
    return np.concatenate([dg, du], axis=1)


def expert_backward(dOv, gu_saved, W: ExpertWeights, exact: bool = False, row_gate=None) -> dict:
    """dgrad part of one expert: dO values [n, d] -> dh, dGU, dX.

    ``row_gate`` [n], when given, multiplies each row of dh (the routed rows'
    gates; ``dOv`` then holds the token's dy rather than w * dy)."""
    dh = dOv @ W.d_bwd.val.T                         # [n, I]
    if row_gate is not None:
        dh = dh * np.asarray(row_gate, dtype=np.float64)[:, None]
    I = W.I
    dgu = swiglu_bwd(dh, gu_saved[:, :I], gu_saved[:, I:])
    if not exact:
        dgu = fp32(dgu)
    dguq = Q(dgu, 1, exact)
    dx = dguq.val @ W.gu_bwd.val.T                   # [n, d]
    return {"dh": dh, "dgu": dgu, "dguq": dguq, "dx": dx if exact else bf16(dx)}


def wgrad(a_tok: Q, b_tok: Q) -> np.ndarray:
    """sum over ranks of token-axis operands: a_tok.val [M, n], b_tok.val [N, n] -> [M, N]."""
    return a_tok.val @ b_tok.val.T


# ---------------------------------------------------------------- whole layer
def layer_forward(inp: dict, shape, exact: bool = False, logits=None, weights=None) -> dict:
    """Full forward on host arrays. ``inp`` holds float arrays of the bf16 inputs."""
    T, d, E, k = shape.T, shape.d, shape.E, shape.k
    x = np.asarray(inp["x"], dtype=np.float64)
    if exact:
        lg = x @ np.asarray(inp["w_router"], dtype=np.float64).T
        idx, w, s_sel = select_f64(lg, inp["bias"], k, shape.G, shape.g_top)
    elif logits is None:
        idx, w, s_sel, lg = route(x, inp["w_router"], inp["bias"], k, shape.G, shape.g_top)
    else:
        lg = np.asarray(logits, dtype=np.float32)
        idx, w, s_sel = select(lg, inp["bias"], k, shape.G, shape.g_top)
    sch = schedule(idx, E, shape.C)
    if weights is None:
        weights = [ExpertWeights(inp["w_gu"][e], inp["w_d"][e], exact) for e in range(E)]
    shared = [ExpertWeights(inp["ws_gu"][e], inp["ws_d"][e], exact) for e in range(shape.S)]
    xq = Q(x, 1, exact)
    O = np.zeros((T * k, d))
    per_expert = []
    for e in range(E):
        a = expert_rows(sch, e)
        r = expert_forward(xq.val[a // k], weights[e], exact)
        O[a] = r["o"]
        per_expert.append(r)
    S = np.zeros((T, d))
    shared_res = []
    for e in range(shape.S):
        r = expert_forward(xq.val, shared[e], exact)
        S += r["o"]
        shared_res.append(r)
    y = combine(w, O.reshape(T, k, d), S, exact)
    return {"idx": idx, "w": w, "s_sel": s_sel, "logits": lg, "sched": sch, "xq": xq,
            "O": O.reshape(T, k, d), "S": S, "y": y, "experts": per_expert,
            "shared": shared_res, "weights": weights, "shared_weights": shared}


def combine(w, O, S, exact: bool = False) -> np.ndarray:
    """y[t] = sum_j w[t,j] O[t,j] + S[t] in fp64, then bf16 (the layer output)."""
    y = (np.asarray(w, dtype=np.float64)[:, :, None] * np.asarray(O, dtype=np.float64)).sum(axis=1)
    y = y + np.asarray(S, dtype=np.float64)
    return y if exact else bf16(y)


def router_backward(dw, w, s_sel, idx, x, w_router, E: int) -> dict:
    dw = np.asarray(dw, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    s = np.asarray(s_sel, dtype=np.float64)
    Z = s.sum(axis=1, keepdims=True)
    ds = (dw - (dw * w).sum(axis=1, keepdims=True)) / Z
    dl = ds * s * (1.0 - s)
    wr = np.asarray(w_router, dtype=np.float64)
    x = np.asarray(x, dtype=np.float64)
    dx_r = np.einsum("tj,tjc->tc", dl, wr[idx])
    dwr = np.zeros((E, x.shape[1]))
    T, k = idx.shape
    for t in range(T):
        for j in range(k):
            dwr[idx[t, j]] += dl[t, j] * x[t]
    return {"dl": dl, "dx_r": dx_r, "dw_router": dwr}


def layer_backward(fwd: dict, inp: dict, shape, exact: bool = False) -> dict:
    T, d, E, k, I = shape.T, shape.d, shape.E, shape.k, shape.I
    dy = np.asarray(inp["dy"], dtype=np.float64)
    x = np.asarray(inp["x"], dtype=np.float64)
    O = fwd["O"]
    sch = fwd["sched"]
    w = fwd["w"]
    dw = np.einsum("tc,tjc->tj", dy, O)
    if not exact:
        dw = fp32(dw)
    if exact:
        dO = np.asarray(w, dtype=np.float64)[:, :, None] * dy[:, None, :]
    else:
        dO = (np.asarray(w, dtype=np.float32)[:, :, None] * dy.astype(np.float32)[:, None, :]).astype(np.float64)
    dO = dO.reshape(T * k, d)
    gates = (np.asarray(w, dtype=np.float64) if exact else
             np.asarray(w, dtype=np.float32).astype(np.float64)).reshape(T * k)
    DX = np.zeros((T * k, d))
    dW_gu = np.zeros((E, 2 * I, d))
    dW_d = np.zeros((E, d, I))
    per_expert = []
    for e in range(E):
        a = expert_rows(sch, e)
        W = fwd["weights"][e]
        r = fwd["experts"][e]
        dOq = Q(dy[a // k], 1, exact)               # the tokens' MX(dy) rows
        b = expert_backward(dOq.val, r["gu_saved"], W, exact, row_gate=gates[a])
        DX[a] = b["dx"]
        dO_tok = tokq(dO[a], exact)
        h_tok = tokq(r["h"], exact)
        dgu_tok = tokq(b["dgu"], exact)
        x_tok = tokq(x[a // k], exact)
        gd = wgrad(dO_tok, h_tok)
        ggu = wgrad(dgu_tok, x_tok)
        dW_d[e] = gd if exact else bf16(gd)
        dW_gu[e] = ggu if exact else bf16(ggu)
        b.update({"dOq": dOq, "dO_tok": dO_tok, "h_tok": h_tok, "dgu_tok": dgu_tok, "x_tok": x_tok})
        per_expert.append(b)
    DXs = np.zeros((T, d))
    dWs_gu = np.zeros((shape.S, 2 * I, d))
    dWs_d = np.zeros((shape.S, d, I))
    shared = []
    for e in range(shape.S):
        W = fwd["shared_weights"][e]
        r = fwd["shared"][e]
        dOq = Q(dy, 1, exact)
        b = expert_backward(dOq.val, r["gu_saved"], W, exact)
        DXs += b["dx"]
        dO_tok = tokq(dy, exact)
        h_tok = tokq(r["h"], exact)
        dgu_tok = tokq(b["dgu"], exact)
        x_tok = tokq(x, exact)
        gd = wgrad(dO_tok, h_tok)
        ggu = wgrad(dgu_tok, x_tok)
        dWs_d[e] = gd if exact else bf16(gd)
        dWs_gu[e] = ggu if exact else bf16(ggu)
        b.update({"dOq": dOq, "dO_tok": dO_tok, "h_tok": h_tok, "dgu_tok": dgu_tok, "x_tok": x_tok})
        shared.append(b)
    rb = router_backward(dw, w, fwd["s_sel"], fwd["idx"], x, inp["w_router"], E)
    dx = DX.reshape(T, k, d).sum(axis=1) + DXs + rb["dx_r"]
    dwr = rb["dw_router"]
    if not exact:
        dx = bf16(dx)
        dwr = bf16(dwr)
    return {"dw": dw, "dO": dO, "DX": DX.reshape(T, k, d), "DXs": DXs, "dx": dx,
            "dW_gu": dW_gu, "dW_d": dW_d, "dWs_gu": dWs_gu, "dWs_d": dWs_d,
            "dw_router": dwr, "dl": rb["dl"], "dx_r": rb["dx_r"],
            "experts": per_expert, "shared": shared}


def loss(y, dy) -> float:
    """Scalar whose gradient w.r.t. y is dy (used by the finite-difference pins)."""
    return float((np.asarray(y, dtype=np.float64) * np.asarray(dy, dtype=np.float64)).sum())
