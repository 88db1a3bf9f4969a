"""Router: logits, sigmoid + bias, group-limited top-k, gate normalisation.

The write-ups only say "DeepSeek-V3 (DSV3)-style MoE layer" (Cursor blog
summary, "method points"). The plain reading of a DSV3-style router, as
fixed for this layer:

1. logits l[t,e] = sum_c x[t,c] * Wr[e,c]  (bf16 inputs, exact products,
   fp64 sums, stored as fp32);
2. scores s = sigmoid(l) in the specified fp32 arithmetic (oracle.sigmoid);
3. selection scores v = s + b (fp32), b a per-expert bias that steers
   selection only;
4. with G groups of E/G consecutive experts: group score = sum of the two
   largest v in the group (fp32); keep the g_top best groups, ties to the
   lower group index;
5. pick the k largest v among experts of kept groups, ties to the lower
   expert index; slot j = 0..k-1 lists them by descending v;
6. gates w_j = s_j / sum_j' s_j' (unbiased scores, fp32, the sum taken in
   slot order), routed scaling factor 1, so sum_j w_j = 1.
"""
from __future__ import annotations

import numpy as np

from .sigmoid import sigmoid_spec

f32 = np.float32


def router_logits(x, w_router) -> np.ndarray:
    """fp32 logits [T,E] of bf16-valued x [T,d] and Wr [E,d] (fp64 sums)."""
    x = np.asarray(x, dtype=np.float64)
    w = np.asarray(w_router, dtype=np.float64)
    return (x @ w.T).astype(np.float32)


def _order_desc(v: np.ndarray) -> np.ndarray:
    """Indices sorting the last axis by descending value, ties to lower index."""
    return np.argsort(-v, axis=-1, kind="stable")


def select(logits, bias, k: int, G: int = 1, g_top: int = 1):
    """Steps 2-6 on fp32 logits. Returns (idx int32 [T,k], w f32 [T,k], s_sel f32 [T,k])."""
    logits = np.asarray(logits, dtype=np.float32)
    T, E = logits.shape
    s = sigmoid_spec(logits)
    v = (s + np.asarray(bias, dtype=np.float32)[None, :]).astype(np.float32)
    allowed = np.ones((T, E), dtype=bool)
    if G > 1:
        per = E // G
        vg = v.reshape(T, G, per)
        top2 = np.sort(vg, axis=-1)[..., ::-1][..., :2]
        gscore = (top2[..., 0] + top2[..., 1]).astype(np.float32)    # [T,G]
        keep = _order_desc(gscore)[:, :g_top]
        gmask = np.zeros((T, G), dtype=bool)
        np.put_along_axis(gmask, keep, True, axis=1)
        allowed = np.repeat(gmask, per, axis=1)
    vm = np.where(allowed, v, -np.inf).astype(np.float32)
    idx = _order_desc(vm)[:, :k].astype(np.int32)
    s_sel = np.take_along_axis(s, idx, axis=1).astype(np.float32)
    tot = s_sel[:, 0].copy()
    for j in range(1, k):
        tot = (tot + s_sel[:, j]).astype(np.float32)
    w = (s_sel / tot[:, None]).astype(np.float32)
    return idx, w, s_sel


def route(x, w_router, bias, k: int, G: int = 1, g_top: int = 1):
    """Steps 1-6. Returns (idx, w, s_sel, logits)."""
    lg = router_logits(x, w_router)
    idx, w, s_sel = select(lg, bias, k, G, g_top)
    return idx, w, s_sel, lg


def selection_margin(logits, bias, idx, G: int = 1, g_top: int = 1) -> np.ndarray:
    """Per-token gap between the k-th chosen v and the best unchosen allowed v.

    Used to judge whether an index disagreement is a near-tie.
    """
    s = sigmoid_spec(np.asarray(logits, dtype=np.float32))
    v = (s + np.asarray(bias, dtype=np.float32)[None, :]).astype(np.float64)
    T, E = v.shape
    chosen = np.zeros((T, E), dtype=bool)
    np.put_along_axis(chosen, np.asarray(idx, dtype=np.int64), True, axis=1)
    kth = np.where(chosen, v, np.inf).min(axis=1)
    rest = np.where(chosen, -np.inf, v).max(axis=1)
    return kth - rest


def select_f64(logits, bias, k: int, G: int = 1, g_top: int = 1):
    """The same selection in fp64 with the textbook sigmoid (exact-mode algebra).

    Used only by the finite-difference pins, where scores must be smooth
    functions of the logits.
    """
    l = np.asarray(logits, dtype=np.float64)
    T, E = l.shape
    s = 1.0 / (1.0 + np.exp(-l))
    v = s + np.asarray(bias, dtype=np.float64)[None, :]
    allowed = np.ones((T, E), dtype=bool)
    if G > 1:
        per = E // G
        top2 = np.sort(v.reshape(T, G, per), axis=-1)[..., ::-1][..., :2]
        keep = _order_desc(top2.sum(axis=-1))[:, :g_top]
        gmask = np.zeros((T, G), dtype=bool)
        np.put_along_axis(gmask, keep, True, axis=1)
        allowed = np.repeat(gmask, per, axis=1)
    idx = _order_desc(np.where(allowed, v, -np.inf))[:, :k].astype(np.int32)
    s_sel = np.take_along_axis(s, idx, axis=1)
    w = s_sel / s_sel.sum(axis=1, keepdims=True)
    return idx, w, s_sel
