"""Seeded synthetic workloads for the DSV3-style MXFP8 MoE layer.

This module only draws random inputs and fixes the layer shapes. It holds
none of the layer's arithmetic (no quantiser, no router, no schedule), so
that the CPU oracle and the CUDA path can both consume its tensors without
sharing any code of the method.

Shapes follow the five workloads of the Mixture-of-Kittens write-ups
(a DeepSeek-V3-style MoE layer in MXFP8; Cursor blog summary, "method
points"), made concrete:

  tiny        T=256    d=256   E=8        k=2 G=1/1 I=128  bias 0
  small       T=4096   d=2048  E=128      k=8 G=1/1 I=768  bias 0
  dsv3_fwd    T=4096   d=7168  E=256 (+1) k=8 G=8/4 I=2048 bias N(0,0.1)
  dsv3_zipf   T=16384  d=7168  E=256 (+1) k=8 G=8/4 I=2048 bias Zipf(1.1), C=640
  e384        T in {512..65536} d=7168 E=384 (+1) k=8 G=1/1 I=2048 bias 0
  dsv3_e64    T=4096   d=7168  E=64 (+1)  k=8 G=8/4 I=2048 bias N(0,0.1)  (profiling case)

Value recipe: x ~ N(0,1), dy ~ N(0,1) (seed+1), router W ~ N(0,0.02),
expert and shared-expert W ~ N(0, w_std); all drawn in fp32 by torch's
seeded generator on the requested device and rounded to bf16.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class LayerShape:
    name: str
    T: int            # tokens
    d: int            # hidden size
    E: int            # routed experts
    k: int            # experts per token
    G: int            # expert groups
    g_top: int        # groups kept per token
    I: int            # expert SwiGLU inner size
    S: int            # shared experts (0 or 1)
    C: int            # ring capacity per expert (multiple of 128)
    bias: str         # "zero" | "normal0.1" | "zipf1.1" | "custom"
    w_std: float      # std of expert weights

    @property
    def assignments(self) -> int:
        return self.T * self.k


def _ceil(a: int, b: int) -> int:
    return -(-a // b) * b


def make_shape(name: str, T: int, d: int, E: int, k: int, G: int, g_top: int,
               I: int, S: int, bias: str, w_std: float, C: int | None = None) -> LayerShape:
    # Default ring capacity per routed expert: twice the mean load, rounded
    # to the 128-row tile (the layer's own default). Hot experts wrap.
    if C is None:
        C = max(128, _ceil(-(-2 * T * k // E), 128))
    return LayerShape(name, T, d, E, k, G, g_top, I, S, C, bias, w_std)


def config(name: str, T: int | None = None) -> LayerShape:
    """The named workloads. ``T`` overrides the token count (e384 sweep)."""
    if name == "tiny":
        return make_shape("tiny", T or 256, 256, 8, 2, 1, 1, 128, 0, "zero", 0.02)
    if name == "small":
        return make_shape("small", T or 4096, 2048, 128, 8, 1, 1, 768, 0, "zero", 0.02)
    if name == "dsv3_fwd":
        return make_shape("dsv3_fwd", T or 4096, 7168, 256, 8, 8, 4, 2048, 1, "normal0.1", 0.006)
    if name == "dsv3_zipf":
        t = T or 16384
        # capacity 1.25 * T * k / E, rounded to the 128-row tile
        cap = _ceil(int(round(1.25 * t * 8 / 256)), 128)
        return make_shape("dsv3_zipf", t, 7168, 256, 8, 8, 4, 2048, 1, "zipf1.1", 0.006, C=cap)
    if name == "dsv3_e64":
        # DSV3 expert shape with a quarter of the experts and tokens: the same mean
        # rows per expert (512) in a few GB, for detailed kernel profiles.
        return make_shape("dsv3_e64", T or 4096, 7168, 64, 8, 8, 4, 2048, 1, "normal0.1", 0.006)
    if name == "e384":
        return make_shape("e384", T or 4096, 7168, 384, 8, 1, 1, 2048, 1, "zero", 0.006)
    raise KeyError(name)


E384_SWEEP = (512, 1024, 2368, 4096, 16384, 65536)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _normal_bf16(shape, std: float, g: torch.Generator, device) -> torch.Tensor:
    return (torch.randn(shape, generator=g, device=device, dtype=torch.float32) * std).to(torch.bfloat16)


def zipf_bias(E: int, s: float, d: int, k: int, seed: int) -> np.ndarray:
    """Per-expert bias that skews expert popularity toward Zipf(s).

    Target share of the expert at popularity rank r is p_r ~ r^-s over a
    seeded random ranking of the experts. The bias is b_e = beta * ln(p_e/p_1).
    beta is picked on a 1024-token calibration batch of synthetic router
    scores (sigmoid of N(0, (0.02*sqrt(d))^2), the logit spread implied by
    x ~ N(0,1) and router W ~ N(0,0.02)), with a plain top-k, by a grid
    search that minimises the L1 gap between realised and target shares.
    This is input preparation only; it does not call the layer's router.
    """
    rng = np.random.default_rng(seed)
    ranks = rng.permutation(E)                      # expert -> popularity rank
    p = (np.arange(1, E + 1, dtype=np.float64)) ** (-s)
    p /= p.sum()
    logp = np.log(p[ranks] / p[0])
    sig = 0.02 * math.sqrt(d)
    scores = 1.0 / (1.0 + np.exp(-rng.normal(0.0, sig, size=(1024, E))))
    target = p[ranks]
    best = (np.inf, 0.0)
    for beta in np.linspace(0.0, 1.0, 101):
        v = scores + beta * logp[None, :]
        top = np.argpartition(-v, k - 1, axis=1)[:, :k]
        share = np.bincount(top.ravel(), minlength=E) / top.size
        gap = np.abs(share - target).sum()
        if gap < best[0] - 1e-12:
            best = (gap, beta)
    return (best[1] * logp).astype(np.float32)


def make_bias(shape: LayerShape, seed: int) -> torch.Tensor:
    if shape.bias == "zero":
        b = np.zeros(shape.E, np.float32)
    elif shape.bias == "normal0.1":
        b = np.random.default_rng(seed + 7).normal(0.0, 0.1, shape.E).astype(np.float32)
    elif shape.bias == "zipf1.1":
        b = zipf_bias(shape.E, 1.1, shape.d, shape.k, seed + 2)
    else:
        raise ValueError(shape.bias)
    return torch.from_numpy(b)


def make_inputs(shape: LayerShape, seed: int = 0, device="cpu", weights: bool = True) -> dict:
    """All layer inputs as torch tensors on ``device``.

    x [T,d] bf16, dy [T,d] bf16, w_router [E,d] bf16, bias [E] f32,
    w_gu [E,2I,d] bf16 (rows 0..I-1 gate, I..2I-1 up), w_d [E,d,I] bf16,
    ws_gu [S,2I,d] bf16, ws_d [S,d,I] bf16.
    Expert weights are drawn one expert at a time to bound temporary memory.
    """
    dev = torch.device(device)
    out = {}
    g = _gen(seed, dev)
    out["x"] = _normal_bf16((shape.T, shape.d), 1.0, g, dev)
    out["w_router"] = _normal_bf16((shape.E, shape.d), 0.02, g, dev)
    out["bias"] = make_bias(shape, seed).to(dev)
    if weights:
        w_gu = torch.empty((shape.E, 2 * shape.I, shape.d), dtype=torch.bfloat16, device=dev)
        w_d = torch.empty((shape.E, shape.d, shape.I), dtype=torch.bfloat16, device=dev)
        for e in range(shape.E):
            w_gu[e] = _normal_bf16((2 * shape.I, shape.d), shape.w_std, g, dev)
            w_d[e] = _normal_bf16((shape.d, shape.I), shape.w_std, g, dev)
        out["w_gu"], out["w_d"] = w_gu, w_d
        ws_gu = torch.empty((shape.S, 2 * shape.I, shape.d), dtype=torch.bfloat16, device=dev)
        ws_d = torch.empty((shape.S, shape.d, shape.I), dtype=torch.bfloat16, device=dev)
        for e in range(shape.S):
            ws_gu[e] = _normal_bf16((2 * shape.I, shape.d), shape.w_std, g, dev)
            ws_d[e] = _normal_bf16((shape.d, shape.I), shape.w_std, g, dev)
        out["ws_gu"], out["ws_d"] = ws_gu, ws_d
    g2 = _gen(seed + 1, dev)
    out["dy"] = _normal_bf16((shape.T, shape.d), 1.0, g2, dev)
    return out


def bf16_to_f32_np(t: torch.Tensor) -> np.ndarray:
    """Host copy of a bf16 tensor as float32 (exact widening)."""
    return t.detach().to("cpu").to(torch.float32).numpy()
