"""GPU parity on the layer's degenerate shapes, end to end against the oracle.

- A single token with one expert per token.
- Every expert picked by every token (k = E), with a shared expert.
- A router whose logits are all zero: every score is a tie, so the
  selection must fall to the lowest indices.
- A capacity of one tile with a long wrap (C = 128 < the busiest expert's rows).

Route indices and counts must be bit-exact. y, dx and the weight gradients
are held to the same bars as the other layer tests: 1e-3 for y, 5e-3 for
gradients (bf16 outputs of MXFP8 products).
"""
import numpy as np
import pytest
import torch

import gen
from oracle import layer as OL
from tests.helpers import np_f64, rel_frob

pytestmark = pytest.mark.gpu


def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")


CASES = {
    "one_token": gen.make_shape("one_token", 1, 128, 4, 1, 1, 1, 128, 0, "zero", 0.05, C=128),
    "all_experts": gen.make_shape("all_experts", 130, 128, 8, 8, 1, 1, 128, 1, "zero", 0.05, C=256),
    "all_ties": gen.make_shape("all_ties", 200, 256, 16, 4, 4, 2, 128, 1, "zero", 0.05, C=128),
    "long_wrap": gen.make_shape("long_wrap", 1000, 128, 4, 2, 1, 1, 128, 0, "zero", 0.05, C=128),
}


@pytest.mark.parametrize("name", list(CASES))
def test_degenerate_shape(name):
    _need_gpu()
    from moe_layer_dsv3_gb300.layer import MoELayer
    s = CASES[name]
    inp = gen.make_inputs(s, seed=3)
    if name == "all_ties":
        inp["w_router"] = torch.zeros_like(inp["w_router"])
    dev = {k: v.cuda() for k, v in inp.items()}
    L = MoELayer.from_shape(s)
    L.quantize_weights(dev["w_gu"], dev["w_d"], dev["ws_gu"], dev["ws_d"])
    L.forward(dev["x"], dev["w_router"], dev["bias"])
    L.backward(dev["dy"])
    torch.cuda.synchronize()
    assert L.status() == (0, 0)
    host = {k: (v.to(torch.float64).numpy() if v.dtype == torch.bfloat16 else v.numpy()) for k, v in inp.items()}
    logits = L.ws_tensor("LOGITS", torch.float32, (s.T, s.E)).cpu().numpy()
    f = OL.layer_forward(host, s, logits=logits)
    b = OL.layer_backward(f, host, s)
    idx = L.topk_idx.cpu().numpy()
    assert np.array_equal(idx, f["idx"])
    counts = L.ws_tensor("COUNTS", torch.int32, (s.E + s.S,)).cpu().numpy()
    assert np.array_equal(counts[:s.E], np.bincount(f["idx"].ravel(), minlength=s.E))
    if name == "all_ties":       # equal scores: the lowest-index groups and experts win
        assert (idx == np.arange(s.k)[None, :]).all()
    if name == "all_experts":    # k = E: each token takes every expert
        assert (np.sort(idx, axis=1) == np.arange(s.E)[None, :]).all()
    if name == "long_wrap":
        assert counts[:s.E].max() > 3 * s.C
    assert rel_frob(np_f64(L.y), f["y"]) < 1e-3
    assert rel_frob(np_f64(L.dx), b["dx"]) < 5e-3
    assert rel_frob(np_f64(L.dw_gu), OL.bf16(b["dW_gu"])) < 5e-3
    assert rel_frob(np_f64(L.dw_d), OL.bf16(b["dW_d"])) < 5e-3
