"""Failure detection without a GPU fault: every spin-wait of the library is
bounded, and when one runs out the kernel records MOE_ERR_TIMEOUT and a site
in a status word and returns. The test makes a wait run out on a barrier that
nothing arrives on, reads the status, and checks that the context still runs
the layer afterwards."""
import time

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import moe_layer_dsv3_gb300 as M
    import gen
    from moe_layer_dsv3_gb300.layer import MoELayer
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    t0 = time.time()
    M.moe_selftest_wait_timeout(status.data_ptr(), 200_000_000)       # 0.2 s
    torch.cuda.synchronize()
    assert time.time() - t0 < 5.0
    st = status.cpu().numpy()
    assert st[0] == M.MOE_ERR_TIMEOUT and st[1] == 900
    # the context is still usable: a small layer step runs and reports a clean status
    shape = gen.config("tiny")
    inp = {k: v.cuda() for k, v in gen.make_inputs(shape, seed=0).items()}
    L = MoELayer.from_shape(shape)
    L.quantize_weights(inp["w_gu"], inp["w_d"])
    y = L.forward(inp["x"], inp["w_router"], inp["bias"])
    L.backward(inp["dy"])
    torch.cuda.synchronize()
    assert L.status() == (0, 0)
    assert np.isfinite(y.float().cpu().numpy()).all()


def test_invalid_arguments_rejected_before_launch():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import moe_layer_dsv3_gb300 as M
    cfg = M.config(256, 256, 8, 2)
    with pytest.raises(M.MoeError) as e:
        M.moe_route(cfg, 0, 0, 0, 0, 0, 0)          # null pointers
    assert e.value.code == M.MOE_ERR_INVALID_ARG
    with pytest.raises(M.MoeError):
        M.moe_selftest_wait_timeout(0, 1000)
