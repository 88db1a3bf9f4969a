"""Host-side error paths of the C ABI.

A failed TMA tensor-map encoding is injected on the host
(moe_debug_fail_tensor_maps: nothing reaches the GPU). The entry point that
needed the map must return MOE_ERR_CUDA without launching anything that
depends on the failed GEMM: the router's top-k must not run on stale logits,
combine must not write y, reverse-dispatch must not write dx. The next call,
with no injection, must give the bytes of a clean run, so a failed call
leaves no state behind that corrupts the next one.
"""
import pytest
import torch

import gen

pytestmark = pytest.mark.gpu

# small layer with a shared expert and ring wrap-around (capacity 128 < the hottest count)
SHAPE = gen.make_shape("errpath", 512, 256, 8, 2, 1, 1, 128, 1, "normal0.1", 0.02, C=128)


@pytest.fixture(scope="module")
def env():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import moe_layer_dsv3_gb300 as lib
    from moe_layer_dsv3_gb300.layer import MoELayer
    inp = gen.make_inputs(SHAPE, seed=11, device="cuda")
    L = MoELayer.from_shape(SHAPE)
    L.quantize_weights(inp["w_gu"], inp["w_d"], inp["ws_gu"], inp["ws_d"])
    L.forward(inp["x"], inp["w_router"], inp["bias"])
    L.backward(inp["dy"])
    torch.cuda.synchronize()
    assert L.status() == (0, 0)
    ref = {n: getattr(L, n).clone() for n in ("topk_idx", "topk_w", "y", "dx", "dw_router", "dw_gu", "dw_d",
                                             "dws_gu", "dws_d")}
    yield lib, L, inp, ref
    lib.moe_debug_fail_tensor_maps(0)


def _fails_with_cuda_error(lib, fn):
    lib.moe_debug_fail_tensor_maps(1)
    try:
        with pytest.raises(lib.MoeError) as e:
            fn()
        assert e.value.code == lib.MOE_ERR_CUDA
    finally:
        lib.moe_debug_fail_tensor_maps(0)
    torch.cuda.synchronize()


def _same(a, b):
    return torch.equal(a.view(torch.uint8), b.view(torch.uint8))


def test_route_failed_router_gemm(env):
    lib, L, inp, ref = env
    L.topk_idx.fill_(-7)
    L.topk_w.fill_(-7.0)
    _fails_with_cuda_error(lib, lambda: L.route(inp["x"], inp["w_router"], inp["bias"]))
    assert (L.topk_idx == -7).all() and (L.topk_w == -7.0).all()   # top-k did not run
    L.route(inp["x"], inp["w_router"], inp["bias"])
    torch.cuda.synchronize()
    assert _same(L.topk_idx, ref["topk_idx"]) and _same(L.topk_w, ref["topk_w"])


def test_route_noalloc_failed_router_gemm(env):
    lib, L, inp, ref = env
    cfg = L.cfg
    idx = torch.full_like(ref["topk_idx"], -7)
    w = torch.full_like(ref["topk_w"], -7.0)
    args = (cfg, inp["x"].data_ptr(), inp["w_router"].data_ptr(), inp["bias"].data_ptr(), idx.data_ptr(),
            w.data_ptr())
    _fails_with_cuda_error(lib, lambda: lib.moe_route_noalloc(*args))
    assert (idx == -7).all() and (w == -7.0).all()
    lib.moe_route_noalloc(*args)
    torch.cuda.synchronize()
    assert _same(idx, ref["topk_idx"]) and _same(w, ref["topk_w"])


def test_forward_failed_expert_gemm(env):
    lib, L, inp, ref = env
    L.route(inp["x"], inp["w_router"], inp["bias"])
    L.schedule()
    L.y.fill_(7.0)
    _fails_with_cuda_error(lib, lambda: L.forward_experts(inp["x"]))
    assert (L.y == 7.0).all()                                          # combine did not run
    assert L.status() == (0, 0)
    L.forward_experts(inp["x"])
    torch.cuda.synchronize()
    assert _same(L.y, ref["y"])


def test_backward_failed_dgrad_gemm(env):
    lib, L, inp, ref = env
    L.forward(inp["x"], inp["w_router"], inp["bias"])
    L.dx.fill_(7.0)
    _fails_with_cuda_error(lib, lambda: L.backward(inp["dy"]))
    assert (L.dx == 7.0).all()                                         # reverse-dispatch did not run
    assert L.status() == (0, 0)
    L.backward(inp["dy"])
    torch.cuda.synchronize()
    for name in ("dx", "dw_router", "dw_gu", "dw_d", "dws_gu", "dws_d"):
        assert _same(getattr(L, name), ref[name]), name


def test_plain_gemm_failed_map(env):
    lib, _, _, _ = env
    M = N = K = 128
    a = torch.zeros(M * K, dtype=torch.uint8, device="cuda")
    sf = torch.zeros(M * K // 32, dtype=torch.uint8, device="cuda")
    c = torch.full((M, N), 7.0, dtype=torch.float32, device="cuda")
    call = lambda: lib.moe_gemm_mxfp8(M, N, K, a.data_ptr(), sf.data_ptr(), a.data_ptr(), sf.data_ptr(),
                                      c.data_ptr())
    _fails_with_cuda_error(lib, call)
    assert (c == 7.0).all()
    call()
    torch.cuda.synchronize()
    assert not c.any()                                                  # zero operands: zero product
