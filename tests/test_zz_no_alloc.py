"""moe_route_noalloc: the router for callers that cannot allocate device memory.

Some callers cannot call cudaMalloc: code running while another allocator
(such as a framework's caching allocator) has reserved the GPU's memory, or
code on a path where an allocation's implicit device synchronisation is not
allowed. For them the library keeps the router's fp32 logits in a fixed
16 MiB device array of its own. This file checks, through the C ABI, that two
calls in a row give exactly the indices and gates of moe_route (the route
tests' bar: bit-exact), and that a size beyond the array is refused.
It also checks the entry point as the first library call of a fresh process,
where its first call sets up the array on the device. It sits last in
collection order so that a -x run has run every other test before it.
"""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import gen

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import moe_layer_dsv3_gb300 as m
    return m


def _route_both(lib, shape, seed):
    inp = gen.make_inputs(shape, seed=seed, device="cuda", weights=False)
    cfg = lib.config(shape.T, shape.d, shape.E, shape.k, shape.G, shape.g_top, shape.I, shape.S, shape.C)
    ws = torch.zeros(lib.moe_workspace_size(cfg), dtype=torch.uint8, device="cuda")
    idx_ref = torch.empty((shape.T, shape.k), dtype=torch.int32, device="cuda")
    w_ref = torch.empty((shape.T, shape.k), dtype=torch.float32, device="cuda")
    lib.moe_route(cfg, inp["x"].data_ptr(), inp["w_router"].data_ptr(), inp["bias"].data_ptr(),
                  idx_ref.data_ptr(), w_ref.data_ptr(), ws.data_ptr())
    idx = torch.full((shape.T, shape.k), -1, dtype=torch.int32, device="cuda")
    w = torch.full((shape.T, shape.k), -1.0, dtype=torch.float32, device="cuda")
    lib.moe_route_noalloc(cfg, inp["x"].data_ptr(), inp["w_router"].data_ptr(), inp["bias"].data_ptr(),
                          idx.data_ptr(), w.data_ptr())
    torch.cuda.synchronize()
    return idx_ref.cpu().numpy(), w_ref.cpu().numpy(), idx.cpu().numpy(), w.cpu().numpy()


def test_noalloc_route_matches_route_on_two_calls(lib):
    shapes = [gen.make_shape("na1", 4096, 1024, 256, 8, 8, 4, 128, 1, "normal0.1", 0.02),
              gen.make_shape("na2", 300, 512, 64, 4, 1, 1, 128, 0, "zero", 0.02)]
    for seed, shape in enumerate(shapes):
        idx_ref, w_ref, idx, w = _route_both(lib, shape, seed)
        assert np.array_equal(idx, idx_ref), shape.name
        assert np.array_equal(w.view(np.uint32), w_ref.view(np.uint32)), shape.name


def test_noalloc_route_refuses_oversize(lib):
    cfg = lib.config(16385, 256, 256, 8, 1, 1, 128, 0)      # T * E = 4,194,560 > 4,194,304
    dummy = torch.zeros(16, dtype=torch.uint8, device="cuda")
    p = dummy.data_ptr()
    with pytest.raises(lib.MoeError) as e:
        lib.moe_route_noalloc(cfg, p, p, p, p, p)
    assert e.value.code == lib.MOE_ERR_SCRATCH


_FIRST_CALL = r"""
import sys
import numpy as np
import torch
sys.path.insert(0, sys.argv[1])
import gen
import moe_layer_dsv3_gb300 as lib
shape = gen.make_shape("na_first", 512, 512, 64, 4, 8, 4, 128, 0, "normal0.1", 0.02)
inp = gen.make_inputs(shape, seed=5, device="cuda", weights=False)
cfg = lib.config(shape.T, shape.d, shape.E, shape.k, shape.G, shape.g_top, shape.I, shape.S, shape.C)
args = (inp["x"].data_ptr(), inp["w_router"].data_ptr(), inp["bias"].data_ptr())
outs = []
for _ in range(2):              # the library's first call in this process, then a second one
    idx = torch.full((shape.T, shape.k), -1, dtype=torch.int32, device="cuda")
    w = torch.full((shape.T, shape.k), -1.0, dtype=torch.float32, device="cuda")
    lib.moe_route_noalloc(cfg, *args, idx.data_ptr(), w.data_ptr())
    outs.append((idx, w))
ws = torch.zeros(lib.moe_workspace_size(cfg), dtype=torch.uint8, device="cuda")
idx_ref = torch.empty((shape.T, shape.k), dtype=torch.int32, device="cuda")
w_ref = torch.empty((shape.T, shape.k), dtype=torch.float32, device="cuda")
lib.moe_route(cfg, *args, idx_ref.data_ptr(), w_ref.data_ptr(), ws.data_ptr())
torch.cuda.synchronize()
for idx, w in outs:
    assert torch.equal(idx, idx_ref) and torch.equal(w.view(torch.int32), w_ref.view(torch.int32))
print("first-call OK")
"""


def test_noalloc_route_as_first_library_call(lib):
    """In a fresh process whose first library call is moe_route_noalloc (so that call
    looks up, and under lazy loading reserves, the fixed array), two calls still give
    exactly moe_route's indices and gates."""
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", _FIRST_CALL, root], cwd=root, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0 and "first-call OK" in r.stdout, r.stdout + r.stderr
