"""GPU parity of the NVFP4 quantiser (bit-exact) and the NVFP4 tcgen05 GEMM
(kind::mxf4nvf4) against the oracle's NVFP4 codec and an fp64 product."""
import numpy as np
import pytest
import torch

from oracle import nvfp4 as N
from tests.helpers import np_u8, rel_frob

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import moe_layer_dsv3_gb300 as m
    return m


def _tile16(canon, rows, K):
    """Canonical [rows][K/16] scales -> the tiled atom layout (128 rows x 4 blocks of 16)."""
    nb = K // 16
    out = np.zeros(rows * nb, np.uint8)
    r = np.arange(rows)[:, None]
    kb = np.arange(nb)[None, :]
    off = ((r // 128) * (K // 64) + kb // 4) * 512 + (r % 32) * 16 + ((r // 32) % 4) * 4 + kb % 4
    out[off] = canon
    return out


def _edge(rows, K, seed):
    rng = np.random.default_rng(seed)
    v = rng.normal(0, 1, (rows, K)) * np.exp2(rng.integers(-8, 8, (rows, 1)))
    v[0, :16] = 0.0                                                  # zero block
    v[1, :16] = [6, 5, 3.5, 2.5, 1.75, 1.25, 0.75, 0.25, -0.25, -5, -3.5, 2, -6, 0.5, -0.0, 4]   # E2M1 ties at X = 1
    v[2, :16] = -1e-3                                                # tiny negatives in a block of their own
    v[2, 16:32] = np.linspace(-448, 448, 16)
    t = torch.from_numpy(v.astype(np.float32)).to(torch.bfloat16)
    return t, t.float().numpy()


@pytest.mark.parametrize("rows,K,g", [(37, 96, None), (256, 512, None), (128, 64, 1.0 / 6.0)])
def test_quantize_nvfp4_bit_exact(lib, rows, K, g):
    t, v = _edge(rows, K, rows + K)
    g = N.tensor_scale(v) if g is None else np.float32(g)
    codes, sb, _ = N.quantize(v, g)
    x = t.cuda()
    q = torch.empty((rows, K // 2), dtype=torch.uint8, device="cuda")
    s = torch.empty((rows, K // 16), dtype=torch.uint8, device="cuda")
    lib.moe_quantize_nvfp4(x.data_ptr(), rows, K, float(g), q.data_ptr(), s.data_ptr(), tiled=False)
    torch.cuda.synchronize()
    assert np.array_equal(np_u8(s), sb)
    assert np.array_equal(np_u8(q), N.pack(codes))
    if rows % 128 == 0 and K % 64 == 0:
        st = torch.empty(rows * K // 16, dtype=torch.uint8, device="cuda")
        lib.moe_quantize_nvfp4(x.data_ptr(), rows, K, float(g), q.data_ptr(), st.data_ptr(), tiled=True)
        torch.cuda.synchronize()
        assert np.array_equal(np_u8(st), _tile16(sb, rows, K))


def _gemm_case(lib, M, Nn, K, seed, unit=False):
    rng = np.random.default_rng(seed)
    if unit:
        mags = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6.0])
        a = rng.choice(mags, (M, K)) * rng.choice([-1, 1], (M, K))
        b = rng.choice(mags, (Nn, K)) * rng.choice([-1, 1], (Nn, K))
        a[:, :16] = 6.0                                              # every block's amax is 6: scales 1, g = 1/6
        b[:, :16] = 6.0
    else:
        a = rng.normal(0, 1, (M, K)) * np.exp2(rng.integers(-3, 4, (M, 1)))
        b = rng.normal(0, 1, (Nn, K)) * np.exp2(rng.integers(-3, 4, (Nn, 1)))
    a, b = a.astype(np.float32), b.astype(np.float32)
    qa, sa, ga = N.quantize(a, np.float32(1.0 / 6.0) if unit else None)
    qb, sbb, gb = N.quantize(b, np.float32(1.0 / 6.0) if unit else None)
    ref = N.dequantize(qa, sa, 1.0) @ N.dequantize(qb, sbb, 1.0).T * (float(ga) * float(gb))
    dev = lambda z: torch.from_numpy(np.ascontiguousarray(z)).cuda()   # noqa: E731
    A, B = dev(N.pack(qa)), dev(N.pack(qb))
    Asf, Bsf = dev(_tile16(sa, M, K)), dev(_tile16(sbb, Nn, K))
    C = torch.zeros((M, Nn), dtype=torch.float32, device="cuda")
    alpha = np.float32(np.float32(ga) * np.float32(gb))
    lib.moe_gemm_nvfp4(M, Nn, K, A.data_ptr(), Asf.data_ptr(), B.data_ptr(), Bsf.data_ptr(), float(alpha), C.data_ptr())
    torch.cuda.synchronize()
    return C.cpu().numpy().astype(np.float64), ref


def test_gemm_nvfp4_unit_scales(lib):
    got, ref = _gemm_case(lib, 128, 128, 256, 0, unit=True)
    assert rel_frob(got, ref) < 1e-6, rel_frob(got, ref)


@pytest.mark.parametrize("M,Nn,K", [(128, 128, 256), (256, 256, 512), (384, 512, 1024), (256, 384, 2048)])
def test_gemm_nvfp4_block_scaled(lib, M, Nn, K):
    got, ref = _gemm_case(lib, M, Nn, K, M + Nn + K)
    assert rel_frob(got, ref) < 1e-5, rel_frob(got, ref)


def test_quantise_then_gemm_matches_oracle_chain(lib):
    """bf16 operands -> GPU NVFP4 quantiser -> GPU GEMM, against the oracle's quantiser and
    an fp64 product: the GPU's codes equal the oracle's, so the products agree to fp32 rounding."""
    rng = np.random.default_rng(9)
    M, Nn, K = 256, 256, 1024
    a = torch.from_numpy(rng.normal(size=(M, K)).astype(np.float32)).to(torch.bfloat16)
    b = torch.from_numpy(rng.normal(size=(Nn, K)).astype(np.float32)).to(torch.bfloat16)
    ga, gb = N.tensor_scale(a.float().numpy()), N.tensor_scale(b.float().numpy())
    out = []
    for t, g, rows in ((a, ga, M), (b, gb, Nn)):
        q = torch.empty((rows, K // 2), dtype=torch.uint8, device="cuda")
        s = torch.empty(rows * K // 16, dtype=torch.uint8, device="cuda")
        x = t.cuda()
        lib.moe_quantize_nvfp4(x.data_ptr(), rows, K, float(g), q.data_ptr(), s.data_ptr(), tiled=True)
        out.append((q, s, x))
    C = torch.empty((M, Nn), dtype=torch.float32, device="cuda")
    alpha = float(np.float32(ga) * np.float32(gb))
    lib.moe_gemm_nvfp4(M, Nn, K, out[0][0].data_ptr(), out[0][1].data_ptr(), out[1][0].data_ptr(),
                       out[1][1].data_ptr(), alpha, C.data_ptr())
    torch.cuda.synchronize()
    qa, sa, _ = N.quantize(a.float().numpy(), ga)
    qb, sb, _ = N.quantize(b.float().numpy(), gb)
    ref = N.dequantize(qa, sa, 1.0) @ N.dequantize(qb, sb, 1.0).T * (float(ga) * float(gb))
    assert rel_frob(C.cpu().numpy(), ref) < 1e-5


@pytest.mark.parametrize("Nn,K", [(384, 512), (256, 1024)])
def test_expert_gemm_nvfp4_grouped(lib, Nn, K):
    """The grouped NVFP4 expert GEMM over a real schedule (routed and shared experts, ragged
    counts, one expert without tokens) against per-expert fp64 products of the oracle's codes;
    rows past the last segment stay untouched."""
    import gen
    from moe_layer_dsv3_gb300.layer import MoELayer
    shape = gen.make_shape("nv4g", 300, 256, 8, 2, 1, 1, 128, 1, "normal0.1", 0.02)
    inp = gen.make_inputs(shape, seed=21, device="cuda", weights=False)
    bias = inp["bias"].clone()
    bias[3] = -1.0e4                                                   # expert 3 never selected
    L = MoELayer.from_shape(shape)
    L.route(inp["x"], inp["w_router"], bias)
    L.schedule()
    torch.cuda.synchronize()
    Ep = shape.E + shape.S
    poff = L.ws_tensor("POFF", torch.int32, (Ep + 1,)).cpu().numpy().astype(np.int64)
    counts = L.ws_tensor("COUNTS", torch.int32, (Ep,)).cpu().numpy()
    assert counts[3] == 0 and counts[shape.E] == shape.T
    Rmax = -(-shape.T * (shape.k + shape.S) // 128) * 128 + 128 * Ep
    R = int(poff[Ep])
    rng = np.random.default_rng(Nn + K)
    a = rng.normal(0, 1, (Rmax, K)) * np.exp2(rng.integers(-3, 4, (Rmax, 1)))
    a[R:] = 0.0
    w = rng.normal(0, 1, (Ep * Nn, K)) * np.exp2(rng.integers(-3, 4, (Ep * Nn, 1)))
    qa, sa, ga = N.quantize(a.astype(np.float32))
    qw, sw, gw = N.quantize(w.astype(np.float32))
    dev = lambda z: torch.from_numpy(np.ascontiguousarray(z)).cuda()   # noqa: E731
    A, W = dev(N.pack(qa)), dev(N.pack(qw))
    Asf, Wsf = dev(_tile16(sa, Rmax, K)), dev(_tile16(sw, Ep * Nn, K))
    out = torch.full((Rmax, Nn), 7.0, dtype=torch.float32, device="cuda")
    alpha = np.float32(np.float32(ga) * np.float32(gw))
    lib.moe_expert_gemm_nvfp4(L.cfg, Nn, K, A.data_ptr(), Asf.data_ptr(), W.data_ptr(), Wsf.data_ptr(), float(alpha),
                              out.data_ptr(), L.ws.data_ptr())
    torch.cuda.synchronize()
    got = out.cpu().numpy().astype(np.float64)
    da, dw = N.dequantize(qa, sa, 1.0), N.dequantize(qw, sw, 1.0)
    for e in range(Ep):
        rows = slice(int(poff[e]), int(poff[e + 1]))
        if poff[e + 1] == poff[e]:
            continue
        ref = da[rows] @ dw[e * Nn:(e + 1) * Nn].T * (float(ga) * float(gw))
        assert rel_frob(got[rows], ref) < 1e-5, e
    assert (got[R:] == 7.0).all()
    # the push form (GEMM2's epilogue): each assignment's row is the fp32 product rounded to bf16
    Ap = shape.T * (shape.k + shape.S)
    O = torch.full((Ap, Nn), float("nan"), dtype=torch.bfloat16, device="cuda")
    lib.moe_expert_gemm_nvfp4_push(L.cfg, Nn, K, A.data_ptr(), Asf.data_ptr(), W.data_ptr(), Wsf.data_ptr(),
                                   float(alpha), O.data_ptr(), L.ws.data_ptr())
    torch.cuda.synchronize()
    row_src = L.ws_tensor("ROWSRC", torch.int32, (Rmax,)).cpu().numpy()
    live = np.flatnonzero(row_src >= 0)
    assert len(live) == Ap and sorted(row_src[live]) == list(range(Ap))
    want = out[torch.as_tensor(live, device="cuda")].to(torch.bfloat16)
    assert torch.equal(O[torch.as_tensor(row_src[live], device="cuda").long()].view(torch.int16), want.view(torch.int16))
