"""GPU parity of the standalone kernels against the oracle: MX quantiser
(bit-exact), scale re-tiling (bit-exact), and the tcgen05 MXFP8 GEMM."""
import numpy as np
import pytest
import torch

from oracle import mxfp8
from tests.helpers import np_u8, rel_frob, tile_scales, untile_scales

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import moe_layer_dsv3_gb300 as m
    return m


def _edge_matrix(rows, K, seed):
    rng = np.random.default_rng(seed)
    v = rng.normal(0, 1, (rows, K)) * np.exp2(rng.integers(-30, 30, (rows, 1)))
    v[0, :32] = 0.0                                   # all-zero block
    v[1, :32] = 2.0 ** -130                           # subnormal-range block (bf16 keeps it)
    v[2, :32] = np.linspace(-448, 448, 32)            # exact E4M3 range
    v[3, :32] = 2.0 ** np.arange(-15, 17)             # powers of two over 32 binades
    v[4, :] = -0.0
    t = torch.from_numpy(v.astype(np.float32)).to(torch.bfloat16)
    return t, t.to(torch.float64).numpy()


@pytest.mark.parametrize("rows,K", [(37, 96), (256, 7168), (1, 32)])
def test_quantize_rows_bit_exact(lib, rows, K):
    t, v = _edge_matrix(max(rows, 5), K, 0)
    t, v = t[:rows], v[:rows]
    x = t.cuda()
    codes = torch.empty((rows, K), dtype=torch.uint8, device="cuda")
    sf = torch.empty((rows, K // 32), dtype=torch.uint8, device="cuda")
    lib.moe_quantize_mxfp8(x.data_ptr(), rows, K, 1, codes.data_ptr(), sf.data_ptr())
    torch.cuda.synchronize()
    q, s = mxfp8.quantize(v, axis=1)
    assert np.array_equal(np_u8(sf), s)
    assert np.array_equal(np_u8(codes), q)


@pytest.mark.parametrize("rows,K", [(45, 64), (300, 256)])
def test_quantize_token_axis_bit_exact(lib, rows, K):
    t, v = _edge_matrix(rows, K, 1)
    x = t.cuda()
    rp = -(-rows // 32) * 32
    codes = torch.empty((K, rp), dtype=torch.uint8, device="cuda")
    sf = torch.empty((K, rp // 32), dtype=torch.uint8, device="cuda")
    lib.moe_quantize_mxfp8(x.data_ptr(), rows, K, 0, codes.data_ptr(), sf.data_ptr())
    torch.cuda.synchronize()
    q, s = mxfp8.quantize_tokens(v)
    assert np.array_equal(np_u8(sf), s)
    assert np.array_equal(np_u8(codes), q)


def test_scales_to_tiled(lib):
    rng = np.random.default_rng(2)
    canon = rng.integers(0, 255, (256, 512 // 32)).astype(np.uint8)
    c = torch.from_numpy(canon).cuda()
    out = torch.empty(256 * 512 // 32, dtype=torch.uint8, device="cuda")
    lib.moe_scales_to_tiled(c.data_ptr(), 256, 512, out.data_ptr())
    torch.cuda.synchronize()
    got = np_u8(out)
    assert np.array_equal(got, tile_scales(canon, 256, 512))
    assert np.array_equal(untile_scales(got, 256, 512), canon)


def _gemm_case(lib, M, N, K, seed, unit_scales=False, pair=False):
    rng = np.random.default_rng(seed)
    a = rng.normal(0, 1, (M, K)) * np.exp2(rng.integers(-3, 4, (M, 1)))
    b = rng.normal(0, 1, (N, K)) * np.exp2(rng.integers(-3, 4, (N, 1)))
    if unit_scales:
        a = np.clip(np.round(a * 4) / 4, -8, 8)
        b = np.clip(np.round(b * 4) / 4, -8, 8)
    aq, asf = mxfp8.quantize(a, 1)
    bq, bsf = mxfp8.quantize(b, 1)
    if unit_scales:
        # rescale codes so every block scale is 2^0: values exactly representable as E4M3
        aq = mxfp8.e4m3_encode(a)
        bq = mxfp8.e4m3_encode(b)
        asf = np.full((M, K // 32), 127, np.uint8)
        bsf = np.full((N, K // 32), 127, np.uint8)
    ref = mxfp8.dequantize(aq, asf, 1) @ mxfp8.dequantize(bq, bsf, 1).T
    dev = lambda z: torch.from_numpy(np.ascontiguousarray(z)).cuda()
    A, B = dev(aq), dev(bq)
    Asf, Bsf = dev(tile_scales(asf, M, K)), dev(tile_scales(bsf, N, K))
    C = torch.zeros((M, N), dtype=torch.float32, device="cuda")
    fn = lib.moe_gemm_mxfp8_pair if pair else lib.moe_gemm_mxfp8
    fn(M, N, K, A.data_ptr(), Asf.data_ptr(), B.data_ptr(), Bsf.data_ptr(), C.data_ptr())
    torch.cuda.synchronize()
    return C.cpu().numpy().astype(np.float64), ref


def test_gemm_unit_scales_single_tile(lib):
    got, ref = _gemm_case(lib, 128, 256, 128, 0, unit_scales=True)
    assert rel_frob(got, ref) < 1e-6, rel_frob(got, ref)


@pytest.mark.parametrize("M,N,K", [(128, 256, 128), (256, 512, 512), (384, 128, 1024), (640, 768, 2048)])
def test_gemm_block_scaled(lib, M, N, K):
    got, ref = _gemm_case(lib, M, N, K, M + N + K)
    assert rel_frob(got, ref) < 1e-5, rel_frob(got, ref)


def _block_errors(got, ref):
    """Relative error per (128-row, 64-column) block: locates a wrong operand half."""
    M, N = ref.shape
    out = {}
    for i in range(0, M, 128):
        for j in range(0, N, 64):
            out[(i, j)] = rel_frob(got[i:i + 128, j:j + 64], ref[i:i + 128, j:j + 64])
    return out


@pytest.mark.parametrize("M,N,K", [(256, 128, 128), (512, 256, 384), (768, 384, 1024), (512, 512, 640)])
def test_gemm_pair_block_scaled(lib, M, N, K):
    """The CTA-pair GEMM (256-row tiles over two SMs, 256 or 128 columns, scales per row and
    per 32-block, an odd number of K atoms so the last stage is partial) against the fp64
    product of the dequantised operands, and against the one-CTA GEMM."""
    got, ref = _gemm_case(lib, M, N, K, M + N + K, pair=True)
    err = rel_frob(got, ref)
    assert err < 1e-5, (err, {k: v for k, v in _block_errors(got, ref).items() if v > 1e-5})
    one, _ = _gemm_case(lib, M, N, K, M + N + K)
    assert rel_frob(got, one) < 1e-6


def test_gemm_pair_unit_scales(lib):
    got, ref = _gemm_case(lib, 256, 128, 128, 0, unit_scales=True, pair=True)
    assert rel_frob(got, ref) < 1e-6, rel_frob(got, ref)
