"""GPU parity at the workloads' full sizes, in the same launch sequence the
benchmark times (moe_route -> moe_schedule -> moe_forward -> moe_backward).

The oracle cannot run a whole DSV3-size layer, so each check is either
complete but cheap (selection on the GPU's logits for every token, the whole
schedule), or sampled and computed one output at a time by the oracle from
the GPU's own quantised operands: sampled tokens, and the rows, token-axis
operands and weight-gradient rows of sampled experts (the busiest one, whose
rows wrap the ring many times, a median one, and the shared expert).
"""
import gc

import numpy as np
import pytest
import torch

import gen
from oracle import layer as OL
from oracle import mxfp8
from oracle import route as OR
from oracle import schedule as OS
from tests.helpers import gu_split, np_f64, np_u8, rel_frob, untile_scales

pytestmark = pytest.mark.gpu
TOL = 1e-3

# Every configuration of the workload set, the 384-expert shape at each token count of
# its sweep (a few rows per expert at T = 512 up to 1.5K per expert at T = 65536).
WORKLOADS = [("small", None), ("dsv3_fwd", None), ("dsv3_zipf", None)] + \
    [("e384", T) for T in (512, 1024, 2368, 4096, 16384, 65536)]


def _f64(t):
    return t.detach().to("cpu").to(torch.float64).numpy()


def _gu_interleave_rows(I, block=128):
    """Row of the GEMM1 weight blob holding canonical row i of [gate | up] (blocks of 128)."""
    i = np.arange(2 * I)
    up = (i >= I).astype(np.int64)
    ii = i - up * I
    return (ii // block) * (2 * block) + up * block + ii % block


class Full:
    def __init__(self, name, T):
        from moe_layer_dsv3_gb300.layer import MoELayer
        self.shape = s = gen.config(name, T=T)
        self.inp = gen.make_inputs(s, seed=0, device="cuda")
        L = MoELayer.from_shape(s)
        self.L = L
        i = self.inp
        L.quantize_weights(i["w_gu"], i["w_d"], i["ws_gu"], i["ws_d"])
        L.forward(i["x"], i["w_router"], i["bias"])
        L.backward(i["dy"])
        torch.cuda.synchronize()
        self.status = L.status()
        self.Ep, self.A = s.E + s.S, s.T * s.k
        self.Ap = s.T * (s.k + s.S)
        self.Rmax = -(-self.Ap // 128) * 128 + 128 * self.Ep
        self.Tpad = -(-s.T // 128) * 128
        self.logits = L.ws_tensor("LOGITS", torch.float32, (s.T, s.E)).cpu().numpy()
        self.idx = L.topk_idx.cpu().numpy()
        self.w = L.topk_w.cpu().numpy()
        self.bias = i["bias"].cpu().numpy()
        self.wr = _f64(i["w_router"])
        self.sched = OS.schedule(self.idx, s.E, s.C)
        self.poff = L.ws_tensor("POFF", torch.int32, (self.Ep + 1,)).cpu().numpy().astype(np.int64)
        self.rng = np.random.default_rng(1)
        self.tokens = np.sort(self.rng.choice(s.T, min(256, s.T), replace=False))
        counts = self.sched["counts"]
        busiest = int(np.argmax(counts))
        nz = np.flatnonzero(counts)
        median = int(nz[np.argsort(counts[nz])[len(nz) // 2]])
        self.experts = sorted({busiest, median}) + ([s.E] if s.S else [])
        self._w = {}

    def ws(self, name, dtype=torch.uint8, shape=None):
        return self.L.ws_tensor(name, dtype, shape)

    def rows_u8(self, name, rows, cols, sel):
        """Rows `sel` of a [rows][cols] u8 workspace buffer."""
        t = self.ws(name, torch.uint8, (rows, cols))
        return np_u8(t[torch.as_tensor(sel, device=t.device)])

    def rows_sf(self, name, rows, K, sel):
        """Canonical scales of rows `sel` of a tiled-scale buffer (only the atoms touched are read)."""
        t = self.ws(name)
        sel = np.asarray(sel, dtype=np.int64)
        nb = K // 32
        kb = np.arange(nb)[None, :]
        r = sel[:, None]
        off = ((r // 128) * (K // 128) + kb // 4) * 512 + (r % 32) * 16 + ((r // 32) % 4) * 4 + kb % 4
        got = t[torch.as_tensor(off.reshape(-1), device=t.device)].cpu().numpy()
        return got.reshape(len(sel), nb)

    def expert_assignments(self, e):
        s = self.shape
        if e < s.E:
            return OS.expert_rows(self.sched, e)
        return self.A + (e - s.E) * s.T + np.arange(s.T)

    def token_of(self, a):
        s = self.shape
        a = np.asarray(a)
        return np.where(a < self.A, a // s.k, (a - self.A) % s.T)

    def weights(self, e):
        s = self.shape
        if e not in self._w:
            if e < s.E:
                self._w[e] = OL.ExpertWeights(_f64(self.inp["w_gu"][e]), _f64(self.inp["w_d"][e]))
            else:
                self._w[e] = OL.ExpertWeights(_f64(self.inp["ws_gu"][e - s.E]), _f64(self.inp["ws_d"][e - s.E]))
        return self._w[e]


def _release_device_memory():
    gc.collect()
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


@pytest.fixture(scope="module", params=WORKLOADS, ids=lambda p: "%s-%s" % p)
def full(request):
    """One workload on the device at a time: the previous one is released before this
    one is built (a 384-expert layer holds about 100 GB: weights, MX weights, gradients)."""
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    _release_device_memory()
    f = Full(*request.param)
    yield f
    f.L = f.inp = f._w = None
    del f
    _release_device_memory()


def test_status_and_route(full):
    s = full.shape
    assert full.status == (0, 0)
    x_rows = _f64(full.inp["x"][torch.as_tensor(full.tokens, device="cuda")])
    ref = OR.router_logits(x_rows, full.wr)
    assert rel_frob(full.logits[full.tokens], ref) < 1e-5
    idx, w, ssel = OR.select(full.logits, full.bias, s.k, s.G, s.g_top)      # every token
    assert np.array_equal(full.idx, idx)
    assert np.array_equal(full.w.view(np.uint32), w.view(np.uint32))
    g = full.ws("SSEL", torch.float32, (s.T, s.k)).cpu().numpy()
    assert np.array_equal(g.view(np.uint32), ssel.view(np.uint32))


def test_schedule(full):
    s = full.shape
    sch = full.sched
    counts = full.ws("COUNTS", torch.int32, (full.Ep,)).cpu().numpy()
    assert np.array_equal(counts[:s.E], sch["counts"]) and np.all(counts[s.E:] == s.T)
    offs = full.ws("OFFSETS", torch.int32, (full.Ep + 1,)).cpu().numpy()
    assert np.array_equal(offs[:s.E + 1], sch["offsets"])
    for name, ref in (("RANK", sch["rank"]), ("POS", sch["pos"]), ("INV", sch["inv"])):
        got = full.ws(name, torch.int32, (full.Ap,)).cpu().numpy()
        assert np.array_equal(got[:full.A], ref), name
    rs = full.ws("ROWSRC", torch.int32, (full.Rmax,)).cpu().numpy()
    for e in full.experts:
        a = full.expert_assignments(e)
        assert np.array_equal(rs[full.poff[e]:full.poff[e] + len(a)], a)
        assert np.all(rs[full.poff[e] + len(a):full.poff[e + 1]] == -1)
    meta = full.ws("META", torch.int32, (16,)).cpu().numpy()
    assert meta[0] == sch["n_laps"] and meta[1] == full.poff[-1]


def _rank_sample(n):
    """First and last 128 ranks of an expert: its first tile, and its last lap's ragged tail."""
    return np.unique(np.concatenate([np.arange(min(n, 128)), np.arange(max(0, n - 128), n)]))


def test_weight_bytes(full):
    s = full.shape
    I, d = s.I, s.d
    rng = np.random.default_rng(3)
    il = _gu_interleave_rows(I)
    for e in full.experts:
        W = full.weights(e)
        ri = np.sort(rng.choice(2 * I, 32, replace=False))
        rows = e * 2 * I + il[ri]
        assert np.array_equal(full.L.wq_tensor("W1F", (full.Ep * 2 * I, d))[torch.as_tensor(rows, device="cuda")]
                              .cpu().numpy(), W.gu_fwd.codes[ri])
        for name, codes, scales, R, K, n_rows in (("W1F", W.gu_fwd.codes, W.gu_fwd.scales, 2 * I, d, None),
                                                   ("W2F", W.d_fwd.codes, W.d_fwd.scales, d, I, None),
                                                   ("W2B", W.d_bwd.codes, W.d_bwd.scales, I, d, None),
                                                   ("W1B", W.gu_bwd.codes, W.gu_bwd.scales, d, 2 * I, None)):
            r = np.sort(rng.choice(R, 32, replace=False))
            blob_rows = e * R + (il[r] if name == "W1F" else r)
            t = full.L.wq_tensor(name, (full.Ep * R, K))
            assert np.array_equal(t[torch.as_tensor(blob_rows, device="cuda")].cpu().numpy(), codes[r]), name
            sft = full.L.wq_tensor(name + "_SF")
            kb = np.arange(K // 32)[None, :]
            rr = blob_rows[:, None]
            off = ((rr // 128) * (K // 128) + kb // 4) * 512 + (rr % 32) * 16 + ((rr // 32) % 4) * 4 + kb % 4
            got = sft[torch.as_tensor(off.reshape(-1), device="cuda")].cpu().numpy().reshape(len(r), -1)
            assert np.array_equal(got, scales[r]), name + "_SF"


def test_expert_stages(full):
    s = full.shape
    I, d = s.I, s.d
    dy = full.inp["dy"]
    topk_w = full.w.reshape(-1)
    for e in full.experts:
        a = full.expert_assignments(e)
        n = len(a)
        sel = _rank_sample(n)
        prow = full.poff[e] + sel
        tok = full.token_of(a[sel])
        W = full.weights(e)
        x = _f64(full.inp["x"][torch.as_tensor(tok, device="cuda")])
        xq = OL.Q(x, 1, False)
        assert np.array_equal(full.rows_u8("XQ", full.Tpad, d, tok), xq.codes)
        assert np.array_equal(full.rows_sf("XQ_SF", full.Tpad, d, tok), xq.scales)
        # GEMM1 + SwiGLU on identical MX x rows
        r1 = OL.expert_gemm1(xq.val, W)
        gu = gu_split(_f64(full.ws("GU", torch.bfloat16, (full.Rmax, 2 * I))[torch.as_tensor(prow, device="cuda")]), I)
        assert rel_frob(gu, r1["gu_saved"]) < TOL, e
        hq = mxfp8.dequantize(full.rows_u8("HQ", full.Rmax, I, prow), full.rows_sf("HQ_SF", full.Rmax, I, prow), 1)
        assert rel_frob(hq, mxfp8.roundtrip(r1["h"], 1)) < TOL, e
        # GEMM2 on the GPU's MX h
        O = _f64(full.ws("O", torch.bfloat16, (full.Ap, d))[torch.as_tensor(a[sel], device="cuda")])
        assert rel_frob(O, OL.expert_gemm2(hq, W)) < TOL, e
        # backward: MX(dy) rows, dh scaled by the gate, SwiGLU bwd on the GPU's saved g,u, dgrad gate/up
        wa = np.where(a[sel] < full.A, topk_w[np.minimum(a[sel], full.A - 1)], 1.0).astype(np.float32)
        dyr = dy[torch.as_tensor(tok, device="cuda")].float().cpu().numpy().astype(np.float64)
        dOq = OL.Q(dyr, 1, False)
        rb = OL.expert_backward(dOq.val, gu, W, row_gate=wa)
        dgu = mxfp8.dequantize(full.rows_u8("DGU", full.Rmax, 2 * I, prow),
                               full.rows_sf("DGU_SF", full.Rmax, 2 * I, prow), 1)
        assert rel_frob(dgu, mxfp8.roundtrip(rb["dgu"], 1)) < TOL, e
        DX = _f64(full.ws("DXE", torch.bfloat16, (full.Ap, d))[torch.as_tensor(a[sel], device="cuda")])
        assert rel_frob(DX, OL.bf16(dgu @ W.gu_bwd.val.T)) < TOL, e


def test_token_axis_and_wgrad(full):
    s = full.shape
    I, d = s.I, s.d
    rng = np.random.default_rng(4)
    topk_w = full.w.reshape(-1)
    for e in full.experts:
        a = full.expert_assignments(e)
        n = len(a)
        tok = full.token_of(a)
        seg = slice(full.poff[e], full.poff[e + 1])
        npad = full.poff[e + 1] - full.poff[e]
        cs = np.sort(rng.choice(d, 32, replace=False))          # sampled columns of x / dO (rows of the operands)
        xs = full.inp["x"][torch.as_tensor(tok, device="cuda")][:, torch.as_tensor(cs, device="cuda")]
        q, sc = mxfp8.quantize_tokens(_f64(xs), npad)
        assert np.array_equal(full.rows_u8("XTOK", d, full.Rmax, cs)[:, seg], q), e
        assert np.array_equal(full.rows_sf("XTOK_SF", d, full.Rmax, cs)[:, seg.start // 32:seg.stop // 32], sc), e
        wa = np.where(a < full.A, topk_w[np.minimum(a, full.A - 1)], 1.0).astype(np.float32)
        dys = full.inp["dy"][torch.as_tensor(tok, device="cuda")][:, torch.as_tensor(cs, device="cuda")]
        dO = (wa[:, None] * dys.float().cpu().numpy()).astype(np.float64)
        q, sc = mxfp8.quantize_tokens(dO, npad)
        assert np.array_equal(full.rows_u8("DOTOK", d, full.Rmax, cs)[:, seg], q), e
        # weight gradients on the GPU's token-axis operands, sampled rows x columns
        def tokop(name, R, rows):
            c = full.rows_u8(name, R, full.Rmax, rows)[:, seg]
            f = full.rows_sf(name + "_SF", R, full.Rmax, rows)[:, seg.start // 32:seg.stop // 32]
            return mxfp8.dequantize(c, f, 1)
        ri = np.sort(rng.choice(I, 32, replace=False))
        ref = OL.bf16(tokop("DOTOK", d, cs) @ tokop("HTOK", I, ri).T)
        gd = full.L.dw_d[e] if e < s.E else full.L.dws_d[e - s.E]
        got = _f64(gd[torch.as_tensor(cs, device="cuda")][:, torch.as_tensor(ri, device="cuda")])
        if npad == 0:
            assert not got.any()
        else:
            assert rel_frob(got, ref) < TOL, e
        rg = np.sort(rng.choice(2 * I, 32, replace=False))
        ref = OL.bf16(tokop("DGUTOK", 2 * I, rg) @ tokop("XTOK", d, cs).T)
        gg = full.L.dw_gu[e] if e < s.E else full.L.dws_gu[e - s.E]
        got = _f64(gg[torch.as_tensor(rg, device="cuda")][:, torch.as_tensor(cs, device="cuda")])
        assert rel_frob(got, ref) < TOL, e


def test_combine_and_reverse_dispatch(full):
    s = full.shape
    d, k = s.d, s.k
    t = full.tokens
    a = (t[:, None] * k + np.arange(k)[None, :]).reshape(-1)
    ash = full.A + t                                     # shared-expert assignments (S = 1)
    O = full.ws("O", torch.bfloat16, (full.Ap, d))
    Or = _f64(O[torch.as_tensor(a, device="cuda")]).reshape(len(t), k, d)
    Os = _f64(O[torch.as_tensor(ash, device="cuda")]) if s.S else np.zeros((len(t), d))
    y = _f64(full.L.y[torch.as_tensor(t, device="cuda")])
    assert rel_frob(y, OL.combine(full.w[t], Or, Os)) < 1e-4
    DX = full.ws("DXE", torch.bfloat16, (full.Ap, d))
    DXr = _f64(DX[torch.as_tensor(a, device="cuda")]).reshape(len(t), k, d).sum(axis=1)
    DXs = _f64(DX[torch.as_tensor(ash, device="cuda")]) if s.S else 0.0
    dl = full.ws("DL", torch.float32, (s.T, k)).cpu().numpy()[t].astype(np.float64)
    dxr = np.einsum("tj,tjc->tc", dl, full.wr[full.idx[t]])
    dx = _f64(full.L.dx[torch.as_tensor(t, device="cuda")])
    assert rel_frob(dx, OL.bf16(DXr + DXs + dxr)) < TOL


def test_router_backward(full):
    s = full.shape
    t = full.tokens
    dw = full.ws("DW", torch.float32, (s.T, s.k)).cpu().numpy()
    O = full.ws("O", torch.bfloat16, (full.Ap, s.d))
    a = (t[:, None] * s.k + np.arange(s.k)[None, :]).reshape(-1)
    Or = _f64(O[torch.as_tensor(a, device="cuda")]).reshape(len(t), s.k, s.d)
    dy = _f64(full.inp["dy"][torch.as_tensor(t, device="cuda")])
    assert rel_frob(dw[t], np.einsum("tc,tjc->tj", dy, Or)) < 1e-5
    ssel = full.ws("SSEL", torch.float32, (s.T, s.k)).cpu().numpy()
    dl = full.ws("DL", torch.float32, (s.T, s.k)).cpu().numpy()
    rb = OL.router_backward(dw[t], full.w[t], ssel[t], full.idx[t], np.zeros((len(t), 1)), np.zeros((s.E, 1)), s.E)
    assert rel_frob(dl[t], rb["dl"]) < 1e-5
    for e in full.experts:
        if e >= s.E:
            continue
        rows = OS.expert_rows(full.sched, e)
        x = _f64(full.inp["x"][torch.as_tensor(rows // s.k, device="cuda")])
        ref = OL.bf16(dl.reshape(-1)[rows].astype(np.float64) @ x)
        assert rel_frob(_f64(full.L.dw_router[e]), ref) < TOL, e


def _checksum(t):
    """Position-weighted int64 checksum of a tensor's 16-bit words, a few experts at a time."""
    total = 0
    for c in t.view(torch.int16).split(8):
        w = c.reshape(c.shape[0], -1).to(torch.int64)
        total += int((w * torch.arange(1, w.shape[1] + 1, device=w.device) % 65521).sum().item())
        total += int(w.sum().item())
    return total


def test_bitwise_rerun(full):
    L, i = full.L, full.inp
    before = [t.clone() for t in (L.y, L.dx, L.dw_router, L.topk_w)]
    h_gu, h_d = _checksum(L.dw_gu), _checksum(L.dw_d)
    L.forward(i["x"], i["w_router"], i["bias"])
    L.backward(i["dy"])
    torch.cuda.synchronize()
    for a_, b_ in zip(before, (L.y, L.dx, L.dw_router, L.topk_w)):
        assert torch.equal(a_.view(torch.uint8), b_.view(torch.uint8))
    assert _checksum(L.dw_gu) == h_gu
    assert _checksum(L.dw_d) == h_d


def test_walk_order_full_size(full):
    """LAPORDER at full size (17 laps at dsv3_zipf) equals the host model's walk order."""
    from tests.test_ring_protocol import walk_order
    s = full.shape
    counts = [int(c) for c in full.L.ws_tensor("COUNTS", torch.int32, (full.Ep,)).cpu().numpy()]
    ref = walk_order(counts, s.E, s.S, s.C, s.T)
    got = full.L.ws_tensor("LAPORDER", torch.int32, (len(ref),)).cpu().numpy()
    assert np.array_equal(got, np.asarray(ref))


def test_decode_tables_full_size(full):
    """The GEMMs' decode tables at full size equal the host restatement."""
    from tests.test_ring_protocol import decode_tables
    s = full.shape
    counts = [int(c) for c in full.L.ws_tensor("COUNTS", torch.int32, (full.Ep,)).cpu().numpy()]
    ring, push, wg = decode_tables(counts, s.E, s.S, s.C, s.T)
    assert np.array_equal(full.L.ws_tensor("RINGINFO", torch.int32, ring.shape).cpu().numpy(), ring)
    assert np.array_equal(full.L.ws_tensor("PUSHINFO", torch.int32, push.shape).cpu().numpy(), push)
    assert np.array_equal(full.L.ws_tensor("WGINFO", torch.int32, wg.shape).cpu().numpy(), wg)


def test_idle_expert_weight_grads_full_size(full):
    """Experts without tokens get all-zero weight gradients whatever the buffers held (their
    tiles are the weight-gradient kernels' zero tiles), and rewriting the buffers
    from a NaN pattern leaves the other experts' gradient bytes unchanged."""
    L, i = full.L, full.inp
    s = full.shape
    idle = np.flatnonzero(full.sched["counts"][:s.E] == 0)
    h_gu, h_d = _checksum(L.dw_gu), _checksum(L.dw_d)
    L.dw_gu.view(torch.uint8).fill_(0xFF)
    L.dw_d.view(torch.uint8).fill_(0xFF)
    L.backward(i["dy"])
    torch.cuda.synchronize()
    assert L.status() == (0, 0)
    for e in idle:
        assert not L.dw_gu[int(e)].view(torch.int16).any() and not L.dw_d[int(e)].view(torch.int16).any(), e
    assert _checksum(L.dw_gu) == h_gu
    assert _checksum(L.dw_d) == h_d


def test_lap_launch_form_bitwise(full):
    """At full size, with ring wrap-around (17 laps at dsv3_zipf), the per-lap launch form
    (MOE_FLAG_LAP_LAUNCHES: a mover launch and a GEMM launch per lap, laps on two streams)
    gives the same bytes as the default all-laps launch with mover warps."""
    if full.shape.name != "dsv3_zipf" and not (full.shape.name == "e384" and full.shape.T == 2368):
        pytest.skip("the wrap-around workload and one wide one (a second layer at T=65536 does not fit beside this one)")
    import moe_layer_dsv3_gb300 as M
    from moe_layer_dsv3_gb300.layer import MoELayer
    s, i = full.shape, full.inp
    Lp = MoELayer.from_shape(s, flags=M.MOE_FLAG_LAP_LAUNCHES)
    Lp.wq = full.L.wq
    Lp.forward(i["x"], i["w_router"], i["bias"])
    Lp.backward(i["dy"])
    torch.cuda.synchronize()
    assert Lp.status() == (0, 0)
    L = full.L
    for name in ("y", "dx", "dw_router", "dw_gu", "dw_d", "dws_gu", "dws_d"):
        assert torch.equal(getattr(L, name).view(torch.int16), getattr(Lp, name).view(torch.int16)), name
    del Lp
    torch.cuda.empty_cache()


def test_wgrad_pair_form_bitwise(full):
    """At the benchmark workload, the CTA-pair weight-gradient form (MOE_FLAG_WGRAD_PAIR)
    gives the same gradient bytes as the default single-CTA form."""
    if full.shape.name != "dsv3_zipf":
        pytest.skip("the benchmark workload only (a second layer's gradients are 22.5 GB)")
    import moe_layer_dsv3_gb300 as M
    from moe_layer_dsv3_gb300.layer import MoELayer
    s, i = full.shape, full.inp
    L2 = MoELayer.from_shape(s, flags=M.MOE_FLAG_WGRAD_PAIR)
    L2.wq = full.L.wq
    L2.forward(i["x"], i["w_router"], i["bias"])
    L2.backward(i["dy"])
    torch.cuda.synchronize()
    assert L2.status() == (0, 0)
    L = full.L
    for name in ("dw_gu", "dw_d", "dws_gu", "dws_d"):
        assert torch.equal(getattr(L, name).view(torch.int16), getattr(L2, name).view(torch.int16)), name
    del L2
    torch.cuda.empty_cache()


def test_dispatch_alone_fills_the_ring_full_size(full):
    """moe_dispatch (one launch over all laps) leaves the same ring bytes as the forward's mover
    warps, at the workloads with ring wrap-around and at the widest expert count."""
    if full.shape.name not in ("dsv3_zipf", "small") and not (full.shape.name == "e384" and full.shape.T == 2368):
        pytest.skip("the wrap-around workload and two without wrap")
    L, i = full.L, full.inp
    L.ws_tensor("RING_X").fill_(0x5A)
    L.ws_tensor("RING_X_SF").fill_(0x5A)
    L.forward(i["x"], i["w_router"], i["bias"])
    torch.cuda.synchronize()
    ref = L.ws_tensor("RING_X").clone(), L.ws_tensor("RING_X_SF").clone()
    L.ws_tensor("RING_X").fill_(0x5A)
    L.ws_tensor("RING_X_SF").fill_(0x5A)
    L.dispatch(i["x"])
    torch.cuda.synchronize()
    assert L.status() == (0, 0)
    assert torch.equal(L.ws_tensor("RING_X"), ref[0])
    assert torch.equal(L.ws_tensor("RING_X_SF"), ref[1])
    del ref
    torch.cuda.empty_cache()
