#!/usr/bin/env python
"""Benchmark of the MXFP8 DSV3-style MoE layer, forward + backward, on GB300.

One step = route -> schedule -> forward -> backward of one synthetic batch
(every row of the hot path). Prints ONE JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload dsv3_zipf|dsv3_fwd|small|tiny|e384] [--T tokens]

N > 1 runs under torch.distributed.run, one rank per GPU, each rank an
independent replica of the layer on its own batch ("replicas only": the
layer has no exchange step on one GPU, so no collective is on the data path;
scaling is weak). `--impl reference` times the C++ fp64 CPU oracle on a
bounded sample of the same workload on all host cores.
"""
from __future__ import annotations

import argparse
import atexit
import dataclasses
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import gen  # noqa: E402

METRIC = "MoE-layer tokens/s fwd+bwd MXFP8 (1xGB300)"


# ---------------------------------------------------------------- helpers
PEAK_FILE = os.path.join(ROOT, "profiles", "mxfp8_peak.json")


def peaks():
    """Roofline denominators: HBM and bf16 from MEASURED_PEAKS.json (else the
    recipe's fallback); dense MXFP8 from the library GEMM measured by
    `bench.py --probe-peak` (profiles/mxfp8_peak.json) when present, else
    2 x the sustained bf16 figure (the nominal fp8/bf16 ratio)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        pk = {"hbm_gbs": d["hbm_gbs"], "bf16": d["bf16_tflops"], "bf16_sus": d["bf16_tflops_sustained"],
              "src": "measured"}
    else:
        pk = {"hbm_gbs": 6800.0, "bf16": 1900.0, "bf16_sus": 1700.0, "src": "fallback"}
    pk["fp8"] = 2.0 * pk["bf16_sus"]
    pk["fp8_note"] = ("dense MXFP8 = 2 x %s sustained bf16 (%s TFLOP/s), the nominal fp8/bf16 ratio"
                      % ("measured" if pk["src"] == "measured" else "fallback", pk["bf16_sus"]))
    if os.path.exists(PEAK_FILE):
        with open(PEAK_FILE) as f:
            m = json.load(f)
        lib = m.get("library") or {}
        if lib.get("tflops_sustained"):
            pk["fp8"] = lib["tflops_sustained"]
            pk["fp8_note"] = ("measured MXFP8: %s, %s, sustained (profiles/mxfp8_peak.json)"
                              % (lib.get("name"), lib.get("shape")))
    return pk


def probe_peak(args):
    """Dense MXFP8 GEMM throughput on this GPU: a library GEMM (cuBLASLt through
    torch._scaled_mm with E8M0 block scales, 32 elements per scale) and this
    repo's own plain tcgen05 GEMM (moe_gemm_mxfp8), at M = N = K = n. Burst =
    best of 10 launches; sustained = back-to-back launches for ~4 s."""
    import moe_layer_dsv3_gb300 as M
    n = args.probe_n
    dev = "cuda"
    torch.manual_seed(0)
    a8 = (torch.randn(n, n, device=dev) * 0.5).to(torch.float8_e4m3fn)
    b8 = (torch.randn(n, n, device=dev) * 0.5).to(torch.float8_e4m3fn)
    flop = 2.0 * n ** 3

    def timeit(fn):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        best = None
        for _ in range(10):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            t = e0.elapsed_time(e1)
            best = t if best is None else min(best, t)
        reps = max(1, int(4000.0 / best))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        sus = e0.elapsed_time(e1) / reps
        return flop / (best / 1e3) / 1e12, flop / (sus / 1e3) / 1e12

    out = {"n": n, "gpu": torch.cuda.get_device_name(0), "torch": torch.__version__}
    clocks = ClockSampler(0)
    # library: MX block scales, all 2^0 (E8M0 byte 127), one per 32 elements along K
    lib = {"name": "cuBLASLt via torch._scaled_mm (E4M3 x E4M3, E8M0 scale per 32 along K)",
           "shape": "M=N=K=%d" % n}
    try:
        sa = torch.full((n, n // 32), 127, dtype=torch.uint8, device=dev).view(torch.float8_e8m0fnu)
        sb = torch.full((n, n // 32), 127, dtype=torch.uint8, device=dev).view(torch.float8_e8m0fnu)
        fn = lambda: torch._scaled_mm(a8, b8.t(), sa, sb, out_dtype=torch.bfloat16)  # noqa: E731
        ref = fn().float()
        chk = (a8.float() @ b8.float().t())
        lib["rel_err"] = float((ref - chk).norm() / chk.norm())
        lib["tflops_burst"], lib["tflops_sustained"] = timeit(fn)
    except Exception as e:   # record why the library path is unavailable
        lib["error"] = "%s: %s" % (type(e).__name__, str(e)[:300])
    out["library"] = lib
    # this repo's plain MXFP8 GEMM (fp32 output)
    ours = {"name": "moe_gemm_mxfp8 (tcgen05 kind::mxf8f6f4.block_scale, fp32 out)", "shape": "M=N=K=%d" % n}
    sf = torch.full((n * n // 32,), 127, dtype=torch.uint8, device=dev)
    c = torch.empty((n, n), dtype=torch.float32, device=dev)
    sp = torch.cuda.current_stream().cuda_stream
    fn = lambda: M.moe_gemm_mxfp8(n, n, n, a8.data_ptr(), sf.data_ptr(), b8.data_ptr(), sf.data_ptr(),  # noqa: E731
                                  c.data_ptr(), sp)
    fn()
    torch.cuda.synchronize()
    ours["rel_err"] = float((c - a8.float() @ b8.float().t()).norm() / (a8.float() @ b8.float().t()).norm())
    ours["tflops_burst"], ours["tflops_sustained"] = timeit(fn)
    out["ours"] = ours
    # this repo's NVFP4 GEMM (E2M1 codes, E4M3 scale per 16; all scales 1, alpha 1)
    nv = {"name": "moe_gemm_nvfp4 (tcgen05 kind::mxf4nvf4.block_scale.scale_vec::4X, fp32 out)",
          "shape": "M=N=K=%d" % n}
    a4 = torch.randint(0, 256, (n, n // 2), dtype=torch.uint8, device=dev)
    b4 = torch.randint(0, 256, (n, n // 2), dtype=torch.uint8, device=dev)
    sf4 = torch.full((n * n // 16,), 0x38, dtype=torch.uint8, device=dev)     # E4M3 1.0
    fn = lambda: M.moe_gemm_nvfp4(n, n, n, a4.data_ptr(), sf4.data_ptr(), b4.data_ptr(), sf4.data_ptr(),  # noqa: E731
                                  1.0, c.data_ptr(), sp)
    nv["tflops_burst"], nv["tflops_sustained"] = timeit(fn)
    out["ours_nvfp4"] = nv
    del a4, b4, sf4, c
    # the grouped NVFP4 expert GEMM over a real schedule (dsv3_e64 routing), GEMM2's
    # shape: rank rows x d, K = I; FLOPs on the T*(k+S) assignment rows only
    from moe_layer_dsv3_gb300.layer import MoELayer
    shp = gen.config("dsv3_e64")
    inp = gen.make_inputs(shp, seed=0, device=dev, weights=False)
    L = MoELayer.from_shape(shp)
    L.route(inp["x"], inp["w_router"], inp["bias"])
    L.schedule()
    Ep = shp.E + shp.S
    Rmax = -(-shp.T * (shp.k + shp.S) // 128) * 128 + 128 * Ep
    Ng, Kg = shp.d, shp.I
    ag = torch.randint(0, 256, (Rmax, Kg // 2), dtype=torch.uint8, device=dev)
    wg = torch.randint(0, 256, (Ep * Ng, Kg // 2), dtype=torch.uint8, device=dev)
    sfa = torch.full((Rmax * Kg // 16,), 0x38, dtype=torch.uint8, device=dev)
    sfw = torch.full((Ep * Ng * Kg // 16,), 0x38, dtype=torch.uint8, device=dev)
    og = torch.empty((Rmax, Ng), dtype=torch.float32, device=dev)
    fn = lambda: M.moe_expert_gemm_nvfp4(L.cfg, Ng, Kg, ag.data_ptr(), sfa.data_ptr(), wg.data_ptr(),  # noqa: E731
                                         sfw.data_ptr(), 1.0, og.data_ptr(), L.ws.data_ptr(), sp)
    flop_g = 2.0 * shp.T * (shp.k + shp.S) * Ng * Kg
    b, su = timeit(fn)
    out["ours_nvfp4_grouped"] = {
        "name": "moe_expert_gemm_nvfp4 (grouped over the schedule, fp32 rank-ordered rows)",
        "shape": "dsv3_e64 routing: %d assignment rows x N=%d x K=%d, %d experts" % (shp.T * (shp.k + shp.S), Ng, Kg, Ep),
        "tflops_burst": b * flop_g / flop, "tflops_sustained": su * flop_g / flop}
    # the same product with GEMM2's epilogue: bf16 rows pushed to their assignments
    ob = torch.empty((shp.T * (shp.k + shp.S), Ng), dtype=torch.bfloat16, device=dev)
    fn = lambda: M.moe_expert_gemm_nvfp4_push(L.cfg, Ng, Kg, ag.data_ptr(), sfa.data_ptr(), wg.data_ptr(),  # noqa: E731
                                              sfw.data_ptr(), 1.0, ob.data_ptr(), L.ws.data_ptr(), sp)
    b, su = timeit(fn)
    out["ours_nvfp4_push"] = {
        "name": "moe_expert_gemm_nvfp4_push (grouped over the schedule, bf16 rows pushed to their assignments)",
        "shape": out["ours_nvfp4_grouped"]["shape"],
        "tflops_burst": b * flop_g / flop, "tflops_sustained": su * flop_g / flop}
    out["clocks"] = clocks.stop()
    print(json.dumps(out), flush=True)


def gemm_flops(shape):
    """Algorithmic FLOPs per step of each grouped GEMM (rows = all expert assignments)."""
    R = shape.T * (shape.k + shape.S)
    d, I = shape.d, shape.I
    return {
        "gemm1_fwd": 2.0 * R * 2 * I * d,
        "gemm2_fwd": 2.0 * R * d * I,
        "gemm_dgrad_down": 2.0 * R * I * d,
        "gemm_dgrad_gu": 2.0 * R * d * 2 * I,
        "gemm_wgrad_d": 2.0 * d * I * R,
        "gemm_wgrad_gu": 2.0 * 2 * I * d * R,
        "router_gemm": 2.0 * shape.T * shape.E * d,
    }


def hbm_bytes(shape):
    """Algorithmic bytes per step of the memory-bound kernels: every tensor a
    kernel needs read once and every output written once. A gather reads each
    source row once however many rows it is copied to (the repeats come from
    L2), so its bytes are the source once plus the gathered rows written."""
    T, d, k, S, E = shape.T, shape.d, shape.k, shape.S, shape.E
    Rr = T * k                    # routed rows (ring traffic)
    R = T * (k + S)
    row_q = d + d // 32           # one MX row (codes + scales)
    return {
        "permute_lap": T * row_q + Rr * row_q,
        "combine": T * (k + S) * d * 2.0 + T * k * 4.0 + T * d * 2.0,
        "rev_combine_dw": T * k * d * 2.0 + T * d * 2.0 + T * k * 12.0,
        "permute_lap_dO": T * row_q + Rr * row_q,
        "reverse_dispatch": T * (k + S) * d * 2.0 + T * k * 12.0 + T * d * 2.0,
        "tok_gather_x": T * d * 2.0 + R * row_q,
        "tok_gather_dO": T * d * 2.0 + R * row_q,
        "quant_rows": 2 * (T * d * 2.0 + T * row_q),          # MX(x) forward, MX(dy) backward
        # dh fp32 and saved g|u bf16 in; dGU codes + scales out along 2I and along ranks
        "swiglu_bwd_quant": R * (shape.I * 4.0 + 2 * shape.I * 2.0 + 2 * (2 * shape.I + 2 * shape.I / 32.0)),
    }


class ClockSampler:
    """nvidia-smi clock / throttle samples, every 50 ms with their timestamps.

    Start it before the warm-up (nvidia-smi takes a moment to start), bracket
    the timed region with window(), and stop() keeps the samples taken inside
    that window. A window shorter than the sampling period may hold none: the
    samples nearest to it are kept then, and "in_window" says so.
    """

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.path = None
        self.t0 = self.t1 = None
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=self.fh, stderr=subprocess.DEVNULL)
            atexit.register(self._end)   # no sampler outlives the bench, even one that raised before stop()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _end(self):
        if self.proc is not None and self.proc.poll() is None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def window(self, start: bool):
        if start:
            self.t0 = time.time()
        else:
            self.t1 = time.time()

    @staticmethod
    def _when(stamp):
        import datetime
        try:
            return datetime.datetime.strptime(stamp.strip(), "%Y/%m/%d %H:%M:%S.%f").timestamp()
        except ValueError:
            return None

    def stop(self):
        if self.proc is None:
            return None
        self._end()
        self.fh.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [q.strip() for q in line.split(",")]
                if len(parts) >= 10:
                    rows.append((self._when(parts[0]), parts[1:]))
        os.unlink(self.path)
        if not rows:
            return None
        in_window = True
        if self.t0 is not None and self.t1 is not None:
            sel = [r for w, r in rows if w is not None and self.t0 <= w <= self.t1]
            if not sel:   # window shorter than the sampling period: the nearest samples
                in_window = False
                timed = [(abs(w - 0.5 * (self.t0 + self.t1)), r) for w, r in rows if w is not None]
                sel = [r for _, r in sorted(timed, key=lambda x: x[0])[:2]] or [r for _, r in rows]
        else:
            sel = [r for _, r in rows]
        sm = [float(r[1]) for r in sel if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in sel if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in sel for i in range(4) if r[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(sel), "in_window": in_window}


# ---------------------------------------------------------------- CPU oracle sample
def oracle_sample(shape, host, idx_full=None, w_full=None, n_experts=2, shared_rows=256, seed=0, nthreads=0):
    """Time the C++ fp64 oracle (oracle/cpp, std::thread over `nthreads` host
    cores) on a bounded sample of one layer step and extrapolate.

    Sample: router logits + selection for 1024 tokens, the schedule of all
    tokens, the full forward+backward of `n_experts` routed experts of
    near-average load (all their rows) and of the shared expert on
    `shared_rows` tokens, and combine + router backward for 1024 tokens.
    Each timed part is scaled by the share of the step it stands for. Weight
    MX quantisation is done before timing (it is not part of a layer step).
    Returns (tokens/s, description).
    """
    from oracle import cxx

    T, d, E, k, I, S = shape.T, shape.d, shape.E, shape.k, shape.I, shape.S
    x, dy = host["x"], host["dy"]
    nt = min(1024, T)
    t0 = time.perf_counter()
    idx_s, w_s, s_s, _ = cxx.route(x[:nt], host["w_router"], host["bias"], k, shape.G, shape.g_top, nthreads)
    t_route = (time.perf_counter() - t0) * T / nt
    if idx_full is None:
        idx_full, w_full, _, _ = cxx.route(x, host["w_router"], host["bias"], k, shape.G, shape.g_top, nthreads)
    t0 = time.perf_counter()
    sch = cxx.schedule(idx_full, E, shape.C)
    t_sched = time.perf_counter() - t0
    counts = sch["counts"]
    order = np.argsort(np.abs(counts - counts.mean()), kind="stable")
    experts = [int(e) for e in order[:n_experts] if counts[e] > 0]
    rng = np.random.default_rng(seed)
    wcache = host.setdefault("_cxx_weights", {})     # MX weights are prepared once, outside the timing

    def expert_weights(e):
        if e not in wcache:
            if e < E:
                wcache[e] = cxx.ExpertWeights(host["w_gu_of"](e), host["w_d_of"](e), nthreads)
            else:
                wcache[e] = cxx.ExpertWeights(host["ws_gu_of"](e - E), host["ws_d_of"](e - E), nthreads)
        return wcache[e]

    wflat = np.asarray(w_full, dtype=np.float32).reshape(-1)
    prepared = []
    for e in experts:
        a = sch["inv"][sch["offsets"][e]:sch["offsets"][e + 1]]
        prepared.append((e, expert_weights(e), a // k, wflat[a]))
    if S:
        toks = np.sort(rng.choice(T, min(shared_rows, T), replace=False))
        prepared.append((E, expert_weights(E), toks, None))
    rows_done = 0
    t0 = time.perf_counter()
    for e, W, toks, gate in prepared:
        cxx.expert_q(x[toks], dy[toks], gate, W, nthreads)
        rows_done += len(toks)
    t_exp = time.perf_counter() - t0
    R = T * (k + S)
    t0 = time.perf_counter()
    cxx.combine(w_s, np.zeros((nt, k, d)), np.zeros((nt, d)) if S else None)
    cxx.router_backward(np.zeros((nt, k)), w_s, s_s, idx_s, x[:nt], host["w_router"], E)
    t_comb = (time.perf_counter() - t0) * T / nt
    total = t_route + t_sched + t_exp * R / max(rows_done, 1) + t_comb
    n_shared_rows = len(prepared[-1][2]) if S else 0
    desc = ("C++ fp64 oracle, %d threads: router on %d tokens, schedule of all %d tokens, fwd+bwd of %d routed "
            "experts (%d rows) and the shared expert on %d tokens, combine/router-bwd on %d tokens; extrapolated to "
            "the %d-row step" % (nthreads, nt, T, len(experts), rows_done - n_shared_rows, n_shared_rows, nt, R))
    return T / total, desc


def host_inputs_for_oracle(shape, dev_inputs):
    """Host copies the oracle sample needs; expert weights fetched one expert at a time."""
    h = {
        "x": dev_inputs["x"].float().cpu().numpy().astype(np.float64),
        "dy": dev_inputs["dy"].float().cpu().numpy().astype(np.float64),
        "w_router": dev_inputs["w_router"].float().cpu().numpy().astype(np.float64),
        "bias": dev_inputs["bias"].cpu().numpy(),
    }
    h["w_gu_of"] = lambda e: dev_inputs["w_gu"][e].float().cpu().numpy().astype(np.float64)
    h["w_d_of"] = lambda e: dev_inputs["w_d"][e].float().cpu().numpy().astype(np.float64)
    h["ws_gu_of"] = lambda e: dev_inputs["ws_gu"][e].float().cpu().numpy().astype(np.float64)
    h["ws_d_of"] = lambda e: dev_inputs["ws_d"][e].float().cpu().numpy().astype(np.float64)
    return h


def cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


def workload_config(shape, extra=None):
    c = {"workload": "%s: T=%d d=%d E=%d(+%d shared) top-%d groups %d/%d I=%d ring C=%d bias %s"
         % (shape.name, shape.T, shape.d, shape.E, shape.S, shape.k, shape.G, shape.g_top, shape.I, shape.C,
            shape.bias),
         "T": shape.T, "d": shape.d, "E": shape.E, "n_shared": shape.S, "k": shape.k, "I": shape.I,
         "ring_capacity": shape.C, "l2": "inputs larger than L2 (x, dy 2*T*d bytes each; weights >10 GB)",
         "parallelism": "replicas"}
    if extra:
        c.update(extra)
    return c


# ---------------------------------------------------------------- reference arm
def run_reference(args, rank, world):
    if rank != 0:
        return
    shape = _shape(args)
    inp = gen.make_inputs(shape, seed=0, device="cpu", weights=False)
    host = {
        "x": inp["x"].double().numpy(), "dy": inp["dy"].double().numpy(),
        "w_router": inp["w_router"].double().numpy(), "bias": inp["bias"].numpy(),
    }
    # Expert weights: same shapes and distribution, drawn per expert from their own seed
    # (the oracle sample touches only a few experts).
    def wgen(e, shp, shared=False):
        g = torch.Generator().manual_seed(1000 + e + (100000 if shared else 0))
        return (torch.randn(shp, generator=g) * shape.w_std).to(torch.bfloat16).double().numpy()
    host["w_gu_of"] = lambda e: wgen(e, (2 * shape.I, shape.d))
    host["w_d_of"] = lambda e: wgen(e + 5000, (shape.d, shape.I))
    host["ws_gu_of"] = lambda e: wgen(e, (2 * shape.I, shape.d), True)
    host["ws_d_of"] = lambda e: wgen(e + 5000, (shape.d, shape.I), True)
    from oracle import cxx
    nthreads = cores()
    idx_full, w_full, _, _ = cxx.route(host["x"], host["w_router"], host["bias"], shape.k, shape.G, shape.g_top,
                                       nthreads)
    vals = []
    desc = ""
    for i in range(args.warmup + args.steps):
        v, desc = oracle_sample(shape, host, idx_full=idx_full, w_full=w_full, n_experts=1, shared_rows=128, seed=i,
                                nthreads=nthreads)
        if i >= args.warmup:
            vals.append(v)
    val = statistics.median(vals)
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 * shape.T / val,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(shape),
            "cpu_baseline": {"value": val, "unit": "tokens/s", "cores": nthreads, "kind": "oracle", "sample": desc},
            "e2e": {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- multi-rank timing
def rank_barrier(world):
    """Barrier over the ranks of a --gpus N run (no-op for one rank)."""
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(value, world, device):
    """The slowest rank's value: the job's time is the max over ranks."""
    if world > 1:
        t = torch.tensor([value], device=device, dtype=torch.float64)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        value = float(t.item())
    return value


def job_tokens_per_s(tokens_per_rank, world, ms_step):
    """Whole-job throughput: every rank processes its own tokens_per_rank each step."""
    return tokens_per_rank * world / (ms_step / 1000.0)


# ---------------------------------------------------------------- our arm
def standalone_movers(shape, L, inp, sp, hb):
    """GB/s of the ring gather run as its own kernel: moe_dispatch (MX(x), then
    one gather launch over all laps) timed alone after the timed region. In the
    default form the same moves run inside GEMM1's mover warps, overlapped
    with the MMAs, and have no time of their own. The backward pull of the
    MX(dy) rows into the dO ring (permute_lap_dO) is timed in one per-lap pass
    of a second layer."""
    import moe_layer_dsv3_gb300 as M
    from moe_layer_dsv3_gb300.layer import MoELayer
    x, dy, wr, bias = inp["x"], inp["dy"], inp["w_router"], inp["bias"]
    out = {}
    for _ in range(2):
        L.dispatch(x, sp)
    torch.cuda.synchronize()
    M.moe_profile_enable(True)
    M.moe_profile_read()
    for _ in range(3):
        L.dispatch(x, sp)
    torch.cuda.synchronize()
    kern = M.moe_profile_read()
    M.moe_profile_enable(False)
    if "dispatch_all" in kern and kern["dispatch_all"][1] > 0:
        out["permute_lap"] = 3 * hb["permute_lap"] / (kern["dispatch_all"][1] / 1000.0) / 1e9
    Lp = MoELayer.from_shape(shape, flags=M.MOE_FLAG_LAP_LAUNCHES)
    Lp.wq = L.wq                                   # the same quantised weights
    for _ in range(2):
        Lp.forward(x, wr, bias, sp)
        Lp.backward(dy, sp)
    torch.cuda.synchronize()
    M.moe_profile_enable(True)
    M.moe_profile_read()
    Lp.backward(dy, sp)
    torch.cuda.synchronize()
    kern = M.moe_profile_read()
    M.moe_profile_enable(False)
    if "permute_lap_dO" in kern and kern["permute_lap_dO"][1] > 0:
        out["permute_lap_dO"] = hb["permute_lap_dO"] / (kern["permute_lap_dO"][1] / 1000.0) / 1e9
    del Lp
    torch.cuda.empty_cache()
    return out


def run_ours(args, rank, world, local_rank):
    import moe_layer_dsv3_gb300 as M
    from moe_layer_dsv3_gb300.layer import MoELayer

    torch.cuda.set_device(local_rank)
    shape = _shape(args)
    inp = gen.make_inputs(shape, seed=rank, device="cuda")
    flags = (M.MOE_FLAG_LAP_LAUNCHES if args.lap_launches else 0) | (M.MOE_FLAG_WGRAD_PAIR if args.wgrad_pair else 0)
    L = MoELayer.from_shape(shape, flags=flags, n_mover_warps=args.mover_warps)
    L.quantize_weights(inp["w_gu"], inp["w_d"], inp["ws_gu"], inp["ws_d"])
    stream = torch.cuda.current_stream()
    sp = stream.cuda_stream
    x, dy, wr, bias = inp["x"], inp["dy"], inp["w_router"], inp["bias"]

    def step():
        L.forward(x, wr, bias, sp)
        L.backward(dy, sp)

    clocks = ClockSampler(local_rank)   # started before the warm-up: nvidia-smi takes a moment to start
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    code, site = L.status()
    if code:
        raise RuntimeError("device status %d at site %d after warm-up" % (code, site))

    def barrier():
        rank_barrier(world)

    # ---- timed region: K steps, inputs resident in HBM
    M.moe_profile_enable(True)
    M.moe_profile_read()
    n0 = M.moe_launch_count()
    barrier()
    torch.cuda.synchronize()
    clocks.window(True)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    clocks.window(False)
    barrier()
    launches = M.moe_launch_count() - n0
    kern = M.moe_profile_read()
    M.moe_profile_enable(False)
    clk = clocks.stop()
    ms = max_over_ranks(e0.elapsed_time(e1), world, "cuda")
    ms_step = ms / args.steps
    value = job_tokens_per_s(shape.T, world, ms_step)

    # ---- per-stage split (one extra, separately timed step)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
    ev[0].record(stream)
    L.route(x, wr, bias, sp)
    ev[1].record(stream)
    L.schedule(sp)
    ev[2].record(stream)
    L.forward_experts(x, sp)
    ev[3].record(stream)
    L.backward(dy, sp)
    ev[4].record(stream)
    torch.cuda.synchronize()
    stages = {n: ev[i].elapsed_time(ev[i + 1]) for i, n in enumerate(("route", "schedule", "forward", "backward"))}

    # ---- the same step replayed from a CUDA graph of its launches (launch-overhead check)
    graph_ms = None
    if not args.no_graph:
        g = L.capture_step(x, wr, bias, dy)
        for _ in range(2):
            g.replay()
        torch.cuda.synchronize()
        ge0, ge1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ge0.record(stream)
        for _ in range(args.steps):
            g.replay()
        ge1.record(stream)
        torch.cuda.synchronize()
        graph_ms = ge0.elapsed_time(ge1) / args.steps
        del g

    # ---- end to end through the C ABI with host buffers (H2D of x, dy; D2H of y, dx).
    # Every step copies its inputs from pinned host memory and its outputs back.
    # The copies run on two copy streams into NB device buffers per tensor, so a
    # step's inputs are uploaded NB - 1 steps ahead and its outputs have NB steps
    # to leave, which absorbs copy jitter on shared hosts; within a step the
    # forward waits only for x and y leaves during the backward.
    NB = 3
    xh = x.cpu().pin_memory()
    dyh = dy.cpu().pin_memory()
    yh = torch.empty_like(xh).pin_memory()
    dxh = torch.empty_like(xh).pin_memory()
    xd = [torch.empty_like(x) for _ in range(NB)]
    dyd = [torch.empty_like(dy) for _ in range(NB)]
    yd = [torch.empty_like(x) for _ in range(NB)]
    dxd = [torch.empty_like(x) for _ in range(NB)]
    h2d_s, d2h_s = torch.cuda.Stream(), torch.cuda.Stream()

    def e2e_run(n, start_ev):
        ev = lambda: [torch.cuda.Event() for _ in range(NB)]   # noqa: E731
        loaded_x, loaded_dy, fwd_done, done, drained_y, drained_dx = ev(), ev(), ev(), ev(), ev(), ev()

        def upload(i):
            # step i's inputs into buffer i % NB once step i - NB has finished with it;
            # x first: the forward starts once x is in, dy is only needed by the backward
            b = i % NB
            h2d_s.wait_event(done[b] if i >= NB else start_ev)
            with torch.cuda.stream(h2d_s):
                xd[b].copy_(xh, non_blocking=True)
                loaded_x[b].record(h2d_s)
                dyd[b].copy_(dyh, non_blocking=True)
                loaded_dy[b].record(h2d_s)

        for i in range(min(NB - 1, n)):
            upload(i)
        for i in range(n):
            b = i % NB
            if i + NB - 1 < n:
                upload(i + NB - 1)
            stream.wait_event(loaded_x[b])
            if i >= NB:
                stream.wait_event(drained_y[b])
            L.forward(xd[b], wr, bias, sp, y=yd[b])          # outputs go straight to this step's buffers
            fwd_done[b].record(stream)
            d2h_s.wait_event(fwd_done[b])                     # y leaves while the backward runs
            with torch.cuda.stream(d2h_s):
                yh.copy_(yd[b], non_blocking=True)
            drained_y[b].record(d2h_s)
            stream.wait_event(loaded_dy[b])
            if i >= NB:
                stream.wait_event(drained_dx[b])
            L.backward(dyd[b], sp, dx=dxd[b])
            done[b].record(stream)
            d2h_s.wait_event(done[b])
            with torch.cuda.stream(d2h_s):
                dxh.copy_(dxd[b], non_blocking=True)
            drained_dx[b].record(d2h_s)
        stream.wait_stream(d2h_s)
        stream.wait_stream(h2d_s)

    s0 = torch.cuda.Event()
    s0.record(stream)
    e2e_run(2, s0)
    torch.cuda.synchronize()
    barrier()
    e0.record(stream)
    e2e_run(args.steps, e0)
    e1.record(stream)
    torch.cuda.synchronize()
    ms_e2e = max_over_ranks(e0.elapsed_time(e1) / args.steps, world, "cuda")
    # the machine's host link alone: one copy of x each way between pinned host memory and the device
    link = {}
    for name, dst, src, st in (("h2d_gbs", xd[0], xh, h2d_s), ("d2h_gbs", yh, yd[0], d2h_s)):
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c0.record(st)
        with torch.cuda.stream(st):
            dst.copy_(src, non_blocking=True)
        c1.record(st)
        c1.synchronize()
        link[name] = xh.numel() * xh.element_size() / (c0.elapsed_time(c1) * 1e-3) / 1e9
    code, site = L.status()
    if code:
        raise RuntimeError("device status %d at site %d" % (code, site))
    if rank != 0:
        return

    # ---- roofline of the dominant kernel and per-kernel summary
    pk = peaks()
    fl = gemm_flops(shape)
    hb = hbm_bytes(shape)
    per_kernel = {}
    for name, (n, tms) in sorted(kern.items(), key=lambda kv: -kv[1][1]):
        ent = {"launches": n, "ms_per_step": tms / args.steps, "share": tms / ms if ms > 0 else None}
        if name in fl:
            ent["tflops"] = fl[name] * args.steps / (tms / 1000.0) / 1e12
        if name in hb:
            ent["gbs"] = hb[name] * args.steps / (tms / 1000.0) / 1e9
        per_kernel[name] = ent
    # Ring-lap kernels run on two streams and overlap one another, so their
    # event times are not additive; the dominant kernel is taken among the
    # kernels that run alone on the launch stream.
    lap_kernels = {"gemm1_fwd", "gemm_dgrad_down", "permute_lap", "permute_lap_dO"} if args.lap_launches else set()
    dom = max(((n, v) for n, v in kern.items() if n not in lap_kernels), key=lambda kv: kv[1][1])[0]
    fp8_peak = pk["fp8"]
    if dom in fl:
        achieved = per_kernel[dom]["tflops"]
        roof = {"kernel": dom, "bound": "tensor", "achieved": achieved, "peak": fp8_peak, "unit": "TFLOP/s",
                "frac": achieved / fp8_peak, "traffic": None, "peak_note": pk["fp8_note"],
                "flop_per_step": fl[dom]}
    else:
        achieved = per_kernel[dom].get("gbs", 0.0)
        roof = {"kernel": dom, "bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / pk["hbm_gbs"], "traffic": None}
    traffic_file = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(traffic_file):
        with open(traffic_file) as f:
            tr = json.load(f)
        ent = tr.get(shape.name, {}).get(dom)
        if ent is not None:
            roof["traffic"] = ent
    gemm_names = [n for n in fl if n in kern and n != "router_gemm"]
    gemm_ms = sum(kern[n][1] for n in gemm_names) / args.steps
    gemm_tflops = sum(fl[n] for n in gemm_names) / (gemm_ms / 1000.0) / 1e12 if gemm_ms else None
    perm = per_kernel.get("permute_lap", {}).get("gbs")
    movers = None
    if not args.lap_launches and not args.no_standalone_movers:
        movers = standalone_movers(shape, L, inp, sp, hb)
        perm = movers.get("permute_lap")
    extra = {
        "stages_ms": stages,
        "grouped_gemm_tflops": gemm_tflops,
        "grouped_gemm_frac_fp8_peak": gemm_tflops / fp8_peak if gemm_tflops else None,
        "graph_ms_per_step": graph_ms,
        "permute_gbs": perm,
        "standalone_movers_gbs": movers,
        "permute_frac_hbm": perm / pk["hbm_gbs"] if perm else None,
        "schedule_share": (stages["schedule"]) / sum(stages.values()),
        "lap_kernels_overlap": sorted(lap_kernels),
        "kernels": per_kernel,
    }
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        host = host_inputs_for_oracle(shape, inp)
        idx = L.topk_idx.cpu().numpy()
        v, desc = oracle_sample(shape, host, idx_full=idx, w_full=L.topk_w.cpu().numpy(), nthreads=cores())
        cpu = {"value": v, "unit": "tokens/s", "cores": cores(), "kind": "oracle", "sample": desc}
    counts = L.ws_tensor("COUNTS", torch.int32, (shape.E + shape.S,)).cpu().numpy()[:shape.E]
    # Waves of each grouped GEMM: output tiles / SM count (the commentary's rule asks for >= 2).
    sms = torch.cuda.get_device_properties(local_rank).multi_processor_count
    all_counts = L.ws_tensor("COUNTS", torch.int32, (shape.E + shape.S,)).cpu().numpy().astype(np.int64)
    mt = int(((all_counts + 127) // 128).sum())
    E_all = shape.E + shape.S
    extra["waves"] = {"sm_count": sms,
                      "gemm1_fwd": mt * (2 * shape.I // 256) / sms, "gemm2_fwd": mt * (shape.d // 256) / sms,
                      "gemm_dgrad_down": mt * (shape.I // 256) / sms, "gemm_dgrad_gu": mt * (shape.d // 256) / sms,
                      "gemm_wgrad_d": E_all * (shape.d // 128) * (shape.I // 256) / sms,
                      "gemm_wgrad_gu": E_all * (2 * shape.I // 128) * (shape.d // 256) / sms}
    extra["routing"] = {"max_count": int(counts.max()), "min_count": int(counts.min()),
                        "laps": int(L.ws_tensor("META", torch.int32, (16,))[0].item()),
                        "ring_capacity": shape.C}
    h2d = 2 * x.numel() * x.element_size()
    d2h = 2 * x.numel() * x.element_size()
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "mxfp8", "data": "synthetic (seeded, random-init weights)",
        "config": dict(workload_config(shape),
                       ring_laps="per-lap launches" if args.lap_launches else "one launch, mover warps",
                       wgrad_tiles="CTA pairs 256-row" if args.wgrad_pair else "single CTA 128x256",
                       mover_warps=args.mover_warps or 2),
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": {"value": job_tokens_per_s(shape.T, world, ms_e2e), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": ms_e2e, "host_link_gbs": {k: round(v, 1) for k, v in link.items()}},
        "gpu_launches": launches,
        "clocks": clk,
    }
    line.update(extra)
    print(json.dumps(line), flush=True)


def _shape(args):
    shape = gen.config(args.workload, T=args.T)
    if args.capacity is not None:
        if args.capacity <= 0 or args.capacity % 128:
            raise SystemExit("--capacity must be a positive multiple of 128")
        shape = dataclasses.replace(shape, C=args.capacity)
    return shape


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="dsv3_zipf")
    ap.add_argument("--T", type=int, default=None)
    ap.add_argument("--capacity", type=int, default=None,
                    help="ring capacity per expert (multiple of 128) instead of the workload's")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="skip the CUDA-graph replay timing")
    ap.add_argument("--no-standalone-movers", action="store_true",
                    help="skip the extra per-lap pass that times the ring movers as their own launches")
    ap.add_argument("--lap-launches", action="store_true",
                    help="one mover launch + one GEMM launch per ring lap instead of one all-laps launch")
    ap.add_argument("--mover-warps", type=int, default=0, choices=[0, 1, 2, 4],
                    help="mover warps per CTA of the all-laps ring GEMMs (0 = library default)")
    ap.add_argument("--wgrad-pair", action="store_true",
                    help="weight gradients on CTA pairs (256-row tiles) instead of single-CTA tiles (for comparison)")
    ap.add_argument("--probe-peak", action="store_true",
                    help="measure dense MXFP8 GEMM throughput (library and this repo's plain GEMM) and exit")
    ap.add_argument("--probe-n", type=int, default=8192)
    args = ap.parse_args()
    if args.probe_peak:
        probe_peak(args)
        return
    if args.warmup < 3:
        args.warmup = 3
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        backend = "nccl" if torch.cuda.is_available() and args.impl == "ours" else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group(backend=backend)
    try:
        if args.impl == "reference":
            run_reference(args, rank, world)
        else:
            run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
