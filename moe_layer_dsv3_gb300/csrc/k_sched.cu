// Device-side schedule (write-ups: the schedule is built on the device, costs
// under 3 % of the MoE runtime and is reused by backward without re-sorting;
// Cursor blog summary, "method points").
//
// Assignments are taken in (t, j) order over k routed slots plus the shared
// experts' slots (slot k + s always picks shared expert E + s). Three passes:
//   1. per-unit histograms (unit = 256 consecutive assignments, one warp);
//   2. per-expert exclusive scan over units, then a single-block pass for
//      offsets, 128-row padded offsets and the per-lap tile lists;
//   3. stable ranks: each warp walks its unit in order, 32 assignments at a
//      time, ranking equal experts with __match_any_sync.
// Only integer arithmetic; the result does not depend on scheduling order.
#include "moe_internal.h"
#include "ptx.cuh"
#include "prof.h"

namespace moe {

namespace {

constexpr int kWarps = 8;

__device__ __forceinline__ int expert_of(const int32_t* idx, int64_t ap, int k, int kp, int E) {
  const int64_t t = ap / kp;
  const int j = static_cast<int>(ap - t * kp);
  return j < k ? idx[t * k + j] : E + (j - k);
}

// Canonical assignment id: routed a = t*k + j, shared a = T*k + s*T + t.
__device__ __forceinline__ int canon_of(int64_t ap, int T, int k, int kp) {
  const int64_t t = ap / kp;
  const int j = static_cast<int>(ap - t * kp);
  return static_cast<int>(j < k ? t * k + j : static_cast<int64_t>(T) * k + static_cast<int64_t>(j - k) * T + t);
}

__global__ void sched_hist_kernel(const int32_t* __restrict__ idx, int k, int kp, int E, int Ep, int64_t Ap,
                                  int units, int* __restrict__ hist, int* status) {
  extern __shared__ int sh[];
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int u = blockIdx.x * kWarps + w;
  int* h = sh + w * Ep;
  for (int e = lane; e < Ep; e += 32) h[e] = 0;
  __syncwarp();
  if (u < units) {
    for (int i = lane; i < kSchedUnit; i += 32) {
      const int64_t ap = static_cast<int64_t>(u) * kSchedUnit + i;
      if (ap < Ap) {
        const int e = expert_of(idx, ap, k, kp, E);
        if (e >= 0 && e < Ep) atomicAdd(&h[e], 1);
        else report_error(status, kErrBounds, 100);
      }
    }
  }
  __syncwarp();
  if (u < units)
    for (int e = lane; e < Ep; e += 32) hist[static_cast<int64_t>(u) * Ep + e] = h[e];
}

// One block per expert: exclusive scan of hist[.][e] over units.
__global__ void sched_scan_kernel(const int* __restrict__ hist, int Ep, int units, int* __restrict__ base,
                                  int* __restrict__ counts) {
  __shared__ int sums[256];
  const int e = blockIdx.x;
  const int per = (units + 255) / 256;
  const int u0 = threadIdx.x * per;
  int s = 0;
  for (int u = u0; u < u0 + per && u < units; ++u) s += hist[static_cast<int64_t>(u) * Ep + e];
  sums[threadIdx.x] = s;
  __syncthreads();
  if (threadIdx.x == 0) {
    int run = 0;
    for (int i = 0; i < 256; ++i) {
      const int v = sums[i];
      sums[i] = run;
      run += v;
    }
    counts[e] = run;
  }
  __syncthreads();
  int run = sums[threadIdx.x];
  for (int u = u0; u < u0 + per && u < units; ++u) {
    const int64_t o = static_cast<int64_t>(u) * Ep + e;
    const int v = hist[o];
    base[o] = run;
    run += v;
  }
}

// Offsets, padded offsets, laps and per-lap tile prefix sums.
// lap_tiles[L][e] = sum_{e' < e} ceil(len(e', L) / 128), where a routed
// expert's lap L holds ranks [L*C, min(n, (L+1)*C)) and a shared expert is
// processed whole in lap 0 (it is read in token order, not from the ring).
__global__ void sched_offsets_kernel(const int* counts, int E, int Ep, int C, int Lb,
                                     int* __restrict__ offsets, int* __restrict__ poff, int* __restrict__ lap_tiles,
                                     int* __restrict__ meta, int* __restrict__ lapbase) {
  __shared__ int sc[1024];   // counts, Ep <= 513
  for (int e = threadIdx.x; e < Ep; e += blockDim.x) sc[e] = counts[e];
  __syncthreads();
  counts = sc;
  if (threadIdx.x == 0) {
    int o = 0, po = 0, nmax = 0, active = 0;
    for (int e = 0; e < Ep; ++e) {
      offsets[e] = o;
      poff[e] = po;
      const int n = counts[e];
      o += n;
      po += (n + 127) & ~127;
      if (e < E) nmax = max(nmax, n);
      active += n > 0 ? 1 : 0;
    }
    offsets[Ep] = o;
    poff[Ep] = po;
    meta[0] = (nmax + C - 1) / C;   // laps of the busiest routed expert
    meta[1] = po;
    meta[2] = active;
  }
  for (int L = threadIdx.x; L < Lb; L += blockDim.x) {
    int run = 0;
    int* lt = lap_tiles + static_cast<int64_t>(L) * (Ep + 1);
    for (int e = 0; e < Ep; ++e) {
      lt[e] = run;
      const int n = counts[e];
      int len;
      if (e < E) {
        len = n - L * C;
        len = len < 0 ? 0 : (len > C ? C : len);
      } else {
        len = L == 0 ? n : 0;
      }
      run += (len + 127) / 128;
    }
    lt[Ep] = run;
  }
  __syncthreads();
  if (threadIdx.x == 0) {       // lapbase[L] = sum over laps L' < L of their m-tiles
    int run = 0;
    for (int L = 0; L < Lb; ++L) {
      lapbase[L] = run;
      run += lap_tiles[static_cast<int64_t>(L) * (Ep + 1) + Ep];
    }
    lapbase[Lb] = run;
  }
}

// Exclusive prefix sum of one value per thread over the block (1024 threads).
__device__ __forceinline__ int block_exscan(int v, int* sm, int& total) {
  sm[threadIdx.x] = v;
  __syncthreads();
  for (int off = 1; off < blockDim.x; off <<= 1) {
    const int t = threadIdx.x >= off ? sm[threadIdx.x - off] : 0;
    __syncthreads();
    sm[threadIdx.x] += t;
    __syncthreads();
  }
  const int incl = sm[threadIdx.x];
  total = sm[blockDim.x - 1];
  __syncthreads();
  return incl - v;
}

constexpr int kKeyUnits = 2048;

// Walk order of the all-laps launches (order[position] = lap-major m-tile gm).
// A unit is an expert's lap pair P (laps 2P and 2P + 1, whose tiles stay side
// by side, lap 2P first, so the expert's weights stream once for both). An
// expert with two or more pairs has its pairs at key (2P + 1) / (2 pairs),
// spread evenly over the walk; the experts with one pair (at most two laps,
// and the shared experts) take (2i + 1) / (2 n_one) in expert order. Units go
// by ascending key (compared exactly as integers), then expert, then pair.
// One block of 1024 threads; scratch holds 3 * cap ints (units, their ranks,
// the tile counts in rank order, then their prefix sums).
//
// The same kernel writes the decode tables of the grouped GEMMs, so that a
// tile's expert, rows and ring slot cost one load instead of a chain of
// dependent searches through the lap and expert prefix sums:
//   info[2 pos]     = {gm, e | valid << 16 | ok << 24 | shared << 25, A row, padded rank row}
//   info[2 pos + 1] = {gm of the slot's previous tenant (lap L - kRingBufs) or -1,
//                      rank of the tile's first row, count of e, poff[e]}
//   push_info[g]    = e | valid << 16 for m-tile g of the padded rank rows.
__global__ void __launch_bounds__(1024) sched_laporder_kernel(const int* __restrict__ counts,
                                                              const int* __restrict__ poff, int E, int Ep, int C,
                                                              int Lb, const int* __restrict__ lapbase,
                                                              const int* __restrict__ lap_tiles, int64_t cap,
                                                              int* __restrict__ scratch, int* __restrict__ order,
                                                              int4* __restrict__ info, int* __restrict__ push_info) {
  __shared__ int sm[1024];
  __shared__ int s_pairs[1024], s_one[1024];
  __shared__ int s_num[kKeyUnits], s_den[kKeyUnits], s_unit[kKeyUnits];
  int* unit = scratch;             // e | P << 16
  int* urank = scratch + cap;
  int* stile = scratch + 2 * cap;  // tiles by rank, then their exclusive prefix
  const int e = threadIdx.x;
  int pairs = 0;
  if (e < Ep) {
    const int n = counts[e];
    const int laps = e < E ? (n + C - 1) / C : (n > 0 ? 1 : 0);
    pairs = (laps + 1) / 2;
  }
  int U = 0, n_one = 0;
  const int ubase = block_exscan(pairs, sm, U);
  const int one = block_exscan(pairs == 1 ? 1 : 0, sm, n_one);
  s_pairs[e] = pairs;
  s_one[e] = one;
  for (int P = 0; P < pairs; ++P) unit[ubase + P] = e | (P << 16);
  __syncthreads();
  auto tiles_of = [&](int ue, int P) {
    int t = 0;
    for (int L = 2 * P; L < 2 * P + 2 && L < Lb; ++L) {
      const int* lt = lap_tiles + static_cast<int64_t>(L) * (Ep + 1);
      t += lt[ue + 1] - lt[ue];
    }
    return t;
  };
  // key of unit u: num / den; units of up to kKeyUnits are compared from shared memory
  auto key_of = [&](int u, int& num, int& den) {
    const int ue = unit[u] & 0xFFFF, P = unit[u] >> 16;
    const bool spread = s_pairs[ue] >= 2;
    num = spread ? 2 * P + 1 : 2 * s_one[ue] + 1;
    den = spread ? 2 * s_pairs[ue] : 2 * n_one;
  };
  const bool in_smem = U <= kKeyUnits;
  if (in_smem) {
    for (int u = threadIdx.x; u < U; u += blockDim.x) {
      key_of(u, s_num[u], s_den[u]);
      s_unit[u] = unit[u];
    }
    __syncthreads();
  }
  for (int u = threadIdx.x; u < U; u += blockDim.x) {
    const int uu = unit[u];
    int num, den;
    key_of(u, num, den);
    int rank = 0;
    for (int v = 0; v < U; ++v) {
      int vn, vd, vu;
      if (in_smem) {
        vn = s_num[v]; vd = s_den[v]; vu = s_unit[v];
      } else {
        key_of(v, vn, vd);
        vu = unit[v];
      }
      const int64_t lhs = static_cast<int64_t>(vn) * den, rhs = static_cast<int64_t>(num) * vd;   // key(v) < key(u)
      // ties: lower expert, then lower pair (unit = e | P << 16 with e < 2^16)
      const bool before = lhs < rhs || (lhs == rhs && ((vu & 0xFFFF) < (uu & 0xFFFF) ||
                                                        ((vu & 0xFFFF) == (uu & 0xFFFF) && (vu >> 16) < (uu >> 16))));
      rank += before ? 1 : 0;
    }
    urank[u] = rank;
    stile[rank] = tiles_of(uu & 0xFFFF, uu >> 16);
  }
  __syncthreads();
  int carry = 0;   // exclusive prefix of stile over ranks, 1024 at a time
  for (int c0 = 0; c0 < U; c0 += blockDim.x) {
    const int r = c0 + threadIdx.x;
    const int v = r < U ? stile[r] : 0;
    int chunk = 0;
    const int ex = block_exscan(v, sm, chunk);
    if (r < U) stile[r] = carry + ex;
    carry += chunk;
    __syncthreads();
  }
  for (int u = threadIdx.x; u < U; u += blockDim.x) {
    const int ue = unit[u] & 0xFFFF, P = unit[u] >> 16;
    const bool shared = ue >= E;
    const int cnt = counts[ue], pe = poff[ue], pe1 = poff[ue + 1];
    int pos = stile[urank[u]];
    for (int L = 2 * P; L < 2 * P + 2 && L < Lb; ++L) {
      const int* lt = lap_tiles + static_cast<int64_t>(L) * (Ep + 1);
      const int base = lapbase[L] + lt[ue];
      for (int mt = 0; mt < lt[ue + 1] - lt[ue]; ++mt) {
        // A shared expert is read in place (token rows mt*128..); a routed
        // expert's lap L sits in ring buffer L % kRingBufs at row e*C + mt*128.
        const int rank0 = shared ? mt * 128 : L * C + mt * 128;
        const int a_row = shared ? mt * 128 : ((L % kRingBufs) * E + ue) * C + mt * 128;
        const int prow0 = pe + rank0;
        const int v = cnt - rank0;
        const int valid = v < 0 ? 0 : (v > 128 ? 128 : v);
        const int ok = (prow0 + 128 <= pe1 && valid > 0) ? 1 : 0;
        int gp = -1;
        if (!shared && L >= kRingBufs) {
          const int Lp = L - kRingBufs;
          gp = lapbase[Lp] + lap_tiles[static_cast<int64_t>(Lp) * (Ep + 1) + ue] + mt;
        }
        order[pos] = base + mt;
        info[2 * pos] = make_int4(base + mt, ue | (valid << 16) | (ok << 24) | ((shared ? 1 : 0) << 25), a_row, prow0);
        info[2 * pos + 1] = make_int4(gp, rank0, cnt, pe);
        ++pos;
      }
    }
  }
  for (int e = threadIdx.x; e < Ep; e += blockDim.x) {
    const int pe = poff[e], pe1 = poff[e + 1], cnt = counts[e];
    for (int g = pe / 128; g < pe1 / 128; ++g) {
      const int v = cnt - (g * 128 - pe);
      push_info[g] = e | ((v < 0 ? 0 : (v > 128 ? 128 : v)) << 16);
    }
  }
}

// Experts ordered by descending count, ties to the lower index (order[rank] = e),
// and the weight gradients' decode table: wg_info[rank] = {e, first K tile,
// K tiles, 0} (K = the expert's padded token rows).
__global__ void sched_order_kernel(const int* __restrict__ counts, const int* __restrict__ poff, int Ep,
                                   int* __restrict__ order, int4* __restrict__ wg_info) {
  for (int e = threadIdx.x; e < Ep; e += blockDim.x) {
    const int n = counts[e];
    int r = 0;
    for (int f = 0; f < Ep; ++f) {
      const int m = counts[f];
      r += (m > n || (m == n && f < e)) ? 1 : 0;
    }
    order[r] = e;
    wg_info[r] = make_int4(e, poff[e] / 128, (poff[e + 1] - poff[e]) / 128, 0);
  }
}

__global__ void sched_rank_kernel(const int32_t* __restrict__ idx, int T, int k, int kp, int E, int Ep, int64_t Ap,
                                  int units, const int* __restrict__ base, const int* __restrict__ offsets,
                                  const int* __restrict__ poff, int* __restrict__ rank, int* __restrict__ pos,
                                  int* __restrict__ inv, int* __restrict__ row_src) {
  extern __shared__ int sh[];
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int u = blockIdx.x * kWarps + w;
  if (u >= units) return;
  int* run = sh + w * Ep;
  for (int e = lane; e < Ep; e += 32) run[e] = base[static_cast<int64_t>(u) * Ep + e];
  __syncwarp();
  const unsigned lt_mask = (1u << lane) - 1u;
  for (int b = 0; b < kSchedUnit / 32; ++b) {
    const int64_t ap = static_cast<int64_t>(u) * kSchedUnit + b * 32 + lane;
    const bool valid = ap < Ap;
    int e = valid ? expert_of(idx, ap, k, kp, E) : -1 - lane;
    if (valid && (e < 0 || e >= Ep)) e = -1000 - lane;   // already reported by the histogram pass
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const bool ok = valid && e >= 0;
    int r = 0;
    if (ok) r = run[e] + __popc(peers & lt_mask);
    __syncwarp();
    if (ok && (31 - __clz(peers)) == lane) run[e] += __popc(peers);
    __syncwarp();
    if (ok) {
      const int a = canon_of(ap, T, k, kp);
      rank[a] = r;
      const int p = offsets[e] + r;
      pos[a] = p;
      inv[p] = a;
      row_src[static_cast<int64_t>(poff[e]) + r] = a;
    }
  }
}

}  // namespace

void launch_schedule(const Dims& m, const int32_t* idx, const Layout& L, void* ws, cudaStream_t s) {
  int* hist = ws_ptr<int>(L, ws, MOE_WS_HIST);
  int* base = ws_ptr<int>(L, ws, MOE_WS_BASE);
  int* counts = ws_ptr<int>(L, ws, MOE_WS_COUNTS);
  int* offsets = ws_ptr<int>(L, ws, MOE_WS_OFFSETS);
  int* poff = ws_ptr<int>(L, ws, MOE_WS_POFF);
  int* lap_tiles = ws_ptr<int>(L, ws, MOE_WS_LAPTILES);
  int* meta = ws_ptr<int>(L, ws, MOE_WS_META);
  int* status = ws_ptr<int>(L, ws, MOE_WS_STATUS);
  const unsigned blocks = static_cast<unsigned>(ceil_div(m.units, kWarps));
  const size_t shm = static_cast<size_t>(kWarps) * m.Ep * sizeof(int);
  note(cudaMemsetAsync(ws_ptr<int>(L, ws, MOE_WS_ROWSRC), 0xFF, L.bytes[MOE_WS_ROWSRC], s));
  if (m.units > 0) {
    launch_kernel("sched_hist", sched_hist_kernel, dim3(blocks), dim3(kWarps * 32), shm, s, idx, m.k, m.kp, m.E, m.Ep,
                  m.Ap, m.units, hist, status);
    launch_kernel("sched_scan", sched_scan_kernel, dim3(m.Ep), dim3(256), 0, s, hist, m.Ep, m.units, base, counts);
  } else {
    note(cudaMemsetAsync(counts, 0, sizeof(int) * m.Ep, s));
  }
  launch_kernel("sched_offsets", sched_offsets_kernel, dim3(1), dim3(256), 0, s, counts, m.E, m.Ep, m.C, m.Lb, offsets,
                poff, lap_tiles, meta, ws_ptr<int>(L, ws, MOE_WS_LAPBASE));
  launch_kernel("sched_laporder", sched_laporder_kernel, dim3(1), dim3(1024), 0, s, counts, poff, m.E, m.Ep, m.C,
                m.Lb, ws_ptr<int>(L, ws, MOE_WS_LAPBASE), lap_tiles, lap_mtiles_max(m),
                ws_ptr<int>(L, ws, MOE_WS_LAPKEY), ws_ptr<int>(L, ws, MOE_WS_LAPORDER),
                ws_ptr<int4>(L, ws, MOE_WS_RINGINFO), ws_ptr<int>(L, ws, MOE_WS_PUSHINFO));
  launch_kernel("sched_order", sched_order_kernel, dim3(1), dim3(512), 0, s, counts, poff, m.Ep,
                ws_ptr<int>(L, ws, MOE_WS_ORDER), ws_ptr<int4>(L, ws, MOE_WS_WGINFO));
  if (m.units > 0) {
    launch_kernel("sched_rank", sched_rank_kernel, dim3(blocks), dim3(kWarps * 32), shm, s, idx, m.T, m.k, m.kp, m.E,
                  m.Ep, m.Ap, m.units, base, offsets, poff, ws_ptr<int>(L, ws, MOE_WS_RANK),
                  ws_ptr<int>(L, ws, MOE_WS_POS), ws_ptr<int>(L, ws, MOE_WS_INV), ws_ptr<int>(L, ws, MOE_WS_ROWSRC));
  }
}

}  // namespace moe
