// Data movement on the schedule: dispatch into the ring (permute), combine,
// reverse-combine and reverse-dispatch, and the router's backward reductions.
//
// Write-ups: dispatch pulls tokens into fixed-capacity ring token buffers
// whose regions are reused once a batch is computed (techlab report, section
// on the ring buffer); combine pushes expert results back to their token;
// backward reverse-combine pulls and reverse-dispatch pushes on the same
// schedule (Cursor blog summary, "method points"). On one GPU the pull is a
// gather through the schedule and the push a fixed-order per-token sum.
#include "moe_internal.h"
#include "mx.cuh"
#include "ptx.cuh"
#include "prof.h"

namespace moe {

namespace {

__device__ __forceinline__ int token_of(int a, int T, int k) {
  const int A = T * k;
  return a < A ? a / k : (a - A) % T;
}

__device__ __forceinline__ int seg_search_dev(const int* v, int n, int64_t x) {
  int lo = 0, hi = n;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (v[mid] <= x) lo = mid; else hi = mid;
  }
  return lo;
}

// Locate routed tile g of lap L. Returns false when g is past the lap's routed tiles.
struct LapTile { int e; int slot0; int rows; int64_t rank0; };
__device__ __forceinline__ bool lap_tile(const int* lap_tiles, const int* counts, int E, int Ep, int C, int L, int g,
                                         LapTile& lt) {
  const int* v = lap_tiles + static_cast<int64_t>(L) * (Ep + 1);
  if (g >= v[E]) return false;
  const int e = seg_search_dev(v, E, g);
  const int mt = g - v[e];
  int len = counts[e] - L * C;
  len = len > C ? C : len;
  lt.e = e;
  lt.slot0 = mt * 128;
  lt.rows = min(128, len - mt * 128);
  lt.rank0 = static_cast<int64_t>(L) * C + mt * 128;
  return lt.rows > 0;
}

// The rows of lap L are the 128-row tiles of its tile list; each tile is
// covered by 16 groups of 8 rows and each row by one warp, so that even a
// lap with a few hot experts spreads over the whole GPU. Grid-stride loop
// over row groups. Rows past an expert's segment are written as zeros.
constexpr int kRowsPerGroup = 8;

__device__ __forceinline__ bool lap_row(const int* lap_tiles, const int* counts, const int* poff,
                                        const int* row_src, int T, int k, int E, int Ep, int C, int L, int gid,
                                        int warp, int64_t& ring_row, int& tok, int& a_out) {
  LapTile lt;
  if (!lap_tile(lap_tiles, counts, E, Ep, C, L, gid >> 4, lt)) return false;
  const int r = (gid & 15) * kRowsPerGroup + warp;
  ring_row = static_cast<int64_t>(lt.e) * C + lt.slot0 + r;
  tok = -1;
  a_out = -1;
  if (r < lt.rows) {
    a_out = row_src[poff[lt.e] + lt.rank0 + r];
    tok = token_of(a_out, T, k);
  }
  return true;
}

constexpr int kPermChunks = 14;   // 16-byte chunks a lane keeps in flight (a whole 7168-byte row per warp)

// ring[e*C + slot] <- the MX row of token t (codes and scales) for the rows of lap L:
// x_q into the x ring in the forward, MX(dy) into the dO ring in the backward.
__global__ void __launch_bounds__(256, 3) permute_lap_kernel(
    const uint8_t* __restrict__ xq, const uint8_t* __restrict__ xq_sf, const int* __restrict__ lap_tiles,
    const int* __restrict__ counts, const int* __restrict__ poff, const int* __restrict__ row_src, int T, int k,
    int d, int E, int Ep, int C, int L, uint8_t* __restrict__ ring, uint8_t* __restrict__ ring_sf) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_groups = lap_tiles[static_cast<int64_t>(L) * (Ep + 1) + E] * 16;
  const int chunks = d / 16, ktiles = d / 128;
  for (int gid = blockIdx.x; gid < n_groups; gid += gridDim.x) {
    int64_t row;
    int t, a;
    if (!lap_row(lap_tiles, counts, poff, row_src, T, k, E, Ep, C, L, gid, warp, row, t, a)) continue;
    const uint4* src = reinterpret_cast<const uint4*>(xq + static_cast<int64_t>(t < 0 ? 0 : t) * d);
    uint4* dst = reinterpret_cast<uint4*>(ring + row * d);
    for (int c0 = 0; c0 < chunks; c0 += 32 * kPermChunks) {   // all of a lane's chunks in flight
      uint4 v[kPermChunks];
#pragma unroll
      for (int u = 0; u < kPermChunks; ++u) {
        const int c = c0 + u * 32 + lane;
        v[u] = (t >= 0 && c < chunks) ? __ldg(src + c) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < kPermChunks; ++u) {
        const int c = c0 + u * 32 + lane;
        if (c < chunks) dst[c] = v[u];
      }
    }
    for (int kt = lane; kt < ktiles; kt += 32) {
      const uint32_t v = t >= 0 ? *reinterpret_cast<const uint32_t*>(xq_sf + sf_off(t, kt * 4, ktiles)) : 0u;
      *reinterpret_cast<uint32_t*>(ring_sf + sf_off(row, kt * 4, ktiles)) = v;
    }
  }
}

// Dispatch of every ring lap in one launch (moe_dispatch). Item = (expert e,
// ring buffer b, kDispSlots consecutive ring slots), experts taken in
// descending-count order so that the slots with the most laps start first.
// The item's warp writes, for each lap L = b, b + 2, ... of e in that order,
// the lap's rows for those slots (zero past the lap's rows up to its last
// 128-row tile): the same writes, in the same per-slot order, as the per-lap
// kernels; one thread's stores to a row are ordered, so the last lap wins.
// Lane l looks up the token of slot l % kDispSlots in lap l / kDispSlots of a
// batch of 32 / kDispSlots laps, so one dependent chain of index loads serves
// many rows; each row is then copied with kDispChunks 16-byte chunks a lane
// in flight. Measured (one GB300, dsv3_zipf): 2 slots per item beat 1, 4 and
// 8, and a TMA bulk-copy form through shared memory.
// L2 cache policies of the dispatch copies: the gathered MX(x) rows (about
// the size of L2 at the benchmark shape, each read k times) are kept, and the
// ring rows this stand-alone form writes, read by nothing soon after, go first.
__device__ __forceinline__ uint64_t pol_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t pol_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint4 ld_hint(const uint4* a, uint64_t pol) {
  uint4 v;
  asm volatile("ld.global.nc.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(a), "l"(pol));
  return v;
}
__device__ __forceinline__ void st_hint(uint4* a, uint4 v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.v4.u32 [%0], {%1, %2, %3, %4}, %5;"
               :: "l"(a), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "l"(pol) : "memory");
}
constexpr int kDispSlots = 2;
constexpr int kDispScaleJobs = 16;   // warps sharing one ring m-tile's scales
constexpr int kDispChunks = 7;

__global__ void __launch_bounds__(256, 4) dispatch_all_kernel(
    const uint8_t* __restrict__ xq, const int* __restrict__ counts, const int* __restrict__ poff,
    const int* __restrict__ row_src, const int* __restrict__ order, int k, int d, int E, int Ep, int C,
    uint8_t* __restrict__ ring) {
  constexpr int kLapsPerBatch = 32 / kDispSlots;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int groups = C / kDispSlots;
  const int64_t item = static_cast<int64_t>(blockIdx.x) * 8 + warp;
  if (item >= static_cast<int64_t>(Ep) * 2 * groups) return;
  const int ei = static_cast<int>(item / (2 * groups));
  const int rem = static_cast<int>(item - static_cast<int64_t>(ei) * 2 * groups);
  const int e = order[ei];              // every expert once; the shared one has no ring rows
  if (e >= E) return;
  const int b = rem / groups, s0 = (rem - b * groups) * kDispSlots;
  const int n = counts[e];
  if (static_cast<int64_t>(b) * C >= n) return;
  const int laps = static_cast<int>((n - static_cast<int64_t>(b) * C + 2LL * C - 1) / (2LL * C));   // laps b, b+2, ...
  const int p0 = poff[e];
  const int chunks = d >> 4;
  const uint64_t pfirst = pol_evict_first(), plast = pol_evict_last();
  for (int jb = 0; jb < laps; jb += kLapsPerBatch) {
    // lane: lap jb + lane / kDispSlots, slot s0 + lane % kDispSlots -> token, -1 (zero row) or -2 (no row)
    int tok = -2;
    {
      const int j = jb + lane / kDispSlots, slot = s0 + lane % kDispSlots;
      if (j < laps) {
        const int64_t L = b + 2LL * j;
        const int len = static_cast<int>(min(static_cast<int64_t>(C), n - L * C));
        if (slot < len) tok = row_src[p0 + L * C + slot] / k;
        else if (slot < (len + 127) / 128 * 128) tok = -1;
      }
    }
    const int nj = min(kLapsPerBatch, laps - jb);
    for (int jj = 0; jj < nj; ++jj) {
#pragma unroll 1
      for (int ss = 0; ss < kDispSlots; ++ss) {
        const int t = __shfl_sync(0xffffffffu, tok, jj * kDispSlots + ss);
        if (t == -2) continue;
        const int64_t row = (static_cast<int64_t>(b) * E + e) * C + s0 + ss;
        const uint4* src = reinterpret_cast<const uint4*>(xq + static_cast<int64_t>(t < 0 ? 0 : t) * d);
        uint4* dst = reinterpret_cast<uint4*>(ring + row * d);
        for (int c0 = 0; c0 < chunks; c0 += 32 * kDispChunks) {
          uint4 v[kDispChunks];
#pragma unroll
          for (int u = 0; u < kDispChunks; ++u) {
            const int c = c0 + u * 32 + lane;
            v[u] = (t >= 0 && c < chunks) ? ld_hint(src + c, plast) : make_uint4(0, 0, 0, 0);
          }
#pragma unroll
          for (int u = 0; u < kDispChunks; ++u) {
            const int c = c0 + u * 32 + lane;
            if (c < chunks) st_hint(dst + c, v[u], pfirst);
          }
        }

      }
    }
  }
}

// Scales of the ring dispatch: job (expert rank ei, buffer b, m-tile mt,
// k-tile group g) writes the tile's scales of k-tile groups g,
// g + kDispScaleJobs, ... for laps b, b + 2, ... in lap order (the last lap's
// stay), 128 rows at a time (tile_scales_from_rows).
__global__ void __launch_bounds__(256) dispatch_scales_kernel(
    const uint8_t* __restrict__ xq_sfr, const int* __restrict__ counts, const int* __restrict__ poff,
    const int* __restrict__ row_src, const int* __restrict__ order, int k, int d, int E, int Ep, int C,
    uint8_t* __restrict__ ring_sf) {
  const int lane = threadIdx.x & 31;
  const int64_t jb = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int mts = C / 128;
  if (jb >= static_cast<int64_t>(Ep) * 2 * mts * kDispScaleJobs) return;
  const int g = static_cast<int>(jb % kDispScaleJobs);
  const int64_t jt = jb / kDispScaleJobs;
  const int ei = static_cast<int>(jt / (2 * mts));
  const int rem = static_cast<int>(jt - static_cast<int64_t>(ei) * 2 * mts);
  const int e = order[ei];
  if (e >= E) return;
  const int b = rem / mts, mt = rem - b * mts;
  const int n = counts[e];
  uint8_t* atoms = ring_sf + ((static_cast<int64_t>(b) * E + e) * C / 128 + mt) * (d >> 7) * 512 + lane * 16;
  for (int64_t L = b; L * C < n; L += 2) {
    const int64_t len = min(static_cast<int64_t>(C), n - L * C);
    if (static_cast<int64_t>(mt) * 128 >= len) break;   // only the last lap can be shorter
    int tok[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t slot = static_cast<int64_t>(mt) * 128 + lane + 32 * j;
      tok[j] = slot < len ? row_src[poff[e] + L * C + slot] / k : -1;
    }
    tile_scales_from_rows(xq_sfr, tok, d, atoms, g, kDispScaleJobs);
  }
}

// y[t] = bf16(sum_{j<k} w[t,j] O[t,j] + sum_s O_shared[s][t]), fp32 in slot order.
__global__ void combine_kernel(const __nv_bfloat16* __restrict__ O, const float* __restrict__ topk_w, int T, int k,
                               int S, int d, __nv_bfloat16* __restrict__ y) {
  const int chunks = d / 8;
  const int64_t gid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (gid >= static_cast<int64_t>(T) * chunks) return;
  const int t = static_cast<int>(gid / chunks), c = static_cast<int>(gid - static_cast<int64_t>(t) * chunks);
  float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  for (int j = 0; j < k; ++j) {
    const int64_t a = static_cast<int64_t>(t) * k + j;
    const float w = topk_w[a];
    const uint4 u = reinterpret_cast<const uint4*>(O + a * d)[c];
    const uint32_t q[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      acc[2 * i] = fmaf(w, __uint_as_float(q[i] << 16), acc[2 * i]);
      acc[2 * i + 1] = fmaf(w, __uint_as_float(q[i] & 0xFFFF0000u), acc[2 * i + 1]);
    }
  }
  for (int s = 0; s < S; ++s) {
    const int64_t a = static_cast<int64_t>(T) * k + static_cast<int64_t>(s) * T + t;
    const uint4 u = reinterpret_cast<const uint4*>(O + a * d)[c];
    const uint32_t q[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      acc[2 * i] += __uint_as_float(q[i] << 16);
      acc[2 * i + 1] += __uint_as_float(q[i] & 0xFFFF0000u);
    }
  }
  reinterpret_cast<uint4*>(y + static_cast<int64_t>(t) * d)[c] =
      make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]), pack_bf16x2(acc[4], acc[5]),
                 pack_bf16x2(acc[6], acc[7]));
}

// One warp per token: dw[t,j] = <dy[t], O[t,j]> (fixed lane-strided order and
// a fixed butterfly), then the router logit gradient
//   Z = sum_j s_j, c = sum_j dw_j w_j, dl_j = (dw_j - c) / Z * s_j (1 - s_j).
__global__ void rev_combine_dw_kernel(const __nv_bfloat16* __restrict__ dy, const __nv_bfloat16* __restrict__ O,
                                      const float* __restrict__ topk_w, const float* __restrict__ s_sel, int T, int k,
                                      int d, float* __restrict__ dw, float* __restrict__ dl) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x >> 5) + warp;
  if (t >= T) return;
  const int chunks = d / 8;
  // One pass over the row: each dy chunk is loaded once and multiplied with
  // the k output rows; every per-slot sum still runs over the chunks in
  // increasing order, then a fixed xor-shuffle tree.
  float dws[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) dws[j] = 0.0f;
  const uint4* pdy = reinterpret_cast<const uint4*>(dy + static_cast<int64_t>(t) * d);
  const uint4* po = reinterpret_cast<const uint4*>(O + static_cast<int64_t>(t) * k * d);
#pragma unroll 2
  for (int c = lane; c < chunks; c += 32) {
    const uint4 u = pdy[c];
    uint4 o[8];
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (j < k) o[j] = po[static_cast<int64_t>(j) * chunks + c];
    const uint32_t qu[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (j < k) {
        const uint32_t qo[4] = {o[j].x, o[j].y, o[j].z, o[j].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          dws[j] = fmaf(__uint_as_float(qu[i] << 16), __uint_as_float(qo[i] << 16), dws[j]);
          dws[j] = fmaf(__uint_as_float(qu[i] & 0xFFFF0000u), __uint_as_float(qo[i] & 0xFFFF0000u), dws[j]);
        }
      }
    }
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) dws[j] += __shfl_xor_sync(0xffffffffu, dws[j], o);
  }
  if (lane == 0) {
    const int64_t base = static_cast<int64_t>(t) * k;
    float Z = s_sel[base];
    for (int j = 1; j < k; ++j) Z = __fadd_rn(Z, s_sel[base + j]);
    float c = 0.0f;
    for (int j = 0; j < k; ++j) c = fmaf(dws[j], topk_w[base + j], c);
    for (int j = 0; j < k; ++j) {
      const float s = s_sel[base + j];
      dw[base + j] = dws[j];
      dl[base + j] = (dws[j] - c) / Z * (s * (1.0f - s));
    }
  }
}

// dx[t] = bf16(sum_{j<k} DX[t,j] + sum_s DX_shared[s][t] + sum_j dl[t,j] Wr[idx[t,j]]), fixed order.
__global__ void reverse_dispatch_kernel(const __nv_bfloat16* __restrict__ DX, const float* __restrict__ dl,
                                        const int32_t* __restrict__ idx, const __nv_bfloat16* __restrict__ wr, int T,
                                        int k, int S, int d, __nv_bfloat16* __restrict__ dx) {
  const int chunks = d / 8;
  const int64_t gid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (gid >= static_cast<int64_t>(T) * chunks) return;
  const int t = static_cast<int>(gid / chunks), c = static_cast<int>(gid - static_cast<int64_t>(t) * chunks);
  float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  auto add_row = [&](const __nv_bfloat16* row, float scale, bool scaled) {
    const uint4 u = reinterpret_cast<const uint4*>(row)[c];
    const uint32_t q[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float lo = __uint_as_float(q[i] << 16), hi = __uint_as_float(q[i] & 0xFFFF0000u);
      if (scaled) {
        acc[2 * i] = fmaf(scale, lo, acc[2 * i]);
        acc[2 * i + 1] = fmaf(scale, hi, acc[2 * i + 1]);
      } else {
        acc[2 * i] += lo;
        acc[2 * i + 1] += hi;
      }
    }
  };
  for (int j = 0; j < k; ++j) add_row(DX + (static_cast<int64_t>(t) * k + j) * d, 1.0f, false);
  for (int s = 0; s < S; ++s) add_row(DX + (static_cast<int64_t>(T) * k + static_cast<int64_t>(s) * T + t) * d, 1.0f, false);
  for (int j = 0; j < k; ++j) {
    const int64_t a = static_cast<int64_t>(t) * k + j;
    add_row(wr + static_cast<int64_t>(idx[a]) * d, dl[a], true);
  }
  reinterpret_cast<uint4*>(dx + static_cast<int64_t>(t) * d)[c] =
      make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]), pack_bf16x2(acc[4], acc[5]),
                 pack_bf16x2(acc[6], acc[7]));
}

// dWr[e][c] = bf16(sum over the 32-row blocks of expert e of part[b][c]).
// 8 groups of 32 threads each sum a contiguous run of blocks; the 8 group
// sums are then added in group order (a fixed order).
__global__ void router_dwr_kernel(const float* __restrict__ part, const int* __restrict__ poff, int d,
                                  __nv_bfloat16* __restrict__ dwr) {
  __shared__ float4 red[8][32];
  const int e = blockIdx.y;
  const int grp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = (blockIdx.x * 32 + lane) * 4;
  const int b0 = poff[e] / 32, b1 = poff[e + 1] / 32;
  const int nb = b1 - b0;
  const int per = (nb + 7) / 8;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (c < d) {
    for (int b = b0 + grp * per; b < b0 + (grp + 1) * per && b < b1; ++b) {
      const float4 v = *reinterpret_cast<const float4*>(part + static_cast<int64_t>(b) * d + c);
      acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
    }
  }
  red[grp][lane] = acc;
  __syncthreads();
  if (grp == 0 && c < d) {
    float4 s = red[0][lane];
    for (int g = 1; g < 8; ++g) {
      const float4 v = red[g][lane];
      s.x += v.x; s.y += v.y; s.z += v.z; s.w += v.w;
    }
    uint2 o = make_uint2(pack_bf16x2(s.x, s.y), pack_bf16x2(s.z, s.w));
    *reinterpret_cast<uint2*>(dwr + static_cast<int64_t>(e) * d + c) = o;
  }
}

}  // namespace

// Bytes of one ring buffer (codes), E * C rows of d.
static size_t ring_bytes(const Dims& m) { return static_cast<size_t>(m.E) * m.C * m.d; }

// Blocks of the lap kernels: enough row groups to cover a full lap, capped at 16 per SM.
static int lap_blocks(const Dims& m) {
  const int64_t groups = static_cast<int64_t>(m.E) * (m.C / 128) * 16;
  const int64_t cap = static_cast<int64_t>(num_sms()) * 16;
  return static_cast<int>(groups < cap ? groups : cap);
}

void launch_dispatch_all(const Dims& m, const Layout& L, void* ws, cudaStream_t s) {
  // codes: items (expert, buffer, slot pair); scales: jobs (expert, buffer, m-tile, k-tile group).
  // Both launches carry the same profile name: together they are the dispatch.
  const int64_t items = static_cast<int64_t>(m.Ep) * 2 * (m.C / kDispSlots);
  const int64_t jobs = static_cast<int64_t>(m.Ep) * 2 * (m.C / 128) * kDispScaleJobs;
  if (items == 0) return;
  launch_kernel("dispatch_all", dispatch_all_kernel, dim3(static_cast<unsigned>(ceil_div(items, 8))), dim3(256), 0, s,
      ws_ptr<uint8_t>(L, ws, MOE_WS_XQ), ws_ptr<int>(L, ws, MOE_WS_COUNTS), ws_ptr<int>(L, ws, MOE_WS_POFF),
      ws_ptr<int>(L, ws, MOE_WS_ROWSRC), ws_ptr<int>(L, ws, MOE_WS_ORDER), m.k, m.d, m.E, m.Ep, m.C,
      ws_ptr<uint8_t>(L, ws, MOE_WS_RING_X));
  launch_kernel("dispatch_all", dispatch_scales_kernel, dim3(static_cast<unsigned>(ceil_div(jobs, 8))), dim3(256), 0, s,
      ws_ptr<uint8_t>(L, ws, MOE_WS_XQ_SFC), ws_ptr<int>(L, ws, MOE_WS_COUNTS), ws_ptr<int>(L, ws, MOE_WS_POFF),
      ws_ptr<int>(L, ws, MOE_WS_ROWSRC), ws_ptr<int>(L, ws, MOE_WS_ORDER), m.k, m.d, m.E, m.Ep, m.C,
      ws_ptr<uint8_t>(L, ws, MOE_WS_RING_X_SF));
}

void launch_permute_lap(const Dims& m, int lap, bool dO, const Layout& L, void* ws, cudaStream_t s) {
  const int blocks = lap_blocks(m);
  if (blocks == 0) return;
  launch_kernel(dO ? "permute_lap_dO" : "permute_lap", permute_lap_kernel, dim3(blocks), dim3(256), 0, s,
      ws_ptr<uint8_t>(L, ws, dO ? MOE_WS_DOS : MOE_WS_XQ), ws_ptr<uint8_t>(L, ws, dO ? MOE_WS_DOS_SF : MOE_WS_XQ_SF),
      ws_ptr<int>(L, ws, MOE_WS_LAPTILES), ws_ptr<int>(L, ws, MOE_WS_COUNTS), ws_ptr<int>(L, ws, MOE_WS_POFF),
      ws_ptr<int>(L, ws, MOE_WS_ROWSRC), m.T, m.k, m.d, m.E, m.Ep, m.C, lap,
      ws_ptr<uint8_t>(L, ws, dO ? MOE_WS_RING_DO : MOE_WS_RING_X) + (lap % kRingBufs) * ring_bytes(m),
      ws_ptr<uint8_t>(L, ws, dO ? MOE_WS_RING_DO_SF : MOE_WS_RING_X_SF) + (lap % kRingBufs) * ring_bytes(m) / 32);
}

void launch_combine(const Dims& m, const float* topk_w, const Layout& L, void* ws, void* y, cudaStream_t s) {
  const int64_t n = static_cast<int64_t>(m.T) * (m.d / 8);
  if (n == 0) return;
  launch_kernel("combine", combine_kernel, dim3(static_cast<unsigned>(ceil_div(n, 256))), dim3(256), 0, s,
      ws_ptr<__nv_bfloat16>(L, ws, MOE_WS_O), topk_w, m.T, m.k, m.S, m.d, static_cast<__nv_bfloat16*>(y));
}

void launch_rev_combine_dw(const Dims& m, const void* dy, const float* topk_w, const Layout& L, void* ws,
                           cudaStream_t s) {
  if (m.T == 0) return;
  launch_kernel("rev_combine_dw", rev_combine_dw_kernel, dim3(static_cast<unsigned>(ceil_div(m.T, 8))), dim3(256), 0, s,
      static_cast<const __nv_bfloat16*>(dy), ws_ptr<__nv_bfloat16>(L, ws, MOE_WS_O), topk_w,
      ws_ptr<float>(L, ws, MOE_WS_SSEL), m.T, m.k, m.d, ws_ptr<float>(L, ws, MOE_WS_DW),
      ws_ptr<float>(L, ws, MOE_WS_DL));
}

void launch_reverse_dispatch(const Dims& m, const int32_t* idx, const void* w_router, const Layout& L, void* ws,
                             void* dx, cudaStream_t s) {
  const int64_t n = static_cast<int64_t>(m.T) * (m.d / 8);
  if (n == 0) return;
  launch_kernel("reverse_dispatch", reverse_dispatch_kernel, dim3(static_cast<unsigned>(ceil_div(n, 256))), dim3(256), 0,
                s, ws_ptr<__nv_bfloat16>(L, ws, MOE_WS_DXE), ws_ptr<float>(L, ws, MOE_WS_DL), idx,
      static_cast<const __nv_bfloat16*>(w_router), m.T, m.k, m.S, m.d, static_cast<__nv_bfloat16*>(dx));
}

void launch_router_dwr(const Dims& m, const Layout& L, void* ws, void* dw_router, cudaStream_t s) {
  dim3 grid(static_cast<unsigned>(ceil_div(m.d, 128)), static_cast<unsigned>(m.E));
  launch_kernel("router_dwr", router_dwr_kernel, grid, dim3(256), 0, s, ws_ptr<float>(L, ws, MOE_WS_DWR_PART),
                ws_ptr<int>(L, ws, MOE_WS_POFF), m.d, static_cast<__nv_bfloat16*>(dw_router));
}

}  // namespace moe
