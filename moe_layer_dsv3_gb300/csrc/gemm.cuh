// Persistent, warp-specialised grouped GEMM on the 5th-generation tensor cores.
//
//   D[128 x BN] (TMEM, fp32) = sum_k A[128 x k] . B[BN x k]^T
//
// A and B are K-major tiles staged by TMA (128-byte swizzle, 128 bytes of K
// per stage: 128 E4M3 values or 64 bf16 values). For MXFP8 the E8M0 scales
// of each stage arrive by bulk copy in the tiled atom layout and are moved
// into TMEM with tcgen05.cp; tcgen05.mma.kind::mxf8f6f4.block_scale applies
// them per 32-element block. The bf16 path (router logits) uses
// tcgen05.mma.kind::f16.
//
// Roles (192 threads): warp 0 = TMA producer, warp 1 = MMA issuer and TMEM
// owner, warps 2-5 = epilogue (each reads the TMEM lane quarter warp%4).
// Work list: "tiles" of 128 rows x BN columns, decoded from the device-side
// schedule, so the host never learns per-expert counts.
//
// The all-laps ring modes add mover warps (two by default: 256 threads) that
// fill the ring token buffers while the other warps compute, so one persistent launch
// covers every lap. Ordering goes through per-m-tile device counters:
//   moved[gm]    8-row groups of m-tile gm written into its ring slot; the
//                producer waits for all 16 before its first TMA load of gm;
//   consumed[gm] tiles of gm whose accumulators are complete (so all their A
//                loads have landed), bumped by the epilogue; the movers of
//                the same slot's next tenant (lap + 2) wait for all N / BN.
// Both lists are walked by every CTA in increasing position of the schedule's
// walk order (LAPORDER: laps 2P and 2P+1 of an expert side by side, so its
// weights stream once for both, and each expert's pairs spread evenly over
// the launch). Every position's previous ring tenant (lap - 2) sits at an
// earlier position, so every wait points to an earlier position or to a move
// of the same one, and the waits cannot form a cycle once all CTAs are
// resident (cooperative launch).
//
// A tile learns its expert, rows and ring slot from one entry of a table the
// schedule writes (the ring positions' entries, the push m-tiles' experts, the
// weight gradients' per-expert K ranges). Searching the lap and expert prefix
// sums instead costs a chain of dependent global loads per tile, which the
// producer and MMA threads would pay between tiles while the tensor pipe idles.
#pragma once
#include <cuda_bf16.h>

#include "moe_internal.h"
#include "mx.cuh"
#include "ptx.cuh"

namespace moe {

constexpr int kRouterMode = 5;   // bf16 x bf16 router logits

// Host-side tensor-map helpers (k_gemm.cu).
bool get_encode();
// 2-D K-major operand [rows][cols] (1- or 2-byte elements), box 128 bytes x box_rows, 128-byte swizzle.
bool make_tmap(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int box_rows, bool bf16);
// 2-D bf16 output [rows][cols] written by TMA stores, box 64 columns x 128 rows, 128-byte swizzle.
bool make_tmap_out(CUtensorMap* m, void* base, int64_t rows, int64_t cols);
// Tiled scale array as uint32 [atoms][128]: one box = one 512-byte scale atom.
bool make_tmap_sf(CUtensorMap* m, const void* base, int64_t atoms);

// The epilogue / tile shape a mode shares with its per-lap form.
__host__ __device__ constexpr int base_mode(int mode) {
  return mode == kSwigluFwdRing ? kSwigluFwd : (mode == kSwigluBwdRing ? kSwigluBwd : (mode == kPushNv4 ? kPush : mode));
}
__host__ __device__ constexpr bool ring_mode(int mode) { return mode == kSwigluFwdRing || mode == kSwigluBwdRing; }
// 192 threads (producer, MMA, 4 epilogue warps), plus MV mover warps in the all-laps ring modes.
__host__ __device__ constexpr int gemm_threads(int mode, int mv) { return ring_mode(mode) ? 192 + 32 * mv : 192; }

// Mover warps per CTA of the all-laps ring modes: the library default, and
// the largest count GEMM1 can take (its SwiGLU epilogue warps hold 255
// registers, so 8 warps already fill the register file).
constexpr int kMoverWarpsDefault = 2;
constexpr int kMoverWarpsGemm1Max = 2;
constexpr int kMoveRows = 8;                    // ring rows per move item
constexpr int kMoveItems = 128 / kMoveRows;     // move items per m-tile

struct GemmParams {
  int N;                 // B rows per expert (output columns per expert)
  int K;                 // reduction length (elements) for fixed-K modes
  int a_ktiles, b_ktiles;// 128-wide K tiles per row of the stored A / B operand (scale atoms)
  const uint8_t* a_sf; const uint8_t* a2_sf; const uint8_t* b_sf;
  const int* counts; const int* poff; const int* lap_tiles; const int* row_src;
  const int* order;      // experts by descending count (weight-gradient tile order)
  int E, Ep, C, lap, T, k;
  int M;                 // plain / router / wgrad output rows per expert
  int static_tiles;      // tile count when it does not depend on the schedule
  void* out; void* out2; int ldo;
  float alpha;           // NVFP4 plain mode: product of the operands' tensor scales
  uint8_t* q_rows; uint8_t* q_rows_sf; int q_rows_ktiles;
  uint8_t* q_tok; uint8_t* q_tok_sf; int64_t q_tok_pitch;
  __nv_bfloat16* gu; int I;
  const float* gate;
  int* status;
  // all-laps ring modes
  const int* lapbase; int Lb; int d;
  const int4* ring_info; // per walk position (pair-spread order): the decoded ring m-tile (two int4,
                         // written by the schedule); tiles and move items go in position order
  const int* push_info;  // push modes, per m-tile of the padded rank rows: e | valid << 16 (or null: search)
  const int4* wg_info;   // weight gradients, per rank of `order`: {e, first K tile, K tiles, 0} (or null)
  int* moved; int* consumed;
  const uint8_t* mv_xq; const uint8_t* mv_xq_sf;
  const uint8_t* mv_xq_sfr;   // the same scales row-major [T][d/32]
  uint8_t* ring; uint8_t* ring_sf;
};

template <int BN, int MODE>
struct GemmCfg {
  static constexpr bool kBf16 = MODE == kRouterMode;
  // NVFP4: a 128-byte stage row holds 256 E2M1 values; the scales (one E4M3
  // per 16) of a stage are 4 atoms per 128 rows, one atom per K = 64 MMA.
  static constexpr bool kNv4 = MODE == kPlainNv4 || MODE == kGroupedNv4 || MODE == kPushNv4;
  // Weight gradients stage their bf16 output tile in shared memory and write
  // it with TMA stores, so the tile's DRAM write overlaps the next mainloop.
  static constexpr bool kTmaOut = MODE == kWgrad;
  // (the NVFP4 push mode's stages carry 4 scale atoms per operand tile and
  // its epilogue a scratch tile per warp: 3 stages fit at BN = 256, 5 at 128)
  static constexpr int kStages = kTmaOut ? (BN >= 256 ? 3 : 5)
                                         : (MODE == kPushNv4 ? (BN >= 256 ? 3 : 5)
                                                             : (BN >= 256 ? 4 : (BN >= 128 ? 6 : 8)));
  static constexpr int kOutBytes = kTmaOut ? 128 * BN * 2 : 0;
  static constexpr int kABytes = 128 * 128;
  static constexpr int kBBytes = BN * 128;
  static constexpr int kSfAtoms = kNv4 ? 4 : 1;                    // scale atoms per 128 rows per stage
  static constexpr int kSfaBytes = kBf16 ? 0 : 512 * kSfAtoms;
  static constexpr int kSfbBytes = kBf16 ? 0 : (BN / 128) * 512 * kSfAtoms;
  static constexpr int kTx = kABytes + kBBytes + kSfaBytes + kSfbBytes;
  static constexpr int kStageBytes = ((kTx + 1023) / 1024) * 1024;
  static constexpr int kSfCols = kBf16 ? 0 : kSfAtoms * (4 + (BN / 128) * 4);   // TMEM columns of scales per stage
  static constexpr int kSfCol0 = 256;
  // Accumulator buffers in TMEM: two when they fit below the scale columns, so
  // the epilogue of one tile overlaps the mainloop of the next.
  static constexpr int kNumAcc = (2 * BN <= kSfCol0) ? 2 : 1;
  static constexpr int kKElems = kBf16 ? 64 : (kNv4 ? 256 : 128);   // K elements per stage
  static constexpr int kTmaX = kBf16 ? 64 : 128;                     // tensor-map x extent per stage (elements / bytes)
  static constexpr int kBarBytes = 256;
  static constexpr int kBase = base_mode(MODE);
  // Per epilogue warp, 32 x 33 fp32: the SwiGLU forward's transpose tile, or
  // the 32-row x 128-byte store-coalescing tile of the push and dh epilogues.
  static constexpr int kScratchBytes = (kBase == kSwigluFwd || kBase == kPush || kBase == kSwigluBwd) ? 4 * 32 * 33 * 4 : 0;
  static constexpr int kSmem = 1024 + kStages * kStageBytes + kOutBytes + kBarBytes + kScratchBytes;
  static_assert(kSmem <= 232448, "shared memory budget");
  static_assert(kSfCol0 + kStages * kSfCols <= 512, "TMEM budget");
  static_assert(BN <= 256, "accumulator budget");
};

struct TileInfo {
  int e;
  int64_t a_row;     // A row of the tile's first row
  int64_t b_row;     // B row of the tile's first column
  int k0;            // first K stage
  int nk;            // number of K stages
  int64_t prow0;     // padded rank row of the tile's first row (grouped-M modes)
  int valid;         // rows of the tile that hold real assignments
  int n0;            // first output column
  int m0;            // first output row (wgrad / plain / router)
  bool use_a2;
  int gm;            // all-laps ring modes: global m-tile of a ring tile, else -1
};

// Largest e in [0, n) with v[e] <= x < v[e+1] (v nondecreasing, v[0] <= x < v[n]).
__device__ __forceinline__ int seg_search(const int* v, int n, int64_t x) {
  int lo = 0, hi = n;   // invariant v[lo] <= x < v[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (v[mid] <= x) lo = mid; else hi = mid;
  }
  return lo;
}

template <int BN, int MODE>
__device__ __forceinline__ int gemm_num_tiles(const GemmParams& p) {
  if constexpr (ring_mode(MODE)) {
    return p.lapbase[p.Lb] * (p.N / BN);
  } else if constexpr (MODE == kSwigluFwd || MODE == kSwigluBwd) {
    return p.lap_tiles[p.lap * (p.Ep + 1) + p.Ep] * (p.N / BN);
  } else if constexpr (MODE == kPush || MODE == kGroupedNv4 || MODE == kPushNv4) {
    return (p.poff[p.Ep] / 128) * (p.N / BN);
  } else if constexpr (MODE == kWgrad) {
    // positions of the two-ended schedule (see gemm_decode): enough rounds for the heavy half
    const int N = p.static_tiles;
    const int g = gridDim.x;
    if (g < 2 || (g & 1)) return N;
    const int heavy = (N + 1) / 2;
    return ((heavy + g / 2 - 1) / (g / 2)) * g;
  } else {
    return p.static_tiles;
  }
}

// Tile (g, n) of ring lap L: g indexes the lap's m-tiles (experts in order;
// the shared expert's tiles, read in place from A2, only in lap 0). The ring
// rows of lap L start at ring_row0.
template <int BN>
__device__ __forceinline__ bool lap_decode(const GemmParams& p, int L, int g, int n, int64_t ring_row0,
                                           TileInfo& t) {
  const int* lt = p.lap_tiles + static_cast<int64_t>(L) * (p.Ep + 1);
  const int e = seg_search(lt, p.Ep, g);
  const int mt = g - lt[e];
  const bool shared = e >= p.E;
  const int64_t rank0 = shared ? static_cast<int64_t>(mt) * 128 : static_cast<int64_t>(L) * p.C + mt * 128;
  const int cnt = p.counts[e];
  t.e = e;
  t.use_a2 = shared;
  t.a_row = shared ? static_cast<int64_t>(mt) * 128 : ring_row0 + static_cast<int64_t>(e) * p.C + mt * 128;
  t.b_row = static_cast<int64_t>(e) * p.N + static_cast<int64_t>(n) * BN;
  t.k0 = 0;
  t.nk = p.K / kTileK;
  t.prow0 = p.poff[e] + rank0;
  const int64_t v = cnt - rank0;
  t.valid = v < 0 ? 0 : (v > 128 ? 128 : static_cast<int>(v));
  t.n0 = n * BN;
  t.m0 = 0;
  t.gm = -1;
  return t.prow0 + 128 <= p.poff[e + 1] && t.valid > 0;
}

template <int BN, int MODE>
__device__ __forceinline__ bool gemm_decode(const GemmParams& p, int tile, TileInfo& t) {
  using Cf = GemmCfg<BN, MODE>;
  t.gm = -1;
  if constexpr (ring_mode(MODE)) {
    // position pos of the walk, n-tile n; the schedule decoded the position's
    // m-tile (lap-major global m-tile gm, expert, rows) into one table entry
    const int nt = p.N / BN;
    const int pos = tile / nt, n = tile - pos * nt;
    const int4 a = p.ring_info[2 * pos];
    const int e = a.y & 0xFFFF;
    t.e = e;
    t.use_a2 = ((a.y >> 25) & 1) != 0;
    t.a_row = a.z;
    t.b_row = static_cast<int64_t>(e) * p.N + static_cast<int64_t>(n) * BN;
    t.k0 = 0;
    t.nk = p.K / kTileK;
    t.prow0 = a.w;
    t.valid = (a.y >> 16) & 0xFF;
    t.n0 = n * BN;
    t.m0 = 0;
    t.gm = t.use_a2 ? -1 : a.x;
    return ((a.y >> 24) & 1) != 0;
  } else if constexpr (MODE == kSwigluFwd || MODE == kSwigluBwd) {
    const int nt = p.N / BN;
    const int g = tile / nt, n = tile - (tile / nt) * nt;
    return lap_decode<BN>(p, p.lap, g, n, 0, t);
  } else if constexpr (MODE == kPush || MODE == kGroupedNv4 || MODE == kPushNv4) {
    // padded rank rows of the schedule: m-tile g belongs to the expert whose segment holds it
    const int nt = p.N / BN;
    const int g = tile / nt, n = tile - (tile / nt) * nt;
    const int64_t prow0 = static_cast<int64_t>(g) * 128;
    int e, valid;
    if (p.push_info != nullptr) {   // decoded by the schedule
      const int v = p.push_info[g];
      e = v & 0xFFFF;
      valid = v >> 16;
    } else {
      e = seg_search(p.poff, p.Ep, prow0);
      const int64_t v = p.counts[e] - (prow0 - p.poff[e]);
      valid = v < 0 ? 0 : (v > 128 ? 128 : static_cast<int>(v));
    }
    t.e = e;
    t.use_a2 = false;
    t.a_row = prow0;
    t.b_row = static_cast<int64_t>(e) * p.N + static_cast<int64_t>(n) * BN;
    t.k0 = 0;
    t.nk = p.K / Cf::kKElems;
    t.prow0 = prow0;
    t.valid = valid;
    t.n0 = n * BN;
    t.m0 = MODE == kGroupedNv4 ? static_cast<int>(prow0) : 0;   // rank-ordered output rows
    return true;
  } else if constexpr (MODE == kWgrad) {
    // Two-ended schedule: in each round half of the CTAs take the next tile from
    // the front of the tile list (experts with the most tokens: long K,
    // compute-bound) and half from the back (experts with few or no tokens:
    // bound by writing their gradient tile); a CTA alternates ends from round
    // to round. Compute and DRAM writes then overlap throughout the launch.
    const int nt = p.N / BN, mt = p.M / 128;
    const int per = nt * mt;
    const int N = p.static_tiles;
    int q = tile;
    const int g = gridDim.x;
    if (g >= 2 && !(g & 1)) {
      const int round = tile / g, b = tile - round * g;
      const int k = round * (g / 2) + (b >> 1);
      if (((b + round) & 1) == 0) {
        if (k >= (N + 1) / 2) return false;
        q = k;
      } else {
        if (k >= N / 2) return false;
        q = N - 1 - k;
      }
    }
    const int rem = q - (q / per) * per;
    const int mi = rem / nt, n = rem - (rem / nt) * nt;
    if (p.wg_info != nullptr) {   // decoded by the schedule
      const int4 w = p.wg_info[q / per];
      t.e = w.x;
      t.k0 = w.y;
      t.nk = w.z;
    } else {
      const int e = p.order[q / per];
      t.e = e;
      t.k0 = p.poff[e] / 128;
      t.nk = (p.poff[e + 1] - p.poff[e]) / 128;
    }
    t.use_a2 = false;
    t.a_row = static_cast<int64_t>(mi) * 128;
    t.b_row = static_cast<int64_t>(n) * BN;
    t.prow0 = 0;
    t.valid = 128;
    t.n0 = n * BN;
    t.m0 = mi * 128;
    return true;
  } else {   // plain, router
    const int nt = (p.N + BN - 1) / BN;
    const int mi = tile / nt, n = tile - (tile / nt) * nt;
    t.e = 0;
    t.use_a2 = false;
    t.a_row = static_cast<int64_t>(mi) * 128;
    t.b_row = static_cast<int64_t>(n) * BN;
    t.k0 = 0;
    t.nk = p.K / Cf::kKElems;
    t.prow0 = 0;
    t.valid = 128;
    t.n0 = n * BN;
    t.m0 = mi * 128;
    return true;
  }
}

__device__ __forceinline__ void store_bf16x32(__nv_bfloat16* dst, const float* v) {
  uint4* p = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int q = 0; q < 4; ++q)
    p[q] = make_uint4(pack_bf16x2(v[8 * q], v[8 * q + 1]), pack_bf16x2(v[8 * q + 2], v[8 * q + 3]),
                      pack_bf16x2(v[8 * q + 4], v[8 * q + 5]), pack_bf16x2(v[8 * q + 6], v[8 * q + 7]));
}

// Read this thread's whole accumulator row (BN fp32 columns) into packed bf16
// pairs, then hand the TMEM buffer back to the MMA warp at once, so the next
// tile's MMAs start while the row is still being written out.
// kAlpha: the row is scaled by alpha first (NVFP4: the operands' tensor scales).
template <int BN, bool kAlpha = false>
__device__ __forceinline__ void drain_acc_bf16(uint32_t tacc, bool have_acc, uint32_t* packed, uint64_t* acce,
                                               float alpha = 1.0f) {
  if (have_acc && kAlpha) {
    // one load per wait: the scaling leaves no registers for a second one
#pragma unroll
    for (int c = 0; c < BN / 32; ++c) {
      uint32_t r0[32];
      tmem_ld32_async(tacc + c * 32, r0);
      tmem_wait_ld();
#pragma unroll
      for (int j = 0; j < 32; ++j) reg_fence(r0[j]);
#pragma unroll
      for (int j = 0; j < 16; ++j)
        packed[c * 16 + j] = pack_bf16x2(__fmul_rn(__uint_as_float(r0[2 * j]), alpha),
                                         __fmul_rn(__uint_as_float(r0[2 * j + 1]), alpha));
    }
  } else if (have_acc) {
    // two loads in flight per wait
#pragma unroll
    for (int c = 0; c < BN / 32; c += 2) {
      uint32_t r0[32], r1[32];
      tmem_ld32_async(tacc + c * 32, r0);
      tmem_ld32_async(tacc + (c + 1) * 32, r1);
      tmem_wait_ld();
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        reg_fence(r0[j]);
        reg_fence(r1[j]);
      }
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        packed[c * 16 + j] = pack_bf16x2(__uint_as_float(r0[2 * j]), __uint_as_float(r0[2 * j + 1]));
        packed[(c + 1) * 16 + j] = pack_bf16x2(__uint_as_float(r1[2 * j]), __uint_as_float(r1[2 * j + 1]));
      }
    }
  } else {
#pragma unroll
    for (int j = 0; j < BN / 2; ++j) packed[j] = 0u;
  }
  tc_fence_before();
  mbar_arrive(acce);
}

// ---------------------------------------------------------------- ring movers
// One move item = kMoveRows consecutive ring rows of one m-tile. Lane r < 8
// holds the assignment of row r (-1 past the expert's count: zero row).

// A finished item becomes visible (to TMA reads too) before moved[gm] counts it.
__device__ __forceinline__ void publish_move(int* ctr, int lane) {
  fence_proxy_async_global();
  __threadfence();
  __syncwarp();
  if (lane == 0) red_release_add(ctr, 1);
}

// Ring row <- the MX row codes of its token (x in the forward, dy in the
// backward). The item's 16-byte chunks are walked flat (consecutive lanes,
// consecutive chunks) in rounds of kFwdU chunks a lane; the next round's loads
// are issued before this round's stores, so two rounds are in flight. The
// scales go per m-tile (move_tile_scales).
constexpr int kFwdU = 8;

__device__ __forceinline__ void move_rows(const GemmParams& p, int lane, int a_lane, int64_t ring_row0) {
  const int d = p.d;
  const int chunks = d >> 4;   // 16-byte chunks per row (d is a multiple of 128: at least 8)
  const int rounds = (kMoveRows * chunks + 32 * kFwdU - 1) / (32 * kFwdU);
  const int tok_l = a_lane >= 0 ? a_lane / p.k : -1;
  const uint4 zero = make_uint4(0, 0, 0, 0);
  // Flat chunk f = (round * kFwdU + u) * 32 + lane is (row r, chunk c); both
  // cursors advance by 32 chunks a step, so no division per chunk.
  int lr = lane / chunks, lc = lane - lr * chunks;   // load cursor
  int sr = lr, sc = lc;                              // store cursor (one round behind)
  auto step = [&](int& r, int& c) {
    c += 32;
    while (c >= chunks) { c -= chunks; ++r; }   // at most 32 / chunks times
  };
  uint4 nxt[kFwdU];
  auto load = [&](uint4* v) {
#pragma unroll
    for (int u = 0; u < kFwdU; ++u) {
      const int t = __shfl_sync(0xffffffffu, tok_l, lr < kMoveRows ? lr : kMoveRows - 1);
      v[u] = (lr < kMoveRows && t >= 0)
                 ? ld_global_u4(reinterpret_cast<const uint4*>(p.mv_xq + static_cast<int64_t>(t) * d) + lc)
                 : zero;
      step(lr, lc);
    }
  };
  load(nxt);
  for (int rd = 0; rd < rounds; ++rd) {
    uint4 cur[kFwdU];
#pragma unroll
    for (int u = 0; u < kFwdU; ++u) cur[u] = nxt[u];
    if (rd + 1 < rounds) load(nxt);
    __syncwarp();   // keeps the next round's loads ahead of this round's stores
#pragma unroll
    for (int u = 0; u < kFwdU; ++u) {
      if (sr < kMoveRows) reinterpret_cast<uint4*>(p.ring + (ring_row0 + sr) * d)[sc] = cur[u];
      step(sr, sc);
    }
  }
}

// Scales of one ring m-tile (128 rows) in the tiled atom layout, copied from
// the row-major scales of the rows' tokens (tile_scales_from_rows): the
// tile's item `part` takes k-tile groups part, part + kMoveItems, ...
__device__ __forceinline__ void move_tile_scales(const GemmParams& p, const uint8_t* sfr, int lane, int cnt,
                                                 int poff_e, int64_t rank_tile0, int64_t ring_tile_row0, int part) {
  int tok[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int64_t rank = rank_tile0 + lane + 32 * j;
    const int a = rank < cnt ? p.row_src[poff_e + rank] : -1;
    tok[j] = a >= 0 ? a / p.k : -1;
  }
  tile_scales_from_rows(sfr, tok, p.d, p.ring_sf + (ring_tile_row0 >> 7) * (p.d >> 7) * 512 + lane * 16, part,
                        kMoveItems);
}

// Mover warp `wid` of this CTA (MV per CTA): items j = blockIdx.x * MV + wid,
// then every gridDim.x * MV, i.e. in increasing (lap-major) order.
template <int BN, int MODE, int MV>
__device__ void ring_mover(const GemmParams& p, int wid, int lane) {
  const int nt = p.N / BN;
  const int total = p.lapbase[p.Lb] * kMoveItems;
  const int stride = gridDim.x * MV;
  for (int j = blockIdx.x * MV + wid; j < total; j += stride) {
    const int pos = j / kMoveItems, part = j - pos * kMoveItems;
    const int4 a = p.ring_info[2 * pos];        // the position's m-tile, decoded by the schedule
    if ((a.y >> 25) & 1) continue;              // shared-expert tile: A2 is read in place
    const int4 b = p.ring_info[2 * pos + 1];
    const int gm = a.x;
    const int gp = b.x;
    if (gp >= 0) {
      // The slot's previous tenant: the same expert's m-tile of lap L - kRingBufs.
      int ok = 1;
      if (lane == 0) ok = wait_counter(p.consumed + gp, nt, p.status, 40) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      (void)ld_acquire_gpu(p.consumed + gp);   // every lane orders its writes after the reads
    }
    const int64_t rank0 = static_cast<int64_t>(b.y) + part * kMoveRows;
    const int64_t ring_row0 = static_cast<int64_t>(a.z) + part * kMoveRows;
    const int cnt = b.z, poff_e = b.w;
    const int src = (lane < kMoveRows && rank0 + lane < cnt) ? p.row_src[poff_e + rank0 + lane] : -1;
    move_rows(p, lane, src, ring_row0);
    // this item's share of the m-tile's scales (all 128 rows, some k-tiles)
    move_tile_scales(p, p.mv_xq_sfr, lane, cnt, poff_e, rank0 - part * kMoveRows, ring_row0 - part * kMoveRows, part);
    publish_move(p.moved + gm, lane);
  }
}

// Stores 32 rows x 128 bytes that a warp holds one row per lane (8 uint4 in
// v) so that each store instruction writes 4 whole 128-byte row segments
// instead of 32 scattered 16-byte pieces: the rows pass through a swizzled
// 4 KB shared tile. dst(r) gives row r's destination (null: skip the row).
template <typename DstOf>
__device__ __forceinline__ void warp_store_rows128(uint8_t* buf, int lane, const uint4* v, DstOf dst) {
#pragma unroll
  for (int i = 0; i < 8; ++i) *reinterpret_cast<uint4*>(buf + lane * 128 + ((i ^ (lane & 7)) << 4)) = v[i];
  __syncwarp();
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int r = 4 * j + (lane >> 3), ch = lane & 7;
    const uint4 val = *reinterpret_cast<const uint4*>(buf + r * 128 + ((ch ^ (r & 7)) << 4));
    uint4* d = dst(r);
    if (d != nullptr) d[ch] = val;
  }
  __syncwarp();
}

// All-laps ring tiles (t.gm >= 0): the accumulator is complete, so every A
// load of the tile landed long ago; one thread reports the tile's ring rows
// consumed, and the movers of the slot's next tenant may overwrite them.
__device__ __forceinline__ void ring_consumed(const GemmParams& p, const TileInfo& t, int q, int lane) {
  if (t.gm >= 0 && q == 0 && lane == 0) {
    fence_proxy_async_global();
    red_release_add(p.consumed + t.gm, 1);
  }
}

// HOLD: accumulator chunks of 32 columns the dh epilogue keeps in registers
// at once (5 at 256 threads per CTA; fewer when more warps share the file).
// kAlpha: push rows scaled by p.alpha (the NVFP4 push mode).
template <int BN, int MODE, int HOLD = 5, bool kAlpha = false>
__device__ __forceinline__ void gemm_epilogue_tile(const GemmParams& p, const TileInfo& t, uint32_t tacc, int q,
                                                   int lane, float* scr, uint8_t* out_smem, const CUtensorMap* tma_o,
                                                   const CUtensorMap* tma_o2, uint64_t* acce) {
  const int row = q * 32 + lane;
  const bool have_acc = t.nk > 0;
  const bool valid = row < t.valid;
  if constexpr (MODE == kSwigluFwd) {
    const int64_t prow = t.prow0 + row;
    const int I = p.I;
    const int i_base = t.n0 / 2;                     // interleaved: BN/2 gate + BN/2 up columns
    // Drain g, u from TMEM (saving them as bf16) and keep h in registers, then
    // hand the accumulator back before the two MX quantisations of h.
    float h[BN / 2];
#pragma unroll
    for (int c = 0; c < BN / 64; ++c) {
      uint32_t rg[32], ru[32];
      tmem_ld32_async(tacc + c * 32, rg);
      tmem_ld32_async(tacc + BN / 2 + c * 32, ru);
      tmem_wait_ld();
      float g[32], u[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        reg_fence(rg[j]);
        reg_fence(ru[j]);
        g[j] = valid ? __uint_as_float(rg[j]) : 0.0f;
        u[j] = valid ? __uint_as_float(ru[j]) : 0.0f;
        // silu(g) u with the fast reciprocal-based divide (about 2 ulp)
        h[c * 32 + j] = __fdividef(g[j], 1.0f + __expf(-g[j])) * u[j];
      }
      // saved g,u: 32-column chunk k of a row holds g then u (128 contiguous bytes),
      // stored 4 rows x 128 bytes per instruction through this warp's scratch tile
      const int64_t chunk = (i_base >> 5) + c;
      uint4 v[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        v[i] = make_uint4(pack_bf16x2(g[8 * i], g[8 * i + 1]), pack_bf16x2(g[8 * i + 2], g[8 * i + 3]),
                          pack_bf16x2(g[8 * i + 4], g[8 * i + 5]), pack_bf16x2(g[8 * i + 6], g[8 * i + 7]));
        v[4 + i] = make_uint4(pack_bf16x2(u[8 * i], u[8 * i + 1]), pack_bf16x2(u[8 * i + 2], u[8 * i + 3]),
                              pack_bf16x2(u[8 * i + 4], u[8 * i + 5]), pack_bf16x2(u[8 * i + 6], u[8 * i + 7]));
      }
      __nv_bfloat16* gu_rows0 = p.gu + (t.prow0 + q * 32) * (2 * I) + chunk * 64;
      warp_store_rows128(reinterpret_cast<uint8_t*>(scr), lane, v, [&](int r) {
        return reinterpret_cast<uint4*>(gu_rows0 + static_cast<int64_t>(r) * (2 * I));
      });
    }
    tc_fence_before();
    mbar_arrive(acce);
    ring_consumed(p, t, q, lane);
#pragma unroll
    for (int c = 0; c < BN / 64; ++c) {
      const int64_t icol = i_base + c * 32;
      emit_rowq(&h[c * 32], p.q_rows + prow * I + icol, p.q_rows_sf + sf_off(prow, icol >> 5, p.q_rows_ktiles));
      emit_tokq(&h[c * 32], scr, lane, p.q_tok, p.q_tok_sf, p.q_tok_pitch, icol, t.prow0 + q * 32);
    }
  } else if constexpr (MODE == kSwigluBwd) {
    // dh (fp32) to the tile's padded rank rows, each routed row times its
    // assignment's gate (the A rows are the token's MX(dy); the gate is a
    // per-row scalar of the down projection's gradient). The SwiGLU backward
    // and the two MX quantisations of dGU run in their own kernel.
    uint8_t* buf = reinterpret_cast<uint8_t*>(scr);
    float* rows0 = static_cast<float*>(p.out) + (t.prow0 + q * 32) * static_cast<int64_t>(p.ldo) + t.n0;
    const float gw = (valid && t.e < p.E) ? p.gate[p.row_src[t.prow0 + row]] : 1.0f;
    // Up to HOLD of the row's 32-column chunks are held in registers: the first
    // ones are stored while the last ones are read, so the accumulator goes
    // back to the MMA thread after only NC - H chunk stores.
    constexpr int NC = BN / 32;
    constexpr int H = NC < HOLD ? NC : HOLD;
    uint32_t r[H][32];
    auto scale = [&](uint32_t* v) {
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        reg_fence(v[j]);
        v[j] = __float_as_uint(__fmul_rn(__uint_as_float(v[j]), gw));
      }
    };
    auto store = [&](const uint32_t* v, int c) {
      uint4 w[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) w[k] = make_uint4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
      warp_store_rows128(buf, lane, w, [&](int rr) {
        return reinterpret_cast<uint4*>(rows0 + static_cast<int64_t>(rr) * p.ldo + c * 32);
      });
    };
    // chunk c lives in slot c % H
#pragma unroll
    for (int c = 0; c < H; ++c) tmem_ld32_async(tacc + c * 32, r[c]);
    tmem_wait_ld();
#pragma unroll
    for (int c = 0; c < H; ++c) scale(r[c]);
#pragma unroll
    for (int c = H; c < NC; ++c) {       // chunk c - H leaves its slot to chunk c
      store(r[c % H], c - H);
      tmem_ld32_async(tacc + c * 32, r[c % H]);
      tmem_wait_ld();
      scale(r[c % H]);
    }
    tc_fence_before();                   // whole accumulator row read: hand TMEM back
    mbar_arrive(acce);
    ring_consumed(p, t, q, lane);
#pragma unroll
    for (int c = NC - H; c < NC; ++c) store(r[c % H], c);
  } else if constexpr (MODE == kPush) {
    const int64_t prow = t.prow0 + row;
    const int a = valid ? p.row_src[prow] : -1;
    uint32_t packed[BN / 2];
    drain_acc_bf16<BN, kAlpha>(tacc, true, packed, acce, p.alpha);
    // Each lane holds one row; rows go to scattered assignments. Per 64-column
    // chunk the warp swaps the tile through shared memory so that each store
    // instruction writes 4 rows x 128 contiguous bytes instead of 32 x 16.
    uint8_t* buf = reinterpret_cast<uint8_t*>(scr);
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out);
#pragma unroll
    for (int c = 0; c < BN / 64; ++c) {
      uint4 v[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int w = (c * 8 + i) * 4;
        v[i] = make_uint4(packed[w], packed[w + 1], packed[w + 2], packed[w + 3]);
      }
      warp_store_rows128(buf, lane, v, [&](int r) {
        const int ar = __shfl_sync(0xffffffffu, a, r);
        return ar >= 0 ? reinterpret_cast<uint4*>(out + static_cast<int64_t>(ar) * p.ldo + t.n0 + c * 64) : nullptr;
      });
    }
  } else if constexpr (MODE == kWgrad) {
    // bf16 tile -> shared staging (boxes of 128 rows x 64 columns, 128-byte
    // swizzle) -> TMA store to dW[e][m0.., n0..]. One thread issues the stores.
    const bool leader = (q == 2 && lane == 0);
    uint32_t packed[BN / 2];
    drain_acc_bf16<BN>(tacc, have_acc, packed, acce);
    if (leader) bulk_wait_read_all();          // the previous tile's stores have read the staging
    named_barrier(1, 128);
#pragma unroll
    for (int i = 0; i < BN / 8; ++i) {         // 16-byte chunk i of the row: box i / 8, chunk i % 8
      uint8_t* box = out_smem + (i >> 3) * (128 * 128) + row * 128;
      *reinterpret_cast<uint4*>(box + (((i & 7) ^ (row & 7)) << 4)) =
          make_uint4(packed[4 * i], packed[4 * i + 1], packed[4 * i + 2], packed[4 * i + 3]);
    }
    fence_proxy_async();
    named_barrier(1, 128);
    if (leader) {
      const bool routed = t.e < p.E;
      const int y = (routed ? t.e : t.e - p.E) * p.M + t.m0;
#pragma unroll
      for (int b = 0; b < BN / 64; ++b) tma_store_2d(routed ? tma_o : tma_o2, t.n0 + 64 * b, y, out_smem + b * 128 * 128);
      bulk_commit();
    }
  } else {   // plain and grouped NVFP4 (fp32 out, M x N) and router logits (fp32 [M][N] for columns < N)
    float* out = static_cast<float*>(p.out);
    const int64_t orow = t.m0 + row;
#pragma unroll 1
    for (int c = 0; c < BN / 32; ++c) {
      float v[32];
      tmem_ld32(tacc + c * 32, v);
      if constexpr (MODE == kPlainNv4 || MODE == kGroupedNv4) {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = __fmul_rn(v[j], p.alpha);
      }
      if (orow < p.M) {
        const int col0 = t.n0 + c * 32;
        if (col0 + 32 <= p.N && (p.ldo % 4) == 0) {
          float4* dst = reinterpret_cast<float4*>(out + orow * p.ldo + col0);
#pragma unroll
          for (int j = 0; j < 8; ++j) dst[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
        } else {
          for (int j = 0; j < 32; ++j)
            if (col0 + j < p.N) out[orow * p.ldo + col0 + j] = v[j];
        }
      }
    }
  }
}

template <int BN, int MODE, int MV = kMoverWarpsDefault>
__global__ void __launch_bounds__(gemm_threads(MODE, MV), 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tma_a, const __grid_constant__ CUtensorMap tma_a2,
                const __grid_constant__ CUtensorMap tma_b, const __grid_constant__ CUtensorMap tma_o,
                const __grid_constant__ CUtensorMap tma_o2, const __grid_constant__ GemmParams p) {
  using Cf = GemmCfg<BN, MODE>;
  constexpr int BM = base_mode(MODE);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* out_smem = smem + Cf::kStages * Cf::kStageBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(out_smem + Cf::kOutBytes);
  uint64_t* empty = full + Cf::kStages;
  uint64_t* accf = empty + Cf::kStages;
  uint64_t* acce = accf + Cf::kNumAcc;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(acce + Cf::kNumAcc);
  float* scratch = reinterpret_cast<float*>(out_smem + Cf::kOutBytes + Cf::kBarBytes);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < Cf::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < Cf::kNumAcc; ++a) {
      mbar_init(&accf[a], 1);
      mbar_init(&acce[a], 128);
    }
    fence_barrier_init();
    fence_proxy_async();
    tma_prefetch(&tma_a);
    tma_prefetch(&tma_b);
    if (BM == kSwigluFwd || BM == kSwigluBwd) tma_prefetch(&tma_a2);
    if (Cf::kTmaOut) {
      tma_prefetch(&tma_o);
      tma_prefetch(&tma_o2);
    }
  }
  if (warp == 1) {
    tmem_alloc(tslot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  const int n_tiles = gemm_num_tiles<BN, MODE>(p);

  if (warp == 0) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x) {
        TileInfo t;
        if (!gemm_decode<BN, MODE>(p, tile, t)) continue;
        if constexpr (ring_mode(MODE)) {
          if (t.gm >= 0) {   // the movers have filled this m-tile's ring slot
            if (!wait_counter(p.moved + t.gm, kMoveItems, p.status, 12)) { ok = false; break; }
            fence_proxy_async_global();
          }
        }
        for (int ks = 0; ks < t.nk; ++ks) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, p.status, 10)) { ok = false; break; }
          uint8_t* sa = smem + stage * Cf::kStageBytes;
          uint8_t* sb = sa + Cf::kABytes;
          mbar_arrive_expect_tx(&full[stage], Cf::kTx);
          const int kt = t.k0 + ks;
          const int kx = kt * Cf::kTmaX;
          tma_load_2d(sa, t.use_a2 ? &tma_a2 : &tma_a, kx, static_cast<int>(t.a_row), &full[stage]);
          tma_load_2d(sb, &tma_b, kx, static_cast<int>(t.b_row), &full[stage]);
          if constexpr (Cf::kNv4) {
            // a stage's 4 atoms of one 128-row tile are contiguous (a_ktiles = atoms per row tile)
            uint8_t* ssfa = sb + Cf::kBBytes;
            bulk_load(ssfa, p.a_sf + ((t.a_row >> 7) * p.a_ktiles + kt * 4) * 512, 2048, &full[stage]);
#pragma unroll
            for (int j = 0; j < BN / 128; ++j)
              bulk_load(ssfa + 2048 + 2048 * j, p.b_sf + (((t.b_row >> 7) + j) * p.b_ktiles + kt * 4) * 512, 2048,
                        &full[stage]);
          } else if constexpr (!Cf::kBf16) {
            uint8_t* ssfa = sb + Cf::kBBytes;
            const uint8_t* asf = (t.use_a2 ? p.a2_sf : p.a_sf) + ((t.a_row >> 7) * p.a_ktiles + kt) * 512;
            bulk_load(ssfa, asf, 512, &full[stage]);
#pragma unroll
            for (int j = 0; j < BN / 128; ++j)
              bulk_load(ssfa + 512 + 512 * j, p.b_sf + (((t.b_row >> 7) + j) * p.b_ktiles + kt) * 512, 512,
                        &full[stage]);
          }
          ++issued;
          if (++stage == Cf::kStages) { stage = 0; phase ^= 1u; }
        }
      }
      // Let every copy this CTA started land before its shared memory is released.
      const int tail = issued < Cf::kStages ? issued : Cf::kStages;
      for (int i = 0; i < tail; ++i) {
        if (--stage < 0) { stage = Cf::kStages - 1; phase ^= 1u; }
        mbar_wait(&full[stage], phase, p.status, 11);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      constexpr uint32_t idesc0 = Cf::kBf16 ? idesc_bf16(128, BN) : (Cf::kNv4 ? idesc_nvf4(128, BN) : idesc_mxf8(128, BN));
      for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x) {
        TileInfo t;
        if (!gemm_decode<BN, MODE>(p, tile, t)) continue;
        if (!mbar_wait(&acce[acc], acc_phase ^ 1u, p.status, 20)) break;
        tc_fence_after();
        const uint32_t dacc = tmem + static_cast<uint32_t>(acc * BN);
        for (int ks = 0; ks < t.nk; ++ks) {
          if (!mbar_wait(&full[stage], phase, p.status, 21)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + stage * Cf::kStageBytes);
          const uint32_t sb = sa + Cf::kABytes;
          if constexpr (Cf::kBf16) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              tc_mma_bf16(dacc, desc_kmajor_sw128(sa + kk * 32), desc_kmajor_sw128(sb + kk * 32), idesc0,
                          (ks | kk) != 0);
          } else if constexpr (Cf::kNv4) {
            // per K = 64 step kk: A's atom kk at columns sfa_t + 4 kk; B's atoms (kk, row tile j)
            // side by side at sfb_t + (BN / 128) 4 kk + 4 j
            const uint32_t sfa_t = tmem + Cf::kSfCol0 + stage * Cf::kSfCols;
            const uint32_t sfb_t = sfa_t + 16;
            const uint32_t ssf = sb + Cf::kBBytes;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              tc_cp_sf(sfa_t + 4 * kk, desc_sf_chunk(ssf + 512 * kk));
#pragma unroll
              for (int j = 0; j < BN / 128; ++j)
                tc_cp_sf(sfb_t + (BN / 128) * 4 * kk + 4 * j, desc_sf_chunk(ssf + 2048 + 2048 * j + 512 * kk));
            }
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              tc_mma_nvf4(dacc, desc_kmajor_sw128(sa + kk * 32), desc_kmajor_sw128(sb + kk * 32), idesc0,
                          sfa_t + 4 * kk, sfb_t + (BN / 128) * 4 * kk, (ks | kk) != 0);
          } else {
            const uint32_t sfa_t = tmem + Cf::kSfCol0 + stage * Cf::kSfCols;
            const uint32_t sfb_t = sfa_t + 4;
            const uint32_t ssf = sb + Cf::kBBytes;
            tc_cp_sf(sfa_t, desc_sf_chunk(ssf));
#pragma unroll
            for (int j = 0; j < BN / 128; ++j) tc_cp_sf(sfb_t + 4 * j, desc_sf_chunk(ssf + 512 + 512 * j));
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              tc_mma_mxf8(dacc, desc_kmajor_sw128(sa + kk * 32), desc_kmajor_sw128(sb + kk * 32),
                          idesc_mxf8_sf(idesc0, kk, kk), sfa_t, sfb_t, (ks | kk) != 0);
          }
          tc_commit(&empty[stage]);
          if (++stage == Cf::kStages) { stage = 0; phase ^= 1u; }
        }
        // (ring modes: the epilogue reports the tile's ring rows consumed once
        // the accumulator is complete, so this thread never waits on a proxy
        // fence behind its queued MMAs)
        tc_commit(&accf[acc]);
        if (++acc == Cf::kNumAcc) { acc = 0; acc_phase ^= 1u; }
      }
    }
  } else if (warp < 6) {
    const int q = warp & 3;
    float* scr = scratch + (warp - 2) * 32 * 33;
    uint32_t acc_phase = 0;
    int acc = 0;
    for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x) {
      TileInfo t;
      if (!gemm_decode<BN, MODE>(p, tile, t)) continue;
      if (!mbar_wait(&accf[acc], acc_phase, p.status, 30)) break;
      tc_fence_after();
      gemm_epilogue_tile<BN, BM, (gemm_threads(MODE, MV) > 256 ? 2 : 5), MODE == kPushNv4>(
          p, t, tmem + static_cast<uint32_t>(acc * BN) + (static_cast<uint32_t>(q * 32) << 16),
                                   q, lane, scr, out_smem, &tma_o, &tma_o2, &acce[acc]);
      if constexpr (BM != kPush && BM != kWgrad && BM != kSwigluFwd && BM != kSwigluBwd) {   // others release TMEM inside
        tc_fence_before();
        mbar_arrive(&acce[acc]);
      }
      if (++acc == Cf::kNumAcc) { acc = 0; acc_phase ^= 1u; }
    }
    if (Cf::kTmaOut && q == 2 && lane == 0) bulk_wait_all();
  } else {
    if constexpr (ring_mode(MODE)) ring_mover<BN, MODE, MV>(p, warp - 6, lane);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace moe
