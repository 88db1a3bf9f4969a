// Grouped MXFP8 GEMM on CTA pairs: tcgen05 .cta_group::2 with 256-row tiles.
//
//   D[256 x 128] (TMEM of two SMs, fp32) = sum_k A[256 x k] . B[128 x k]^T
//
// A cluster of two CTAs on two SMs computes one 256 x 128 tile. CTA r of the
// pair loads A rows [128 r, 128 r + 128) and B rows [64 r, 64 r + 64) of the
// tile into its own shared memory (at the same offsets in both CTAs), plus
// the E8M0 scale atoms of its A rows and of all 128 B rows. The even CTA
// issues every MMA (M = 256, N = 128, K = 32); each MMA reads A and B from
// both CTAs' shared memory and writes the 256 x 128 accumulator into the two
// CTAs' TMEM, rows 128 r.. of CTA r. Per SM this is a 128 x 128 x 32 MMA fed
// by 128 + 64 operand rows, the operand bytes per FLOP of a 128 x 256 tile
// on one SM, while each SM keeps TWO 128-column accumulators in TMEM: the
// epilogue of one tile overlaps the MMAs of the next instead of holding the
// only accumulator.
//
// Roles (192 threads per CTA): warp 0 = TMA producer (both CTAs; completions
// counted on the even CTA's barriers), warp 1 = MMA issuer (even CTA) and
// TMEM owner (both), warps 2-5 = epilogue (both CTAs, each its own rows).
// Synchronisation:
//   full[s]   (even CTA) stage s landed in both CTAs (TMA transaction bytes);
//   empty[s]  (both)     stage s consumed: MMA commit multicast to the pair;
//   accf[a]   (both)     accumulator a complete: MMA commit multicast;
//   acce[a]   (even CTA) accumulator a drained by the 8 epilogue warps of the
//                        pair (one arrival per warp, 4 of them remote).
// Barriers completed by hardware (TMA transaction bytes, MMA commits) are
// waited on at CTA scope, as in a one-CTA pipeline; only the drained-
// accumulator barrier, which the odd CTA's threads arrive on, is waited on
// with cluster-scope acquire (once per tile). Every wait is bounded
// (kWaitLimitNs) and reports (kErrTimeout, site).
#pragma once
#include <cuda_bf16.h>

#include "gemm.cuh"

namespace moe {

constexpr int kPairM = 256;            // output rows of a pair tile

// Tile shape of a pair kernel instance: BN output columns per pair tile (each
// CTA loads BN / 2 rows of B), KS 128-element K atoms per pipeline stage.
template <int MODE, int BN, int KS>
struct PairCfg {
  static constexpr bool kTmaOut = MODE == kWgrad;
  static constexpr int kHalfN = BN / 2;
  static constexpr int kAAtom = 128 * 128;                    // A bytes per K atom
  static constexpr int kBAtom = kHalfN * 128;                 // B bytes per K atom (this CTA's half)
  static constexpr int kSfbAtoms = BN / 128;                  // B scale atoms per K atom
  static constexpr int kABytes = KS * kAAtom;
  static constexpr int kBBytes = KS * kBAtom;
  static constexpr int kSfaBytes = KS * 512;
  static constexpr int kSfbBytes = KS * kSfbAtoms * 512;
  static constexpr int kAtomTx = kAAtom + kBAtom + 512 + kSfbAtoms * 512;  // per CTA per K atom
  static constexpr int kTx = KS * kAtomTx;                                 // per CTA per full stage
  static constexpr int kStageBytes = ((kTx + 1023) / 1024) * 1024;
  static constexpr int kOutTile = 128 * BN * 2;               // bf16 staging tile of one CTA
  static constexpr int kOutBufs = kTmaOut ? (BN <= 128 ? 2 : 1) : 0;
  static constexpr int kOutBytes = kOutBufs * kOutTile;
  static constexpr int kBarBytes = 256;
  static constexpr int kSfCols = KS * (4 + 4 * kSfbAtoms);    // TMEM scale columns per stage
  static constexpr int kStagesSmem = (232448 - 1024 - kOutBytes - kBarBytes) / kStageBytes;
  static constexpr int kStages = kStagesSmem < 8 ? kStagesSmem : 8;
  // Two accumulators when they fit beside the scale columns in TMEM.
  static constexpr int kNumAcc = (2 * BN + kStages * kSfCols <= 512) ? 2 : 1;
  static constexpr int kSfCol0 = kNumAcc * BN;
  static constexpr int kSmem = 1024 + kStages * kStageBytes + kOutBytes + kBarBytes;
  static_assert(kStages >= 2, "pipeline depth");
  static_assert(kSmem <= 232448, "shared memory budget");
  static_assert(kSfCol0 + kStages * kSfCols <= 512, "TMEM budget");
};

struct PairTile {
  int e;
  int64_t a_row;   // this CTA's first A row
  int64_t b_row;   // this CTA's first B row (its half of the tile's columns)
  int64_t sfb_rt;  // first 128-row tile of B holding the tile's columns
  int k0, nk;      // first K atom, number of K atoms
  int m0;          // this CTA's first output row (per expert)
  int n0;          // first output column
};

// Tile list position of pair tile `tile` (the cluster's share of the
// two-ended weight-gradient order, or row-major for the plain GEMM).
template <int MODE, int BN>
__device__ __forceinline__ bool pair_decode(const GemmParams& p, int tile, uint32_t rank, PairTile& t) {
  const int nt = p.N / BN, mp = p.M / kPairM;
  const int per = nt * mp;
  int q = tile;
  int e = 0;
  if constexpr (MODE == kWgrad) {
    // Two-ended schedule over clusters: in each round half of the clusters
    // take the next tile from the front of the list (experts with the most
    // tokens: long K) and half from the back (few or no tokens: bound by
    // writing their gradient tile), alternating ends from round to round.
    const int N = p.static_tiles;
    const int g = static_cast<int>(pair::num_clusters());
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
    e = p.order[q / per];
    q -= (q / per) * per;
  }
  const int mi = q / nt, n = q - (q / nt) * nt;
  t.e = e;
  t.m0 = mi * kPairM + static_cast<int>(rank) * 128;
  t.n0 = n * BN;
  t.a_row = t.m0;
  t.b_row = static_cast<int64_t>(n) * BN + static_cast<int64_t>(rank) * (BN / 2);
  t.sfb_rt = static_cast<int64_t>(n) * (BN / 128);
  if constexpr (MODE == kWgrad) {
    t.k0 = p.poff[e] / 128;
    t.nk = (p.poff[e + 1] - p.poff[e]) / 128;
  } else {
    t.k0 = 0;
    t.nk = p.K / 128;
  }
  return true;
}

template <int MODE>
__device__ __forceinline__ int pair_num_tiles(const GemmParams& p) {
  if constexpr (MODE == kWgrad) {
    const int N = p.static_tiles;
    const int g = static_cast<int>(pair::num_clusters());
    if (g < 2 || (g & 1)) return N;
    const int heavy = (N + 1) / 2;
    return ((heavy + g / 2 - 1) / (g / 2)) * g;
  } else {
    return p.static_tiles;
  }
}

template <int MODE, int BN, int KS>
__global__ void __launch_bounds__(192, 1)
    gemm_pair_kernel(const __grid_constant__ CUtensorMap tma_a, const __grid_constant__ CUtensorMap tma_b,
                     const __grid_constant__ CUtensorMap tma_sfa, const __grid_constant__ CUtensorMap tma_sfb,
                     const __grid_constant__ CUtensorMap tma_o, const __grid_constant__ CUtensorMap tma_o2,
                     const __grid_constant__ GemmParams p) {
  using Cf = PairCfg<MODE, BN, KS>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* out_smem = smem + Cf::kStages * Cf::kStageBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(out_smem + Cf::kOutBytes);
  uint64_t* empty = full + Cf::kStages;
  uint64_t* accf = empty + Cf::kStages;
  uint64_t* acce = accf + Cf::kNumAcc;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(acce + Cf::kNumAcc);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = pair::cta_rank();
  const int cid = static_cast<int>(pair::cluster_id());
  const int ncl = static_cast<int>(pair::num_clusters());

  if (threadIdx.x == 0) {
    for (int s = 0; s < Cf::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < Cf::kNumAcc; ++a) {
      mbar_init(&accf[a], 1);
      mbar_init(&acce[a], 8);
    }
    fence_barrier_init();
    tma_prefetch(&tma_a);
    tma_prefetch(&tma_b);
    tma_prefetch(&tma_sfa);
    tma_prefetch(&tma_sfb);
    if (Cf::kTmaOut) {
      tma_prefetch(&tma_o);
      tma_prefetch(&tma_o2);
    }
  }
  if (warp == 1) {
    pair::tmem_alloc(tslot, 512);
    pair::tmem_relinquish();
  }
  // Both CTAs' barriers are initialised (and TMEM allocated) before either
  // CTA signals the other.
  tc_fence_before();
  __syncwarp();
  pair::cluster_sync();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  const int n_tiles = pair_num_tiles<MODE>(p);

  if (warp == 0) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;
      bool ok = true;
      for (int tile = cid; tile < n_tiles && ok; tile += ncl) {
        PairTile t;
        if (!pair_decode<MODE, BN>(p, tile, rank, t)) continue;
        for (int ks = 0; ks < t.nk; ks += KS) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, p.status, 110)) { ok = false; break; }
          const uint32_t bar = pair::map_rank(smem_u32(&full[stage]), 0);
          // atoms of this stage: KS, or fewer in the tile's last stage
          const int nv = t.nk - ks < KS ? t.nk - ks : KS;
          if (rank == 0) mbar_arrive_expect_tx(&full[stage], 2 * nv * Cf::kAtomTx);
          uint8_t* sa = smem + stage * Cf::kStageBytes;
          uint8_t* sb = sa + Cf::kABytes;
          uint8_t* ssfa = sb + Cf::kBBytes;
          uint8_t* ssfb = ssfa + Cf::kSfaBytes;
#pragma unroll
          for (int j = 0; j < KS; ++j) {   // K atom kt of the stage
            if (j >= nv) break;
            const int kt = t.k0 + ks + j;
            pair::tma_load_2d(sa + j * Cf::kAAtom, &tma_a, kt * 128, static_cast<int>(t.a_row), bar);
            pair::tma_load_2d(sb + j * Cf::kBAtom, &tma_b, kt * 128, static_cast<int>(t.b_row), bar);
            pair::tma_load_2d(ssfa + j * 512, &tma_sfa, 0, static_cast<int>((t.a_row >> 7) * p.a_ktiles + kt), bar);
#pragma unroll
            for (int b = 0; b < Cf::kSfbAtoms; ++b)
              pair::tma_load_2d(ssfb + (j * Cf::kSfbAtoms + b) * 512, &tma_sfb, 0,
                                static_cast<int>((t.sfb_rt + b) * p.b_ktiles + kt), bar);
          }
          ++issued;
          if (++stage == Cf::kStages) { stage = 0; phase ^= 1u; }
        }
      }
      // Every copy into either CTA has landed before the pair may exit (the
      // even CTA's full barriers count both CTAs' bytes; the final cluster
      // barrier holds the odd CTA until then).
      if (rank == 0) {
        const int tail = issued < Cf::kStages ? issued : Cf::kStages;
        for (int i = 0; i < tail; ++i) {
          if (--stage < 0) { stage = Cf::kStages - 1; phase ^= 1u; }
          mbar_wait(&full[stage], phase, p.status, 111);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      constexpr uint32_t idesc0 = idesc_mxf8(kPairM, BN);
      for (int tile = cid; tile < n_tiles && ok; tile += ncl) {
        PairTile t;
        if (!pair_decode<MODE, BN>(p, tile, rank, t)) continue;
        if (!pair::mbar_wait_cluster(&acce[acc], acc_phase ^ 1u, p.status, 120)) break;
        tc_fence_after();
        const uint32_t dacc = tmem + static_cast<uint32_t>(acc * BN);
        for (int ks = 0; ks < t.nk; ks += KS) {
          if (!mbar_wait(&full[stage], phase, p.status, 121)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + stage * Cf::kStageBytes);
          const uint32_t sb = sa + Cf::kABytes;
          const uint32_t ssfa = sb + Cf::kBBytes;
          const uint32_t ssfb = ssfa + Cf::kSfaBytes;
          const int nv = t.nk - ks < KS ? t.nk - ks : KS;
#pragma unroll
          for (int j = 0; j < KS; ++j) {
            if (j >= nv) break;
            const uint32_t sfa_t = tmem + Cf::kSfCol0 + stage * Cf::kSfCols + j * (4 + 4 * Cf::kSfbAtoms);
            const uint32_t sfb_t = sfa_t + 4;
            pair::tc_cp_sf(sfa_t, desc_sf_chunk(ssfa + j * 512));
#pragma unroll
            for (int b = 0; b < Cf::kSfbAtoms; ++b)
              pair::tc_cp_sf(sfb_t + 4 * b, desc_sf_chunk(ssfb + (j * Cf::kSfbAtoms + b) * 512));
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              pair::tc_mma_mxf8(dacc, desc_kmajor_sw128(sa + j * Cf::kAAtom + kk * 32),
                                desc_kmajor_sw128(sb + j * Cf::kBAtom + kk * 32), idesc_mxf8_sf(idesc0, kk, kk),
                                sfa_t, sfb_t, (ks | j | kk) != 0);
          }
          pair::tc_commit_mc(&empty[stage], 0x3);
          if (++stage == Cf::kStages) { stage = 0; phase ^= 1u; }
        }
        pair::tc_commit_mc(&accf[acc], 0x3);
        if (++acc == Cf::kNumAcc) { acc = 0; acc_phase ^= 1u; }
      }
    }
  } else {
    const int q = warp & 3;
    const int row = q * 32 + lane;
    const bool leader = (q == 2 && lane == 0);
    // drained accumulators are reported on the even CTA's acce barriers
    const uint32_t acce_cl = pair::map_rank(smem_u32(acce), 0);
    uint32_t acc_phase = 0;
    int acc = 0, done = 0;
    for (int tile = cid; tile < n_tiles; tile += ncl) {
      PairTile t;
      if (!pair_decode<MODE, BN>(p, tile, rank, t)) continue;
      if (!mbar_wait(&accf[acc], acc_phase, p.status, 130)) break;
      tc_fence_after();
      const uint32_t tacc = tmem + static_cast<uint32_t>(acc * BN) + (static_cast<uint32_t>(q * 32) << 16);
      if constexpr (MODE == kWgrad) {
        // The whole accumulator row goes to registers (packed bf16) before the
        // accumulator is handed back, so the MMAs of the next tile can start.
        uint32_t packed[BN / 2];
        if (t.nk > 0) {
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
        __syncwarp();
        if (lane == 0) pair::mbar_arrive_cluster(acce_cl + acc * 8);
        // bf16 tile -> staging buffer -> TMA store. The store that last used
        // this buffer (kOutBufs tiles back) must have read it.
        uint8_t* st = out_smem + (Cf::kOutBufs > 1 ? (done & 1) : 0) * Cf::kOutTile;
        if (leader) {
          if constexpr (Cf::kOutBufs > 1) asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
          else bulk_wait_read_all();
        }
        named_barrier(1, 128);
#pragma unroll
        for (int i = 0; i < BN / 8; ++i) {   // 16-byte chunk i of the row: box i / 8, chunk i % 8
          uint8_t* box = st + (i >> 3) * (128 * 128) + row * 128;
          *reinterpret_cast<uint4*>(box + (((i & 7) ^ (row & 7)) << 4)) =
              make_uint4(packed[4 * i], packed[4 * i + 1], packed[4 * i + 2], packed[4 * i + 3]);
        }
        fence_proxy_async();
        named_barrier(1, 128);
        if (leader) {
          const bool routed = t.e < p.E;
          const int y = (routed ? t.e : t.e - p.E) * p.M + t.m0;
#pragma unroll
          for (int b = 0; b < BN / 64; ++b)
            tma_store_2d(routed ? &tma_o : &tma_o2, t.n0 + 64 * b, y, st + b * 128 * 128);
          bulk_commit();
        }
        ++done;
      } else {   // plain: fp32 [M][N]
        float* out = static_cast<float*>(p.out);
        const int64_t orow = t.m0 + row;
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          float v[32];
          tmem_ld32(tacc + c * 32, v);
          float4* dst = reinterpret_cast<float4*>(out + orow * p.ldo + t.n0 + c * 32);
#pragma unroll
          for (int j = 0; j < 8; ++j) dst[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) pair::mbar_arrive_cluster(acce_cl + acc * 8);
      }
      if (++acc == Cf::kNumAcc) { acc = 0; acc_phase ^= 1u; }
    }
    if (Cf::kTmaOut && leader) bulk_wait_all();
  }
  // Neither CTA leaves (or frees TMEM) while the other may still use its
  // shared memory, its TMEM or its barriers.
  tc_fence_before();
  __syncwarp();
  pair::cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    pair::tmem_dealloc(tmem, 512);
  }
}

}  // namespace moe
