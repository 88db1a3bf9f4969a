// Host side of the tcgen05 grouped GEMM: tensor maps, grid sizing, dispatch.
#include <cudaTypedefs.h>

#include <atomic>
#include <mutex>

#include "gemm.cuh"
#include "prof.h"

namespace moe {

namespace {
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;
std::atomic<int> g_fail_tmaps{0};   // injected encode failures still to hand out

// Takes one injected failure, if any is pending.
bool injected_failure() {
  int n = g_fail_tmaps.load(std::memory_order_relaxed);
  while (n > 0)
    if (g_fail_tmaps.compare_exchange_weak(n, n - 1, std::memory_order_relaxed)) return true;
  return false;
}
}  // namespace

bool get_encode() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode != nullptr;
}

// 2-D K-major operand [rows][cols] (elements of `esize` bytes), box 128 bytes x box_rows.
bool make_tmap(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int box_rows, bool bf16) {
  if (injected_failure()) return false;
  const int esize = bf16 ? 2 : 1;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols * esize)};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(128 / esize), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  const CUresult r = g_encode(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
                              const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 2-D bf16 output [rows][cols] written by TMA stores, box 64 columns x 128 rows, 128-byte swizzle.
bool make_tmap_out(CUtensorMap* m, void* base, int64_t rows, int64_t cols) {
  if (injected_failure()) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols * 2)};
  cuuint32_t box[2] = {64, 128};
  cuuint32_t estr[2] = {1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Scale atoms of a tiled-scale array as a 2-D map of uint32 [atoms][128]: one
// box = one 512-byte atom (128 rows x 4 blocks), selected by its row coordinate.
bool make_tmap_sf(CUtensorMap* m, const void* base, int64_t atoms) {
  if (injected_failure()) return false;
  cuuint64_t dims[2] = {128, static_cast<cuuint64_t>(atoms)};
  cuuint64_t strides[1] = {512};
  cuuint32_t box[2] = {128, 1};
  cuuint32_t estr[2] = {1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {

// Per device: 0 = not yet set up, 1 = ready, 2 = set-up failed.
struct DevOnce {
  std::mutex mu;
  int state[kMaxDev] = {};
  int per_sm[kMaxDev] = {};
};

template <int BN, int MODE, int MV = kMoverWarpsDefault>
int run(const char* name, const CUtensorMap& ta, const CUtensorMap& ta2, const CUtensorMap& tb, const CUtensorMap& to,
        const CUtensorMap& to2, const GemmParams& p, int grid, cudaStream_t s) {
  using Cf = GemmCfg<BN, MODE>;
  // The shared-memory opt-in (and, for cooperative launches, the resident
  // limit) belongs to the current device: set up once per device.
  static DevOnce once;
  const int dev = current_device();
  if (dev < 0) return MOE_ERR_CUDA;
  int per_sm = 0;
  {
    std::lock_guard<std::mutex> lk(once.mu);
    if (once.state[dev] == 0) {
      bool ok = cudaFuncSetAttribute(gemm_kernel<BN, MODE, MV>, cudaFuncAttributeMaxDynamicSharedMemorySize, Cf::kSmem) ==
                cudaSuccess;
      if (ok && ring_mode(MODE))
        ok = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&once.per_sm[dev], gemm_kernel<BN, MODE, MV>,
                                                           gemm_threads(MODE, MV), Cf::kSmem) == cudaSuccess &&
             once.per_sm[dev] >= 1;
      once.state[dev] = ok ? 1 : 2;
    }
    if (once.state[dev] != 1) return MOE_ERR_CUDA;
    per_sm = once.per_sm[dev];
  }
  if (grid <= 0) return MOE_OK;
  cudaLaunchConfig_t lc = {};
  cudaLaunchAttribute attr[1];
  if constexpr (ring_mode(MODE)) {
    // CTAs wait on one another's counters: all of them must be resident, so
    // the launch is cooperative and no larger than the co-resident limit.
    if (grid > per_sm * num_sms()) grid = per_sm * num_sms();
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    lc.attrs = attr;
    lc.numAttrs = 1;
  }
  lc.gridDim = dim3(static_cast<unsigned>(grid));
  lc.blockDim = dim3(gemm_threads(MODE, MV));
  lc.dynamicSmemBytes = Cf::kSmem;
  lc.stream = s;
  Prof prof(name, s);
  const cudaError_t e = cudaLaunchKernelEx(&lc, gemm_kernel<BN, MODE, MV>, ta, ta2, tb, to, to2, p);
  note(e);
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace

int num_sms() {
  static std::atomic<int> cache[kMaxDev];
  const int dev = current_device();
  if (dev < 0) return 1;
  int n = cache[dev].load(std::memory_order_relaxed);
  if (n <= 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 1;
    cache[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

// Dispatch one grouped GEMM. Returns an MOE_* code.
int gemm_dispatch(const char* name, int mode, const Dims& m, int lap, int N, int K, int M, const GemmOperands& op,
                  const GemmEpilogue& ep, const int* counts, const int* poff, const int* lap_tiles,
                  const int* row_src, int* status, cudaStream_t s, int bn_hint, const int* order,
                  const RingMovers* mv, const void* tile_info) {
  if (!get_encode()) return MOE_ERR_CUDA;
  const bool bf16 = mode == kRouterMode;
  int BN;
  if (ring_mode(mode) && mv == nullptr) return MOE_ERR_INVALID_ARG;
  if (base_mode(mode) == kSwigluFwd) BN = kGemm1BN;
  else if (mode == kRouterMode) BN = N <= 32 ? 32 : (N % 256 == 0 ? 256 : 128);
  else if ((bn_hint == 128 || bn_hint == 256) && N % bn_hint == 0) BN = bn_hint;
  else BN = (N % 256 == 0) ? 256 : 128;
  if (!bf16 && N % BN) return MOE_ERR_INVALID_ARG;

  CUtensorMap ta, ta2, tb;
  if (!make_tmap(&ta, op.a, op.a_rows, op.a_cols, 128, bf16)) return MOE_ERR_CUDA;
  if (op.a2 != nullptr) {
    if (!make_tmap(&ta2, op.a2, op.a2_rows, op.a_cols, 128, bf16)) return MOE_ERR_CUDA;
  } else {
    ta2 = ta;
  }
  if (!make_tmap(&tb, op.b, op.b_rows, op.b_cols, BN, bf16)) return MOE_ERR_CUDA;
  CUtensorMap to = tb, to2 = tb;
  if (mode == kWgrad) {
    if (!make_tmap_out(&to, ep.out, static_cast<int64_t>(m.E) * M, N)) return MOE_ERR_CUDA;
    if (m.S > 0 && ep.out2 != nullptr) {
      if (!make_tmap_out(&to2, ep.out2, static_cast<int64_t>(m.S) * M, N)) return MOE_ERR_CUDA;
    } else {
      to2 = to;
    }
  }

  GemmParams p{};
  p.N = N;
  p.K = K;
  p.a_ktiles = op.a_cols / 128;
  p.b_ktiles = op.b_cols / 128;
  p.a_sf = op.a_sf;
  p.a2_sf = op.a2_sf;
  p.b_sf = op.b_sf;
  p.counts = counts;
  p.poff = poff;
  p.lap_tiles = lap_tiles;
  p.row_src = row_src;
  p.order = order;
  p.E = m.E;
  p.Ep = m.Ep;
  p.C = m.C;
  p.lap = lap;
  p.T = m.T;
  p.k = m.k;
  p.M = M;
  p.out = ep.out;
  p.out2 = ep.out2;
  p.ldo = ep.ldo;
  p.alpha = ep.alpha;
  if (mode == kPlainNv4 || mode == kGroupedNv4 || mode == kPushNv4)
    p.a_ktiles = p.b_ktiles = K / 64;   // scale atoms (64 elements) per 128-row tile
  p.q_rows = ep.q_rows;
  p.q_rows_sf = ep.q_rows_sf;
  p.q_rows_ktiles = ep.q_rows_ktiles;
  p.q_tok = ep.q_tok;
  p.q_tok_sf = ep.q_tok_sf;
  p.q_tok_pitch = ep.q_tok_pitch;
  p.gu = static_cast<__nv_bfloat16*>(ep.gu);
  p.gate = ep.gate;
  p.I = m.I;
  p.status = status;
  // decode tables written by the schedule (one load per tile instead of searches)
  if (mode == kPush || mode == kGroupedNv4 || mode == kPushNv4) p.push_info = static_cast<const int*>(tile_info);
  if (mode == kWgrad) p.wg_info = static_cast<const int4*>(tile_info);
  if (mv != nullptr) {
    p.lapbase = mv->lapbase;
    p.ring_info = mv->ring_info;
    p.Lb = m.Lb;
    p.d = m.d;
    p.moved = mv->moved;
    p.consumed = mv->consumed;
    p.mv_xq = mv->xq;
    p.mv_xq_sf = mv->xq_sf;
    p.mv_xq_sfr = mv->xq_sfr;
    p.ring = mv->ring;
    p.ring_sf = mv->ring_sf;
  }

  const int nt = (N + BN - 1) / BN;
  int64_t upper;
  if (ring_mode(mode)) {
    upper = lap_mtiles_max(m) * nt;
  } else if (mode == kSwigluFwd || mode == kSwigluBwd) {
    upper = (static_cast<int64_t>(m.E) * (m.C / 128) + (lap == 0 ? m.S * (m.Tpad / 128) : 0)) * nt;
  } else if (mode == kPush || mode == kGroupedNv4 || mode == kPushNv4) {
    upper = (m.Rmax / 128) * nt;
  } else if (mode == kWgrad) {
    upper = static_cast<int64_t>(m.Ep) * (M / 128) * nt;
    p.static_tiles = static_cast<int>(upper);
  } else {
    upper = ceil_div(M, 128) * nt;
    p.static_tiles = static_cast<int>(upper);
  }
  const int grid = static_cast<int>(upper < num_sms() ? upper : num_sms());

  switch (mode) {
    case kSwigluFwd:
      if (BN == 128) return run<128, kSwigluFwd>(name, ta, ta2, tb, to, to2, p, grid, s);
      return run<256, kSwigluFwd>(name, ta, ta2, tb, to, to2, p, grid, s);
    case kSwigluFwdRing:
      return m.MV == 1 ? run<kGemm1BN, kSwigluFwdRing, 1>(name, ta, ta2, tb, to, to2, p, grid, s)
                       : run<kGemm1BN, kSwigluFwdRing, kMoverWarpsGemm1Max>(name, ta, ta2, tb, to, to2, p, grid, s);
    case kSwigluBwdRing:
      if (BN == 256) {
        return m.MV == 1   ? run<256, kSwigluBwdRing, 1>(name, ta, ta2, tb, to, to2, p, grid, s)
               : m.MV == 4 ? run<256, kSwigluBwdRing, 4>(name, ta, ta2, tb, to, to2, p, grid, s)
                           : run<256, kSwigluBwdRing, 2>(name, ta, ta2, tb, to, to2, p, grid, s);
      }
      return m.MV == 1   ? run<128, kSwigluBwdRing, 1>(name, ta, ta2, tb, to, to2, p, grid, s)
             : m.MV == 4 ? run<128, kSwigluBwdRing, 4>(name, ta, ta2, tb, to, to2, p, grid, s)
                         : run<128, kSwigluBwdRing, 2>(name, ta, ta2, tb, to, to2, p, grid, s);
    case kSwigluBwd:
      return BN == 256 ? run<256, kSwigluBwd>(name, ta, ta2, tb, to, to2, p, grid, s) : run<128, kSwigluBwd>(name, ta, ta2, tb, to, to2, p, grid, s);
    case kPush:
      return BN == 256 ? run<256, kPush>(name, ta, ta2, tb, to, to2, p, grid, s) : run<128, kPush>(name, ta, ta2, tb, to, to2, p, grid, s);
    case kWgrad:
      return BN == 256 ? run<256, kWgrad>(name, ta, ta2, tb, to, to2, p, grid, s) : run<128, kWgrad>(name, ta, ta2, tb, to, to2, p, grid, s);
    case kPlain:
      return BN == 256 ? run<256, kPlain>(name, ta, ta2, tb, to, to2, p, grid, s) : run<128, kPlain>(name, ta, ta2, tb, to, to2, p, grid, s);
    case kPlainNv4:
      return BN == 256 ? run<256, kPlainNv4>(name, ta, ta2, tb, to, to2, p, grid, s) : run<128, kPlainNv4>(name, ta, ta2, tb, to, to2, p, grid, s);
    case kGroupedNv4:
      return BN == 256 ? run<256, kGroupedNv4>(name, ta, ta2, tb, to, to2, p, grid, s)
                       : run<128, kGroupedNv4>(name, ta, ta2, tb, to, to2, p, grid, s);
    case kPushNv4:
      return BN == 256 ? run<256, kPushNv4>(name, ta, ta2, tb, to, to2, p, grid, s)
                       : run<128, kPushNv4>(name, ta, ta2, tb, to, to2, p, grid, s);
    case kRouterMode:
      if (BN == 32) return run<32, kRouterMode>(name, ta, ta2, tb, to, to2, p, grid, s);
      return BN == 256 ? run<256, kRouterMode>(name, ta, ta2, tb, to, to2, p, grid, s) : run<128, kRouterMode>(name, ta, ta2, tb, to, to2, p, grid, s);
    default: return MOE_ERR_INVALID_ARG;
  }
}

}  // namespace moe

extern "C" int moe_debug_fail_tensor_maps(int count) {
  moe::g_fail_tmaps.store(count > 0 ? count : 0, std::memory_order_relaxed);
  return MOE_OK;
}

extern "C" int moe_gemm_mxfp8(int M, int N, int K, const void* a, const void* a_sf, const void* b, const void* b_sf,
                              float* c, moe_stream_t stream) {
  if (M <= 0 || N <= 0 || K <= 0 || M % 128 || N % 128 || K % 128 || !a || !a_sf || !b || !b_sf || !c)
    return MOE_ERR_INVALID_ARG;
  moe::Dims m{};
  moe::GemmOperands op{};
  op.a = static_cast<const uint8_t*>(a);
  op.a_rows = M;
  op.a_cols = K;
  op.a_sf = static_cast<const uint8_t*>(a_sf);
  op.b = static_cast<const uint8_t*>(b);
  op.b_rows = N;
  op.b_cols = K;
  op.b_sf = static_cast<const uint8_t*>(b_sf);
  moe::GemmEpilogue ep{};
  ep.out = c;
  ep.ldo = N;
  return moe::gemm_dispatch("gemm_plain", moe::kPlain, m, 0, N, K, M, op, ep, nullptr, nullptr, nullptr, nullptr, nullptr,
                            static_cast<cudaStream_t>(stream));
}
