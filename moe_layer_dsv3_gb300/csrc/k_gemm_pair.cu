// Host side of the CTA-pair grouped GEMM (gemm_pair.cuh): tensor maps,
// cluster launch, grid sizing.
#include <mutex>

#include "gemm_pair.cuh"
#include "prof.h"

namespace moe {

// Pair tiles are 256 x 256 when N allows, else 256 x 128; two 128-element K
// atoms per pipeline stage (the fastest of 128/256 wide x 1/2 atoms measured
// on a long-K product).
constexpr int kPairKS = 2;
inline int pair_bn(int N) { return N % 256 == 0 ? 256 : 128; }

namespace {

struct PairOnce {
  std::mutex mu;
  int state[kMaxDev] = {};        // 0 = not yet set up, 1 = ready, 2 = set-up failed
  int clusters[kMaxDev] = {};     // co-resident clusters of two CTAs
};

template <int MODE, int BN, int KS>
int run_pair(const char* name, const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tsa,
             const CUtensorMap& tsb, const CUtensorMap& to, const CUtensorMap& to2, const GemmParams& p, int tiles,
             cudaStream_t s) {
  using Cf = PairCfg<MODE, BN, KS>;
  static PairOnce once;
  const int dev = current_device();
  if (dev < 0) return MOE_ERR_CUDA;
  cudaLaunchConfig_t lc = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  lc.attrs = attr;
  lc.numAttrs = 1;
  lc.blockDim = dim3(192);
  lc.dynamicSmemBytes = Cf::kSmem;
  lc.stream = s;
  int clusters = 0;
  {
    std::lock_guard<std::mutex> lk(once.mu);
    if (once.state[dev] == 0) {
      bool ok = cudaFuncSetAttribute(gemm_pair_kernel<MODE, BN, KS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     Cf::kSmem) == cudaSuccess;
      if (ok) {
        cudaLaunchConfig_t q = lc;
        q.gridDim = dim3(static_cast<unsigned>(2 * num_sms()));
        ok = cudaOccupancyMaxActiveClusters(&once.clusters[dev], gemm_pair_kernel<MODE, BN, KS>, &q) == cudaSuccess &&
             once.clusters[dev] >= 1;
      }
      once.state[dev] = ok ? 1 : 2;
    }
    if (once.state[dev] != 1) return MOE_ERR_CUDA;
    clusters = once.clusters[dev];
  }
  if (tiles <= 0) return MOE_OK;
  if (clusters > 1 && (clusters & 1)) --clusters;   // the two-ended order pairs clusters up
  if (clusters > tiles) clusters = tiles;
  lc.gridDim = dim3(static_cast<unsigned>(2 * clusters));
  Prof prof(name, s);
  const cudaError_t e = cudaLaunchKernelEx(&lc, gemm_pair_kernel<MODE, BN, KS>, ta, tb, tsa, tsb, to, to2, p);
  note(e);
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace

int gemm_pair_dispatch(const char* name, int mode, const Dims& m, int N, int M, int K, const GemmOperands& op,
                       const GemmEpilogue& ep, const int* poff, const int* order, int* status, cudaStream_t s) {
  if (!get_encode()) return MOE_ERR_CUDA;
  const int bn = pair_bn(N);
  if (N % 128 || M % kPairM || op.a_cols % 128 || op.b_cols % 128 || op.a_rows % 128 || op.b_rows % 128)
    return MOE_ERR_INVALID_ARG;
  CUtensorMap ta, tb, tsa, tsb;
  if (!make_tmap(&ta, op.a, op.a_rows, op.a_cols, 128, false)) return MOE_ERR_CUDA;
  if (!make_tmap(&tb, op.b, op.b_rows, op.b_cols, bn / 2, false)) return MOE_ERR_CUDA;
  if (!make_tmap_sf(&tsa, op.a_sf, (op.a_rows / 128) * (op.a_cols / 128))) return MOE_ERR_CUDA;
  if (!make_tmap_sf(&tsb, op.b_sf, (op.b_rows / 128) * (op.b_cols / 128))) return MOE_ERR_CUDA;
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
  p.M = M;
  p.a_ktiles = op.a_cols / 128;
  p.b_ktiles = op.b_cols / 128;
  p.poff = poff;
  p.order = order;
  p.E = m.E;
  p.Ep = m.Ep;
  p.out = ep.out;
  p.out2 = ep.out2;
  p.ldo = ep.ldo;
  p.status = status;
  const int64_t per = static_cast<int64_t>(M / kPairM) * (N / bn);
  const int64_t tiles = mode == kWgrad ? m.Ep * per : per;
  p.static_tiles = static_cast<int>(tiles);
  switch (mode) {
    case kWgrad:
      return bn == 256 ? run_pair<kWgrad, 256, kPairKS>(name, ta, tb, tsa, tsb, to, to2, p, static_cast<int>(tiles), s)
                       : run_pair<kWgrad, 128, kPairKS>(name, ta, tb, tsa, tsb, to, to2, p, static_cast<int>(tiles), s);
    case kPlain:
      return bn == 256 ? run_pair<kPlain, 256, kPairKS>(name, ta, tb, tsa, tsb, to, to2, p, static_cast<int>(tiles), s)
                       : run_pair<kPlain, 128, kPairKS>(name, ta, tb, tsa, tsb, to, to2, p, static_cast<int>(tiles), s);
    default: return MOE_ERR_INVALID_ARG;
  }
}

}  // namespace moe

extern "C" int moe_gemm_mxfp8_pair(int M, int N, int K, const void* a, const void* a_sf, const void* b,
                                   const void* b_sf, float* c, moe_stream_t stream) {
  if (M <= 0 || N <= 0 || K <= 0 || M % moe::kPairM || N % 128 || K % 128 || !a || !a_sf || !b || !b_sf ||
      !c)
    return MOE_ERR_INVALID_ARG;
  if (!moe::arch_ok()) return MOE_ERR_UNSUPPORTED_ARCH;
  moe::CallScope call;
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
  if (int r = moe::gemm_pair_dispatch("gemm_plain_pair", moe::kPlain, m, N, M, K, op, ep, nullptr, nullptr, nullptr,
                                      static_cast<cudaStream_t>(stream)))
    return r;
  return call.status();
}
