// Router: logits on the tensor cores, then sigmoid + bias + group-limited
// top-k + gate normalisation as warp-shuffle reductions (one warp per token).
//
// Reading of "DSV3-style router" (Cursor blog summary, "method points"):
// s = sigmoid(logit) in the specified fp32 arithmetic below, v = s + bias,
// group score = sum of the two largest v of the group, keep the topk_groups
// best groups (ties to the lower group), take the k best v among kept
// experts (ties to the lower expert), slots in descending-v order, gates
// w = s / sum(s) summed in slot order.
#include <cudaTypedefs.h>

#include <mutex>

#include "moe_internal.h"
#include "gemm.cuh"
#include "prof.h"

namespace moe {

// sigma(l) = 1 / (1 + E(-clamp(l, -80, 80))), E by Cody-Waite reduction
// (W. J. Cody and W. Waite, 1980) and a degree-7 Taylor polynomial, every
// operation an IEEE binary32 round-to-nearest op without contraction.
__device__ __forceinline__ float sigmoid_spec(float l) {
  constexpr double kLn2 = 0.6931471805599453094;
  constexpr float kLog2e = static_cast<float>(1.0 / kLn2);
  constexpr float kC1 = 355.0f / 512.0f;                               // ln2 to 9 significant bits
  constexpr float kC2 = static_cast<float>(kLn2 - 355.0 / 512.0);      // remainder
  constexpr float c0 = 1.0f, c1 = 1.0f, c2 = 0.5f;
  constexpr float c3 = static_cast<float>(1.0 / 6.0), c4 = static_cast<float>(1.0 / 24.0);
  constexpr float c5 = static_cast<float>(1.0 / 120.0), c6 = static_cast<float>(1.0 / 720.0);
  constexpr float c7 = static_cast<float>(1.0 / 5040.0);
  const float lc = fminf(fmaxf(l, -80.0f), 80.0f);
  const float z = -lc;
  const float n = rintf(__fmul_rn(z, kLog2e));
  const float r = __fsub_rn(__fsub_rn(z, __fmul_rn(n, kC1)), __fmul_rn(n, kC2));
  float p = c7;
  p = __fadd_rn(__fmul_rn(p, r), c6);
  p = __fadd_rn(__fmul_rn(p, r), c5);
  p = __fadd_rn(__fmul_rn(p, r), c4);
  p = __fadd_rn(__fmul_rn(p, r), c3);
  p = __fadd_rn(__fmul_rn(p, r), c2);
  p = __fadd_rn(__fmul_rn(p, r), c1);
  p = __fadd_rn(__fmul_rn(p, r), c0);
  const float two_n = __int_as_float((static_cast<int>(n) + 127) << 23);
  const float e = __fmul_rn(p, two_n);
  return __fdiv_rn(1.0f, __fadd_rn(1.0f, e));
}

// (v1, e1) ranks above (v2, e2): larger value, ties to the lower index.
__device__ __forceinline__ bool better(float v1, int e1, float v2, int e2) {
  return v1 > v2 || (v1 == v2 && e1 < e2);
}

__device__ __forceinline__ void warp_best(float& v, int& e) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, v, o);
    const int oe = __shfl_xor_sync(0xffffffffu, e, o);
    if (better(ov, oe, v, e)) { v = ov; e = oe; }
  }
}

// One warp per token. Lane l owns experts e = l + 32 i, i < kMaxPerLane
// (a compile-time bound on ceil(E / 32), so the per-lane loops have no dead
// iterations at the common expert counts).
template <int kMaxPerLane>
__global__ void router_topk_kernel(const float* __restrict__ logits, const float* __restrict__ bias, int T, int E,
                                   int k, int G, int gtop, int32_t* __restrict__ idx_out,
                                   float* __restrict__ w_out, float* __restrict__ s_out) {
  extern __shared__ float sv_all[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x >> 5) + warp;
  float* sv = sv_all + warp * E;
  if (t >= T) return;
  float s[kMaxPerLane], v[kMaxPerLane];
  const int per_lane = (E + 31) / 32;
#pragma unroll
  for (int i = 0; i < kMaxPerLane; ++i) {
    const int e = lane + 32 * i;
    if (i < per_lane && e < E) {
      s[i] = sigmoid_spec(logits[static_cast<int64_t>(t) * E + e]);
      v[i] = __fadd_rn(s[i], bias[e]);
      sv[e] = v[i];
    } else {
      s[i] = 0.0f;
      v[i] = -INFINITY;
    }
  }
  __syncwarp();
  uint32_t kept = 0xffffffffu;
  if (G > 1) {
    const int per = E / G;
    float gs = -INFINITY;
    if (lane < G) {
      float m1 = -INFINITY, m2 = -INFINITY;
      for (int e = lane * per; e < (lane + 1) * per; ++e) {
        const float x = sv[e];
        if (x > m1) { m2 = m1; m1 = x; } else if (x > m2) { m2 = x; }
      }
      gs = __fadd_rn(m1, m2);
    }
    kept = 0;
    for (int r = 0; r < gtop; ++r) {
      float bv = (lane < G && !((kept >> lane) & 1u)) ? gs : -INFINITY;
      int be = lane < G && !((kept >> lane) & 1u) ? lane : 0x7fffffff;
      warp_best(bv, be);
      kept |= 1u << be;
    }
  }
  // This lane's candidates (experts of kept groups), one bit per slot i:
  // the group of each slot is found once, not in every selection round.
  const int per = G > 1 ? E / G : E;
  uint32_t cand = 0;
#pragma unroll
  for (int i = 0; i < kMaxPerLane; ++i) {
    const int e = lane + 32 * i;
    if (i < per_lane && e < E && ((kept >> (e / per)) & 1u)) cand |= 1u << i;
  }
  uint32_t taken = 0;
  int sel_e[8];          // k <= 8 (checked by the API); unrolled, so both stay in registers
  float sel_s[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    if (j >= k) break;   // k is the same in every lane
    float bv = -INFINITY;
    int be = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < kMaxPerLane; ++i) {
      const int e = lane + 32 * i;
      if (((cand & ~taken) >> i) & 1u) {
        if (better(v[i], e, bv, be)) { bv = v[i]; be = e; }
      }
    }
    warp_best(bv, be);
    if ((be & 31) == lane) taken |= 1u << (be >> 5);
    float sw = 0.0f;
#pragma unroll
    for (int i = 0; i < kMaxPerLane; ++i)
      if (i == (be >> 5)) sw = s[i];
    sel_s[j] = __shfl_sync(0xffffffffu, sw, be & 31);
    sel_e[j] = be;
  }
  // Every lane sums the selected scores in slot order; lane j writes slot j.
  float tot = sel_s[0];
#pragma unroll
  for (int j = 1; j < 8; ++j)
    if (j < k) tot = __fadd_rn(tot, sel_s[j]);
  float my_s = 0.0f;
  int my_e = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j)
    if (j == lane && j < k) { my_s = sel_s[j]; my_e = sel_e[j]; }
  if (lane < k) {
    const int64_t o = static_cast<int64_t>(t) * k + lane;
    idx_out[o] = my_e;
    w_out[o] = __fdiv_rn(my_s, tot);
    if (s_out != nullptr) s_out[o] = my_s;
  }
}

int launch_router_logits(const Dims& m, const void* x, const void* w_router, float* logits, cudaStream_t s) {
  GemmOperands op{};
  op.a = static_cast<const uint8_t*>(x);
  op.a_rows = m.T;
  op.a_cols = m.d;
  op.b = static_cast<const uint8_t*>(w_router);
  op.b_rows = m.E;
  op.b_cols = m.d;
  GemmEpilogue ep{};
  ep.out = logits;
  ep.ldo = m.E;
  return gemm_dispatch("router_gemm", kRouterMode, m, 0, m.E, m.d, m.T, op, ep, nullptr, nullptr, nullptr, nullptr,
                       nullptr, s);
}

void launch_router_topk(const Dims& m, const float* logits, const float* bias, int32_t* idx, float* w, float* s_sel,
                        cudaStream_t s) {
  if (m.T == 0) return;
  const int warps = 4;
  const int per = (m.E + 31) / 32;   // E <= 512
  auto kern = per <= 4 ? router_topk_kernel<4> : per <= 8 ? router_topk_kernel<8> : per <= 12 ? router_topk_kernel<12>
                                                                                    : router_topk_kernel<16>;
  launch_kernel("router_topk", kern, dim3(static_cast<unsigned>(ceil_div(m.T, warps))), dim3(warps * 32),
                warps * m.E * sizeof(float), s, logits, bias, m.T, m.E, m.k, m.G, m.gtop, idx, w, s_sel);
}

// ---------------------------------------------------------------- router without allocation
// Scratch of moe_route_noalloc: the fp32 logits of one call, in a fixed
// file-scope device array (every GPU that loads the library holds it until
// the process exits). Host code must not pass the array's name to a kernel:
// on the host it is only a stand-in symbol, so its device address is looked
// up with cudaGetSymbolAddress, once per CUDA context of a device.
constexpr int64_t kRouteScratchFloats = int64_t(1) << 22;   // 16 MiB: T * E <= 4,194,304
static __device__ __align__(256) float g_route_scratch[kRouteScratchFloats];

namespace {
std::mutex g_scratch_mu;
struct ScratchSlot {
  unsigned long long ctx_id = 0;   // context the address belongs to (0 = none yet)
  float* addr = nullptr;
};
ScratchSlot g_scratch[kMaxDev];

PFN_cuCtxGetCurrent_v4000 g_ctx_current = nullptr;
PFN_cuCtxGetId_v12000 g_ctx_id = nullptr;

// Unique id of the calling thread's current context (ids are never reused in a
// process, so a context created after cudaDeviceReset gets a new one); 0 if
// it cannot be read.
unsigned long long current_ctx_id() {
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(f);
  });
  if (g_ctx_current == nullptr || g_ctx_id == nullptr) return 0;
  CUcontext c = nullptr;
  unsigned long long id = 0;
  if (g_ctx_current(&c) != CUDA_SUCCESS || c == nullptr || g_ctx_id(c, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Device address of the scratch in the current context (looked up on the
// first call in each context).
int route_scratch(float** out) {
  const int dev = current_device();
  if (dev < 0) return MOE_ERR_CUDA;
  const unsigned long long id = current_ctx_id();
  if (id == 0) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  ScratchSlot& slot = g_scratch[dev];
  if (slot.ctx_id != id) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_route_scratch) != cudaSuccess || p == nullptr) {
      (void)cudaGetLastError();   // the failed lookup's own error: not left for the caller to find
      return MOE_ERR_CUDA;
    }
    slot.addr = static_cast<float*>(p);
    slot.ctx_id = id;
  }
  *out = slot.addr;
  return MOE_OK;
}
}  // namespace

}  // namespace moe

extern "C" int moe_route_noalloc(const moe_config_t* cfg, const void* x, const void* w_router, const float* bias,
                                 int32_t* topk_idx, float* topk_w, moe_stream_t stream) {
  if (int r = moe::validate(cfg)) return r;
  const bool no_tokens = cfg->T == 0;   // per-token arrays may be null then
  if ((!x && !no_tokens) || !w_router || !bias || (!topk_idx && !no_tokens) || (!topk_w && !no_tokens))
    return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(w_router)) & 15u) return MOE_ERR_INVALID_ARG;
  if (static_cast<int64_t>(cfg->T) * cfg->E > moe::kRouteScratchFloats) return MOE_ERR_SCRATCH;
  if (!moe::arch_ok()) return MOE_ERR_UNSUPPORTED_ARCH;
  if (cfg->T == 0) return MOE_OK;
  float* logits = nullptr;
  if (int r = moe::route_scratch(&logits)) return r;
  const moe::Dims m = moe::make_dims(cfg);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  moe::CallScope call;
  if (int r = moe::launch_router_logits(m, x, w_router, logits, s)) return r;
  moe::launch_router_topk(m, logits, bias, topk_idx, topk_w, nullptr, s);
  return call.status();
}
