// NVFP4: quantiser (bf16 -> E2M1 codes + E4M3 block scales) and the plain
// NVFP4 GEMM entry point on the tcgen05 kernel (kind::mxf4nvf4).
//
// Reading of "NVFP4" (Cursor blog summary, opening paragraph: Cursor's earlier
// NVFP4 training kernels; no further detail): NVIDIA's 4-bit format, E2M1
// elements, one E4M3 scale per 16 elements, one fp32 scale g per tensor.
// Rounding points, every step an IEEE binary32 operation:
//   denom = 6 g;  sb = E4M3_RNE_satfinite(amax(block) / denom);
//   X = decode(sb) g;  q = E2M1_RNE_satfinite(v / X) (0 when X = 0).
// The GEMM multiplies the fp32 product by alpha = g_a g_b.
#include <cuda_fp4.h>
#include <cuda_fp8.h>

#include "gemm.cuh"
#include "prof.h"

namespace moe {

__device__ __forceinline__ float e4m3_value(uint8_t b) {
  const __half_raw h = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(b), __NV_E4M3);
  return __half2float(__half(h));
}

// One thread per 16-element block along K.
__global__ void quant_nvfp4_kernel(const __nv_bfloat16* __restrict__ src, int64_t rows, int K, float g,
                                   uint8_t* __restrict__ codes, uint8_t* __restrict__ sf, int tiled) {
  const int64_t nb = K / 16;
  const int64_t gid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (gid >= rows * nb) return;
  const int64_t r = gid / nb;
  const int64_t kb = gid - r * nb;
  const uint4* p = reinterpret_cast<const uint4*>(src + r * K + kb * 16);
  const uint4 u0 = p[0], u1 = p[1];
  const uint32_t w[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
  float v[16];
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    amax = fmaxf(amax, fmaxf(fabsf(v[2 * i]), fabsf(v[2 * i + 1])));
  }
  const float denom = __fmul_rn(6.0f, g);
  const uint8_t sb = static_cast<uint8_t>(
      __nv_cvt_float_to_fp8(__fdiv_rn(amax, denom), __NV_SATFINITE, __NV_E4M3));
  const float X = __fmul_rn(e4m3_value(sb), g);
  uint32_t packed[2] = {0u, 0u};
  if (X > 0.0f) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t b = static_cast<uint32_t>(__nv_cvt_float2_to_fp4x2(
          make_float2(__fdiv_rn(v[2 * i], X), __fdiv_rn(v[2 * i + 1], X)), __NV_E2M1, cudaRoundNearest));
      packed[i >> 2] |= (b & 0xFFu) << (8 * (i & 3));
    }
  }
  *reinterpret_cast<uint2*>(codes + r * (K / 2) + kb * 8) = make_uint2(packed[0], packed[1]);
  sf[tiled ? sf_off(r, kb, K / 64) : r * nb + kb] = sb;
}

void launch_quant_nvfp4(const void* src, int64_t rows, int K, float g, uint8_t* codes, uint8_t* sf, bool tiled,
                        cudaStream_t s) {
  const int64_t n = rows * (K / 16);
  if (n == 0) return;
  launch_kernel("quant_nvfp4", quant_nvfp4_kernel, dim3(static_cast<unsigned>(ceil_div(n, 256))), dim3(256), 0, s,
                static_cast<const __nv_bfloat16*>(src), rows, K, g, codes, sf, tiled ? 1 : 0);
}

}  // namespace moe

extern "C" int moe_quantize_nvfp4(const void* src, int rows, int K, float g, void* codes, void* scales, int tiled,
                                  moe_stream_t stream) {
  if (src == nullptr || codes == nullptr || scales == nullptr || rows < 0 || K <= 0 || K % 16) return MOE_ERR_INVALID_ARG;
  if (!(g > 0.0f) || (tiled && (rows % 128 || K % 64))) return MOE_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(src) % 16 || reinterpret_cast<uintptr_t>(codes) % 8) return MOE_ERR_INVALID_ARG;
  if (!moe::arch_ok()) return MOE_ERR_UNSUPPORTED_ARCH;
  if (rows == 0) return MOE_OK;
  moe::CallScope call;
  moe::launch_quant_nvfp4(src, rows, K, g, static_cast<uint8_t*>(codes), static_cast<uint8_t*>(scales), tiled != 0,
                          static_cast<cudaStream_t>(stream));
  return call.status();
}

namespace {

// The NVFP4 expert GEMM over the schedule in ws: fp32 rank-ordered rows
// (kGroupedNv4) or bf16 rows pushed to their assignment (kPushNv4).
int expert_gemm_nvfp4(const moe_config_t* cfg, int mode, int N, int K, const void* a, const void* a_sf,
                      const void* w, const void* w_sf, float alpha, void* out, void* ws, moe_stream_t stream) {
  if (int r = moe::validate(cfg)) return r;
  if (N <= 0 || K <= 0 || N % 128 || K % 256 || !a || !a_sf || !w || !w_sf || !out || !ws) return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(a) | reinterpret_cast<uintptr_t>(w) | reinterpret_cast<uintptr_t>(a_sf) |
       reinterpret_cast<uintptr_t>(w_sf) | reinterpret_cast<uintptr_t>(out) | reinterpret_cast<uintptr_t>(ws)) & 15u)
    return MOE_ERR_INVALID_ARG;
  if (!moe::arch_ok()) return MOE_ERR_UNSUPPORTED_ARCH;
  moe::CallScope call;
  const moe::Layout L = moe::make_layout(cfg);
  const moe::Dims& m = L.m;
  if (m.T == 0) return MOE_OK;
  moe::GemmOperands op{};
  op.a = static_cast<const uint8_t*>(a);
  op.a_rows = m.Rmax;
  op.a_cols = K / 2;      // packed bytes per row
  op.a_sf = static_cast<const uint8_t*>(a_sf);
  op.b = static_cast<const uint8_t*>(w);
  op.b_rows = static_cast<int64_t>(m.Ep) * N;
  op.b_cols = K / 2;
  op.b_sf = static_cast<const uint8_t*>(w_sf);
  moe::GemmEpilogue ep{};
  ep.out = out;
  ep.ldo = N;
  ep.alpha = alpha;
  if (int r = moe::gemm_dispatch(mode == moe::kPushNv4 ? "expert_gemm_nvfp4_push" : "expert_gemm_nvfp4", mode, m, 0,
                                 N, K, static_cast<int>(m.Rmax), op, ep, moe::ws_ptr<int>(L, ws, MOE_WS_COUNTS),
                                 moe::ws_ptr<int>(L, ws, MOE_WS_POFF), nullptr, moe::ws_ptr<int>(L, ws, MOE_WS_ROWSRC),
                                 moe::ws_ptr<int>(L, ws, MOE_WS_STATUS), static_cast<cudaStream_t>(stream), 0, nullptr,
                                 nullptr, moe::ws_ptr<int>(L, ws, MOE_WS_PUSHINFO)))
    return r;
  return call.status();
}

}  // namespace

extern "C" int moe_expert_gemm_nvfp4(const moe_config_t* cfg, int N, int K, const void* a, const void* a_sf,
                                     const void* w, const void* w_sf, float alpha, float* out, void* ws,
                                     moe_stream_t stream) {
  return expert_gemm_nvfp4(cfg, moe::kGroupedNv4, N, K, a, a_sf, w, w_sf, alpha, out, ws, stream);
}

extern "C" int moe_expert_gemm_nvfp4_push(const moe_config_t* cfg, int N, int K, const void* a, const void* a_sf,
                                          const void* w, const void* w_sf, float alpha, void* out, void* ws,
                                          moe_stream_t stream) {
  return expert_gemm_nvfp4(cfg, moe::kPushNv4, N, K, a, a_sf, w, w_sf, alpha, out, ws, stream);
}

extern "C" int moe_gemm_nvfp4(int M, int N, int K, const void* a, const void* a_sf, const void* b, const void* b_sf,
                              float alpha, float* c, moe_stream_t stream) {
  if (M <= 0 || N <= 0 || K <= 0 || M % 128 || N % 128 || K % 256 || !a || !a_sf || !b || !b_sf || !c)
    return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(a) | reinterpret_cast<uintptr_t>(b) | reinterpret_cast<uintptr_t>(a_sf) |
       reinterpret_cast<uintptr_t>(b_sf) | reinterpret_cast<uintptr_t>(c)) & 15u)
    return MOE_ERR_INVALID_ARG;
  if (!moe::arch_ok()) return MOE_ERR_UNSUPPORTED_ARCH;
  moe::CallScope call;
  moe::Dims m{};
  moe::GemmOperands op{};
  op.a = static_cast<const uint8_t*>(a);
  op.a_rows = M;
  op.a_cols = K / 2;      // packed bytes per row
  op.a_sf = static_cast<const uint8_t*>(a_sf);
  op.b = static_cast<const uint8_t*>(b);
  op.b_rows = N;
  op.b_cols = K / 2;
  op.b_sf = static_cast<const uint8_t*>(b_sf);
  moe::GemmEpilogue ep{};
  ep.out = c;
  ep.ldo = N;
  ep.alpha = alpha;
  if (int r = moe::gemm_dispatch("gemm_nvfp4", moe::kPlainNv4, m, 0, N, K, M, op, ep, nullptr, nullptr, nullptr,
                                 nullptr, nullptr, static_cast<cudaStream_t>(stream)))
    return r;
  return call.status();
}
