// MX quantisers: along rows (K axis), along columns (token axis, transposed),
// token-axis gathers through the schedule, and scale re-tiling.
#include "moe_internal.h"
#include "mx.cuh"
#include "ptx.cuh"
#include "prof.h"

namespace moe {

// Row of the interleaved GEMM1 weight layout for source row r of w_gu:
// blocks of kGuBlock gate rows followed by the matching kGuBlock up rows.
__device__ __forceinline__ int64_t gu_interleave_row(int64_t r, int I) {
  const int64_t e = r / (2 * I);
  const int64_t i = r % (2 * I);
  const int64_t up = i >= I ? 1 : 0;
  const int64_t ii = i - up * I;
  return e * 2 * I + (ii / kGuBlock) * (2 * kGuBlock) + up * kGuBlock + (ii % kGuBlock);
}

// One thread per 32-element block along K.
// sf_rows (optional): a second, row-major copy of the scale bytes.
__global__ void quant_rows_kernel(const __nv_bfloat16* __restrict__ src, int64_t rows, int K, int64_t ld,
                                  uint8_t* __restrict__ codes, uint8_t* __restrict__ sf, int tiled,
                                  int interleave_I, uint8_t* __restrict__ sf_rows) {
  const int64_t nb = K / 32;
  const int64_t gid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (gid >= rows * nb) return;
  const int64_t r = gid / nb;
  const int64_t kb = gid - r * nb;
  float v[32];
  load_bf16x32(src + r * ld + kb * 32, v);
  const int b = mx_scale_byte(amax32(v));
  uint32_t w[8];
  mx_pack32(v, mx_inv_scale(b), w);
  const int64_t orow = interleave_I > 0 ? gu_interleave_row(r, interleave_I) : r;
  store32(codes + orow * K + kb * 32, w);
  sf[tiled ? sf_off(orow, kb, K / 128) : orow * nb + kb] = static_cast<uint8_t>(b);
  if (sf_rows != nullptr) sf_rows[orow * nb + kb] = static_cast<uint8_t>(b);
}

// Token-axis MX of src[rows][K]: block = 32 consecutive rows of one column.
// codes[K][rows_pad], scales per (column, row block). CTA: 32 rows x 256 cols.
__global__ void quant_cols_kernel(const __nv_bfloat16* __restrict__ src, int64_t rows, int K, int64_t ld,
                                  int64_t rows_pad, uint8_t* __restrict__ codes, uint8_t* __restrict__ sf,
                                  int tiled) {
  // blockIdx.z selects one matrix of a batch of equally shaped ones.
  src += static_cast<int64_t>(blockIdx.z) * rows * ld;
  codes += static_cast<int64_t>(blockIdx.z) * K * rows_pad;
  sf += static_cast<int64_t>(blockIdx.z) * K * (rows_pad / 32);
  const int c = blockIdx.x * 256 + threadIdx.x;
  const int64_t r0 = static_cast<int64_t>(blockIdx.y) * 32;
  if (c >= K) return;
  float v[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const int64_t r = r0 + i;
    v[i] = r < rows ? __bfloat162float(src[r * ld + c]) : 0.0f;
  }
  const int b = mx_scale_byte(amax32(v));
  uint32_t w[8];
  mx_pack32(v, mx_inv_scale(b), w);
  store32(codes + static_cast<int64_t>(c) * rows_pad + r0, w);
  const int64_t kb = r0 / 32;
  sf[tiled ? sf_off(c, kb, rows_pad / 128) : static_cast<int64_t>(c) * (rows_pad / 32) + kb] = static_cast<uint8_t>(b);
}

// Token of assignment a (routed a < T*k: a / k; shared: (a - T*k) % T).
__device__ __forceinline__ int token_of(int a, int T, int k) {
  const int A = T * k;
  return a < A ? a / k : (a - A) % T;
}

// Token-axis MX of gathered rows: padded row pr holds assignment a = row_src[pr]
// (or padding). value = src[t_a][c], times the gate w_a when scale_by_gate
// (shared-expert assignments have gate 1). Optionally also accumulates the
// router weight-gradient partial sums part[pr/32][c] = sum_r dl_a x[t_a][c]
// over the routed rows of the 32-row block, in rank order.
// CTA: 128 rows x 128 columns (blockIdx.x: row tile, blockIdx.y: column
// block), warp g on rows 32g..32g+31; lane l loads 8 bytes (columns
// 4l..4l+3) of each of its 32 rows and owns those 4 columns.
// The 4 warps' codes meet in shared memory, so each column's 128 rows are
// stored as one 128-byte run.
constexpr int kTokCols = 4;
constexpr int kTokThreads = 128;

__device__ __forceinline__ float bf16_lane(const uint2& u, int j) {
  const uint32_t w = j < 2 ? u.x : u.y;
  return (j & 1) ? __uint_as_float(w & 0xFFFF0000u) : __uint_as_float(w << 16);
}

// The gate-scaled form runs 3 CTAs per SM: the registers it needs for the
// gates of both passes then fit without spilling (0.55 -> 0.52 ms at the
// benchmark shape, against 4 CTAs per SM with a 96-byte spill).
template <bool kGate, bool kPart>
__global__ void __launch_bounds__(kTokThreads, kGate ? 3 : 4) tok_gather_kernel(
    const __nv_bfloat16* __restrict__ src, const int* __restrict__ row_src, const int* __restrict__ poff_end, int T,
    int k, int d, int64_t Rmax, const float* __restrict__ topk_w, const float* __restrict__ dl,
    float* __restrict__ part, uint8_t* __restrict__ codes, uint8_t* __restrict__ sf) {
  const int64_t r0 = static_cast<int64_t>(blockIdx.x) * 128;
  if (r0 >= *poff_end) return;
  __shared__ int s_tok[128];
  __shared__ float s_w[128];
  __shared__ float s_dl[128];
  __shared__ __align__(16) uint8_t st[128 * 128];   // [column][128 rows], 16-byte chunks swizzled
  __shared__ uint32_t ssf[128];                      // [column]: scale bytes of the 4 row blocks
  {
    const int a = row_src[r0 + threadIdx.x];
    float w = 1.0f, g = 0.0f;
    if (a >= 0 && a < T * k) {
      if (kGate) w = topk_w[a];
      if (kPart) g = dl[a];
    }
    s_tok[threadIdx.x] = a >= 0 ? token_of(a, T, k) : -1;
    s_w[threadIdx.x] = w;
    s_dl[threadIdx.x] = g;
  }
  __syncthreads();
  const int q = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cb = blockIdx.y * 128;
  const int c0 = cb + lane * kTokCols;
  const int* tok = s_tok + 32 * q;
  const float* wr = s_w + 32 * q;
  const float* dr = s_dl + 32 * q;
  uint2 raw[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const int t = tok[i];
    raw[i] = t >= 0 ? *reinterpret_cast<const uint2*>(src + static_cast<int64_t>(t) * d + c0) : make_uint2(0, 0);
  }
  float amax[kTokCols], acc[kTokCols];
#pragma unroll
  for (int j = 0; j < kTokCols; ++j) { amax[j] = 0.0f; acc[j] = 0.0f; }
#pragma unroll
  for (int i = 0; i < 32; ++i) {
#pragma unroll
    for (int j = 0; j < kTokCols; ++j) {
      float x = bf16_lane(raw[i], j);
      if (kPart) acc[j] = fmaf(dr[i], x, acc[j]);
      if (kGate) x = wr[i] * x;
      amax[j] = fmaxf(amax[j], fabsf(x));
    }
  }
#pragma unroll
  for (int j = 0; j < kTokCols; ++j) {
    const int b = mx_scale_byte(amax[j]);
    const float inv = mx_inv_scale(b);
    uint32_t w[8];
#pragma unroll
    for (int h = 0; h < 8; ++h) {
      float v4[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        float x = bf16_lane(raw[4 * h + u], j);
        if (kGate) x = wr[4 * h + u] * x;
        v4[u] = x * inv;
      }
      w[h] = e4m3x2(v4[0], v4[1]) | (e4m3x2(v4[2], v4[3]) << 16);
    }
    const int col = lane * kTokCols + j;
    uint8_t* run = st + col * 128;
    *reinterpret_cast<uint4*>(run + (((2 * q) ^ (lane & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
    *reinterpret_cast<uint4*>(run + (((2 * q + 1) ^ (lane & 7)) << 4)) = make_uint4(w[4], w[5], w[6], w[7]);
    reinterpret_cast<uint8_t*>(ssf)[col * 4 + q] = static_cast<uint8_t>(b);
  }
  if (kPart)
    *reinterpret_cast<float4*>(part + (r0 / 32 + q) * d + c0) = make_float4(acc[0], acc[1], acc[2], acc[3]);
  __syncthreads();
  // 128 columns x 128 rows of codes: 8 threads per 128-byte column run.
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int idx = threadIdx.x + kTokThreads * i;
    const int col = idx >> 3, ch = idx & 7;
    const uint4 v = *reinterpret_cast<const uint4*>(st + col * 128 + ((ch ^ ((col >> 2) & 7)) << 4));
    *reinterpret_cast<uint4*>(codes + static_cast<int64_t>(cb + col) * Rmax + r0 + ch * 16) = v;
  }
  *reinterpret_cast<uint32_t*>(sf + sf_off(cb + threadIdx.x, r0 >> 5, Rmax >> 7)) = ssf[threadIdx.x];
}

// Packed two-wide fp32 arithmetic (one instruction for two lanes of values;
// each result rounded to nearest like the scalar operation).
__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "mov.b64 rc, {%6, %7};\n\tfma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}
// Two E4M3 codes of (a.x, a.y) * inv.
__device__ __forceinline__ uint32_t e4m3x2_scaled(float2 a, float inv) {
  const float2 v = fmul2(a, make_float2(inv, inv));
  return e4m3x2(v.x, v.y);
}

// SwiGLU backward of padded rank rows and the two MX forms of dGU = [dg | du]:
// along 2I per row (q_rows, tiled scales) and along ranks per column (q_tok,
// [2I][Rmax], tiled scales). Row pr is an assignment iff row_src[pr] >= 0;
// other rows of an expert's padded segment give zeros.
//   sg = sigmoid(g), dg = dh u sg (1 + g (1 - sg)), du = dh g sg   (fp32;
//   sg from __expf and a fast divide, a few ulp, as in the forward)
// CTA: 128 rows x 32 columns of I; warp q takes rows 32q..32q+31. Lane
// (gq = lane / 8, cq = lane % 8) holds rows 8gq..8gq+7 of the warp's block
// and columns 4cq..4cq+3, so each load instruction reads 4 rows' contiguous
// 128-byte (dh) or 64-byte (g, u) runs, and a row's 32-column MX block is
// spread over the 8 lanes of one group (amax by 3 shuffles) while a column's
// 32-row token block is spread over the 4 groups (amax by 2 shuffles). The
// token-axis codes of the 4 warps meet in shared memory, so each column's
// 128 rows are stored as one 128-byte run. 6 CTAs per SM (80 registers, a
// 20-byte spill): faster than 5 CTAs without a spill (0.76 against 0.77 ms).
__global__ void __launch_bounds__(128, 6) swiglu_bwd_quant_kernel(
    const float* __restrict__ dh, const __nv_bfloat16* __restrict__ gu, const int* __restrict__ row_src,
    const int* __restrict__ poff_end, int I, int64_t Rmax, uint8_t* __restrict__ q_rows,
    uint8_t* __restrict__ q_rows_sf, uint8_t* __restrict__ q_tok, uint8_t* __restrict__ q_tok_sf) {
  __shared__ __align__(16) uint8_t tst[2][32 * 128];   // [dg|du][column][128 rows], 16-byte chunks swizzled
  __shared__ uint32_t tsf[2][32];                        // [dg|du][column]: 4 scale bytes (row blocks)
  const int q = threadIdx.x >> 5, lane = threadIdx.x & 31, gq = lane >> 3, cq = lane & 7;
  const int64_t r0 = static_cast<int64_t>(blockIdx.y) * 128;
  if (r0 >= *poff_end) return;
  const int c0 = blockIdx.x * 32;
  const int64_t wrow = r0 + q * 32;                       // first row of this warp's block
  const uint32_t valid = __ballot_sync(0xFFFFFFFFu, row_src[wrow + lane] >= 0);
  // All 24 loads are issued before any arithmetic (coherent ld_global_* loads and the
  // warp barrier after them): left to itself the compiler sinks them toward
  // their uses, and the kernel took 1.22 instead of 0.78 ms at full size.
  float4 hv[8];
  uint2 gv[8], uv[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int64_t prow = wrow + 8 * gq + i;
    hv[i] = ld_global_f4(dh + prow * I + c0 + 4 * cq);
    // saved g,u: 32-column chunk c0 / 32 of the row holds g then u
    const __nv_bfloat16* pg = gu + prow * (2 * I) + 2 * c0 + 4 * cq;
    gv[i] = ld_global_u2(pg);
    uv[i] = ld_global_u2(pg + 32);
  }
  __syncwarp();
  float dg[8][4], du[8][4];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float h[4] = {hv[i].x, hv[i].y, hv[i].z, hv[i].w};
    const float g[4] = {__uint_as_float(gv[i].x << 16), __uint_as_float(gv[i].x & 0xFFFF0000u),
                        __uint_as_float(gv[i].y << 16), __uint_as_float(gv[i].y & 0xFFFF0000u)};
    const float u[4] = {__uint_as_float(uv[i].x << 16), __uint_as_float(uv[i].x & 0xFFFF0000u),
                        __uint_as_float(uv[i].y << 16), __uint_as_float(uv[i].y & 0xFFFF0000u)};
    const bool ok = (valid >> (8 * gq + i)) & 1u;
#pragma unroll
    for (int j = 0; j < 4; j += 2) {   // columns j, j + 1 as one packed pair
      if (ok) {
        const float2 sg = make_float2(__fdividef(1.0f, 1.0f + __expf(-g[j])),
                                      __fdividef(1.0f, 1.0f + __expf(-g[j + 1])));
        const float2 hh = make_float2(h[j], h[j + 1]), gg = make_float2(g[j], g[j + 1]);
        const float2 uu = make_float2(u[j], u[j + 1]), one = make_float2(1.0f, 1.0f);
        const float2 om = ffma2(sg, make_float2(-1.0f, -1.0f), one);            // 1 - sg
        const float2 d = fmul2(fmul2(fmul2(hh, uu), sg), ffma2(gg, om, one));   // h u sg (1 + g (1 - sg))
        const float2 e = fmul2(hh, fmul2(gg, sg));                              // h (g sg)
        dg[i][j] = d.x; dg[i][j + 1] = d.y;
        du[i][j] = e.x; du[i][j + 1] = e.y;
      } else {
        dg[i][j] = dg[i][j + 1] = 0.0f;
        du[i][j] = du[i][j + 1] = 0.0f;
      }
    }
  }
  // Row form: 32-column block of one row = the 8 lanes of a group, 4 code bytes each.
  // The lane's 8 rows lie in one 32-row block of the tiled scales: row i's byte is 16 i past row 0's.
  const int ktl = 2 * I / 128;
  const int64_t prow0 = wrow + 8 * gq;
#pragma unroll
  for (int x = 0; x < 2; ++x) {
    float (*v)[4] = x == 0 ? dg : du;
    const int col = x * I + c0;
    uint8_t* qr = q_rows + prow0 * (2 * I) + col + 4 * cq;
    uint8_t* qs = q_rows_sf + sf_off(prow0, col >> 5, ktl);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float m = fmaxf(fmaxf(fabsf(v[i][0]), fabsf(v[i][1])), fmaxf(fabsf(v[i][2]), fabsf(v[i][3])));
      m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
      m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
      m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 4));
      const int b = mx_scale_byte(m);
      const float inv = mx_inv_scale(b);
      *reinterpret_cast<uint32_t*>(qr + static_cast<int64_t>(i) * (2 * I)) =
          e4m3x2_scaled(make_float2(v[i][0], v[i][1]), inv) | (e4m3x2_scaled(make_float2(v[i][2], v[i][3]), inv) << 16);
      if (cq == 0) qs[16 * i] = static_cast<uint8_t>(b);
    }
  }
  // Token form: column 4cq + j, 32 rows = 4 groups x 8 rows; this lane's 8 rows give 8 contiguous code bytes.
#pragma unroll
  for (int x = 0; x < 2; ++x) {
    float (*v)[4] = x == 0 ? dg : du;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float m = fmaxf(fmaxf(fmaxf(fabsf(v[0][j]), fabsf(v[1][j])), fmaxf(fabsf(v[2][j]), fabsf(v[3][j]))),
                      fmaxf(fmaxf(fabsf(v[4][j]), fabsf(v[5][j])), fmaxf(fabsf(v[6][j]), fabsf(v[7][j]))));
      m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 8));
      m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 16));
      const int b = mx_scale_byte(m);
      const float inv = mx_inv_scale(b);
      const uint32_t w0 = e4m3x2_scaled(make_float2(v[0][j], v[1][j]), inv) |
                          (e4m3x2_scaled(make_float2(v[2][j], v[3][j]), inv) << 16);
      const uint32_t w1 = e4m3x2_scaled(make_float2(v[4][j], v[5][j]), inv) |
                          (e4m3x2_scaled(make_float2(v[6][j], v[7][j]), inv) << 16);
      const int col = 4 * cq + j;
      // rows 32q + 8gq .. +7 of the column: chunk 2q + gq/2, half gq % 2; chunks swizzled by col / 4
      const int ch = (2 * q + (gq >> 1)) ^ cq;
      *reinterpret_cast<uint2*>(tst[x] + col * 128 + ch * 16 + (gq & 1) * 8) = make_uint2(w0, w1);
      if (gq == 0) reinterpret_cast<uint8_t*>(tsf[x])[col * 4 + q] = static_cast<uint8_t>(b);
    }
  }
  __syncthreads();
  // 2 x 32 columns x 128 rows of codes: 8 threads per 128-byte column run.
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int idx = threadIdx.x + 128 * i;
    const int x = idx >> 8, col = (idx >> 3) & 31, ch = idx & 7;
    const uint4 v = *reinterpret_cast<const uint4*>(tst[x] + col * 128 + ((ch ^ ((col >> 2) & 7)) << 4));
    *reinterpret_cast<uint4*>(q_tok + static_cast<int64_t>(x * I + c0 + col) * Rmax + r0 + ch * 16) = v;
  }
  if (threadIdx.x < 64) {
    const int x = threadIdx.x >> 5, col = threadIdx.x & 31;
    *reinterpret_cast<uint32_t*>(q_tok_sf + sf_off(x * I + c0 + col, r0 >> 5, Rmax >> 7)) = tsf[x][col];
  }
}

__global__ void scales_to_tiled_kernel(const uint8_t* __restrict__ canon, int64_t rows, int nb, uint8_t* tiled) {
  const int64_t gid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (gid >= rows * nb) return;
  const int64_t r = gid / nb, kb = gid - (gid / nb) * nb;
  tiled[sf_off(r, kb, nb / 4)] = canon[gid];
}

void launch_quant_rows(const void* src, int64_t rows, int K, int64_t ld, uint8_t* codes, uint8_t* sf, bool tiled,
                       int interleave_I, cudaStream_t s, uint8_t* sf_rows) {
  const int64_t n = rows * (K / 32);
  if (n == 0) return;
  const int threads = 256;
  launch_kernel("quant_rows", quant_rows_kernel, dim3(static_cast<unsigned>(ceil_div(n, threads))), dim3(threads), 0, s,
      static_cast<const __nv_bfloat16*>(src), rows, K, ld, codes, sf, tiled ? 1 : 0, interleave_I, sf_rows);
}

void launch_quant_cols(const void* src, int64_t rows, int K, int64_t ld, int64_t rows_pad, uint8_t* codes,
                       uint8_t* sf, bool tiled, int batch, cudaStream_t s) {
  if (rows_pad == 0 || K == 0 || batch == 0) return;
  dim3 grid(static_cast<unsigned>(ceil_div(K, 256)), static_cast<unsigned>(rows_pad / 32), static_cast<unsigned>(batch));
  launch_kernel("quant_cols", quant_cols_kernel, grid, dim3(256), 0, s, static_cast<const __nv_bfloat16*>(src), rows, K,
                ld, rows_pad, codes, sf, tiled ? 1 : 0);
}

void launch_swiglu_bwd_quant(const Dims& m, const Layout& L, void* ws, cudaStream_t s) {
  if (m.Rmax == 0) return;
  dim3 grid(static_cast<unsigned>(m.I / 32), static_cast<unsigned>(m.Rmax / 128));
  launch_kernel("swiglu_bwd_quant", swiglu_bwd_quant_kernel, grid, dim3(128), 0, s,
      ws_ptr<float>(L, ws, MOE_WS_DH), ws_ptr<__nv_bfloat16>(L, ws, MOE_WS_GU), ws_ptr<int>(L, ws, MOE_WS_ROWSRC),
      ws_ptr<int>(L, ws, MOE_WS_POFF) + m.Ep, m.I, m.Rmax, ws_ptr<uint8_t>(L, ws, MOE_WS_DGU),
      ws_ptr<uint8_t>(L, ws, MOE_WS_DGU_SF), ws_ptr<uint8_t>(L, ws, MOE_WS_DGUTOK),
      ws_ptr<uint8_t>(L, ws, MOE_WS_DGUTOK_SF));
}

void launch_tok_gather(const Dims& m, const void* src_rows, bool scale_by_gate, const float* topk_w,
                       bool router_partials, const Layout& L, void* ws, uint8_t* codes, uint8_t* sf,
                       cudaStream_t s) {
  // Rank tiles vary fastest: the CTAs resident at one time share one 128-column
  // block, whose slice of every token (256 bytes of each source row) stays in
  // L2 across the token's k + S gathered copies.
  dim3 grid(static_cast<unsigned>(m.Rmax / 128), static_cast<unsigned>(m.d / 128));
  const int* poff = ws_ptr<int>(L, ws, MOE_WS_POFF);
  const auto* sp = static_cast<const __nv_bfloat16*>(src_rows);
  const int* rs = ws_ptr<int>(L, ws, MOE_WS_ROWSRC);
  const float* dl = router_partials ? ws_ptr<float>(L, ws, MOE_WS_DL) : nullptr;
  float* part = router_partials ? ws_ptr<float>(L, ws, MOE_WS_DWR_PART) : nullptr;
  auto kern = scale_by_gate ? (router_partials ? tok_gather_kernel<true, true> : tok_gather_kernel<true, false>)
                            : (router_partials ? tok_gather_kernel<false, true> : tok_gather_kernel<false, false>);
  launch_kernel(scale_by_gate ? "tok_gather_dO" : "tok_gather_x", kern, grid, dim3(kTokThreads), 0, s, sp, rs,
                poff + m.Ep, m.T, m.k, m.d, m.Rmax, topk_w, dl, part, codes, sf);
}

}  // namespace moe

extern "C" int moe_scales_to_tiled(const void* canon, int rows, int K, void* tiled, moe_stream_t stream) {
  if (canon == nullptr || tiled == nullptr || rows <= 0 || K <= 0 || rows % 128 || K % 128) return MOE_ERR_INVALID_ARG;
  const int nb = K / 32;
  const int64_t n = static_cast<int64_t>(rows) * nb;
  moe::CallScope call;
  moe::launch_kernel("scales_to_tiled", moe::scales_to_tiled_kernel, dim3(static_cast<unsigned>(moe::ceil_div(n, 256))),
                     dim3(256), 0, static_cast<cudaStream_t>(stream), static_cast<const uint8_t*>(canon),
                     static_cast<int64_t>(rows), nb, static_cast<uint8_t*>(tiled));
  return call.status();
}
