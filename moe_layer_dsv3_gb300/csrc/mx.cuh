// MXFP8 device helpers: E8M0 block scale and E4M3 element conversion.
//
// Reading of "MXFP8" (Cursor blog summary, "method points"): OCP MX v1.0,
// E4M3 elements, one E8M0 scale per 32 elements, scale byte
// floor(log2(amax)) - 8 + 127 clamped to [0, 254] (0 for an all-zero block),
// elements converted by round-to-nearest-even with saturation to +-448.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp8.h>

namespace moe {

// Scale byte of a block from its absolute maximum. floor(log2(amax)) is the
// unbiased exponent field of the fp32 value; subnormal amax clamps to 0.
__device__ __forceinline__ int mx_scale_byte(float amax) {
  const int e = static_cast<int>((__float_as_uint(amax) >> 23) & 0xFFu) - 127;
  int b = e - 8 + 127;
  b = b < 0 ? 0 : (b > 254 ? 254 : b);
  return amax > 0.0f ? b : 0;
}

// 2^(127 - b) for b in [0, 253] (b <= 246 for any finite fp32 amax).
__device__ __forceinline__ float mx_inv_scale(int b) { return __uint_as_float(static_cast<uint32_t>(254 - b) << 23); }

__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  return static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3));
}

// Quantise 32 values with a common inverse scale into 8 packed words.
__device__ __forceinline__ void mx_pack32(const float* v, float inv, uint32_t* w) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t a = e4m3x2(v[4 * i] * inv, v[4 * i + 1] * inv);
    const uint32_t b = e4m3x2(v[4 * i + 2] * inv, v[4 * i + 3] * inv);
    w[i] = a | (b << 16);
  }
}

// Absolute maximum of 32 values as four interleaved chains of 8 (10
// dependent maxima deep rather than 32, with 4 live temporaries).
__device__ __forceinline__ float amax32(const float* v) {
  float m[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) m[j] = fmaxf(m[j], fabsf(v[4 * i + j]));
  return fmaxf(fmaxf(m[0], m[1]), fmaxf(m[2], m[3]));
}

__device__ __forceinline__ void store32(uint8_t* dst, const uint32_t* w) {
  uint4* p = reinterpret_cast<uint4*>(dst);
  p[0] = make_uint4(w[0], w[1], w[2], w[3]);
  p[1] = make_uint4(w[4], w[5], w[6], w[7]);
}

__device__ __forceinline__ void load_bf16x32(const __nv_bfloat16* src, float* v) {
  const uint4* p = reinterpret_cast<const uint4*>(src);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint4 u = p[q];
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[8 * q + 2 * i] = __uint_as_float(w[i] << 16);
      v[8 * q + 2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&p);
}

// Tiled scale layout offset (see moe_scales_to_tiled in the public header).
__device__ __forceinline__ int64_t sf_off(int64_t r, int64_t kb, int64_t k_tiles) {
  return ((r >> 7) * k_tiles + (kb >> 2)) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4 + (kb & 3);
}

// Scales of one 128-row tile in the tiled atom layout, from row-major scales
// sfr [tokens][d/32]. Lane l covers tile rows l, l+32, l+64, l+96 (tokens
// tok[0..3], -1 for a zero row), whose words of one k-tile form one 16-byte
// chunk of the atom, so a warp writes each atom as 512 contiguous bytes.
// atoms = the tile's first atom + 16 * lane. With d a multiple of 512 each
// row's words of 4 k-tiles are one 16-byte load: the call covers the k-tile
// groups first, first + step, ... (k-tiles first, first + step, ... otherwise),
// so that several warps can share a tile, each with one round of loads.
__device__ __forceinline__ void tile_scales_from_rows(const uint8_t* sfr, const int* tok, int d, uint8_t* atoms,
                                                      int first, int step) {
  const int ktiles = d >> 7;
  const int64_t rowb = d >> 5;
  if ((d & 511) == 0) {
    for (int kc = first; kc < ktiles / 4; kc += step) {
      uint4 v[4];
#pragma unroll
      for (int j = 0; j < 4; ++j)
        v[j] = tok[j] >= 0 ? __ldg(reinterpret_cast<const uint4*>(sfr + tok[j] * rowb) + kc) : make_uint4(0, 0, 0, 0);
      *reinterpret_cast<uint4*>(atoms + (4 * kc + 0) * 512) = make_uint4(v[0].x, v[1].x, v[2].x, v[3].x);
      *reinterpret_cast<uint4*>(atoms + (4 * kc + 1) * 512) = make_uint4(v[0].y, v[1].y, v[2].y, v[3].y);
      *reinterpret_cast<uint4*>(atoms + (4 * kc + 2) * 512) = make_uint4(v[0].z, v[1].z, v[2].z, v[3].z);
      *reinterpret_cast<uint4*>(atoms + (4 * kc + 3) * 512) = make_uint4(v[0].w, v[1].w, v[2].w, v[3].w);
    }
  } else {
    for (int kt = first; kt < ktiles; kt += step) {
      uint32_t w[4];
#pragma unroll
      for (int j = 0; j < 4; ++j)
        w[j] = tok[j] >= 0 ? __ldg(reinterpret_cast<const uint32_t*>(sfr + tok[j] * rowb) + kt) : 0u;
      *reinterpret_cast<uint4*>(atoms + kt * 512) = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
}

// Row-wise MX of 32 values: codes to dst (16-byte aligned), scale byte to sf.
__device__ __forceinline__ void emit_rowq(const float* v, uint8_t* dst, uint8_t* sf_byte) {
  const int b = mx_scale_byte(amax32(v));
  uint32_t w[8];
  mx_pack32(v, mx_inv_scale(b), w);
  store32(dst, w);
  *sf_byte = static_cast<uint8_t>(b);
}

// Token-axis MX of a warp's 32x32 block (lane = row): transposes through
// shared memory so that lane j owns column j, then writes 32 codes of that
// column (32 consecutive ranks) and its scale.
__device__ __forceinline__ void emit_tokq(const float* v, float* scr, int lane, uint8_t* q_tok, uint8_t* q_tok_sf,
                                          int64_t pitch, int64_t col0, int64_t prow_base) {
#pragma unroll
  for (int j = 0; j < 32; ++j) scr[lane * 33 + j] = v[j];
  __syncwarp();
  float c[32];
#pragma unroll
  for (int r = 0; r < 32; ++r) c[r] = scr[r * 33 + lane];
  __syncwarp();
  const int b = mx_scale_byte(amax32(c));
  uint32_t w[8];
  mx_pack32(c, mx_inv_scale(b), w);
  const int64_t col = col0 + lane;
  store32(q_tok + col * pitch + prow_base, w);
  q_tok_sf[sf_off(col, prow_base >> 5, pitch >> 7)] = static_cast<uint8_t>(b);
}

}  // namespace moe
