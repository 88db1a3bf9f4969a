// CPU oracle of the DSV3-style MXFP8 MoE layer in plain C++ -- TEST INFRASTRUCTURE ONLY.
//
// A plain, slow, fp64 statement of what the layer computes, written from the
// Mixture-of-Kittens write-ups (Cursor blog summary, "method points"; techlab
// report, ring-buffer paragraph; mlqm commentary, sections "two scorecards"
// and "deterministic training") and the readings they leave open. Only the
// tests and the CPU-baseline leg of bench.py load it. It shares no code with
// the CUDA library and includes none of its headers; its inputs come from the
// seeded generators (gen/), as plain arrays.
//
// Every floating-point step is IEEE binary64 or binary32 with
// round-to-nearest and no contraction (built with -ffp-contract=off), in the
// order written here; the MX codec and the router's sigmoid are stated from
// their definitions:
//   MXFP8 (OCP MX v1.0 reading): E4M3 elements, one E8M0 scale per 32
//     elements, scale byte floor(log2 amax) - 8 + 127 clamped to [0, 254]
//     (0 for an all-zero block), elements v / 2^(byte-127) rounded to
//     nearest-even and saturated to +-448;
//   router: logits in fp64 sums rounded to fp32; s = sigma(l) by the
//     specified fp32 arithmetic (Cody-Waite reduction, degree-7 Taylor
//     polynomial in Horner form); v = s + bias; groups scored by the sum of
//     their two best v; top-k of kept experts, ties to the lower index, slots
//     by descending v; gates w = s / sum(s) in slot order;
//   schedule: assignments a = t k + j in (t, j) order; stable ranks per
//     expert; positions offsets[e] + rank;
//   expert: GEMM1 on MX(x) rows and MX weights in fp64, saved g, u rounded to
//     bf16, h = fp32(silu(g) u) from the unrounded g, u, MX(h) along I, GEMM2
//     rounded to bf16; the shared expert on every token;
//   combine: y = bf16(sum_j w O_j + S) in fp64;
//   backward: dw = fp32(<dy, O>), the expert dgrad on each token's MX(dy) with
//     the routed row's gate applied to dh, SwiGLU backward on the saved bf16
//     g, u, dGU = fp32, MX(dGU) along 2I, DX = bf16; weight gradients on
//     token-axis MX operands (blocks of 32 consecutive ranks, zero-padded
//     tail): dO = fp32(w dy), h, dGU and x; router backward through the gate
//     normalisation and the sigmoid; dx = bf16(sum_j DX + DX_shared + dx_r).
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <functional>
#include <thread>
#include <vector>

namespace {

// ---------------------------------------------------------------- threads
void parallel_for(int64_t n, int nthreads, const std::function<void(int64_t, int64_t)>& body) {
  if (n <= 0) return;
  int nt = nthreads > 0 ? nthreads : static_cast<int>(std::thread::hardware_concurrency());
  if (nt < 1) nt = 1;
  if (nt > n) nt = static_cast<int>(n);
  if (nt == 1) {
    body(0, n);
    return;
  }
  std::vector<std::thread> th;
  const int64_t chunk = (n + nt - 1) / nt;
  for (int i = 0; i < nt; ++i) {
    const int64_t lo = i * chunk, hi = std::min(n, lo + chunk);
    if (lo < hi) th.emplace_back(body, lo, hi);
  }
  for (auto& t : th) t.join();
}

// ---------------------------------------------------------------- roundings
// bf16, nearest-even: keep 8 significant bits of a = m 2^e, m in [0.5, 1).
double bf16(double a) {
  int e = 0;
  const double m = std::frexp(a, &e);
  return std::ldexp(std::nearbyint(m * 256.0) / 256.0, e);
}
double fp32(double a) { return static_cast<double>(static_cast<float>(a)); }

// ---------------------------------------------------------------- E4M3 / E8M0
double e4m3_decode(uint8_t c) {
  const double sign = (c & 0x80) ? -1.0 : 1.0;
  const int e = (c >> 3) & 0xF, m = c & 7;
  if ((c & 0x7F) == 0x7F) return NAN;
  const double mag = e == 0 ? m * std::ldexp(1.0, -9) : (1.0 + m / 8.0) * std::ldexp(1.0, e - 7);
  return sign * mag;
}

// Nearest E4M3 code (ties to even mantissa), saturating to 448; the sign bit
// follows the sign of v.
uint8_t e4m3_encode(double v) {
  const bool neg = std::signbit(v);
  const double a = std::fabs(v);
  int code;
  if (a < std::ldexp(1.0, -6)) {
    code = static_cast<int>(std::nearbyint(a * 512.0));          // subnormals (8 = 2^-6)
  } else {
    int ex = 0;
    std::frexp(a, &ex);
    int e = ex - 1;                                               // floor(log2 a)
    const double frac = a / std::ldexp(1.0, e);                   // [1, 2), exact
    int qm = static_cast<int>(std::nearbyint((frac - 1.0) * 8.0));
    if (qm == 8) { ++e; qm = 0; }
    code = ((e + 7) << 3) | qm;
    if (code > 0x7E) code = 0x7E;
  }
  return static_cast<uint8_t>(neg ? (code | 0x80) : code);
}

uint8_t scale_byte(double amax) {
  if (!(amax > 0.0)) return 0;
  int ex = 0;
  std::frexp(amax, &ex);
  const int b = (ex - 1) - 8 + 127;
  return static_cast<uint8_t>(b < 0 ? 0 : (b > 254 ? 254 : b));
}

// One block of 32 values (stride apart) -> codes, scale byte; returns the byte.
uint8_t quant_block(const double* v, int64_t stride, uint8_t* codes, int64_t cstride) {
  double amax = 0.0;
  for (int i = 0; i < 32; ++i) amax = std::max(amax, std::fabs(v[i * stride]));
  const uint8_t b = scale_byte(amax);
  const double X = std::ldexp(1.0, static_cast<int>(b) - 127);
  for (int i = 0; i < 32; ++i) codes[i * cstride] = e4m3_encode(v[i * stride] / X);
  return b;
}

// MX along K of a [rows][K] matrix: codes [rows][K], scales [rows][K/32], and
// (optional) the dequantised values [rows][K].
void mx_rows(const double* v, int64_t rows, int64_t K, uint8_t* codes, uint8_t* scales, double* val) {
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t b = 0; b < K / 32; ++b) {
      const int64_t o = r * K + b * 32;
      const uint8_t s = quant_block(v + o, 1, codes + o, 1);
      if (scales) scales[r * (K / 32) + b] = s;
      if (val) {
        const double X = std::ldexp(1.0, static_cast<int>(s) - 127);
        for (int i = 0; i < 32; ++i) val[o + i] = e4m3_decode(codes[o + i]) * X;
      }
    }
}

// Values of MX(v) along K (the operand a GEMM sees); rows split over threads.
std::vector<double> mx_values(const double* v, int64_t rows, int64_t K, int nthreads = 0) {
  std::vector<double> val(rows * K);
  std::vector<uint8_t> codes(rows * K);
  parallel_for(rows, nthreads, [&](int64_t lo, int64_t hi) {
    mx_rows(v + lo * K, hi - lo, K, codes.data() + lo * K, nullptr, val.data() + lo * K);
  });
  return val;
}

// Token-axis MX of rank-ordered rows [n][K]: column c, blocks of 32
// consecutive ranks, ranks past n are zero. Returns the values transposed,
// [K][n_pad].
std::vector<double> mx_tokens(const double* rows, int64_t n, int64_t K, int64_t* n_pad_out) {
  const int64_t n_pad = (n + 31) / 32 * 32;
  std::vector<double> col(n_pad), val(K * n_pad);
  std::vector<uint8_t> codes(32);
  for (int64_t c = 0; c < K; ++c) {
    for (int64_t r = 0; r < n_pad; ++r) col[r] = r < n ? rows[r * K + c] : 0.0;
    for (int64_t b = 0; b < n_pad / 32; ++b) {
      const uint8_t s = quant_block(col.data() + b * 32, 1, codes.data(), 1);
      const double X = std::ldexp(1.0, static_cast<int>(s) - 127);
      for (int i = 0; i < 32; ++i) val[c * n_pad + b * 32 + i] = e4m3_decode(codes[i]) * X;
    }
  }
  *n_pad_out = n_pad;
  return val;
}

// ---------------------------------------------------------------- sigmoid (fp32, specified)
float exp_spec(float z) {
  const float log2e = static_cast<float>(1.0 / std::log(2.0));
  const float c1 = static_cast<float>(std::nearbyint(std::log(2.0) * 512.0) / 512.0);   // 355/512
  const float c2 = static_cast<float>(std::log(2.0) - static_cast<double>(c1));
  float coef[8];
  double f = 1.0;
  for (int i = 0; i < 8; ++i) {
    if (i > 0) f *= i;
    coef[i] = static_cast<float>(1.0 / f);
  }
  const float n = std::nearbyint(z * log2e);
  const float r = (z - n * c1) - n * c2;
  float p = coef[7];
  for (int i = 6; i >= 0; --i) p = p * r + coef[i];
  uint32_t bits = static_cast<uint32_t>(static_cast<int32_t>(n) + 127) << 23;
  float two_n;
  std::memcpy(&two_n, &bits, 4);
  return p * two_n;
}

float sigmoid_spec(float l) {
  const float lc = std::min(std::max(l, -80.0f), 80.0f);
  return 1.0f / (1.0f + exp_spec(-lc));
}

// (v1, e1) ranks before (v2, e2): larger value, ties to the lower index.
bool better(float v1, int e1, float v2, int e2) { return v1 > v2 || (v1 == v2 && e1 < e2); }

// ---------------------------------------------------------------- GEMM (fp64, K-major operands)
// C[i][j] = sum_k A[i][k] B[j][k], rows of C split over threads.
void gemm_nt(const double* A, const double* B, int64_t M, int64_t N, int64_t K, double* C, int nthreads) {
  parallel_for(M, nthreads, [&](int64_t lo, int64_t hi) {
    for (int64_t i = lo; i < hi; ++i)
      for (int64_t j = 0; j < N; ++j) {
        double s = 0.0;
        const double* a = A + i * K;
        const double* b = B + j * K;
        for (int64_t k = 0; k < K; ++k) s += a[k] * b[k];
        C[i * N + j] = s;
      }
  });
}

std::vector<double> transpose(const double* a, int64_t rows, int64_t cols) {
  std::vector<double> t(rows * cols);
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t c = 0; c < cols; ++c) t[c * rows + r] = a[r * cols + c];
  return t;
}

double silu(double g) { return g / (1.0 + std::exp(-g)); }

// ---------------------------------------------------------------- NVFP4
// E2M1 magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6: the nearest (ties to the even
// code), saturating at 6; the sign bit follows the sign of v.
uint8_t e2m1_encode(double v) {
  static const double mag[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};
  const double a = std::min(std::fabs(v), 6.0);
  int best = 0;
  for (int c = 1; c < 8; ++c) {
    const double dc = std::fabs(a - mag[c]), db = std::fabs(a - mag[best]);
    if (dc < db || (dc == db && (c & 1) == 0)) best = c;
  }
  return static_cast<uint8_t>(best | (std::signbit(v) ? 8 : 0));
}

}  // namespace

extern "C" {

// NVFP4 along K of fp32 v [rows][K] (K a multiple of 16) with tensor scale g:
// codes [rows][K] (one 4-bit code per byte), E4M3 block scales [rows][K/16].
//   denom = fp32(6 g); sb = E4M3(fp32(amax / denom)); X = fp32(decode(sb) g);
//   q = E2M1(fp32(v / X)), or 0 when X = 0.
void orc_nvfp4_quantize(const float* v, int64_t rows, int64_t K, float g, uint8_t* codes, uint8_t* scales) {
  const float denom = 6.0f * g;
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t b = 0; b < K / 16; ++b) {
      const float* blk = v + r * K + b * 16;
      float amax = 0.0f;
      for (int i = 0; i < 16; ++i) amax = std::max(amax, std::fabs(blk[i]));
      const uint8_t sb = e4m3_encode(static_cast<double>(amax / denom));
      scales[r * (K / 16) + b] = sb;
      const float X = static_cast<float>(e4m3_decode(sb)) * g;
      for (int i = 0; i < 16; ++i)
        codes[r * K + b * 16 + i] = X > 0.0f ? e2m1_encode(static_cast<double>(blk[i] / X)) : 0;
    }
}
void orc_e2m1_encode(const double* v, int64_t n, uint8_t* codes) {
  for (int64_t i = 0; i < n; ++i) codes[i] = e2m1_encode(v[i]);
}

// ---------------------------------------------------------------- codec and router pieces (pins)
void orc_e4m3_encode(const double* v, int64_t n, uint8_t* codes) {
  for (int64_t i = 0; i < n; ++i) codes[i] = e4m3_encode(v[i]);
}
void orc_e4m3_decode(const uint8_t* c, int64_t n, double* v) {
  for (int64_t i = 0; i < n; ++i) v[i] = e4m3_decode(c[i]);
}
void orc_scale_byte(const double* amax, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = scale_byte(amax[i]);
}
// MX along K of [rows][K] (K a multiple of 32): codes, scales, values.
void orc_mx_quantize(const double* v, int64_t rows, int64_t K, uint8_t* codes, uint8_t* scales, double* val) {
  mx_rows(v, rows, K, codes, scales, val);
}
// Token-axis MX of rows [n][K]: column c, blocks of 32 consecutive ranks,
// zero past n. Codes [K][n_pad], scales [K][n_pad/32], n_pad = ceil32(n).
void orc_mx_quantize_tokens(const double* rows, int64_t n, int64_t K, uint8_t* codes, uint8_t* scales) {
  const int64_t n_pad = (n + 31) / 32 * 32;
  std::vector<double> col(n_pad);
  for (int64_t c = 0; c < K; ++c) {
    for (int64_t r = 0; r < n_pad; ++r) col[r] = r < n ? rows[r * K + c] : 0.0;
    for (int64_t b = 0; b < n_pad / 32; ++b)
      scales[c * (n_pad / 32) + b] = quant_block(col.data() + b * 32, 1, codes + c * n_pad + b * 32, 1);
  }
}
void orc_exp_spec(const float* z, int64_t n, float* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = exp_spec(z[i]);
}
void orc_sigmoid_spec(const float* l, int64_t n, float* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = sigmoid_spec(l[i]);
}

// logits[t][e] = fp32(sum_c x[t][c] wr[e][c]) (fp64 sum in c order).
void orc_router_logits(const double* x, const double* wr, int T, int d, int E, float* logits, int nthreads) {
  parallel_for(T, nthreads, [&](int64_t lo, int64_t hi) {
    for (int64_t t = lo; t < hi; ++t)
      for (int e = 0; e < E; ++e) {
        double s = 0.0;
        for (int c = 0; c < d; ++c) s += x[t * d + c] * wr[static_cast<int64_t>(e) * d + c];
        logits[t * E + e] = static_cast<float>(s);
      }
  });
}

// Selection of every token from its fp32 logits (see the header comment).
void orc_select(const float* logits, const float* bias, int T, int E, int k, int G, int gtop, int32_t* idx, float* w,
                float* ssel) {
  std::vector<float> s(E), v(E);
  std::vector<char> allowed(E), taken(E);
  for (int64_t t = 0; t < T; ++t) {
    for (int e = 0; e < E; ++e) {
      s[e] = sigmoid_spec(logits[t * E + e]);
      v[e] = s[e] + bias[e];
    }
    std::fill(allowed.begin(), allowed.end(), 1);
    if (G > 1) {
      const int per = E / G;
      std::vector<float> gs(G);
      for (int g = 0; g < G; ++g) {
        float m1 = -INFINITY, m2 = -INFINITY;
        for (int e = g * per; e < (g + 1) * per; ++e) {
          if (v[e] > m1) { m2 = m1; m1 = v[e]; } else if (v[e] > m2) { m2 = v[e]; }
        }
        gs[g] = m1 + m2;
      }
      std::vector<char> kept(G, 0);
      for (int r = 0; r < gtop; ++r) {
        int bg = -1;
        for (int g = 0; g < G; ++g)
          if (!kept[g] && (bg < 0 || better(gs[g], g, gs[bg], bg))) bg = g;
        kept[bg] = 1;
      }
      for (int e = 0; e < E; ++e) allowed[e] = kept[e / per];
    }
    std::fill(taken.begin(), taken.end(), 0);
    float tot = 0.0f;
    for (int j = 0; j < k; ++j) {
      int be = -1;
      for (int e = 0; e < E; ++e)
        if (allowed[e] && !taken[e] && (be < 0 || better(v[e], e, v[be], be))) be = e;
      taken[be] = 1;
      idx[t * k + j] = be;
      ssel[t * k + j] = s[be];
      tot = j == 0 ? s[be] : tot + s[be];
    }
    for (int j = 0; j < k; ++j) w[t * k + j] = ssel[t * k + j] / tot;
  }
}

// Counts, exclusive offsets (E + 1), stable ranks, positions and their inverse.
void orc_schedule(const int32_t* idx, int64_t A, int E, int64_t* counts, int64_t* offsets, int64_t* rank,
                  int64_t* pos, int64_t* inv) {
  for (int e = 0; e < E; ++e) counts[e] = 0;
  for (int64_t a = 0; a < A; ++a) rank[a] = counts[idx[a]]++;
  offsets[0] = 0;
  for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
  for (int64_t a = 0; a < A; ++a) {
    pos[a] = offsets[idx[a]] + rank[a];
    inv[pos[a]] = a;
  }
}

// One expert's weights in the four MX orientations the layer uses (values):
//   W1 [2I][d] along d (GEMM1), W2 [d][I] along I (GEMM2),
//   W2b = W_d^T [I][d] along d (dgrad of GEMM2), W1b = W_gu^T [d][2I] along 2I
//   (dgrad of GEMM1). w_gu [2I][d] (gate rows, then up rows), w_d [d][I].
void orc_expert_weights(const double* w_gu, const double* w_d, int d, int I, int nthreads, double* W1, double* W2,
                        double* W2b, double* W1b) {
  const int64_t I2 = 2LL * I;
  std::vector<double> v = mx_values(w_gu, I2, d, nthreads);
  std::memcpy(W1, v.data(), sizeof(double) * v.size());
  v = mx_values(w_d, d, I, nthreads);
  std::memcpy(W2, v.data(), sizeof(double) * v.size());
  const std::vector<double> wdT = transpose(w_d, d, I);
  v = mx_values(wdT.data(), I, d, nthreads);
  std::memcpy(W2b, v.data(), sizeof(double) * v.size());
  const std::vector<double> wguT = transpose(w_gu, I2, d);
  v = mx_values(wguT.data(), d, I2, nthreads);
  std::memcpy(W1b, v.data(), sizeof(double) * v.size());
}

// One expert's forward and backward on its rows in rank order, on weights
// from orc_expert_weights.
//   x_rows, dy_rows [n][d]: the rows' tokens' x and dy (bf16 values);
//   gate [n]: the routed rows' gates (fp32), or null for the shared expert.
// Outputs: O [n][d] and DX [n][d] (bf16 values), dW_gu [2I][d] and
// dW_d [d][I] (bf16 values).
void orc_expert_q(const double* x_rows, const double* dy_rows, const float* gate, int64_t n, int d, int I,
                  const double* W1, const double* W2, const double* W2b, const double* W1b, int nthreads, double* O,
                  double* DX, double* dW_gu, double* dW_d) {
  const int64_t I2 = 2LL * I;
  if (n == 0) {
    std::fill(dW_gu, dW_gu + I2 * d, 0.0);
    std::fill(dW_d, dW_d + static_cast<int64_t>(d) * I, 0.0);
    return;
  }
  // forward
  const std::vector<double> xq = mx_values(x_rows, n, d, nthreads);
  std::vector<double> gu(n * I2), h(n * I), gus(n * I2);
  gemm_nt(xq.data(), W1, n, I2, d, gu.data(), nthreads);
  for (int64_t r = 0; r < n; ++r)
    for (int64_t i = 0; i < I; ++i) {
      const double g = gu[r * I2 + i], u = gu[r * I2 + I + i];
      h[r * I + i] = fp32(silu(g) * u);
      gus[r * I2 + i] = bf16(g);
      gus[r * I2 + I + i] = bf16(u);
    }
  const std::vector<double> hq = mx_values(h.data(), n, I, nthreads);
  gemm_nt(hq.data(), W2, n, d, I, O, nthreads);
  for (int64_t i = 0; i < n * d; ++i) O[i] = bf16(O[i]);
  // backward: dh = gate * (MX(dy) . W_d) along d, SwiGLU backward on the saved bf16 g, u
  const std::vector<double> dyq = mx_values(dy_rows, n, d, nthreads);
  std::vector<double> dh(n * I), dgu(n * I2);
  gemm_nt(dyq.data(), W2b, n, I, d, dh.data(), nthreads);
  for (int64_t r = 0; r < n; ++r) {
    const double gw = gate ? static_cast<double>(gate[r]) : 1.0;
    for (int64_t i = 0; i < I; ++i) {
      const double dhv = dh[r * I + i] * gw;
      const double g = gus[r * I2 + i], u = gus[r * I2 + I + i];
      const double sg = 1.0 / (1.0 + std::exp(-g));
      dgu[r * I2 + i] = fp32(dhv * u * sg * (1.0 + g * (1.0 - sg)));
      dgu[r * I2 + I + i] = fp32(dhv * (g * sg));
    }
  }
  const std::vector<double> dguq = mx_values(dgu.data(), n, I2, nthreads);
  gemm_nt(dguq.data(), W1b, n, d, I2, DX, nthreads);
  for (int64_t i = 0; i < n * d; ++i) DX[i] = bf16(DX[i]);
  // weight gradients on token-axis MX operands
  std::vector<double> dO(n * d);
  for (int64_t r = 0; r < n; ++r) {
    const float gw = gate ? gate[r] : 1.0f;
    for (int64_t c = 0; c < d; ++c)
      dO[r * d + c] = static_cast<double>(gw * static_cast<float>(dy_rows[r * d + c]));
  }
  int64_t np = 0;
  const std::vector<double> dO_t = mx_tokens(dO.data(), n, d, &np);      // [d][np]
  const std::vector<double> h_t = mx_tokens(h.data(), n, I, &np);        // [I][np]
  const std::vector<double> dgu_t = mx_tokens(dgu.data(), n, I2, &np);   // [2I][np]
  const std::vector<double> x_t = mx_tokens(x_rows, n, d, &np);          // [d][np]
  gemm_nt(dO_t.data(), h_t.data(), d, I, np, dW_d, nthreads);
  gemm_nt(dgu_t.data(), x_t.data(), I2, d, np, dW_gu, nthreads);
  for (int64_t i = 0; i < static_cast<int64_t>(d) * I; ++i) dW_d[i] = bf16(dW_d[i]);
  for (int64_t i = 0; i < I2 * d; ++i) dW_gu[i] = bf16(dW_gu[i]);
}

// orc_expert_weights followed by orc_expert_q, from bf16 master weights.
void orc_expert(const double* x_rows, const double* dy_rows, const float* gate, int64_t n, int d, int I,
                const double* w_gu, const double* w_d, int nthreads, double* O, double* DX, double* dW_gu,
                double* dW_d) {
  const int64_t I2 = 2LL * I;
  std::vector<double> W1(I2 * d), W2(static_cast<int64_t>(d) * I), W2b(static_cast<int64_t>(I) * d),
      W1b(static_cast<int64_t>(d) * I2);
  orc_expert_weights(w_gu, w_d, d, I, nthreads, W1.data(), W2.data(), W2b.data(), W1b.data());
  orc_expert_q(x_rows, dy_rows, gate, n, d, I, W1.data(), W2.data(), W2b.data(), W1b.data(), nthreads, O, DX, dW_gu,
               dW_d);
}

// y[t] = bf16(sum_j w[t][j] O[t][j] + S[t]) (fp64, j in slot order); S may be null.
void orc_combine(const float* w, const double* O, const double* S, int T, int k, int d, double* y) {
  for (int64_t t = 0; t < T; ++t)
    for (int64_t c = 0; c < d; ++c) {
      double s = 0.0;
      for (int j = 0; j < k; ++j) s += static_cast<double>(w[t * k + j]) * O[(t * k + j) * d + c];
      if (S) s += S[t * d + c];
      y[t * d + c] = bf16(s);
    }
}

// Router backward: dw [T][k] gate gradients (fp32 values), w and ssel (fp32),
// x [T][d], wr [E][d]. dl = ((dw - sum_i dw_i w_i) / sum(ssel)) s (1 - s) on
// the selected experts; dx_r[t] = sum_j dl_j wr[idx_j]; dWr[e] = sum over the
// assignments to e of dl x[t] (fp64, unrounded). The bias gets no gradient.
void orc_router_backward(const double* dw, const float* w, const float* ssel, const int32_t* idx, const double* x,
                         const double* wr, int T, int k, int d, int E, double* dl, double* dx_r, double* dWr) {
  std::fill(dWr, dWr + static_cast<int64_t>(E) * d, 0.0);
  for (int64_t t = 0; t < T; ++t) {
    double Z = 0.0, dot = 0.0;
    for (int j = 0; j < k; ++j) {
      Z += ssel[t * k + j];
      dot += dw[t * k + j] * w[t * k + j];
    }
    for (int j = 0; j < k; ++j) {
      const double s = ssel[t * k + j];
      dl[t * k + j] = (dw[t * k + j] - dot) / Z * s * (1.0 - s);
    }
    for (int64_t c = 0; c < d; ++c) {
      double acc = 0.0;
      for (int j = 0; j < k; ++j) acc += dl[t * k + j] * wr[static_cast<int64_t>(idx[t * k + j]) * d + c];
      dx_r[t * d + c] = acc;
    }
    for (int j = 0; j < k; ++j) {
      double* row = dWr + static_cast<int64_t>(idx[t * k + j]) * d;
      for (int64_t c = 0; c < d; ++c) row[c] += dl[t * k + j] * x[t * d + c];
    }
  }
}

// The whole layer, forward and backward.
//   x [T][d], dy [T][d], w_router [E][d], w_gu [E][2I][d], w_d [E][d][I],
//   ws_gu [S][2I][d], ws_d [S][d][I]: bf16 values; bias [E] fp32.
//   logits_in: fp32 [T][E] to select from instead of computing them (null =
//   compute them here).
// Outputs: idx, w [T][k]; logits [T][E]; y, dx [T][d]; dW_gu, dW_d, dWs_gu,
// dWs_d, dW_r [E][d] (bf16 values).
void orc_layer(int T, int d, int E, int k, int G, int gtop, int I, int S, const double* x, const double* w_router,
               const float* bias, const double* w_gu, const double* w_d, const double* ws_gu, const double* ws_d,
               const double* dy, const float* logits_in, int nthreads, int32_t* idx, float* w, float* logits,
               double* y, double* dx, double* dW_gu, double* dW_d, double* dWs_gu, double* dWs_d, double* dW_r) {
  const int64_t A = static_cast<int64_t>(T) * k, I2 = 2LL * I;
  if (logits_in)
    std::memcpy(logits, logits_in, sizeof(float) * T * E);
  else
    orc_router_logits(x, w_router, T, d, E, logits, nthreads);
  std::vector<float> ssel(A);
  orc_select(logits, bias, T, E, k, G, gtop, idx, w, ssel.data());
  std::vector<int64_t> counts(E), offsets(E + 1), rank(A), pos(A), inv(A);
  orc_schedule(idx, A, E, counts.data(), offsets.data(), rank.data(), pos.data(), inv.data());
  std::vector<double> O(A * d, 0.0), DX(A * d, 0.0), S_out(static_cast<int64_t>(T) * d, 0.0),
      DXs(static_cast<int64_t>(T) * d, 0.0);
  for (int e = 0; e < E; ++e) {
    const int64_t n = counts[e];
    std::vector<double> xr(n * d), dyr(n * d), Oe(n * d), DXe(n * d);
    std::vector<float> ge(n);
    for (int64_t r = 0; r < n; ++r) {
      const int64_t a = inv[offsets[e] + r], t = a / k;
      std::memcpy(&xr[r * d], x + t * d, sizeof(double) * d);
      std::memcpy(&dyr[r * d], dy + t * d, sizeof(double) * d);
      ge[r] = w[a];
    }
    orc_expert(xr.data(), dyr.data(), ge.data(), n, d, I, w_gu + static_cast<int64_t>(e) * I2 * d,
               w_d + static_cast<int64_t>(e) * d * I, nthreads, Oe.data(), DXe.data(),
               dW_gu + static_cast<int64_t>(e) * I2 * d, dW_d + static_cast<int64_t>(e) * d * I);
    for (int64_t r = 0; r < n; ++r) {
      const int64_t a = inv[offsets[e] + r];
      std::memcpy(&O[a * d], &Oe[r * d], sizeof(double) * d);
      std::memcpy(&DX[a * d], &DXe[r * d], sizeof(double) * d);
    }
  }
  for (int s = 0; s < S; ++s) {
    std::vector<double> Os(static_cast<int64_t>(T) * d), DXo(static_cast<int64_t>(T) * d);
    orc_expert(x, dy, nullptr, T, d, I, ws_gu + static_cast<int64_t>(s) * I2 * d,
               ws_d + static_cast<int64_t>(s) * d * I, nthreads, Os.data(), DXo.data(),
               dWs_gu + static_cast<int64_t>(s) * I2 * d, dWs_d + static_cast<int64_t>(s) * d * I);
    for (int64_t i = 0; i < static_cast<int64_t>(T) * d; ++i) {
      S_out[i] += Os[i];
      DXs[i] += DXo[i];
    }
  }
  orc_combine(w, O.data(), S > 0 ? S_out.data() : nullptr, T, k, d, y);
  // backward
  std::vector<double> dwv(A), dl(A), dxr(static_cast<int64_t>(T) * d);
  for (int64_t a = 0; a < A; ++a) {
    const int64_t t = a / k;
    double s = 0.0;
    for (int64_t c = 0; c < d; ++c) s += dy[t * d + c] * O[a * d + c];
    dwv[a] = fp32(s);
  }
  orc_router_backward(dwv.data(), w, ssel.data(), idx, x, w_router, T, k, d, E, dl.data(), dxr.data(), dW_r);
  for (int64_t i = 0; i < static_cast<int64_t>(E) * d; ++i) dW_r[i] = bf16(dW_r[i]);
  for (int64_t t = 0; t < T; ++t)
    for (int64_t c = 0; c < d; ++c) {
      double s = 0.0;
      for (int j = 0; j < k; ++j) s += DX[(t * k + j) * d + c];
      s += DXs[t * d + c] + dxr[t * d + c];
      dx[t * d + c] = bf16(s);
    }
}

}  // extern "C"
