// Internal host-side declarations: workspace layout and kernel launchers.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/moe.h"

namespace moe {

constexpr int kTileM = 128;     // rows per GEMM tile / scale atom
constexpr int kTileK = 128;     // fp8 elements per K stage (one 128-byte swizzle row)
constexpr int kSchedUnit = 256; // assignments per schedule unit (one warp)
constexpr int kRingBufs = 2;    // ring token buffers; lap L uses buffer L % kRingBufs
// Tile width of the GEMM1 (gate|up) kernel. Its weight rows are interleaved
// in blocks of kGemm1BN / 2 gate rows followed by the matching up rows, so a
// tile holds matching g and u columns.
constexpr int kGemm1BN = 256;
constexpr int kGuBlock = kGemm1BN / 2;
// Output rows of a CTA-pair GEMM tile (gemm_pair.cuh).
constexpr int kPairRows = 256;

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline int64_t round_up(int64_t a, int64_t b) { return ceil_div(a, b) * b; }

// Byte offset of scale byte (row r, 32-block kb) in the MMA-ready tiled scale
// layout of a [R][K] MX operand: 512-byte atoms of 128 rows x 4 blocks,
// atoms ordered (row tile, k tile), inside an atom (r%32)*16 + (r/32%4)*4 + kb%4.
__host__ __device__ inline int64_t sf_tiled_offset(int64_t r, int64_t kb, int64_t k_tiles) {
  return ((r >> 7) * k_tiles + (kb >> 2)) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4 + (kb & 3);
}

struct Dims {
  int T, d, E, k, G, gtop, I, S, C;
  int Ep;          // routed + shared experts
  int kp;          // routed + shared slots per token
  int64_t A;       // routed assignments T*k
  int64_t Ap;      // all assignments T*(k+S)
  int64_t Tpad;    // ceil128(T)
  int64_t Rmax;    // padded-row capacity of rank-ordered buffers
  int Lb;          // upper bound on ring laps: ceil(T / C)
  int units;       // schedule units
  int MV;          // mover warps per CTA of the all-laps ring GEMMs (1, 2 or 4)
};

struct Layout {
  Dims m;
  size_t off[MOE_WS_COUNT];
  size_t bytes[MOE_WS_COUNT];
  size_t total;
};

struct WLayout {
  size_t off[MOE_WQ_COUNT];
  size_t bytes[MOE_WQ_COUNT];
  size_t total;
};

// Upper bound on the m-tiles of all ring laps together: sum over experts of
// (ceil(n_e / 128) + laps_e) <= Rmax / 128 + Ep * Lb.
inline int64_t lap_mtiles_max(const Dims& m) { return m.Rmax / 128 + static_cast<int64_t>(m.Ep) * (m.Lb > 0 ? m.Lb : 1); }

int validate(const moe_config_t* cfg);
Dims make_dims(const moe_config_t* cfg);
Layout make_layout(const moe_config_t* cfg);
WLayout make_wlayout(const moe_config_t* cfg);

template <typename T>
inline T* ws_ptr(const Layout& L, void* ws, int which) {
  return reinterpret_cast<T*>(static_cast<char*>(ws) + L.off[which]);
}
template <typename T>
inline T* wq_ptr(const WLayout& L, void* wq, int which) {
  return reinterpret_cast<T*>(static_cast<char*>(wq) + L.off[which]);
}

// Per-device caches are indexed by the device ordinal, below this bound.
constexpr int kMaxDev = 64;
// Current device ordinal, or -1 when it cannot be read or is past kMaxDev.
int current_device();
// SM count of the current device (cached per device).
int num_sms();
// Current device is compute capability 10.3 (GB300) (cached per device).
bool arch_ok();

// ---------------------------------------------------------------- call errors
// An entry point collects the return codes of its own kernel launches and
// stream operations in a slot of the calling host thread, so its result
// reflects only those calls: an error that other code left in the CUDA
// runtime's last-error state is neither read nor cleared by the library.
cudaError_t& call_error();
inline void note(cudaError_t e) {
  if (e != cudaSuccess && call_error() == cudaSuccess) call_error() = e;
}
// Opened at the top of an entry point: clears the slot; status() reads it.
struct CallScope {
  CallScope() { call_error() = cudaSuccess; }
  int status() const { return call_error() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }
};

// ---------------------------------------------------------------- quantisers
// Row-wise MX quantisation of bf16 src[rows][K] (row pitch ld elements).
// Output row r goes to row out_row(r) = (interleave ? gate/up interleave : r).
// Scales canonical [rows][K/32] (sf_k_tiles == 0) or tiled with K/128 k-tiles.
// sf_rows (optional): also write the scales row-major [rows][K/32].
void launch_quant_rows(const void* src, int64_t rows, int K, int64_t ld, uint8_t* codes, uint8_t* sf, bool tiled,
                       int interleave_I, cudaStream_t s, uint8_t* sf_rows = nullptr);
// Column-wise (token-axis) MX quantisation: src[rows][K] bf16 -> codes[K][rows_pad], blocks of 32 rows.
// `batch` equally shaped matrices laid out back to back (grid z).
void launch_quant_cols(const void* src, int64_t rows, int K, int64_t ld, int64_t rows_pad, uint8_t* codes,
                       uint8_t* sf, bool tiled, int batch, cudaStream_t s);

// NVFP4 quantisation of bf16 src[rows][K] along K with tensor scale g: packed
// E2M1 codes [rows][K/2] (element 2i in the low nibble), E4M3 block scales
// (16 elements) canonical [rows][K/16] or, when tiled, in the 512-byte atoms
// of 128 rows x 4 blocks the tensor cores read.
void launch_quant_nvfp4(const void* src, int64_t rows, int K, float g, uint8_t* codes, uint8_t* sf, bool tiled,
                        cudaStream_t s);

// ---------------------------------------------------------------- router
// Returns an MOE_* code: host-side failures (tensor-map encoding, launch
// attributes) come back here, since they launch nothing.
int launch_router_logits(const Dims& m, const void* x, const void* w_router, float* logits, cudaStream_t s);
void launch_router_topk(const Dims& m, const float* logits, const float* bias, int32_t* idx, float* w,
                        float* s_sel, cudaStream_t s);

// ---------------------------------------------------------------- schedule
void launch_schedule(const Dims& m, const int32_t* idx, const Layout& L, void* ws, cudaStream_t s);

// ---------------------------------------------------------------- data movement
void launch_permute_lap(const Dims& m, int lap, bool dO, const Layout& L, void* ws, cudaStream_t s);
// Every lap of the ring dispatch in one launch (same writes, same per-slot lap order).
void launch_dispatch_all(const Dims& m, const Layout& L, void* ws, cudaStream_t s);
void launch_combine(const Dims& m, const float* topk_w, const Layout& L, void* ws, void* y, cudaStream_t s);
void launch_rev_combine_dw(const Dims& m, const void* dy, const float* topk_w, const Layout& L, void* ws,
                           cudaStream_t s);
// SwiGLU backward of the padded rank rows and MX of dGU = [dg | du] two ways
// (along 2I per row, and along ranks per column).
void launch_swiglu_bwd_quant(const Dims& m, const Layout& L, void* ws, cudaStream_t s);
void launch_tok_gather(const Dims& m, const void* src_rows, bool scale_by_gate, const float* topk_w,
                       bool router_partials, const Layout& L, void* ws, uint8_t* codes, uint8_t* sf,
                       cudaStream_t s);
void launch_reverse_dispatch(const Dims& m, const int32_t* idx, const void* w_router, const Layout& L, void* ws,
                             void* dx, cudaStream_t s);
void launch_router_dwr(const Dims& m, const Layout& L, void* ws, void* dw_router, cudaStream_t s);

// ---------------------------------------------------------------- GEMM
enum GemmMode : int {
  kSwigluFwd = 0,   // lap tiles, A = ring / x_q, epilogue SwiGLU + MX(h) two ways + saved g,u
  kPush = 1,        // padded tiles, epilogue bf16 rows pushed to their assignment
  kSwigluBwd = 2,   // lap tiles, A = ring of MX(dy) rows / MX(dy) in place, epilogue fp32 dh rows times the gate
  kWgrad = 3,       // per-expert K ranges, epilogue bf16 weight gradient
  kPlain = 4,       // single dense problem, fp32 output (unit test entry)
  // 5 is the bf16 router-logit mode (gemm.cuh)
  kSwigluFwdRing = 6,  // kSwigluFwd over all ring laps in one launch, mover warps fill the ring
  kSwigluBwdRing = 7,  // kSwigluBwd over all ring laps in one launch, mover warps fill the dO ring
  kPlainNv4 = 8,       // single dense NVFP4 problem (E2M1, E4M3 scale per 16), fp32 output times alpha
  kGroupedNv4 = 9,     // NVFP4 expert GEMM over the schedule's padded rank rows, fp32 rank-ordered rows times alpha
  kPushNv4 = 10,       // the same NVFP4 expert GEMM with the kPush epilogue: bf16 rows times alpha to their assignment
};

// Where the mover warps of the all-laps ring modes take each ring row from.
struct RingMovers {
  const int* lapbase;            // [Lb+1] first global m-tile of each lap
  const int4* ring_info;         // per walk position: the decoded m-tile (two int4, see MOE_WS_RINGINFO);
                                 // CTAs walk tiles and move items in position order
  int* moved;                    // per global m-tile: 8-row groups written (target 16)
  int* consumed;                 // per global m-tile: GEMM tiles whose accumulators completed (target N / BN)
  const uint8_t* xq; const uint8_t* xq_sf;   // MX rows along d (x forward, dy backward), tiled scales
  const uint8_t* xq_sfr;                     // the same scales row-major [T][d/32]
  uint8_t* ring; uint8_t* ring_sf;           // [kRingBufs][E][C] rows, tiled scales
};

struct GemmOperands {
  const uint8_t* a;  int64_t a_rows; int a_cols; const uint8_t* a_sf;
  const uint8_t* a2; int64_t a2_rows; const uint8_t* a2_sf;   // identity-ordered A for shared experts
  const uint8_t* b;  int64_t b_rows; int b_cols; const uint8_t* b_sf;
};

struct GemmEpilogue {
  void* out;            // bf16 rows (push / wgrad) or fp32 (plain)
  void* out2;           // second output (shared-expert wgrad)
  uint8_t* q_rows; uint8_t* q_rows_sf; int q_rows_ktiles;     // MX along the N axis
  uint8_t* q_tok;  uint8_t* q_tok_sf;  int64_t q_tok_pitch;   // MX along tokens (transposed)
  void* gu;             // saved bf16 g|u rows
  const float* gate;    // dh epilogue: per-assignment gate that scales each routed row
  int ldo;              // output row pitch (elements)
  float alpha = 1.0f;   // NVFP4 plain mode: scale of the fp32 product
};

int gemm_dispatch(const char* name, int mode, const Dims& m, int lap, int N, int K, int M, const GemmOperands& op,
                  const GemmEpilogue& ep, const int* counts, const int* poff, const int* lap_tiles,
                  const int* row_src, int* status, cudaStream_t s, int bn_hint = 0, const int* order = nullptr,
                  const RingMovers* mv = nullptr, const void* tile_info = nullptr);

// The weight-gradient (kWgrad) or plain (kPlain, fp32 out) GEMM on CTA pairs:
// 256 x 128 output tiles, tcgen05 MMAs issued for both SMs of a cluster of two
// (gemm_pair.cuh). M a multiple of 256, N of 128; operands as for gemm_dispatch.
int gemm_pair_dispatch(const char* name, int mode, const Dims& m, int N, int M, int K, const GemmOperands& op,
                       const GemmEpilogue& ep, const int* poff, const int* order, int* status, cudaStream_t s);

}  // namespace moe
