/*
 * moe.h -- C ABI of the GB300 (sm_103a) DSV3-style MXFP8 MoE layer.
 *
 * The layer is the one the Mixture-of-Kittens write-ups describe: a
 * DeepSeek-V3-style MoE layer trained in MXFP8 (Cursor blog summary, "method
 * points"), whose forward pass dispatches tokens to experts, runs the expert
 * FFNs and combines the results, and whose backward pass runs reverse-combine
 * and reverse-dispatch on the forward schedule (same section, bullet on
 * communication direction). On one GPU, dispatch is a schedule-driven gather
 * into fixed-capacity ring token buffers and combine a fixed-order weighted
 * sum (techlab report, section on ring buffers; mlqm commentary, section
 * "signalling cut to 18 us").
 *
 * Conventions for every entry point
 *   - Pointers named in the signature are DEVICE pointers unless stated.
 *     bf16 tensors are row-major, dense (row pitch = row length). Tensor,
 *     weight, gradient and workspace buffers must start on a 16-byte boundary
 *     (MOE_ERR_INVALID_ARG otherwise); topk_idx, topk_w and bias only need
 *     their element alignment.
 *   - The caller allocates and frees every buffer, including the workspace
 *     (moe_workspace_size) and the quantised-weight blob (moe_weights_size).
 *     The library never allocates device memory and never synchronises the
 *     stream, except moe_status, which reads one device word.
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and runs asynchronously.
 *   - Return value: MOE_OK, or an MOE_ERR_* code for argument, architecture
 *     or launch errors, in which case nothing further was enqueued.
 *     MOE_ERR_CUDA reflects the entry point's own launches and stream
 *     operations only: an error that other code left in the CUDA runtime's
 *     last-error state is neither reported nor cleared.
 *     Device-side failures (a bounded wait that ran out, a bounds check)
 *     are recorded in a status word in the workspace; read it with
 *     moe_status after synchronising.
 *   - Streams: moe_forward (with MOE_FLAG_LAP_LAUNCHES) and moe_backward fork
 *     part of their work onto an auxiliary stream and join it back before
 *     returning. The library creates one auxiliary stream per (device,
 *     caller stream) on first use and keeps it until the process exits, so
 *     layers driven from different streams do not wait on each other.
 *   - Results are bitwise deterministic: no floating-point atomics, every
 *     reduction has a fixed order.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

typedef void* moe_stream_t; /* cudaStream_t */

enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,     /* bad shape, null pointer, misaligned pointer */
  MOE_ERR_UNSUPPORTED_ARCH = 2,/* current device is not compute capability 10.3 */
  MOE_ERR_CUDA = 3,            /* a CUDA runtime / driver call failed */
  MOE_ERR_WORKSPACE = 4,       /* workspace or weight blob too small */
  MOE_ERR_TIMEOUT = 5,         /* (device status) a bounded wait gave up */
  MOE_ERR_BOUNDS = 6,          /* (device status) an index check failed */
  MOE_ERR_SCRATCH = 7          /* moe_route_noalloc: T * E exceeds its fixed scratch */
};

/* Layer shape.
 *   T tokens, d hidden size, E routed experts, k experts per token,
 *   n_groups / topk_groups: DSV3 group-limited routing (1/1 = plain top-k),
 *   I expert SwiGLU inner size, n_shared shared experts (0 or 1),
 *   capacity: ring capacity per routed expert (rows); 0 = default
 *   ceil128(2*T*k/E). Constraints: d, I, capacity multiples of 128;
 *   E a multiple of n_groups with at least 2 experts per group when
 *   n_groups > 1; 1 <= k <= 8 and k <= E; E <= 512. T = 0 is valid: every
 *   call then succeeds, moe_backward writes zero weight gradients, and the
 *   per-token arrays (x, topk_idx, topk_w, y, dy, dx) may be null. */
typedef struct moe_config {
  int T, d, E, k, n_groups, topk_groups, I, n_shared;
  int capacity;
  int flags; /* MOE_FLAG_* bits below; other bits are rejected */
  /* Mover warps per CTA of the all-laps ring GEMMs (the counterpart, on one
   * GPU, of the write-ups' "communication SM count" tuning knob: techlab
   * report, section on the two scorecards): 0 = default (2), 1, 2 or 4. The
   * forward GEMM1 takes at most 2 (its SwiGLU epilogue needs the register
   * file of 8 warps); the backward dgrad GEMM takes any of the three. Results
   * do not depend on it. */
  int n_mover_warps;
} moe_config_t;

/* Ring-lap execution. By default each ring direction (forward GEMM1, backward
 * dgrad of the down projection) is ONE persistent cooperative launch over all
 * laps: two mover warps per CTA fill ring slots (lap L in buffer L % 2) while
 * the other warps run the MMAs, and per-tile device counters order a slot's
 * refill after its previous lap's tiles have read it. With this flag each lap
 * is instead a mover launch followed by a GEMM launch, laps alternating
 * between two streams. Both give bitwise-identical results. */
#define MOE_FLAG_LAP_LAUNCHES 1

/* Weight gradients. By default each weight-gradient GEMM runs on single-CTA
 * 128 x 256 tiles (one persistent CTA per SM). With this flag they run on CTA
 * pairs instead, wherever the gradient's row count (d for dW_d, 2I for dW_gu)
 * is a multiple of 256: clusters of two CTAs on two SMs compute 256 x 256
 * (or 256 x 128) output tiles with tcgen05 .cta_group::2 MMAs, each SM
 * staging half of the tile's B rows. Both forms give the same bytes (the same
 * products summed in the same K order). The pair form is the faster product
 * on long K but the slower weight gradient at this layer's per-expert K. */
#define MOE_FLAG_WGRAD_PAIR 2

/* Bytes of workspace the layer needs for this shape (schedule, saved
 * activations for backward, ring buffers, staging). */
MOE_API int moe_workspace_size(const moe_config_t* cfg, size_t* bytes);

/* Bytes of the quantised-weight blob written by moe_quantize_weights. */
MOE_API int moe_weights_size(const moe_config_t* cfg, size_t* bytes);

/* MXFP8 quantisation (write-ups: the layer runs "in MXFP8", Cursor blog
 * summary "method points"; read as OCP MX v1.0: E4M3 elements, one E8M0
 * scale per 32 elements, scale byte floor(log2 amax) - 8 + 127, elements
 * rounded to nearest-even and saturated to +-448).
 *   src: bf16 [rows][K] row-major.
 *   axis = 1: blocks of 32 along K. codes [rows][K], scales [rows][K/32].
 *             K must be a multiple of 32.
 *   axis = 0: blocks of 32 consecutive rows of one column (token axis).
 *             codes [K][rows_pad], scales [K][rows_pad/32] (transposed),
 *             rows_pad = ceil32(rows), zero-padded. K must be a multiple of 32.
 * Scales are written in this canonical row-major layout. */
MOE_API int moe_quantize_mxfp8(const void* src_bf16, int rows, int K, int axis, void* codes, void* scales,
                       moe_stream_t stream);

/* Quantise the expert weights (bf16 masters) into the blob in the four MX
 * orientations the forward and backward GEMMs read.
 *   w_gu [E][2I][d]  rows 0..I-1 gate, I..2I-1 up;   w_d [E][d][I];
 *   ws_gu [n_shared][2I][d], ws_d [n_shared][d][I] (may be NULL if n_shared = 0).
 *   wq: blob of moe_weights_size bytes. Layout is private to the library
 *   (see moe_wq_view). Run once per optimiser step; not part of a layer step. */
MOE_API int moe_quantize_weights(const moe_config_t* cfg, const void* w_gu, const void* w_d, const void* ws_gu,
                         const void* ws_d, void* wq, moe_stream_t stream);

/* Router (write-ups: DSV3-style router, Cursor blog summary "method points").
 *   x [T][d] bf16, w_router [E][d] bf16, bias [E] fp32.
 *   logits = x w_router^T (fp32), s = sigmoid(logits) in a specified fp32
 *   arithmetic, v = s + bias; keep the topk_groups groups with the largest
 *   sum of their two best v; pick the k best v of kept experts (ties to the
 *   lower index), slots ordered by descending v; gates w = s / sum(s).
 *   Outputs topk_idx [T][k] int32 and topk_w [T][k] fp32. Saves logits and
 *   selected scores in ws for backward. */
MOE_API int moe_route(const moe_config_t* cfg, const void* x, const void* w_router, const float* bias, int32_t* topk_idx,
              float* topk_w, void* ws, moe_stream_t stream);

/* moe_route without a workspace, for callers that cannot allocate device
 * memory: code that runs while another allocator (for example a framework's
 * caching allocator) has reserved all of the GPU's memory, or code on a path
 * where cudaMalloc's implicit device-wide synchronisation is not allowed.
 * The write-ups have no counterpart to this entry point.
 *   Same arguments and outputs (topk_idx, topk_w) as moe_route, minus ws;
 *   the selected scores are not saved, so backward still needs moe_route.
 *   The fp32 logits live in a fixed 16 MiB array of device memory inside
 *   the library (held by every GPU that loads it, until the process exits):
 *   T * E must be at most 4,194,304 (T = 16384 at E = 256), otherwise the
 *   call returns MOE_ERR_SCRATCH and enqueues nothing.
 *   It calls no cudaMalloc, cudaFree or other allocating routine. Its first
 *   call in each CUDA context of a device looks up the array's device
 *   address (with that device current); make that first call before any
 *   stream capture. Under lazy module loading (the CUDA default) the device
 *   also reserves the array's 16 MiB at that first call, or at an earlier
 *   moe_route on the device, whichever comes first: so make one of them
 *   before another allocator reserves the GPU's memory. Every call shares
 *   the one array and overwrites the logits it reads, so nothing needs
 *   clearing between calls; calls that overlap on the GPU (different
 *   streams, or different host threads, on one device) race on it and must
 *   be ordered by the caller. */
MOE_API int moe_route_noalloc(const moe_config_t* cfg, const void* x, const void* w_router, const float* bias,
                              int32_t* topk_idx, float* topk_w, moe_stream_t stream);

/* Device-side schedule (write-ups: scheduling runs entirely on the device,
 * under 3 % of MoE time, reused by backward without re-sorting; Cursor blog
 * summary "method points").
 *   topk_idx [T][k] int32. Builds in ws: per-expert counts, exclusive
 *   offsets, stable ranks in (t, j) order, positions offsets[e] + rank,
 *   the inverse permutation, 128-row padded segments and per-lap tile
 *   lists of the ring buffers. No host synchronisation. */
MOE_API int moe_schedule(const moe_config_t* cfg, const int32_t* topk_idx, void* ws, moe_stream_t stream);

/* Forward pass on the schedule in ws (write-ups: dispatch -> expert FFN ->
 * combine, Cursor blog summary "method points"; ring token buffers reused
 * lap by lap without dropping tokens, techlab report).
 *   x [T][d] bf16, wq from moe_quantize_weights, topk_w [T][k] fp32 (from
 *   moe_route). y [T][d] bf16 = sum_j w[t,j] expert_{idx[t,j]}(x_t) +
 *   shared(x_t), each expert a SwiGLU FFN on MXFP8 operands. Saves what
 *   backward needs in ws.
 * All pointers are device memory owned by the caller (the library allocates
 * nothing); ws must hold the schedule of moe_schedule for the same topk_idx.
 * Asynchronous on `stream`; the two ring GEMMs are cooperative launches, so
 * they start once all their CTAs can be resident. Errors (returned before
 * any launch): MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED_ARCH; MOE_ERR_CUDA
 * for a launch failure. A bounded device wait that gives up is reported
 * through moe_status (MOE_ERR_TIMEOUT), not by the return value. */
MOE_API int moe_forward(const moe_config_t* cfg, const void* x, const void* wq, const float* topk_w, void* y, void* ws,
                moe_stream_t stream);

/* Dispatch alone: MX(x) along d into the workspace, then every ring lap's
 * rows gathered into the ring token buffers by the schedule of the last
 * moe_schedule on this workspace (lap L of an expert into buffer L % 2; on
 * return the buffers hold each expert's last two laps). This is the
 * dispatch step the pages describe (tokens pulled into fixed-capacity ring
 * buffers; techlab report, ring token buffer paragraph) run as its own
 * kernel on `stream`. moe_forward does the same moves
 * inside its GEMM1 launch, so a forward needs no dispatch call; this entry
 * serves callers that want the dispatched ring by itself. One launch covers
 * all laps: a warp per (expert, buffer, 8 slots) writes that slot group's
 * laps in lap order, so the final bytes equal those of lap-by-lap dispatch.
 * x: bf16 [T][d] (device). ws: the workspace. Errors: MOE_ERR_INVALID_ARG,
 * MOE_ERR_UNSUPPORTED_ARCH, MOE_ERR_CUDA (launch failure). */
MOE_API int moe_dispatch(const moe_config_t* cfg, const void* x, void* ws, moe_stream_t stream);

/* Backward pass (write-ups: reverse-combine and reverse-dispatch on the
 * reused schedule, Cursor blog summary "method points").
 *   x, w_router, topk_idx, topk_w: the forward inputs / router outputs.
 *   dy [T][d] bf16. Outputs (bf16): dx [T][d], dw_router [E][d],
 *   dw_gu [E][2I][d], dw_d [E][d][I], dws_gu [n_shared][2I][d],
 *   dws_d [n_shared][d][I]. The router bias receives no gradient.
 * Rounding points of the expert dgrad: each token's dy is quantised once,
 * MX along d; a routed row's gate w multiplies its down-projection gradient
 * dh = w (MX(dy) . W_d) in fp32, the same quantity as (w dy) . W_d. The
 * weight gradient of W_d quantises w dy along tokens.
 * ws must be the workspace of the matching moe_forward (its saved g,u, MX(h)
 * and schedule are read). Ownership, stream and error behaviour as for
 * moe_forward; dws_gu / dws_d may be null when n_shared = 0. */
MOE_API int moe_backward(const moe_config_t* cfg, const void* x, const void* w_router, const int32_t* topk_idx,
                 const float* topk_w, const void* dy, const void* wq, void* dx, void* dw_router, void* dw_gu,
                 void* dw_d, void* dws_gu, void* dws_d, void* ws, moe_stream_t stream);

/* Device status word of the workspace: MOE_OK or the first device-side
 * error (code, site). Synchronous: copies 8 bytes to the host on `stream`
 * and waits for it. Clears the word when `clear` is non-zero. */
MOE_API int moe_status(const moe_config_t* cfg, void* ws, int* code, int* site, int clear, moe_stream_t stream);

/* Named views into the workspace (for inspection and tests). */
enum {
  MOE_WS_STATUS = 0,   /* int32[4] */
  MOE_WS_META,         /* int32[16]: [0] laps used, [1] padded rows used, [2] experts with tokens */
  MOE_WS_COUNTS,       /* int32[E+S]   per-expert assignment counts (shared last) */
  MOE_WS_OFFSETS,      /* int32[E+S+1] exclusive prefix sum of counts */
  MOE_WS_POFF,         /* int32[E+S+1] prefix sum of ceil128(counts) */
  MOE_WS_RANK,         /* int32[T*(k+S)] rank of assignment a within its expert */
  MOE_WS_POS,          /* int32[T*(k+S)] offsets[e] + rank */
  MOE_WS_INV,          /* int32[T*(k+S)] inverse of POS */
  MOE_WS_ROWSRC,       /* int32[Rmax]   padded row -> assignment (-1 = padding) */
  MOE_WS_LAPTILES,     /* int32[Lb][E+S+1] per-lap tile prefix sums */
  MOE_WS_HIST,         /* int32[units][E+S] schedule histogram */
  MOE_WS_BASE,         /* int32[units][E+S] schedule scan */
  MOE_WS_LOGITS,       /* fp32[T][E] */
  MOE_WS_SSEL,         /* fp32[T][k] selected sigmoid scores */
  MOE_WS_XQ,           /* u8[Tpad][d]       MX(x) along d */
  MOE_WS_XQ_SF,        /* tiled scales of XQ */
  MOE_WS_RING_X,       /* u8[2][E][C][d]    two ring token buffers (dispatch); lap L uses buffer L % 2 */
  MOE_WS_RING_X_SF,
  MOE_WS_GU,           /* bf16[Rmax][2I]    saved g, u: chunk j (columns 64j..64j+63) of a row holds
                          g[32j..32j+31] then u[32j..32j+31] */
  MOE_WS_HQ,           /* u8[Rmax][I]       MX(h) along I */
  MOE_WS_HQ_SF,
  MOE_WS_HTOK,         /* u8[I][Rmax]       MX(h) along tokens */
  MOE_WS_HTOK_SF,
  MOE_WS_O,            /* bf16[T*(k+S)][d]  expert outputs per assignment */
  MOE_WS_DW,           /* fp32[T][k]        gate gradients */
  MOE_WS_DL,           /* fp32[T][k]        router logit gradients */
  MOE_WS_RING_DO,      /* u8[2][E][C][d]    two ring buffers of the MX(dy) rows (reverse-combine), as RING_X */
  MOE_WS_RING_DO_SF,
  MOE_WS_DOS,          /* u8[Tpad][d]       MX(dy) along d: the dO ring source and the shared expert A */
  MOE_WS_DOS_SF,
  MOE_WS_DOTOK,        /* u8[d][Rmax]       MX(w dy) along tokens */
  MOE_WS_DOTOK_SF,
  MOE_WS_DGU,          /* u8[Rmax][2I]      MX(dGU) along 2I */
  MOE_WS_DGU_SF,
  MOE_WS_DGUTOK,       /* u8[2I][Rmax]      MX(dGU) along tokens */
  MOE_WS_DGUTOK_SF,
  MOE_WS_XTOK,         /* u8[d][Rmax]       MX(x) along tokens */
  MOE_WS_XTOK_SF,
  MOE_WS_DXE,          /* bf16[T*(k+S)][d]  expert input gradients per assignment */
  MOE_WS_DWR_PART,     /* fp32[Rmax/32][d]  router weight-gradient partial sums */
  MOE_WS_ORDER,        /* int32[E+S]   experts by descending count (ties: lower index first) */
  MOE_WS_LAPBASE,      /* int32[Lb+1]  prefix over laps of the lap tile counts */
  MOE_WS_MOVED,        /* int32[...]   per lap m-tile: 8-row groups moved into the ring */
  MOE_WS_CONSUMED,     /* int32[...]   per lap m-tile: GEMM tiles that finished reading it */
  MOE_WS_DH,           /* f32[Rmax][I] dh = dO W_d at padded rank rows (input of the SwiGLU backward) */
  MOE_WS_LAPORDER,     /* int32[...]   position -> lap-major m-tile: the order the all-laps launches walk
                          (an expert's laps 2P and 2P+1 side by side; its pairs spread over the walk) */
  MOE_WS_LAPKEY,       /* int32[3][...] scratch of the walk-order sort: lap-pair units, their ranks, prefix sums */
  MOE_WS_XQ_SFC,       /* u8[T][d/32]   scales of XQ, row-major (the ring movers' source) */
  MOE_WS_DOS_SFC,      /* u8[T][d/32]   scales of DOS, row-major (the dO-ring movers' source) */
  MOE_WS_RINGINFO,     /* int32[...][8] per walk position: the decoded ring m-tile the all-laps launches
                          and their movers read with one load instead of searching the lap and expert
                          prefix sums: {gm, e | valid << 16 | ok << 24 | shared << 25, A row, padded rank
                          row}, {previous tenant's gm or -1, rank of the first row, count, poff[e]} */
  MOE_WS_PUSHINFO,     /* int32[Rmax/128] per m-tile of the padded rank rows: e | valid rows << 16 */
  MOE_WS_WGINFO,       /* int32[E+S][4] per rank of ORDER: {e, first K tile, K tiles, 0} of the weight gradients */
  MOE_WS_COUNT
};
MOE_API int moe_ws_view(const moe_config_t* cfg, void* ws, int which, void** ptr, size_t* bytes);

/* Named views into the quantised-weight blob. Expert e's rows start at
 * e * rows_per_expert; shared experts follow the E routed ones.
 *   W1F: [E+S][2I][d] along d, rows interleaved in 128-row blocks
 *        (gate 128b..128b+127, then up 128b..128b+127);
 *   W2F: [E+S][d][I] along I;  W2B: [E+S][I][d] along d (W_d^T);
 *   W1B: [E+S][d][2I] along 2I (W_gu^T). Scales in the tiled layout. */
enum {
  MOE_WQ_W1F = 0, MOE_WQ_W1F_SF, MOE_WQ_W2F, MOE_WQ_W2F_SF,
  MOE_WQ_W2B, MOE_WQ_W2B_SF, MOE_WQ_W1B, MOE_WQ_W1B_SF, MOE_WQ_COUNT
};
MOE_API int moe_wq_view(const moe_config_t* cfg, void* wq, int which, void** ptr, size_t* bytes);

/* Plain MXFP8 GEMM on the tensor cores (the expert GEMMs' core, exposed for
 * testing): c[M][N] (fp32) = dequant(a)[M][K] . dequant(b)[N][K]^T.
 *   a, b: E4M3 codes, K-major. a_sf, b_sf: scales in the tiled layout
 *   (moe_scales_to_tiled). M, N, K multiples of 128. */
MOE_API int moe_gemm_mxfp8(int M, int N, int K, const void* a, const void* a_sf, const void* b, const void* b_sf, float* c,
                   moe_stream_t stream);

/* moe_gemm_mxfp8 on CTA pairs (exposed for testing; the kernel of the
 * MOE_FLAG_WGRAD_PAIR weight gradients). Clusters of two CTAs on two SMs
 * compute 256 x 256 tiles (256 x 128 when N is not a multiple of 256) with
 * tcgen05 .cta_group::2 MMAs issued by the even CTA; each CTA stages its 128
 * rows of A and half of the tile's rows of B, two 128-element K atoms per
 * pipeline stage. Same operands and result as moe_gemm_mxfp8; M a multiple
 * of 256, N and K of 128. */
MOE_API int moe_gemm_mxfp8_pair(int M, int N, int K, const void* a, const void* a_sf, const void* b,
                                const void* b_sf, float* c, moe_stream_t stream);

/* NVFP4 (exposed as a stand-alone quantiser and GEMM; the write-ups name
 * NVFP4 training kernels beside the MXFP8 ones, Cursor blog summary, opening
 * paragraph, and give no detail). Read as NVIDIA's 4-bit format: E2M1
 * elements (magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6), one E4M3 scale per 16
 * elements along K, one fp32 scale g per tensor (g = amax / (6 * 448) is the
 * usual choice; the caller supplies it). Every step is an IEEE binary32
 * operation: sb = E4M3_RNE_satfinite(amax(block) / (6 g)),
 * X = decode(sb) g, q = E2M1_RNE_satfinite(v / X) (0 when X = 0).
 *   src: bf16 [rows][K], K a multiple of 16. codes: [rows][K/2] bytes, element
 *   2i in the low nibble (8-byte aligned). scales: canonical [rows][K/16]
 *   (tiled = 0) or the tiled layout of 512-byte atoms of 128 rows x 4 blocks
 *   of 16 (tiled = 1; rows a multiple of 128, K of 64), byte offset
 *   ((r/128)*(K/64) + kb/4)*512 + (r%32)*16 + (r/32%4)*4 + kb%4.
 * Errors: MOE_ERR_INVALID_ARG (shapes, g <= 0, alignment), MOE_ERR_UNSUPPORTED_ARCH. */
MOE_API int moe_quantize_nvfp4(const void* src_bf16, int rows, int K, float g, void* codes, void* scales, int tiled,
                               moe_stream_t stream);

/* NVFP4 GEMM on the tensor cores (tcgen05 kind::mxf4nvf4, scale_vec::4X):
 * c[M][N] (fp32) = alpha * dequant(a)[M][K] . dequant(b)[N][K]^T, where a, b are
 * packed E2M1 codes [rows][K/2] and a_sf, b_sf their E4M3 block scales in the
 * tiled layout of moe_quantize_nvfp4; alpha is the product of the two tensor
 * scales. M, N multiples of 128, K of 256; 16-byte aligned pointers. */
MOE_API int moe_gemm_nvfp4(int M, int N, int K, const void* a, const void* a_sf, const void* b, const void* b_sf,
                           float alpha, float* c, moe_stream_t stream);

/* NVFP4 expert GEMM grouped by the schedule in `ws` (moe_schedule must have
 * run on the same stream): for every expert e, routed and shared, and every
 * padded rank row r of its segment [POFF[e], POFF[e+1]) (moe_ws_view),
 *   out[r][n] (fp32) = alpha * sum_k dequant(a)[r][k] * dequant(w)[e*N + n][k],
 * n < N: the expert GEMMs' grouped product in the 4-bit format (NVFP4 read as
 * above; Cursor blog summary, opening paragraph).
 *   a: packed E2M1 codes [Rmax][K/2] in rank order, a_sf their tiled E4M3
 *      scales (moe_quantize_nvfp4, rows = Rmax); Rmax = the padded rank rows
 *      of the workspace, ceil128(T*(k+S)) + 128*(E+S). Rows a segment pads
 *      (past its expert's count) are multiplied like any other.
 *   w: packed codes [(E+S)*N][K/2], expert e's block at rows e*N, w_sf tiled.
 *   alpha: the product of the two tensor scales.
 *   out: fp32 [Rmax][N]; rows at or past POFF[E+S] are not written.
 * N a multiple of 128, K of 256; 16-byte aligned pointers.
 * Errors: MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED_ARCH, MOE_ERR_CUDA. */
MOE_API int moe_expert_gemm_nvfp4(const moe_config_t* cfg, int N, int K, const void* a, const void* a_sf,
                                  const void* w, const void* w_sf, float alpha, float* out, void* ws,
                                  moe_stream_t stream);

/* The same NVFP4 expert GEMM with GEMM2's epilogue: each row r of an expert's
 * segment that holds an assignment a = ROWSRC[r] (moe_ws_view) is written as
 *   out[a][n] (bf16, round to nearest even) = alpha * sum_k dequant(a)[r][k] * dequant(w)[e*N + n][k],
 * the fp32 product of moe_expert_gemm_nvfp4 rounded to bf16, at the
 * assignment's row (a < T*(k+S), the routed then the shared assignments, as
 * the layer's expert outputs O). Padding rows are not written.
 *   out: bf16 [T*(k+S)][N], 16-byte aligned. Other arguments, requirements and
 *   errors as moe_expert_gemm_nvfp4. */
MOE_API int moe_expert_gemm_nvfp4_push(const moe_config_t* cfg, int N, int K, const void* a, const void* a_sf,
                                       const void* w, const void* w_sf, float alpha, void* out, void* ws,
                                       moe_stream_t stream);

/* Re-lay canonical scales [rows][K/32] into the tiled layout the tensor
 * cores read: 512-byte atoms of 128 rows x 4 blocks, atom (r/128, kb/4) at
 * ((r/128)*(K/128) + kb/4)*512, byte (r%32)*16 + (r/32%4)*4 + kb%4.
 * rows, K multiples of 128. */
MOE_API int moe_scales_to_tiled(const void* canon, int rows, int K, void* tiled, moe_stream_t stream);

/* Measurement hooks (process-wide, for benchmarks; not part of the layer).
 * moe_profile_enable(1): every kernel launch of the library is bracketed by a
 * pair of CUDA events recorded on its launch stream (events come from a pool
 * created here; no device memory is allocated). moe_profile_read synchronises
 * the recorded events and returns, per kernel name, the number of launches
 * and their total device time in milliseconds, then clears the records.
 * moe_launch_count: kernels launched by the library since it was loaded. */
typedef struct moe_kernel_time {
  char name[32];
  int launches;
  double ms;
} moe_kernel_time_t;
MOE_API int moe_profile_enable(int enable);
MOE_API int moe_profile_read(moe_kernel_time_t* out, int max_entries, int* n_entries);
/* Like moe_profile_read, but returns every recorded launch in issue order with
 * its start and end in milliseconds after the first recorded start (launches
 * on different streams may overlap), then clears the records. */
typedef struct moe_kernel_span {
  char name[32];
  double start_ms, end_ms;
} moe_kernel_span_t;
MOE_API int moe_profile_trace(moe_kernel_span_t* out, int max_entries, int* n_entries);
MOE_API long long moe_launch_count(void);

/* Failure-detection self-test: launches one kernel that waits on a barrier
 * nothing arrives on, through the same bounded wait every pipeline wait of
 * the library uses. After limit_ns (at most 10 s) the wait gives up and
 * writes MOE_ERR_TIMEOUT and site 900 into status[0..1] (a device int32[2]
 * that the caller zeroes), and the kernel returns: no hang, no trap, and the
 * context stays usable. */
MOE_API int moe_selftest_wait_timeout(int* status, unsigned long long limit_ns, moe_stream_t stream);

/* Host-side fault injection, for tests of the error paths. The next `count`
 * TMA tensor-map encodings made by this process fail as a failed
 * cuTensorMapEncodeTiled would: the GEMM that needed the map is not launched,
 * nothing that depends on it is launched, and the entry point returns
 * MOE_ERR_CUDA. count <= 0 clears a pending injection. Nothing reaches the
 * GPU. Returns MOE_OK. */
MOE_API int moe_debug_fail_tensor_maps(int count);

#ifdef __cplusplus
}
#endif
#endif /* MOE_GB300_H */
