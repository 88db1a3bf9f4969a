// C ABI: argument checks, workspace layout, and the launch sequence of the
// forward and backward passes. Every step runs in this library's kernels.
#include <atomic>
#include <cstring>
#include <map>
#include <mutex>

#include "moe_internal.h"

namespace moe {

namespace {

constexpr size_t kAlign = 256;

struct Builder {
  size_t cur = 0;
  void add(size_t* off, size_t* bytes, int which, size_t n) {
    off[which] = cur;
    bytes[which] = n;
    cur += (n + kAlign - 1) / kAlign * kAlign;
  }
};

}  // namespace

int current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return -1;
  return dev;
}

cudaError_t& call_error() {
  thread_local cudaError_t e = cudaSuccess;
  return e;
}

bool arch_ok() {
  static std::atomic<int> cache[kMaxDev];   // 0 unknown, 1 sm_103, 2 other
  const int dev = current_device();
  if (dev < 0) return false;
  int v = cache[dev].load(std::memory_order_relaxed);
  if (v == 0) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return false;
    v = (major == 10 && minor == 3) ? 1 : 2;
    cache[dev].store(v, std::memory_order_relaxed);
  }
  return v == 1;
}

namespace {

inline cudaStream_t S(moe_stream_t s) { return static_cast<cudaStream_t>(s); }

// Ring lap L runs on lap stream L % kRingBufs (stream 0 is the caller's, the
// others are auxiliary streams) and uses ring buffer L % kRingBufs, so up to
// kRingBufs laps are in flight: a lap waits only for the lap that used its
// ring buffer before. The backward's side work (reverse-dispatch, router
// weight gradient) runs on the first auxiliary stream. Each caller stream of
// each device gets auxiliary streams and fork / join events of its own, so
// layers driven from different streams do not serialise on a shared one;
// they are created on first use and kept until the process exits. Fork and
// join are event record / wait pairs on the caller's stream.
struct LapStreams {
  std::mutex mu;
  cudaStream_t aux[kRingBufs - 1] = {};
  cudaEvent_t fork = nullptr;
  cudaEvent_t join[kRingBufs - 1] = {};
};
std::mutex g_lap_mu;
std::map<cudaStream_t, LapStreams> g_lap[kMaxDev];

LapStreams* lap_streams(cudaStream_t caller) {
  const int dev = current_device();
  if (dev < 0) return nullptr;
  LapStreams* l;
  {
    std::lock_guard<std::mutex> lk(g_lap_mu);
    l = &g_lap[dev][caller];   // std::map nodes stay put while others are added
  }
  std::lock_guard<std::mutex> lk(l->mu);
  if (l->fork == nullptr) {
    for (int i = 0; i < kRingBufs - 1; ++i)
      if (cudaStreamCreateWithFlags(&l->aux[i], cudaStreamNonBlocking) != cudaSuccess ||
          cudaEventCreateWithFlags(&l->join[i], cudaEventDisableTiming) != cudaSuccess)
        return nullptr;
    if (cudaEventCreateWithFlags(&l->fork, cudaEventDisableTiming) != cudaSuccess) return nullptr;
  }
  return l;
}

// A per-token array (x, topk_idx, topk_w, y, dy, dx) may be null only when there are no tokens.
inline bool tok_ok(const void* p, const moe_config_t* c) { return p != nullptr || c->T == 0; }

// Device buffers read or written with 16-byte vectors or by TMA must start on
// a 16-byte boundary; null (allowed where tok_ok allows it) passes.
inline bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
template <typename... P>
inline bool all_al16(const P*... p) { return (al16(p) && ...); }

// Counters of an all-laps ring launch, zeroed on the stream before it.
RingMovers ring_movers(const Layout& L, void* ws, cudaStream_t s) {
  RingMovers mv{};
  mv.lapbase = ws_ptr<int>(L, ws, MOE_WS_LAPBASE);
  mv.ring_info = ws_ptr<int4>(L, ws, MOE_WS_RINGINFO);
  mv.moved = ws_ptr<int>(L, ws, MOE_WS_MOVED);
  mv.consumed = ws_ptr<int>(L, ws, MOE_WS_CONSUMED);
  note(cudaMemsetAsync(mv.moved, 0, L.bytes[MOE_WS_MOVED], s));
  note(cudaMemsetAsync(mv.consumed, 0, L.bytes[MOE_WS_CONSUMED], s));
  return mv;
}

}  // namespace

int validate(const moe_config_t* c) {
  if (c == nullptr) return MOE_ERR_INVALID_ARG;
  if (c->T < 0 || c->d <= 0 || c->E <= 0 || c->k <= 0 || c->I <= 0) return MOE_ERR_INVALID_ARG;
  if (c->d % 128 || c->I % 128) return MOE_ERR_INVALID_ARG;
  if (c->E > 512 || c->k > 8 || c->k > c->E) return MOE_ERR_INVALID_ARG;
  if (c->n_shared < 0 || c->n_shared > 1) return MOE_ERR_INVALID_ARG;
  if (c->n_groups <= 0 || c->topk_groups <= 0 || c->topk_groups > c->n_groups || c->n_groups > 32)
    return MOE_ERR_INVALID_ARG;
  if (c->E % c->n_groups) return MOE_ERR_INVALID_ARG;
  if (c->n_groups > 1 && (c->E / c->n_groups < 2 || c->k > c->topk_groups * (c->E / c->n_groups)))
    return MOE_ERR_INVALID_ARG;
  if (c->capacity < 0 || c->capacity % 128) return MOE_ERR_INVALID_ARG;
  if (c->flags & ~(MOE_FLAG_LAP_LAUNCHES | MOE_FLAG_WGRAD_PAIR)) return MOE_ERR_INVALID_ARG;
  if (c->n_mover_warps != 0 && c->n_mover_warps != 1 && c->n_mover_warps != 2 && c->n_mover_warps != 4)
    return MOE_ERR_INVALID_ARG;
  const int64_t Ap = static_cast<int64_t>(c->T) * (c->k + c->n_shared);
  if (Ap + 128LL * (c->E + c->n_shared) >= (1LL << 31)) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

Dims make_dims(const moe_config_t* c) {
  Dims m{};
  m.T = c->T;
  m.d = c->d;
  m.E = c->E;
  m.k = c->k;
  m.G = c->n_groups;
  m.gtop = c->topk_groups;
  m.I = c->I;
  m.S = c->n_shared;
  const int64_t avg2 = c->E > 0 ? ceil_div(2LL * c->T * c->k, c->E) : 0;
  m.C = c->capacity > 0 ? c->capacity : static_cast<int>(round_up(avg2 > 128 ? avg2 : 128, 128));
  m.Ep = m.E + m.S;
  m.kp = m.k + m.S;
  m.A = static_cast<int64_t>(m.T) * m.k;
  m.Ap = static_cast<int64_t>(m.T) * m.kp;
  m.Tpad = round_up(m.T, 128);
  m.Rmax = round_up(m.Ap, 128) + 128LL * m.Ep;
  m.Lb = m.T > 0 ? static_cast<int>(ceil_div(m.T, m.C)) : 0;
  m.units = static_cast<int>(ceil_div(m.Ap, kSchedUnit));
  m.MV = c->n_mover_warps > 0 ? c->n_mover_warps : 2;
  return m;
}

Layout make_layout(const moe_config_t* c) {
  Layout L{};
  L.m = make_dims(c);
  const Dims& m = L.m;
  Builder b;
  const size_t T = m.T, d = m.d, E = m.E, k = m.k, I = m.I, Ep = m.Ep;
  const size_t Ap = m.Ap, R = m.Rmax, Tp = m.Tpad, C = m.C;
  b.add(L.off, L.bytes, MOE_WS_STATUS, 16);
  b.add(L.off, L.bytes, MOE_WS_META, 64);
  b.add(L.off, L.bytes, MOE_WS_COUNTS, 4 * Ep);
  b.add(L.off, L.bytes, MOE_WS_OFFSETS, 4 * (Ep + 1));
  b.add(L.off, L.bytes, MOE_WS_POFF, 4 * (Ep + 1));
  b.add(L.off, L.bytes, MOE_WS_RANK, 4 * Ap);
  b.add(L.off, L.bytes, MOE_WS_POS, 4 * Ap);
  b.add(L.off, L.bytes, MOE_WS_INV, 4 * Ap);
  b.add(L.off, L.bytes, MOE_WS_ROWSRC, 4 * R);
  b.add(L.off, L.bytes, MOE_WS_LAPTILES, 4 * static_cast<size_t>(m.Lb > 0 ? m.Lb : 1) * (Ep + 1));
  b.add(L.off, L.bytes, MOE_WS_HIST, 4 * static_cast<size_t>(m.units) * Ep);
  b.add(L.off, L.bytes, MOE_WS_BASE, 4 * static_cast<size_t>(m.units) * Ep);
  b.add(L.off, L.bytes, MOE_WS_LOGITS, 4 * T * E);
  b.add(L.off, L.bytes, MOE_WS_SSEL, 4 * T * k);
  b.add(L.off, L.bytes, MOE_WS_XQ, Tp * d);
  b.add(L.off, L.bytes, MOE_WS_XQ_SF, Tp * d / 32);
  b.add(L.off, L.bytes, MOE_WS_RING_X, kRingBufs * E * C * d);
  b.add(L.off, L.bytes, MOE_WS_RING_X_SF, kRingBufs * E * C * d / 32);
  b.add(L.off, L.bytes, MOE_WS_GU, 2 * R * 2 * I);
  b.add(L.off, L.bytes, MOE_WS_HQ, R * I);
  b.add(L.off, L.bytes, MOE_WS_HQ_SF, R * I / 32);
  b.add(L.off, L.bytes, MOE_WS_HTOK, I * R);
  b.add(L.off, L.bytes, MOE_WS_HTOK_SF, I * R / 32);
  b.add(L.off, L.bytes, MOE_WS_O, 2 * Ap * d);
  b.add(L.off, L.bytes, MOE_WS_DW, 4 * T * k);
  b.add(L.off, L.bytes, MOE_WS_DL, 4 * T * k);
  b.add(L.off, L.bytes, MOE_WS_RING_DO, kRingBufs * E * C * d);
  b.add(L.off, L.bytes, MOE_WS_RING_DO_SF, kRingBufs * E * C * d / 32);
  b.add(L.off, L.bytes, MOE_WS_DOS, Tp * d);
  b.add(L.off, L.bytes, MOE_WS_DOS_SF, Tp * d / 32);
  b.add(L.off, L.bytes, MOE_WS_DOTOK, d * R);
  b.add(L.off, L.bytes, MOE_WS_DOTOK_SF, d * R / 32);
  b.add(L.off, L.bytes, MOE_WS_DGU, R * 2 * I);
  b.add(L.off, L.bytes, MOE_WS_DGU_SF, R * 2 * I / 32);
  b.add(L.off, L.bytes, MOE_WS_DGUTOK, 2 * I * R);
  b.add(L.off, L.bytes, MOE_WS_DGUTOK_SF, 2 * I * R / 32);
  b.add(L.off, L.bytes, MOE_WS_XTOK, d * R);
  b.add(L.off, L.bytes, MOE_WS_XTOK_SF, d * R / 32);
  b.add(L.off, L.bytes, MOE_WS_DXE, 2 * Ap * d);
  b.add(L.off, L.bytes, MOE_WS_DWR_PART, 4 * (R / 32) * d);
  b.add(L.off, L.bytes, MOE_WS_ORDER, 4 * Ep);
  b.add(L.off, L.bytes, MOE_WS_LAPBASE, 4 * static_cast<size_t>(m.Lb + 1));
  b.add(L.off, L.bytes, MOE_WS_MOVED, 4 * static_cast<size_t>(lap_mtiles_max(m)));
  b.add(L.off, L.bytes, MOE_WS_CONSUMED, 4 * static_cast<size_t>(lap_mtiles_max(m)));
  b.add(L.off, L.bytes, MOE_WS_DH, 4 * static_cast<size_t>(m.Rmax) * m.I);
  b.add(L.off, L.bytes, MOE_WS_LAPORDER, 4 * static_cast<size_t>(lap_mtiles_max(m)));
  b.add(L.off, L.bytes, MOE_WS_LAPKEY, 12 * static_cast<size_t>(lap_mtiles_max(m)));
  b.add(L.off, L.bytes, MOE_WS_XQ_SFC, T * d / 32);
  b.add(L.off, L.bytes, MOE_WS_DOS_SFC, T * d / 32);
  b.add(L.off, L.bytes, MOE_WS_RINGINFO, 32 * static_cast<size_t>(lap_mtiles_max(m)));
  b.add(L.off, L.bytes, MOE_WS_PUSHINFO, 4 * static_cast<size_t>(m.Rmax / 128));
  b.add(L.off, L.bytes, MOE_WS_WGINFO, 16 * Ep);
  L.total = b.cur;
  return L;
}

WLayout make_wlayout(const moe_config_t* c) {
  WLayout W{};
  const Dims m = make_dims(c);
  Builder b;
  const size_t Ep = m.Ep, d = m.d, I = m.I;
  b.add(W.off, W.bytes, MOE_WQ_W1F, Ep * 2 * I * d);
  b.add(W.off, W.bytes, MOE_WQ_W1F_SF, Ep * 2 * I * d / 32);
  b.add(W.off, W.bytes, MOE_WQ_W2F, Ep * d * I);
  b.add(W.off, W.bytes, MOE_WQ_W2F_SF, Ep * d * I / 32);
  b.add(W.off, W.bytes, MOE_WQ_W2B, Ep * I * d);
  b.add(W.off, W.bytes, MOE_WQ_W2B_SF, Ep * I * d / 32);
  b.add(W.off, W.bytes, MOE_WQ_W1B, Ep * d * 2 * I);
  b.add(W.off, W.bytes, MOE_WQ_W1B_SF, Ep * d * 2 * I / 32);
  W.total = b.cur;
  return W;
}

}  // namespace moe

using namespace moe;

extern "C" {

int moe_workspace_size(const moe_config_t* cfg, size_t* bytes) {
  if (bytes == nullptr) return MOE_ERR_INVALID_ARG;
  if (int r = validate(cfg)) return r;
  *bytes = make_layout(cfg).total;
  return MOE_OK;
}

int moe_weights_size(const moe_config_t* cfg, size_t* bytes) {
  if (bytes == nullptr) return MOE_ERR_INVALID_ARG;
  if (int r = validate(cfg)) return r;
  *bytes = make_wlayout(cfg).total;
  return MOE_OK;
}

int moe_ws_view(const moe_config_t* cfg, void* ws, int which, void** ptr, size_t* bytes) {
  if (int r = validate(cfg)) return r;
  if (which < 0 || which >= MOE_WS_COUNT || ptr == nullptr) return MOE_ERR_INVALID_ARG;
  const Layout L = make_layout(cfg);
  *ptr = static_cast<char*>(ws) + L.off[which];
  if (bytes) *bytes = L.bytes[which];
  return MOE_OK;
}

int moe_wq_view(const moe_config_t* cfg, void* wq, int which, void** ptr, size_t* bytes) {
  if (int r = validate(cfg)) return r;
  if (which < 0 || which >= MOE_WQ_COUNT || ptr == nullptr) return MOE_ERR_INVALID_ARG;
  const WLayout W = make_wlayout(cfg);
  *ptr = static_cast<char*>(wq) + W.off[which];
  if (bytes) *bytes = W.bytes[which];
  return MOE_OK;
}

int moe_quantize_mxfp8(const void* src, int rows, int K, int axis, void* codes, void* scales, moe_stream_t stream) {
  if (src == nullptr || codes == nullptr || scales == nullptr || rows < 0 || K <= 0 || K % 32)
    return MOE_ERR_INVALID_ARG;
  if (axis != 0 && axis != 1) return MOE_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(src) % 16 || reinterpret_cast<uintptr_t>(codes) % 16) return MOE_ERR_INVALID_ARG;
  if (!arch_ok()) return MOE_ERR_UNSUPPORTED_ARCH;
  CallScope call;
  if (rows == 0) return MOE_OK;
  if (axis == 1) {
    launch_quant_rows(src, rows, K, K, static_cast<uint8_t*>(codes), static_cast<uint8_t*>(scales), false, 0, S(stream));
  } else {
    launch_quant_cols(src, rows, K, K, round_up(rows, 32), static_cast<uint8_t*>(codes), static_cast<uint8_t*>(scales),
                      false, 1, S(stream));
  }
  return call.status();
}

int moe_quantize_weights(const moe_config_t* cfg, const void* w_gu, const void* w_d, const void* ws_gu,
                         const void* ws_d, void* wq, moe_stream_t stream) {
  if (int r = validate(cfg)) return r;
  if (w_gu == nullptr || w_d == nullptr || wq == nullptr) return MOE_ERR_INVALID_ARG;
  if (cfg->n_shared > 0 && (ws_gu == nullptr || ws_d == nullptr)) return MOE_ERR_INVALID_ARG;
  if (!all_al16(w_gu, w_d, ws_gu, ws_d, wq)) return MOE_ERR_INVALID_ARG;
  if (!arch_ok()) return MOE_ERR_UNSUPPORTED_ARCH;
  CallScope call;
  const Dims m = make_dims(cfg);
  const WLayout W = make_wlayout(cfg);
  cudaStream_t s = S(stream);
  const int64_t d = m.d, I = m.I, E = m.E;
  uint8_t* w1f = wq_ptr<uint8_t>(W, wq, MOE_WQ_W1F);
  uint8_t* w1f_sf = wq_ptr<uint8_t>(W, wq, MOE_WQ_W1F_SF);
  uint8_t* w2f = wq_ptr<uint8_t>(W, wq, MOE_WQ_W2F);
  uint8_t* w2f_sf = wq_ptr<uint8_t>(W, wq, MOE_WQ_W2F_SF);
  uint8_t* w2b = wq_ptr<uint8_t>(W, wq, MOE_WQ_W2B);
  uint8_t* w2b_sf = wq_ptr<uint8_t>(W, wq, MOE_WQ_W2B_SF);
  uint8_t* w1b = wq_ptr<uint8_t>(W, wq, MOE_WQ_W1B);
  uint8_t* w1b_sf = wq_ptr<uint8_t>(W, wq, MOE_WQ_W1B_SF);
  for (int part = 0; part < 2; ++part) {
    const void* gu = part == 0 ? w_gu : ws_gu;
    const void* dd = part == 0 ? w_d : ws_d;
    const int64_t n = part == 0 ? E : m.S;
    const int64_t e0 = part == 0 ? 0 : E;
    if (n == 0) continue;
    // GEMM1 forward operand: [2I][d] along d, gate/up rows interleaved by 128.
    launch_quant_rows(gu, n * 2 * I, static_cast<int>(d), d, w1f + e0 * 2 * I * d, w1f_sf + e0 * 2 * I * d / 32, true,
                      static_cast<int>(I), s);
    // GEMM2 forward operand: [d][I] along I.
    launch_quant_rows(dd, n * d, static_cast<int>(I), I, w2f + e0 * d * I, w2f_sf + e0 * d * I / 32, true, 0, s);
    // GEMM2 dgrad operand: W_d^T = [I][d] along d.
    launch_quant_cols(dd, d, static_cast<int>(I), I, d, w2b + e0 * I * d, w2b_sf + e0 * I * d / 32, true,
                      static_cast<int>(n), s);
    // GEMM1 dgrad operand: W_gu^T = [d][2I] along 2I.
    launch_quant_cols(gu, 2 * I, static_cast<int>(d), d, 2 * I, w1b + e0 * d * 2 * I, w1b_sf + e0 * d * 2 * I / 32,
                      true, static_cast<int>(n), s);
  }
  return call.status();
}

int moe_route(const moe_config_t* cfg, const void* x, const void* w_router, const float* bias, int32_t* topk_idx,
              float* topk_w, void* ws, moe_stream_t stream) {
  if (int r = validate(cfg)) return r;
  if (!tok_ok(x, cfg) || !w_router || !bias || !tok_ok(topk_idx, cfg) || !tok_ok(topk_w, cfg) || !ws)
    return MOE_ERR_INVALID_ARG;
  if (!all_al16(x, w_router, ws)) return MOE_ERR_INVALID_ARG;
  if (!arch_ok()) return MOE_ERR_UNSUPPORTED_ARCH;
  CallScope call;
  const Layout L = make_layout(cfg);
  const Dims& m = L.m;
  if (m.T == 0) return MOE_OK;
  float* logits = ws_ptr<float>(L, ws, MOE_WS_LOGITS);
  if (int r = launch_router_logits(m, x, w_router, logits, S(stream))) return r;
  launch_router_topk(m, logits, bias, topk_idx, topk_w, ws_ptr<float>(L, ws, MOE_WS_SSEL), S(stream));
  return call.status();
}

int moe_schedule(const moe_config_t* cfg, const int32_t* topk_idx, void* ws, moe_stream_t stream) {
  if (int r = validate(cfg)) return r;
  if (!tok_ok(topk_idx, cfg) || !ws) return MOE_ERR_INVALID_ARG;
  if (!all_al16(ws)) return MOE_ERR_INVALID_ARG;
  if (!arch_ok()) return MOE_ERR_UNSUPPORTED_ARCH;
  CallScope call;
  const Layout L = make_layout(cfg);
  launch_schedule(L.m, topk_idx, L, ws, S(stream));
  return call.status();
}

int moe_dispatch(const moe_config_t* cfg, const void* x, void* ws, moe_stream_t stream) {
  if (int r = validate(cfg)) return r;
  if (!tok_ok(x, cfg) || !ws) return MOE_ERR_INVALID_ARG;
  if (!all_al16(x, ws)) return MOE_ERR_INVALID_ARG;
  if (!arch_ok()) return MOE_ERR_UNSUPPORTED_ARCH;
  CallScope call;
  const Layout L = make_layout(cfg);
  const Dims& m = L.m;
  if (m.T == 0) return MOE_OK;
  cudaStream_t s = S(stream);
  uint8_t* xq = ws_ptr<uint8_t>(L, ws, MOE_WS_XQ);
  uint8_t* xq_sf = ws_ptr<uint8_t>(L, ws, MOE_WS_XQ_SF);
  if (m.Tpad > m.T) {
    note(cudaMemsetAsync(xq + m.T * m.d, 0, (m.Tpad - m.T) * m.d, s));
    note(cudaMemsetAsync(xq_sf + (m.T / 128) * 128 * (m.d / 32), 0, (m.Tpad - m.T / 128 * 128) * (m.d / 32), s));
  }
  launch_quant_rows(x, m.T, m.d, m.d, xq, xq_sf, true, 0, s, ws_ptr<uint8_t>(L, ws, MOE_WS_XQ_SFC));
  launch_dispatch_all(m, L, ws, s);
  return call.status();
}

int moe_forward(const moe_config_t* cfg, const void* x, const void* wq, const float* topk_w, void* y, void* ws,
                moe_stream_t stream) {
  if (int r = validate(cfg)) return r;
  if (!tok_ok(x, cfg) || !wq || !tok_ok(topk_w, cfg) || !tok_ok(y, cfg) || !ws) return MOE_ERR_INVALID_ARG;
  if (!all_al16(x, wq, y, ws)) return MOE_ERR_INVALID_ARG;
  if (!arch_ok()) return MOE_ERR_UNSUPPORTED_ARCH;
  CallScope call;
  const Layout L = make_layout(cfg);
  const WLayout W = make_wlayout(cfg);
  const Dims& m = L.m;
  if (m.T == 0) return MOE_OK;
  cudaStream_t s = S(stream);
  void* wqm = const_cast<void*>(wq);
  uint8_t* xq = ws_ptr<uint8_t>(L, ws, MOE_WS_XQ);
  uint8_t* xq_sf = ws_ptr<uint8_t>(L, ws, MOE_WS_XQ_SF);
  if (m.Tpad > m.T) {
    note(cudaMemsetAsync(xq + m.T * m.d, 0, (m.Tpad - m.T) * m.d, s));
    note(cudaMemsetAsync(xq_sf + (m.T / 128) * 128 * (m.d / 32), 0, (m.Tpad - m.T / 128 * 128) * (m.d / 32), s));
  }
  launch_quant_rows(x, m.T, m.d, m.d, xq, xq_sf, true, 0, s, ws_ptr<uint8_t>(L, ws, MOE_WS_XQ_SFC));
  int* counts = ws_ptr<int>(L, ws, MOE_WS_COUNTS);
  int* poff = ws_ptr<int>(L, ws, MOE_WS_POFF);
  int* lap_tiles = ws_ptr<int>(L, ws, MOE_WS_LAPTILES);
  int* row_src = ws_ptr<int>(L, ws, MOE_WS_ROWSRC);
  int* status = ws_ptr<int>(L, ws, MOE_WS_STATUS);

  GemmOperands op1{};
  op1.a = ws_ptr<uint8_t>(L, ws, MOE_WS_RING_X);
  op1.a_rows = static_cast<int64_t>(m.E) * m.C;
  op1.a_cols = m.d;
  op1.a_sf = ws_ptr<uint8_t>(L, ws, MOE_WS_RING_X_SF);
  op1.a2 = xq;
  op1.a2_rows = m.Tpad;
  op1.a2_sf = xq_sf;
  op1.b = wq_ptr<uint8_t>(W, wqm, MOE_WQ_W1F);
  op1.b_rows = static_cast<int64_t>(m.Ep) * 2 * m.I;
  op1.b_cols = m.d;
  op1.b_sf = wq_ptr<uint8_t>(W, wqm, MOE_WQ_W1F_SF);
  GemmEpilogue ep1{};
  ep1.gu = ws_ptr<void>(L, ws, MOE_WS_GU);
  ep1.q_rows = ws_ptr<uint8_t>(L, ws, MOE_WS_HQ);
  ep1.q_rows_sf = ws_ptr<uint8_t>(L, ws, MOE_WS_HQ_SF);
  ep1.q_rows_ktiles = m.I / 128;
  ep1.q_tok = ws_ptr<uint8_t>(L, ws, MOE_WS_HTOK);
  ep1.q_tok_sf = ws_ptr<uint8_t>(L, ws, MOE_WS_HTOK_SF);
  ep1.q_tok_pitch = m.Rmax;
  if (!(cfg->flags & MOE_FLAG_LAP_LAUNCHES)) {
    // One persistent launch over all laps; its mover warps fill the ring.
    RingMovers mv = ring_movers(L, ws, s);
    mv.xq = xq;
    mv.xq_sf = xq_sf;
    mv.xq_sfr = ws_ptr<uint8_t>(L, ws, MOE_WS_XQ_SFC);
    mv.ring = ws_ptr<uint8_t>(L, ws, MOE_WS_RING_X);
    mv.ring_sf = ws_ptr<uint8_t>(L, ws, MOE_WS_RING_X_SF);
    op1.a_rows = static_cast<int64_t>(kRingBufs) * m.E * m.C;
    if (int r = gemm_dispatch("gemm1_fwd", kSwigluFwdRing, m, 0, 2 * m.I, m.d, 0, op1, ep1, counts, poff, lap_tiles,
                              row_src, status, s, 0, nullptr, &mv))
      return r;
  } else {
    LapStreams* ls = lap_streams(s);
    if (ls == nullptr) return MOE_ERR_CUDA;
    std::lock_guard<std::mutex> lk(ls->mu);
    note(cudaEventRecord(ls->fork, s));
    for (int i = 0; i < kRingBufs - 1; ++i) note(cudaStreamWaitEvent(ls->aux[i], ls->fork, 0));
    const uint8_t* ring = op1.a;
    const uint8_t* ring_sf = op1.a_sf;
    const size_t rb = static_cast<size_t>(m.E) * m.C * m.d;
    int rc = MOE_OK;
    for (int lap = 0; lap < m.Lb && rc == MOE_OK; ++lap) {
      const int rbuf = lap % kRingBufs;
      cudaStream_t cs = rbuf ? ls->aux[rbuf - 1] : s;
      op1.a = ring + rbuf * rb;
      op1.a_sf = ring_sf + rbuf * rb / 32;
      launch_permute_lap(m, lap, false, L, ws, cs);
      rc = gemm_dispatch("gemm1_fwd", kSwigluFwd, m, lap, 2 * m.I, m.d, 0, op1, ep1, counts, poff, lap_tiles, row_src,
                         status, cs);
    }
    for (int i = 0; i < kRingBufs - 1; ++i) {
      note(cudaEventRecord(ls->join[i], ls->aux[i]));
      note(cudaStreamWaitEvent(s, ls->join[i], 0));
    }
    if (rc) return rc;
  }
  GemmOperands op2{};
  op2.a = ws_ptr<uint8_t>(L, ws, MOE_WS_HQ);
  op2.a_rows = m.Rmax;
  op2.a_cols = m.I;
  op2.a_sf = ws_ptr<uint8_t>(L, ws, MOE_WS_HQ_SF);
  op2.b = wq_ptr<uint8_t>(W, wqm, MOE_WQ_W2F);
  op2.b_rows = static_cast<int64_t>(m.Ep) * m.d;
  op2.b_cols = m.I;
  op2.b_sf = wq_ptr<uint8_t>(W, wqm, MOE_WQ_W2F_SF);
  GemmEpilogue ep2{};
  ep2.out = ws_ptr<void>(L, ws, MOE_WS_O);
  ep2.ldo = m.d;
  if (int r = gemm_dispatch("gemm2_fwd", kPush, m, 0, m.d, m.I, 0, op2, ep2, counts, poff, lap_tiles, row_src, status,
                            s, 0, nullptr, nullptr, ws_ptr<int>(L, ws, MOE_WS_PUSHINFO)))
    return r;
  launch_combine(m, topk_w, L, ws, y, s);
  return call.status();
}

int moe_backward(const moe_config_t* cfg, const void* x, const void* w_router, const int32_t* topk_idx,
                 const float* topk_w, const void* dy, const void* wq, void* dx, void* dw_router, void* dw_gu,
                 void* dw_d, void* dws_gu, void* dws_d, void* ws, moe_stream_t stream) {
  if (int r = validate(cfg)) return r;
  if (!tok_ok(x, cfg) || !w_router || !tok_ok(topk_idx, cfg) || !tok_ok(topk_w, cfg) || !tok_ok(dy, cfg) || !wq ||
      !tok_ok(dx, cfg) || !dw_router || !dw_gu || !dw_d || !ws)
    return MOE_ERR_INVALID_ARG;
  if (cfg->n_shared > 0 && (!dws_gu || !dws_d)) return MOE_ERR_INVALID_ARG;
  if (!all_al16(x, w_router, dy, wq, dx, dw_router, dw_gu, dw_d, dws_gu, dws_d, ws)) return MOE_ERR_INVALID_ARG;
  if (!arch_ok()) return MOE_ERR_UNSUPPORTED_ARCH;
  CallScope call;
  const Layout L = make_layout(cfg);
  const WLayout W = make_wlayout(cfg);
  const Dims& m = L.m;
  cudaStream_t s = S(stream);
  void* wqm = const_cast<void*>(wq);
  int* counts = ws_ptr<int>(L, ws, MOE_WS_COUNTS);
  int* poff = ws_ptr<int>(L, ws, MOE_WS_POFF);
  int* lap_tiles = ws_ptr<int>(L, ws, MOE_WS_LAPTILES);
  int* row_src = ws_ptr<int>(L, ws, MOE_WS_ROWSRC);
  int* status = ws_ptr<int>(L, ws, MOE_WS_STATUS);
  if (m.T == 0) {
    // No tokens: every gradient is zero.
    note(cudaMemsetAsync(dw_router, 0, static_cast<size_t>(m.E) * m.d * 2, s));
    note(cudaMemsetAsync(dw_gu, 0, static_cast<size_t>(m.E) * 2 * m.I * m.d * 2, s));
    note(cudaMemsetAsync(dw_d, 0, static_cast<size_t>(m.E) * m.d * m.I * 2, s));
    if (m.S) {
      note(cudaMemsetAsync(dws_gu, 0, static_cast<size_t>(m.S) * 2 * m.I * m.d * 2, s));
      note(cudaMemsetAsync(dws_d, 0, static_cast<size_t>(m.S) * m.d * m.I * 2, s));
    }
    return call.status();
  }
  // Reverse-combine: gate gradients, router logit gradients.
  launch_rev_combine_dw(m, dy, topk_w, L, ws, s);
  // MX(dy) along d, once per token (token order; rows past T zero): the rows
  // the dO ring is filled from, and the shared expert's dgrad input in place.
  // The gate of a routed row scales its dh in the dgrad-down epilogue.
  uint8_t* dos = ws_ptr<uint8_t>(L, ws, MOE_WS_DOS);
  uint8_t* dos_sf = ws_ptr<uint8_t>(L, ws, MOE_WS_DOS_SF);
  if (m.Tpad > m.T) {
    note(cudaMemsetAsync(dos + m.T * m.d, 0, (m.Tpad - m.T) * m.d, s));
    note(cudaMemsetAsync(dos_sf + (m.T / 128) * 128 * (m.d / 32), 0, (m.Tpad - m.T / 128 * 128) * (m.d / 32), s));
  }
  launch_quant_rows(dy, m.T, m.d, m.d, dos, dos_sf, true, 0, s, ws_ptr<uint8_t>(L, ws, MOE_WS_DOS_SFC));
  // Token-axis operands of the weight gradients (and router dW partial sums).
  launch_tok_gather(m, x, false, topk_w, true, L, ws, ws_ptr<uint8_t>(L, ws, MOE_WS_XTOK),
                    ws_ptr<uint8_t>(L, ws, MOE_WS_XTOK_SF), s);
  launch_tok_gather(m, dy, true, topk_w, false, L, ws, ws_ptr<uint8_t>(L, ws, MOE_WS_DOTOK),
                    ws_ptr<uint8_t>(L, ws, MOE_WS_DOTOK_SF), s);
  // dgrad of GEMM2 + SwiGLU backward, lap by lap through the dO ring.
  GemmOperands opb2{};
  opb2.a = ws_ptr<uint8_t>(L, ws, MOE_WS_RING_DO);
  opb2.a_rows = static_cast<int64_t>(m.E) * m.C;
  opb2.a_cols = m.d;
  opb2.a_sf = ws_ptr<uint8_t>(L, ws, MOE_WS_RING_DO_SF);
  opb2.a2 = dos;
  opb2.a2_rows = m.Tpad;
  opb2.a2_sf = dos_sf;
  opb2.b = wq_ptr<uint8_t>(W, wqm, MOE_WQ_W2B);
  opb2.b_rows = static_cast<int64_t>(m.Ep) * m.I;
  opb2.b_cols = m.d;
  opb2.b_sf = wq_ptr<uint8_t>(W, wqm, MOE_WQ_W2B_SF);
  GemmEpilogue epb2{};
  epb2.out = ws_ptr<void>(L, ws, MOE_WS_DH);
  epb2.gate = topk_w;
  epb2.ldo = m.I;
  if (!(cfg->flags & MOE_FLAG_LAP_LAUNCHES)) {
    RingMovers mv = ring_movers(L, ws, s);
    mv.xq = dos;
    mv.xq_sf = dos_sf;
    mv.xq_sfr = ws_ptr<uint8_t>(L, ws, MOE_WS_DOS_SFC);
    mv.ring = ws_ptr<uint8_t>(L, ws, MOE_WS_RING_DO);
    mv.ring_sf = ws_ptr<uint8_t>(L, ws, MOE_WS_RING_DO_SF);
    opb2.a_rows = static_cast<int64_t>(kRingBufs) * m.E * m.C;
    if (int r = gemm_dispatch("gemm_dgrad_down", kSwigluBwdRing, m, 0, m.I, m.d, 0, opb2, epb2, counts, poff,
                              lap_tiles, row_src, status, s, 256, nullptr, &mv))
      return r;
  } else {
    LapStreams* ls = lap_streams(s);
    if (ls == nullptr) return MOE_ERR_CUDA;
    std::lock_guard<std::mutex> lk(ls->mu);
    note(cudaEventRecord(ls->fork, s));
    for (int i = 0; i < kRingBufs - 1; ++i) note(cudaStreamWaitEvent(ls->aux[i], ls->fork, 0));
    const uint8_t* ring = opb2.a;
    const uint8_t* ring_sf = opb2.a_sf;
    const size_t rb = static_cast<size_t>(m.E) * m.C * m.d;
    int rc = MOE_OK;
    for (int lap = 0; lap < m.Lb && rc == MOE_OK; ++lap) {
      const int rbuf = lap % kRingBufs;
      cudaStream_t cs = rbuf ? ls->aux[rbuf - 1] : s;
      opb2.a = ring + rbuf * rb;
      opb2.a_sf = ring_sf + rbuf * rb / 32;
      launch_permute_lap(m, lap, true, L, ws, cs);
      rc = gemm_dispatch("gemm_dgrad_down", kSwigluBwd, m, lap, m.I, m.d, 0, opb2, epb2, counts, poff, lap_tiles,
                         row_src, status, cs, 256);
    }
    for (int i = 0; i < kRingBufs - 1; ++i) {
      note(cudaEventRecord(ls->join[i], ls->aux[i]));
      note(cudaStreamWaitEvent(s, ls->join[i], 0));
    }
    if (rc) return rc;
  }
  // SwiGLU backward on dh and the saved g,u; MX(dGU) along 2I and along ranks.
  launch_swiglu_bwd_quant(m, L, ws, s);
  // dgrad of GEMM1: DX rows pushed to their assignment.
  GemmOperands opb4{};
  opb4.a = ws_ptr<uint8_t>(L, ws, MOE_WS_DGU);
  opb4.a_rows = m.Rmax;
  opb4.a_cols = 2 * m.I;
  opb4.a_sf = ws_ptr<uint8_t>(L, ws, MOE_WS_DGU_SF);
  opb4.b = wq_ptr<uint8_t>(W, wqm, MOE_WQ_W1B);
  opb4.b_rows = static_cast<int64_t>(m.Ep) * m.d;
  opb4.b_cols = 2 * m.I;
  opb4.b_sf = wq_ptr<uint8_t>(W, wqm, MOE_WQ_W1B_SF);
  GemmEpilogue epb4{};
  epb4.out = ws_ptr<void>(L, ws, MOE_WS_DXE);
  epb4.ldo = m.d;
  if (int r = gemm_dispatch("gemm_dgrad_gu", kPush, m, 0, m.d, 2 * m.I, 0, opb4, epb4, counts, poff, lap_tiles,
                            row_src, status, s, 0, nullptr, nullptr, ws_ptr<int>(L, ws, MOE_WS_PUSHINFO)))
    return r;
  // Weight gradients: K = the expert's ranks (token axis), all laps at once.
  GemmOperands opw{};
  opw.a = ws_ptr<uint8_t>(L, ws, MOE_WS_DOTOK);
  opw.a_rows = m.d;
  opw.a_cols = static_cast<int>(m.Rmax);
  opw.a_sf = ws_ptr<uint8_t>(L, ws, MOE_WS_DOTOK_SF);
  opw.b = ws_ptr<uint8_t>(L, ws, MOE_WS_HTOK);
  opw.b_rows = m.I;
  opw.b_cols = static_cast<int>(m.Rmax);
  opw.b_sf = ws_ptr<uint8_t>(L, ws, MOE_WS_HTOK_SF);
  GemmEpilogue epw{};
  epw.out = dw_d;
  epw.out2 = dws_d;
  epw.ldo = m.I;
  // Reverse-dispatch (+ router input gradient) and the router weight gradient
  // depend on no weight gradient: they run on a side stream beside them, in
  // the SM resources the persistent weight-gradient CTAs leave free.
  LapStreams* ls = lap_streams(s);
  if (ls == nullptr) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lk(ls->mu);
  note(cudaEventRecord(ls->fork, s));
  // Weight gradients on single-CTA 128 x 256 tiles, or on CTA pairs (256-row
  // tiles) when asked for and the output rows allow it.
  const bool pair_d = (cfg->flags & MOE_FLAG_WGRAD_PAIR) && m.d % kPairRows == 0;
  const bool pair_gu = (cfg->flags & MOE_FLAG_WGRAD_PAIR) && (2 * m.I) % kPairRows == 0;
  const int* order = ws_ptr<int>(L, ws, MOE_WS_ORDER);
  const int4* wg_info = ws_ptr<int4>(L, ws, MOE_WS_WGINFO);
  if (int r = pair_d ? gemm_pair_dispatch("gemm_wgrad_d", kWgrad, m, m.I, m.d, 0, opw, epw, poff, order, status, s)
                     : gemm_dispatch("gemm_wgrad_d", kWgrad, m, 0, m.I, 0, m.d, opw, epw, counts, poff, lap_tiles,
                                     row_src, status, s, 256, order, nullptr, wg_info))
    return r;
  note(cudaStreamWaitEvent(ls->aux[0], ls->fork, 0));
  launch_reverse_dispatch(m, topk_idx, w_router, L, ws, dx, ls->aux[0]);
  launch_router_dwr(m, L, ws, dw_router, ls->aux[0]);
  note(cudaEventRecord(ls->join[0], ls->aux[0]));
  opw.a = ws_ptr<uint8_t>(L, ws, MOE_WS_DGUTOK);
  opw.a_rows = 2 * m.I;
  opw.a_sf = ws_ptr<uint8_t>(L, ws, MOE_WS_DGUTOK_SF);
  opw.b = ws_ptr<uint8_t>(L, ws, MOE_WS_XTOK);
  opw.b_rows = m.d;
  opw.b_sf = ws_ptr<uint8_t>(L, ws, MOE_WS_XTOK_SF);
  epw.out = dw_gu;
  epw.out2 = dws_gu;
  epw.ldo = m.d;
  const int r = pair_gu ? gemm_pair_dispatch("gemm_wgrad_gu", kWgrad, m, m.d, 2 * m.I, 0, opw, epw, poff, order,
                                             status, s)
                        : gemm_dispatch("gemm_wgrad_gu", kWgrad, m, 0, m.d, 0, 2 * m.I, opw, epw, counts, poff,
                                        lap_tiles, row_src, status, s, 256, order, nullptr, wg_info);
  note(cudaStreamWaitEvent(s, ls->join[0], 0));
  if (r) return r;
  return call.status();
}

int moe_status(const moe_config_t* cfg, void* ws, int* code, int* site, int clear, moe_stream_t stream) {
  if (int r = validate(cfg)) return r;
  if (!ws || !code || !site) return MOE_ERR_INVALID_ARG;
  const Layout L = make_layout(cfg);
  int h[2] = {0, 0};
  int* st = ws_ptr<int>(L, ws, MOE_WS_STATUS);
  if (cudaMemcpyAsync(h, st, sizeof(h), cudaMemcpyDeviceToHost, S(stream)) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(S(stream)) != cudaSuccess) return MOE_ERR_CUDA;
  *code = h[0];
  *site = h[1];
  if (clear && cudaMemsetAsync(st, 0, 16, S(stream)) != cudaSuccess) return MOE_ERR_CUDA;
  return MOE_OK;
}

}  // extern "C"
