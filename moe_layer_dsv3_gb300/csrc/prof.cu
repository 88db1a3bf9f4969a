// Launch accounting and event timing behind moe_profile_* / moe_launch_count.
#include <atomic>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "moe_internal.h"
#include "prof.h"
#include "ptx.cuh"

namespace moe {

// Self-test of the bounded waits: waits on an mbarrier that nothing ever
// arrives on, so the wait must give up after limit_ns and record
// (kErrTimeout, 900) in status, leaving the context usable.
__global__ void wait_timeout_selftest_kernel(int* status, unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
    mbar_wait(&bar, 0, status, 900, limit_ns);
  }
}

namespace {

struct Rec {
  const char* name;
  cudaEvent_t a, b;
};

std::mutex g_mu;
bool g_enabled = false;
std::vector<Rec> g_recs;
std::vector<cudaEvent_t> g_pool;
std::atomic<long long> g_launches{0};

cudaEvent_t take_event() {
  if (g_pool.empty()) {
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    return e;
  }
  cudaEvent_t e = g_pool.back();
  g_pool.pop_back();
  return e;
}

}  // namespace

Prof::Prof(const char* name, cudaStream_t s) : name_(name), s_(s) {
  g_launches.fetch_add(1, std::memory_order_relaxed);
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_enabled) return;
  a_ = take_event();
  b_ = take_event();
  if (a_ && b_) cudaEventRecord(a_, s_);
}

Prof::~Prof() {
  if (!a_ || !b_) return;
  cudaEventRecord(b_, s_);
  std::lock_guard<std::mutex> lk(g_mu);
  g_recs.push_back({name_, a_, b_});
}

}  // namespace moe

extern "C" {

int moe_profile_enable(int enable) {
  std::lock_guard<std::mutex> lk(moe::g_mu);
  moe::g_enabled = enable != 0;
  if (moe::g_enabled && moe::g_pool.size() < 1024) {
    while (moe::g_pool.size() < 1024) {
      cudaEvent_t e = nullptr;
      if (cudaEventCreate(&e) != cudaSuccess) return MOE_ERR_CUDA;
      moe::g_pool.push_back(e);
    }
  }
  return MOE_OK;
}

int moe_profile_read(moe_kernel_time_t* out, int max_entries, int* n_entries) {
  if (n_entries == nullptr || (max_entries > 0 && out == nullptr)) return MOE_ERR_INVALID_ARG;
  std::vector<moe::Rec> recs;
  {
    std::lock_guard<std::mutex> lk(moe::g_mu);
    recs.swap(moe::g_recs);
  }
  std::vector<std::string> names;
  std::vector<int> counts;
  std::vector<double> ms;
  int rc = MOE_OK;
  for (const auto& r : recs) {
    float t = 0.0f;
    if (cudaEventSynchronize(r.b) != cudaSuccess || cudaEventElapsedTime(&t, r.a, r.b) != cudaSuccess) rc = MOE_ERR_CUDA;
    size_t i = 0;
    while (i < names.size() && names[i] != r.name) ++i;
    if (i == names.size()) {
      names.emplace_back(r.name);
      counts.push_back(0);
      ms.push_back(0.0);
    }
    counts[i] += 1;
    ms[i] += t;
  }
  {
    std::lock_guard<std::mutex> lk(moe::g_mu);
    for (const auto& r : recs) {
      moe::g_pool.push_back(r.a);
      moe::g_pool.push_back(r.b);
    }
  }
  const int n = static_cast<int>(names.size());
  for (int i = 0; i < n && i < max_entries; ++i) {
    std::memset(out[i].name, 0, sizeof(out[i].name));
    std::strncpy(out[i].name, names[i].c_str(), sizeof(out[i].name) - 1);
    out[i].launches = counts[i];
    out[i].ms = ms[i];
  }
  *n_entries = n;
  return rc;
}

int moe_profile_trace(moe_kernel_span_t* out, int max_entries, int* n_entries) {
  if (n_entries == nullptr || (max_entries > 0 && out == nullptr)) return MOE_ERR_INVALID_ARG;
  std::vector<moe::Rec> recs;
  {
    std::lock_guard<std::mutex> lk(moe::g_mu);
    recs.swap(moe::g_recs);
  }
  int rc = MOE_OK;
  const int n = static_cast<int>(recs.size());
  for (int i = 0; i < n; ++i) {
    float t0 = 0.0f, t1 = 0.0f;
    if (cudaEventSynchronize(recs[i].b) != cudaSuccess ||
        cudaEventElapsedTime(&t0, recs[0].a, recs[i].a) != cudaSuccess ||
        cudaEventElapsedTime(&t1, recs[0].a, recs[i].b) != cudaSuccess)
      rc = MOE_ERR_CUDA;
    if (i < max_entries) {
      std::memset(out[i].name, 0, sizeof(out[i].name));
      std::strncpy(out[i].name, recs[i].name, sizeof(out[i].name) - 1);
      out[i].start_ms = t0;
      out[i].end_ms = t1;
    }
  }
  {
    std::lock_guard<std::mutex> lk(moe::g_mu);
    for (const auto& r : recs) {
      moe::g_pool.push_back(r.a);
      moe::g_pool.push_back(r.b);
    }
  }
  *n_entries = n;
  return rc;
}

long long moe_launch_count(void) { return moe::g_launches.load(); }

int moe_selftest_wait_timeout(int* status, unsigned long long limit_ns, moe_stream_t stream) {
  if (status == nullptr || limit_ns == 0 || limit_ns > 10000000000ull) return MOE_ERR_INVALID_ARG;
  moe::CallScope call;
  moe::launch_kernel("selftest_wait", moe::wait_timeout_selftest_kernel, dim3(1), dim3(32), 0,
                     static_cast<cudaStream_t>(stream), status, limit_ns);
  return call.status();
}

}  // extern "C"
