// Process-wide launch counter and optional per-launch CUDA-event timing.
#pragma once
#include <cuda_runtime.h>

namespace moe {

// Bracket one kernel launch: counts it and, when profiling is enabled,
// records a CUDA event before and after it on the launch stream.
class Prof {
 public:
  Prof(const char* name, cudaStream_t s);
  ~Prof();
  Prof(const Prof&) = delete;
  Prof& operator=(const Prof&) = delete;

 private:
  const char* name_;
  cudaStream_t s_;
  cudaEvent_t a_ = nullptr, b_ = nullptr;
};

}  // namespace moe
