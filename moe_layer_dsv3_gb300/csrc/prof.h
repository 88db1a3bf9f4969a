// Process-wide launch counter, optional per-launch CUDA-event timing, and the
// launch helper every kernel launch of the library goes through.
#pragma once
#include <cuda_runtime.h>

#include <utility>

#include "moe_internal.h"

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

// Launch `kern` with the given shape on `s` through cudaLaunchKernelEx and
// note its return code in the calling entry point's error slot.
template <typename... Kp, typename... Ar>
inline void launch_kernel(const char* name, void (*kern)(Kp...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                          Ar&&... args) {
  cudaLaunchConfig_t lc = {};
  lc.gridDim = grid;
  lc.blockDim = block;
  lc.dynamicSmemBytes = smem;
  lc.stream = s;
  Prof prof(name, s);
  note(cudaLaunchKernelEx(&lc, kern, std::forward<Ar>(args)...));
}

}  // namespace moe
