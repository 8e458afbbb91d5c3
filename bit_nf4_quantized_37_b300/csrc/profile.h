// profile.h -- RAII scope that brackets one kernel launch with CUDA events when profiling
// is on (qlora_profile_start / qlora_profile_stop in the C ABI).
#pragma once

#include <cuda_runtime.h>

namespace qlora {

bool profiling_enabled();

class ProfileScope {
 public:
  ProfileScope(const char* name, cudaStream_t stream);
  ~ProfileScope();
  ProfileScope(const ProfileScope&) = delete;
  ProfileScope& operator=(const ProfileScope&) = delete;

 private:
  const char* name_;
  cudaStream_t stream_;
  cudaEvent_t start_ = nullptr;
};

}  // namespace qlora
