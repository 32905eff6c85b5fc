// Optional per-kernel timing: when enabled with fbob_profile_enable, every
// kernel launch of the library is bracketed by two CUDA events recorded on its
// stream; fbob_profile_report turns them into per-kernel counts and times.
#pragma once

#include <cuda_runtime_api.h>

namespace fbob {

// Both are no-ops unless profiling is enabled.
void prof_begin(cudaStream_t s, const char* kernel);
void prof_end(cudaStream_t s);

}  // namespace fbob
