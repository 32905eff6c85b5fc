// The device status word that kernels set when a bounded wait gives up.
#include <cuda_runtime.h>

#include "internal.h"

namespace fbob {

__device__ unsigned int g_status_word = 0u;

// cudaGetSymbolAddress resolves the address for the current device's context;
// callers fetch it per call so that every device gets its own word.
cudaError_t dev_status_word(unsigned int** ptr) {
  return cudaGetSymbolAddress((void**)ptr, g_status_word);
}

}  // namespace fbob
