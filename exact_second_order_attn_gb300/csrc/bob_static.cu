// Fixed device-resident workspace for fbob_attn_bob_noalloc.
//
// fbob_attn_bob needs an (alpha, E) workspace of 8 * B * H * N bytes from the
// caller.  Some callers cannot provide one: hosts that hand the library only
// their own input and output buffers (an embedding framework whose caching
// allocator has already reserved the device memory, a plug-in interface with
// fixed tensor arguments), or latency-bound loops that must not call
// cudaMalloc / cudaFree because those calls can synchronise the device.  For
// them the workspace lives in one file-scope device array instead, which
// every GPU that loads this library holds until the process exits.
//
// In host code the array's name is only a host-side handle, not a device
// address: its device address is fetched with cudaGetSymbolAddress once per
// device, with that device current, on the first fbob_attn_bob_noalloc call
// on that device, and cached.  Every call on a device shares the array and
// the last call's values stay in it; calls that run at the same time on the
// GPU (different streams with no ordering between them) race on it.  Pass 1
// writes every (alpha, E) element that pass 2 reads, so nothing has to be
// cleared between calls.
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"

namespace fbob {

namespace {

// 2 floats (alpha, E) per query row; 2^21 rows = 16 MiB per device.
constexpr size_t kStaticRows = size_t(1) << 21;

static __device__ __align__(256) float g_bob_static_ws[2 * kStaticRows];

constexpr int kMaxDevices = 64;
float* g_ptr[kMaxDevices] = {};
std::mutex g_mu;

}  // namespace

size_t static_workspace_rows() { return kStaticRows; }

cudaError_t static_workspace(float** ptr) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_bob_static_ws);
    if (e != cudaSuccess) return e;
    g_ptr[dev] = static_cast<float*>(p);
  }
  *ptr = g_ptr[dev];
  return cudaSuccess;
}

}  // namespace fbob
