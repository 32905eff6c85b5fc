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
// address.  Its device address belongs to the CUDA context the library's
// device code is loaded into, so it is looked up with cudaGetSymbolAddress,
// with the caller's device current, once per context: the saved address is
// keyed by the device and the context's process-unique id (cuCtxGetId), so a
// context created later on the same device - after cudaDeviceReset, or a
// non-primary context made current by the caller - gets its own lookup and
// never a stale address.  Every call on a device shares the array and the
// last call's values stay in it; calls that run at the same time on the GPU
// (different streams with no ordering between them) race on it.  Pass 1
// writes every (alpha, E) element that pass 2 reads, so nothing has to be
// cleared between calls.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "internal.h"

namespace fbob {

namespace {

// 2 floats (alpha, E) per query row; 2^21 rows = 16 MiB per device.
constexpr size_t kStaticRows = size_t(1) << 21;

static __device__ __align__(256) float g_bob_static_ws[2 * kStaticRows];

constexpr int kMaxDevices = 64;

struct Saved {
  unsigned long long ctx_id;  // 0: nothing saved (context ids start at 1)
  float* ptr;
};
Saved g_saved[kMaxDevices] = {};
std::mutex g_mu;

// Driver entry points, reached through the runtime (the library does not link
// libcuda directly).
struct CtxFns {
  PFN_cuCtxGetCurrent_v4000 current = nullptr;
  PFN_cuCtxGetId_v12000 id = nullptr;
};

const CtxFns& ctx_fns() {
  static const CtxFns fns = [] {
    CtxFns f;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      f.current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      f.id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
    return f;
  }();
  return fns;
}

}  // namespace

// Process-unique id of the current context, or 0 if it cannot be read.
unsigned long long current_ctx_id() {
  const CtxFns& f = ctx_fns();
  if (!f.current || !f.id) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (f.current(&ctx) != CUDA_SUCCESS || !ctx) return 0;
  if (f.id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

size_t static_workspace_rows() { return kStaticRows; }

cudaError_t static_workspace(float** ptr) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  const unsigned long long id = current_ctx_id();
  if (id != 0 && g_saved[dev].ctx_id == id) {
    *ptr = g_saved[dev].ptr;
    return cudaSuccess;
  }
  // First call in this context (or its id is unreadable): look the address up.
  // This also makes the device's primary context current if none was.
  void* p = nullptr;
  e = cudaGetSymbolAddress(&p, g_bob_static_ws);
  if (e != cudaSuccess) return e;
  const unsigned long long id_after = id != 0 ? id : current_ctx_id();
  g_saved[dev] = Saved{id_after, id_after != 0 ? static_cast<float*>(p) : nullptr};
  *ptr = static_cast<float*>(p);
  return cudaSuccess;
}

}  // namespace fbob
