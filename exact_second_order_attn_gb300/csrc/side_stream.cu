// A second stream per CUDA context, for launchers that split their work into
// two independent halves run at the same time (see SideStream in internal.h).
//
// Why: BoB launches pass 1 and then pass 2 over all heads.  When the number
// of CTAs is a few multiprocessors' worth past a multiple of the SM count,
// the last wave of each launch leaves most SMs idle.  Two head groups on two
// streams let one group's pass 2 start on the SMs the other group's pass 1
// leaves free.
//
// The stream and the two events are created once per (device, context) and
// kept for the life of the process; a context created later on the same
// device (after cudaDeviceReset, or a non-primary context) gets its own.  A
// per-context lock is held from fork() to join(), so two host threads that
// split on the same context take turns queueing their halves (the GPU work
// itself still overlaps).
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"

namespace fbob {

namespace {

constexpr int kMaxDevices = 64;

struct Slot {
  std::mutex mu;
  unsigned long long ctx_id = 0;   // 0: not created
  cudaStream_t side = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};
Slot g_slots[kMaxDevices];
int g_sms[kMaxDevices] = {};

}  // namespace

int sm_count() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  if (g_sms[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    g_sms[dev] = n;
  }
  return g_sms[dev];
}

cudaError_t SideStream::fork(cudaStream_t s) {
  if (slot_) return cudaErrorInvalidValue;   // already forked
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  const unsigned long long id = current_ctx_id();
  if (id == 0) return cudaErrorNotSupported;   // no way to key the cache: the caller runs unsplit
  Slot& sl = g_slots[dev];
  sl.mu.lock();
  if (sl.ctx_id != id) {
    // first fork in this context (handles of an earlier context are dropped, not destroyed)
    cudaStream_t st = nullptr;
    cudaEvent_t f = nullptr, j = nullptr;
    e = cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&f, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&j, cudaEventDisableTiming);
    if (e != cudaSuccess) {
      if (j) cudaEventDestroy(j);
      if (f) cudaEventDestroy(f);
      if (st) cudaStreamDestroy(st);
      sl.mu.unlock();
      cudaGetLastError();   // the failure is returned here, not left for the next launch check
      return e;
    }
    sl.ctx_id = id;
    sl.side = st;
    sl.fork = f;
    sl.join = j;
  }
  e = cudaEventRecord(sl.fork, s);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(sl.side, sl.fork, 0);
  if (e != cudaSuccess) {
    sl.mu.unlock();
    cudaGetLastError();
    return e;
  }
  origin_ = s;
  side_ = sl.side;
  slot_ = &sl;
  return cudaSuccess;
}

cudaError_t SideStream::join() {
  if (!slot_) return cudaSuccess;
  Slot& sl = *static_cast<Slot*>(slot_);
  cudaError_t e = cudaEventRecord(sl.join, side_);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(origin_, sl.join, 0);
  slot_ = nullptr;
  side_ = nullptr;
  sl.mu.unlock();
  return e;
}

SideStream::~SideStream() { join(); }

}  // namespace fbob
