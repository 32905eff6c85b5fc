// Internal launch interface between the C ABI (api.cpp) and the kernels.
// Every launcher assumes its arguments were validated by api.cpp and only
// enqueues work on the given stream; it returns the cudaError_t of the launch.
#pragma once

#include <cuda_runtime_api.h>
#include <stddef.h>

namespace fbob {

// Device-side give-up state shared by all kernels: a status word the kernels
// set on a timed-out wait, and the wait limit in nanoseconds.
struct DevCtx {
  unsigned int* err;           // device address of the status word
  unsigned long long wait_ns;  // per-wait time limit
  int stall;                   // test hook: producer withholds its first tile
};

struct FwdArgs {
  const void *Q, *K, *V;
  float *O, *L;
  int BH, N, d;
  float tau;
  int causal;  // query i attends to keys j <= i
};

struct BwdArgs {
  const void *Q, *K, *V, *dO;
  const float *O, *L;
  float *dQ, *dK, *dV, *D;
  int BH, N, d;
  float tau;
  int causal;
};

struct BobArgs {
  const void *Q, *K, *V, *dO, *UQ, *UK, *UV;
  const float *O, *L, *D;
  float *gQ, *gK, *gV, *gdO;
  float* ws;  // [BH, N, 2]: alpha, E
  int BH, N, d;
  float tau;
  int causal;
};

// Status word bits.
constexpr unsigned int kErrTimeout = 1u;

// errword.cu: device address of the status word on the current device.
cudaError_t dev_status_word(unsigned int** ptr);

// simt.cu: fp32-FMA kernels for fp32 inputs (any N >= 1).
cudaError_t simt_fwd(const FwdArgs& a, const DevCtx& c, cudaStream_t s);
cudaError_t simt_bwd(const BwdArgs& a, const DevCtx& c, cudaStream_t s);
cudaError_t simt_bob(const BobArgs& a, const DevCtx& c, cudaStream_t s);

// tc_fwd.cu / tc_bwd.cu / tc_bob.cu: tcgen05 kernels for bf16 inputs (any N).
cudaError_t tc_fwd(const FwdArgs& a, const DevCtx& c, cudaStream_t s);
cudaError_t tc_bwd(const BwdArgs& a, const DevCtx& c, cudaStream_t s);
cudaError_t tc_bob(const BobArgs& a, const DevCtx& c, cudaStream_t s);
cudaError_t tc_bob_four_pass(const BobArgs& a, const DevCtx& c, cudaStream_t s);  // ablation schedule
// tc_bob_cols.cu: BoB pass 2 (gK, gV) for heads of 65 to 128 columns.
cudaError_t tc_bob_cols_wide(const BobArgs& a, const DevCtx& c, cudaStream_t s);

// bob_static.cu: the fixed (alpha, E) workspace of fbob_attn_bob_noalloc.
size_t static_workspace_rows();           // capacity in query rows (B*H*N)
cudaError_t static_workspace(float** ptr);  // device address on the current device
unsigned long long current_ctx_id();       // process-unique id of the current context, 0 if unknown

// side_stream.cu: a second stream of the current context for a launcher that
// runs two independent halves of its work at the same time.  fork() makes the
// side stream wait for the work queued so far on s; join() makes s wait for
// everything queued on the side stream since.  The shared stream and events
// are held (host lock) from fork() to join(), which the destructor runs if
// the launcher did not.  Stream capture: both calls are capture-legal and the
// side stream leaves the capture at join(); the first fork() in a context
// creates the stream and events, so it should precede a capture.
class SideStream {
 public:
  SideStream() = default;
  SideStream(const SideStream&) = delete;
  SideStream& operator=(const SideStream&) = delete;
  ~SideStream();
  cudaError_t fork(cudaStream_t s);
  cudaError_t join();
  cudaStream_t stream() const { return side_; }

 private:
  cudaStream_t origin_ = nullptr, side_ = nullptr;
  void* slot_ = nullptr;   // the context's cached stream and events (locked while forked)
};

// Multiprocessors of the current device (0 if unknown).
int sm_count();

}  // namespace fbob
