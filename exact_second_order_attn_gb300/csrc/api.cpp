// C ABI of libfbob.so: argument validation, dispatch to the kernel launchers
// and status reporting.  See include/fbob.h for the contract of each call.
#include "fbob.h"

#include <cuda_runtime_api.h>
#include <math.h>
#include <stdarg.h>
#include <stdint.h>
#include <stdio.h>

#include <atomic>

#include "internal.h"

namespace {

thread_local char g_last_error[512] = "";
std::atomic<unsigned long long> g_wait_ns{2000000000ull};
std::atomic<int> g_stall{0};
constexpr unsigned long long kDefaultWaitNs = 2000000000ull;

fbob_status fail(fbob_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return s;
}

fbob_status cuda_fail(cudaError_t e, const char* where) {
  return fail(FBOB_ERR_CUDA, "%s: %s (%s)", where, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Shared checks of the problem descriptor.  Returns FBOB_OK and sets *empty
// when there is nothing to compute.
fbob_status check_problem(const fbob_problem* p, bool* empty) {
  if (!p) return fail(FBOB_ERR_INVALID_ARG, "problem descriptor is null");
  if (p->B < 0 || p->H < 0 || p->N < 0 || p->d <= 0)
    return fail(FBOB_ERR_INVALID_ARG, "bad sizes B=%d H=%d N=%d d=%d", p->B, p->H, p->N, p->d);
  if (!isfinite(p->tau) || p->tau == 0.f)
    return fail(FBOB_ERR_INVALID_ARG, "tau must be finite and nonzero (got %g)", (double)p->tau);
  if (p->dtype != FBOB_BF16 && p->dtype != FBOB_FP32)
    return fail(FBOB_ERR_INVALID_ARG, "unknown dtype %d", p->dtype);
  if (p->d != 32 && p->d != 64 && p->d != 96 && p->d != 128)
    return fail(FBOB_ERR_UNSUPPORTED, "head size d=%d (supported: 32, 64, 96, 128)", p->d);
  const long long heads = (long long)p->B * p->H;
  if (heads > 65535) return fail(FBOB_ERR_UNSUPPORTED, "B*H=%lld exceeds 65535", heads);
  if ((long long)p->N * p->d * heads > (1ll << 40))
    return fail(FBOB_ERR_UNSUPPORTED, "problem of %lld elements per tensor is too large",
                (long long)p->N * p->d * heads);
  *empty = (heads == 0 || p->N == 0);
  return FBOB_OK;
}

struct Ptr {
  const void* p;
  const char* name;
};

fbob_status check_ptrs(const Ptr* ps, int n) {
  for (int i = 0; i < n; ++i) {
    if (!ps[i].p) return fail(FBOB_ERR_INVALID_ARG, "pointer %s is null", ps[i].name);
    if (!aligned16(ps[i].p)) return fail(FBOB_ERR_INVALID_ARG, "pointer %s is not 16-byte aligned", ps[i].name);
  }
  return FBOB_OK;
}

fbob_status make_ctx(fbob::DevCtx* c) {
  cudaError_t e = fbob::dev_status_word(&c->err);
  if (e != cudaSuccess) return cuda_fail(e, "device status word");
  c->wait_ns = g_wait_ns.load();
  c->stall = g_stall.load();
  return FBOB_OK;
}

}  // namespace

extern "C" {

int fbob_abi_version(void) { return FBOB_ABI_VERSION; }

const char* fbob_status_string(fbob_status s) {
  switch (s) {
    case FBOB_OK: return "FBOB_OK";
    case FBOB_ERR_INVALID_ARG: return "FBOB_ERR_INVALID_ARG";
    case FBOB_ERR_UNSUPPORTED: return "FBOB_ERR_UNSUPPORTED";
    case FBOB_ERR_WORKSPACE: return "FBOB_ERR_WORKSPACE";
    case FBOB_ERR_CUDA: return "FBOB_ERR_CUDA";
    case FBOB_ERR_TIMEOUT: return "FBOB_ERR_TIMEOUT";
  }
  return "FBOB_UNKNOWN_STATUS";
}

const char* fbob_last_error(void) { return g_last_error; }

unsigned long long fbob_set_wait_limit_ns(unsigned long long ns) {
  return g_wait_ns.exchange(ns == 0 ? kDefaultWaitNs : ns);
}

int fbob_debug_stall_producer(int stall) { return g_stall.exchange(stall ? 1 : 0); }

size_t fbob_bob_workspace_bytes(const fbob_problem* p) {
  if (!p || p->B < 0 || p->H < 0 || p->N < 0) return 0;
  return (size_t)2 * sizeof(float) * (size_t)p->B * (size_t)p->H * (size_t)p->N;
}

fbob_status fbob_attn_fwd(const fbob_problem* p, const void* Q, const void* K, const void* V, float* O, float* L,
                          cudaStream_t stream) {
  bool empty = false;
  fbob_status st = check_problem(p, &empty);
  if (st != FBOB_OK) return st;
  if (empty) return FBOB_OK;
  const Ptr ps[] = {{Q, "Q"}, {K, "K"}, {V, "V"}, {O, "O"}, {L, "L"}};
  if ((st = check_ptrs(ps, 5)) != FBOB_OK) return st;
  fbob::DevCtx c;
  if ((st = make_ctx(&c)) != FBOB_OK) return st;
  fbob::FwdArgs a{Q, K, V, O, L, p->B * p->H, p->N, p->d, p->tau, p->causal != 0};
  cudaError_t e = p->dtype == FBOB_BF16 ? fbob::tc_fwd(a, c, stream) : fbob::simt_fwd(a, c, stream);
  if (e != cudaSuccess) return cuda_fail(e, "attn_fwd launch");
  return FBOB_OK;
}

fbob_status fbob_attn_bwd(const fbob_problem* p, const void* Q, const void* K, const void* V, const float* O,
                          const void* dO, const float* L, float* dQ, float* dK, float* dV, float* D,
                          cudaStream_t stream) {
  bool empty = false;
  fbob_status st = check_problem(p, &empty);
  if (st != FBOB_OK) return st;
  if (empty) return FBOB_OK;
  const Ptr ps[] = {{Q, "Q"},   {K, "K"},   {V, "V"},   {O, "O"},   {dO, "dO"},
                    {L, "L"},   {dQ, "dQ"}, {dK, "dK"}, {dV, "dV"}, {D, "D"}};
  if ((st = check_ptrs(ps, 10)) != FBOB_OK) return st;
  fbob::DevCtx c;
  if ((st = make_ctx(&c)) != FBOB_OK) return st;
  fbob::BwdArgs a{Q, K, V, dO, O, L, dQ, dK, dV, D, p->B * p->H, p->N, p->d, p->tau, p->causal != 0};
  cudaError_t e = p->dtype == FBOB_BF16 ? fbob::tc_bwd(a, c, stream) : fbob::simt_bwd(a, c, stream);
  if (e != cudaSuccess) return cuda_fail(e, "attn_bwd launch");
  return FBOB_OK;
}

fbob_status fbob_attn_bob(const fbob_problem* p, const void* Q, const void* K, const void* V, const float* O,
                          const void* dO, const float* L, const float* D, const void* UQ, const void* UK,
                          const void* UV, float* gQ, float* gK, float* gV, float* gdO, float* workspace,
                          size_t workspace_bytes, cudaStream_t stream) {
  bool empty = false;
  fbob_status st = check_problem(p, &empty);
  if (st != FBOB_OK) return st;
  if (empty) return FBOB_OK;
  const Ptr ps[] = {{Q, "Q"},   {K, "K"},   {V, "V"},   {O, "O"},   {dO, "dO"}, {L, "L"},    {D, "D"},
                    {UQ, "UQ"}, {UK, "UK"}, {UV, "UV"}, {gQ, "gQ"}, {gK, "gK"}, {gV, "gV"}, {gdO, "gdO"}};
  if ((st = check_ptrs(ps, 14)) != FBOB_OK) return st;
  if (!workspace) return fail(FBOB_ERR_WORKSPACE, "workspace pointer is null");
  if (!aligned16(workspace)) return fail(FBOB_ERR_WORKSPACE, "workspace is not 16-byte aligned");
  const size_t need = fbob_bob_workspace_bytes(p);
  if (workspace_bytes < need)
    return fail(FBOB_ERR_WORKSPACE, "workspace of %zu bytes is smaller than the %zu needed", workspace_bytes, need);
  fbob::DevCtx c;
  if ((st = make_ctx(&c)) != FBOB_OK) return st;
  fbob::BobArgs a{Q, K, V, dO, UQ, UK, UV, O, L, D, gQ, gK, gV, gdO, workspace, p->B * p->H, p->N, p->d, p->tau,
                  p->causal != 0};
  cudaError_t e = p->dtype == FBOB_BF16 ? fbob::tc_bob(a, c, stream) : fbob::simt_bob(a, c, stream);
  if (e != cudaSuccess) return cuda_fail(e, "attn_bob launch");
  return FBOB_OK;
}

fbob_status fbob_attn_bob_four_pass(const fbob_problem* p, const void* Q, const void* K, const void* V,
                                    const float* O, const void* dO, const float* L, const float* D, const void* UQ,
                                    const void* UK, const void* UV, float* gQ, float* gK, float* gV, float* gdO,
                                    float* workspace, size_t workspace_bytes, cudaStream_t stream) {
  bool empty = false;
  fbob_status st = check_problem(p, &empty);
  if (st != FBOB_OK) return st;
  if (p->dtype != FBOB_BF16)
    return fail(FBOB_ERR_UNSUPPORTED, "fbob_attn_bob_four_pass: the ablation schedule runs bf16 inputs only");
  if (empty) return FBOB_OK;
  const Ptr ps[] = {{Q, "Q"},   {K, "K"},   {V, "V"},   {O, "O"},   {dO, "dO"}, {L, "L"},    {D, "D"},
                    {UQ, "UQ"}, {UK, "UK"}, {UV, "UV"}, {gQ, "gQ"}, {gK, "gK"}, {gV, "gV"}, {gdO, "gdO"}};
  if ((st = check_ptrs(ps, 14)) != FBOB_OK) return st;
  if (!workspace) return fail(FBOB_ERR_WORKSPACE, "workspace pointer is null");
  if (!aligned16(workspace)) return fail(FBOB_ERR_WORKSPACE, "workspace is not 16-byte aligned");
  const size_t need = fbob_bob_workspace_bytes(p);
  if (workspace_bytes < need)
    return fail(FBOB_ERR_WORKSPACE, "workspace of %zu bytes is smaller than the %zu needed", workspace_bytes, need);
  fbob::DevCtx c;
  if ((st = make_ctx(&c)) != FBOB_OK) return st;
  fbob::BobArgs a{Q, K, V, dO, UQ, UK, UV, O, L, D, gQ, gK, gV, gdO, workspace, p->B * p->H, p->N, p->d, p->tau,
                  p->causal != 0};
  cudaError_t e = fbob::tc_bob_four_pass(a, c, stream);
  if (e != cudaSuccess) return cuda_fail(e, "attn_bob_four_pass launch");
  return FBOB_OK;
}

fbob_status fbob_attn_bob_noalloc(const fbob_problem* p, const void* Q, const void* K, const void* V,
                                  const float* O, const void* dO, const float* L, const float* D, const void* UQ,
                                  const void* UK, const void* UV, float* gQ, float* gK, float* gV, float* gdO,
                                  cudaStream_t stream) {
  bool empty = false;
  fbob_status st = check_problem(p, &empty);
  if (st != FBOB_OK) return st;
  if (empty) return FBOB_OK;
  const Ptr ps[] = {{Q, "Q"},   {K, "K"},   {V, "V"},   {O, "O"},   {dO, "dO"}, {L, "L"},    {D, "D"},
                    {UQ, "UQ"}, {UK, "UK"}, {UV, "UV"}, {gQ, "gQ"}, {gK, "gK"}, {gV, "gV"}, {gdO, "gdO"}};
  if ((st = check_ptrs(ps, 14)) != FBOB_OK) return st;
  const size_t rows = (size_t)p->B * (size_t)p->H * (size_t)p->N;
  if (rows > fbob::static_workspace_rows())
    return fail(FBOB_ERR_UNSUPPORTED,
                "fbob_attn_bob_noalloc: B*H*N = %zu exceeds the fixed workspace of %zu rows; "
                "use fbob_attn_bob with a caller workspace",
                rows, fbob::static_workspace_rows());
  float* ws = nullptr;
  cudaError_t e = fbob::static_workspace(&ws);
  if (e != cudaSuccess) return cuda_fail(e, "fixed workspace address");
  fbob::DevCtx c;
  if ((st = make_ctx(&c)) != FBOB_OK) return st;
  fbob::BobArgs a{Q, K, V, dO, UQ, UK, UV, O, L, D, gQ, gK, gV, gdO, ws, p->B * p->H, p->N, p->d, p->tau,
                  p->causal != 0};
  e = p->dtype == FBOB_BF16 ? fbob::tc_bob(a, c, stream) : fbob::simt_bob(a, c, stream);
  if (e != cudaSuccess) return cuda_fail(e, "attn_bob_noalloc launch");
  return FBOB_OK;
}

fbob_status fbob_device_status(cudaStream_t stream) {
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
  unsigned int* word = nullptr;
  if ((e = fbob::dev_status_word(&word)) != cudaSuccess) return cuda_fail(e, "device status word");
  unsigned int v = 0;
  if ((e = cudaMemcpy(&v, word, sizeof(v), cudaMemcpyDeviceToHost)) != cudaSuccess)
    return cuda_fail(e, "read device status word");
  if (v != 0) {
    const unsigned int zero = 0;
    if ((e = cudaMemcpy(word, &zero, sizeof(zero), cudaMemcpyHostToDevice)) != cudaSuccess)
      return cuda_fail(e, "clear device status word");
    if (v & fbob::kErrTimeout) return fail(FBOB_ERR_TIMEOUT, "a device-side wait exceeded its time limit");
  }
  return FBOB_OK;
}

}  // extern "C"
