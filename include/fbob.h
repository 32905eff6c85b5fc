/*
 * fbob.h - C ABI of the GB300 (sm_103a) exact attention backward-over-backward
 * library (libfbob.so).
 *
 * The library computes, for softmax attention with scale tau,
 *   forward        O = softmax(tau Q K^T) V,  L = row logsumexp (natural log)
 *   first backward g(Q, K, V, dO) = (dQ, dK, dV) and D = rowsum(dO o O)
 *   BoB            J_g^T applied to (UQ, UK, UV) at (dQ, dK, dV), i.e. the
 *                  gradients gQ, gK, gV, gdO of
 *                  f = <UQ, dQ> + <UK, dK> + <UV, dV>
 *                  with respect to Q, K, V, dO.
 * Sources: "FlashBoB: I/O-Efficient Exact Backward-over-Backward for Softmax
 * Attention" - the abstract (aiqbench.com / arxivdaily.com pages) for the
 * forward / first backward / BoB chain, and the evolve.pub review: "Scope &
 * Claims" (BoB = J_g^T at (dQ, dK, dV), paper section 4.1), Summary and Key
 * claims (two-pass schedule, the row scalars alpha and E are the only length-N
 * vectors that cross the pass boundary, no N x N tensor in HBM; paper
 * Prop. 4.1 and Algorithm 1), FAQ "Is FlashBoB an approximation?" (exact
 * outputs, bf16 inputs with fp32 accumulation).
 *
 * Conventions shared by every call
 * --------------------------------
 * - All tensor arguments are DEVICE pointers owned by the caller.  The library
 *   never allocates device memory, frees or synchronises inside these calls;
 *   every launch is ordered on `stream` (fbob_attn_bwd and fbob_attn_bob may
 *   fork part of their work onto a stream of their own and join it back, see
 *   fbob_attn_bob) and the call
 *   returns before the GPU finishes.
 *   Outputs are overwritten, never accumulated into.
 * - Matrices are [B, H, N, d] row-major and contiguous (element (b, h, i, c)
 *   at ((b*H + h)*N + i)*d + c); row vectors (L, D) are [B, H, N]; the BoB
 *   workspace is [B, H, N, 2] floats (alpha, E interleaved per row).
 * - Inputs Q, K, V, dO, UQ, UK, UV have the element type `dtype` of the
 *   problem (bf16 or fp32); O, L, D, all gradients and the workspace are
 *   fp32.
 * - Every pointer must be 16-byte aligned and tensors must not overlap an
 *   output of the same call.
 * - Supported: d in {32, 64, 96, 128}; any N >= 1 (bf16 and fp32); causal or
 *   not.  (bf16 heads of 32 and 96 run on the 64- and 128-column tensor-core
 *   kernels with the missing columns zero-padded on chip.)
 *   B*H*N == 0 is a valid empty problem
 *   (returns FBOB_OK, launches nothing).
 * - Argument problems are reported BEFORE any launch (nothing is launched on
 *   error).  A failed launch returns FBOB_ERR_CUDA.  Kernels never trap: a
 *   device-side wait that exceeds its time limit makes the kernel give up and
 *   record FBOB_ERR_TIMEOUT in a device status word, read with
 *   fbob_device_status().
 * - No C++ exception crosses this interface.  Functions are thread-safe;
 *   fbob_last_error() is per host thread.
 */
#ifndef FBOB_H_
#define FBOB_H_

#include <stddef.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define FBOB_ABI_VERSION 1

typedef enum {
  FBOB_OK = 0,
  FBOB_ERR_INVALID_ARG = 1,   /* null/misaligned pointer, bad sizes or tau    */
  FBOB_ERR_UNSUPPORTED = 2,   /* valid problem outside the supported set      */
  FBOB_ERR_WORKSPACE = 3,     /* workspace pointer null or too small          */
  FBOB_ERR_CUDA = 4,          /* a CUDA runtime call or launch failed         */
  FBOB_ERR_TIMEOUT = 5        /* a device-side wait ran out (device status)   */
} fbob_status;

typedef enum {
  FBOB_BF16 = 0,              /* inputs are IEEE bfloat16                     */
  FBOB_FP32 = 1               /* inputs are IEEE binary32                     */
} fbob_dtype;

/* One attention problem: B batches x H heads of N x d matrices. */
typedef struct {
  int B, H, N, d;
  float tau;                  /* score scale, S = tau Q K^T; finite, nonzero  */
  int dtype;                  /* fbob_dtype of Q, K, V, dO, UQ, UK, UV        */
  int causal;                 /* 0: full attention; nonzero: causal, query i  */
                              /* attends to keys j <= i                       */
} fbob_problem;

/*
 * Forward (FlashBoB abstract: FlashAttention-style forward).
 *   in : Q, K, V  [B,H,N,d] dtype
 *   out: O [B,H,N,d] fp32, L [B,H,N] fp32 (natural-log row logsumexp of
 *        tau Q K^T)
 */
fbob_status fbob_attn_fwd(const fbob_problem* p,
                          const void* Q, const void* K, const void* V,
                          float* O, float* L, cudaStream_t stream);

/*
 * First backward g (FlashBoB abstract; evolve.pub review FAQ "What is
 * backward-over-backward"):
 *   dV = P^T dO, dP = dO V^T, D = rowsum(dO o O), dS = P o (dP - D),
 *   dQ = tau dS K, dK = tau dS^T Q, with P = exp(tau Q K^T - L).
 *   in : Q, K, V, dO [B,H,N,d] dtype; O [B,H,N,d] fp32 and L [B,H,N] fp32
 *        from fbob_attn_fwd on the same Q, K, V
 *   out: dQ, dK, dV [B,H,N,d] fp32; D [B,H,N] fp32
 * Streams: like fbob_attn_bob (bf16), the heads may run as two groups, the
 * second on the library's forked stream; ordered on `stream` as one call.
 */
fbob_status fbob_attn_bwd(const fbob_problem* p,
                          const void* Q, const void* K, const void* V,
                          const float* O, const void* dO, const float* L,
                          float* dQ, float* dK, float* dV, float* D,
                          cudaStream_t stream);

/* Bytes of BoB workspace: 2 * B * H * N * sizeof(float) (alpha and E). */
size_t fbob_bob_workspace_bytes(const fbob_problem* p);

/*
 * Backward over backward (evolve.pub review, "Scope & Claims", Summary, Key
 * claims; paper section 4.1, Prop. 4.1, Algorithm 1).  Two passes on
 * `stream`:
 *   pass 1, per block of query rows, loops over all key tiles, reduces the
 *     row scalars alpha_i = sum_j P_ij B_ij and
 *     E_i = sum_j P_ij (C_ij + B_ij dP_ij)   (B = tau (UQ K^T + Q UK^T),
 *     C = dO UV^T) while accumulating alpha-free sums, applies the affine
 *     correction at the row end and writes gQ, gdO and (alpha, E);
 *   pass 2, per block of keys, loops over all query tiles and writes gK, gV.
 *   Only alpha and E (the workspace) cross between the passes; no N x N
 *   matrix is ever stored.
 *   in : Q, K, V, dO, UQ, UK, UV [B,H,N,d] dtype; O [B,H,N,d] fp32 and
 *        L [B,H,N] fp32 from fbob_attn_fwd; D [B,H,N] fp32 from fbob_attn_bwd
 *   out: gQ, gK, gV, gdO [B,H,N,d] fp32;
 *        workspace [B,H,N,2] fp32 = (alpha_i, E_i) per row, at least
 *        fbob_bob_workspace_bytes(p) bytes (FBOB_ERR_WORKSPACE otherwise)
 * Streams (bf16 inputs): when B*H >= 2 and each pass would end on a mostly
 * empty wave of thread blocks, the heads run as two groups, the second on a
 * library-owned stream forked from `stream` (it waits for the work already
 * queued there) and joined back (`stream` waits for it before any later
 * work).  Seen from `stream`, the call is ordered exactly as one launch
 * sequence; results do not depend on the grouping.  The first such call in
 * a CUDA context creates that stream and two events (kept until the process
 * exits); make it before any stream capture, like the first
 * fbob_attn_bob_noalloc call.
 */
fbob_status fbob_attn_bob(const fbob_problem* p,
                          const void* Q, const void* K, const void* V,
                          const float* O, const void* dO,
                          const float* L, const float* D,
                          const void* UQ, const void* UK, const void* UV,
                          float* gQ, float* gK, float* gV, float* gdO,
                          float* workspace, size_t workspace_bytes,
                          cudaStream_t stream);

/*
 * BoB on the four-pass schedule, an ablation of the two-pass fbob_attn_bob
 * ("FlashBoB", evolve.pub review - Strengths: the hierarchical affine
 * structure collapses a natural four-pass schedule to two).  The pages name
 * the four-pass schedule without spelling it out; this library's reading is
 * the order plain reverse mode imposes when the row scalars are not split
 * off affinely:
 *   1. row sweep: alpha_i = sum_j P tau B;
 *   2. row sweep: E in its natural form, which uses alpha (the cotangent of
 *      P carries - alpha dP from D = rowsum(dO o O));
 *   3. row sweep: gQ and gdO accumulated directly, alpha and E known;
 *   4. column pass: gK, gV (the same kernel as fbob_attn_bob's pass 2).
 * Same arguments, outputs (identical up to rounding order), workspace and
 * errors as fbob_attn_bob; bf16 inputs only (fp32 returns
 * FBOB_ERR_UNSUPPORTED).  It runs 25 GEMMs of 2 N^2 d per head against the
 * two-pass schedule's 19 counted (20 executed).
 */
fbob_status fbob_attn_bob_four_pass(const fbob_problem* p,
                                    const void* Q, const void* K, const void* V,
                                    const float* O, const void* dO,
                                    const float* L, const float* D,
                                    const void* UQ, const void* UK, const void* UV,
                                    float* gQ, float* gK, float* gV, float* gdO,
                                    float* workspace, size_t workspace_bytes,
                                    cudaStream_t stream);

/*
 * BoB without a caller workspace (the paper has no counterpart; this is a
 * convenience of this library).  Same inputs, outputs, passes and errors as
 * fbob_attn_bob, but the (alpha, E) workspace is a fixed device array inside
 * the library, so the caller passes only inputs and outputs and nothing is
 * allocated.  It serves callers that cannot obtain an extra device buffer:
 * hosts that hand over only their own tensors, or loops that must not call
 * cudaMalloc/cudaFree (they can synchronise the device).
 *   - Capacity: B*H*N <= 2097152 (2^21) query rows; larger problems return
 *     FBOB_ERR_UNSUPPORTED before any launch.  Every GPU that loads the
 *     library holds the array (16 MiB) until the process exits.
 *   - The array's device address belongs to the CUDA context the library's
 *     device code is loaded into.  The first call in a context (per device:
 *     its primary context, a non-primary context the caller made current, or
 *     the new context after cudaDeviceReset) looks the address up with that
 *     device current (cudaGetSymbolAddress, which may load the library's
 *     device code) and saves it for later calls in the same context; make
 *     that first call - on every device, and again after a cudaDeviceReset -
 *     before any stream capture.
 *   - All calls on a device share the array: calls whose kernels overlap on
 *     the GPU (e.g. on two unordered streams) race and give wrong results.
 *     Calls ordered on one stream are safe; no clearing is needed between
 *     them (pass 1 rewrites every element pass 2 reads).
 */
fbob_status fbob_attn_bob_noalloc(const fbob_problem* p,
                                  const void* Q, const void* K, const void* V,
                                  const float* O, const void* dO,
                                  const float* L, const float* D,
                                  const void* UQ, const void* UK, const void* UV,
                                  float* gQ, float* gK, float* gV, float* gdO,
                                  cudaStream_t stream);

/*
 * Device status: waits for `stream` to finish (this call DOES synchronise),
 * then returns FBOB_ERR_TIMEOUT if any kernel of this library on the current
 * device gave up on a bounded wait since the last call, else FBOB_OK (or
 * FBOB_ERR_CUDA if the synchronisation itself failed).  Clears the word.
 */
fbob_status fbob_device_status(cudaStream_t stream);

/*
 * Time limit, in nanoseconds, of every device-side wait of later launches
 * (default 2e9 = 2 s; 0 restores the default).  Meant for tests of the
 * give-up path; returns the previous limit.
 */
unsigned long long fbob_set_wait_limit_ns(unsigned long long ns);

/*
 * Per-kernel timing (measurement aid, off by default).  While enabled, every
 * kernel launch of the library is bracketed by two CUDA events recorded on
 * its stream.  fbob_profile_report waits for the recorded launches, adds
 * them to per-kernel totals and returns the length of the text
 * {"kernel": [launches, total_ms, min_ms, max_ms], ...}; if buf can hold the
 * whole text (len > length) it writes it NUL-terminated and clears the
 * totals, otherwise (e.g. buf == NULL) the totals are kept.
 * fbob_profile_enable returns the previous setting.
 */
int fbob_profile_enable(int on);
int fbob_profile_report(char* buf, size_t len);

/*
 * Test hook for the give-up path (off by default).  With stall = 1 the TMA
 * producer of every tensor-core kernel launched afterwards withholds its
 * first streamed tile, so the consumers' bounded waits run out: the kernels
 * give up, free their resources and return, and fbob_device_status reports
 * FBOB_ERR_TIMEOUT.  Returns the previous setting.
 */
int fbob_debug_stall_producer(int stall);

/* Static text for a status code. */
const char* fbob_status_string(fbob_status s);

/* Detail text of the last non-OK status returned on this host thread. */
const char* fbob_last_error(void);

/* FBOB_ABI_VERSION of the loaded library. */
int fbob_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FBOB_H_ */
