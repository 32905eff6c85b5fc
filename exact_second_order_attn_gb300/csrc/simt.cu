// fp32 CUDA-core (FFMA) kernels for the attention forward, first backward and
// the two-pass BoB.  They serve fp32 inputs (every product and sum in fp32,
// nothing rounded below fp32) and any N >= 1; bf16 inputs go to the tcgen05
// kernels.  The element type stays a template parameter of the loaders.  The tile schedule is the same as
// the tensor-core kernels: a CTA owns a block of 32 rows that stays in shared
// memory and streams 32-row tiles of the other side, recomputing score tiles
// on chip; no N x N matrix is stored.
//
// Thread map (256 threads): r = tid / 8 owns tile row r; q = tid % 8 owns
// score columns 4q..4q+3 and accumulator columns q + 8m (m < d/8).  The eight
// threads of a row are consecutive lanes, so row reductions are 3 shuffles.
//
// Source of the arithmetic: "FlashBoB: I/O-Efficient Exact Backward-over-
// Backward for Softmax Attention", evolve.pub review - Summary and Key claims
// (two passes, row scalars alpha and E, paper Prop. 4.1 / Algorithm 1) and
// Strengths (alpha-free accumulators corrected after the row reduction).
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>

#include "internal.h"
#include "prof.h"

namespace fbob {
namespace {

constexpr int BR = 32;   // resident rows per CTA
constexpr int BC = 32;   // streamed rows per tile
static_assert(BR == BC, "the causal column loops start at the block's first row");
constexpr int NT = 256;  // threads per CTA
constexpr int LO = BC + 1;

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }

// Load rows [row0, row0+32) of a [N, D] matrix into smem with row stride LD
// (as fp32), zero rows at or beyond N.
template <typename T, int D>
__device__ __forceinline__ void load_rows(float* dst, const T* __restrict__ src, int row0, int N) {
  constexpr int LD = D + 1;
  for (int idx = threadIdx.x; idx < 32 * D; idx += NT) {
    const int r = idx / D, c = idx % D;
    const int g = row0 + r;
    dst[r * LD + c] = (g < N) ? to_f(src[(size_t)g * D + c]) : 0.f;
  }
}

__device__ __forceinline__ float row_sum8(float v) {
  v += __shfl_xor_sync(0xffffffffu, v, 1);
  v += __shfl_xor_sync(0xffffffffu, v, 2);
  v += __shfl_xor_sync(0xffffffffu, v, 4);
  return v;
}
__device__ __forceinline__ float row_max8(float v) {
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 1));
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 2));
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 4));
  return v;
}

// ---------------------------------------------------------------------------
// forward: online softmax over key tiles
// ---------------------------------------------------------------------------
template <typename T, int D>
__global__ void __launch_bounds__(NT) simt_fwd_kernel(FwdArgs a) {
  extern __shared__ float sm[];
  constexpr int LD = D + 1, NM = D / 8;
  float* sQ = sm;
  float* sK = sQ + BR * LD;
  float* sV = sK + BC * LD;
  float* oP = sV + BC * LD;
  const int N = a.N, head = blockIdx.y, i0 = blockIdx.x * BR;
  const size_t ho = (size_t)head * N * D;
  const T* Q = (const T*)a.Q + ho;
  const T* K = (const T*)a.K + ho;
  const T* V = (const T*)a.V + ho;
  const int tid = threadIdx.x, r = tid >> 3, q = tid & 7, i = i0 + r;
  load_rows<T, D>(sQ, Q, i0, N);
  float acc[NM];
#pragma unroll
  for (int m = 0; m < NM; ++m) acc[m] = 0.f;
  float mrow = -INFINITY, lrow = 0.f;
  const int jend = a.causal ? min(N, i0 + BR) : N;   // causal: keys up to the block's last row
  for (int j0 = 0; j0 < jend; j0 += BC) {
    __syncthreads();
    load_rows<T, D>(sK, K, j0, N);
    load_rows<T, D>(sV, V, j0, N);
    __syncthreads();
    float s[4] = {0.f, 0.f, 0.f, 0.f};
    for (int k = 0; k < D; ++k) {
      const float qv = sQ[r * LD + k];
#pragma unroll
      for (int m = 0; m < 4; ++m) s[m] = fmaf(qv, sK[(4 * q + m) * LD + k], s[m]);
    }
    float tmax = -INFINITY;
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const int jj = j0 + 4 * q + m;
      s[m] = (jj < N && (!a.causal || jj <= i)) ? a.tau * s[m] : -INFINITY;
      tmax = fmaxf(tmax, s[m]);
    }
    const float mnew = fmaxf(mrow, row_max8(tmax));
    const float scale = expf(mrow - mnew);  // 0 on the first tile
    float psum = 0.f;
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const float p = expf(s[m] - mnew);
      psum += p;
      oP[r * LO + 4 * q + m] = p;
    }
    lrow = lrow * scale + row_sum8(psum);
    mrow = mnew;
#pragma unroll
    for (int m = 0; m < NM; ++m) acc[m] *= scale;
    __syncthreads();
    for (int c = 0; c < BC; ++c) {
      const float p = oP[r * LO + c];
#pragma unroll
      for (int m = 0; m < NM; ++m) acc[m] = fmaf(p, sV[c * LD + q + 8 * m], acc[m]);
    }
  }
  if (i < N) {
    const float inv = 1.f / lrow;
#pragma unroll
    for (int m = 0; m < NM; ++m) a.O[ho + (size_t)i * D + q + 8 * m] = acc[m] * inv;
    if (q == 0) a.L[(size_t)head * N + i] = mrow + logf(lrow);
  }
}

// ---------------------------------------------------------------------------
// first backward, row pass: D = rowsum(dO o O), dQ = tau dS K
// ---------------------------------------------------------------------------
template <typename T, int D>
__global__ void __launch_bounds__(NT) simt_bwd_dq_kernel(BwdArgs a) {
  extern __shared__ float sm[];
  constexpr int LD = D + 1, NM = D / 8;
  float* sQ = sm;
  float* sdO = sQ + BR * LD;
  float* sK = sdO + BR * LD;
  float* sV = sK + BC * LD;
  float* odS = sV + BC * LD;
  const int N = a.N, head = blockIdx.y, i0 = blockIdx.x * BR;
  const size_t ho = (size_t)head * N * D, vo = (size_t)head * N;
  const T* Q = (const T*)a.Q + ho;
  const T* K = (const T*)a.K + ho;
  const T* V = (const T*)a.V + ho;
  const T* dO = (const T*)a.dO + ho;
  const int tid = threadIdx.x, r = tid >> 3, q = tid & 7, i = i0 + r;
  load_rows<T, D>(sQ, Q, i0, N);
  load_rows<T, D>(sdO, dO, i0, N);
  __syncthreads();
  float dpart = 0.f;
  if (i < N) {
#pragma unroll
    for (int m = 0; m < NM; ++m)
      dpart = fmaf(sdO[r * LD + q + 8 * m], a.O[ho + (size_t)i * D + q + 8 * m], dpart);
  }
  const float Dr = row_sum8(dpart);
  const float Lr = (i < N) ? a.L[vo + i] : 0.f;
  if (i < N && q == 0) a.D[vo + i] = Dr;
  float acc[NM];
#pragma unroll
  for (int m = 0; m < NM; ++m) acc[m] = 0.f;
  for (int j0 = 0; j0 < (a.causal ? min(N, i0 + BR) : N); j0 += BC) {
    __syncthreads();
    load_rows<T, D>(sK, K, j0, N);
    load_rows<T, D>(sV, V, j0, N);
    __syncthreads();
    float s[4] = {0.f, 0.f, 0.f, 0.f}, dp[4] = {0.f, 0.f, 0.f, 0.f};
    for (int k = 0; k < D; ++k) {
      const float qv = sQ[r * LD + k], ov = sdO[r * LD + k];
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        s[m] = fmaf(qv, sK[(4 * q + m) * LD + k], s[m]);
        dp[m] = fmaf(ov, sV[(4 * q + m) * LD + k], dp[m]);
      }
    }
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const bool ok = (i < N) && (j0 + 4 * q + m < N) && (!a.causal || j0 + 4 * q + m <= i);
      const float p = ok ? expf(a.tau * s[m] - Lr) : 0.f;
      odS[r * LO + 4 * q + m] = p * (dp[m] - Dr);
    }
    __syncthreads();
    for (int c = 0; c < BC; ++c) {
      const float ds = odS[r * LO + c];
#pragma unroll
      for (int m = 0; m < NM; ++m) acc[m] = fmaf(ds, sK[c * LD + q + 8 * m], acc[m]);
    }
  }
  if (i < N) {
#pragma unroll
    for (int m = 0; m < NM; ++m) a.dQ[ho + (size_t)i * D + q + 8 * m] = a.tau * acc[m];
  }
}

// ---------------------------------------------------------------------------
// first backward, column pass: dV = P^T dO, dK = tau dS^T Q
// ---------------------------------------------------------------------------
template <typename T, int D>
__global__ void __launch_bounds__(NT) simt_bwd_dkdv_kernel(BwdArgs a) {
  extern __shared__ float sm[];
  constexpr int LD = D + 1, NM = D / 8;
  float* sK = sm;
  float* sV = sK + BR * LD;
  float* sQ = sV + BR * LD;
  float* sdO = sQ + BC * LD;
  float* oP = sdO + BC * LD;
  float* odS = oP + BR * LO;
  float* sL = odS + BR * LO;
  float* sD = sL + BC;
  const int N = a.N, head = blockIdx.y, j0 = blockIdx.x * BR;
  const size_t ho = (size_t)head * N * D, vo = (size_t)head * N;
  const T* Q = (const T*)a.Q + ho;
  const T* K = (const T*)a.K + ho;
  const T* V = (const T*)a.V + ho;
  const T* dO = (const T*)a.dO + ho;
  const int tid = threadIdx.x, r = tid >> 3, q = tid & 7, j = j0 + r;
  load_rows<T, D>(sK, K, j0, N);
  load_rows<T, D>(sV, V, j0, N);
  float accK[NM], accV[NM];
#pragma unroll
  for (int m = 0; m < NM; ++m) accK[m] = accV[m] = 0.f;
  for (int c0 = a.causal ? j0 : 0; c0 < N; c0 += BC) {   // causal: queries from the block's first key
    __syncthreads();
    load_rows<T, D>(sQ, Q, c0, N);
    load_rows<T, D>(sdO, dO, c0, N);
    if (tid < BC) {
      const int g = c0 + tid;
      sL[tid] = (g < N) ? a.L[vo + g] : 0.f;
      sD[tid] = (g < N) ? a.D[vo + g] : 0.f;
    }
    __syncthreads();
    float s[4] = {0.f, 0.f, 0.f, 0.f}, dp[4] = {0.f, 0.f, 0.f, 0.f};
    for (int k = 0; k < D; ++k) {
      const float kv = sK[r * LD + k], vv = sV[r * LD + k];
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        s[m] = fmaf(kv, sQ[(4 * q + m) * LD + k], s[m]);
        dp[m] = fmaf(vv, sdO[(4 * q + m) * LD + k], dp[m]);
      }
    }
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const int cc = 4 * q + m;
      const bool ok = (j < N) && (c0 + cc < N) && (!a.causal || c0 + cc >= j);
      const float p = ok ? expf(a.tau * s[m] - sL[cc]) : 0.f;
      oP[r * LO + cc] = p;
      odS[r * LO + cc] = p * (dp[m] - sD[cc]);
    }
    __syncthreads();
    for (int c = 0; c < BC; ++c) {
      const float p = oP[r * LO + c], ds = odS[r * LO + c];
#pragma unroll
      for (int m = 0; m < NM; ++m) {
        accV[m] = fmaf(p, sdO[c * LD + q + 8 * m], accV[m]);
        accK[m] = fmaf(ds, sQ[c * LD + q + 8 * m], accK[m]);
      }
    }
  }
  if (j < N) {
#pragma unroll
    for (int m = 0; m < NM; ++m) {
      a.dK[ho + (size_t)j * D + q + 8 * m] = a.tau * accK[m];
      a.dV[ho + (size_t)j * D + q + 8 * m] = accV[m];
    }
  }
}

// ---------------------------------------------------------------------------
// BoB pass 1 (row blocks): alpha, E and the row-side outputs gQ, gdO.
//   per score element (row i, key j), with Braw = UQ_i.K_j + Q_i.UK_j:
//     P = exp(tau s - L_i), B = tau Braw, t = dP - D_i,
//     dS = P t, X = P (C + B t), PB = P B
//   alpha-free accumulators over keys:
//     U1 = dS UK + X K,  U2 = P K,  W = dS K,  Y = P UV + PB V
//   row scalars: alpha = sum PB, EX = sum X (E = EX + D alpha)
//   row end:  gQ = tau (U1 - EX U2 - alpha W),  gdO = Y - alpha O
// ---------------------------------------------------------------------------
template <typename T, int D>
__global__ void __launch_bounds__(NT) simt_bob_pass1_kernel(BobArgs a) {
  extern __shared__ float sm[];
  constexpr int LD = D + 1, NM = D / 8;
  float* sQ = sm;
  float* sdO = sQ + BR * LD;
  float* sUQ = sdO + BR * LD;
  float* sK = sUQ + BR * LD;
  float* sV = sK + BC * LD;
  float* sUK = sV + BC * LD;
  float* sUV = sUK + BC * LD;
  float* oP = sUV + BC * LD;
  float* odS = oP + BR * LO;
  float* oX = odS + BR * LO;
  float* oPB = oX + BR * LO;
  const int N = a.N, head = blockIdx.y, i0 = blockIdx.x * BR;
  const size_t ho = (size_t)head * N * D, vo = (size_t)head * N;
  const T* Q = (const T*)a.Q + ho;
  const T* K = (const T*)a.K + ho;
  const T* V = (const T*)a.V + ho;
  const T* dO = (const T*)a.dO + ho;
  const T* UQ = (const T*)a.UQ + ho;
  const T* UK = (const T*)a.UK + ho;
  const T* UV = (const T*)a.UV + ho;
  const int tid = threadIdx.x, r = tid >> 3, q = tid & 7, i = i0 + r;
  load_rows<T, D>(sQ, Q, i0, N);
  load_rows<T, D>(sdO, dO, i0, N);
  load_rows<T, D>(sUQ, UQ, i0, N);
  const float Lr = (i < N) ? a.L[vo + i] : 0.f;
  const float Dr = (i < N) ? a.D[vo + i] : 0.f;
  float U1[NM], U2[NM], Wa[NM], Y[NM];
#pragma unroll
  for (int m = 0; m < NM; ++m) U1[m] = U2[m] = Wa[m] = Y[m] = 0.f;
  float alpha_p = 0.f, ex_p = 0.f;
  for (int j0 = 0; j0 < (a.causal ? min(N, i0 + BR) : N); j0 += BC) {
    __syncthreads();
    load_rows<T, D>(sK, K, j0, N);
    load_rows<T, D>(sV, V, j0, N);
    load_rows<T, D>(sUK, UK, j0, N);
    load_rows<T, D>(sUV, UV, j0, N);
    __syncthreads();
    float s[4] = {0.f, 0.f, 0.f, 0.f}, dp[4] = {0.f, 0.f, 0.f, 0.f};
    float cc[4] = {0.f, 0.f, 0.f, 0.f}, bb[4] = {0.f, 0.f, 0.f, 0.f};
    for (int k = 0; k < D; ++k) {
      const float qv = sQ[r * LD + k], ov = sdO[r * LD + k], uqv = sUQ[r * LD + k];
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const int jj = (4 * q + m) * LD + k;
        const float kv = sK[jj];
        s[m] = fmaf(qv, kv, s[m]);
        dp[m] = fmaf(ov, sV[jj], dp[m]);
        cc[m] = fmaf(ov, sUV[jj], cc[m]);
        bb[m] = fmaf(uqv, kv, fmaf(qv, sUK[jj], bb[m]));
      }
    }
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const int jj = 4 * q + m;
      const bool ok = (i < N) && (j0 + jj < N) && (!a.causal || j0 + jj <= i);
      const float p = ok ? expf(a.tau * s[m] - Lr) : 0.f;
      const float b = a.tau * bb[m];
      const float t = dp[m] - Dr;
      const float pb = p * b;
      const float x = p * fmaf(b, t, cc[m]);
      alpha_p += pb;
      ex_p += x;
      oP[r * LO + jj] = p;
      odS[r * LO + jj] = p * t;
      oX[r * LO + jj] = x;
      oPB[r * LO + jj] = pb;
    }
    __syncthreads();
    for (int c = 0; c < BC; ++c) {
      const float p = oP[r * LO + c], ds = odS[r * LO + c], x = oX[r * LO + c], pb = oPB[r * LO + c];
#pragma unroll
      for (int m = 0; m < NM; ++m) {
        const int n = c * LD + q + 8 * m;
        const float kv = sK[n];
        U1[m] = fmaf(ds, sUK[n], fmaf(x, kv, U1[m]));
        U2[m] = fmaf(p, kv, U2[m]);
        Wa[m] = fmaf(ds, kv, Wa[m]);
        Y[m] = fmaf(p, sUV[n], fmaf(pb, sV[n], Y[m]));
      }
    }
  }
  const float alpha = row_sum8(alpha_p);
  const float ex = row_sum8(ex_p);
  if (i < N) {
#pragma unroll
    for (int m = 0; m < NM; ++m) {
      const size_t o = ho + (size_t)i * D + q + 8 * m;
      a.gQ[o] = a.tau * (U1[m] - ex * U2[m] - alpha * Wa[m]);
      a.gdO[o] = Y[m] - alpha * a.O[o];
    }
    if (q == 0) {
      a.ws[2 * (vo + i)] = alpha;
      a.ws[2 * (vo + i) + 1] = fmaf(Dr, alpha, ex);
    }
  }
}

// ---------------------------------------------------------------------------
// BoB pass 2 (key blocks): gK, gV.
//   per element (key j, query i):  P, t = dP - D_i, b' = tau Braw - alpha_i,
//     dS = P t,  Gs = P (C + b' t + alpha_i D_i - E_i),  Gdp = P b'
//   gK = tau (dS^T UQ + Gs^T Q),  gV = Gdp^T dO
// ---------------------------------------------------------------------------
template <typename T, int D>
__global__ void __launch_bounds__(NT) simt_bob_pass2_kernel(BobArgs a) {
  extern __shared__ float sm[];
  constexpr int LD = D + 1, NM = D / 8;
  float* sK = sm;
  float* sV = sK + BR * LD;
  float* sUK = sV + BR * LD;
  float* sUV = sUK + BR * LD;
  float* sQ = sUV + BR * LD;
  float* sdO = sQ + BC * LD;
  float* sUQ = sdO + BC * LD;
  float* odS = sUQ + BC * LD;
  float* oGs = odS + BR * LO;
  float* oGd = oGs + BR * LO;
  float* sL = oGd + BR * LO;
  float* sD = sL + BC;
  float* sA = sD + BC;
  float* sG = sA + BC;
  const int N = a.N, head = blockIdx.y, j0 = blockIdx.x * BR;
  const size_t ho = (size_t)head * N * D, vo = (size_t)head * N;
  const T* Q = (const T*)a.Q + ho;
  const T* K = (const T*)a.K + ho;
  const T* V = (const T*)a.V + ho;
  const T* dO = (const T*)a.dO + ho;
  const T* UQ = (const T*)a.UQ + ho;
  const T* UK = (const T*)a.UK + ho;
  const T* UV = (const T*)a.UV + ho;
  const int tid = threadIdx.x, r = tid >> 3, q = tid & 7, j = j0 + r;
  load_rows<T, D>(sK, K, j0, N);
  load_rows<T, D>(sV, V, j0, N);
  load_rows<T, D>(sUK, UK, j0, N);
  load_rows<T, D>(sUV, UV, j0, N);
  float AK[NM], AV[NM];
#pragma unroll
  for (int m = 0; m < NM; ++m) AK[m] = AV[m] = 0.f;
  for (int c0 = a.causal ? j0 : 0; c0 < N; c0 += BC) {   // causal: queries from the block's first key
    __syncthreads();
    load_rows<T, D>(sQ, Q, c0, N);
    load_rows<T, D>(sdO, dO, c0, N);
    load_rows<T, D>(sUQ, UQ, c0, N);
    if (tid < BC) {
      const int g = c0 + tid;
      const bool ok = g < N;
      const float Dv = ok ? a.D[vo + g] : 0.f;
      const float al = ok ? a.ws[2 * (vo + g)] : 0.f;
      const float E = ok ? a.ws[2 * (vo + g) + 1] : 0.f;
      sL[tid] = ok ? a.L[vo + g] : 0.f;
      sD[tid] = Dv;
      sA[tid] = al;
      sG[tid] = fmaf(al, Dv, -E);  // alpha D - E
    }
    __syncthreads();
    float s[4] = {0.f, 0.f, 0.f, 0.f}, dp[4] = {0.f, 0.f, 0.f, 0.f};
    float cc[4] = {0.f, 0.f, 0.f, 0.f}, bb[4] = {0.f, 0.f, 0.f, 0.f};
    for (int k = 0; k < D; ++k) {
      const float kv = sK[r * LD + k], vv = sV[r * LD + k];
      const float ukv = sUK[r * LD + k], uvv = sUV[r * LD + k];
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const int ii = (4 * q + m) * LD + k;
        const float qv = sQ[ii], ov = sdO[ii];
        s[m] = fmaf(kv, qv, s[m]);
        dp[m] = fmaf(vv, ov, dp[m]);
        cc[m] = fmaf(uvv, ov, cc[m]);
        bb[m] = fmaf(ukv, qv, fmaf(kv, sUQ[ii], bb[m]));
      }
    }
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const int ii = 4 * q + m;
      const bool ok = (j < N) && (c0 + ii < N) && (!a.causal || c0 + ii >= j);
      const float p = ok ? expf(a.tau * s[m] - sL[ii]) : 0.f;
      const float t = dp[m] - sD[ii];
      const float bp = fmaf(a.tau, bb[m], -sA[ii]);
      odS[r * LO + ii] = p * t;
      oGs[r * LO + ii] = p * (fmaf(bp, t, cc[m]) + sG[ii]);
      oGd[r * LO + ii] = p * bp;
    }
    __syncthreads();
    for (int c = 0; c < BC; ++c) {
      const float ds = odS[r * LO + c], gs = oGs[r * LO + c], gd = oGd[r * LO + c];
#pragma unroll
      for (int m = 0; m < NM; ++m) {
        const int n = c * LD + q + 8 * m;
        AK[m] = fmaf(ds, sUQ[n], fmaf(gs, sQ[n], AK[m]));
        AV[m] = fmaf(gd, sdO[n], AV[m]);
      }
    }
  }
  if (j < N) {
#pragma unroll
    for (int m = 0; m < NM; ++m) {
      const size_t o = ho + (size_t)j * D + q + 8 * m;
      a.gK[o] = a.tau * AK[m];
      a.gV[o] = AV[m];
    }
  }
}

template <int D> constexpr size_t fwd_smem() { return sizeof(float) * ((BR + 2 * BC) * (D + 1) + BR * LO); }
template <int D> constexpr size_t dq_smem() { return sizeof(float) * ((2 * BR + 2 * BC) * (D + 1) + BR * LO); }
template <int D> constexpr size_t dkdv_smem() {
  return sizeof(float) * ((2 * BR + 2 * BC) * (D + 1) + 2 * BR * LO + 2 * BC);
}
template <int D> constexpr size_t p1_smem() { return sizeof(float) * ((3 * BR + 4 * BC) * (D + 1) + 4 * BR * LO); }
template <int D> constexpr size_t p2_smem() {
  return sizeof(float) * ((4 * BR + 3 * BC) * (D + 1) + 3 * BR * LO + 4 * BC);
}

template <typename Args, typename Kern>
cudaError_t go(const char* name, Kern kernel, size_t smem, int N, int BH, const Args& args, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((N + BR - 1) / BR, BH);
  prof_begin(s, name);
  kernel<<<grid, NT, smem, s>>>(args);
  prof_end(s);
  return cudaGetLastError();
}

template <typename T, int D>
cudaError_t fwd_t(const FwdArgs& a, cudaStream_t s) {
  return go("simt_fwd", simt_fwd_kernel<T, D>, fwd_smem<D>(), a.N, a.BH, a, s);
}
template <typename T, int D>
cudaError_t bwd_t(const BwdArgs& a, cudaStream_t s) {
  cudaError_t e = go("simt_bwd_dq", simt_bwd_dq_kernel<T, D>, dq_smem<D>(), a.N, a.BH, a, s);
  if (e != cudaSuccess) return e;
  return go("simt_bwd_dkdv", simt_bwd_dkdv_kernel<T, D>, dkdv_smem<D>(), a.N, a.BH, a, s);
}
template <typename T, int D>
cudaError_t bob_t(const BobArgs& a, cudaStream_t s) {
  cudaError_t e = go("simt_bob_pass1", simt_bob_pass1_kernel<T, D>, p1_smem<D>(), a.N, a.BH, a, s);
  if (e != cudaSuccess) return e;
  return go("simt_bob_pass2", simt_bob_pass2_kernel<T, D>, p2_smem<D>(), a.N, a.BH, a, s);
}

}  // namespace

cudaError_t simt_fwd(const FwdArgs& a, const DevCtx&, cudaStream_t s) {
  switch (a.d) {
    case 32: return fwd_t<float, 32>(a, s);
    case 64: return fwd_t<float, 64>(a, s);
    case 96: return fwd_t<float, 96>(a, s);
    default: return fwd_t<float, 128>(a, s);
  }
}
cudaError_t simt_bwd(const BwdArgs& a, const DevCtx&, cudaStream_t s) {
  switch (a.d) {
    case 32: return bwd_t<float, 32>(a, s);
    case 64: return bwd_t<float, 64>(a, s);
    case 96: return bwd_t<float, 96>(a, s);
    default: return bwd_t<float, 128>(a, s);
  }
}
cudaError_t simt_bob(const BobArgs& a, const DevCtx&, cudaStream_t s) {
  switch (a.d) {
    case 32: return bob_t<float, 32>(a, s);
    case 64: return bob_t<float, 64>(a, s);
    case 96: return bob_t<float, 96>(a, s);
    default: return bob_t<float, 128>(a, s);
  }
}

}  // namespace fbob
