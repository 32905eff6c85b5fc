// Tensor-core (tcgen05 + TMEM + TMA) attention forward for bf16 inputs,
// d in {64, 128}, N a multiple of 128: O = softmax(tau Q K^T) V and the
// natural-log row logsumexp L (FlashBoB abstract: the FlashAttention-style
// forward whose outputs the first backward and BoB consume).
//
// A CTA owns two 128-row query blocks (A, B) that share every streamed
// 32-key tile of K and V.  Ten warps: warpgroup 0 (warps 0-3) runs the
// online softmax of block A, warpgroup 1 (warps 4-7) that of block B (thread
// r = TMEM lane r = row r of its block, so row max / sum are thread-local),
// warp 8 issues TMA, warp 9 issues tcgen05.mma and owns TMEM.
// Per tile t and block X:  S_X = Q_X K_t^T (fp32, TMEM);  the group computes
// P = 2^(x - m) with x = tau log2(e) S and its running max m, writes P as bf16
// into TMEM;  O_X += P V_t (A operand from TMEM).  The running max moves only
// when a row's tile max exceeds it by more than 8 (lazy rescale), so P <= 2^8
// stays well inside bf16 and O_X is rescaled in TMEM only then (after the
// group's previous P V product has landed).  O = O_X / l, L = (m + log2 l) ln 2.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>

#include "internal.h"
#include "prof.h"
#include "tc_tile.cuh"

namespace fbob {
namespace {

using namespace tc;
using tile::kBlk;
using tile::kChunk;
using tile::kLog2e;
using tile::kM;
using tile::kT;

constexpr int kThreads = 320;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescale = 8.0f;          // lazy-rescale threshold (log2 units)
constexpr uint64_t kDrainNs = 200000000ull;
constexpr int kNS = 6;                    // K/V stages

struct FwdParams {
  CUtensorMap mQ;          // resident, box {64, 128}
  CUtensorMap mK, mV;      // streamed, box {64, 32}
  float *O, *L;
  int N;
  float tau;
  unsigned int* err;
  unsigned long long wait_ns;
  int stall;
};

template <int D>
struct FwdCfg {
  static constexpr int DC = D / 64;
  static constexpr int RES = 2 * DC * kChunk;    // Q of blocks A and B
  static constexpr int CH = 2 * kBlk;            // [K(32) | V(32)] per 64-column chunk
  static constexpr int STAGE = DC * CH;
  static constexpr int SMEM = RES + kNS * STAGE;
  // TMEM: O_A, O_B, then per block two 32-column S buffers, then per block two
  // 16-column P halves
  static constexpr int S_COL = 2 * D, P_COL = 2 * D + 128;
  static_assert(P_COL + 64 <= 512, "TMEM budget");
  static_assert(SMEM + 1024 <= 232448, "shared memory budget");
};

struct Ctrl {
  uint64_t res_full;
  uint64_t st_full[kNS], st_empty[kNS];
  uint64_t s_full[2][2], s_empty[2][2];   // [block][buffer]
  uint64_t o_full[2][2], o_empty[2][2];   // [block][P half]
  uint64_t acc_full[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1) attn_fwd2_tc(const __grid_constant__ FwdParams p) {
  using C = FwdCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ Ctrl ctrl;
  const int tid = threadIdx.x, warp = tid >> 5;
  const int row0 = blockIdx.x * 2 * kM, head = blockIdx.y;
  const int nblk = (row0 + kM < p.N) ? 2 : 1;   // block B exists unless N is an odd multiple of 128
  const int nt = p.N / kT;
  uint8_t* res = smem;
  uint8_t* stages = res + C::RES;

  if (tid == 0) {
    ctrl.abort_flag = 0;
    mbar_init(&ctrl.res_full, 1);
    for (int s = 0; s < kNS; ++s) {
      mbar_init(&ctrl.st_full[s], 1);
      mbar_init(&ctrl.st_empty[s], nblk);   // one P V commit per block
    }
    for (int x = 0; x < 2; ++x)
      for (int b = 0; b < 2; ++b) {
        mbar_init(&ctrl.s_full[x][b], 1);
        mbar_init(&ctrl.s_empty[x][b], 128);
        mbar_init(&ctrl.o_full[x][b], 128);
        mbar_init(&ctrl.o_empty[x][b], 1);
      }
    mbar_init(&ctrl.acc_full[0], 1);
    mbar_init(&ctrl.acc_full[1], 1);
    mbar_init(&ctrl.drain, 1);
    fence_mbar_init();
    if ((smem_u32(smem) & 1023u) != 0u) {
      ctrl.abort_flag = 1;
      atomicOr(p.err, kErrTimeout);
    }
  }
  if (warp == 9) {
    tmem_alloc(&ctrl.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = ctrl.tmem_base;
  const Waiter wt{&ctrl.abort_flag, p.err, p.wait_ns};
  const bool live = ctrl.abort_flag == 0;

  if (warp == 8) {
    // ------------------------------------------------------------------ TMA
    if (live && (tid & 31) == 0) {
      int issued = 0;
      mbar_arrive_expect_tx(&ctrl.res_full, nblk * C::DC * kChunk);
      for (int x = 0; x < nblk; ++x)
        for (int kc = 0; kc < C::DC; ++kc)
          tma_load_3d(res + (x * C::DC + kc) * kChunk, &p.mQ, &ctrl.res_full, kc * 64, row0 + x * kM, head);
      bool ok = true;
      for (int t = 0; t < nt && ok; ++t) {
        const int s = t % kNS;
        if (!(ok = mbar_wait(&ctrl.st_empty[s], ((t / kNS) & 1) ^ 1, wt))) break;
        if (p.stall && t == 0) continue;  // test hook: nothing will fill this stage
        mbar_arrive_expect_tx(&ctrl.st_full[s], C::STAGE);
        uint8_t* st = stages + s * C::STAGE;
        for (int kc = 0; kc < C::DC; ++kc) {
          tma_load_3d(st + kc * C::CH, &p.mK, &ctrl.st_full[s], kc * 64, t * kT, head);
          tma_load_3d(st + kc * C::CH + kBlk, &p.mV, &ctrl.st_full[s], kc * 64, t * kT, head);
        }
        issued = t + 1;
      }
      if (!ok) {
        mbar_wait_drain(&ctrl.res_full, 0, kDrainNs);
        for (int t = (issued > kNS ? issued - kNS : 0); t < issued; ++t)
          mbar_wait_drain(&ctrl.st_full[t % kNS], (t / kNS) & 1, kDrainNs);
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------------ MMA
    // S(t) for both blocks, and P V per block, each issued in order; the
    // warp issues whatever is ready (P V first), probing without blocking.
    if (live) {  // the whole warp runs the loop; lane 0 issues (elect.sync)
      const uint32_t res_l = desc_lo(smem_u32(res), 16), st_a = smem_u32(stages);
      const uint32_t i32 = idesc_bf16(kM, 32, false, false);
      const uint32_t id = idesc_bf16(kM, D, false, true);
      bool ok = __all_sync(0xffffffffu, mbar_wait(&ctrl.res_full, 0, wt));
      int ns = 0, na[2] = {0, nblk > 1 ? 0 : nt};
      uint64_t idle_since = 0;
      uint32_t idle = 0;  // empty polls since the last check of the clock
      while (ok && (na[0] < nt || na[1] < nt)) {
        bool progressed = false;
        for (int x = 0; x < nblk; ++x) {
          const int u = na[x];
          if (u < ns && mbar_test_w(&ctrl.o_full[x][u & 1], (u >> 1) & 1)) {
            tc_fence_after();
            const uint32_t vmn = desc_lo(st_a + (u % kNS) * C::STAGE, C::CH);
#pragma unroll
            for (int kk = 0; kk < 2; ++kk)
              mma_ts_w(tb + x * D, tb + C::P_COL + x * 32 + (u & 1) * 16 + kk * 8, tile::mn_lo(vmn, 1, kk), id,
                        (u == 0 && kk == 0) ? 0u : 1u);
            mma_commit_w(&ctrl.o_empty[x][u & 1]);
            mma_commit_w(&ctrl.st_empty[u % kNS]);
            if (u + 1 == nt) mma_commit_w(&ctrl.acc_full[x]);
            na[x] = u + 1;
            progressed = true;
          }
        }
        if (ns < nt) {
          const int t = ns;
          bool ready = mbar_test_w(&ctrl.st_full[t % kNS], (t / kNS) & 1);
          if (ready && t >= 2)
            for (int x = 0; x < nblk; ++x) ready = ready && mbar_test_w(&ctrl.s_empty[x][t & 1], ((t - 2) >> 1) & 1);
          if (ready) {
            tc_fence_after();
            const uint32_t klo = desc_lo(st_a + (t % kNS) * C::STAGE, 16);
            for (int x = 0; x < nblk; ++x) {
#pragma unroll
              for (int k = 0; k < D / 16; ++k)
                mma_ss_w(tb + C::S_COL + x * 64 + (t & 1) * 32, tile::res_lo(res_l, x, C::DC, k),
                          tile::kmaj_lo(klo, C::CH, 0, k), i32, k > 0);
              mma_commit_w(&ctrl.s_full[x][t & 1]);
            }
            ++ns;
            progressed = true;
          }
        }
        if (progressed) {
          idle_since = 0;
        } else if ((++idle & 63u) == 0u) {
          // Spin on the probes (a sleep here delays the next issue by far more
          // than the tile period); every 64 empty polls lane 0 reads the clock
          // and the abort flag, and the decision is broadcast so the warp stays
          // converged.
          const uint64_t now = __shfl_sync(0xffffffffu, globaltimer_ns(), 0);
          const int aborting = __shfl_sync(0xffffffffu, *wt.abort, 0);
          if (idle_since == 0) {
            idle_since = now;
          } else if (aborting) {
            ok = false;
          } else if (now - idle_since > wt.limit) {
            if ((tid & 31) == 0) {
              *wt.abort = 1;
              atomicOr(p.err, kErrTimeout);
            }
            ok = false;
          }
        }
      }
      mma_commit_w(&ctrl.drain);
      mbar_wait_drain(&ctrl.drain, 0, kDrainNs);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int x = warp >> 2;                 // block owned by this warpgroup
    const int r = tid & 127;
    const uint32_t lane = (uint32_t)((warp & 3) * 32) << 16;
    const float sc = p.tau * kLog2e;
    float m = -INFINITY, l = 0.f;
    bool ok = live && x < nblk;
    for (int t = 0; t < nt && ok; ++t) {
      const int b = t & 1, k = t >> 1;
      if (!mbar_wait(&ctrl.s_full[x][b], k & 1, wt)) { ok = false; break; }
      tc_fence_after();
      float s[32];
      tmem_ld32(tb + lane + C::S_COL + x * 64 + b * 32, s);
      tc_fence_before();
      mbar_arrive(&ctrl.s_empty[x][b]);
      float mt = -INFINITY;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        s[j] *= sc;
        mt = fmaxf(mt, s[j]);
      }
      if (__any_sync(0xffffffffu, mt > m + kRescale)) {
        const float mn = fmaxf(m, mt);
        if (t > 0) {
          const float scale = tile::ex2(m - mn);
          // the previous P V product of this block must have landed
          if (!mbar_wait(&ctrl.o_empty[x][(t - 1) & 1], ((t - 1) >> 1) & 1, wt)) { ok = false; break; }
          tc_fence_after();
          const uint32_t ob = tb + lane + x * D;
#pragma unroll 1
          for (int c0 = 0; c0 < D; c0 += 16) {
            float o[16];
            tmem_ld16(ob + c0, o);
            uint32_t w[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) w[e] = __float_as_uint(o[e] * scale);
            tmem_st16_nowait(ob + c0, w);
          }
          tmem_st_wait();
          l *= scale;
        }
        m = mn;
      }
      uint32_t w[16];
      float ls = 0.f;
#pragma unroll
      for (int j = 0; j < 32; j += 2) {
        const float p0 = tile::ex2(s[j] - m), p1 = tile::ex2(s[j + 1] - m);
        ls += p0 + p1;
        w[j / 2] = pack_bf16x2(p0, p1);
      }
      l += ls;
      if (!mbar_wait(&ctrl.o_empty[x][b], (k & 1) ^ 1, wt)) { ok = false; break; }
      tmem_st16_nowait(tb + lane + C::P_COL + x * 32 + b * 16, w);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&ctrl.o_full[x][b]);
    }
    if (ok && mbar_wait(&ctrl.acc_full[x], 0, wt)) {
      tc_fence_after();
      const int i = row0 + x * kM + r;
      const size_t ro = ((size_t)head * p.N + i) * D;
      const float inv = 1.f / l;
#pragma unroll 1
      for (int c0 = 0; c0 < D; c0 += 16) {
        float o[16];
        tmem_ld16(tb + lane + x * D + c0, o);
#pragma unroll
        for (int e = 0; e < 16; ++e) o[e] *= inv;
        tile::store16(p.O + ro + c0, o);
      }
      p.L[(size_t)head * p.N + i] = (m + __log2f(l)) * kLn2;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tb, 512);
  }
}

template <int D>
cudaError_t fwd_d(const FwdArgs& a, const DevCtx& c, cudaStream_t s) {
  FwdParams p;
  if (!make_bf16_map(&p.mQ, a.Q, a.BH, a.N, D, kM) || !make_bf16_map(&p.mK, a.K, a.BH, a.N, D, kT) ||
      !make_bf16_map(&p.mV, a.V, a.BH, a.N, D, kT))
    return cudaErrorInvalidValue;
  p.O = a.O;
  p.L = a.L;
  p.N = a.N;
  p.tau = a.tau;
  p.err = c.err;
  p.wait_ns = c.wait_ns;
  p.stall = c.stall;
  auto kernel = attn_fwd2_tc<D>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, FwdCfg<D>::SMEM);
  if (e != cudaSuccess) return e;
  const dim3 grid((a.N + 2 * kM - 1) / (2 * kM), a.BH);
  prof_begin(s, "attn_fwd");
  kernel<<<grid, kThreads, FwdCfg<D>::SMEM, s>>>(p);
  prof_end(s);
  return cudaGetLastError();
}

}  // namespace

cudaError_t tc_fwd(const FwdArgs& a, const DevCtx& c, cudaStream_t s) {
  return a.d == 64 ? fwd_d<64>(a, c, s) : fwd_d<128>(a, c, s);
}

}  // namespace fbob
