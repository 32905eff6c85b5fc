// Tensor-core (tcgen05 + TMEM + TMA) attention forward and first backward for
// bf16 inputs, d in {64, 128}, N a multiple of 128.  They produce O, L and
// D = rowsum(dO o O), the inputs of the two-pass BoB, and dQ, dK, dV.
//
// Source: "FlashBoB: I/O-Efficient Exact Backward-over-Backward for Softmax
// Attention" - the abstract (FlashAttention-style forward and first backward
// that BoB differentiates through).
//
// Same CTA organisation as the BoB kernels: warps 0-3 own TMEM lanes (one tile
// row per thread), warp 4 issues TMA, warp 5 issues tcgen05.mma.
//
// forward (128 query rows per CTA, 32-key tiles): S = Q K^T in TMEM; online
//   softmax in base 2 with a lazy rescale (the running max m only moves when a
//   row's tile max exceeds it by more than 8, so P <= 2^8 stays exact enough in
//   bf16); O += P V in TMEM.  O = O / l, L = (m + log2 l) ln 2.
// first backward:
//   row kernel (128 query rows): D = rowsum(dO o O); S = Q K^T, dP = dO V^T;
//     dS = P (dP - D); dQ += dS K; dQ *= tau.
//   column kernel (128 keys): S^T = K Q^T, dP^T = V dO^T; dV += P^T dO;
//     dK += dS^T Q; dK *= tau.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <math.h>

#include "internal.h"
#include "tc_ptx.cuh"

namespace fbob {
namespace {

using namespace tc;

constexpr int kM = 128;
constexpr int kT = 32;
constexpr int kThreads = 192;
constexpr int kTileBytes = 16384;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr uint64_t kDrainNs = 200000000ull;
constexpr float kRescale = 8.0f;  // lazy-rescale threshold (log2 units)

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

struct Ctrl {
  uint64_t res_full;
  uint64_t stage_full[4], stage_empty[4];
  uint64_t score_full[2], score_empty[2];
  uint64_t op_full[2], op_empty[2];
  uint64_t acc_full, drain;
  uint32_t tmem_base;
  int abort_flag;
};

__device__ __forceinline__ void init_ctrl(Ctrl& c, int ns, int nb, uint32_t stage_empty_count) {
  c.abort_flag = 0;
  mbar_init(&c.res_full, 1);
  for (int s = 0; s < ns; ++s) {
    mbar_init(&c.stage_full[s], 1);
    mbar_init(&c.stage_empty[s], stage_empty_count);
  }
  for (int b = 0; b < nb; ++b) {
    mbar_init(&c.score_full[b], 1);
    mbar_init(&c.score_empty[b], 128);
  }
  for (int h = 0; h < 2; ++h) {
    mbar_init(&c.op_full[h], 128);
    mbar_init(&c.op_empty[h], 1);
  }
  mbar_init(&c.acc_full, 1);
  mbar_init(&c.drain, 1);
  fence_mbar_init();
}

__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void write_op_half(uint32_t tile, uint32_t r, uint32_t h, const uint32_t* w) {
#pragma unroll
  for (int cc = 0; cc < 4; ++cc)
    st_shared_v4(tile + sw128_offset(r, 4 * h + cc), w[4 * cc], w[4 * cc + 1], w[4 * cc + 2], w[4 * cc + 3]);
}

__device__ __forceinline__ void store16(float* dst, const float* v) {
  float4* d4 = reinterpret_cast<float4*>(dst);
#pragma unroll
  for (int q = 0; q < 4; ++q) d4[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float* v) {
  uint32_t r[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) r[i] = __float_as_uint(v[i]);
  tmem_st8(taddr, r);
#pragma unroll
  for (int i = 0; i < 8; ++i) r[i] = __float_as_uint(v[8 + i]);
  tmem_st8(taddr + 8, r);
}

// Common prologue: barriers, TMEM allocation, layout check.
__device__ __forceinline__ void prologue(Ctrl& ctrl, uint8_t* smem, int ns, int nb, uint32_t se_count,
                                         unsigned int* err) {
  const int tid = threadIdx.x, warp = tid >> 5;
  if (tid == 0) {
    init_ctrl(ctrl, ns, nb, se_count);
    if ((smem_u32(smem) & 1023u) != 0u) {
      ctrl.abort_flag = 1;
      atomicOr(err, kErrTimeout);
    }
  }
  if (warp == 5) {
    tmem_alloc(&ctrl.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
}

__device__ __forceinline__ void epilogue_free(const Ctrl& ctrl) {
  tc_fence_before();
  __syncthreads();
  if ((threadIdx.x >> 5) == 5) {
    tc_fence_after();
    tmem_dealloc(ctrl.tmem_base, 512);
  }
}

// Producer give-up path: wait for copies already in flight.
__device__ __forceinline__ void drain_copies(Ctrl& ctrl, int issued, int ns) {
  mbar_wait_drain(&ctrl.res_full, 0, kDrainNs);
  for (int t = (issued > ns ? issued - ns : 0); t < issued; ++t)
    mbar_wait_drain(&ctrl.stage_full[t % ns], (t / ns) & 1, kDrainNs);
}

// ===========================================================================
// forward
// ===========================================================================
struct FwdParams {
  CUtensorMap mQ;          // resident, box {64, 128}
  CUtensorMap mK, mV;      // streamed, box {64, 32}
  float *O, *L;
  int N;
  float tau;
  unsigned int* err;
  unsigned long long wait_ns;
};

template <int D>
struct FwdCfg {
  static constexpr int DC = D / 64;
  static constexpr int STAGE = DC * 8192;  // [K(32) | V(32)] per chunk
  static constexpr int NS = 4;
  static constexpr int RES = DC * kTileBytes;
  static constexpr int OPS = kTileBytes;   // P
  static constexpr int SMEM = RES + NS * STAGE + OPS;
  static constexpr int NB = 2;
  static constexpr int SCOLS = 32;
  static constexpr int A_O = 0;
  static constexpr int ACC_COLS = D;
  static_assert(ACC_COLS + NB * SCOLS <= 512, "TMEM budget");
  static_assert(SMEM + 1024 <= 232448, "shared memory budget");
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1) attn_fwd_tc(const __grid_constant__ FwdParams p) {
  using C = FwdCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ Ctrl ctrl;
  const int tid = threadIdx.x, warp = tid >> 5;
  const int row0 = blockIdx.x * kM, head = blockIdx.y;
  const int ntiles = p.N / kT;
  uint8_t* res = smem;
  uint8_t* stages = res + C::RES;
  uint8_t* ops = stages + C::NS * C::STAGE;
  prologue(ctrl, smem, C::NS, C::NB, 1, p.err);
  const uint32_t tb = ctrl.tmem_base;
  const Waiter wt{&ctrl.abort_flag, p.err, p.wait_ns};
  const bool live = ctrl.abort_flag == 0;

  if (warp == 4) {
    if (live && (tid & 31) == 0) {
      int issued = 0;
      mbar_arrive_expect_tx(&ctrl.res_full, C::RES);
      for (int kc = 0; kc < C::DC; ++kc)
        tma_load_3d(res + kc * kTileBytes, &p.mQ, &ctrl.res_full, kc * 64, row0, head);
      bool ok = true;
      for (int t = 0; t < ntiles && ok; ++t) {
        const int s = t % C::NS;
        if (!(ok = mbar_wait(&ctrl.stage_empty[s], ((t / C::NS) & 1) ^ 1, wt))) break;
        mbar_arrive_expect_tx(&ctrl.stage_full[s], C::STAGE);
        uint8_t* st = stages + s * C::STAGE;
        for (int kc = 0; kc < C::DC; ++kc) {
          tma_load_3d(st + kc * 8192, &p.mK, &ctrl.stage_full[s], kc * 64, t * kT, head);
          tma_load_3d(st + kc * 8192 + 4096, &p.mV, &ctrl.stage_full[s], kc * 64, t * kT, head);
        }
        issued = t + 1;
      }
      if (!ok) drain_copies(ctrl, issued, C::NS);
    }
  } else if (warp == 5) {
    if (live && (tid & 31) == 0) {
      const uint32_t res_a = smem_u32(res), st_a = smem_u32(stages), op_a = smem_u32(ops);
      const uint32_t id_s = idesc_bf16(kM, 32, false, false);
      const uint32_t id_o = idesc_bf16(kM, D, false, true);
      auto score_mmas = [&](int t) {
        const uint32_t sb = st_a + (t % C::NS) * C::STAGE;
        const uint32_t sc = tb + C::ACC_COLS + (t % C::NB) * C::SCOLS;
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint64_t a = sdesc_sw128(res_a + (k >> 2) * kTileBytes + (k & 3) * 32, 16, 1024);
          const uint64_t b = sdesc_sw128(sb + (k >> 2) * 8192 + (k & 3) * 32, 16, 1024);
          mma_ss(sc, a, b, id_s, k > 0);
        }
      };
      auto accum_mmas = [&](int u) {
        const uint32_t sb = st_a + (u % C::NS) * C::STAGE;
        const uint32_t h = u & 1;
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
          const uint64_t a = sdesc_sw128(op_a + h * 64 + kk * 32, 16, 1024);
          const uint64_t b = sdesc_sw128(sb + 4096 + kk * 2048, 8192, 1024);  // V, MN-major
          mma_ss(tb + C::A_O, a, b, id_o, (u == 0 && kk == 0) ? 0u : 1u);
        }
      };
      bool ok = mbar_wait(&ctrl.res_full, 0, wt);
      auto do_accum = [&](int u) {
        if (!mbar_wait(&ctrl.op_full[u & 1], (u >> 1) & 1, wt)) return false;
        tc_fence_after();
        accum_mmas(u);
        mma_commit(&ctrl.op_empty[u & 1]);
        mma_commit(&ctrl.stage_empty[u % C::NS]);
        return true;
      };
      for (int t = 0; t < ntiles && ok; ++t) {
        ok = mbar_wait(&ctrl.stage_full[t % C::NS], (t / C::NS) & 1, wt) &&
             mbar_wait(&ctrl.score_empty[t % C::NB], ((t / C::NB) & 1) ^ 1, wt);
        if (!ok) break;
        tc_fence_after();
        score_mmas(t);
        mma_commit(&ctrl.score_full[t % C::NB]);
        if (t > 0) ok = do_accum(t - 1);
      }
      if (ok) ok = do_accum(ntiles - 1);
      if (ok) mma_commit(&ctrl.acc_full);
      mma_commit(&ctrl.drain);
      mbar_wait_drain(&ctrl.drain, 0, kDrainNs);
    }
  } else {
    const int r = tid, i = row0 + r;
    const float sc = p.tau * kLog2e;
    const uint32_t lane = (uint32_t)(warp * 32) << 16;
    const uint32_t op_a = smem_u32(ops);
    float m = -INFINITY, l = 0.f;
    bool ok = live;
    for (int t = 0; t < ntiles && ok; ++t) {
      const int b = t % C::NB, h = t & 1;
      if (!mbar_wait(&ctrl.score_full[b], (t / C::NB) & 1, wt)) { ok = false; break; }
      tc_fence_after();
      float x[32];
      tmem_ld32(tb + lane + C::ACC_COLS + b * C::SCOLS, x);
      tc_fence_before();
      mbar_arrive(&ctrl.score_empty[b]);
      float mt = -INFINITY;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        x[j] *= sc;
        mt = fmaxf(mt, x[j]);
      }
      // lazy rescale: only when some row of this warp grew by more than 2^8
      const bool grow = mt > m + kRescale;
      if (__any_sync(0xffffffffu, grow)) {
        const float mn = fmaxf(m, mt);
        const float scale = (t == 0) ? 0.f : ex2(m - mn);
        if (t > 0) {
          // every earlier P V product must have landed before O is rescaled
          if (!mbar_wait(&ctrl.op_empty[(t - 1) & 1], ((t - 1) >> 1) & 1, wt)) { ok = false; break; }
          tc_fence_after();
          const uint32_t ob = tb + lane + C::A_O;
#pragma unroll 1
          for (int c0 = 0; c0 < D; c0 += 16) {
            float o[16];
            tmem_ld16(ob + c0, o);
#pragma unroll
            for (int e = 0; e < 16; ++e) o[e] *= scale;
            tmem_st16(ob + c0, o);
          }
          tc_fence_before();
        }
        l *= scale;
        m = mn;
      }
      uint32_t w[16];
      float ls = 0.f;
#pragma unroll
      for (int j = 0; j < 32; j += 2) {
        const float p0 = ex2(x[j] - m), p1 = ex2(x[j + 1] - m);
        ls += p0 + p1;
        w[j / 2] = pack_bf16x2(p0, p1);
      }
      l += ls;
      if (!mbar_wait(&ctrl.op_empty[h], ((t >> 1) & 1) ^ 1, wt)) { ok = false; break; }
      write_op_half(op_a, r, h, w);
      fence_proxy_async_smem();
      mbar_arrive(&ctrl.op_full[h]);
    }
    if (ok && mbar_wait(&ctrl.acc_full, 0, wt)) {
      tc_fence_after();
      const size_t ro = ((size_t)head * p.N + i) * D;
      const float inv = 1.f / l;
#pragma unroll 1
      for (int c0 = 0; c0 < D; c0 += 16) {
        float o[16];
        tmem_ld16(tb + lane + C::A_O + c0, o);
#pragma unroll
        for (int e = 0; e < 16; ++e) o[e] *= inv;
        store16(p.O + ro + c0, o);
      }
      p.L[(size_t)head * p.N + i] = (m + __log2f(l)) * kLn2;
    }
  }
  epilogue_free(ctrl);
}

// ===========================================================================
// first backward, row kernel: D and dQ
// ===========================================================================
struct DqParams {
  CUtensorMap mQ, mdO;     // resident
  CUtensorMap mK, mV;      // streamed
  const float *O, *L;
  const __nv_bfloat16* dO;
  float *dQ, *D;
  int N;
  float tau;
  unsigned int* err;
  unsigned long long wait_ns;
};

template <int D>
struct DqCfg {
  static constexpr int DC = D / 64;
  static constexpr int STAGE = DC * 8192;  // [K(32) | V(32)]
  static constexpr int NS = 4;
  static constexpr int RES = 2 * DC * kTileBytes;
  static constexpr int OPS = kTileBytes;   // dS
  static constexpr int SMEM = RES + NS * STAGE + OPS;
  static constexpr int NB = 2;
  static constexpr int SCOLS = 64;         // [S | dP]
  static constexpr int ACC_COLS = D;
  static_assert(ACC_COLS + NB * SCOLS <= 512, "TMEM budget");
  static_assert(SMEM + 1024 <= 232448, "shared memory budget");
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1) attn_bwd_dq_tc(const __grid_constant__ DqParams p) {
  using C = DqCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ Ctrl ctrl;
  const int tid = threadIdx.x, warp = tid >> 5;
  const int row0 = blockIdx.x * kM, head = blockIdx.y;
  const int ntiles = p.N / kT;
  uint8_t* res = smem;
  uint8_t* stages = res + C::RES;
  uint8_t* ops = stages + C::NS * C::STAGE;
  prologue(ctrl, smem, C::NS, C::NB, 1, p.err);
  const uint32_t tb = ctrl.tmem_base;
  const Waiter wt{&ctrl.abort_flag, p.err, p.wait_ns};
  const bool live = ctrl.abort_flag == 0;

  if (warp == 4) {
    if (live && (tid & 31) == 0) {
      int issued = 0;
      mbar_arrive_expect_tx(&ctrl.res_full, C::RES);
      for (int kc = 0; kc < C::DC; ++kc) {
        tma_load_3d(res + kc * kTileBytes, &p.mQ, &ctrl.res_full, kc * 64, row0, head);
        tma_load_3d(res + (C::DC + kc) * kTileBytes, &p.mdO, &ctrl.res_full, kc * 64, row0, head);
      }
      bool ok = true;
      for (int t = 0; t < ntiles && ok; ++t) {
        const int s = t % C::NS;
        if (!(ok = mbar_wait(&ctrl.stage_empty[s], ((t / C::NS) & 1) ^ 1, wt))) break;
        mbar_arrive_expect_tx(&ctrl.stage_full[s], C::STAGE);
        uint8_t* st = stages + s * C::STAGE;
        for (int kc = 0; kc < C::DC; ++kc) {
          tma_load_3d(st + kc * 8192, &p.mK, &ctrl.stage_full[s], kc * 64, t * kT, head);
          tma_load_3d(st + kc * 8192 + 4096, &p.mV, &ctrl.stage_full[s], kc * 64, t * kT, head);
        }
        issued = t + 1;
      }
      if (!ok) drain_copies(ctrl, issued, C::NS);
    }
  } else if (warp == 5) {
    if (live && (tid & 31) == 0) {
      const uint32_t res_a = smem_u32(res), st_a = smem_u32(stages), op_a = smem_u32(ops);
      const uint32_t id_s = idesc_bf16(kM, 32, false, false);
      const uint32_t id_a = idesc_bf16(kM, D, false, true);
      auto score_mmas = [&](int t) {
        const uint32_t sb = st_a + (t % C::NS) * C::STAGE;
        const uint32_t sc = tb + C::ACC_COLS + (t % C::NB) * C::SCOLS;
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t ko = (k >> 2) * kTileBytes + (k & 3) * 32;
          const uint32_t so = (k >> 2) * 8192 + (k & 3) * 32;
          mma_ss(sc, sdesc_sw128(res_a + ko, 16, 1024), sdesc_sw128(sb + so, 16, 1024), id_s, k > 0);
          mma_ss(sc + 32, sdesc_sw128(res_a + C::DC * kTileBytes + ko, 16, 1024),
                 sdesc_sw128(sb + so + 4096, 16, 1024), id_s, k > 0);
        }
      };
      auto accum_mmas = [&](int u) {
        const uint32_t sb = st_a + (u % C::NS) * C::STAGE;
        const uint32_t h = u & 1;
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
          const uint64_t a = sdesc_sw128(op_a + h * 64 + kk * 32, 16, 1024);
          const uint64_t b = sdesc_sw128(sb + kk * 2048, 8192, 1024);  // K, MN-major
          mma_ss(tb, a, b, id_a, (u == 0 && kk == 0) ? 0u : 1u);
        }
      };
      bool ok = mbar_wait(&ctrl.res_full, 0, wt);
      auto do_accum = [&](int u) {
        if (!mbar_wait(&ctrl.op_full[u & 1], (u >> 1) & 1, wt)) return false;
        tc_fence_after();
        accum_mmas(u);
        mma_commit(&ctrl.op_empty[u & 1]);
        mma_commit(&ctrl.stage_empty[u % C::NS]);
        return true;
      };
      for (int t = 0; t < ntiles && ok; ++t) {
        ok = mbar_wait(&ctrl.stage_full[t % C::NS], (t / C::NS) & 1, wt) &&
             mbar_wait(&ctrl.score_empty[t % C::NB], ((t / C::NB) & 1) ^ 1, wt);
        if (!ok) break;
        tc_fence_after();
        score_mmas(t);
        mma_commit(&ctrl.score_full[t % C::NB]);
        if (t > 0) ok = do_accum(t - 1);
      }
      if (ok) ok = do_accum(ntiles - 1);
      if (ok) mma_commit(&ctrl.acc_full);
      mma_commit(&ctrl.drain);
      mbar_wait_drain(&ctrl.drain, 0, kDrainNs);
    }
  } else {
    const int r = tid, i = row0 + r;
    const size_t vo = (size_t)head * p.N + i;
    const size_t ro = vo * D;
    // D_i = rowsum(dO o O) for this thread's row
    float Di = 0.f;
    {
      const uint4* g = reinterpret_cast<const uint4*>(p.dO + ro);
      const float4* o = reinterpret_cast<const float4*>(p.O + ro);
#pragma unroll 4
      for (int c = 0; c < D / 8; ++c) {
        const uint4 u = g[c];
        const float4 o0 = o[2 * c], o1 = o[2 * c + 1];
        const __nv_bfloat162* hb = reinterpret_cast<const __nv_bfloat162*>(&u);
        const float2 a0 = __bfloat1622float2(hb[0]), a1 = __bfloat1622float2(hb[1]);
        const float2 a2 = __bfloat1622float2(hb[2]), a3 = __bfloat1622float2(hb[3]);
        Di = fmaf(a0.x, o0.x, Di);
        Di = fmaf(a0.y, o0.y, Di);
        Di = fmaf(a1.x, o0.z, Di);
        Di = fmaf(a1.y, o0.w, Di);
        Di = fmaf(a2.x, o1.x, Di);
        Di = fmaf(a2.y, o1.y, Di);
        Di = fmaf(a3.x, o1.z, Di);
        Di = fmaf(a3.y, o1.w, Di);
      }
    }
    p.D[vo] = Di;
    const float nL = -p.L[vo] * kLog2e;
    const float sc = p.tau * kLog2e;
    const uint32_t lane = (uint32_t)(warp * 32) << 16;
    const uint32_t op_a = smem_u32(ops);
    bool ok = live;
    for (int t = 0; t < ntiles && ok; ++t) {
      const int b = t % C::NB, h = t & 1;
      if (!mbar_wait(&ctrl.score_full[b], (t / C::NB) & 1, wt)) { ok = false; break; }
      tc_fence_after();
      const uint32_t sbase = tb + lane + C::ACC_COLS + b * C::SCOLS;
      uint32_t w[16];
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        float s[16], dp[16];
        tmem_ld16(sbase + q * 16, s);
        tmem_ld16(sbase + 32 + q * 16, dp);
#pragma unroll
        for (int j = 0; j < 16; j += 2) {
          const float p0 = ex2(fmaf(s[j], sc, nL)), p1 = ex2(fmaf(s[j + 1], sc, nL));
          w[q * 8 + j / 2] = pack_bf16x2(p0 * (dp[j] - Di), p1 * (dp[j + 1] - Di));
        }
      }
      tc_fence_before();
      mbar_arrive(&ctrl.score_empty[b]);
      if (!mbar_wait(&ctrl.op_empty[h], ((t >> 1) & 1) ^ 1, wt)) { ok = false; break; }
      write_op_half(op_a, r, h, w);
      fence_proxy_async_smem();
      mbar_arrive(&ctrl.op_full[h]);
    }
    if (ok && mbar_wait(&ctrl.acc_full, 0, wt)) {
      tc_fence_after();
#pragma unroll 1
      for (int c0 = 0; c0 < D; c0 += 16) {
        float v[16];
        tmem_ld16(tb + lane + c0, v);
#pragma unroll
        for (int e = 0; e < 16; ++e) v[e] *= p.tau;
        store16(p.dQ + ro + c0, v);
      }
    }
  }
  epilogue_free(ctrl);
}

// ===========================================================================
// first backward, column kernel: dK, dV
// ===========================================================================
struct DkvParams {
  CUtensorMap mK, mV;      // resident
  CUtensorMap mQ, mdO;     // streamed
  const float *L, *D;
  float *dK, *dV;
  int N;
  float tau;
  unsigned int* err;
  unsigned long long wait_ns;
};

template <int D>
struct DkvCfg {
  static constexpr int DC = D / 64;
  static constexpr int STAGE_T = DC * 8192;   // [Q(32) | dO(32)]
  static constexpr int STAGE_TX = STAGE_T + 256;
  static constexpr int STAGE = STAGE_T + 1024;
  static constexpr int NS = 4;
  static constexpr int RES = 2 * DC * kTileBytes;
  static constexpr int OPS = 2 * kTileBytes;  // P, dS
  static constexpr int SMEM = RES + NS * STAGE + OPS;
  static constexpr int NB = 2;
  static constexpr int SCOLS = 64;            // [S^T | dP^T]
  static constexpr int A_K = 0, A_V = D;
  static constexpr int ACC_COLS = 2 * D;
  static_assert(ACC_COLS + NB * SCOLS <= 512, "TMEM budget");
  static_assert(SMEM + 1024 <= 232448, "shared memory budget");
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1) attn_bwd_dkdv_tc(const __grid_constant__ DkvParams p) {
  using C = DkvCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ Ctrl ctrl;
  const int tid = threadIdx.x, warp = tid >> 5;
  const int col0 = blockIdx.x * kM, head = blockIdx.y;
  const int ntiles = p.N / kT;
  uint8_t* res = smem;
  uint8_t* stages = res + C::RES;
  uint8_t* ops = stages + C::NS * C::STAGE;
  prologue(ctrl, smem, C::NS, C::NB, 1 + 4, p.err);
  const uint32_t tb = ctrl.tmem_base;
  const Waiter wt{&ctrl.abort_flag, p.err, p.wait_ns};
  const bool live = ctrl.abort_flag == 0;

  if (warp == 4) {
    if (live && (tid & 31) == 0) {
      int issued = 0;
      mbar_arrive_expect_tx(&ctrl.res_full, C::RES);
      for (int kc = 0; kc < C::DC; ++kc) {
        tma_load_3d(res + kc * kTileBytes, &p.mK, &ctrl.res_full, kc * 64, col0, head);
        tma_load_3d(res + (C::DC + kc) * kTileBytes, &p.mV, &ctrl.res_full, kc * 64, col0, head);
      }
      bool ok = true;
      const size_t vbase = (size_t)head * p.N;
      for (int t = 0; t < ntiles && ok; ++t) {
        const int s = t % C::NS;
        if (!(ok = mbar_wait(&ctrl.stage_empty[s], ((t / C::NS) & 1) ^ 1, wt))) break;
        mbar_arrive_expect_tx(&ctrl.stage_full[s], C::STAGE_TX);
        uint8_t* st = stages + s * C::STAGE;
        for (int kc = 0; kc < C::DC; ++kc) {
          tma_load_3d(st + kc * 8192, &p.mQ, &ctrl.stage_full[s], kc * 64, t * kT, head);
          tma_load_3d(st + kc * 8192 + 4096, &p.mdO, &ctrl.stage_full[s], kc * 64, t * kT, head);
        }
        bulk_load(st + C::STAGE_T, p.L + vbase + t * kT, 128, &ctrl.stage_full[s]);
        bulk_load(st + C::STAGE_T + 128, p.D + vbase + t * kT, 128, &ctrl.stage_full[s]);
        issued = t + 1;
      }
      if (!ok) drain_copies(ctrl, issued, C::NS);
    }
  } else if (warp == 5) {
    if (live && (tid & 31) == 0) {
      const uint32_t res_a = smem_u32(res), st_a = smem_u32(stages), op_a = smem_u32(ops);
      const uint32_t id_s = idesc_bf16(kM, 32, false, false);
      const uint32_t id_a = idesc_bf16(kM, D, false, true);
      auto score_mmas = [&](int t) {
        const uint32_t sb = st_a + (t % C::NS) * C::STAGE;
        const uint32_t sc = tb + C::ACC_COLS + (t % C::NB) * C::SCOLS;
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t ko = (k >> 2) * kTileBytes + (k & 3) * 32;
          const uint32_t so = (k >> 2) * 8192 + (k & 3) * 32;
          mma_ss(sc, sdesc_sw128(res_a + ko, 16, 1024), sdesc_sw128(sb + so, 16, 1024), id_s, k > 0);
          mma_ss(sc + 32, sdesc_sw128(res_a + C::DC * kTileBytes + ko, 16, 1024),
                 sdesc_sw128(sb + so + 4096, 16, 1024), id_s, k > 0);
        }
      };
      auto accum_mmas = [&](int u) {
        const uint32_t sb = st_a + (u % C::NS) * C::STAGE;
        const uint32_t h = u & 1;
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
          const uint32_t acc0 = (u == 0 && kk == 0) ? 0u : 1u;
          const uint64_t aP = sdesc_sw128(op_a + h * 64 + kk * 32, 16, 1024);
          const uint64_t adS = sdesc_sw128(op_a + kTileBytes + h * 64 + kk * 32, 16, 1024);
          mma_ss(tb + C::A_V, aP, sdesc_sw128(sb + 4096 + kk * 2048, 8192, 1024), id_a, acc0);  // P^T dO
          mma_ss(tb + C::A_K, adS, sdesc_sw128(sb + kk * 2048, 8192, 1024), id_a, acc0);        // dS^T Q
        }
      };
      bool ok = mbar_wait(&ctrl.res_full, 0, wt);
      auto do_accum = [&](int u) {
        if (!mbar_wait(&ctrl.op_full[u & 1], (u >> 1) & 1, wt)) return false;
        tc_fence_after();
        accum_mmas(u);
        mma_commit(&ctrl.op_empty[u & 1]);
        mma_commit(&ctrl.stage_empty[u % C::NS]);
        return true;
      };
      for (int t = 0; t < ntiles && ok; ++t) {
        ok = mbar_wait(&ctrl.stage_full[t % C::NS], (t / C::NS) & 1, wt) &&
             mbar_wait(&ctrl.score_empty[t % C::NB], ((t / C::NB) & 1) ^ 1, wt);
        if (!ok) break;
        tc_fence_after();
        score_mmas(t);
        mma_commit(&ctrl.score_full[t % C::NB]);
        if (t > 0) ok = do_accum(t - 1);
      }
      if (ok) ok = do_accum(ntiles - 1);
      if (ok) mma_commit(&ctrl.acc_full);
      mma_commit(&ctrl.drain);
      mbar_wait_drain(&ctrl.drain, 0, kDrainNs);
    }
  } else {
    const int r = tid, j = col0 + r;
    const float sc = p.tau * kLog2e;
    const uint32_t lane = (uint32_t)(warp * 32) << 16;
    const uint32_t op_a = smem_u32(ops);
    bool ok = live;
    for (int t = 0; t < ntiles && ok; ++t) {
      const int b = t % C::NB, h = t & 1, s = t % C::NS;
      if (!mbar_wait(&ctrl.stage_full[s], (t / C::NS) & 1, wt) ||
          !mbar_wait(&ctrl.score_full[b], (t / C::NB) & 1, wt)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const float* vec = reinterpret_cast<const float*>(stages + s * C::STAGE + C::STAGE_T);
      const uint32_t sbase = tb + lane + C::ACC_COLS + b * C::SCOLS;
      uint32_t wP[16], wdS[16];
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        float s_[16], dp[16];
        tmem_ld16(sbase + q * 16, s_);
        tmem_ld16(sbase + 32 + q * 16, dp);
#pragma unroll
        for (int c = 0; c < 16; c += 2) {
          const int ii = q * 16 + c;
          const float p0 = ex2(fmaf(s_[c], sc, -vec[ii] * kLog2e));
          const float p1 = ex2(fmaf(s_[c + 1], sc, -vec[ii + 1] * kLog2e));
          wP[q * 8 + c / 2] = pack_bf16x2(p0, p1);
          wdS[q * 8 + c / 2] = pack_bf16x2(p0 * (dp[c] - vec[32 + ii]), p1 * (dp[c + 1] - vec[32 + ii + 1]));
        }
      }
      tc_fence_before();
      mbar_arrive(&ctrl.score_empty[b]);
      __syncwarp();
      if ((tid & 31) == 0) mbar_arrive(&ctrl.stage_empty[s]);
      if (!mbar_wait(&ctrl.op_empty[h], ((t >> 1) & 1) ^ 1, wt)) { ok = false; break; }
      write_op_half(op_a, r, h, wP);
      write_op_half(op_a + kTileBytes, r, h, wdS);
      fence_proxy_async_smem();
      mbar_arrive(&ctrl.op_full[h]);
    }
    if (ok && mbar_wait(&ctrl.acc_full, 0, wt)) {
      tc_fence_after();
      const size_t ro = ((size_t)head * p.N + j) * D;
#pragma unroll 1
      for (int c0 = 0; c0 < D; c0 += 16) {
        float k_[16], v[16];
        tmem_ld16(tb + lane + C::A_K + c0, k_);
        tmem_ld16(tb + lane + C::A_V + c0, v);
#pragma unroll
        for (int e = 0; e < 16; ++e) k_[e] *= p.tau;
        store16(p.dK + ro + c0, k_);
        store16(p.dV + ro + c0, v);
      }
    }
  }
  epilogue_free(ctrl);
}

// ===========================================================================
// host side
// ===========================================================================
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    cudaDriverEntryPointQueryResult q;
    void* f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }
  return fn;
}

bool make_map(CUtensorMap* m, const void* base, int BH, int N, int D, int rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)N, (cuuint64_t)BH};
  cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)N * D * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename K, typename Params>
cudaError_t launch(K kernel, int smem, dim3 grid, const Params& prm, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kernel<<<grid, kThreads, smem, s>>>(prm);
  return cudaGetLastError();
}

template <int D>
cudaError_t fwd_d(const FwdArgs& a, const DevCtx& c, cudaStream_t s) {
  FwdParams p;
  if (!make_map(&p.mQ, a.Q, a.BH, a.N, D, kM) || !make_map(&p.mK, a.K, a.BH, a.N, D, kT) ||
      !make_map(&p.mV, a.V, a.BH, a.N, D, kT))
    return cudaErrorInvalidValue;
  p.O = a.O;
  p.L = a.L;
  p.N = a.N;
  p.tau = a.tau;
  p.err = c.err;
  p.wait_ns = c.wait_ns;
  return launch(attn_fwd_tc<D>, FwdCfg<D>::SMEM, dim3(a.N / kM, a.BH), p, s);
}

template <int D>
cudaError_t bwd_d(const BwdArgs& a, const DevCtx& c, cudaStream_t s) {
  DqParams q;
  if (!make_map(&q.mQ, a.Q, a.BH, a.N, D, kM) || !make_map(&q.mdO, a.dO, a.BH, a.N, D, kM) ||
      !make_map(&q.mK, a.K, a.BH, a.N, D, kT) || !make_map(&q.mV, a.V, a.BH, a.N, D, kT))
    return cudaErrorInvalidValue;
  q.O = a.O;
  q.L = a.L;
  q.dO = static_cast<const __nv_bfloat16*>(a.dO);
  q.dQ = a.dQ;
  q.D = a.D;
  q.N = a.N;
  q.tau = a.tau;
  q.err = c.err;
  q.wait_ns = c.wait_ns;
  cudaError_t e = launch(attn_bwd_dq_tc<D>, DqCfg<D>::SMEM, dim3(a.N / kM, a.BH), q, s);
  if (e != cudaSuccess) return e;
  DkvParams k;
  if (!make_map(&k.mK, a.K, a.BH, a.N, D, kM) || !make_map(&k.mV, a.V, a.BH, a.N, D, kM) ||
      !make_map(&k.mQ, a.Q, a.BH, a.N, D, kT) || !make_map(&k.mdO, a.dO, a.BH, a.N, D, kT))
    return cudaErrorInvalidValue;
  k.L = a.L;
  k.D = a.D;
  k.dK = a.dK;
  k.dV = a.dV;
  k.N = a.N;
  k.tau = a.tau;
  k.err = c.err;
  k.wait_ns = c.wait_ns;
  return launch(attn_bwd_dkdv_tc<D>, DkvCfg<D>::SMEM, dim3(a.N / kM, a.BH), k, s);
}

}  // namespace

cudaError_t tc_fwd(const FwdArgs& a, const DevCtx& c, cudaStream_t s) {
  return a.d == 64 ? fwd_d<64>(a, c, s) : fwd_d<128>(a, c, s);
}
cudaError_t tc_bwd(const BwdArgs& a, const DevCtx& c, cudaStream_t s) {
  return a.d == 64 ? bwd_d<64>(a, c, s) : bwd_d<128>(a, c, s);
}

}  // namespace fbob
