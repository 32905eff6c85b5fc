// Tensor-core (tcgen05 + TMEM + TMA) kernels of the two-pass BoB for bf16
// inputs, d in {64, 128}, N a multiple of 128.
//
// Source: "FlashBoB: I/O-Efficient Exact Backward-over-Backward for Softmax
// Attention", evolve.pub review - Summary / Key claims (two-pass schedule,
// only alpha and E cross the pass boundary, no N x N tensor in HBM; paper
// Prop. 4.1 and Algorithm 1) and Strengths (alpha-free accumulators corrected
// after the row reduction; transfer ledger of Theorem 4.3).
//
// Per (query row i, key j), with Braw = UQ_i.K_j + Q_i.UK_j:
//   P = exp(tau S - L_i), B = tau Braw, dP = dO_i.V_j, C = dO_i.UV_j,
//   t = dP - D_i, dS = P t, X = P (C + B t), PB = P B
// Pass 1 (block of 128 query rows, loop over 32-key tiles):
//   U1 += dS UK + X K, U2 += P K, W += dS K, Y += P UV + PB V
//   alpha = sum_j PB, EX = sum_j X, E = EX + D alpha
//   gQ = tau (U1 - EX U2 - alpha W), gdO = Y - alpha O
// Pass 2 (block of 128 keys, loop over 32-query tiles):
//   b' = B - alpha_i, Gs = P (C + b' t + alpha_i D_i - E_i), Gdp = P b'
//   gK = tau (dS^T UQ + Gs^T Q), gV = Gdp^T dO
//
// CTA = 6 warps: warps 0-3 own TMEM lanes 0-127 (one tile row per thread:
// softmax-type row sums need no shuffles), warp 4 issues TMA, warp 5 issues
// tcgen05.mma (one thread) and owns the TMEM allocation.  Score tiles are
// computed into TMEM, turned into bf16 operands in registers and written to
// 128B-swizzled shared memory, and consumed by the accumulator MMAs; the
// accumulators stay in TMEM for the whole loop.
//
// TMEM budget (512 columns of 128 lanes x fp32): the d=64 pass 1 holds all four
// accumulators (4 x 64) and two score buffers ([S|B|dP|C] = 128 columns each).
// At d=128 the four accumulators alone fill TMEM, so pass 1 runs as two CTA
// kinds over the same row blocks: the Q side (U1, U2, W: 384 columns + one
// score buffer) writes gQ and alpha/E, the dO side (Y) recomputes S and B and
// writes gdO.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "internal.h"
#include "tc_ptx.cuh"

namespace fbob {
namespace {

using namespace tc;

constexpr int kM = 128;         // rows per CTA (TMEM lanes)
constexpr int kT = 32;          // streamed rows per tile
constexpr int kThreads = 192;   // 4 elementwise warps + TMA warp + MMA warp
constexpr int kTileBytes = 16384;  // 128 rows x 128 B (one 64-column chunk)
constexpr float kLog2e = 1.4426950408889634f;
constexpr uint64_t kDrainNs = 200000000ull;  // 0.2 s for the give-up path

enum Role { kBoth = 0, kQSide = 1, kDoSide = 2 };

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

struct P1Params {
  CUtensorMap mQ, mdO, mUQ;        // resident, box {64, 128}
  CUtensorMap mK, mUK, mV, mUV;    // streamed, box {64, 32}
  const float *L, *D, *O;
  float *gQ, *gdO, *ws;
  int N;
  float tau;
  unsigned int* err;
  unsigned long long wait_ns;
};

struct P2Params {
  CUtensorMap mK, mV, mUK, mUV;    // resident, box {64, 128}
  CUtensorMap mQ, mUQ, mdO;        // streamed, box {64, 32}
  const float *L, *D, *ws;
  float *gK, *gV;
  int N;
  float tau;
  unsigned int* err;
  unsigned long long wait_ns;
};

template <int D, int ROLE>
struct P1Cfg {
  static constexpr int DC = D / 64;
  static constexpr bool kQ = ROLE != kDoSide;   // gQ, alpha, E
  static constexpr bool kDo = ROLE != kQSide;   // gdO
  static constexpr int NRES = kQ ? 3 : 2;       // Q, UQ, dO
  static constexpr int NOPS = 1 + (kQ ? 2 : 0) + (kDo ? 1 : 0);  // P, dS, X, PB
  static constexpr int NACC = (kQ ? 3 : 0) + (kDo ? 1 : 0);
  static constexpr int SCOLS = kQ ? 128 : 64;   // [S|B|dP|C] or [S|B]
  static constexpr int NB = (ROLE == kQSide) ? 1 : 2;
  static constexpr int STAGE = DC * kTileBytes;  // K, UK, V, UV: 32 rows each per chunk
  static constexpr int NS = (ROLE == kQSide) ? 2 : (ROLE == kBoth ? 4 : 3);
  static constexpr int RES = NRES * DC * kTileBytes;
  static constexpr int OPS = NOPS * kTileBytes;
  static constexpr int SMEM = RES + NS * STAGE + OPS;
  static constexpr int ACC_COLS = NACC * D;
  static_assert(ACC_COLS + NB * SCOLS <= 512, "TMEM budget");
  static_assert(SMEM + 1024 <= 232448, "shared memory budget (1 KB static)");
  // resident slots
  static constexpr int R_Q = 0, R_UQ = 1, R_DO = 2;
  // operand slots
  static constexpr int O_P = 0, O_DS = 1, O_X = 2, O_PB = kQ ? 3 : 1;
  // accumulator columns
  static constexpr int A_U1 = 0, A_U2 = D, A_W = 2 * D, A_Y = kQ ? 3 * D : 0;
};

template <int D>
struct P2Cfg {
  static constexpr int DC = D / 64;
  static constexpr int NRES = 4;                 // K, V, UK, UV
  static constexpr int NOPS = 3;                 // dS, Gs, Gdp
  static constexpr int SCOLS = 128;              // [S|B|dP|C]
  static constexpr int NB = 2;
  static constexpr int VEC = 512;                // L, D (128 B each), alpha/E (256 B)
  static constexpr int STAGE_T = DC * 12288;     // Q, UQ, dO: 32 rows each per chunk
  static constexpr int STAGE_TX = STAGE_T + VEC; // bytes landing per stage
  static constexpr int STAGE = STAGE_T + 1024;   // stride keeps stages 1024-byte aligned
  static constexpr int NS = 2;
  static constexpr int RES = NRES * DC * kTileBytes;
  static constexpr int OPS = NOPS * kTileBytes;
  static constexpr int SMEM = RES + OPS + NS * STAGE;
  static constexpr int ACC_COLS = 2 * D;
  static_assert(ACC_COLS + NB * SCOLS <= 512, "TMEM budget");
  static_assert(SMEM + 1024 <= 232448, "shared memory budget (1 KB static)");
  static constexpr int R_K = 0, R_V = 1, R_UK = 2, R_UV = 3;
  static constexpr int O_DS = 0, O_GS = 1, O_GD = 2;
  static constexpr int A_K = 0, A_V = D;
};

// Shared control block (static shared memory).
struct Ctrl {
  uint64_t res_full;
  uint64_t stage_full[4], stage_empty[4];
  uint64_t score_full[2], score_empty[2];
  uint64_t op_full[2], op_empty[2];
  uint64_t acc_full, drain;
  uint32_t tmem_base;
  int abort_flag;
};

__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Write 32 packed bf16 (16 words) of this thread's row r into columns
// [32h, 32h+32) of a 128B-swizzled [128][64] operand tile.
__device__ __forceinline__ void write_op_half(uint32_t tile, uint32_t r, uint32_t h, const uint32_t* w) {
#pragma unroll
  for (int cc = 0; cc < 4; ++cc)
    st_shared_v4(tile + sw128_offset(r, 4 * h + cc), w[4 * cc], w[4 * cc + 1], w[4 * cc + 2], w[4 * cc + 3]);
}

// 16 fp32 values to global memory (64 B, 16-byte aligned).
__device__ __forceinline__ void store16(float* dst, const float* v) {
  float4* d4 = reinterpret_cast<float4*>(dst);
#pragma unroll
  for (int q = 0; q < 4; ++q) d4[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
}

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

// ===========================================================================
// pass 1
// ===========================================================================
template <int D, int ROLE>
__global__ void __launch_bounds__(kThreads, 1) bob_pass1_tc(const __grid_constant__ P1Params p) {
  using C = P1Cfg<D, ROLE>;
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ Ctrl ctrl;
  const int tid = threadIdx.x, warp = tid >> 5;
  const int row0 = blockIdx.x * kM, head = blockIdx.y;
  const int ntiles = p.N / kT;
  uint8_t* res = smem;
  uint8_t* stages = res + C::RES;
  uint8_t* ops = stages + C::NS * C::STAGE;

  if (tid == 0) {
    init_ctrl(ctrl, C::NS, C::NB, 1);
    if ((smem_u32(smem) & 1023u) != 0u) {  // layout assumption; never expected
      ctrl.abort_flag = 1;
      atomicOr(p.err, kErrTimeout);
    }
  }
  if (warp == 5) {
    tmem_alloc(&ctrl.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = ctrl.tmem_base;
  const Waiter wt{&ctrl.abort_flag, p.err, p.wait_ns};
  const bool live = ctrl.abort_flag == 0;

  if (warp == 4) {
    // ------------------------------------------------------------ TMA producer
    if (live && (tid & 31) == 0) {
      int issued = 0;
      mbar_arrive_expect_tx(&ctrl.res_full, C::RES);
      const CUtensorMap* rmap[3] = {&p.mQ, &p.mUQ, &p.mdO};
      for (int r = 0; r < C::NRES; ++r)
        for (int kc = 0; kc < C::DC; ++kc)
          tma_load_3d(res + (r * C::DC + kc) * kTileBytes, rmap[r], &ctrl.res_full, kc * 64, row0, head);
      bool ok = true;
      for (int t = 0; t < ntiles && ok; ++t) {
        const int s = t % C::NS;
        ok = mbar_wait(&ctrl.stage_empty[s], ((t / C::NS) & 1) ^ 1, wt);
        if (!ok) break;
        mbar_arrive_expect_tx(&ctrl.stage_full[s], C::STAGE);
        uint8_t* st = stages + s * C::STAGE;
        for (int kc = 0; kc < C::DC; ++kc) {
          uint8_t* ch = st + kc * kTileBytes;
          tma_load_3d(ch + 0, &p.mK, &ctrl.stage_full[s], kc * 64, t * kT, head);
          tma_load_3d(ch + 4096, &p.mUK, &ctrl.stage_full[s], kc * 64, t * kT, head);
          tma_load_3d(ch + 8192, &p.mV, &ctrl.stage_full[s], kc * 64, t * kT, head);
          tma_load_3d(ch + 12288, &p.mUV, &ctrl.stage_full[s], kc * 64, t * kT, head);
        }
        issued = t + 1;
      }
      if (!ok) {
        // give-up path: let every copy already issued land before exiting
        mbar_wait_drain(&ctrl.res_full, 0, kDrainNs);
        for (int t = (issued > C::NS ? issued - C::NS : 0); t < issued; ++t)
          mbar_wait_drain(&ctrl.stage_full[t % C::NS], (t / C::NS) & 1, kDrainNs);
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (live && (tid & 31) == 0) {
      const uint32_t res_a = smem_u32(res), st_a = smem_u32(stages), op_a = smem_u32(ops);
      const uint32_t id_s64 = idesc_bf16(kM, 64, false, false);
      const uint32_t id_s32 = idesc_bf16(kM, 32, false, false);
      const uint32_t id_acc = idesc_bf16(kM, D, false, true);
      auto res_desc = [&](int slot, int k) {
        return sdesc_sw128(res_a + (slot * C::DC + (k >> 2)) * kTileBytes + (k & 3) * 32, 16, 1024);
      };
      auto score_mmas = [&](int t) {
        const uint32_t sb = st_a + (t % C::NS) * C::STAGE;
        const uint32_t sc = tb + C::ACC_COLS + (t % C::NB) * C::SCOLS;
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = (k >> 2) * kTileBytes + (k & 3) * 32;
          mma_ss(sc, res_desc(C::R_Q, k), sdesc_sw128(sb + off, 16, 1024), id_s64, k > 0);  // [S | Q UK^T]
        }
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = (k >> 2) * kTileBytes + (k & 3) * 32;
          mma_ss(sc + 32, res_desc(C::R_UQ, k), sdesc_sw128(sb + off, 16, 1024), id_s32, 1);  // += UQ K^T
        }
        if (C::kQ) {
#pragma unroll
          for (int k = 0; k < D / 16; ++k) {
            const uint32_t off = (k >> 2) * kTileBytes + (k & 3) * 32 + 8192;
            mma_ss(sc + 64, res_desc(C::R_DO, k), sdesc_sw128(sb + off, 16, 1024), id_s64, k > 0);  // [dP | C]
          }
        }
      };
      auto accum_mmas = [&](int u) {
        const uint32_t sb = st_a + (u % C::NS) * C::STAGE;
        const uint32_t h = u & 1;
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
          const uint32_t acc0 = (u == 0 && kk == 0) ? 0u : 1u;
          auto opd = [&](int slot) { return sdesc_sw128(op_a + slot * kTileBytes + h * 64 + kk * 32, 16, 1024); };
          auto bz = [&](int rows0) { return sdesc_sw128(sb + rows0 * 128 + kk * 2048, kTileBytes, 1024); };
          if (C::kQ) {
            mma_ss(tb + C::A_U1, opd(C::O_DS), bz(32), id_acc, acc0);  // dS UK
            mma_ss(tb + C::A_U1, opd(C::O_X), bz(0), id_acc, 1);       // X K
            mma_ss(tb + C::A_U2, opd(C::O_P), bz(0), id_acc, acc0);    // P K
            mma_ss(tb + C::A_W, opd(C::O_DS), bz(0), id_acc, acc0);    // dS K
          }
          if (C::kDo) {
            mma_ss(tb + C::A_Y, opd(C::O_P), bz(96), id_acc, acc0);    // P UV
            mma_ss(tb + C::A_Y, opd(C::O_PB), bz(64), id_acc, 1);      // PB V
          }
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
      // every issued MMA completes before the TMEM is released
      mma_commit(&ctrl.drain);
      mbar_wait_drain(&ctrl.drain, 0, kDrainNs);
    }
  } else {
    // ------------------------------------------------------------ elementwise
    const int r = tid;  // tile row = TMEM lane
    const int i = row0 + r;
    const size_t vo = (size_t)head * p.N + i;
    const float nL = -p.L[vo] * kLog2e;
    const float Di = p.D[vo];
    const float sc = p.tau * kLog2e;
    const uint32_t lane = (uint32_t)(warp * 32) << 16;
    const uint32_t op_a = smem_u32(ops);
    float alpha = 0.f, ex = 0.f;
    bool ok = live;
    for (int t = 0; t < ntiles && ok; ++t) {
      const int b = t % C::NB, h = t & 1;
      if (!mbar_wait(&ctrl.score_full[b], (t / C::NB) & 1, wt)) { ok = false; break; }
      tc_fence_after();
      const uint32_t sbase = tb + lane + C::ACC_COLS + b * C::SCOLS;
      uint32_t wP[16], wdS[16], wX[16], wPB[16];
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        float s[16], bb[16], dp[16], cc[16];
        tmem_ld16(sbase + q * 16, s);
        tmem_ld16(sbase + 32 + q * 16, bb);
        if (C::kQ) {
          tmem_ld16(sbase + 64 + q * 16, dp);
          tmem_ld16(sbase + 96 + q * 16, cc);
        }
#pragma unroll
        for (int j = 0; j < 16; j += 2) {
          float pv[2], dsv[2], xv[2], pbv[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const float pe = ex2(fmaf(s[j + e], sc, nL));
            const float be = p.tau * bb[j + e];
            pv[e] = pe;
            pbv[e] = pe * be;
            alpha += pbv[e];
            if (C::kQ) {
              const float te = dp[j + e] - Di;
              dsv[e] = pe * te;
              xv[e] = pe * fmaf(be, te, cc[j + e]);
              ex += xv[e];
            }
          }
          const int w = q * 8 + j / 2;
          wP[w] = pack_bf16x2(pv[0], pv[1]);
          wPB[w] = pack_bf16x2(pbv[0], pbv[1]);
          if (C::kQ) {
            wdS[w] = pack_bf16x2(dsv[0], dsv[1]);
            wX[w] = pack_bf16x2(xv[0], xv[1]);
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&ctrl.score_empty[b]);
      if (!mbar_wait(&ctrl.op_empty[h], ((t >> 1) & 1) ^ 1, wt)) { ok = false; break; }
      write_op_half(op_a + C::O_P * kTileBytes, r, h, wP);
      if (C::kQ) {
        write_op_half(op_a + C::O_DS * kTileBytes, r, h, wdS);
        write_op_half(op_a + C::O_X * kTileBytes, r, h, wX);
      }
      if (C::kDo) write_op_half(op_a + C::O_PB * kTileBytes, r, h, wPB);
      fence_proxy_async_smem();
      mbar_arrive(&ctrl.op_full[h]);
    }
    if (ok && mbar_wait(&ctrl.acc_full, 0, wt)) {
      tc_fence_after();
      const size_t ro = ((size_t)head * p.N + i) * D;
      const uint32_t abase = tb + lane;
      if (C::kQ) {
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 16) {
          float u1[16], u2[16], wv[16], o[16];
          tmem_ld16(abase + C::A_U1 + c0, u1);
          tmem_ld16(abase + C::A_U2 + c0, u2);
          tmem_ld16(abase + C::A_W + c0, wv);
#pragma unroll
          for (int j = 0; j < 16; ++j) o[j] = p.tau * (u1[j] - ex * u2[j] - alpha * wv[j]);
          store16(p.gQ + ro + c0, o);
        }
        p.ws[2 * vo] = alpha;
        p.ws[2 * vo + 1] = fmaf(Di, alpha, ex);
      }
      if (C::kDo) {
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 16) {
          float y[16], o[16];
          tmem_ld16(abase + C::A_Y + c0, y);
          const float4* src = reinterpret_cast<const float4*>(p.O + ro + c0);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float4 v = src[q];
            o[4 * q] = y[4 * q] - alpha * v.x;
            o[4 * q + 1] = y[4 * q + 1] - alpha * v.y;
            o[4 * q + 2] = y[4 * q + 2] - alpha * v.z;
            o[4 * q + 3] = y[4 * q + 3] - alpha * v.w;
          }
          store16(p.gdO + ro + c0, o);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tb, 512);
  }
}

// ===========================================================================
// pass 2
// ===========================================================================
template <int D>
__global__ void __launch_bounds__(kThreads, 1) bob_pass2_tc(const __grid_constant__ P2Params p) {
  using C = P2Cfg<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ Ctrl ctrl;
  const int tid = threadIdx.x, warp = tid >> 5;
  const int col0 = blockIdx.x * kM, head = blockIdx.y;
  const int ntiles = p.N / kT;
  uint8_t* res = smem;
  uint8_t* ops = res + C::RES;
  uint8_t* stages = ops + C::OPS;

  if (tid == 0) {
    // stage_empty: one MMA commit + one arrival per elementwise warp (vectors read)
    init_ctrl(ctrl, C::NS, C::NB, 1 + 4);
    if ((smem_u32(smem) & 1023u) != 0u) {
      ctrl.abort_flag = 1;
      atomicOr(p.err, kErrTimeout);
    }
  }
  if (warp == 5) {
    tmem_alloc(&ctrl.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = ctrl.tmem_base;
  const Waiter wt{&ctrl.abort_flag, p.err, p.wait_ns};
  const bool live = ctrl.abort_flag == 0;

  if (warp == 4) {
    if (live && (tid & 31) == 0) {
      int issued = 0;
      mbar_arrive_expect_tx(&ctrl.res_full, C::RES);
      const CUtensorMap* rmap[4] = {&p.mK, &p.mV, &p.mUK, &p.mUV};
      for (int r = 0; r < C::NRES; ++r)
        for (int kc = 0; kc < C::DC; ++kc)
          tma_load_3d(res + (r * C::DC + kc) * kTileBytes, rmap[r], &ctrl.res_full, kc * 64, col0, head);
      bool ok = true;
      const size_t vbase = (size_t)head * p.N;
      for (int t = 0; t < ntiles && ok; ++t) {
        const int s = t % C::NS;
        ok = mbar_wait(&ctrl.stage_empty[s], ((t / C::NS) & 1) ^ 1, wt);
        if (!ok) break;
        mbar_arrive_expect_tx(&ctrl.stage_full[s], C::STAGE_TX);
        uint8_t* st = stages + s * C::STAGE;
        for (int kc = 0; kc < C::DC; ++kc) {
          uint8_t* ch = st + kc * 12288;
          tma_load_3d(ch + 0, &p.mQ, &ctrl.stage_full[s], kc * 64, t * kT, head);
          tma_load_3d(ch + 4096, &p.mUQ, &ctrl.stage_full[s], kc * 64, t * kT, head);
          tma_load_3d(ch + 8192, &p.mdO, &ctrl.stage_full[s], kc * 64, t * kT, head);
        }
        uint8_t* vec = st + C::STAGE_T;
        bulk_load(vec, p.L + vbase + t * kT, 128, &ctrl.stage_full[s]);
        bulk_load(vec + 128, p.D + vbase + t * kT, 128, &ctrl.stage_full[s]);
        bulk_load(vec + 256, p.ws + 2 * (vbase + t * kT), 256, &ctrl.stage_full[s]);
        issued = t + 1;
      }
      if (!ok) {
        mbar_wait_drain(&ctrl.res_full, 0, kDrainNs);
        for (int t = (issued > C::NS ? issued - C::NS : 0); t < issued; ++t)
          mbar_wait_drain(&ctrl.stage_full[t % C::NS], (t / C::NS) & 1, kDrainNs);
      }
    }
  } else if (warp == 5) {
    if (live && (tid & 31) == 0) {
      const uint32_t res_a = smem_u32(res), st_a = smem_u32(stages), op_a = smem_u32(ops);
      const uint32_t id_s64 = idesc_bf16(kM, 64, false, false);
      const uint32_t id_s32 = idesc_bf16(kM, 32, false, false);
      const uint32_t id_acc = idesc_bf16(kM, D, false, true);
      auto res_desc = [&](int slot, int k) {
        return sdesc_sw128(res_a + (slot * C::DC + (k >> 2)) * kTileBytes + (k & 3) * 32, 16, 1024);
      };
      auto score_mmas = [&](int t) {
        const uint32_t sb = st_a + (t % C::NS) * C::STAGE;
        const uint32_t sc = tb + C::ACC_COLS + (t % C::NB) * C::SCOLS;
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = (k >> 2) * 12288 + (k & 3) * 32;
          mma_ss(sc, res_desc(C::R_K, k), sdesc_sw128(sb + off, 16, 1024), id_s64, k > 0);          // [S^T | K UQ^T]
        }
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = (k >> 2) * 12288 + (k & 3) * 32;
          mma_ss(sc + 32, res_desc(C::R_UK, k), sdesc_sw128(sb + off, 16, 1024), id_s32, 1);        // += UK Q^T
        }
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = (k >> 2) * 12288 + (k & 3) * 32 + 8192;
          mma_ss(sc + 64, res_desc(C::R_V, k), sdesc_sw128(sb + off, 16, 1024), id_s32, k > 0);     // dP^T
          mma_ss(sc + 96, res_desc(C::R_UV, k), sdesc_sw128(sb + off, 16, 1024), id_s32, k > 0);    // C^T
        }
      };
      auto accum_mmas = [&](int u) {
        const uint32_t sb = st_a + (u % C::NS) * C::STAGE;
        const uint32_t h = u & 1;
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
          const uint32_t acc0 = (u == 0 && kk == 0) ? 0u : 1u;
          auto opd = [&](int slot) { return sdesc_sw128(op_a + slot * kTileBytes + h * 64 + kk * 32, 16, 1024); };
          auto bz = [&](int rows0) { return sdesc_sw128(sb + rows0 * 128 + kk * 2048, 12288, 1024); };
          mma_ss(tb + C::A_K, opd(C::O_DS), bz(32), id_acc, acc0);   // dS^T UQ
          mma_ss(tb + C::A_K, opd(C::O_GS), bz(0), id_acc, 1);       // Gs^T Q
          mma_ss(tb + C::A_V, opd(C::O_GD), bz(64), id_acc, acc0);   // Gdp^T dO
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
    const int r = tid;  // key row within the block = TMEM lane
    const int j = col0 + r;
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
      uint32_t wdS[16], wGs[16], wGd[16];
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        float s_[16], bb[16], dp[16], cc[16];
        tmem_ld16(sbase + q * 16, s_);
        tmem_ld16(sbase + 32 + q * 16, bb);
        tmem_ld16(sbase + 64 + q * 16, dp);
        tmem_ld16(sbase + 96 + q * 16, cc);
#pragma unroll
        for (int c = 0; c < 16; c += 2) {
          float dsv[2], gsv[2], gdv[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int ii = q * 16 + c + e;          // query column within the tile
            const float Li = vec[ii];
            const float Dq = vec[32 + ii];
            const float al = vec[64 + 2 * ii];
            const float Eq = vec[64 + 2 * ii + 1];
            const float pe = ex2(fmaf(s_[c + e], sc, -Li * kLog2e));
            const float te = dp[c + e] - Dq;
            const float bp = fmaf(p.tau, bb[c + e], -al);
            dsv[e] = pe * te;
            gsv[e] = pe * (fmaf(bp, te, cc[c + e]) + fmaf(al, Dq, -Eq));
            gdv[e] = pe * bp;
          }
          const int w = q * 8 + c / 2;
          wdS[w] = pack_bf16x2(dsv[0], dsv[1]);
          wGs[w] = pack_bf16x2(gsv[0], gsv[1]);
          wGd[w] = pack_bf16x2(gdv[0], gdv[1]);
        }
      }
      tc_fence_before();
      mbar_arrive(&ctrl.score_empty[b]);
      __syncwarp();
      if ((tid & 31) == 0) mbar_arrive(&ctrl.stage_empty[s]);
      if (!mbar_wait(&ctrl.op_empty[h], ((t >> 1) & 1) ^ 1, wt)) { ok = false; break; }
      write_op_half(op_a + C::O_DS * kTileBytes, r, h, wdS);
      write_op_half(op_a + C::O_GS * kTileBytes, r, h, wGs);
      write_op_half(op_a + C::O_GD * kTileBytes, r, h, wGd);
      fence_proxy_async_smem();
      mbar_arrive(&ctrl.op_full[h]);
    }
    if (ok && mbar_wait(&ctrl.acc_full, 0, wt)) {
      tc_fence_after();
      const size_t ro = ((size_t)head * p.N + j) * D;
      const uint32_t abase = tb + lane;
#pragma unroll 1
      for (int c0 = 0; c0 < D; c0 += 16) {
        float ak[16], av[16];
        tmem_ld16(abase + C::A_K + c0, ak);
        tmem_ld16(abase + C::A_V + c0, av);
#pragma unroll
        for (int e = 0; e < 16; ++e) ak[e] *= p.tau;
        store16(p.gK + ro + c0, ak);
        store16(p.gV + ro + c0, av);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tb, 512);
  }
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

// [BH, N, D] bf16 tensor, box {64, rows, 1}, 128-byte swizzle.
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
cudaError_t bob_d(const BobArgs& a, const DevCtx& c, cudaStream_t s) {
  P1Params p1;
  const int BH = a.BH, N = a.N;
  bool ok = make_map(&p1.mQ, a.Q, BH, N, D, kM) && make_map(&p1.mdO, a.dO, BH, N, D, kM) &&
            make_map(&p1.mUQ, a.UQ, BH, N, D, kM) && make_map(&p1.mK, a.K, BH, N, D, kT) &&
            make_map(&p1.mUK, a.UK, BH, N, D, kT) && make_map(&p1.mV, a.V, BH, N, D, kT) &&
            make_map(&p1.mUV, a.UV, BH, N, D, kT);
  if (!ok) return cudaErrorInvalidValue;
  p1.L = a.L;
  p1.D = a.D;
  p1.O = a.O;
  p1.gQ = a.gQ;
  p1.gdO = a.gdO;
  p1.ws = a.ws;
  p1.N = N;
  p1.tau = a.tau;
  p1.err = c.err;
  p1.wait_ns = c.wait_ns;
  const dim3 grid(N / kM, BH);
  cudaError_t e;
  if constexpr (D == 64) {
    e = launch(bob_pass1_tc<D, kBoth>, P1Cfg<D, kBoth>::SMEM, grid, p1, s);
  } else {
    e = launch(bob_pass1_tc<D, kQSide>, P1Cfg<D, kQSide>::SMEM, grid, p1, s);
    if (e == cudaSuccess) e = launch(bob_pass1_tc<D, kDoSide>, P1Cfg<D, kDoSide>::SMEM, grid, p1, s);
  }
  if (e != cudaSuccess) return e;
  P2Params p2;
  ok = make_map(&p2.mK, a.K, BH, N, D, kM) && make_map(&p2.mV, a.V, BH, N, D, kM) &&
       make_map(&p2.mUK, a.UK, BH, N, D, kM) && make_map(&p2.mUV, a.UV, BH, N, D, kM) &&
       make_map(&p2.mQ, a.Q, BH, N, D, kT) && make_map(&p2.mUQ, a.UQ, BH, N, D, kT) &&
       make_map(&p2.mdO, a.dO, BH, N, D, kT);
  if (!ok) return cudaErrorInvalidValue;
  p2.L = a.L;
  p2.D = a.D;
  p2.ws = a.ws;
  p2.gK = a.gK;
  p2.gV = a.gV;
  p2.N = N;
  p2.tau = a.tau;
  p2.err = c.err;
  p2.wait_ns = c.wait_ns;
  return launch(bob_pass2_tc<D>, P2Cfg<D>::SMEM, grid, p2, s);
}

}  // namespace

cudaError_t tc_bob(const BobArgs& a, const DevCtx& c, cudaStream_t s) {
  return a.d == 64 ? bob_d<64>(a, c, s) : bob_d<128>(a, c, s);
}

}  // namespace fbob
