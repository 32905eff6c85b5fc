// Tensor-core (tcgen05 + TMEM + TMA) attention forward for bf16 inputs,
// d in {64, 128}, any N: O = softmax(tau Q K^T) V and the
// natural-log row logsumexp L (FlashBoB abstract: the FlashAttention-style
// forward whose outputs the first backward and BoB consume).
//
// A CTA owns two 128-row query blocks (A, B) and streams K and V in tiles of
// 128 keys.  TMEM: O_A, O_B (d columns each), S_A, S_B (128 columns each: 512
// in all at d = 128).  Per tile t and block X:
//   S_X = Q_X K_t^T         one SS MMA of N = 128 (issued by warp 9);
//   softmax (warpgroup X, thread r = row r): two passes over S_X - the row
//     max, then P = 2^(x - m) with x = tau log2(e) S - written over S_X as
//     two bf16 terms, P = P_hi + P_lo with P_hi = bf16(P) and P_lo =
//     bf16(P - P_hi): each 32-column chunk of S holds the P_hi of its 32
//     keys in its first 16 columns and their P_lo in the last 16;
//   O_X += P_hi V_t + P_lo V_t   TS MMAs, P read from TMEM (issued by warp 10).
// The split makes O exact to about 2^-17 relative instead of the 2^-9 of one
// bf16 rounding of P.  That matters downstream: D = rowsum(dO o O) feeds
// dP - D, which nearly cancels on the dominant key of a peaked softmax row,
// so an O (and D) carrying P's rounding would spoil dQ, dK and every BoB
// output there.  Because P overwrites S, S_X(t+1) is issued only after the
// P V products of tile t have completed.  The running max moves only when a
// row's tile max exceeds it by more than 8 (lazy rescale), so P <= 2^8 stays
// well inside bf16 and O_X is rescaled in TMEM only then (after the previous
// P V products have landed).
// O = O_X / l, L = (m + log2 l) ln 2.  Warp 8 issues TMA.
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
using tile::kChunk;
using tile::kLog2e;
using tile::kM;

constexpr int kThreads = 352;
constexpr int kKT = 128;                  // keys per tile
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescale = 8.0f;          // lazy-rescale threshold (log2 units)
constexpr uint64_t kDrainNs = 200000000ull;

struct FwdParams {
  CUtensorMap mQ, mK, mV;  // box {64, 128}
  float *O, *L;
  int N;
  int dv;                  // head size in global memory (<= D; see tc_tile.cuh)
  float tau;
  int causal;
  unsigned int* err;
  unsigned long long wait_ns;
  int stall;
};

template <int D>
struct FwdCfg {
  static constexpr int DC = D / 64;
  static constexpr int TILE = DC * kChunk;       // one 128 x d tile (Q block, K or V tile)
  static constexpr int NK = D == 128 ? 3 : 4, NV = D == 128 ? 2 : 4;
  static constexpr int Q_OFF = 0, K_OFF = 2 * TILE, V_OFF = K_OFF + NK * TILE;
  static constexpr int SMEM = V_OFF + NV * TILE;
  static constexpr int S_COL = 2 * D;            // S_A at S_COL, S_B at S_COL + 128
  static_assert(S_COL + 2 * kKT <= 512, "TMEM budget");
  static_assert(SMEM + 1024 <= 232448, "shared memory budget");
};

struct Ctrl {
  uint64_t q_full;
  uint64_t k_full[4], k_empty[4], v_full[4], v_empty[4];
  uint64_t s_full[2], p_full[2], o_done[2];   // per block
  uint64_t drain_s, drain_p;
  uint32_t tmem_base;
  int abort_flag;
};

// One tile of the softmax of one row (this thread's TMEM lane): pass 1 finds
// the tile's row max over columns 0..lim, a lazy rescale of O and l follows
// when the max grew by more than 2^8 (after the block's previous P V product
// has landed), pass 2 writes P = 2^(x - m) as P_hi + P_lo over S (chunk c
// reads columns 32c..32c+31 and writes P_hi into 32c..32c+15, P_lo into
// 32c+16..32c+31) and sums P into ls.  MASK = false skips the column test
// (tiles below the diagonal).
template <int D, bool MASK>
__device__ __forceinline__ bool softmax_tile(uint32_t s_col, uint32_t o_col, int lim, float sc, float& m, float& l,
                                             float& ls, uint64_t& o_done, int t, const Waiter& wt) {
  float mt = -INFINITY;
#pragma unroll 1
  for (int c = 0; c < kKT / 32; ++c) {
    float s[32];
    tmem_ld32(s_col + 32 * c, s);
#pragma unroll
    for (int j = 0; j < 32; ++j) mt = fmaxf(mt, (!MASK || 32 * c + j <= lim) ? s[j] : -INFINITY);
  }
  mt *= sc;
  if (__any_sync(0xffffffffu, mt > m + kRescale)) {
    const float mn = fmaxf(m, mt);
    if (t > 0) {
      const float scale = tile::ex2(m - mn);
      // the previous P V product of this block must have landed
      if (!__all_sync(0xffffffffu, mbar_wait(&o_done, (t - 1) & 1, wt))) return false;
      tc_fence_after();
#pragma unroll 1
      for (int c0 = 0; c0 < D; c0 += 16) {
        float o[16];
        tmem_ld16(o_col + c0, o);
        uint32_t w[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) w[e] = __float_as_uint(o[e] * scale);
        tmem_st16_nowait(o_col + c0, w);
      }
      tmem_st_wait();
      l *= scale;
    }
    m = mn;
  }
#pragma unroll 1
  for (int c = 0; c < kKT / 32; ++c) {
    float s[32];
    tmem_ld32(s_col + 32 * c, s);
    uint32_t wh[16], wl[16];
#pragma unroll
    for (int j = 0; j < 32; j += 2) {
      const float p0 = (!MASK || 32 * c + j <= lim) ? tile::ex2(fmaf(s[j], sc, -m)) : 0.f;
      const float p1 = (!MASK || 32 * c + j + 1 <= lim) ? tile::ex2(fmaf(s[j + 1], sc, -m)) : 0.f;
      ls += p0 + p1;
      const __nv_bfloat162 h = __floats2bfloat162_rn(p0, p1);
      const float2 hf = __bfloat1622float2(h);
      wh[j / 2] = *reinterpret_cast<const uint32_t*>(&h);
      wl[j / 2] = pack_bf16x2(p0 - hf.x, p1 - hf.y);   // exact differences, rounded once more
    }
    tmem_st16_nowait(s_col + 32 * c, wh);
    tmem_st16_nowait(s_col + 32 * c + 16, wl);
  }
  return true;
}

// CAUSAL and RAGGED (N not a multiple of 128) are compile-time choices; a
// ragged N reads zeros past the end (TMA), masks keys >= N in the last tile
// and stores only rows < N.
template <int D, bool CAUSAL, bool RAGGED>
__global__ void __launch_bounds__(kThreads, 1) attn_fwd_tc(const __grid_constant__ FwdParams p) {
  using C = FwdCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ Ctrl ctrl;
  const int tid = threadIdx.x, warp = tid >> 5;
  // causal: block X streams the key tiles up to its diagonal (tile
  // row0 / 128 + X), so the last pairs of blocks do the most work and run first
  const int pair = CAUSAL ? (int)(gridDim.x - 1 - blockIdx.x) : (int)blockIdx.x;
  const int row0 = pair * 2 * kM, head = blockIdx.y;
  const int nblk = (row0 + kM < p.N) ? 2 : 1;   // block B exists unless it would start at or past N
  const int t_all = (p.N + kKT - 1) / kKT;
  const int ntx[2] = {CAUSAL ? min(t_all, row0 / kKT + 1) : t_all, CAUSAL ? min(t_all, row0 / kKT + 2) : t_all};
  const int nt = ntx[nblk - 1];                 // key tiles the CTA streams

  if (tid == 0) {
    ctrl.abort_flag = 0;
    mbar_init(&ctrl.q_full, 1);
    for (int s = 0; s < C::NK; ++s) {
      mbar_init(&ctrl.k_full[s], 1);
      mbar_init(&ctrl.k_empty[s], 1);
    }
    for (int s = 0; s < C::NV; ++s) {
      mbar_init(&ctrl.v_full[s], 1);
      mbar_init(&ctrl.v_empty[s], 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(&ctrl.s_full[x], 1);
      mbar_init(&ctrl.p_full[x], 128);
      mbar_init(&ctrl.o_done[x], 1);
    }
    mbar_init(&ctrl.drain_s, 1);
    mbar_init(&ctrl.drain_p, 1);
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
  const uint32_t sm0 = smem_u32(smem);

  if (warp == 8) {
    // ------------------------------------------------------------------ TMA
    if (live && (tid & 31) == 0) {
      mbar_arrive_expect_tx(&ctrl.q_full, nblk * C::TILE);
      for (int x = 0; x < nblk; ++x)
        for (int kc = 0; kc < C::DC; ++kc)
          tma_load_3d(smem + C::Q_OFF + x * C::TILE + kc * kChunk, &p.mQ, &ctrl.q_full, kc * 64, row0 + x * kM, head);
      int ik = 0, iv = 0;
      bool ok = true;
      // K runs up to NK tiles ahead, V up to NV; K(t) is issued before V(t)
      for (int t = 0; t < nt && ok; ++t) {
        const int sk = t % C::NK, sv = t % C::NV;
        if (!(ok = mbar_wait(&ctrl.k_empty[sk], ((t / C::NK) & 1) ^ 1, wt))) break;
        if (!(p.stall && t == 0)) {  // test hook: nothing fills the first K stage
          mbar_arrive_expect_tx(&ctrl.k_full[sk], C::TILE);
          for (int kc = 0; kc < C::DC; ++kc)
            tma_load_3d(smem + C::K_OFF + sk * C::TILE + kc * kChunk, &p.mK, &ctrl.k_full[sk], kc * 64, t * kKT, head);
          ik = t + 1;
        }
        if (!(ok = mbar_wait(&ctrl.v_empty[sv], ((t / C::NV) & 1) ^ 1, wt))) break;
        mbar_arrive_expect_tx(&ctrl.v_full[sv], C::TILE);
        for (int kc = 0; kc < C::DC; ++kc)
          tma_load_3d(smem + C::V_OFF + sv * C::TILE + kc * kChunk, &p.mV, &ctrl.v_full[sv], kc * 64, t * kKT, head);
        iv = t + 1;
      }
      if (!ok) {
        // give-up path: every copy already issued lands before the CTA exits
        mbar_wait_drain(&ctrl.q_full, 0, kDrainNs);
        for (int t = (ik > C::NK ? ik - C::NK : 0); t < ik; ++t)
          mbar_wait_drain(&ctrl.k_full[t % C::NK], (t / C::NK) & 1, kDrainNs);
        for (int t = (iv > C::NV ? iv - C::NV : 0); t < iv; ++t)
          mbar_wait_drain(&ctrl.v_full[t % C::NV], (t / C::NV) & 1, kDrainNs);
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------- S = Q K^T MMAs
    // S_X(t) waits for K(t) and, for t > 0, for O_X += P V_{t-1} to have
    // completed (P_X(t-1) lives in S_X's columns).
    if (live) {  // the whole warp runs the loop; lane 0 issues (elect.sync)
      const uint32_t q_lo = desc_lo(sm0 + C::Q_OFF, 16);
      const uint32_t i128 = idesc_bf16(kM, kKT, false, false);
      bool ok = __all_sync(0xffffffffu, mbar_wait(&ctrl.q_full, 0, wt));
      for (int t = 0; ok && t < nt; ++t) {
        const int sk = t % C::NK;
        const uint32_t k_lo = desc_lo(sm0 + C::K_OFF + sk * C::TILE, 16);
        ok = __all_sync(0xffffffffu, mbar_wait(&ctrl.k_full[sk], (t / C::NK) & 1, wt));
        for (int x = 0; ok && x < nblk; ++x) {
          if (t >= ntx[x]) continue;
          if (t > 0) ok = __all_sync(0xffffffffu, mbar_wait(&ctrl.o_done[x], (t - 1) & 1, wt));
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < D / 16; ++k)
            mma_ss_w(tb + C::S_COL + x * kKT, tile::res_lo(q_lo, x, C::DC, k), tile::res_lo(k_lo, 0, C::DC, k), i128,
                     k > 0);
          mma_commit_w(&ctrl.s_full[x]);
        }
        if (ok) mma_commit_w(&ctrl.k_empty[sk]);
      }
      mma_commit_w(&ctrl.drain_s);
      mbar_wait_drain(&ctrl.drain_s, 0, kDrainNs);
    }
  } else if (warp == 10) {
    // ------------------------------------------------------ O += P V MMAs
    if (live) {
      const uint32_t id = idesc_bf16(kM, D, false, true);
      bool ok = true;
      for (int t = 0; ok && t < nt; ++t) {
        const int sv = t % C::NV;
        const uint32_t v_mn = desc_lo(sm0 + C::V_OFF + sv * C::TILE, kChunk);
        ok = __all_sync(0xffffffffu, mbar_wait(&ctrl.v_full[sv], (t / C::NV) & 1, wt));
        for (int x = 0; ok && x < nblk; ++x) {
          if (t >= ntx[x]) continue;
          ok = __all_sync(0xffffffffu, mbar_wait(&ctrl.p_full[x], t & 1, wt));
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < kKT / 16; ++kk) {
            // keys 16 kk .. 16 kk + 15: P_hi at column 32 (kk / 2) + 8 (kk % 2), P_lo 16 columns on
            const uint32_t a = tb + C::S_COL + x * kKT + 32 * (kk >> 1) + 8 * (kk & 1);
            mma_ts_w(tb + x * D, a, tile::mnmaj(v_mn, 0, kk), id, (t > 0 || kk > 0) ? 1u : 0u);
            mma_ts_w(tb + x * D, a + 16, tile::mnmaj(v_mn, 0, kk), id, 1u);
          }
          mma_commit_w(&ctrl.o_done[x]);
        }
        if (ok) mma_commit_w(&ctrl.v_empty[sv]);
      }
      mma_commit_w(&ctrl.drain_p);
      mbar_wait_drain(&ctrl.drain_p, 0, kDrainNs);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int x = warp >> 2;                 // block owned by this warpgroup
    const int r = tid & 127;
    const uint32_t lane = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t s_col = tb + lane + C::S_COL + x * kKT;
    const float sc = p.tau * kLog2e;
    float m = -INFINITY, l = 0.f;
    bool ok = live && x < nblk;
    const int ntb = ntx[x < nblk ? x : 0];
    for (int t = 0; t < ntb && ok; ++t) {
      // warp-uniform waits: the TMEM loads and stores that follow are warp-collective
      if (!__all_sync(0xffffffffu, mbar_wait(&ctrl.s_full[x], t & 1, wt))) { ok = false; break; }
      tc_fence_after();
      // this row may see tile columns 0..lim (causal: keys up to its own index);
      // the masked variant runs only on a block's diagonal tile
      int lim = CAUSAL ? row0 + x * kM + r - t * kKT : kKT - 1;
      if (RAGGED) lim = min(lim, p.N - 1 - t * kKT);   // keys >= N
      float ls = 0.f;
      const bool fine = ((CAUSAL || RAGGED) && __any_sync(0xffffffffu, lim < kKT - 1))
                            ? softmax_tile<D, CAUSAL || RAGGED>(s_col, tb + lane + x * D, lim, sc, m, l, ls, ctrl.o_done[x], t, wt)
                            : softmax_tile<D, false>(s_col, tb + lane + x * D, lim, sc, m, l, ls, ctrl.o_done[x], t, wt);
      if (!fine) { ok = false; break; }
      l += ls;
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&ctrl.p_full[x]);
    }
    if (ok && __all_sync(0xffffffffu, mbar_wait(&ctrl.o_done[x], (ntb - 1) & 1, wt))) {
      tc_fence_after();
      // every lane runs the (warp-collective) TMEM loads; rows >= N store nothing
      const int i = row0 + x * kM + r;
      const bool keep = i < p.N;
      const size_t ro = ((size_t)head * p.N + (keep ? i : 0)) * p.dv;
      const float inv = 1.f / l;
#pragma unroll 1
      for (int c0 = 0; c0 < p.dv; c0 += 16) {   // columns >= dv hold zeros
        float o[16];
        tmem_ld16(tb + lane + x * D + c0, o);
#pragma unroll
        for (int e = 0; e < 16; ++e) o[e] *= inv;
        if (keep) tile::store16(p.O + ro + c0, o);
      }
      if (keep) p.L[(size_t)head * p.N + i] = (m + __log2f(l)) * kLn2;
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
  if (!make_bf16_map(&p.mQ, a.Q, a.BH, a.N, a.d, kM) || !make_bf16_map(&p.mK, a.K, a.BH, a.N, a.d, kKT) ||
      !make_bf16_map(&p.mV, a.V, a.BH, a.N, a.d, kKT))
    return cudaErrorInvalidValue;
  p.O = a.O;
  p.L = a.L;
  p.N = a.N;
  p.dv = a.d;
  p.tau = a.tau;
  p.causal = a.causal;
  p.err = c.err;
  p.wait_ns = c.wait_ns;
  p.stall = c.stall;
  const bool ragged = a.N % kM != 0;
  auto kernel = a.causal ? (ragged ? attn_fwd_tc<D, true, true> : attn_fwd_tc<D, true, false>)
                         : (ragged ? attn_fwd_tc<D, false, true> : attn_fwd_tc<D, false, false>);
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
  // d = 32, 96 run on the d = 64, 128 kernels with zero-padded columns
  return a.d <= 64 ? fwd_d<64>(a, c, s) : fwd_d<128>(a, c, s);
}

}  // namespace fbob
