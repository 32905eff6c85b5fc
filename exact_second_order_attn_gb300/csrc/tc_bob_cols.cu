// BoB pass 2 (the column pass) for bf16 inputs with 128-column heads (d = 96
// and 128; d = 96 zero-padded on chip), any N: per block of 128 keys, a loop
// over all query tiles that writes gK and gV.
//
// Source: "FlashBoB: I/O-Efficient Exact Backward-over-Backward for Softmax
// Attention", evolve.pub review - Summary / Key claims (the second pass of the
// two-pass schedule reads only the row scalars alpha and E from the first;
// paper Prop. 4.1 and Algorithm 1) and Strengths (transfer ledger of
// Theorem 4.3: pass 2 streams Q, dO, UQ and L, D, alpha, E per key block).
//
// Per (key j = resident row, query i = streamed column), with the final
// alpha_i, E_i of pass 1:
//   P = exp(tau S - L_i), b' = tau B - alpha_i, t = dP - D_i,
//   dS = P t,  Gs = P (C + b' t + alpha_i D_i - E_i),  Gdp = P b',
//   gK = tau (dS^T UQ + Gs^T Q),  gV = Gdp^T dO.
//
// Why a kernel of its own: at d = 128 the two accumulators take 256 of the
// 512 TMEM columns, and the four score tiles (S, B, dP, C) of a 64-query tile
// another 256, so the resident operands cannot all sit in TMEM, and a score
// MMA with its 128-row A operand in shared memory runs near the tensor rate
// only with N >= 128.  So each 64-query tile is computed in two phases through
// one 128-column score buffer:
//   phase A  [S^T | B^T / tau] = K [Q; UQ]^T (one SS MMA, N = 128) + UK Q^T
//            (SS, N = 64): K and UK resident in shared memory;
//   phase B  [dP^T | C^T] = V dO^T, UV dO^T (TS MMAs, N = 64): V and UV
//            resident in TMEM.
// gV needs only phase A's data, so its operand Gdp is written as soon as
// phase A is read and its MMA runs while phase B's scores are read; gK's
// operands dS, Gs follow phase B and its MMAs run while the next tile's
// phase A is read.  The tensor pipe thus sees
//   A(t)  gK(t-1)  B(t)  gV(t)  A(t+1)  gK(t)  ...
// with each score phase's read-out covered by an accumulator batch.  dO
// streams through a one-stage ring of its own (released once gV(t) and B(t)
// are done: the next dO is needed only by B(t+1), behind A(t+1) and
// gK(t)); [Q | UQ] and the per-query vectors (L, D, alpha, E) through a
// three-stage ring released by gK(t).  gK(t) runs after A(t+1), so with two
// stages the load for tile t+2 could start only once gK(t) had finished and
// A(t+2) waited for it; the third stage is paid for by the single dO stage
// and by Gdp and dS sharing one operand tile (Gdp(t) is written once gK(t-1)
// has read dS(t-1), dS(t) once gV(t) has read Gdp(t)).
//
// CTA of 11 warps: warps 0-7 two elementwise warpgroups (both on every tile,
// warpgroup g on query columns 32g..32g+31; thread r owns TMEM lane r = key
// r), warp 8 TMA, warp 9 score MMAs (TMEM owner), warp 10 accumulator MMAs.
// TMEM: gK 0-127 | gV 128-255 | score buffer 256-383 | V 384-447, UV 448-511.
// Every wait is bounded; on give-up every role leaves its loop, copies and
// MMAs in flight are drained and TMEM is freed.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "prof.h"
#include "tc_tile.cuh"

namespace fbob {
namespace {

using namespace tc;
using namespace tile;

constexpr int kQT = 64;                    // queries per streamed tile
constexpr int kD = 128, kDC = 2;           // head columns (padded), 64-column chunks
constexpr int kQB = kQT * 128;             // one 64-column chunk of a 64-row tile: 8 KB
constexpr int kQUCH = 2 * kQB;             // [Q | UQ] rows of one chunk: 16 KB
constexpr int kQU = kDC * kQUCH;           // 32 KB
constexpr int kVEC = 4 * kQT * 4;          // L (64), D (64), (alpha, E) (128) floats
constexpr int kQUS = kQU + kVEC;           // one [Q | UQ] stage with its vectors
constexpr int kDO = kDC * kQB;             // one dO stage: 16 KB
constexpr int kNQ = 3, kND = 1;            // ring stages
constexpr int kRES_OFF = 0;                // K (2 chunks), UK (2 chunks)
constexpr int kQU_OFF = kRES_OFF + 2 * kDC * kChunk;
constexpr int kDO_OFF = kQU_OFF + kNQ * kQUS;
constexpr int kOPS_OFF = kDO_OFF + kND * kDO;   // Gdp-then-dS, Gs tiles [128][64]
constexpr int kREC_OFF = kOPS_OFF + 2 * kChunk; // per elementwise warp: 2 x 32 float2 query records
constexpr int kSMEM = kREC_OFF + 8 * 64 * 8;
static_assert(kQUS % 1024 == 0 && kQU_OFF % 1024 == 0 && kDO_OFF % 1024 == 0 && kOPS_OFF % 1024 == 0,
              "1024-byte aligned tiles");
static_assert(kSMEM + 1024 <= 232448, "shared memory budget (1 KB static)");
constexpr int kACC_K = 0, kACC_V = kD, kSC = 2 * kD, kTRES = kSC + 2 * kQT;   // TMEM columns
static_assert(kTRES + 2 * (kD / 2) == 512, "TMEM budget");
constexpr int kOP_GDP = 0, kOP_DS = 0, kOP_GS = 1;   // Gdp(t) and dS(t) share a tile

struct ColParams {
  CUtensorMap mK, mUK;                       // resident, box {64, 128}
  CUtensorMap mQ, mUQ, mdO;                  // streamed, box {64, 64}
  const __nv_bfloat16 *V, *UV;               // resident (copied into TMEM)
  const float *L, *D, *ws;
  float *gK, *gV;
  int N;
  int dv;                                    // head size in global memory (<= 128)
  float tau;
  unsigned int* err;
  unsigned long long wait_ns;
  int stall;
};

struct ColCtrl {
  uint64_t res_full, tres_full;
  uint64_t qu_full[kNQ], qu_empty[kNQ];
  uint64_t do_full[kND], do_empty[kND];
  uint64_t s_full[2], s_empty[2];            // phase A, phase B of the score buffer
  uint64_t gdp_full, gdp_empty, kop_full, kop_empty;
  uint64_t acc_full, drain_s, drain_a;
  uint32_t tmem_base;
  int abort_flag;
};

// L, D, (alpha, E) of query tile tq with bounds checks, written by the 32
// lanes of the producer warp (a ragged tile, or N not a multiple of 4, where
// a bulk copy would start off a 16-byte boundary).
__device__ __forceinline__ void fill_vectors(const ColParams& p, float* vec, int tq, int head, int lane) {
  for (int k = lane; k < 4 * kQT; k += 32) {
    float v = 0.f;
    if (k < 2 * kQT) {
      const int q = tq * kQT + (k % kQT);
      if (q < p.N) v = (k < kQT ? p.L : p.D)[(size_t)head * p.N + q];
    } else {
      const int q = tq * kQT + (k - 2 * kQT) / 2;
      if (q < p.N) v = p.ws[2 * ((size_t)head * p.N + q) + (k & 1)];
    }
    vec[k] = v;
  }
}

// The elementwise work of one tile for one thread (key row r, query columns
// c0..c0+31).  MASK: some column lies outside [lo, hi] (causal diagonal or
// queries past N) and gets P = 0.  Returns false when a wait gave up.
template <bool MASK>
__device__ __forceinline__ bool ew_tile(const ColParams& p, ColCtrl& c, const Waiter& wt, uint32_t sc_col,
                                        uint32_t ops, const float* vec, float2* rec, int t, int c0, int lo, int hi,
                                        int r) {
  const float sc = p.tau * kLog2e;
  // The tile's per-query constants, formed once per warp instead of once per
  // (key, query): (-L log2e, alpha) for phase A and (D, alpha D - E) for
  // phase B, in this warp's own records (a warp barrier orders them).  The
  // loops read two queries' records with one broadcast 16-byte load: every
  // shared-memory load costs the pipe a wavefront, however few bytes.
  float2* recA = rec;
  float2* recB = rec + 32;
  const float4* recA4 = reinterpret_cast<const float4*>(recA);
  const float4* recB4 = reinterpret_cast<const float4*>(recB);
  {
    const int lane = (int)(threadIdx.x & 31u), i = c0 + lane;
    const float Lq = vec[i], Dq = vec[kQT + i];
    const float2 ae = reinterpret_cast<const float2*>(vec + 2 * kQT)[i];
    __syncwarp();   // every lane has read the previous tile's records
    recA[lane] = make_float2(-Lq * kLog2e, ae.x);
    recB[lane] = make_float2(Dq, fmaf(ae.x, Dq, -ae.y));
    __syncwarp();
  }
  float P[32], bp[32];
  // ---- phase A: S^T and B^T / tau of this warpgroup's 32 queries
  if (!__all_sync(0xffffffffu, mbar_wait(&c.s_full[0], t & 1, wt))) return false;
  tc_fence_after();
  {
    float S[32], B[32];
    tmem_ld16x4(sc_col, sc_col + 16, sc_col + 64, sc_col + 80, S, S + 16, B, B + 16);
    tc_fence_before();
    mbar_arrive(&c.s_empty[0]);
#pragma unroll
    for (int j = 0; j < 32; j += 2) {
      const float4 v = recA4[j / 2];
      const int col = c0 + j;
      P[j] = (!MASK || (col >= lo && col <= hi)) ? ex2(fmaf(S[j], sc, v.x)) : 0.f;
      P[j + 1] = (!MASK || (col + 1 >= lo && col + 1 <= hi)) ? ex2(fmaf(S[j + 1], sc, v.z)) : 0.f;
      bp[j] = fmaf(p.tau, B[j], -v.y);
      bp[j + 1] = fmaf(p.tau, B[j + 1], -v.w);
    }
  }
  // Gdp = P b' for gV.  Its tile held dS(t-1): gK(t-1) must have read it
  // (and Gs(t-1), which the same commit covers).
  if (t > 0 && !__all_sync(0xffffffffu, mbar_wait(&c.kop_empty, (t - 1) & 1, wt))) return false;
  {
    uint32_t w[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) w[j] = pack_bf16x2(P[2 * j] * bp[2 * j], P[2 * j + 1] * bp[2 * j + 1]);
    write_op_cols<16>(ops + kOP_GDP * kChunk, (uint32_t)r, c0, w);
  }
  fence_proxy_async_smem();
  mbar_arrive(&c.gdp_full);
  // ---- phase B: dP^T and C^T
  if (!__all_sync(0xffffffffu, mbar_wait(&c.s_full[1], t & 1, wt))) return false;
  tc_fence_after();
  float dP[32], C[32];
  tmem_ld16x4(sc_col, sc_col + 16, sc_col + 64, sc_col + 80, dP, dP + 16, C, C + 16);
  tc_fence_before();
  mbar_arrive(&c.s_empty[1]);
  // dS goes where Gdp(t) is: gV(t) must have read it
  if (!__all_sync(0xffffffffu, mbar_wait(&c.gdp_empty, t & 1, wt))) return false;
#pragma unroll
  for (int h = 0; h < 2; ++h) {   // 16 columns at a time: dS and Gs for gK
    uint32_t wd[8], wg[8];
#pragma unroll
    for (int j = 0; j < 16; j += 2) {
      float ds[2], gs[2];
      const float4 v4 = recB4[(16 * h + j) / 2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int k = 16 * h + j + e;
        const float2 v = e == 0 ? make_float2(v4.x, v4.y) : make_float2(v4.z, v4.w);
        const float te = dP[k] - v.x;
        ds[e] = P[k] * te;
        gs[e] = P[k] * (fmaf(bp[k], te, C[k]) + v.y);
      }
      wd[j / 2] = pack_bf16x2(ds[0], ds[1]);
      wg[j / 2] = pack_bf16x2(gs[0], gs[1]);
    }
    write_op_cols<8>(ops + kOP_DS * kChunk, (uint32_t)r, c0 + 16 * h, wd);
    write_op_cols<8>(ops + kOP_GS * kChunk, (uint32_t)r, c0 + 16 * h, wg);
  }
  fence_proxy_async_smem();
  mbar_arrive(&c.kop_full);
  return true;
}

template <bool CAUSAL, bool RAGGED>
__global__ void __launch_bounds__(kThreads, 1) bob_cols_wide(const __grid_constant__ ColParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ ColCtrl ctrl;
  const int tid = threadIdx.x, warp = tid >> 5, lane_id = tid & 31;
  const int blk0 = blockIdx.x * kM, head = blockIdx.y;
  const int t_all = (p.N + kQT - 1) / kQT;
  // causal: a key block meets only the queries from its own index on
  const int t_begin = CAUSAL ? blk0 / kQT : 0;
  const int nt = t_all - t_begin;   // >= 1: blk0 < N

  if (tid == 0) {
    ctrl.abort_flag = 0;
    mbar_init(&ctrl.res_full, 1);
    mbar_init(&ctrl.tres_full, 256);
    for (int s = 0; s < kNQ; ++s) {
      mbar_init(&ctrl.qu_full[s], 1);
      mbar_init(&ctrl.qu_empty[s], 1);    // gK(t) done (it follows every other reader)
    }
    for (int s = 0; s < kND; ++s) {
      mbar_init(&ctrl.do_full[s], 1);
      mbar_init(&ctrl.do_empty[s], 2);    // B(t) and gV(t) done (two issuing warps)
    }
    for (int q = 0; q < 2; ++q) {
      mbar_init(&ctrl.s_full[q], 1);
      mbar_init(&ctrl.s_empty[q], 256);
    }
    mbar_init(&ctrl.gdp_full, 256);
    mbar_init(&ctrl.gdp_empty, 1);
    mbar_init(&ctrl.kop_full, 256);
    mbar_init(&ctrl.kop_empty, 1);
    mbar_init(&ctrl.acc_full, 1);
    mbar_init(&ctrl.drain_s, 1);
    mbar_init(&ctrl.drain_a, 1);
    fence_mbar_init();
    if ((smem_u32(smem) & 1023u) != 0u) {  // layout assumption; never expected
      ctrl.abort_flag = 1;
      atomicOr(p.err, kErrTimeout);
    }
  }
  if (warp == kMmaWarp) {
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

  if (warp == kProdWarp) {
    // ------------------------------------------------------------------ TMA
    // The whole warp runs the loop: lane 0 waits and issues the copies, all
    // lanes fill the vectors of a tile that cannot take a bulk copy.
    if (live) {
      if (lane_id == 0) {
        mbar_arrive_expect_tx(&ctrl.res_full, 2 * kDC * kChunk);
        for (int kc = 0; kc < kDC; ++kc) {
          tma_load_3d(smem + kRES_OFF + kc * kChunk, &p.mK, &ctrl.res_full, kc * 64, blk0, head);
          tma_load_3d(smem + kRES_OFF + (kDC + kc) * kChunk, &p.mUK, &ctrl.res_full, kc * 64, blk0, head);
        }
      }
      bool ok = true;
      int iq = 0, id = 0;   // [Q | UQ] and dO stages issued
      for (int t = 0; t < nt && ok; ++t) {
        const int tq = t_begin + t, sq = t % kNQ, sd = t % kND;
        int w = 1;
        if (lane_id == 0) w = mbar_wait(&ctrl.qu_empty[sq], ((t / kNQ) & 1) ^ 1, wt);
        if (!(ok = __shfl_sync(0xffffffffu, w, 0) != 0)) break;
        if (p.stall && t == 0) continue;  // test hook: nothing will fill this tile
        uint8_t* st = smem + kQU_OFF + sq * kQUS;
        // vectors by bulk copy only for whole tiles at 16-byte aligned addresses
        const bool whole = !RAGGED || (p.N % 4 == 0 && (tq + 1) * kQT <= p.N);
        if (!whole) {
          fill_vectors(p, reinterpret_cast<float*>(st + kQU), tq, head, lane_id);
          fence_proxy_async_smem();   // before later bulk copies into the same bytes
          __syncwarp();
        }
        if (lane_id == 0) {
          mbar_arrive_expect_tx(&ctrl.qu_full[sq], kQU + (whole ? kVEC : 0));
          for (int kc = 0; kc < kDC; ++kc) {
            tma_load_3d(st + kc * kQUCH, &p.mQ, &ctrl.qu_full[sq], kc * 64, tq * kQT, head);
            tma_load_3d(st + kc * kQUCH + kQB, &p.mUQ, &ctrl.qu_full[sq], kc * 64, tq * kQT, head);
          }
          if (whole) {
            const size_t v = (size_t)head * p.N + (size_t)tq * kQT;
            bulk_load(st + kQU, p.L + v, 4 * kQT, &ctrl.qu_full[sq]);
            bulk_load(st + kQU + 4 * kQT, p.D + v, 4 * kQT, &ctrl.qu_full[sq]);
            bulk_load(st + kQU + 8 * kQT, p.ws + 2 * v, 8 * kQT, &ctrl.qu_full[sq]);
          }
        }
        iq = t + 1;
        if (lane_id == 0) w = mbar_wait(&ctrl.do_empty[sd], ((t / kND) & 1) ^ 1, wt);
        if (!(ok = __shfl_sync(0xffffffffu, w, 0) != 0)) break;
        if (lane_id == 0) {
          mbar_arrive_expect_tx(&ctrl.do_full[sd], kDO);
          for (int kc = 0; kc < kDC; ++kc)
            tma_load_3d(smem + kDO_OFF + sd * kDO + kc * kQB, &p.mdO, &ctrl.do_full[sd], kc * 64, tq * kQT, head);
        }
        id = t + 1;
      }
      if (!ok && lane_id == 0) {
        // give-up path: every copy already issued lands before the CTA exits
        mbar_wait_drain(&ctrl.res_full, 0, kDrainNs);
        for (int t = (iq > kNQ ? iq - kNQ : 0); t < iq; ++t)
          mbar_wait_drain(&ctrl.qu_full[t % kNQ], (t / kNQ) & 1, kDrainNs);
        for (int t = (id > kND ? id - kND : 0); t < id; ++t)
          mbar_wait_drain(&ctrl.do_full[t % kND], (t / kND) & 1, kDrainNs);
      }
    }
  } else if (warp == kMmaWarp) {
    // --------------------------------------------------------- score MMAs
    // A(t) waits for its [Q | UQ] stage and for phase B of tile t-1 to have
    // been read from the score buffer; B(t) for its dO stage and for phase A
    // of tile t to have been read.
    if (live) {  // the whole warp runs the loop; lane 0 issues (elect.sync)
      const uint32_t res_l = desc_lo(sm0 + kRES_OFF, 16);
      const uint32_t i128 = idesc_bf16(kM, 2 * kQT, false, false), i64 = idesc_bf16(kM, kQT, false, false);
      const uint32_t tres = tb + kTRES;
      bool ok = __all_sync(0xffffffffu, mbar_wait(&ctrl.res_full, 0, wt));
      ok = ok && __all_sync(0xffffffffu, mbar_wait(&ctrl.tres_full, 0, wt));
      for (int t = 0; ok && t < nt; ++t) {
        const int sq = t % kNQ, sd = t % kND;
        ok = __all_sync(0xffffffffu, mbar_wait(&ctrl.qu_full[sq], (t / kNQ) & 1, wt));
        if (ok && t > 0) ok = __all_sync(0xffffffffu, mbar_wait(&ctrl.s_empty[1], (t - 1) & 1, wt));
        if (!ok) break;
        tc_fence_after();
        const uint32_t qu_l = desc_lo(sm0 + kQU_OFF + sq * kQUS, 16);
#pragma unroll
        for (int k = 0; k < kD / 16; ++k)  // [S^T | K UQ^T] = K [Q; UQ]^T
          mma_ss_w(tb + kSC, res_lo(res_l, 0, kDC, k), kmaj(qu_l, kQUCH, 0, k), i128, k > 0);
#pragma unroll
        for (int k = 0; k < kD / 16; ++k)  // B^T / tau += UK Q^T
          mma_ss_w(tb + kSC + kQT, res_lo(res_l, 1, kDC, k), kmaj(qu_l, kQUCH, 0, k), i64, 1);
        mma_commit_w(&ctrl.s_full[0]);
        ok = __all_sync(0xffffffffu, mbar_wait(&ctrl.do_full[sd], (t / kND) & 1, wt));
        ok = ok && __all_sync(0xffffffffu, mbar_wait(&ctrl.s_empty[0], t & 1, wt));
        if (!ok) break;
        tc_fence_after();
        const uint32_t do_l = desc_lo(sm0 + kDO_OFF + sd * kDO, 16);
#pragma unroll
        for (int k = 0; k < kD / 16; ++k) {
          mma_ts_w(tb + kSC, tres_a(tres, 0, kD, k), kmaj(do_l, kQB, 0, k), i64, k > 0);        // dP^T = V dO^T
          mma_ts_w(tb + kSC + kQT, tres_a(tres, 1, kD, k), kmaj(do_l, kQB, 0, k), i64, k > 0);  // C^T = UV dO^T
        }
        mma_commit_w(&ctrl.s_full[1]);
        mma_commit_w(&ctrl.do_empty[sd]);
      }
      mma_commit_w(&ctrl.drain_s);
      mbar_wait_drain(&ctrl.drain_s, 0, kDrainNs);
    }
  } else if (warp == kAccWarp) {
    // --------------------------------------------------- accumulator MMAs
    // gV(t) as soon as Gdp(t) is written (after phase A of tile t was read)
    // and tile t's dO has landed - phase A does not read dO, so Gdp(t) can
    // exist before it; gK(t) as soon as dS(t), Gs(t) are (after phase B).
    // The dO stage is released by gV(t) together with B(t) (other warp), the
    // [Q | UQ] stage by gK(t), which needs phase B's operands and so follows
    // every other reader of the stage.
    if (live) {
      const uint32_t id = idesc_bf16(kM, kD, false, true);
      const uint32_t ops_l = desc_lo(sm0 + kOPS_OFF, 16);
      bool ok = true;
      for (int t = 0; ok && t < nt; ++t) {
        const int sq = t % kNQ, sd = t % kND;
        ok = __all_sync(0xffffffffu, mbar_wait(&ctrl.gdp_full, t & 1, wt));
        ok = ok && __all_sync(0xffffffffu, mbar_wait(&ctrl.do_full[sd], (t / kND) & 1, wt));
        if (!ok) break;
        tc_fence_after();
        const uint32_t do_mn = desc_lo(sm0 + kDO_OFF + sd * kDO, kQB);
#pragma unroll
        for (int kk = 0; kk < kQT / 16; ++kk)  // gV += Gdp^T dO
          mma_ss_w(tb + kACC_V, op_lo(ops_l, kOP_GDP, 0, kk), mnmaj(do_mn, 0, kk), id, (t > 0 || kk > 0) ? 1u : 0u);
        mma_commit_w(&ctrl.gdp_empty);
        mma_commit_w(&ctrl.do_empty[sd]);
        ok = __all_sync(0xffffffffu, mbar_wait(&ctrl.kop_full, t & 1, wt));
        ok = ok && __all_sync(0xffffffffu, mbar_wait(&ctrl.qu_full[sq], (t / kNQ) & 1, wt));
        if (!ok) break;
        tc_fence_after();
        const uint32_t qu_mn = desc_lo(sm0 + kQU_OFF + sq * kQUS, kQUCH);
#pragma unroll
        for (int kk = 0; kk < kQT / 16; ++kk) {
          const uint32_t acc = (t > 0 || kk > 0) ? 1u : 0u;
          mma_ss_w(tb + kACC_K, op_lo(ops_l, kOP_DS, 0, kk), mnmaj(qu_mn, kQB, kk), id, acc);  // gK += dS^T UQ
          mma_ss_w(tb + kACC_K, op_lo(ops_l, kOP_GS, 0, kk), mnmaj(qu_mn, 0, kk), id, 1);      // gK += Gs^T Q
        }
        mma_commit_w(&ctrl.kop_empty);
        mma_commit_w(&ctrl.qu_empty[sq]);
      }
      if (ok) mma_commit_w(&ctrl.acc_full);
      mma_commit_w(&ctrl.drain_a);
      mbar_wait_drain(&ctrl.drain_a, 0, kDrainNs);
    }
  } else {
    // ------------------------------------------------------------ elementwise
    const int g = warp >> 2;                 // warpgroup: query columns 32g..32g+31
    const int r = tid & 127;                 // key row = TMEM lane
    const uint32_t lane = (uint32_t)((warp & 3) * 32) << 16;
    {
      // V (g = 0) or UV (g = 1) rows -> TMEM, two bf16 per column (rows at or
      // beyond N and columns at or beyond the head size are zeros)
      const bool row_ok = blk0 + r < p.N;
      const size_t row_g = (size_t)head * p.N + (row_ok ? blk0 + r : 0);
      const int dv8 = p.dv / 8;
      const uint4* src = reinterpret_cast<const uint4*>(g == 0 ? p.V : p.UV) + row_g * dv8;
      const uint32_t col = tb + lane + kTRES + (uint32_t)(g * (kD / 2));
#pragma unroll
      for (int cc = 0; cc < kD / 32; ++cc) {  // 16 columns = 32 bf16 per store
        uint32_t w[16];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint4 u = (row_ok && 4 * cc + q < dv8) ? src[4 * cc + q] : make_uint4(0u, 0u, 0u, 0u);
          w[4 * q] = u.x;
          w[4 * q + 1] = u.y;
          w[4 * q + 2] = u.z;
          w[4 * q + 3] = u.w;
        }
        tmem_st16_nowait(col + 16 * cc, w);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&ctrl.tres_full);
    }
    const int c0 = 32 * g;
    const uint32_t sc_col = tb + lane + kSC + (uint32_t)c0;
    const uint32_t ops = sm0 + kOPS_OFF;
    float2* rec = reinterpret_cast<float2*>(smem + kREC_OFF) + warp * 64;
    bool ok = live;
    for (int t = 0; t < nt && ok; ++t) {
      const int tq = t_begin + t;
      const float* vec = reinterpret_cast<const float*>(smem + kQU_OFF + (t % kNQ) * kQUS + kQU);
      // the tile's vectors arrive with its [Q | UQ] stage (warp-uniform wait:
      // the TMEM accesses that follow are warp-collective)
      if (!__all_sync(0xffffffffu, mbar_wait(&ctrl.qu_full[t % kNQ], (t / kNQ) & 1, wt))) { ok = false; break; }
      const int diag = blk0 + r - tq * kQT;   // this key's own index, as a tile column
      const int lo = CAUSAL ? diag : 0;
      const int hi = RAGGED ? min(kQT - 1, p.N - 1 - tq * kQT) : kQT - 1;
      // tiles that cross the diagonal or N take the masked variant; the vote
      // keeps the choice warp-uniform
      constexpr bool kMask = CAUSAL || RAGGED;
      if (kMask && __any_sync(0xffffffffu, lo > c0 || hi < c0 + 31))
        ok = ew_tile<kMask>(p, ctrl, wt, sc_col, ops, vec, rec, t, c0, lo, hi, r);
      else
        ok = ew_tile<false>(p, ctrl, wt, sc_col, ops, vec, rec, t, c0, lo, hi, r);
    }
    if (ok && __all_sync(0xffffffffu, mbar_wait(&ctrl.acc_full, 0, wt))) {
      tc_fence_after();
      // every lane runs the (warp-collective) TMEM loads; rows >= N store nothing
      const bool keep = blk0 + r < p.N;
      const size_t ro = ((size_t)head * p.N + (keep ? blk0 + r : 0)) * p.dv;
      const int c_lo = g * (kD / 2), c_hi = min(c_lo + kD / 2, p.dv);   // columns >= dv hold zeros
#pragma unroll 1
      for (int cc = c_lo; cc < c_hi; cc += 16) {
        float ak[16], av[16];
        tmem_ld16x2(tb + lane + kACC_K + cc, tb + lane + kACC_V + cc, ak, av);
#pragma unroll
        for (int j = 0; j < 16; ++j) ak[j] *= p.tau;
        if (keep) {
          store16(p.gK + ro + cc, ak);
          store16(p.gV + ro + cc, av);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tb, 512);
  }
}

}  // namespace

cudaError_t tc_bob_cols_wide(const BobArgs& a, const DevCtx& c, cudaStream_t s) {
  const int BH = a.BH, N = a.N;
  ColParams p;
  const bool ok = make_bf16_map(&p.mK, a.K, BH, N, a.d, kM) && make_bf16_map(&p.mUK, a.UK, BH, N, a.d, kM) &&
                  make_bf16_map(&p.mQ, a.Q, BH, N, a.d, kQT) && make_bf16_map(&p.mUQ, a.UQ, BH, N, a.d, kQT) &&
                  make_bf16_map(&p.mdO, a.dO, BH, N, a.d, kQT);
  if (!ok) return cudaErrorInvalidValue;
  p.V = static_cast<const __nv_bfloat16*>(a.V);
  p.UV = static_cast<const __nv_bfloat16*>(a.UV);
  p.L = a.L;
  p.D = a.D;
  p.ws = a.ws;
  p.gK = a.gK;
  p.gV = a.gV;
  p.N = N;
  p.dv = a.d;
  p.tau = a.tau;
  p.err = c.err;
  p.wait_ns = c.wait_ns;
  p.stall = c.stall;
  const bool ragged = N % kM != 0;
  auto kernel = a.causal ? (ragged ? bob_cols_wide<true, true> : bob_cols_wide<true, false>)
                         : (ragged ? bob_cols_wide<false, true> : bob_cols_wide<false, false>);
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSMEM);
  if (e != cudaSuccess) return e;
  const dim3 grid((N + kM - 1) / kM, BH);
  prof_begin(s, "bob_pass2");
  kernel<<<grid, kThreads, kSMEM, s>>>(p);
  prof_end(s);
  return cudaGetLastError();
}

}  // namespace fbob
