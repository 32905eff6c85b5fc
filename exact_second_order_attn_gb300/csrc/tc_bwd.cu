// Tensor-core (tcgen05 + TMEM + TMA) first backward for bf16 inputs, d in
// {64, 128}, any N, on the tile skeleton of tc_tile.cuh.  It
// produces dQ, dK, dV and D = rowsum(dO o O), the row term BoB reads.
//
// Source: "FlashBoB: I/O-Efficient Exact Backward-over-Backward for Softmax
// Attention" - the abstract (the FlashAttention-style first backward that BoB
// differentiates through) and the evolve.pub review FAQ "What is
// backward-over-backward (BoB)" (BoB is the vector-Jacobian product of this map).
//
//   row kernel (128 query rows): D = rowsum(dO o O); S = Q K^T, dP = dO V^T;
//     dS = P (dP - D); dQ += dS K; dQ *= tau.
//   column kernel (128 keys): S^T = K Q^T, dP^T = V dO^T; dV += P^T dO;
//     dK += dS^T Q; dK *= tau.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "prof.h"
#include "tc_tile.cuh"

namespace fbob {
namespace {

using namespace tc;
using tile::kM;

// ===========================================================================
// first backward on the tile skeleton
// ===========================================================================
struct DqParams {
  CUtensorMap mK, mV;      // streamed
  const __nv_bfloat16 *Q, *dO;   // resident (copied into TMEM)
  const float *O, *L;
  float *dQ, *D;
  int N;
  int dv;                  // head size in global memory (<= D; see tc_tile.cuh)
  float tau;
  int causal;
  unsigned int* err;
  unsigned long long wait_ns;
  int stall;
};

// Row kernel: resident Q, dO in TMEM (A operands of the score MMAs); ring A
// = K (read by dQ += dS K), ring B = V (read only by dP = dO V^T), 64 keys
// per tile.  TMEM: dQ (d) | [S | dP] x 2 | Q, dO (d) and, at d = 64, the dS
// halves (TS MMA); at d = 128 dS goes to shared memory (SS MMA).
template <int D_>
struct DqOp {
  using Params = DqParams;
  static constexpr bool SPLIT = false, ROWS = true;
  static constexpr int D = D_, DC = D / 64, T = 64, BLK = T * 128;
  static constexpr int RES = 0, TRES = 2;
  static constexpr int ACH = BLK, BCH = BLK;
  static constexpr int SA = DC * ACH, SB = DC * BCH, SA_TX = SA, SB_TX = SB;
  static constexpr int NSA = D == 128 ? 5 : 8, NSB = NSA;
  static constexpr bool VEC = false, ROW_SUMS = false, TS = D == 64;
  static constexpr int VEC_OFF = 0, NVEC = 0, VEC_SCRATCH = 0;
  static constexpr int OPS = TS ? 0 : 2 * tile::kChunk;  // dS, one [128][64] tile per half
  static constexpr int ACC = D, SCOLS = 2 * T, NBUF = 2;   // [S | dP]
  static constexpr int OP_HALF = T / 2, OP_COL = ACC + NBUF * SCOLS;
  static constexpr int TRES_COL = OP_COL + (TS ? 2 * OP_HALF : 0);
  static constexpr int SMEM = NSA * SA + NSB * SB + OPS;
  static_assert(TRES_COL + TRES * D / 2 <= 512, "TMEM budget");
  static_assert(SMEM + 1024 <= 232448, "shared memory budget");

  __device__ static const void* tres_src(const Params& p, int s) { return s == 0 ? (const void*)p.Q : (const void*)p.dO; }
  __device__ static void load_res(const Params&, uint8_t*, uint64_t*, int, int) {}
  __device__ static void load_a(const Params& p, uint8_t* st, uint64_t* bar, int t, int head, bool) {
    for (int kc = 0; kc < DC; ++kc) tma_load_3d(st + kc * ACH, &p.mK, bar, kc * 64, t * T, head);
  }
  __device__ static void fill_vec(const Params&, float*, int, int, int) {}
  __device__ static void load_b(const Params& p, uint8_t* st, uint64_t* bar, int t, int head) {
    for (int kc = 0; kc < DC; ++kc) tma_load_3d(st + kc * BCH, &p.mV, bar, kc * 64, t * T, head);
  }
  __device__ static void score_mmas(uint32_t sc, uint32_t tres, uint32_t, uint32_t sa, uint32_t sb) {
    const uint32_t i64 = idesc_bf16(tile::kM, T, false, false);
#pragma unroll
    for (int k = 0; k < D / 16; ++k) {
      mma_ts_w(sc, tile::tres_a(tres, 0, D, k), tile::kmaj(sa, ACH, 0, k), i64, k > 0);      // S = Q K^T
      mma_ts_w(sc + T, tile::tres_a(tres, 1, D, k), tile::kmaj(sb, BCH, 0, k), i64, k > 0);  // dP = dO V^T
    }
  }
  __device__ static void accum_mmas(uint32_t tb, uint32_t ops, uint32_t sa, uint32_t h, bool first) {
    const uint32_t amn = desc_lo(sa, ACH);
    const uint32_t id = idesc_bf16(tile::kM, D, false, true);
#pragma unroll
    for (int kk = 0; kk < T / 16; ++kk) {  // dQ += dS K
      const uint32_t acc = (first && kk == 0) ? 0u : 1u;
      if (TS)
        mma_ts_w(tb, ops + h * OP_HALF + kk * 8, tile::mnmaj(amn, 0, kk), id, acc);
      else
        mma_ss_w(tb, tile::op64_lo(ops, 0, h, kk), tile::mnmaj(amn, 0, kk), id, acc);
    }
  }
  struct Row {
    float nL, Di;
  };
  __device__ static void ew_init(Row& w, const Params& p, int blk0, int r, int head) {
    w.Di = 0.f;
    w.nL = 0.f;
    if (blk0 + r >= p.N) return;   // ragged N: row past the end (never stored)
    const size_t vo = (size_t)head * p.N + blk0 + r;
    const size_t ro = vo * p.dv;
    // D_i = rowsum(dO o O) of this thread's row
    float Di = 0.f;
    const uint4* g = reinterpret_cast<const uint4*>(p.dO + ro);
    const float4* o = reinterpret_cast<const float4*>(p.O + ro);
#pragma unroll 4
    for (int c = 0; c < p.dv / 8; ++c) {
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
    if (threadIdx.x < 128) p.D[vo] = Di;  // one of the two warpgroups writes it
    w.Di = Di;
    w.nL = -p.L[vo] * tile::kLog2e;
  }
  template <bool MASK>
  __device__ static bool ew_tile(Row& w, const Params& p, const tile::TileArgs& a, const tile::TileSync& s, int r) {
    const float sc = p.tau * tile::kLog2e;
    uint32_t wd[T / 2];
#pragma unroll
    for (int q = 0; q < T / 16; ++q) {
      float S[16], dP[16];
      tmem_ld16x2(a.sc + q * 16, a.sc + T + q * 16, S, dP);
      if (q == T / 16 - 1) s.release_scores();
#pragma unroll
      for (int j = 0; j < 16; j += 2) {
        const int c = q * 16 + j;   // tile column (key)
        const float p0 = (!MASK || (c >= a.lo && c <= a.hi)) ? tile::ex2(fmaf(S[j], sc, w.nL)) : 0.f;
        const float p1 = (!MASK || (c + 1 >= a.lo && c + 1 <= a.hi)) ? tile::ex2(fmaf(S[j + 1], sc, w.nL)) : 0.f;
        wd[q * 8 + j / 2] = pack_bf16x2(p0 * (dP[j] - w.Di), p1 * (dP[j + 1] - w.Di));
      }
    }
    if (!s.acquire_ops()) return false;
    if (TS) {
      tmem_st16_nowait(a.ops, wd);
      tmem_st16_nowait(a.ops + 16, wd + 16);
    } else {
      tile::write_op64(a.ops + a.h * tile::kChunk, (uint32_t)r, wd);
    }
    s.publish_ops();
    return true;
  }
  __device__ static void epilogue(Row&, const Params& p, const tile::EpiArgs& e) {
    // every lane runs the (warp-collective) TMEM loads; rows >= N store nothing
    const bool keep = e.blk0 + e.r < p.N;
    const size_t ro = ((size_t)e.head * p.N + (keep ? e.blk0 + e.r : 0)) * p.dv;
    const int c_lo = e.g * (D / 2), c_hi = min(c_lo + D / 2, p.dv);   // columns >= dv hold zeros
#pragma unroll 1
    for (int c0 = c_lo; c0 < c_hi; c0 += 16) {
      float v[16];
      tmem_ld16(e.tm + c0, v);
#pragma unroll
      for (int j = 0; j < 16; ++j) v[j] *= p.tau;
      if (keep) tile::store16(p.dQ + ro + c0, v);
    }
  }
};

struct DkvParams {
  CUtensorMap mQ, mdO;     // streamed
  const __nv_bfloat16 *K, *V;   // resident (copied into TMEM)
  const float *L, *D;
  float *dK, *dV;
  int N;
  int dv;                  // head size in global memory (<= D; see tc_tile.cuh)
  float tau;
  int causal;
  unsigned int* err;
  unsigned long long wait_ns;
  int stall;
};

// Column kernel: resident K, V in TMEM; ring A = [Q | dO] + (L, D) of the
// tile, 64 queries per tile.  P and dS go to shared memory (SS MMAs).
// TMEM: dK, dV (2d) | [S^T | dP^T] x NBUF | K, V (d); one score buffer at d = 128.
template <int D_>
struct DkvOp {
  using Params = DkvParams;
  static constexpr bool ROWS = false;
  static constexpr int D = D_, DC = D / 64, T = 64, BLK = T * 128;
  static constexpr int RES = 0, TRES = 2;
  static constexpr int ACH = 2 * BLK, VEC_OFF = DC * ACH;
  static constexpr int SA = DC * ACH + 1024, SA_TX = DC * ACH + 2 * T * 4, SB = 0, SB_TX = 0;
  static constexpr int NSA = D == 128 ? 4 : 8, NSB = 0;
  static constexpr bool VEC = true, ROW_SUMS = false, TS = false;
  static constexpr int OPS = 4 * tile::kChunk;   // P, dS: one [128][64] tile per operand and half
  static constexpr int ACC = 2 * D, SCOLS = 2 * T, NBUF = D == 128 ? 1 : 2;   // dK, dV; [S^T | dP^T]
  static constexpr int OP_HALF = 0, OP_COL = ACC + NBUF * SCOLS;
  static constexpr int TRES_COL = OP_COL;
  static constexpr int NVEC = 2;                          // L, D per query
  static constexpr int VEC_SCRATCH = NSA * SA + OPS;      // 2 warpgroups x 2 buffers x NVEC x T floats
  static constexpr int SMEM = VEC_SCRATCH + 4 * NVEC * T * 4;
  static_assert(TRES_COL + TRES * D / 2 <= 512, "TMEM budget");
  static_assert(SMEM + 1024 <= 232448, "shared memory budget");

  __device__ static const void* tres_src(const Params& p, int s) { return s == 0 ? (const void*)p.K : (const void*)p.V; }
  __device__ static void load_res(const Params&, uint8_t*, uint64_t*, int, int) {}
  __device__ static void load_a(const Params& p, uint8_t* st, uint64_t* bar, int t, int head, bool whole) {
    for (int kc = 0; kc < DC; ++kc) {
      tma_load_3d(st + kc * ACH, &p.mQ, bar, kc * 64, t * T, head);
      tma_load_3d(st + kc * ACH + BLK, &p.mdO, bar, kc * 64, t * T, head);
    }
    if (!whole) return;   // ragged last tile: fill_vec
    const size_t v = (size_t)head * p.N + (size_t)t * T;
    tile::bulk_load(st + VEC_OFF, p.L + v, T * 4, bar);
    tile::bulk_load(st + VEC_OFF + T * 4, p.D + v, T * 4, bar);
  }
  // L, D of tile t with bounds checks (128 threads, thread i)
  __device__ static void fill_vec(const Params& p, float* dst, int t, int head, int i) {
    for (int k = i; k < 2 * T; k += 128) {
      const int q = t * T + (k % T);
      const float* src = k < T ? p.L : p.D;
      dst[k] = q < p.N ? src[(size_t)head * p.N + q] : 0.f;
    }
  }
  __device__ static void load_b(const Params&, uint8_t*, uint64_t*, int, int) {}
  __device__ static void score_mmas(uint32_t sc, uint32_t tres, uint32_t, uint32_t sa, uint32_t) {
    const uint32_t i64 = idesc_bf16(tile::kM, T, false, false);
#pragma unroll
    for (int k = 0; k < D / 16; ++k) {
      mma_ts_w(sc, tile::tres_a(tres, 0, D, k), tile::kmaj(sa, ACH, 0, k), i64, k > 0);        // S^T = K Q^T
      mma_ts_w(sc + T, tile::tres_a(tres, 1, D, k), tile::kmaj(sa, ACH, BLK, k), i64, k > 0);  // dP^T = V dO^T
    }
  }
  __device__ static void accum_mmas(uint32_t tb, uint32_t ops, uint32_t sa, uint32_t h, bool first) {
    const uint32_t amn = desc_lo(sa, ACH);
    const uint32_t id = idesc_bf16(tile::kM, D, false, true);
#pragma unroll
    for (int kk = 0; kk < T / 16; ++kk) {
      const uint32_t acc = (first && kk == 0) ? 0u : 1u;
      mma_ss_w(tb + D, tile::op64_lo(ops, 0, h, kk), tile::mnmaj(amn, BLK, kk), id, acc);  // dV += P^T dO
      mma_ss_w(tb, tile::op64_lo(ops, 1, h, kk), tile::mnmaj(amn, 0, kk), id, acc);        // dK += dS^T Q
    }
  }
  struct Row {};
  __device__ static void ew_init(Row&, const Params&, int, int, int) {}
  // NC query columns per warpgroup and tile: all T with two score buffers,
  // T / 2 (starting at a.c0) when both warpgroups share the one buffer.
  static constexpr bool SPLIT = NBUF == 1;
  static constexpr int NC = SPLIT ? T / 2 : T;
  template <bool MASK>
  __device__ static bool ew_tile(Row&, const Params& p, const tile::TileArgs& a, const tile::TileSync& s, int r) {
    const float sc = p.tau * tile::kLog2e;
    const float* vL = a.vec + a.c0;
    const float* vD = a.vec + T + a.c0;
    // With one score buffer its release is on the critical path, so the
    // operand tiles are taken only after all scores are read; with two, they
    // are taken first and each 16-column chunk is written as soon as it is
    // computed (fewer live registers).
    constexpr bool kEarly = NBUF > 1;
    if (kEarly && !s.acquire_ops()) return false;
    uint32_t wP[kEarly ? 8 : NC / 2], wd[kEarly ? 8 : NC / 2];
#pragma unroll
    for (int q = 0; q < NC / 16; ++q) {
      float S[16], dP[16];
      tmem_ld16x2(a.sc + a.c0 + q * 16, a.sc + T + a.c0 + q * 16, S, dP);
      if (q == NC / 16 - 1) s.release_scores();
      const int o = kEarly ? 0 : q * 8;
#pragma unroll
      for (int c = 0; c < 16; c += 2) {
        const int ii = q * 16 + c, col = a.c0 + ii;   // tile column (query)
        const float p0 = (!MASK || (col >= a.lo && col <= a.hi)) ? tile::ex2(fmaf(S[c], sc, -vL[ii] * tile::kLog2e)) : 0.f;
        const float p1 =
            (!MASK || (col + 1 >= a.lo && col + 1 <= a.hi)) ? tile::ex2(fmaf(S[c + 1], sc, -vL[ii + 1] * tile::kLog2e)) : 0.f;
        wP[o + c / 2] = pack_bf16x2(p0, p1);
        wd[o + c / 2] = pack_bf16x2(p0 * (dP[c] - vD[ii]), p1 * (dP[c + 1] - vD[ii + 1]));
      }
      if (kEarly) {
        tile::write_op_cols<8>(a.ops + a.h * tile::kChunk, (uint32_t)r, a.c0 + q * 16, wP);
        tile::write_op_cols<8>(a.ops + (2 + a.h) * tile::kChunk, (uint32_t)r, a.c0 + q * 16, wd);
      }
    }
    if (!kEarly) {
      if (!s.acquire_ops()) return false;
      tile::write_op_cols<NC / 2>(a.ops + a.h * tile::kChunk, (uint32_t)r, a.c0, wP);
      tile::write_op_cols<NC / 2>(a.ops + (2 + a.h) * tile::kChunk, (uint32_t)r, a.c0, wd);
    }
    s.publish_ops();
    return true;
  }
  __device__ static void epilogue(Row&, const Params& p, const tile::EpiArgs& e) {
    // every lane runs the (warp-collective) TMEM loads; rows >= N store nothing
    const bool keep = e.blk0 + e.r < p.N;
    const size_t ro = ((size_t)e.head * p.N + (keep ? e.blk0 + e.r : 0)) * p.dv;
    const int c_lo = e.g * (D / 2), c_hi = min(c_lo + D / 2, p.dv);   // columns >= dv hold zeros
#pragma unroll 1
    for (int c0 = c_lo; c0 < c_hi; c0 += 16) {
      float k_[16], v[16];
      tmem_ld16x2(e.tm + c0, e.tm + D + c0, k_, v);
#pragma unroll
      for (int j = 0; j < 16; ++j) k_[j] *= p.tau;
      if (keep) {
        tile::store16(p.dK + ro + c0, k_);
        tile::store16(p.dV + ro + c0, v);
      }
    }
  }
};

// ===========================================================================
// host side
// ===========================================================================
template <typename K, typename Params>
cudaError_t launch(const char* name, K kernel, int smem, int threads, dim3 grid, const Params& prm, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  prof_begin(s, name);
  kernel<<<grid, threads, smem, s>>>(prm);
  prof_end(s);
  return cudaGetLastError();
}

// the instantiation for (causal, ragged N)
template <class Op>
auto pick(bool causal, bool ragged) {
  return causal ? (ragged ? tile::tile_kernel<Op, true, true> : tile::tile_kernel<Op, true, false>)
                : (ragged ? tile::tile_kernel<Op, false, true> : tile::tile_kernel<Op, false, false>);
}

template <int D>
cudaError_t bwd_group(const BwdArgs& a, const DevCtx& c, cudaStream_t s) {
  DqParams q;
  if (!make_bf16_map(&q.mK, a.K, a.BH, a.N, a.d, DqOp<D>::T) || !make_bf16_map(&q.mV, a.V, a.BH, a.N, a.d, DqOp<D>::T))
    return cudaErrorInvalidValue;
  q.Q = static_cast<const __nv_bfloat16*>(a.Q);
  q.O = a.O;
  q.L = a.L;
  q.dO = static_cast<const __nv_bfloat16*>(a.dO);
  q.dQ = a.dQ;
  q.D = a.D;
  q.N = a.N;
  q.dv = a.d;
  q.tau = a.tau;
  q.causal = a.causal;
  q.err = c.err;
  q.wait_ns = c.wait_ns;
  q.stall = c.stall;
  const dim3 grid((a.N + kM - 1) / kM, a.BH);
  const bool ragged = a.N % kM != 0;
  cudaError_t e = launch("attn_bwd_dq", pick<DqOp<D>>(a.causal, ragged), DqOp<D>::SMEM, tile::kThreads, grid, q, s);
  if (e != cudaSuccess) return e;
  DkvParams k;
  if (!make_bf16_map(&k.mQ, a.Q, a.BH, a.N, a.d, DkvOp<D>::T) || !make_bf16_map(&k.mdO, a.dO, a.BH, a.N, a.d, DkvOp<D>::T))
    return cudaErrorInvalidValue;
  k.K = static_cast<const __nv_bfloat16*>(a.K);
  k.V = static_cast<const __nv_bfloat16*>(a.V);
  k.L = a.L;
  k.D = a.D;
  k.dK = a.dK;
  k.dV = a.dV;
  k.N = a.N;
  k.dv = a.d;
  k.tau = a.tau;
  k.causal = a.causal;
  k.err = c.err;
  k.wait_ns = c.wait_ns;
  k.stall = c.stall;
  return launch("attn_bwd_dkdv", pick<DkvOp<D>>(a.causal, ragged), DkvOp<D>::SMEM, tile::kThreads, grid, k, s);
}

// Heads [h0, h0 + n) of a: every per-head array starts h0 heads further on.
BwdArgs head_range(const BwdArgs& a, int h0, int n) {
  const size_t nd = (size_t)a.N * a.d, n1 = (size_t)a.N;
  auto bf = [&](const void* p) { return static_cast<const void*>(static_cast<const char*>(p) + 2 * h0 * nd); };
  BwdArgs b = a;
  b.Q = bf(a.Q), b.K = bf(a.K), b.V = bf(a.V), b.dO = bf(a.dO);
  b.O = a.O + h0 * nd, b.L = a.L + h0 * n1;
  b.dQ = a.dQ + h0 * nd, b.dK = a.dK + h0 * nd, b.dV = a.dV + h0 * nd, b.D = a.D + h0 * n1;
  b.BH = n;
  return b;
}

// The dK/dV kernel reads the D the dq kernel writes, so the two run in stream
// order.  When each launch would end on a mostly empty wave, the heads run as
// two groups on two streams (as BoB does, tc_bob.cu) so that one group's dK/dV
// kernel fills the SMs the other group's dq tail leaves idle.
bool split_heads(const BwdArgs& a) {
  const int sms = sm_count();
  if (a.BH < 2 || sms <= 0) return false;
  const long ctas = (long)a.BH * ((a.N + kM - 1) / kM);
  const long waves = (ctas + sms - 1) / sms;
  return waves <= 16 && (waves * sms - ctas) * 20 > waves * sms;
}

template <int D>
cudaError_t bwd_d(const BwdArgs& a, const DevCtx& c, cudaStream_t s) {
  if (!split_heads(a)) return bwd_group<D>(a, c, s);
  SideStream side;
  if (side.fork(s) != cudaSuccess) return bwd_group<D>(a, c, s);   // no side stream: run unsplit
  const int h1 = a.BH / 2;
  cudaError_t e0 = bwd_group<D>(head_range(a, 0, h1), c, s);
  cudaError_t e1 = bwd_group<D>(head_range(a, h1, a.BH - h1), c, side.stream());
  cudaError_t e2 = side.join();
  return e0 != cudaSuccess ? e0 : e1 != cudaSuccess ? e1 : e2;
}

}  // namespace

cudaError_t tc_bwd(const BwdArgs& a, const DevCtx& c, cudaStream_t s) {
  // d = 32, 96 run on the d = 64, 128 kernels with zero-padded columns
  return a.d <= 64 ? bwd_d<64>(a, c, s) : bwd_d<128>(a, c, s);
}

}  // namespace fbob

#ifdef FBOB_TRACE
FBOB_TRACE_IO(fbob_trace_io_bwd)
#endif
