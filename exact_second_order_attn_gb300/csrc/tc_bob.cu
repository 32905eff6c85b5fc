// Tensor-core (tcgen05 + TMEM + TMA) kernels of the two-pass BoB for bf16
// inputs, d in {64, 128}, N a multiple of 128, built on the tile skeleton of
// tc_tile.cuh.
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
// TMEM budget (512 columns x 128 lanes fp32).  d=64 pass 1 holds all four
// accumulators (4 x 64) and two score buffers ([S|B|dP|C], 128 columns each).
// At d=128 the four accumulators alone fill TMEM, so pass 1 runs as two CTA
// kinds over the same row blocks: the Q side (U1, U2, W = 384 columns + one
// score buffer) writes gQ and alpha/E; the dO side (Y) recomputes S and B and
// writes gdO, with its P / PB operands in TMEM.  Pass 2 keeps gK, gV (2d
// columns), its score buffer(s) and its three operands (dS, Gs, Gdp) in TMEM.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "internal.h"
#include "prof.h"
#include "tc_tile.cuh"

namespace fbob {
namespace {

using namespace tc;
using namespace tile;

enum Role { kBoth = 0, kQSide = 1, kDoSide = 2 };

struct P1Params {
  CUtensorMap mQ, mdO, mUQ;        // resident, box {64, 128}
  CUtensorMap mK, mUK, mV, mUV;    // streamed, box {64, 32}
  const float *L, *D, *O;
  float *gQ, *gdO, *ws;
  int N;
  float tau;
  unsigned int* err;
  unsigned long long wait_ns;
  int stall;
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
  int stall;
};

// ===========================================================================
// pass 1
// ===========================================================================
template <int D_, int ROLE>
struct Pass1 {
  using Params = P1Params;
  static constexpr int D = D_, DC = D / 64;
  static constexpr bool kQ = ROLE != kDoSide;   // gQ, alpha, E
  static constexpr bool kDo = ROLE != kQSide;   // gdO
  // resident slots: Q, UQ, dO
  static constexpr int NRES = kQ ? 3 : 2;
  static constexpr int RES = NRES * DC * kChunk;
  // ring A holds what the accumulator MMAs read, ring B what only the score
  // MMAs read:  both: A = [K UK V UV];  Q side: A = [K UK], B = [V UV];
  // dO side: A = [V UV], B = [K UK]
  static constexpr int ABLK = ROLE == kBoth ? 4 : 2, BBLK = ROLE == kBoth ? 0 : 2;
  static constexpr int ACH = ABLK * kBlk, BCH = BBLK * kBlk;
  static constexpr int SA = DC * ACH, SB = DC * BCH, SA_TX = SA, SB_TX = SB;
  static constexpr int NSA = ROLE == kQSide ? 3 : 4;
  static constexpr int NSB = ROLE == kBoth ? 0 : (ROLE == kQSide ? 2 : 4);
  static constexpr bool VEC = false;
  static constexpr int VEC_OFF = 0;
  static constexpr bool ROW_SUMS = true;
  static constexpr bool TS = ROLE == kDoSide;
  static constexpr int NOPS = TS ? 0 : 1 + (kQ ? 2 : 0) + (kDo ? 1 : 0);  // P, dS, X, PB tiles
  static constexpr int OPS = NOPS * kChunk;
  static constexpr int ACC = ((kQ ? 3 : 0) + (kDo ? 1 : 0)) * D;
  static constexpr int SCOLS = kQ ? 128 : 64;    // [S|B|dP|C] or [S|B]
  static constexpr int NBUF = ROLE == kQSide ? 1 : 2;
  static constexpr int OP_HALF = 32;             // TS: P, PB (16 columns each)
  static constexpr int OP_COL = ACC + NBUF * SCOLS;
  static constexpr int SMEM = RES + NSA * SA + NSB * SB + OPS;
  static_assert(OP_COL + (TS ? 2 * OP_HALF : 0) <= 512, "TMEM budget");
  static_assert(SMEM + 1024 <= 232448, "shared memory budget (1 KB static)");
  static_assert(NSA <= kMaxStages && NSB <= kMaxStages, "stage count");
  // where K, UK (= K block + 1) and V, UV (= V block + 1) live
  static constexpr bool K_IN_B = ROLE == kDoSide, V_IN_B = ROLE == kQSide;
  static constexpr int K_BLK = 0, V_BLK = ROLE == kBoth ? 2 : 0;
  static constexpr int A_U1 = 0, A_U2 = D, A_W = 2 * D, A_Y = kQ ? 3 * D : 0;
  static constexpr int O_P = 0, O_DS = 1, O_X = 2, O_PB = kQ ? 3 : 1;

  __device__ static void load_res(const Params& p, uint8_t* res, uint64_t* bar, int row0, int head) {
    const CUtensorMap* m[3] = {&p.mQ, &p.mUQ, &p.mdO};
    for (int s = 0; s < NRES; ++s)
      for (int kc = 0; kc < DC; ++kc) tma_load_3d(res + (s * DC + kc) * kChunk, m[s], bar, kc * 64, row0, head);
  }
  __device__ static void load_a(const Params& p, uint8_t* st, uint64_t* bar, int t, int head) {
    for (int kc = 0; kc < DC; ++kc) {
      uint8_t* c = st + kc * ACH;
      if (ROLE == kBoth || ROLE == kQSide) {
        tma_load_3d(c, &p.mK, bar, kc * 64, t * kT, head);
        tma_load_3d(c + kBlk, &p.mUK, bar, kc * 64, t * kT, head);
      }
      if (ROLE == kBoth || ROLE == kDoSide) {
        uint8_t* v = c + V_BLK * kBlk;
        tma_load_3d(v, &p.mV, bar, kc * 64, t * kT, head);
        tma_load_3d(v + kBlk, &p.mUV, bar, kc * 64, t * kT, head);
      }
    }
  }
  __device__ static void load_b(const Params& p, uint8_t* st, uint64_t* bar, int t, int head) {
    const CUtensorMap* m0 = ROLE == kQSide ? &p.mV : &p.mK;
    const CUtensorMap* m1 = ROLE == kQSide ? &p.mUV : &p.mUK;
    for (int kc = 0; kc < DC; ++kc) {
      tma_load_3d(st + kc * BCH, m0, bar, kc * 64, t * kT, head);
      tma_load_3d(st + kc * BCH + kBlk, m1, bar, kc * 64, t * kT, head);
    }
  }

  __device__ static void score_mmas(uint32_t sc, uint32_t res, uint32_t sa, uint32_t sb) {
    const uint32_t kst = K_IN_B ? sb : sa, vst = V_IN_B ? sb : sa;
    const int kch = K_IN_B ? BCH : ACH, vch = V_IN_B ? BCH : ACH;
    const uint32_t i64 = idesc_bf16(kM, 64, false, false), i32 = idesc_bf16(kM, 32, false, false);
#pragma unroll
    for (int k = 0; k < D / 16; ++k)  // [S | Q UK^T] = Q [K; UK]^T
      mma_ss_w(sc, res_lo(res, 0, DC, k), kmaj_lo(kst, kch, K_BLK, k), i64, k > 0);
#pragma unroll
    for (int k = 0; k < D / 16; ++k)  // B += UQ K^T
      mma_ss_w(sc + 32, res_lo(res, 1, DC, k), kmaj_lo(kst, kch, K_BLK, k), i32, 1);
    if (kQ) {
#pragma unroll
      for (int k = 0; k < D / 16; ++k)  // [dP | C] = dO [V; UV]^T
        mma_ss_w(sc + 64, res_lo(res, 2, DC, k), kmaj_lo(vst, vch, V_BLK, k), i64, k > 0);
    }
  }

  __device__ static void accum_mmas(uint32_t tb, uint32_t ops, uint32_t sa, uint32_t h, bool first) {
    const uint32_t amn = desc_lo(sa, ACH);
    const uint32_t id = idesc_bf16(kM, D, false, true);
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
      const uint32_t acc0 = (first && kk == 0) ? 0u : 1u;
      auto op = [&](int slot) { return op_lo(ops, slot, h, kk); };
      if (kQ) {
        mma_ss_w(tb + A_U1, op(O_DS), mn_lo(amn, K_BLK + 1, kk), id, acc0);  // dS UK
        mma_ss_w(tb + A_U1, op(O_X), mn_lo(amn, K_BLK, kk), id, 1);          // X K
        mma_ss_w(tb + A_U2, op(O_P), mn_lo(amn, K_BLK, kk), id, acc0);       // P K
        mma_ss_w(tb + A_W, op(O_DS), mn_lo(amn, K_BLK, kk), id, acc0);       // dS K
      }
      if (kDo) {
        if (TS) {
          const uint32_t a = ops + h * OP_HALF + kk * 8;
          mma_ts_w(tb + A_Y, a, mn_lo(amn, V_BLK + 1, kk), id, acc0);        // P UV
          mma_ts_w(tb + A_Y, a + 16, mn_lo(amn, V_BLK, kk), id, 1);          // PB V
        } else {
          mma_ss_w(tb + A_Y, op(O_P), mn_lo(amn, V_BLK + 1, kk), id, acc0);  // P UV
          mma_ss_w(tb + A_Y, op(O_PB), mn_lo(amn, V_BLK, kk), id, 1);        // PB V
        }
      }
    }
  }

  struct Row {
    float nL, Di, alpha, ex;
  };
  __device__ static void ew_init(Row& w, const Params& p, int blk0, int r, int head) {
    const size_t vo = (size_t)head * p.N + blk0 + r;
    w.nL = -p.L[vo] * kLog2e;
    w.Di = p.D[vo];
    w.alpha = 0.f;
    w.ex = 0.f;
  }

  __device__ static bool ew_tile(Row& w, const Params& p, const TileArgs& a, const TileSync& s, int r) {
    const float sc = p.tau * kLog2e;
    uint32_t wP[16], wdS[16], wX[16], wPB[16];
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      float S[16], B[16], dP[16], C[16];
      if (kQ)
        tmem_ld16x4(a.sc + q * 16, a.sc + 32 + q * 16, a.sc + 64 + q * 16, a.sc + 96 + q * 16, S, B, dP, C);
      else
        tmem_ld16x2(a.sc + q * 16, a.sc + 32 + q * 16, S, B);
      if (q == 1) s.release_scores();
#pragma unroll
      for (int j = 0; j < 16; j += 2) {
        float pv[2], dsv[2], xv[2], pbv[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float pe = ex2(fmaf(S[j + e], sc, w.nL));
          const float be = p.tau * B[j + e];
          pv[e] = pe;
          pbv[e] = pe * be;
          w.alpha += pbv[e];
          if (kQ) {
            const float te = dP[j + e] - w.Di;
            dsv[e] = pe * te;
            xv[e] = pe * fmaf(be, te, C[j + e]);
            w.ex += xv[e];
          }
        }
        const int k = q * 8 + j / 2;
        wP[k] = pack_bf16x2(pv[0], pv[1]);
        wPB[k] = pack_bf16x2(pbv[0], pbv[1]);
        if (kQ) {
          wdS[k] = pack_bf16x2(dsv[0], dsv[1]);
          wX[k] = pack_bf16x2(xv[0], xv[1]);
        }
      }
    }
    if (!s.acquire_ops()) return false;
    if (TS) {
      tmem_st16_nowait(a.ops, wP);
      tmem_st16_nowait(a.ops + 16, wPB);
    } else {
      write_op_half(a.ops + O_P * kChunk, r, a.h, wP);
      if (kQ) {
        write_op_half(a.ops + O_DS * kChunk, r, a.h, wdS);
        write_op_half(a.ops + O_X * kChunk, r, a.h, wX);
      }
      if (kDo) write_op_half(a.ops + O_PB * kChunk, r, a.h, wPB);
    }
    s.publish_ops();
    return true;
  }

  __device__ static void epilogue(Row& w, const Params& p, const EpiArgs& e) {
    float alpha = w.alpha, ex = w.ex;
    if (!e.sum_rows(alpha, ex)) return;
    const size_t vo = (size_t)e.head * p.N + e.blk0 + e.r;
    const size_t ro = vo * D;
    const int c_lo = e.g * (D / 2), c_hi = c_lo + D / 2;
    if (kQ) {
#pragma unroll 1
      for (int c0 = c_lo; c0 < c_hi; c0 += 16) {
        float u1[16], u2[16], wv[16], o[16];
        tmem_ld16x2(e.tm + A_U1 + c0, e.tm + A_U2 + c0, u1, u2);
        tmem_ld16(e.tm + A_W + c0, wv);
#pragma unroll
        for (int j = 0; j < 16; ++j) o[j] = p.tau * (u1[j] - ex * u2[j] - alpha * wv[j]);
        store16(p.gQ + ro + c0, o);
      }
      if (e.g == 0) {
        p.ws[2 * vo] = alpha;
        p.ws[2 * vo + 1] = fmaf(w.Di, alpha, ex);
      }
    }
    if (kDo) {
#pragma unroll 1
      for (int c0 = c_lo; c0 < c_hi; c0 += 16) {
        float y[16], o[16];
        tmem_ld16(e.tm + A_Y + c0, y);
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
};

// ===========================================================================
// pass 2
// ===========================================================================
template <int D_>
struct Pass2 {
  using Params = P2Params;
  static constexpr int D = D_, DC = D / 64;
  static constexpr int NRES = 4;                  // K, V, UK, UV
  static constexpr int RES = NRES * DC * kChunk;
  static constexpr int ACH = 3 * kBlk;            // [Q | UQ | dO] per chunk
  static constexpr int VEC_OFF = DC * ACH;        // L (32), D (32), (alpha, E) (64) floats
  static constexpr int SA = DC * ACH + 1024, SA_TX = DC * ACH + 512;
  static constexpr int SB = 0, SB_TX = 0;
  static constexpr int NSA = D == 128 ? 3 : 4, NSB = 0;
  static constexpr bool VEC = true, ROW_SUMS = false, TS = true;
  static constexpr int OPS = 0;
  static constexpr int ACC = 2 * D;               // gK, gV accumulators
  static constexpr int SCOLS = 128;               // [S|B|dP|C]
  static constexpr int NBUF = D == 128 ? 1 : 2;
  static constexpr int OP_HALF = 48;              // dS, Gs, Gdp (16 columns each)
  static constexpr int OP_COL = ACC + NBUF * SCOLS;
  static constexpr int SMEM = RES + NSA * SA;
  static_assert(OP_COL + 2 * OP_HALF <= 512, "TMEM budget");
  static_assert(SMEM + 1024 <= 232448, "shared memory budget (1 KB static)");
  static constexpr int A_K = 0, A_V = D;

  __device__ static void load_res(const Params& p, uint8_t* res, uint64_t* bar, int col0, int head) {
    const CUtensorMap* m[4] = {&p.mK, &p.mV, &p.mUK, &p.mUV};
    for (int s = 0; s < NRES; ++s)
      for (int kc = 0; kc < DC; ++kc) tma_load_3d(res + (s * DC + kc) * kChunk, m[s], bar, kc * 64, col0, head);
  }
  __device__ static void load_a(const Params& p, uint8_t* st, uint64_t* bar, int t, int head) {
    for (int kc = 0; kc < DC; ++kc) {
      uint8_t* c = st + kc * ACH;
      tma_load_3d(c, &p.mQ, bar, kc * 64, t * kT, head);
      tma_load_3d(c + kBlk, &p.mUQ, bar, kc * 64, t * kT, head);
      tma_load_3d(c + 2 * kBlk, &p.mdO, bar, kc * 64, t * kT, head);
    }
    const size_t v = (size_t)head * p.N + (size_t)t * kT;
    uint8_t* vec = st + VEC_OFF;
    bulk_load(vec, p.L + v, 128, bar);
    bulk_load(vec + 128, p.D + v, 128, bar);
    bulk_load(vec + 256, p.ws + 2 * v, 256, bar);
  }
  __device__ static void load_b(const Params&, uint8_t*, uint64_t*, int, int) {}

  __device__ static void score_mmas(uint32_t sc, uint32_t res, uint32_t sa, uint32_t) {
    const uint32_t i64 = idesc_bf16(kM, 64, false, false), i32 = idesc_bf16(kM, 32, false, false);
#pragma unroll
    for (int k = 0; k < D / 16; ++k)  // [S^T | K UQ^T] = K [Q; UQ]^T
      mma_ss_w(sc, res_lo(res, 0, DC, k), kmaj_lo(sa, ACH, 0, k), i64, k > 0);
#pragma unroll
    for (int k = 0; k < D / 16; ++k)  // B^T += UK Q^T
      mma_ss_w(sc + 32, res_lo(res, 2, DC, k), kmaj_lo(sa, ACH, 0, k), i32, 1);
#pragma unroll
    for (int k = 0; k < D / 16; ++k) {
      mma_ss_w(sc + 64, res_lo(res, 1, DC, k), kmaj_lo(sa, ACH, 2, k), i32, k > 0);  // dP^T = V dO^T
      mma_ss_w(sc + 96, res_lo(res, 3, DC, k), kmaj_lo(sa, ACH, 2, k), i32, k > 0);  // C^T = UV dO^T
    }
  }

  __device__ static void accum_mmas(uint32_t tb, uint32_t ops, uint32_t sa, uint32_t h, bool first) {
    const uint32_t amn = desc_lo(sa, ACH);
    const uint32_t id = idesc_bf16(kM, D, false, true);
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
      const uint32_t acc0 = (first && kk == 0) ? 0u : 1u;
      const uint32_t a = ops + h * OP_HALF + kk * 8;
      mma_ts_w(tb + A_K, a, mn_lo(amn, 1, kk), id, acc0);        // dS^T UQ
      mma_ts_w(tb + A_K, a + 16, mn_lo(amn, 0, kk), id, 1);      // Gs^T Q
      mma_ts_w(tb + A_V, a + 32, mn_lo(amn, 2, kk), id, acc0);   // Gdp^T dO
    }
  }

  struct Row {};
  __device__ static void ew_init(Row&, const Params&, int, int, int) {}

  __device__ static bool ew_tile(Row&, const Params& p, const TileArgs& a, const TileSync& s, int) {
    const float sc = p.tau * kLog2e;
    const float* vL = a.vec;
    const float* vD = a.vec + 32;
    const float2* vAE = reinterpret_cast<const float2*>(a.vec + 64);
    uint32_t wdS[16], wGs[16], wGd[16];
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      float S[16], B[16], dP[16], C[16];
      tmem_ld16x4(a.sc + q * 16, a.sc + 32 + q * 16, a.sc + 64 + q * 16, a.sc + 96 + q * 16, S, B, dP, C);
      if (q == 1) s.release_scores();
#pragma unroll
      for (int c = 0; c < 16; c += 2) {
        float dsv[2], gsv[2], gdv[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int ii = q * 16 + c + e;   // query column within the tile
          const float Dq = vD[ii];
          const float2 ae = vAE[ii];
          const float pe = ex2(fmaf(S[c + e], sc, -vL[ii] * kLog2e));
          const float te = dP[c + e] - Dq;
          const float bp = fmaf(p.tau, B[c + e], -ae.x);
          dsv[e] = pe * te;
          gsv[e] = pe * (fmaf(bp, te, C[c + e]) + fmaf(ae.x, Dq, -ae.y));
          gdv[e] = pe * bp;
        }
        const int k = q * 8 + c / 2;
        wdS[k] = pack_bf16x2(dsv[0], dsv[1]);
        wGs[k] = pack_bf16x2(gsv[0], gsv[1]);
        wGd[k] = pack_bf16x2(gdv[0], gdv[1]);
      }
    }
    if (!s.acquire_ops()) return false;
    tmem_st16_nowait(a.ops, wdS);
    tmem_st16_nowait(a.ops + 16, wGs);
    tmem_st16_nowait(a.ops + 32, wGd);
    s.publish_ops();
    return true;
  }

  __device__ static void epilogue(Row&, const Params& p, const EpiArgs& e) {
    const size_t ro = ((size_t)e.head * p.N + e.blk0 + e.r) * D;
    const int c_lo = e.g * (D / 2), c_hi = c_lo + D / 2;
#pragma unroll 1
    for (int c0 = c_lo; c0 < c_hi; c0 += 16) {
      float ak[16], av[16];
      tmem_ld16x2(e.tm + A_K + c0, e.tm + A_V + c0, ak, av);
#pragma unroll
      for (int j = 0; j < 16; ++j) ak[j] *= p.tau;
      store16(p.gK + ro + c0, ak);
      store16(p.gV + ro + c0, av);
    }
  }
};

// ===========================================================================
// host side
// ===========================================================================
template <class Op>
cudaError_t launch(const char* name, const typename Op::Params& prm, dim3 grid, cudaStream_t s) {
  auto kernel = tile_kernel<Op>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, Op::SMEM);
  if (e != cudaSuccess) return e;
  prof_begin(s, name);
  kernel<<<grid, kThreads, Op::SMEM, s>>>(prm);
  prof_end(s);
  return cudaGetLastError();
}

template <int D>
cudaError_t bob_d(const BobArgs& a, const DevCtx& c, cudaStream_t s) {
  P1Params p1;
  const int BH = a.BH, N = a.N;
  bool ok = make_bf16_map(&p1.mQ, a.Q, BH, N, D, kM) && make_bf16_map(&p1.mdO, a.dO, BH, N, D, kM) &&
            make_bf16_map(&p1.mUQ, a.UQ, BH, N, D, kM) && make_bf16_map(&p1.mK, a.K, BH, N, D, kT) &&
            make_bf16_map(&p1.mUK, a.UK, BH, N, D, kT) && make_bf16_map(&p1.mV, a.V, BH, N, D, kT) &&
            make_bf16_map(&p1.mUV, a.UV, BH, N, D, kT);
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
  p1.stall = c.stall;
  const dim3 grid(N / kM, BH);
  cudaError_t e;
  if constexpr (D == 64) {
    e = launch<Pass1<D, kBoth>>("bob_pass1", p1, grid, s);
  } else {
    e = launch<Pass1<D, kQSide>>("bob_pass1_qside", p1, grid, s);
    if (e == cudaSuccess) e = launch<Pass1<D, kDoSide>>("bob_pass1_doside", p1, grid, s);
  }
  if (e != cudaSuccess) return e;
  P2Params p2;
  ok = make_bf16_map(&p2.mK, a.K, BH, N, D, kM) && make_bf16_map(&p2.mV, a.V, BH, N, D, kM) &&
       make_bf16_map(&p2.mUK, a.UK, BH, N, D, kM) && make_bf16_map(&p2.mUV, a.UV, BH, N, D, kM) &&
       make_bf16_map(&p2.mQ, a.Q, BH, N, D, kT) && make_bf16_map(&p2.mUQ, a.UQ, BH, N, D, kT) &&
       make_bf16_map(&p2.mdO, a.dO, BH, N, D, kT);
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
  p2.stall = c.stall;
  return launch<Pass2<D>>("bob_pass2", p2, grid, s);
}

}  // namespace

cudaError_t tc_bob(const BobArgs& a, const DevCtx& c, cudaStream_t s) {
  return a.d == 64 ? bob_d<64>(a, c, s) : bob_d<128>(a, c, s);
}

}  // namespace fbob
