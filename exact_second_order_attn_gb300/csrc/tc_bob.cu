// Tensor-core (tcgen05 + TMEM + TMA) kernels of the two-pass BoB for bf16
// inputs, d in {64, 128}, any N, built on the tile skeleton of
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
// The identity the pass-1 split rests on: with the row totals alpha and EX
// known, EX U2 + alpha W = sum_j (EX P + alpha dS) K_j, so
//   gQ = tau (U1 - Z),  Z = sum_j G K_j,  G = EX P + alpha dS.
//
// The score MMAs read their resident operands (Q, UQ and, at d = 64, dO in
// pass 1; K, UK and, at d = 64, V, UV in pass 2) from TMEM where it has room,
// so mostly only the streamed 32-row tile is read from shared memory.  TMEM
// (512 columns x 128 lanes fp32) holds one kernel's accumulators, so pass 1
// runs as two kernels over the same 128-row blocks, in stream order:
//   U1-and-Y kernel  U1, Y (2d) | [S|B|dP|C] x NBUF | Q, UQ (, dO)
//              (the dS, X, P, PB operands in shared memory; at d = 128 one
//              score buffer, dO in shared memory)
//              writes U1 into gQ, (alpha, E) into the workspace and
//              gdO = Y - alpha O;
//   Z kernel   Z (d) | [S|dP] x 2 | G halves | Q, dO
//              reads (alpha, E) and U1, writes gQ = tau (U1 - Z).
// Pass 2: gK, gV (2d) | [S|B|dP|C] | then, at d = 64, the (dS, Gs, Gdp)
// halves and K, UK, V, UV; at d = 128, K and UK (V, UV stay in shared memory
// and the three operands go to shared memory).
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

struct P1Params {
  CUtensorMap mK, mUK, mV, mUV;              // streamed, box {64, 32} (U1-and-Y sweep)
  CUtensorMap mK64, mV64;                    // streamed, box {64, 64} (Z sweep)
  CUtensorMap mUK64;                         // streamed, box {64, 64} (four-pass alpha sweep only)
  CUtensorMap mdO_res, mUQ_res;              // resident, box {64, 128} (U1-and-Y sweeps, in shared memory)
  const __nv_bfloat16 *Q, *UQ, *dO;          // resident (copied into TMEM)
  const float *L, *D, *O;
  float *gQ, *gdO, *ws;
  int N;
  int dv;                                    // head size in global memory (<= D; see tc_tile.cuh)
  float tau;
  int causal;
  unsigned int* err;
  unsigned long long wait_ns;
  int stall;
};

struct P2Params {
  CUtensorMap mV, mUV;                       // resident in shared memory at d = 128, box {64, 128}
  CUtensorMap mQ, mUQ, mdO;                  // streamed, box {64, 32}
  const __nv_bfloat16 *K, *UK, *V, *UV;      // resident (copied into TMEM)
  const float *L, *D, *ws;
  float *gK, *gV;
  int N;
  int dv;                                    // head size in global memory (<= D; see tc_tile.cuh)
  float tau;
  int causal;
  unsigned int* err;
  unsigned long long wait_ns;
  int stall;
};

// ===========================================================================
// pass 1
// ===========================================================================
__device__ __forceinline__ void load_tile2(const CUtensorMap* m0, const CUtensorMap* m1, uint8_t* st, int dc, int ch,
                                           int blk, uint64_t* bar, int row, int head) {
  for (int kc = 0; kc < dc; ++kc) {
    tma_load_3d(st + kc * ch, m0, bar, kc * 64, row, head);
    if (m1) tma_load_3d(st + kc * ch + blk, m1, bar, kc * 64, row, head);
  }
}

// U1-and-Y sweep (32 keys per tile): U1 += dS UK + X K, Y += P UV + PB V,
// alpha, EX; writes U1 (into gQ, finished by the Z sweep), (alpha, E) and
// gdO = Y - alpha O.  Ring A = [K UK V UV] (all read by the accumulator
// MMAs).  The four operands dS, X, P, PB go to shared memory.  At d = 128,
// Q and UQ sit in TMEM and dO in shared memory, with one score buffer whose
// columns the two warpgroups split; at d = 64 Q, UQ, dO sit in TMEM with two
// score buffers.
//
// DIRECT (the four-pass ablation's row-output sweep): alpha and E are known
// from the two reduction sweeps before it, so the second operand is the full
// cotangent of S, Sbar = P (Pbar - En) with Pbar = tau B (dP - D) + C - alpha dP
// and En = sum_j P Pbar, and the kernel writes gQ = tau (dS UK + Sbar K)
// summed over all keys - no row totals, no correction sweep.
//
// The fourth operand P o B enters gdO = Y - alpha O, which on a peaked
// softmax row nearly cancels (P o B ~ alpha P on the dominant key); one bf16
// rounding of it would show in gdO at a few 1e-3 of its maximum.  So the
// two-pass sweeps carry it as two bf16 terms, PB = PB_hi + PB_lo (a fifth
// operand tile and one more MMA per 16 keys).  DIRECT knows alpha and instead
// writes the centred P o (B - alpha) (gdO = Y, nothing cancels).
//
// FULL (d = 64: the whole of pass 1 in one sweep): TMEM also holds the two
// remaining alpha-free accumulators U2 += P K and W += dS K, so the row end
// applies the affine correction gQ = tau (U1 - EX U2 - alpha W) directly and
// no Z sweep follows.  The five operands go to TMEM as well (the accumulator
// MMAs read only their B tiles from shared memory, and the elementwise warps
// store no operand tiles there): TMEM = four accumulators of 64 columns, one
// score buffer of 128, one operand buffer of 5 x 16 (shared by consecutive
// tiles) and Q (32) = 496 of 512.  UQ and dO stay in shared memory as the A
// operands of their score MMAs.
template <int D_, bool DIRECT = false, bool FULL = false>
struct PassU1Y {
  using Params = P1Params;
  static constexpr int D = D_, DC = D / 64, T = 32;
  static constexpr bool kWide = D == 128;
  static_assert(!FULL || (D == 64 && !DIRECT), "the one-sweep pass 1 fits TMEM at d = 64");
  static constexpr bool ROWS = true, SPLIT = kWide || FULL;
  static constexpr int TRES = FULL ? 1 : kWide ? 2 : 3;                      // Q (, UQ (, dO))
  static constexpr int RES = FULL ? 2 * DC * kChunk : kWide ? DC * kChunk : 0;  // (UQ,) dO in shared memory
  static constexpr int ACH = 4 * kBlk;                  // [K | UK | V | UV] per 64-column chunk
  static constexpr int SA = DC * ACH, SA_TX = SA, SB = 0, SB_TX = 0;
  static constexpr bool kSplitPB = !DIRECT;             // PB as bf16 hi + lo (see above)
  static constexpr int NSA = kWide ? (kSplitPB ? 3 : 4) : 8, NSB = 0;
  static constexpr bool VEC = false, ROW_SUMS = !DIRECT, TS = FULL, ONE_OPS = FULL;
  static constexpr int VEC_OFF = 0, NVEC = 0, VEC_SCRATCH = 0;
  // dS, X, P, PB (, PB_lo) tiles; half h = columns 32h..32h+31
  static constexpr int OPS = FULL ? 0 : (kSplitPB ? 5 : 4) * kChunk;
  static constexpr int TOPS = FULL ? 5 * (T / 2) : 0;   // TMEM operand columns (bf16 pairs)
  static constexpr int ACC = (FULL ? 4 : 2) * D;        // U1 | Y (| U2 | W)
  static constexpr int SCOLS = 128, NBUF = (kWide || FULL) ? 1 : 2;   // [S|B|dP|C]
  static constexpr int OP_HALF = 0, OP_COL = ACC + NBUF * SCOLS;
  static constexpr int TRES_COL = OP_COL + TOPS;
  static constexpr int SMEM = RES + NSA * SA + OPS;
  // Ring-A order of the four 32-row blocks: [K | UK | V | UV], or with FULL
  // [V | UV | K | UK], where UV, K and K, UK are neighbours, so that two
  // pairs of accumulator products share their A operand as one N = 2d MMA:
  // P [UV | K] -> [Y | U2] and dS [K | UK] -> [W | U1] (TMEM Y | U2 | W | U1).
  static constexpr int BK = FULL ? 2 : 0, BUK = BK + 1, BV = FULL ? 0 : 2, BUV = BV + 1;
  static constexpr int A_U1 = FULL ? 3 * D : 0, A_Y = FULL ? 0 : D, A_U2 = FULL ? D : 2 * D, A_W = FULL ? 2 * D : 3 * D;
  static_assert(!FULL || (A_U2 == A_Y + D && A_U1 == A_W + D), "paired accumulators are adjacent");
  static constexpr int NC = SPLIT ? T / 2 : T;          // key columns per warpgroup and tile
  static_assert(TRES_COL + TRES * D / 2 <= 512, "TMEM budget");
  static_assert(SMEM + 1024 <= 232448, "shared memory budget (1 KB static)");

  __device__ static const void* tres_src(const Params& p, int s) {
    return s == 0 ? (const void*)p.Q : s == 1 ? (const void*)p.UQ : (const void*)p.dO;
  }
  __device__ static void load_res(const Params& p, uint8_t* res, uint64_t* bar, int row0, int head) {
    if (FULL) {   // UQ then dO
      for (int kc = 0; kc < DC; ++kc) tma_load_3d(res + kc * kChunk, &p.mUQ_res, bar, kc * 64, row0, head);
      res += DC * kChunk;
    }
    for (int kc = 0; kc < DC; ++kc) tma_load_3d(res + kc * kChunk, &p.mdO_res, bar, kc * 64, row0, head);
  }
  __device__ static void load_a(const Params& p, uint8_t* st, uint64_t* bar, int t, int head, bool) {
    load_tile2(&p.mK, &p.mUK, st + BK * kBlk, DC, ACH, kBlk, bar, t * T, head);
    load_tile2(&p.mV, &p.mUV, st + BV * kBlk, DC, ACH, kBlk, bar, t * T, head);
  }
  __device__ static void load_b(const Params&, uint8_t*, uint64_t*, int, int) {}
  __device__ static void fill_vec(const Params&, float*, int, int, int) {}

  __device__ static void score_mmas(uint32_t sc, uint32_t tres, uint32_t res, uint32_t sa, uint32_t) {
    const uint32_t i64 = idesc_bf16(kM, 64, false, false), i32 = idesc_bf16(kM, 32, false, false);
#pragma unroll
    for (int k = 0; k < D / 16; ++k)  // [S | Q UK^T] = Q [K; UK]^T
      mma_ts_w(sc, tres_a(tres, 0, D, k), kmaj(sa, ACH, BK * kBlk, k), i64, k > 0);
#pragma unroll
    for (int k = 0; k < D / 16; ++k) {  // B += UQ K^T
      if (FULL)
        mma_ss_w(sc + 32, res_lo(res, 0, DC, k), kmaj(sa, ACH, BK * kBlk, k), i32, 1);
      else
        mma_ts_w(sc + 32, tres_a(tres, 1, D, k), kmaj(sa, ACH, BK * kBlk, k), i32, 1);
    }
#pragma unroll
    for (int k = 0; k < D / 16; ++k) {  // [dP | C] = dO [V; UV]^T
      if (FULL)
        mma_ss_w(sc + 64, res_lo(res, 1, DC, k), kmaj(sa, ACH, BV * kBlk, k), i64, k > 0);
      else if (kWide)
        mma_ss_w(sc + 64, res_lo(res, 0, DC, k), kmaj(sa, ACH, BV * kBlk, k), i64, k > 0);
      else
        mma_ts_w(sc + 64, tres_a(tres, 2, D, k), kmaj(sa, ACH, BV * kBlk, k), i64, k > 0);
    }
  }
  __device__ static void accum_mmas(uint32_t tb, uint32_t ops, uint32_t sa, uint32_t h, bool first) {
    const uint32_t amn = desc_lo(sa, ACH);
    const uint32_t id = idesc_bf16(kM, D, false, true);
#pragma unroll
    for (int kk = 0; kk < T / 16; ++kk) {
      const uint32_t acc0 = (first && kk == 0) ? 0u : 1u;
      if constexpr (FULL) {
        // N = 2d over two neighbouring 64-column blocks: LBO = one block;
        // operand s of this tile at TMEM columns ops + 16 s, 16 keys per 8 columns
        const uint32_t amn2 = desc_lo(sa, kBlk);
        const uint32_t id2 = idesc_bf16(kM, 2 * D, false, true);
        const uint32_t a = ops + (uint32_t)(kk * 8);
        mma_ts_w(tb + A_Y, a + 2 * 16, mnmaj(amn2, BUV * kBlk, kk), id2, acc0);  // [Y | U2] += P [UV | K]
        mma_ts_w(tb + A_Y, a + 3 * 16, mnmaj(amn, BV * kBlk, kk), id, 1);        // Y += PB V
        mma_ts_w(tb + A_Y, a + 4 * 16, mnmaj(amn, BV * kBlk, kk), id, 1);        // + PB_lo V
        mma_ts_w(tb + A_W, a, mnmaj(amn2, BK * kBlk, kk), id2, acc0);            // [W | U1] += dS [K | UK]
        mma_ts_w(tb + A_U1, a + 16, mnmaj(amn, BK * kBlk, kk), id, 1);           // U1 += X K
      } else {
        mma_ss_w(tb + A_U1, op_lo(ops, 0, h, kk), mnmaj(amn, BUK * kBlk, kk), id, acc0);   // U1 += dS UK
        mma_ss_w(tb + A_U1, op_lo(ops, 1, h, kk), mnmaj(amn, BK * kBlk, kk), id, 1);       // U1 += X K
        mma_ss_w(tb + A_Y, op_lo(ops, 2, h, kk), mnmaj(amn, BUV * kBlk, kk), id, acc0);    // Y += P UV
        mma_ss_w(tb + A_Y, op_lo(ops, 3, h, kk), mnmaj(amn, BV * kBlk, kk), id, 1);        // Y += PB V
        if (kSplitPB) mma_ss_w(tb + A_Y, op_lo(ops, 4, h, kk), mnmaj(amn, BV * kBlk, kk), id, 1);  // + PB_lo V
      }
    }
  }
  struct Row {
    float nL, Di, alpha, ex;   // DIRECT: alpha and ex = En are read, not summed
  };
  __device__ static void ew_init(Row& w, const Params& p, int blk0, int r, int head) {
    const bool ok = blk0 + r < p.N;   // ragged N: rows past the end are never stored
    const size_t vo = (size_t)head * p.N + (ok ? blk0 + r : 0);
    w.nL = ok ? -p.L[vo] * kLog2e : 0.f;
    w.Di = ok ? p.D[vo] : 0.f;
    if (DIRECT && ok) {
      // the workspace holds (alpha, E) with E = sum_j P (C + tau B dP) = En + 2 alpha D
      w.alpha = p.ws[2 * vo];
      w.ex = fmaf(-2.f * w.alpha, w.Di, p.ws[2 * vo + 1]);
    } else {
      w.alpha = 0.f;
      w.ex = 0.f;
    }
  }
  // Operands are written 16 columns at a time.  With two score buffers the
  // operand half is acquired first (as in the dK/dV kernel); with one (split
  // columns, a single 16-column chunk per warpgroup) the scores are released
  // first so the next tile's score MMAs can start.
  static constexpr bool kEarly = NBUF > 1;
  static_assert(kEarly || NC == 16, "late acquire needs a single chunk");
  template <bool MASK>
  __device__ static bool ew_tile(Row& w, const Params& p, const TileArgs& a, const TileSync& s, int r) {
    const float sc = p.tau * kLog2e;
    if (kEarly && !s.acquire_ops()) return false;
#pragma unroll
    for (int q = 0; q < NC / 16; ++q) {
      float S[16], B[16], dP[16], C[16];
      const uint32_t c = a.sc + a.c0 + q * 16;
      tmem_ld16x4(c, c + 32, c + 64, c + 96, S, B, dP, C);
      if (q == NC / 16 - 1) s.release_scores();
      uint32_t wdS[8], wX[8], wP[8], wPB[8], wPBl[8];
#pragma unroll
      for (int j = 0; j < 16; j += 2) {
        float ds[2], x[2], pv[2], pb[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int col = a.c0 + q * 16 + j + e;   // tile column (key)
          const float pe = (!MASK || (col >= a.lo && col <= a.hi)) ? ex2(fmaf(S[j + e], sc, w.nL)) : 0.f;
          const float be = p.tau * B[j + e];
          const float te = dP[j + e] - w.Di;
          pv[e] = pe;
          ds[e] = pe * te;
          if (DIRECT) {
            pb[e] = pe * (be - w.alpha);   // the centred P o (B - alpha)
            // Sbar = P (tau B (dP - D) + C - alpha dP - En)
            x[e] = pe * (fmaf(be, te, C[j + e]) - fmaf(w.alpha, dP[j + e], w.ex));
          } else {
            pb[e] = pe * be;
            w.alpha += pb[e];
            x[e] = pe * fmaf(be, te, C[j + e]);
            w.ex += x[e];
          }
        }
        wdS[j / 2] = pack_bf16x2(ds[0], ds[1]);
        wX[j / 2] = pack_bf16x2(x[0], x[1]);
        wP[j / 2] = pack_bf16x2(pv[0], pv[1]);
        const __nv_bfloat162 hi = __floats2bfloat162_rn(pb[0], pb[1]);
        wPB[j / 2] = *reinterpret_cast<const uint32_t*>(&hi);
        if (kSplitPB) {
          const float2 hf = __bfloat1622float2(hi);
          wPBl[j / 2] = pack_bf16x2(pb[0] - hf.x, pb[1] - hf.y);   // exact differences, rounded once more
        }
      }
      if (!kEarly && !s.acquire_ops()) return false;
      if constexpr (FULL) {   // TMEM operands: 16 keys = 8 columns of each
        const uint32_t o = a.ops + (uint32_t)((a.c0 + q * 16) / 2);
        tmem_st8_nowait(o, wdS);
        tmem_st8_nowait(o + 16, wX);
        tmem_st8_nowait(o + 2 * 16, wP);
        tmem_st8_nowait(o + 3 * 16, wPB);
        tmem_st8_nowait(o + 4 * 16, wPBl);
      } else {
        const int col = 32 * (int)a.h + a.c0 + q * 16;
        write_op_cols<8>(a.ops, (uint32_t)r, col, wdS);
        write_op_cols<8>(a.ops + kChunk, (uint32_t)r, col, wX);
        write_op_cols<8>(a.ops + 2 * kChunk, (uint32_t)r, col, wP);
        write_op_cols<8>(a.ops + 3 * kChunk, (uint32_t)r, col, wPB);
        if (kSplitPB) write_op_cols<8>(a.ops + 4 * kChunk, (uint32_t)r, col, wPBl);
      }
    }
    s.publish_ops();
    return true;
  }
  __device__ static void epilogue(Row& w, const Params& p, const EpiArgs& e) {
    float alpha = w.alpha, ex = w.ex;
    if (!DIRECT && !e.sum_rows(alpha, ex)) return;   // DIRECT: alpha was read whole
    // every lane runs the (warp-collective) TMEM loads; rows >= N touch no memory
    const bool keep = e.blk0 + e.r < p.N;
    const size_t vo = (size_t)e.head * p.N + (keep ? e.blk0 + e.r : 0);
    const size_t ro = vo * p.dv;
    const int c_lo = e.g * (D / 2), c_hi = min(c_lo + D / 2, p.dv);   // columns >= dv hold zeros
#pragma unroll 1
    for (int c0 = c_lo; c0 < c_hi; c0 += 16) {
      float u1[16], y[16], o[16];
      tmem_ld16x2(e.tm + A_U1 + c0, e.tm + A_Y + c0, u1, y);
      if (FULL) {
        float u2[16], w2[16];
        tmem_ld16x2(e.tm + A_U2 + c0, e.tm + A_W + c0, u2, w2);
#pragma unroll
        for (int j = 0; j < 16; ++j)   // gQ = tau (U1 - EX U2 - alpha W)
          u1[j] = p.tau * (u1[j] - fmaf(ex, u2[j], alpha * w2[j]));
      }
      if (!keep) continue;
      if (DIRECT) {
#pragma unroll
        for (int j = 0; j < 16; ++j) u1[j] *= p.tau;   // gQ = tau (dS UK + Sbar K)
      }
      store16(p.gQ + ro + c0, u1);   // two-pass at d = 128: U1, finished by the Z sweep
      if (DIRECT) {
        store16(p.gdO + ro + c0, y);   // gdO = P UV + P o (B - alpha) V
        continue;
      }
      const float4* src = reinterpret_cast<const float4*>(p.O + ro + c0);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float4 v = src[q];
        o[4 * q] = fmaf(-alpha, v.x, y[4 * q]);          // gdO = Y - alpha O
        o[4 * q + 1] = fmaf(-alpha, v.y, y[4 * q + 1]);
        o[4 * q + 2] = fmaf(-alpha, v.z, y[4 * q + 2]);
        o[4 * q + 3] = fmaf(-alpha, v.w, y[4 * q + 3]);
      }
      store16(p.gdO + ro + c0, o);
    }
    if (!DIRECT && keep && e.g == 0) {
      p.ws[2 * vo] = alpha;
      p.ws[2 * vo + 1] = fmaf(w.Di, alpha, ex);
    }
  }
};

// Z sweep (64 keys per tile): Z += G K, G = EX P + alpha dS, gQ = tau (U1 - Z).
// Ring A = K, ring B = V.  G goes to TMEM at d = 64, to shared memory at d = 128.
template <int D_>
struct PassZ {
  using Params = P1Params;
  static constexpr bool SPLIT = false, ROWS = true;
  static constexpr int D = D_, DC = D / 64, T = 64, BLK = T * 128;
  static constexpr int RES = 0, TRES = 2;   // Q, dO
  static constexpr int ACH = BLK, BCH = BLK;
  static constexpr int SA = DC * ACH, SB = DC * BCH, SA_TX = SA, SB_TX = SB;
  static constexpr int NSA = D == 128 ? 5 : 8, NSB = NSA;
  static constexpr bool VEC = false, ROW_SUMS = false, TS = D == 64;
  static constexpr int VEC_OFF = 0, NVEC = 0, VEC_SCRATCH = 0;
  static constexpr int OPS = TS ? 0 : 2 * kChunk;
  static constexpr int ACC = D, SCOLS = 2 * T, NBUF = 2;   // [S | dP]
  static constexpr int OP_HALF = T / 2, OP_COL = ACC + NBUF * SCOLS;
  static constexpr int TRES_COL = OP_COL + (TS ? 2 * OP_HALF : 0);
  static constexpr int SMEM = NSA * SA + NSB * SB + OPS;
  static_assert(TRES_COL + TRES * D / 2 <= 512, "TMEM budget");
  static_assert(SMEM + 1024 <= 232448, "shared memory budget (1 KB static)");

  __device__ static const void* tres_src(const Params& p, int s) { return s == 0 ? (const void*)p.Q : (const void*)p.dO; }
  __device__ static void load_res(const Params&, uint8_t*, uint64_t*, int, int) {}
  __device__ static void load_a(const Params& p, uint8_t* st, uint64_t* bar, int t, int head, bool) {
    load_tile2(&p.mK64, nullptr, st, DC, ACH, BLK, bar, t * T, head);
  }
  __device__ static void fill_vec(const Params&, float*, int, int, int) {}
  __device__ static void load_b(const Params& p, uint8_t* st, uint64_t* bar, int t, int head) {
    load_tile2(&p.mV64, nullptr, st, DC, BCH, BLK, bar, t * T, head);
  }
  __device__ static void score_mmas(uint32_t sc, uint32_t tres, uint32_t, uint32_t sa, uint32_t sb) {
    const uint32_t i64 = idesc_bf16(kM, T, false, false);
#pragma unroll
    for (int k = 0; k < D / 16; ++k) {
      mma_ts_w(sc, tres_a(tres, 0, D, k), kmaj(sa, ACH, 0, k), i64, k > 0);      // S = Q K^T
      mma_ts_w(sc + T, tres_a(tres, 1, D, k), kmaj(sb, BCH, 0, k), i64, k > 0);  // dP = dO V^T
    }
  }
  __device__ static void accum_mmas(uint32_t tb, uint32_t ops, uint32_t sa, uint32_t h, bool first) {
    const uint32_t amn = desc_lo(sa, ACH);
    const uint32_t id = idesc_bf16(kM, D, false, true);
#pragma unroll
    for (int kk = 0; kk < T / 16; ++kk) {  // Z += G K
      const uint32_t acc = (first && kk == 0) ? 0u : 1u;
      if (TS)
        mma_ts_w(tb, ops + h * OP_HALF + kk * 8, mnmaj(amn, 0, kk), id, acc);
      else
        mma_ss_w(tb, op64_lo(ops, 0, h, kk), mnmaj(amn, 0, kk), id, acc);
    }
  }
  struct Row {
    float nL, Di, alpha, ex;
  };
  __device__ static void ew_init(Row& w, const Params& p, int blk0, int r, int head) {
    const bool ok = blk0 + r < p.N;   // ragged N: rows past the end are never stored
    const size_t vo = (size_t)head * p.N + (ok ? blk0 + r : 0);
    w.nL = ok ? -p.L[vo] * kLog2e : 0.f;
    w.Di = ok ? p.D[vo] : 0.f;
    w.alpha = ok ? p.ws[2 * vo] : 0.f;                            // row totals of the U1-and-Y sweep
    w.ex = ok ? fmaf(-w.Di, w.alpha, p.ws[2 * vo + 1]) : 0.f;     // EX = E - D alpha
  }
  template <bool MASK>
  __device__ static bool ew_tile(Row& w, const Params& p, const TileArgs& a, const TileSync& s, int r) {
    const float sc = p.tau * kLog2e;
    uint32_t wg[T / 2];
#pragma unroll
    for (int q = 0; q < T / 16; ++q) {
      float S[16], dP[16];
      tmem_ld16x2(a.sc + q * 16, a.sc + T + q * 16, S, dP);
      if (q == T / 16 - 1) s.release_scores();
#pragma unroll
      for (int j = 0; j < 16; j += 2) {
        float g[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int col = q * 16 + j + e;   // tile column (key)
          const float pe = (!MASK || (col >= a.lo && col <= a.hi)) ? ex2(fmaf(S[j + e], sc, w.nL)) : 0.f;
          g[e] = pe * fmaf(w.alpha, dP[j + e] - w.Di, w.ex);   // EX P + alpha dS
        }
        wg[q * 8 + j / 2] = pack_bf16x2(g[0], g[1]);
      }
    }
    if (!s.acquire_ops()) return false;
    if (TS) {
      tmem_st16_nowait(a.ops, wg);
      tmem_st16_nowait(a.ops + 16, wg + 16);
    } else {
      write_op64(a.ops + a.h * kChunk, (uint32_t)r, wg);
    }
    s.publish_ops();
    return true;
  }
  __device__ static void epilogue(Row&, const Params& p, const EpiArgs& e) {
    // every lane runs the (warp-collective) TMEM loads; rows >= N touch no memory
    const bool keep = e.blk0 + e.r < p.N;
    const size_t ro = ((size_t)e.head * p.N + (keep ? e.blk0 + e.r : 0)) * p.dv;
    const int c_lo = e.g * (D / 2), c_hi = min(c_lo + D / 2, p.dv);   // columns >= dv hold zeros
#pragma unroll 1
    for (int c0 = c_lo; c0 < c_hi; c0 += 16) {
      float z[16], o[16];
      tmem_ld16(e.tm + c0, z);
      if (!keep) continue;
      const float4* u1 = reinterpret_cast<const float4*>(p.gQ + ro + c0);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float4 v = u1[q];
        o[4 * q] = p.tau * (v.x - z[4 * q]);
        o[4 * q + 1] = p.tau * (v.y - z[4 * q + 1]);
        o[4 * q + 2] = p.tau * (v.z - z[4 * q + 2]);
        o[4 * q + 3] = p.tau * (v.w - z[4 * q + 3]);
      }
      store16(p.gQ + ro + c0, o);
    }
  }
};

// ===========================================================================
// four-pass ablation: the reduction sweeps
// ===========================================================================
// Without the affine structure, reverse mode needs the row scalars in order:
// alpha first (the cotangent of D), then E, whose natural form uses alpha,
// then the row outputs with both known (PassU1Y<D, true>), then the column
// pass.  These two kernels are the first two sweeps; they only reduce, so
// they issue score MMAs alone (the accumulator warp just passes the
// operand barriers through).

// alpha sweep (64 keys per tile): alpha = sum_j P tau B.  Ring A = [K | UK];
// Q, UQ in TMEM.
template <int D_>
struct PassAlpha {
  using Params = P1Params;
  static constexpr bool SPLIT = false, ROWS = true;
  static constexpr int D = D_, DC = D / 64, T = 64, BLK = T * 128;
  static constexpr int RES = 0, TRES = 2;   // Q, UQ
  static constexpr int ACH = 2 * BLK;       // [K | UK] per 64-column chunk
  static constexpr int SA = DC * ACH, SA_TX = SA, SB = 0, SB_TX = 0;
  static constexpr int NSA = D == 128 ? 6 : 8, NSB = 0;
  static constexpr bool VEC = false, ROW_SUMS = true, TS = false;
  static constexpr int VEC_OFF = 0, NVEC = 0, VEC_SCRATCH = 0, OPS = 0;
  static constexpr int ACC = 0, SCOLS = 2 * T, NBUF = 2;   // [S | B]
  static constexpr int OP_HALF = 0, OP_COL = ACC + NBUF * SCOLS, TRES_COL = OP_COL;
  static constexpr int SMEM = NSA * SA;
  static_assert(TRES_COL + TRES * D / 2 <= 512, "TMEM budget");
  static_assert(SMEM + 1024 <= 232448, "shared memory budget (1 KB static)");

  __device__ static const void* tres_src(const Params& p, int s) { return s == 0 ? (const void*)p.Q : (const void*)p.UQ; }
  __device__ static void load_res(const Params&, uint8_t*, uint64_t*, int, int) {}
  __device__ static void load_a(const Params& p, uint8_t* st, uint64_t* bar, int t, int head, bool) {
    load_tile2(&p.mK64, &p.mUK64, st, DC, ACH, BLK, bar, t * T, head);
  }
  __device__ static void load_b(const Params&, uint8_t*, uint64_t*, int, int) {}
  __device__ static void fill_vec(const Params&, float*, int, int, int) {}
  __device__ static void score_mmas(uint32_t sc, uint32_t tres, uint32_t, uint32_t sa, uint32_t) {
    const uint32_t i128 = idesc_bf16(kM, 2 * T, false, false), i64 = idesc_bf16(kM, T, false, false);
#pragma unroll
    for (int k = 0; k < D / 16; ++k)  // [S | Q UK^T] = Q [K; UK]^T
      mma_ts_w(sc, tres_a(tres, 0, D, k), kmaj(sa, ACH, 0, k), i128, k > 0);
#pragma unroll
    for (int k = 0; k < D / 16; ++k)  // B += UQ K^T
      mma_ts_w(sc + T, tres_a(tres, 1, D, k), kmaj(sa, ACH, 0, k), i64, 1);
  }
  __device__ static void accum_mmas(uint32_t, uint32_t, uint32_t, uint32_t, bool) {}
  struct Row {
    float nL, alpha;
  };
  __device__ static void ew_init(Row& w, const Params& p, int blk0, int r, int head) {
    w.nL = blk0 + r < p.N ? -p.L[(size_t)head * p.N + blk0 + r] * kLog2e : 0.f;
    w.alpha = 0.f;
  }
  template <bool MASK>
  __device__ static bool ew_tile(Row& w, const Params& p, const TileArgs& a, const TileSync& s, int) {
    const float sc = p.tau * kLog2e;
#pragma unroll
    for (int q = 0; q < T / 16; ++q) {
      float S[16], B[16];
      tmem_ld16x2(a.sc + q * 16, a.sc + T + q * 16, S, B);
      if (q == T / 16 - 1) s.release_scores();
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int col = q * 16 + j;   // tile column (key)
        const float pe = (!MASK || (col >= a.lo && col <= a.hi)) ? ex2(fmaf(S[j], sc, w.nL)) : 0.f;
        w.alpha = fmaf(pe, p.tau * B[j], w.alpha);
      }
    }
    // no operands: pass the operand barriers through to the accumulator warp
    if (!s.acquire_ops()) return false;
    s.publish_ops();
    return true;
  }
  __device__ static void epilogue(Row& w, const Params& p, const EpiArgs& e) {
    float alpha = w.alpha, unused = 0.f;
    if (!e.sum_rows(alpha, unused)) return;
    if (e.g == 0 && e.blk0 + e.r < p.N) p.ws[2 * ((size_t)e.head * p.N + e.blk0 + e.r)] = alpha;
  }
};

// E sweep (32 keys per tile): En = sum_j P Pbar, Pbar = tau B (dP - D) + C -
// alpha dP with alpha from the alpha sweep; stores E = En + 2 alpha D, the
// form the column pass reads.  Same streamed tile, residents and score MMAs
// as the U1-and-Y sweep, two score buffers, no accumulators.
template <int D_>
struct PassE {
  using Params = P1Params;
  using Scores = PassU1Y<D_>;
  static constexpr bool SPLIT = false, ROWS = true;
  static constexpr int D = D_, DC = D / 64, T = 32;
  static constexpr int TRES = Scores::TRES, RES = Scores::RES, ACH = Scores::ACH;
  static constexpr int SA = DC * ACH, SA_TX = SA, SB = 0, SB_TX = 0;
  static constexpr int NSA = D == 128 ? 5 : 8, NSB = 0;
  static constexpr bool VEC = false, ROW_SUMS = true, TS = false;
  static constexpr int VEC_OFF = 0, NVEC = 0, VEC_SCRATCH = 0, OPS = 0;
  static constexpr int ACC = 0, SCOLS = 128, NBUF = 2;   // [S|B|dP|C]
  static constexpr int OP_HALF = 0, OP_COL = ACC + NBUF * SCOLS, TRES_COL = OP_COL;
  static constexpr int SMEM = RES + NSA * SA;
  static_assert(TRES_COL + TRES * D / 2 <= 512, "TMEM budget");
  static_assert(SMEM + 1024 <= 232448, "shared memory budget (1 KB static)");

  __device__ static const void* tres_src(const Params& p, int s) { return Scores::tres_src(p, s); }
  __device__ static void load_res(const Params& p, uint8_t* res, uint64_t* bar, int row0, int head) {
    Scores::load_res(p, res, bar, row0, head);
  }
  __device__ static void load_a(const Params& p, uint8_t* st, uint64_t* bar, int t, int head, bool w) {
    Scores::load_a(p, st, bar, t, head, w);
  }
  __device__ static void load_b(const Params&, uint8_t*, uint64_t*, int, int) {}
  __device__ static void fill_vec(const Params&, float*, int, int, int) {}
  __device__ static void score_mmas(uint32_t sc, uint32_t tres, uint32_t res, uint32_t sa, uint32_t sb) {
    Scores::score_mmas(sc, tres, res, sa, sb);
  }
  __device__ static void accum_mmas(uint32_t, uint32_t, uint32_t, uint32_t, bool) {}
  struct Row {
    float nL, Di, alpha, en;
  };
  __device__ static void ew_init(Row& w, const Params& p, int blk0, int r, int head) {
    const bool ok = blk0 + r < p.N;
    const size_t vo = (size_t)head * p.N + (ok ? blk0 + r : 0);
    w.nL = ok ? -p.L[vo] * kLog2e : 0.f;
    w.Di = ok ? p.D[vo] : 0.f;
    w.alpha = ok ? p.ws[2 * vo] : 0.f;
    w.en = 0.f;
  }
  template <bool MASK>
  __device__ static bool ew_tile(Row& w, const Params& p, const TileArgs& a, const TileSync& s, int) {
    const float sc = p.tau * kLog2e;
#pragma unroll
    for (int q = 0; q < T / 16; ++q) {
      float S[16], B[16], dP[16], C[16];
      const uint32_t c = a.sc + q * 16;
      tmem_ld16x4(c, c + 32, c + 64, c + 96, S, B, dP, C);
      if (q == T / 16 - 1) s.release_scores();
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int col = q * 16 + j;   // tile column (key)
        const float pe = (!MASK || (col >= a.lo && col <= a.hi)) ? ex2(fmaf(S[j], sc, w.nL)) : 0.f;
        const float pbar = fmaf(p.tau * B[j], dP[j] - w.Di, C[j]) - w.alpha * dP[j];
        w.en = fmaf(pe, pbar, w.en);
      }
    }
    if (!s.acquire_ops()) return false;
    s.publish_ops();
    return true;
  }
  __device__ static void epilogue(Row& w, const Params& p, const EpiArgs& e) {
    float en = w.en, unused = 0.f;
    if (!e.sum_rows(en, unused)) return;
    if (e.g == 0 && e.blk0 + e.r < p.N)
      p.ws[2 * ((size_t)e.head * p.N + e.blk0 + e.r) + 1] = fmaf(2.f * w.alpha, w.Di, en);
  }
};

// ===========================================================================
// pass 2
// ===========================================================================
template <int D_>
struct Pass2 {
  using Params = P2Params;
  static constexpr bool ROWS = false;
  static constexpr int D = D_, DC = D / 64, T = kT;
  static constexpr bool kAllTmem = D == 64;        // V, UV also in TMEM; operands in TMEM
  static constexpr int TRES = kAllTmem ? 4 : 2;    // K, UK (, V, UV)
  static constexpr int RES = kAllTmem ? 0 : 2 * DC * kChunk;   // V, UV in shared memory
  static constexpr int ACH = 3 * kBlk;            // [Q | UQ | dO] per chunk
  static constexpr int VEC_OFF = DC * ACH;        // L (T), D (T), (alpha, E) (2T) floats
  static constexpr int SA = DC * ACH + 1024, SA_TX = DC * ACH + 512;
  static constexpr int SB = 0, SB_TX = 0;
  static constexpr int NSA = kAllTmem ? 8 : 4, NSB = 0;
  static constexpr bool VEC = true, ROW_SUMS = false, TS = kAllTmem;
  static constexpr int OPS = kAllTmem ? 0 : 3 * kChunk;   // dS, Gs, Gdp tiles [128][64]
  static constexpr int ACC = 2 * D;               // gK, gV accumulators
  static constexpr int SCOLS = 128;               // [S|B|dP|C]
  static constexpr int NBUF = 1;
  static constexpr int OP_HALF = 48;              // TMEM operands: dS, Gs, Gdp (16 columns each)
  static constexpr int OP_COL = ACC + NBUF * SCOLS;
  static constexpr int TRES_COL = OP_COL + (kAllTmem ? 2 * OP_HALF : 0);
  static constexpr int NVEC = 4;                   // L, D, (alpha, E) per query
  static constexpr int VEC_SCRATCH = RES + NSA * SA + OPS;   // 2 warpgroups x 2 buffers x NVEC x T floats
  static constexpr int QREC = VEC_SCRATCH + 4 * NVEC * T * 4; // per elementwise warp: T query records
  static constexpr int SMEM = QREC + kEwWarps * T * 16;
  static_assert(TRES_COL + TRES * D / 2 <= 512, "TMEM budget");
  static_assert(SMEM + 1024 <= 232448, "shared memory budget (1 KB static)");
  static constexpr int A_K = 0, A_V = D;

  __device__ static const void* tres_src(const Params& p, int s) {
    return s == 0 ? (const void*)p.K : s == 1 ? (const void*)p.UK : s == 2 ? (const void*)p.V : (const void*)p.UV;
  }
  __device__ static void load_res(const Params& p, uint8_t* res, uint64_t* bar, int col0, int head) {
    const CUtensorMap* m[2] = {&p.mV, &p.mUV};
    for (int s = 0; s < 2; ++s)
      for (int kc = 0; kc < DC; ++kc) tma_load_3d(res + (s * DC + kc) * kChunk, m[s], bar, kc * 64, col0, head);
  }
  __device__ static void load_a(const Params& p, uint8_t* st, uint64_t* bar, int t, int head, bool whole) {
    for (int kc = 0; kc < DC; ++kc) {
      uint8_t* c = st + kc * ACH;
      tma_load_3d(c, &p.mQ, bar, kc * 64, t * kT, head);
      tma_load_3d(c + kBlk, &p.mUQ, bar, kc * 64, t * kT, head);
      tma_load_3d(c + 2 * kBlk, &p.mdO, bar, kc * 64, t * kT, head);
    }
    if (!whole) return;   // ragged last tile: fill_vec
    const size_t v = (size_t)head * p.N + (size_t)t * kT;
    uint8_t* vec = st + VEC_OFF;
    bulk_load(vec, p.L + v, 128, bar);
    bulk_load(vec + 128, p.D + v, 128, bar);
    bulk_load(vec + 256, p.ws + 2 * v, 256, bar);
  }
  __device__ static void load_b(const Params&, uint8_t*, uint64_t*, int, int) {}
  // L, D, (alpha, E) of tile t with bounds checks (128 threads, thread i)
  __device__ static void fill_vec(const Params& p, float* dst, int t, int head, int i) {
    for (int k = i; k < 4 * T; k += 128) {
      float v = 0.f;
      if (k < 2 * T) {
        const int q = t * T + (k % T);
        if (q < p.N) v = (k < T ? p.L : p.D)[(size_t)head * p.N + q];
      } else {
        const int q = t * T + (k - 2 * T) / 2;
        if (q < p.N) v = p.ws[2 * ((size_t)head * p.N + q) + (k & 1)];
      }
      dst[k] = v;
    }
  }

  __device__ static void score_mmas(uint32_t sc, uint32_t tres, uint32_t res, uint32_t sa, uint32_t) {
    const uint32_t i64 = idesc_bf16(kM, 64, false, false), i32 = idesc_bf16(kM, 32, false, false);
#pragma unroll
    for (int k = 0; k < D / 16; ++k)  // [S^T | K UQ^T] = K [Q; UQ]^T
      mma_ts_w(sc, tres_a(tres, 0, D, k), kmaj_lo(sa, ACH, 0, k), i64, k > 0);
#pragma unroll
    for (int k = 0; k < D / 16; ++k)  // B^T += UK Q^T
      mma_ts_w(sc + 32, tres_a(tres, 1, D, k), kmaj_lo(sa, ACH, 0, k), i32, 1);
#pragma unroll
    for (int k = 0; k < D / 16; ++k) {
      if (kAllTmem) {
        mma_ts_w(sc + 64, tres_a(tres, 2, D, k), kmaj_lo(sa, ACH, 2, k), i32, k > 0);  // dP^T = V dO^T
        mma_ts_w(sc + 96, tres_a(tres, 3, D, k), kmaj_lo(sa, ACH, 2, k), i32, k > 0);  // C^T = UV dO^T
      } else {
        mma_ss_w(sc + 64, res_lo(res, 0, DC, k), kmaj_lo(sa, ACH, 2, k), i32, k > 0);
        mma_ss_w(sc + 96, res_lo(res, 1, DC, k), kmaj_lo(sa, ACH, 2, k), i32, k > 0);
      }
    }
  }

  __device__ static void accum_mmas(uint32_t tb, uint32_t ops, uint32_t sa, uint32_t h, bool first) {
    const uint32_t amn = desc_lo(sa, ACH);
    const uint32_t id = idesc_bf16(kM, D, false, true);
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
      const uint32_t acc0 = (first && kk == 0) ? 0u : 1u;
      if (kAllTmem) {
        const uint32_t a = ops + h * OP_HALF + kk * 8;
        mma_ts_w(tb + A_K, a, mn_lo(amn, 1, kk), id, acc0);        // dS^T UQ
        mma_ts_w(tb + A_K, a + 16, mn_lo(amn, 0, kk), id, 1);      // Gs^T Q
        mma_ts_w(tb + A_V, a + 32, mn_lo(amn, 2, kk), id, acc0);   // Gdp^T dO
      } else {
        mma_ss_w(tb + A_K, op_lo(ops, 0, h, kk), mn_lo(amn, 1, kk), id, acc0);
        mma_ss_w(tb + A_K, op_lo(ops, 1, h, kk), mn_lo(amn, 0, kk), id, 1);
        mma_ss_w(tb + A_V, op_lo(ops, 2, h, kk), mn_lo(amn, 2, kk), id, acc0);
      }
    }
  }

  struct Row {};
  __device__ static void ew_init(Row&, const Params&, int, int, int) {}

  // Query columns per warpgroup and tile (all of them: the split of columns
  // between the warpgroups measured slower here).
  static constexpr bool SPLIT = false;
  static constexpr int NC = SPLIT ? T / 2 : T;
  template <bool MASK>
  __device__ static bool ew_tile(Row&, const Params& p, const TileArgs& a, const TileSync& s, int r) {
    static_assert(NC == 32, "one query record per lane");
    const float sc = p.tau * kLog2e;
    // The tile's per-query constants, formed once per warp instead of once
    // per (key, query): (-L log2e, D, alpha, alpha D - E) in this warp's own
    // records (no other warp reads them, so a warp barrier orders them).
    float4* rec = reinterpret_cast<float4*>(a.smem + QREC) + (threadIdx.x >> 5) * T;
    {
      const int i = a.c0 + (int)(threadIdx.x & 31u);
      const float Lq = a.vec[i], Dq = a.vec[T + i];
      const float2 ae = reinterpret_cast<const float2*>(a.vec + 2 * T)[i];
      __syncwarp();   // every lane has read the previous tile's records
      rec[threadIdx.x & 31u] = make_float4(-Lq * kLog2e, Dq, ae.x, fmaf(ae.x, Dq, -ae.y));
      __syncwarp();
    }
    // one score buffer: its release comes first, the operands are taken after
    uint32_t wdS[NC / 2], wGs[NC / 2], wGd[NC / 2];
#pragma unroll
    for (int q = 0; q < NC / 16; ++q) {
      float S[16], B[16], dP[16], C[16];
      const uint32_t c = a.sc + a.c0 + q * 16;
      tmem_ld16x4(c, c + T, c + 2 * T, c + 3 * T, S, B, dP, C);
      if (q == NC / 16 - 1) s.release_scores();
#pragma unroll
      for (int j = 0; j < 16; j += 2) {
        float dsv[2], gsv[2], gdv[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int ii = q * 16 + j + e;   // query column (relative to a.c0)
          const float4 v = rec[ii];
          const int col = a.c0 + ii;         // tile column (query)
          const float pe = (!MASK || (col >= a.lo && col <= a.hi)) ? ex2(fmaf(S[j + e], sc, v.x)) : 0.f;
          const float te = dP[j + e] - v.y;
          const float bp = fmaf(p.tau, B[j + e], -v.z);
          dsv[e] = pe * te;
          gsv[e] = pe * (fmaf(bp, te, C[j + e]) + v.w);
          gdv[e] = pe * bp;
        }
        const int k = q * 8 + j / 2;
        wdS[k] = pack_bf16x2(dsv[0], dsv[1]);
        wGs[k] = pack_bf16x2(gsv[0], gsv[1]);
        wGd[k] = pack_bf16x2(gdv[0], gdv[1]);
      }
    }
    if (!s.acquire_ops()) return false;
#pragma unroll
    for (int q = 0; q < NC / 16; ++q) {
      if (kAllTmem) {
        const uint32_t o = a.ops + (a.c0 + q * 16) / 2;
        tmem_st8_nowait(o, wdS + 8 * q);
        tmem_st8_nowait(o + 16, wGs + 8 * q);
        tmem_st8_nowait(o + 32, wGd + 8 * q);
      } else {
        const int col = 32 * (int)a.h + a.c0 + q * 16;
        write_op_cols<8>(a.ops, (uint32_t)r, col, wdS + 8 * q);
        write_op_cols<8>(a.ops + kChunk, (uint32_t)r, col, wGs + 8 * q);
        write_op_cols<8>(a.ops + 2 * kChunk, (uint32_t)r, col, wGd + 8 * q);
      }
    }
    s.publish_ops();
    return true;
  }

  __device__ static void epilogue(Row&, const Params& p, const EpiArgs& e) {
    // every lane runs the (warp-collective) TMEM loads; rows >= N store nothing
    const bool keep = e.blk0 + e.r < p.N;
    const size_t ro = ((size_t)e.head * p.N + (keep ? e.blk0 + e.r : 0)) * p.dv;
    const int c_lo = e.g * (D / 2), c_hi = min(c_lo + D / 2, p.dv);   // columns >= dv hold zeros
#pragma unroll 1
    for (int c0 = c_lo; c0 < c_hi; c0 += 16) {
      float ak[16], av[16];
      tmem_ld16x2(e.tm + A_K + c0, e.tm + A_V + c0, ak, av);
#pragma unroll
      for (int j = 0; j < 16; ++j) ak[j] *= p.tau;
      if (keep) {
        store16(p.gK + ro + c0, ak);
        store16(p.gV + ro + c0, av);
      }
    }
  }
};

// ===========================================================================
// host side
// ===========================================================================
template <class Op>
cudaError_t launch(const char* name, const typename Op::Params& prm, dim3 grid, cudaStream_t s) {
  // the instantiation for (causal, ragged N)
  const bool ragged = prm.N % kM != 0;
  auto kernel = prm.causal ? (ragged ? tile_kernel<Op, true, true> : tile_kernel<Op, true, false>)
                           : (ragged ? tile_kernel<Op, false, true> : tile_kernel<Op, false, false>);
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, Op::SMEM);
  if (e != cudaSuccess) return e;
  prof_begin(s, name);
  kernel<<<grid, kThreads, Op::SMEM, s>>>(prm);
  prof_end(s);
  return cudaGetLastError();
}

// Pass-1 parameters (the row sweeps of either schedule).
bool make_p1(P1Params& p1, const BobArgs& a, const DevCtx& c, bool four_pass) {
  const int BH = a.BH, N = a.N;
  bool ok = make_bf16_map(&p1.mK, a.K, BH, N, a.d, kT) && make_bf16_map(&p1.mUK, a.UK, BH, N, a.d, kT) &&
            make_bf16_map(&p1.mV, a.V, BH, N, a.d, kT) && make_bf16_map(&p1.mUV, a.UV, BH, N, a.d, kT) &&
            make_bf16_map(&p1.mK64, a.K, BH, N, a.d, 64) && make_bf16_map(&p1.mV64, a.V, BH, N, a.d, 64) &&
            make_bf16_map(&p1.mdO_res, a.dO, BH, N, a.d, kM) && make_bf16_map(&p1.mUQ_res, a.UQ, BH, N, a.d, kM);
  if (four_pass) ok = ok && make_bf16_map(&p1.mUK64, a.UK, BH, N, a.d, 64);
  if (!ok) return false;
  p1.Q = static_cast<const __nv_bfloat16*>(a.Q);
  p1.UQ = static_cast<const __nv_bfloat16*>(a.UQ);
  p1.dO = static_cast<const __nv_bfloat16*>(a.dO);
  p1.L = a.L;
  p1.D = a.D;
  p1.O = a.O;
  p1.gQ = a.gQ;
  p1.gdO = a.gdO;
  p1.ws = a.ws;
  p1.N = N;
  p1.dv = a.d;
  p1.tau = a.tau;
  p1.causal = a.causal;
  p1.err = c.err;
  p1.wait_ns = c.wait_ns;
  p1.stall = c.stall;
  return true;
}

// Pass 2 (the column pass, shared by both schedules): reads (alpha, E).
template <int D>
cudaError_t pass2_d(const BobArgs& a, const DevCtx& c, const dim3& grid, cudaStream_t s) {
  const int BH = a.BH, N = a.N;
  P2Params p2;
  const bool ok = make_bf16_map(&p2.mQ, a.Q, BH, N, a.d, kT) && make_bf16_map(&p2.mUQ, a.UQ, BH, N, a.d, kT) &&
                  make_bf16_map(&p2.mdO, a.dO, BH, N, a.d, kT) && make_bf16_map(&p2.mV, a.V, BH, N, a.d, kM) &&
                  make_bf16_map(&p2.mUV, a.UV, BH, N, a.d, kM);
  if (!ok) return cudaErrorInvalidValue;
  p2.K = static_cast<const __nv_bfloat16*>(a.K);
  p2.UK = static_cast<const __nv_bfloat16*>(a.UK);
  p2.V = static_cast<const __nv_bfloat16*>(a.V);
  p2.UV = static_cast<const __nv_bfloat16*>(a.UV);
  p2.L = a.L;
  p2.D = a.D;
  p2.ws = a.ws;
  p2.gK = a.gK;
  p2.gV = a.gV;
  p2.N = N;
  p2.dv = a.d;
  p2.tau = a.tau;
  p2.causal = a.causal;
  p2.err = c.err;
  p2.wait_ns = c.wait_ns;
  p2.stall = c.stall;
  return launch<Pass2<D>>("bob_pass2", p2, grid, s);
}

template <int D>
cudaError_t bob_group(const BobArgs& a, const DevCtx& c, cudaStream_t s) {
  P1Params p1;
  if (!make_p1(p1, a, c, false)) return cudaErrorInvalidValue;
  const dim3 grid((a.N + kM - 1) / kM, a.BH);
  cudaError_t e;
  if constexpr (D == 64) {
    e = launch<PassU1Y<64, false, true>>("bob_pass1", p1, grid, s);   // one sweep
  } else {
    // the Z kernel reads what the U1-and-Y kernel wrote (U1 in gQ, alpha and E)
    e = launch<PassU1Y<D>>("bob_pass1_u1y", p1, grid, s);
    if (e == cudaSuccess) e = launch<PassZ<D>>("bob_pass1_z", p1, grid, s);
  }
  if (e != cudaSuccess) return e;
  if constexpr (D == 128) return tc_bob_cols_wide(a, c, s);
  else return pass2_d<D>(a, c, grid, s);
}

// Heads [h0, h0 + n) of a: every per-head array starts h0 heads further on.
BobArgs head_range(const BobArgs& a, int h0, int n) {
  const size_t nd = (size_t)a.N * a.d, n1 = (size_t)a.N;
  auto bf = [&](const void* p) { return static_cast<const void*>(static_cast<const char*>(p) + 2 * h0 * nd); };
  BobArgs b = a;
  b.Q = bf(a.Q), b.K = bf(a.K), b.V = bf(a.V), b.dO = bf(a.dO), b.UQ = bf(a.UQ), b.UK = bf(a.UK), b.UV = bf(a.UV);
  b.O = a.O + h0 * nd, b.L = a.L + h0 * n1, b.D = a.D + h0 * n1;
  b.gQ = a.gQ + h0 * nd, b.gK = a.gK + h0 * nd, b.gV = a.gV + h0 * nd, b.gdO = a.gdO + h0 * nd;
  b.ws = a.ws + 2 * h0 * n1;
  b.BH = n;
  return b;
}

// Whether to run the heads as two groups on two streams: when each pass's
// launch is a few waves long and its last wave is mostly empty, one group's
// pass 2 fills the SMs the other group's pass 1 tail leaves idle.  (One CTA
// per SM at a time: every kernel here takes all 512 TMEM columns.)
bool split_heads(const BobArgs& a) {
  const int sms = sm_count();
  if (a.BH < 2 || sms <= 0) return false;
  const long ctas = (long)a.BH * ((a.N + kM - 1) / kM);
  const long waves = (ctas + sms - 1) / sms;
  const long idle = waves * sms - ctas;
  return waves <= 16 && idle * 20 > waves * sms;   // more than 5 % of the slots idle
}

template <int D>
cudaError_t bob_d(const BobArgs& a, const DevCtx& c, cudaStream_t s) {
  if (!split_heads(a)) return bob_group<D>(a, c, s);
  SideStream side;
  if (side.fork(s) != cudaSuccess) return bob_group<D>(a, c, s);   // no side stream: run unsplit
  const int h1 = a.BH / 2;
  cudaError_t e0 = bob_group<D>(head_range(a, 0, h1), c, s);
  cudaError_t e1 = bob_group<D>(head_range(a, h1, a.BH - h1), c, side.stream());
  cudaError_t e2 = side.join();
  return e0 != cudaSuccess ? e0 : e1 != cudaSuccess ? e1 : e2;
}

// The four-pass schedule: alpha sweep, E sweep, row-output sweep, column pass.
template <int D>
cudaError_t bob4_d(const BobArgs& a, const DevCtx& c, cudaStream_t s) {
  P1Params p1;
  if (!make_p1(p1, a, c, true)) return cudaErrorInvalidValue;
  const dim3 grid((a.N + kM - 1) / kM, a.BH);
  cudaError_t e = launch<PassAlpha<D>>("bob4_alpha", p1, grid, s);
  if (e == cudaSuccess) e = launch<PassE<D>>("bob4_e", p1, grid, s);
  if (e == cudaSuccess) e = launch<PassU1Y<D, true>>("bob4_rows", p1, grid, s);
  if (e != cudaSuccess) return e;
  if constexpr (D == 128) return tc_bob_cols_wide(a, c, s);
  else return pass2_d<D>(a, c, grid, s);
}

}  // namespace

cudaError_t tc_bob(const BobArgs& a, const DevCtx& c, cudaStream_t s) {
  // d = 32, 96 run on the d = 64, 128 kernels with zero-padded columns
  return a.d <= 64 ? bob_d<64>(a, c, s) : bob_d<128>(a, c, s);
}

cudaError_t tc_bob_four_pass(const BobArgs& a, const DevCtx& c, cudaStream_t s) {
  return a.d <= 64 ? bob4_d<64>(a, c, s) : bob4_d<128>(a, c, s);
}

}  // namespace fbob

#ifdef FBOB_TRACE
FBOB_TRACE_IO(fbob_trace_io_bob)
#endif
