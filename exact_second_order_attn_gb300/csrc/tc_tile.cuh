// Warp-specialised tile-loop skeleton shared by the tensor-core kernels that
// stream one side of the attention matrix against a resident 128-row block:
// BoB pass 1 (query rows resident, key tiles streamed), BoB pass 2 (keys
// resident, query tiles streamed) and the two first-backward kernels.
//
// CTA of 10 warps:
//   warps 0-7  two elementwise warpgroups; warpgroup g handles the streamed
//              tiles t with t % 2 == g, so one group works on tile t while the
//              other works on tile t+1.  Thread r of either group owns TMEM
//              lane r = tile row r (row sums are thread-local).
//   warp 8     TMA producer (one thread).
//   warp 9     tcgen05.mma issuer (one thread) and TMEM owner (512 columns).
//
// Per 32-row streamed tile t:
//   1. TMA fills ring A (operands the accumulator MMAs also read, plus any
//      per-tile vectors) and ring B (operands only the score MMAs read).
//   2. Score MMAs write fp32 score tiles into TMEM buffer t % NBUF; ring B's
//      stage is released as soon as they complete.
//   3. The owning warpgroup loads the scores, releases the TMEM buffer,
//      computes bf16 operands and writes them to operand half t % 2 (shared
//      memory for SS MMAs, TMEM for TS MMAs).
//   4. Accumulator MMAs read the operand half and ring A's stage; their
//      completion releases both.  The MMA thread issues whichever of the next
//      score batch and the next accumulator batch is ready, so the tensor pipe
//      works on later tiles while a warpgroup still computes operands.
// Every wait is bounded (tc_ptx.cuh mbar_wait); on give-up every role leaves
// its loop, copies and MMAs in flight are drained and TMEM is freed.
//
// A kernel is a policy class Op providing the layout constants and the
// device functions called below (see tc_bob.cu, tc_bwd.cu).
#pragma once

#include "tc_ptx.cuh"

namespace fbob {

// tmap.cu: TMA map of a [B*H, N, d] bf16 tensor, box {64, rows, 1}, 128B swizzle.
bool make_bf16_map(CUtensorMap* m, const void* base, int BH, int N, int D, int rows);

namespace tile {

using namespace tc;

constexpr int kM = 128;            // resident rows per CTA = TMEM lanes
constexpr int kT = 32;             // streamed rows per tile
constexpr int kEwWarps = 8;
constexpr int kProdWarp = 8, kMmaWarp = 9;
constexpr int kThreads = 320;
constexpr int kChunk = 16384;      // 128 rows x 128 B: one 64-column chunk of a resident tile
constexpr int kBlk = 4096;         // 32 rows x 128 B: one 64-column chunk of a streamed tensor
constexpr float kLog2e = 1.4426950408889634f;
constexpr uint64_t kDrainNs = 200000000ull;
constexpr int kMaxStages = 4;

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

struct Ctrl {
  uint64_t res_full;
  uint64_t a_full[kMaxStages], a_empty[kMaxStages];
  uint64_t b_full[kMaxStages], b_empty[kMaxStages];
  uint64_t s_full[2], s_empty[2];
  uint64_t o_full[2], o_empty[2];
  uint64_t acc_full, drain;
  uint64_t red;          // epilogue: both warpgroups' row partials written
  uint32_t tmem_base;
  int abort_flag;
};

// Synchronisation handle given to the policy's per-tile elementwise code.
struct TileSync {
  Ctrl* c;
  const Waiter* w;
  int q;          // tile parity = warpgroup
  int k;          // tile index within this warpgroup
  int sa;         // ring-A stage of the tile
  bool vec;       // the tile's ring-A stage carries vectors read by the warpgroup
  bool ts;        // operands go to TMEM

  // scores of this tile are in registers: the TMEM buffer may be reused
  __device__ __forceinline__ void release_scores() const {
    tc_fence_before();
    mbar_arrive(&c->s_empty[q]);
  }
  // wait until the accumulator MMAs of this group's previous tile have read
  // the operand half
  __device__ __forceinline__ bool acquire_ops() const { return mbar_wait(&c->o_empty[q], (k & 1) ^ 1, *w); }
  // operands written: hand them to the MMA thread (and release the ring-A
  // vectors this warpgroup read)
  __device__ __forceinline__ void publish_ops() const {
    if (ts) {
      tmem_st_wait();
      tc_fence_before();
    } else {
      fence_proxy_async_smem();
    }
    mbar_arrive(&c->o_full[q]);
    if (vec) {
      __syncwarp();
      if ((threadIdx.x & 31u) == 0u) mbar_arrive(&c->a_empty[sa]);
    }
  }
};

// What the policy's epilogue gets: this thread's TMEM lane base, a scratch
// area (ring A, idle once every tile is consumed) and the reduction barrier.
struct EpiArgs {
  uint32_t tm;         // TMEM address with this warp's lane bits, column 0
  float* scratch;      // >= 2 KB of shared memory
  Ctrl* c;
  const Waiter* w;
  int blk0, r, head, g;

  // Sum two per-row partials (a, b) over both warpgroups, in a fixed order.
  // Every elementwise thread calls this once; the wait is bounded.
  __device__ __forceinline__ bool sum_rows(float& a, float& b) const {
    float2* red = reinterpret_cast<float2*>(scratch);
    red[g * 128 + r] = make_float2(a, b);
    mbar_arrive(&c->red);
    if (!mbar_wait(&c->red, 0, *w)) return false;
    const float2 x = red[r], y = red[128 + r];
    a = x.x + y.x;
    b = x.y + y.y;
    return true;
  }
};

// Everything the policy's elementwise code needs for one tile.
struct TileArgs {
  uint32_t sc;         // TMEM address (lane bits included) of the tile's score buffer
  const float* vec;    // ring-A vectors of the tile (shared memory) or nullptr
  uint32_t ops;        // SS: shared address of operand tile 0; TS: TMEM address of the half's first column
  uint32_t h;          // operand half (SS: columns 32h..32h+31 of each [128][64] operand tile)
  int t;               // tile index
};

template <class Op>
__global__ void __launch_bounds__(kThreads, 1) tile_kernel(const __grid_constant__ typename Op::Params p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ Ctrl ctrl;
  const int tid = threadIdx.x, warp = tid >> 5;
  const int blk0 = blockIdx.x * kM, head = blockIdx.y;
  const int nt = p.N / kT;
  uint8_t* res = smem;
  uint8_t* ring_a = res + Op::RES;
  uint8_t* ring_b = ring_a + Op::NSA * Op::SA;
  uint8_t* ops = ring_b + Op::NSB * Op::SB;

  if (tid == 0) {
    ctrl.abort_flag = 0;
    mbar_init(&ctrl.res_full, 1);
    for (int s = 0; s < Op::NSA; ++s) {
      mbar_init(&ctrl.a_full[s], 1);
      mbar_init(&ctrl.a_empty[s], Op::VEC ? 1 + 4 : 1);
    }
    for (int s = 0; s < Op::NSB; ++s) {
      mbar_init(&ctrl.b_full[s], 1);
      mbar_init(&ctrl.b_empty[s], 1);
    }
    for (int q = 0; q < 2; ++q) {
      mbar_init(&ctrl.s_full[q], 1);
      mbar_init(&ctrl.s_empty[q], 128);
      mbar_init(&ctrl.o_full[q], 128);
      mbar_init(&ctrl.o_empty[q], 1);
    }
    mbar_init(&ctrl.acc_full, 1);
    mbar_init(&ctrl.drain, 1);
    mbar_init(&ctrl.red, 256);
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

  if (warp == kProdWarp) {
    // ------------------------------------------------------------------ TMA
    if (live && (tid & 31) == 0) {
      int ia = 0, ib = 0;
      mbar_arrive_expect_tx(&ctrl.res_full, Op::RES);
      Op::load_res(p, res, &ctrl.res_full, blk0, head);
      bool ok = true;
      for (int t = 0; t < nt && ok; ++t) {
        const int sa = t % Op::NSA;
        if (!(ok = mbar_wait(&ctrl.a_empty[sa], ((t / Op::NSA) & 1) ^ 1, wt))) break;
        if (p.stall && t == 0) continue;  // test hook: nothing will fill this stage
        mbar_arrive_expect_tx(&ctrl.a_full[sa], Op::SA_TX);
        Op::load_a(p, ring_a + sa * Op::SA, &ctrl.a_full[sa], t, head);
        ia = t + 1;
        if constexpr (Op::NSB > 0) {
          const int sb = t % Op::NSB;
          if (!(ok = mbar_wait(&ctrl.b_empty[sb], ((t / Op::NSB) & 1) ^ 1, wt))) break;
          mbar_arrive_expect_tx(&ctrl.b_full[sb], Op::SB_TX);
          Op::load_b(p, ring_b + sb * Op::SB, &ctrl.b_full[sb], t, head);
          ib = t + 1;
        }
      }
      if (!ok) {
        // give-up path: every copy already issued lands before the CTA exits
        mbar_wait_drain(&ctrl.res_full, 0, kDrainNs);
        for (int t = (ia > Op::NSA ? ia - Op::NSA : 0); t < ia; ++t)
          mbar_wait_drain(&ctrl.a_full[t % Op::NSA], (t / Op::NSA) & 1, kDrainNs);
        if constexpr (Op::NSB > 0) {
          for (int t = (ib > Op::NSB ? ib - Op::NSB : 0); t < ib; ++t)
            mbar_wait_drain(&ctrl.b_full[t % Op::NSB], (t / Op::NSB) & 1, kDrainNs);
        }
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------------ MMA
    // Score batches S(t) and accumulator batches A(u) are each issued in
    // order; between them the thread issues whichever is ready (A first: it
    // frees stages), so a warpgroup still computing A(u)'s operands does not
    // hold back S(t+1).  Readiness is probed without blocking; one bounded
    // timer covers any stretch without progress.
    if (live) {  // the whole warp runs the loop; lane 0 issues (elect.sync)
      const uint32_t res_l = desc_lo(smem_u32(res), 16), ra = smem_u32(ring_a), rb = smem_u32(ring_b);
      const uint32_t ops_a = Op::TS ? (tb + Op::OP_COL) : desc_lo(smem_u32(ops), 16);
      bool ok = __all_sync(0xffffffffu, mbar_wait(&ctrl.res_full, 0, wt));
      int ns = 0, na = 0;  // next score batch, next accumulator batch
      uint64_t idle_since = 0;
      while (ok && na < nt) {
        bool progressed = false;
        if (na < ns && mbar_test_w(&ctrl.o_full[na & 1], (na >> 1) & 1)) {
          tc_fence_after();
          Op::accum_mmas(tb, ops_a, ra + (na % Op::NSA) * Op::SA, na & 1, na == 0);
          mma_commit_w(&ctrl.o_empty[na & 1]);
          mma_commit_w(&ctrl.a_empty[na % Op::NSA]);
          ++na;
          progressed = true;
        }
        if (ns < nt) {
          const int t = ns;
          bool ready = mbar_test_w(&ctrl.a_full[t % Op::NSA], (t / Op::NSA) & 1);
          uint32_t stage_b = rb;
          if constexpr (Op::NSB > 0) {
            ready = ready && mbar_test_w(&ctrl.b_full[t % Op::NSB], (t / Op::NSB) & 1);
            stage_b = rb + (t % Op::NSB) * Op::SB;
          }
          if (ready && t >= Op::NBUF) {  // the previous user of this score buffer has read it
            const int u = t - Op::NBUF;
            ready = mbar_test_w(&ctrl.s_empty[u & 1], (u >> 1) & 1);
          }
          if (ready) {
            tc_fence_after();
            Op::score_mmas(tb + Op::ACC + (t % Op::NBUF) * Op::SCOLS, res_l, desc_lo(ra + (t % Op::NSA) * Op::SA, 16),
                           desc_lo(stage_b, 16));
            mma_commit_w(&ctrl.s_full[t & 1]);
            if constexpr (Op::NSB > 0) mma_commit_w(&ctrl.b_empty[t % Op::NSB]);
            ++ns;
            progressed = true;
          }
        }
        if (progressed) {
          idle_since = 0;
        } else {
          __nanosleep(20);
          // lane 0 decides; the decision is broadcast so the warp stays converged
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
      if (ok) mma_commit_w(&ctrl.acc_full);
      mma_commit_w(&ctrl.drain);
      mbar_wait_drain(&ctrl.drain, 0, kDrainNs);
    }
  } else {
    // ------------------------------------------------------------ elementwise
    const int g = warp >> 2;                 // warpgroup
    const int r = tid & 127;                 // tile row = TMEM lane
    const uint32_t lane = (uint32_t)((warp & 3) * 32) << 16;
    typename Op::Row row;
    Op::ew_init(row, p, blk0, r, head);
    bool ok = live;
    for (int t = g; t < nt && ok; t += 2) {
      const int k = t >> 1, sa = t % Op::NSA;
      if (Op::VEC && !mbar_wait(&ctrl.a_full[sa], (t / Op::NSA) & 1, wt)) { ok = false; break; }
      if (!mbar_wait(&ctrl.s_full[g], k & 1, wt)) { ok = false; break; }
      tc_fence_after();
      const TileSync sync{&ctrl, &wt, g, k, sa, Op::VEC, Op::TS};
      TileArgs ta;
      ta.sc = tb + lane + Op::ACC + (t % Op::NBUF) * Op::SCOLS;
      ta.vec = Op::VEC ? reinterpret_cast<const float*>(ring_a + sa * Op::SA + Op::VEC_OFF) : nullptr;
      ta.ops = Op::TS ? (tb + lane + Op::OP_COL + (uint32_t)g * Op::OP_HALF) : smem_u32(ops);
      ta.h = (uint32_t)g;
      ta.t = t;
      ok = Op::ew_tile(row, p, ta, sync, r);
    }
    const EpiArgs ea{tb + lane, reinterpret_cast<float*>(ring_a), &ctrl, &wt, blk0, r, head, g};
    if (ok && mbar_wait(&ctrl.acc_full, 0, wt)) {
      tc_fence_after();
      Op::epilogue(row, p, ea);
    } else if (Op::ROW_SUMS) {
      mbar_arrive(&ctrl.red);  // keep the other warpgroup's bounded wait short
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tb, 512);
  }
}

// ---------------------------------------------------------------------------
// helpers shared by the policies
// ---------------------------------------------------------------------------

// Descriptor low words (see tc_ptx.cuh desc_lo).  Offsets are in bytes and
// compile-time constants once the k loops are unrolled, so each operand of an
// MMA costs one add.
// K-major resident tile: slot of `dc` 64-column chunks of 16 KB, k-th 16-column step.
__device__ __forceinline__ uint32_t res_lo(uint32_t res_lo0, int slot, int dc, int k) {
  return res_lo0 + (uint32_t)(((slot * dc + (k >> 2)) * kChunk + (k & 3) * 32) >> 4);
}
// K-major streamed stage with 64-column chunks `chunk` bytes apart, 32-row block `blk`.
__device__ __forceinline__ uint32_t kmaj_lo(uint32_t st_lo0, int chunk, int blk, int k) {
  return st_lo0 + (uint32_t)(((k >> 2) * chunk + blk * kBlk + (k & 3) * 32) >> 4);
}
// MN-major streamed 32-row block `blk` (rows = the MMA's K), kk-th 16-row step;
// st_mn_lo0 = desc_lo(stage address, chunk stride).
__device__ __forceinline__ uint32_t mn_lo(uint32_t st_mn_lo0, int blk, int kk) {
  return st_mn_lo0 + (uint32_t)((blk * kBlk + kk * 2048) >> 4);
}
// K-major operand tile `slot` ([128][64], 16 KB each), half h, kk-th 16-column step.
__device__ __forceinline__ uint32_t op_lo(uint32_t ops_lo0, int slot, uint32_t h, int kk) {
  return ops_lo0 + (uint32_t)((slot * kChunk + kk * 32) >> 4) + h * 4u;
}

// Write 32 packed bf16 (16 words) of row r into columns [32h, 32h+32) of a
// 128B-swizzled [128][64] operand tile.
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

__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

}  // namespace tile
}  // namespace fbob
