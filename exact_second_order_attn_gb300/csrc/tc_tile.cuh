// Warp-specialised tile-loop skeleton shared by the tensor-core kernels that
// stream one side of the attention matrix against a resident 128-row block:
// BoB pass 1 (query rows resident, key tiles streamed), BoB pass 2 (keys
// resident, query tiles streamed) and the two first-backward kernels.
//
// CTA of 11 warps:
//   warps 0-7  two elementwise warpgroups; warpgroup g handles the streamed
//              tiles t with t % 2 == g, so one group works on tile t while
//              the other works on tile t+1 - or, for a policy with one score
//              buffer that asks for it (SPLIT), both work on every tile, group
//              g on its half of the tile's columns, so the buffer is read and
//              released in half the time.  Thread r of either group owns TMEM
//              lane r = resident row r (row sums are thread-local partials).
//   warp 8     TMA producer (one thread).
//   warp 9     issues the score MMAs; TMEM owner (512 columns).
//   warp 10    issues the accumulator MMAs.
//
// Resident operands of the score MMAs live in TMEM when the policy says so
// (TRES > 0): at kernel start each elementwise warpgroup copies its share of
// the resident rows from global memory into TMEM (lane r = resident row r,
// two bf16 per column), and the score MMAs read them as the A operand (TS
// MMA).  Only the streamed tile then comes from shared memory, which keeps
// the 32- and 64-column score MMAs off the shared-memory bandwidth limit.
// Residents the policy keeps in shared memory (RES > 0) arrive by TMA.
//
// Per streamed tile t (Op::T = 32 or 64 rows):
//   1. TMA fills ring A (operands the accumulator MMAs also read, plus any
//      per-tile vectors) and ring B (operands only the score MMAs read); both
//      stages of a tile complete one barrier.
//   2. Score MMAs write fp32 score tiles into TMEM buffer t % NBUF; ring B's
//      stage is released as soon as they complete.
//   3. The owning warpgroup loads the scores, releases the TMEM buffer,
//      computes bf16 operands and writes them to operand half t % 2 (shared
//      memory for SS MMAs, TMEM for TS MMAs).
//   4. Accumulator MMAs read the operand half and ring A's stage; their
//      completion releases both.  Score and accumulator MMAs come from two
//      warps, so the tensor pipe works on later tiles' scores while a
//      warpgroup still computes tile t's operands.
// Every wait is bounded (tc_ptx.cuh mbar_wait); on give-up every role leaves
// its loop, copies and MMAs in flight are drained and TMEM is freed.
//
// A kernel is a policy class Op providing the layout constants and the
// device functions called below (see tc_bob.cu, tc_bwd.cu).
#pragma once

#include <type_traits>

#include "tc_ptx.cuh"

namespace fbob {

// tmap.cu: TMA map of a [B*H, N, d] bf16 tensor, box {64, rows, 1}, 128B swizzle.
bool make_bf16_map(CUtensorMap* m, const void* base, int BH, int N, int D, int rows);

namespace tile {

using namespace tc;

// Timeline instrumentation, compiled only with -DFBOB_TRACE: clock64 stamps of
// CTA (0, 0) of the kernel whose layout id matches g_trace_sel, one slot per
// (event, tile < 64).  Off in every normal build.
#ifdef FBOB_TRACE
static __device__ unsigned long long g_trace[16 * 64];
static __device__ int g_trace_sel;
#define FBOB_STAMP(ev, i)                                                                                  \
  do {                                                                                                     \
    if (trace_on && (i) < 64) g_trace[(ev)*64 + (i)] = clock64();                                          \
  } while (0)
#define FBOB_TRACE_IO(fn)                                                                                  \
  extern "C" int fn(int sel, void* out) {                                                                  \
    if (out) return (int)cudaMemcpyFromSymbol(out, fbob::tile::g_trace, sizeof(fbob::tile::g_trace));      \
    static unsigned long long zero[16 * 64];                                                               \
    cudaError_t e = cudaMemcpyToSymbol(fbob::tile::g_trace, zero, sizeof(zero));                           \
    if (e == cudaSuccess) e = cudaMemcpyToSymbol(fbob::tile::g_trace_sel, &sel, sizeof(int));              \
    return (int)e;                                                                                         \
  }
#else
#define FBOB_STAMP(ev, i) \
  do {                    \
  } while (0)
#endif

constexpr int kM = 128;            // resident rows per CTA = TMEM lanes
constexpr int kT = 32;             // streamed rows per tile
constexpr int kEwWarps = 8;
constexpr int kProdWarp = 8, kMmaWarp = 9, kAccWarp = 10;
constexpr int kThreads = 352;
constexpr int kChunk = 16384;      // 128 rows x 128 B: one 64-column chunk of a resident tile
constexpr int kBlk = 4096;         // 32 rows x 128 B: one 64-column chunk of a streamed tensor
constexpr float kLog2e = 1.4426950408889634f;
constexpr uint64_t kDrainNs = 200000000ull;
constexpr int kMaxStages = 8;

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

struct Ctrl {
  uint64_t res_full;
  uint64_t tres_full;    // TMEM residents written (both warpgroups)
  uint64_t a_full[kMaxStages], a_empty[kMaxStages];
  uint64_t b_empty[kMaxStages];
  uint64_t s_full[2], s_empty[2];
  uint64_t o_full[2], o_empty[2];
  uint64_t acc_full, drain, drain_acc;
  uint64_t red;          // epilogue: both warpgroups' row partials written
  uint64_t vfill[2];     // ragged N: a warpgroup's vectors written to its scratch
  uint32_t tmem_base;
  int abort_flag;
};

// Synchronisation handle given to the policy's per-tile elementwise code.
struct TileSync {
  Ctrl* c;
  const Waiter* w;
  int q;          // tile parity: score/operand barrier and operand half
  int k;          // t >> 1
  int sa;         // ring-A stage of the tile
  bool vec;       // the tile's ring-A stage carries vectors read by the warpgroup
  bool ts;        // operands go to TMEM
  bool one_ops;   // a single operand buffer (split columns): tile t reuses tile t-1's
#ifdef FBOB_TRACE
  bool trace_on, trace_all;
  int t;
#endif

  // scores of this tile are in registers: the TMEM buffer may be reused
  __device__ __forceinline__ void release_scores() const {
    FBOB_STAMP(3, t);
#ifdef FBOB_TRACE
    if (trace_all && t < 64) g_trace[(11 + ((threadIdx.x >> 5) & 7) / 2) * 64 + t] = clock64();  // warps 1,3,5,7 -> 11..14
#endif
    tc_fence_before();
    mbar_arrive(&c->s_empty[q]);
  }
  // wait until the accumulator MMAs of this group's previous tile have read
  // the operand half - with one operand buffer, those of the previous tile
  // (warp-uniform: the TMEM stores that follow are warp-collective)
  __device__ __forceinline__ bool acquire_ops() const {
    if (one_ops) {
      const int tp = 2 * k + q - 1;   // A(tp) completes phase tp >> 1 of o_empty[tp & 1]
      if (tp < 0) return true;
      return __all_sync(0xffffffffu, mbar_wait(&c->o_empty[tp & 1], (tp >> 1) & 1, *w));
    }
    return __all_sync(0xffffffffu, mbar_wait(&c->o_empty[q], (k & 1) ^ 1, *w));
  }
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
    // warp-uniform: the caller's TMEM loads that follow are warp-collective
    if (!__all_sync(0xffffffffu, mbar_wait(&c->red, 0, *w))) return false;
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
  int t;               // streamed tile index (data)
  int c0;              // first tile column this warpgroup handles (0, or T/2 when the columns are split)
  int lo, hi;          // tile columns [lo, hi] this thread's row may see (causal mask; else [0, T-1])
  uint8_t* smem;       // the kernel's dynamic shared memory (policy scratch at the policy's offsets)
};

// CAUSAL and RAGGED (N not a multiple of 128) are compile-time choices, so
// the kernels for full attention on whole tiles carry no mask code; the host
// launches the instantiation that matches the problem.
//
// Ragged N: TMA fills rows at or beyond N with zeros; the streamed tile that
// crosses N masks its columns >= N like the causal mask; resident rows >= N
// are computed on zeros and never stored; per-tile vectors (column kernels)
// of that last tile - of every tile when N is not a multiple of 4, since a
// bulk copy needs a 16-byte aligned source and head h starts at float h N -
// are read with bounds checks instead of a bulk copy.
//
// Narrower heads: a kernel built for D serves any head size p.dv <= D (a
// multiple of 16): global rows are p.dv wide, TMA fills the box columns at or
// beyond p.dv with zeros (the tensor maps carry the true width), the TMEM
// residents are padded with zeros, so the score MMAs see zero-padded rows and
// the accumulator columns >= p.dv stay zero and are never stored.
// Op::ONE_OPS (optional, default false): one operand buffer shared by
// consecutive tiles, for split columns where TMEM has no room for two.
template <class Op, class = void>
struct OneOps : std::false_type {};
template <class Op>
struct OneOps<Op, std::void_t<decltype(Op::ONE_OPS)>> : std::bool_constant<Op::ONE_OPS> {};

template <class Op, bool CAUSAL, bool RAGGED>
__global__ void __launch_bounds__(kThreads, 1) tile_kernel(const __grid_constant__ typename Op::Params p) {
  static_assert(Op::NSB == 0 || Op::NSB == Op::NSA, "ring B stages pair with ring A stages");
  static_assert(Op::NBUF < Op::NSA, "the MMA order needs more stages than score buffers");
  constexpr bool kSplit = Op::SPLIT;  // both warpgroups on every tile, half the columns each
  static_assert(!kSplit || Op::NBUF == 1, "split columns only with one score buffer");
  constexpr int kEwPerTile = kSplit ? 256 : 128;
  constexpr bool kOneOps = OneOps<Op>::value;
  static_assert(!kOneOps || (kSplit && Op::OP_HALF == 0), "one operand buffer: both warpgroups on every tile");
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ Ctrl ctrl;
  const int tid = threadIdx.x, warp = tid >> 5;
  // Causal: a row block (ROWS: resident queries) streams the key tiles up to
  // its diagonal, a column block (resident keys) the query tiles from its
  // diagonal.  Row blocks then run the heaviest (last) blocks first.
  const int blk = (Op::ROWS && CAUSAL) ? (int)(gridDim.x - 1 - blockIdx.x) : (int)blockIdx.x;
  const int blk0 = blk * kM, head = blockIdx.y;
  const int t_all = (p.N + Op::T - 1) / Op::T;
  const int t_begin = (CAUSAL && !Op::ROWS) ? blk0 / Op::T : 0;
  const int t_end = (CAUSAL && Op::ROWS) ? min(t_all, (blk0 + kM) / Op::T) : t_all;
  const int nt = t_end - t_begin;   // loop steps; step t streams tile t_begin + t
  uint8_t* res = smem;
  uint8_t* ring_a = res + Op::RES;
  uint8_t* ring_b = ring_a + Op::NSA * Op::SA;
  uint8_t* ops = ring_b + Op::NSB * Op::SB;

  if (tid == 0) {
    ctrl.abort_flag = 0;
    mbar_init(&ctrl.res_full, 1);
    mbar_init(&ctrl.tres_full, 256);
    for (int s = 0; s < Op::NSA; ++s) {
      mbar_init(&ctrl.a_full[s], 1);
      mbar_init(&ctrl.a_empty[s], Op::VEC ? 1 + kEwPerTile / 32 : 1);
    }
    for (int s = 0; s < Op::NSB; ++s) mbar_init(&ctrl.b_empty[s], 1);
    for (int q = 0; q < 2; ++q) {
      mbar_init(&ctrl.s_full[q], 1);
      mbar_init(&ctrl.s_empty[q], kEwPerTile);
      mbar_init(&ctrl.o_full[q], kEwPerTile);
      mbar_init(&ctrl.o_empty[q], 1);
    }
    mbar_init(&ctrl.acc_full, 1);
    mbar_init(&ctrl.drain, 1);
    mbar_init(&ctrl.drain_acc, 1);
    mbar_init(&ctrl.red, 256);
    mbar_init(&ctrl.vfill[0], 128);
    mbar_init(&ctrl.vfill[1], 128);
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
#ifdef FBOB_TRACE
  constexpr int kTraceId = Op::ACC * 1000000 + Op::SCOLS * 1000 + Op::TRES * 100 + Op::OP_HALF / 16 * 10 + Op::T / 32;
  const bool trace_cta = blockIdx.x == 0 && blockIdx.y == 0 && g_trace_sel == kTraceId && (tid & 31) == 0;
  const bool trace_on = trace_cta && (warp >= kEwWarps || (warp & 3) == 0);
#endif

  if (warp == kProdWarp) {
    // ------------------------------------------------------------------ TMA
    // Ring A and ring B stages of tile t fill together and complete one
    // barrier (a_full), so the MMA warp waits once per tile for its operands.
    if (live && (tid & 31) == 0) {
      int ia = 0;
      if constexpr (Op::RES > 0) {
        mbar_arrive_expect_tx(&ctrl.res_full, Op::RES);
        Op::load_res(p, res, &ctrl.res_full, blk0, head);
      }
      bool ok = true;
      for (int t = 0; t < nt && ok; ++t) {
        const int sa = t % Op::NSA;
        if (!(ok = mbar_wait(&ctrl.a_empty[sa], ((t / Op::NSA) & 1) ^ 1, wt))) break;
        if constexpr (Op::NSB > 0) {
          if (!(ok = mbar_wait(&ctrl.b_empty[sa], ((t / Op::NSA) & 1) ^ 1, wt))) break;
        }
        if (p.stall && t == 0) continue;  // test hook: nothing will fill this stage
        // vectors by bulk copy only for whole tiles at 16-byte aligned addresses
        const bool whole = !RAGGED || (p.N % 4 == 0 && (t_begin + t + 1) * Op::T <= p.N);
        mbar_arrive_expect_tx(&ctrl.a_full[sa],
                              Op::SA_TX + (Op::NSB > 0 ? Op::SB_TX : 0) - (Op::VEC && !whole ? 4 * Op::T * Op::NVEC : 0));
        Op::load_a(p, ring_a + sa * Op::SA, &ctrl.a_full[sa], t_begin + t, head, whole);
        if constexpr (Op::NSB > 0) Op::load_b(p, ring_b + sa * Op::SB, &ctrl.a_full[sa], t_begin + t, head);
        FBOB_STAMP(7, t);
        ia = t + 1;
      }
      if (!ok) {
        // give-up path: every copy already issued lands before the CTA exits
        if constexpr (Op::RES > 0) mbar_wait_drain(&ctrl.res_full, 0, kDrainNs);
        for (int t = (ia > Op::NSA ? ia - Op::NSA : 0); t < ia; ++t)
          mbar_wait_drain(&ctrl.a_full[t % Op::NSA], (t / Op::NSA) & 1, kDrainNs);
      }
    }
  } else if (warp == kMmaWarp) {
    // --------------------------------------------------------- score MMAs
    // Two warps issue MMAs: this one the score batches S(t), warp kAccWarp
    // the accumulator batches A(t).  An mbarrier probe costs an issuing warp
    // one to two hundred cycles, about as much as a batch of 32-column MMAs,
    // so each warp pays only for its own waits and the tensor pipe takes
    // work from both.  The two warps write disjoint TMEM (score buffers vs
    // accumulators) and each commit tracks its own warp's MMAs.  Ring A's
    // stage t is released by A(t)'s commit although S(t) also read it: A(t)
    // needs tile t's operands, which exist only after S(t) completed.
    // S(t) waits for its stage and, for t >= NBUF, for tile t - NBUF's
    // warpgroup to have read the score buffer; no wait depends on work issued
    // later (NBUF < NSA), so the order cannot deadlock.
    if (live) {  // the whole warp runs the loop; lane 0 issues (elect.sync)
      const uint32_t res_l = desc_lo(smem_u32(res), 16), ra = smem_u32(ring_a), rb = smem_u32(ring_b);
      bool ok = true;
      if constexpr (Op::RES > 0) ok = __all_sync(0xffffffffu, mbar_wait(&ctrl.res_full, 0, wt));
      if constexpr (Op::TRES > 0) ok = ok && __all_sync(0xffffffffu, mbar_wait(&ctrl.tres_full, 0, wt));
      const uint32_t tres = tb + Op::TRES_COL;
      for (int t = 0; ok && t < nt; ++t) {
        const int sa = t % Op::NSA, u = t - Op::NBUF;
        // both conditions probed in one go (their latencies overlap); the
        // bounded blocking waits only run when a probe found one incomplete
        FBOB_STAMP(4, t);
        // both conditions probed in one go (their latencies overlap); the
        // bounded blocking waits only run when the probe found one incomplete
        uint64_t* eb = &ctrl.s_empty[(u < 0 ? 0 : u) & 1];
        const uint32_t ep = u < 0 ? 1u : (uint32_t)((u >> 1) & 1);
        if (u < 0 || !__all_sync(0xffffffffu, mbar_test2(&ctrl.a_full[sa], (t / Op::NSA) & 1, eb, ep))) {
          ok = __all_sync(0xffffffffu, mbar_wait(&ctrl.a_full[sa], (t / Op::NSA) & 1, wt));
          FBOB_STAMP(15, t);
          ok = ok && __all_sync(0xffffffffu, u < 0 || mbar_wait(&ctrl.s_empty[u & 1], (u >> 1) & 1, wt));
        }
        if (!ok) break;
        FBOB_STAMP(5, t);
        tc_fence_after();
        FBOB_STAMP(9, t);
        Op::score_mmas(tb + Op::ACC + (t % Op::NBUF) * Op::SCOLS, tres, res_l, desc_lo(ra + sa * Op::SA, 16),
                       desc_lo(rb + sa * Op::SB, 16));
        mma_commit_w(&ctrl.s_full[t & 1]);
        if constexpr (Op::NSB > 0) mma_commit_w(&ctrl.b_empty[sa]);
        FBOB_STAMP(0, t);
      }
      mma_commit_w(&ctrl.drain);
      mbar_wait_drain(&ctrl.drain, 0, kDrainNs);
    }
  } else if (warp == kAccWarp) {
    // --------------------------------------------------- accumulator MMAs
    if (live) {
      const uint32_t ra = smem_u32(ring_a);
      const uint32_t ops_a = Op::TS ? (tb + Op::OP_COL) : desc_lo(smem_u32(ops), 16);
      bool ok = true;
      for (int t = 0; ok && t < nt; ++t) {
        ok = __all_sync(0xffffffffu, mbar_wait(&ctrl.o_full[t & 1], (t >> 1) & 1, wt));
        // With one score buffer read by one warpgroup per tile, S(t+2) waits
        // for that warpgroup to have read S(t+1), a turnaround during which
        // the tensor pipe has nothing queued; A(t), issued as soon as its
        // operands exist, would instead run interleaved with S(t+1).  So A(t)
        // waits for S(t+1) to complete and fills that turnaround.  (With
        // split columns the buffer is released soon enough that A(t) would
        // only delay S(t+2).  The barrier cannot run two phases ahead of this
        // wait: that needs S(t+3) to complete, two score batches later.)
        if (Op::NBUF == 1 && !Op::SPLIT && t + 1 < nt)
          ok = ok && __all_sync(0xffffffffu, mbar_wait(&ctrl.s_full[(t + 1) & 1], ((t + 1) >> 1) & 1, wt));
        if (!ok) break;
        tc_fence_after();
        FBOB_STAMP(10, t);
        Op::accum_mmas(tb, ops_a, ra + (t % Op::NSA) * Op::SA, t & 1, t == 0);
        mma_commit_w(&ctrl.o_empty[t & 1]);
        mma_commit_w(&ctrl.a_empty[t % Op::NSA]);
        FBOB_STAMP(1, t);
      }
      if (ok) mma_commit_w(&ctrl.acc_full);
      mma_commit_w(&ctrl.drain_acc);
      mbar_wait_drain(&ctrl.drain_acc, 0, kDrainNs);
    }
  } else {
    // ------------------------------------------------------------ elementwise
    const int g = warp >> 2;                 // warpgroup
    const int r = tid & 127;                 // tile row = TMEM lane
    const uint32_t lane = (uint32_t)((warp & 3) * 32) << 16;
    typename Op::Row row;
    if constexpr (Op::TRES > 0) {
      // resident rows -> TMEM: warpgroup g copies residents g, g + 2, ...
      // (rows at or beyond N, and columns at or beyond the head size p.dv
      // of a narrower head, are zeros)
      const bool row_ok = blk0 + r < p.N;
      const size_t row_g = (size_t)head * p.N + (row_ok ? blk0 + r : 0);
      const int dv8 = p.dv / 8;
      for (int s = g; s < Op::TRES; s += 2) {
        const uint4* src = reinterpret_cast<const uint4*>(Op::tres_src(p, s)) + row_g * dv8;
        const uint32_t col = tb + lane + Op::TRES_COL + (uint32_t)(s * (Op::D / 2));
#pragma unroll
        for (int c = 0; c < Op::D / 32; ++c) {  // 16 columns = 32 bf16 per store
          uint32_t w[16];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint4 u = (row_ok && 4 * c + q < dv8) ? src[4 * c + q] : make_uint4(0u, 0u, 0u, 0u);
            w[4 * q] = u.x;
            w[4 * q + 1] = u.y;
            w[4 * q + 2] = u.z;
            w[4 * q + 3] = u.w;
          }
          tmem_st16_nowait(col + 16 * c, w);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&ctrl.tres_full);
    }
    Op::ew_init(row, p, blk0, r, head);
    bool ok = live;
    int nfill = 0;   // uses of this warpgroup's vector scratch (double-buffered)
    for (int t = kSplit ? 0 : g; t < nt && ok; t += kSplit ? 1 : 2) {
      const int q = t & 1, k = t >> 1, sa = t % Op::NSA;
      FBOB_STAMP(8, t);
      // waits are warp-uniform: a warp must never split in front of the
      // warp-collective TMEM loads and stores of the tile
      if (Op::VEC && !__all_sync(0xffffffffu, mbar_wait(&ctrl.a_full[sa], (t / Op::NSA) & 1, wt))) { ok = false; break; }
      if (!__all_sync(0xffffffffu, mbar_wait(&ctrl.s_full[q], k & 1, wt))) { ok = false; break; }
      FBOB_STAMP(2, t);
      tc_fence_after();
#ifdef FBOB_TRACE
      const TileSync sync{&ctrl, &wt, q, k, sa, Op::VEC, Op::TS, kOneOps, trace_on, trace_cta && ((warp & 1) == 1), t};
#else
      const TileSync sync{&ctrl, &wt, q, k, sa, Op::VEC, Op::TS, kOneOps};
#endif
      TileArgs ta;
      ta.sc = tb + lane + Op::ACC + (t % Op::NBUF) * Op::SCOLS;
      ta.vec = Op::VEC ? reinterpret_cast<const float*>(ring_a + sa * Op::SA + Op::VEC_OFF) : nullptr;
      if (Op::VEC && RAGGED && (p.N % 4 != 0 || (t_begin + t + 1) * Op::T > p.N)) {
        // no bulk copy for this tile (see the producer): the warpgroup reads
        // the tile's vectors itself
        // buffer nfill % 2: its previous reader finished before this
        // warpgroup's previous rendezvous, which every thread has passed
        float* scr = reinterpret_cast<float*>(smem + Op::VEC_SCRATCH) + (2 * g + (nfill & 1)) * (Op::NVEC * Op::T);
        Op::fill_vec(p, scr, t_begin + t, head, r);
        mbar_arrive(&ctrl.vfill[g]);   // bounded rendezvous of the warpgroup
        if (!__all_sync(0xffffffffu, mbar_wait(&ctrl.vfill[g], nfill & 1, wt))) { ok = false; break; }
        ++nfill;
        ta.vec = scr;
      }
      ta.ops = Op::TS ? (tb + lane + Op::OP_COL + (uint32_t)q * Op::OP_HALF) : smem_u32(ops);
      ta.h = (uint32_t)q;
      ta.t = t_begin + t;
      ta.c0 = kSplit ? g * (Op::T / 2) : 0;
      ta.smem = smem;
      // causal: column c of the tile is key / query (t_begin + t) T + c
      const int diag = blk0 + r - ta.t * Op::T;   // this row's own index, as a tile column
      ta.lo = (CAUSAL && !Op::ROWS) ? diag : 0;
      ta.hi = (CAUSAL && Op::ROWS) ? diag : Op::T - 1;
      if (RAGGED) ta.hi = min(ta.hi, p.N - 1 - ta.t * Op::T);   // columns >= N
      // tiles that cross the diagonal (causal) take the masked variant; the
      // vote keeps the choice warp-uniform
      constexpr bool kMask = CAUSAL || RAGGED;
      if (kMask && __any_sync(0xffffffffu, ta.lo > 0 || ta.hi < Op::T - 1))
        ok = Op::template ew_tile<kMask>(row, p, ta, sync, r);
      else
        ok = Op::template ew_tile<false>(row, p, ta, sync, r);
      FBOB_STAMP(6, t);

    }
    const EpiArgs ea{tb + lane, reinterpret_cast<float*>(ring_a), &ctrl, &wt, blk0, r, head, g};
    if (ok && __all_sync(0xffffffffu, mbar_wait(&ctrl.acc_full, 0, wt))) {
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
// TMEM-resident operand `slot` (d/2 columns each, two bf16 per column), k-th
// 16-element step: the A address of a TS MMA.
__device__ __forceinline__ uint32_t tres_a(uint32_t tres, int slot, int d, int k) {
  return tres + (uint32_t)(slot * (d / 2) + k * 8);
}
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

// Byte-offset forms for any streamed tile height: `off` is the byte offset
// of the operand block inside a 64-column chunk (block b of T rows: b * T * 128).
__device__ __forceinline__ uint32_t kmaj(uint32_t st_lo0, int chunk, int off, int k) {
  return st_lo0 + (uint32_t)(((k >> 2) * chunk + off + (k & 3) * 32) >> 4);
}
__device__ __forceinline__ uint32_t mnmaj(uint32_t st_mn_lo0, int off, int kk) {
  return st_mn_lo0 + (uint32_t)((off + kk * 2048) >> 4);
}
// 64-row tiles: operand `slot` of half h is its own [128][64] tile
// ((2 slot + h)-th 16 KB tile), kk-th 16-column step.
__device__ __forceinline__ uint32_t op64_lo(uint32_t ops_lo0, int slot, uint32_t h, int kk) {
  return ops_lo0 + (uint32_t)(((2 * slot + (int)h) * kChunk + kk * 32) >> 4);
}
// Write 64 packed bf16 (32 words) of row r into a 128B-swizzled [128][64] tile.
__device__ __forceinline__ void write_op64(uint32_t tile, uint32_t r, const uint32_t* w) {
#pragma unroll
  for (int cc = 0; cc < 8; ++cc)
    st_shared_v4(tile + sw128_offset(r, cc), w[4 * cc], w[4 * cc + 1], w[4 * cc + 2], w[4 * cc + 3]);
}

// Write NW packed words (2 NW bf16) of row r into columns [col0, col0 + 2 NW)
// of a 128B-swizzled [128][64] operand tile (col0 a multiple of 8).
template <int NW>
__device__ __forceinline__ void write_op_cols(uint32_t tile, uint32_t r, int col0, const uint32_t* w) {
#pragma unroll
  for (int cc = 0; cc < NW / 4; ++cc)
    st_shared_v4(tile + sw128_offset(r, (uint32_t)(col0 / 8 + cc)), w[4 * cc], w[4 * cc + 1], w[4 * cc + 2],
                 w[4 * cc + 3]);
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
