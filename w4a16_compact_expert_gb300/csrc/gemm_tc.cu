// Prefill regime: persistent grouped GEMM on the 5th-generation tensor cores
// (tcgen05.mma, FP16 operands in shared memory, FP32 accumulators in TMEM).
//
// The compact int4 weights are the MMA A operand: two 128-row A matrices per
// tile share every token stage (gate/up: the gate and up rows m0 .. m0 + 127;
// down: rows m0 .. m0 + 255 of the down matrix as two halves).  The tokens of
// one expert are the N dimension (a token chunk of <= 256, or <= 128 in the
// narrow variant, padded only to a multiple of 16, so ragged expert loads
// waste little work).  Per 64-wide K
// step:
//   producer warp : 4-D TMA loads fetch the int4 chunks of the 8 row tiles of
//                   each A matrix (and, at scale-block starts, their block
//                   scales) into a raw ring; the token rows of B come as 2-D
//                   TMA tiles, 128-byte swizzled (for gate/up x rows in
//                   sorted-row order, copied there by the router or by a small
//                   kernel; h for down)
//   dequant warps : int4 -> FP16 (nearest q*s) written into a 128-byte
//                   swizzled K-major A ring (the only place an expanded value
//                   exists: one 64-wide K step of 2 x 128 rows, per CTA)
//   MMA warp      : one thread issues tcgen05.mma M128 x N x K16 for each A
//                   matrix into the two halves of one TMEM accumulator (the
//                   narrow variant alternates between two accumulators of
//                   2 x 128 columns) and commits stage releases
//   epilogue      : tcgen05.ld of the accumulator; gate/up: h = SiLU(g) * u
//                   rounded to FP16; down: y [pair][H] FP16.  With one
//                   accumulator split over the 4 epilogue warps and the 8
//                   dequant warps, a third each; with two, the 4 epilogue
//                   warps alone, under the next tile's MMAs
// A last kernel gathers out[t] = (x[t]) + sum_j w[t,j] y[t*k+j] in rank order.
// Every wait is bounded (status word + early exit), nothing spins forever.
// Sources: compact weights converted in-kernel with FP32 accumulation stages
// and explicit rounding (Horizon RunMap landing page, "08 / Precision &
// quality"); a grouped executor for the full-residency regime ("Horizon
// RunMap - architecture", "Regimes and executor boundaries").
#include <cuda.h>

#include "internal.h"

namespace {

constexpr int kMTile = 128;     // weight rows per tile (MMA M)
constexpr int kBK = 64;         // K per pipeline stage (one 128-byte swizzle row of FP16)
constexpr int kDqWarps = 8;     // dequant warps of one group (one 16-row tile of each A matrix each)
constexpr int kMaxE = 256;
constexpr uint32_t kTmemCols = 512;

// NMAX: tokens per tile (MMA N, max).
//  256 (prefill): many tokens per weight byte.  The dequant warps write the
//      FP16 weights into a shared-memory A ring; a shallow int4 ring keeps the
//      tensor cores fed; one accumulator of 2 x 256 TMEM columns.
//  32 (a few to ~16 tokens per expert): few tokens per weight byte, so the
//      tile must stream its weights at HBM speed.  There every 64-wide K step
//      of the shared-memory design cost ~1,400 cycles whatever the ring
//      depths: the MMA thread spent ~550 cycles issuing its 8 MMAs (M = 128,
//      N <= 64 costs ~60 cycles per MMA whatever N) and ~800 on the fixed
//      cost of a step (barrier wait, commits, loop).  So here a pipeline
//      stage is two 64-wide K chunks (16 MMAs per barrier round trip), the
//      dequant warps store the FP16 weights straight into tensor memory
//      (tcgen05.st, one row per TMEM lane, no shared-memory A ring) and the
//      MMA takes A from there; two groups of dequant warps take alternate
//      stages, a deep int4 ring covers HBM latency, and two accumulators let
//      one tile's epilogue run under the next tile's MMAs.
//  128 (prefill, alternative): the 256-token variant's A ring with two
//      accumulators of 2 x 128 columns (the epilogue of one tile runs under
//      the next tile's MMAs instead of stalling them: a trace of the 256-token
//      variant showed the MMA warp waiting 9,000-13,000 cycles for the
//      accumulator at each tile start) and two groups of dequant warps (each
//      expert's weights are converted once per 128-token tile).
template <bool GU, int NMAX>
struct Cfg {
  static constexpr bool kWide = NMAX > 64;
  static constexpr bool kTS = !kWide;                 // A (weights) from tensor memory
  static constexpr int kCh = kTS ? 2 : 1;             // 64-wide K chunks per A / int4 stage
  // two 128-row A tiles share every token stage: gate and up (gate/up), rows
  // m0 and m0 + 128 of the down matrix (down)
  static constexpr int kMats = 2;
  static constexpr int kAcc = NMAX <= 128 ? 2 : 1;    // accumulators
  static constexpr int kHalf = NMAX <= 128 ? NMAX : 256;   // TMEM column of the second A matrix's half
  // Warp roles: two MMA warps (0 and 3, each issuing the MMAs of one A
  // matrix: one thread issuing every MMA of a K step was the bottleneck of
  // the small-token pipeline, ~60 cycles per M = 128, N <= 64 MMA in
  // isolation and ~160 among busy dequant warps), the int4 producer (1), the
  // token producer (2), then 4 epilogue warps (one per TMEM lane quarter
  // warp % 4), then kDqGroups groups of 8 dequant warps (group g converts
  // the K steps s with s % kDqGroups == g).
  static constexpr int kDqGroups = NMAX <= 128 ? 2 : 1;
  static constexpr int kDqAll = kDqWarps * kDqGroups;
  static constexpr int kMmaWarps = 2;
  static constexpr int kWarpMma = 0, kWarpProd = 1, kWarpProdB = 2, kWarpMma2 = 3;
  static constexpr int kWarpEpi = 2 + kMmaWarps, kWarpDq = kWarpEpi + 4;
  static constexpr int kThreads = (kWarpDq + kDqAll) * 32;
  // every int4 stage carries its block scales when a group does not see the
  // first K step of every block
  static constexpr bool kScalesEveryStage = kDqGroups > 1;
  static constexpr int kStagesA = 3;                  // dequantised FP16 A stages
  static constexpr int kASmemStages = kTS ? 0 : kStagesA;
  static constexpr int kTmemA = 2 * kAcc * kHalf;     // TS: first TMEM column of the A stages
  static constexpr int kTmemAMat = kCh * kBK / 2;     // TS: columns of one matrix in an A stage (FP16 pairs)
  static constexpr int kTmemAStage = kMats * kTmemAMat;
  static constexpr int kStagesB = kTS ? 8 : 3;
  static constexpr int kBoxRows = kWide ? 64 : 16;    // token rows per TMA box of a B stage
  static constexpr int kAMat = kMTile * kBK * 2;          // 16 KB per matrix per stage
  static constexpr int kABytes = kMats * kAMat;
  static constexpr int kBBytes = NMAX * kBK * 2;          // 32 KB (256) or 4 KB (32)
  // per K chunk, the int4 chunks of 8 row tiles per matrix; then (at block
  // boundaries, or in every stage) the 16 block scales of the same 8 row
  // tiles per matrix
  static constexpr int kRawQ = kMats * 8 * 512;
  static constexpr int kRawBytes = kCh * kRawQ + kMats * 8 * 32;
  static constexpr int kSchedBytes = (4 * (kMaxE + 1) + 4) * 4;
  // int4 chunks (+ scales) from HBM: whatever the other rings leave
  static constexpr int kFixed = kASmemStages * kABytes + kStagesB * kBBytes + kSchedBytes +
                                (2 * kStagesA + 2 * kStagesB + 4) * 8 + 16 + 1024;
  static constexpr int kRawFit = (227 * 1024 - kFixed) / (kRawBytes + 16);
  static constexpr int kStagesRaw = NMAX > 128 ? 3 : (kRawFit < 16 ? kRawFit : 16);
  static constexpr int kOffA = 0;
  static constexpr int kOffB = kOffA + kASmemStages * kABytes;
  static constexpr int kOffRaw = kOffB + kStagesB * kBBytes;
  static constexpr int kOffSched = kOffRaw + kStagesRaw * kRawBytes;   // 4 x (kMaxE + 1) ints + count
  static constexpr int kOffBar = kOffSched + kSchedBytes;
  static constexpr int kNumBars = 2 * kStagesRaw + 2 * kStagesA + 2 * kStagesB + 4;
  static constexpr int kSmem = kOffBar + kNumBars * 8 + 16 + 1024;   // + TMEM slot + alignment slack
  static_assert(kSmem <= 227 * 1024, "shared memory budget");
  static_assert(kStagesRaw >= 3, "int4 ring depth");
  static_assert(kRawBytes % 128 == 0 && kBBytes % 1024 == 0, "ring alignment");
  static_assert(!kTS || kTmemA + kStagesA * kTmemAStage <= (int)kTmemCols, "tensor memory budget");
};

// K steps per token stage for a tile of n tokens: a stage holds NMAX rows of
// one K step, or, for fewer tokens, that many bytes of several consecutive K
// steps (each a K-major swizzled block of the tile's rows rounded up to the
// TMA box), so that a small tile keeps as many K steps in flight as the
// bytes allow.
template <class C>
DEV_INLINE int kb_per_stage(int n) {
  const int rows = (n + C::kBoxRows - 1) / C::kBoxRows * C::kBoxRows;
  const int kpb = C::kBBytes / (rows * 128);
  return kpb > 0 ? kpb : 1;
}

struct Ring {
  int i = 0;
  uint32_t ph = 0;
  DEV_INLINE void next(int n) {
    if (++i == n) {
      i = 0;
      ph ^= 1u;
    }
  }
};

struct Tile {
  int slot, r0, n, m0, u;
};

// The active-expert schedule written by the routing kernels, copied to shared
// memory once per CTA so that every role decodes tiles without global loads.
struct Sched {
  int n;            // active experts
  int* tile;        // [n + 1] prefix of token chunks
  int* slot;        // [n]
  int* start;       // [n]
  int* count;       // [n]
  int lo, hi;       // the tiles this launch covers
  // Tail split (256-token tile): the tiles [F, hi) of the last, partial wave
  // are taken as two token halves each, virtual tiles [F, vhi) = [F, F + 2 (hi - F)),
  // so that no CTA runs a whole tile more than the others
  int F, vhi;
  bool split;
};

DEV_INLINE Sched load_sched(const FwdCtx& c, int* sm) {
  Sched s;
  s.tile = sm;
  s.slot = sm + (kMaxE + 1);
  s.start = sm + 2 * (kMaxE + 1);
  s.count = sm + 3 * (kMaxE + 1);
  int* sn = sm + 4 * (kMaxE + 1);
  const int n = *c.n_active;
  for (int u = threadIdx.x; u <= n; u += blockDim.x) {
    const int tv = c.act_tile[u];
    int sl = 0, st = 0, ct = 0;
    if (u < n) {
      sl = c.act_slot[u];
      st = c.act_start[u];
      ct = c.act_count[u];
    }
    s.tile[u] = tv;
    if (u < n) {
      s.slot[u] = sl;
      s.start[u] = st;
      s.count[u] = ct;
    }
  }
  if (threadIdx.x == 0) *sn = n;
  __syncthreads();
  s.n = *sn;
  return s;
}

// Tile t -> (active expert, token chunk, weight-row tile).  Chunks split an
// expert's rows into ceil(count / tile_tokens) near-equal parts (the routing
// kernels wrote that prefix into act_tile).
DEV_INLINE bool get_tile(const Sched& s, int t, int mtiles, int mstep, Tile& out) {
  if (s.n <= 0) return false;
  if (t >= s.vhi) return false;
  int half = -1;
  if (s.split && t >= s.F) {   // a token half of a tail tile
    half = (t - s.F) & 1;
    t = s.F + ((t - s.F) >> 1);
  }
  const int mt = t % mtiles, ct = t / mtiles;
  int lo = 0, hi = s.n - 1;
  while (lo < hi) {   // last u with tile[u] <= ct
    const int mid = (lo + hi + 1) >> 1;
    if (s.tile[mid] <= ct) lo = mid;
    else hi = mid - 1;
  }
  const int u = lo;
  const int nch = s.tile[u + 1] - s.tile[u], ch = ct - s.tile[u];
  const int cnt = s.count[u];
  const int b0 = (int)((long long)ch * cnt / nch), b1 = (int)((long long)(ch + 1) * cnt / nch);
  out.slot = s.slot[u];
  out.r0 = s.start[u] + b0;
  out.n = b1 - b0;
  out.m0 = mt * mstep;
  out.u = u;
  if (half >= 0) {
    const int h0 = out.n >> 1;
    if (half == 0) {
      out.n = h0;
    } else {
      out.r0 += h0;
      out.n -= h0;
    }
  }
  return true;
}

// TMA: one box at (c0, c1, c2) of a 3-D tensor map.
DEV_INLINE void tma_load_3d(void* dst, const void* tmap, int c0, int c1, int c2, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cta.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
      "l"(tmap), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
      : "memory");
}

DEV_INLINE void st_shared_v4_b32(uint32_t addr, uint32_t v0, uint32_t v1, uint32_t v2, uint32_t v3) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v0), "r"(v1), "r"(v2), "r"(v3) : "memory");
}


// DENSE: the offload-qpacked comparison.  A comes as FP16 tiles of the
// execution slots of the active experts [c.ub0, c.ub1) (tmA0 / tmA1: 3-D maps,
// 128 rows x 64 K per load, 128-byte swizzled straight into the A ring), no
// dequantisation; the tile schedule covers only those experts.
template <bool GU, bool DENSE, int NMAX>
__global__ void __launch_bounds__(Cfg<GU, NMAX>::kThreads, 1)
    grouped_gemm_kernel(FwdCtx c, const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmA0,
                        const __grid_constant__ CUtensorMap tmA1, const __grid_constant__ CUtensorMap tmS0,
                        const __grid_constant__ CUtensorMap tmS1) {
  using C = Cfg<GU, NMAX>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* raw_full = bars;
  uint64_t* raw_empty = raw_full + C::kStagesRaw;
  uint64_t* a_full = raw_empty + C::kStagesRaw;
  uint64_t* a_empty = a_full + C::kStagesA;
  uint64_t* b_full = a_empty + C::kStagesA;
  uint64_t* b_empty = b_full + C::kStagesB;
  uint64_t* acc_full = b_empty + C::kStagesB;   // [2]
  uint64_t* acc_empty = acc_full + 2;           // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  pdl_wait();      // routing (and, for down, h) of the preceding grids
  pdl_trigger();
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStagesRaw; ++s) {
      mbar_init(&raw_full[s], 1);
      mbar_init(&raw_empty[s], kDqWarps);
    }
    for (int s = 0; s < C::kStagesA; ++s) {
      mbar_init(&a_full[s], DENSE ? 1 : kDqWarps);
      mbar_init(&a_empty[s], C::kMmaWarps);   // one commit per MMA warp
    }
    for (int s = 0; s < C::kStagesB; ++s) {
      mbar_init(&b_full[s], 1);
      mbar_init(&b_empty[s], C::kMmaWarps);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&acc_full[s], C::kMmaWarps);
      mbar_init(&acc_empty[s], C::kAcc == 1 ? 12 : 4);   // one arrive per warp that reads the accumulator
    }
    fence_mbar_init();
  }
  if (warp == C::kWarpMma) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  Sched sch = load_sched(c, reinterpret_cast<int*>(smem + C::kOffSched));   // contains __syncthreads
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const MatLayout& LA = GU ? c.lay.gate : c.lay.down;
  // gate/up: tiles of 128 rows of gate and up; down: tiles of 256 rows, the
  // second 128 rows as the second A matrix (row offset m1off)
  const int mstep = GU ? kMTile : 2 * kMTile, m1off = GU ? 0 : kMTile;
  // nks: 64-wide K chunks of a tile (token stages); nst: A / int4 stages
  const int K = (int)LA.k, nks = K / kBK, nst = nks / C::kCh, mtiles = (int)LA.rows / mstep;
  if (DENSE) {
    sch.lo = sch.tile[min(c.ub0, sch.n)] * mtiles;
    sch.hi = sch.tile[min(c.ub1, sch.n)] * mtiles;
  } else {
    sch.lo = 0;
    sch.hi = sch.n > 0 ? sch.tile[sch.n] * mtiles : 0;
  }
  sch.F = sch.vhi = sch.hi;
  sch.split = false;
  if (!DENSE && C::kAcc == 1) {
    // 256-token tile: with R tiles in the last, partial wave (R <= half the
    // grid), run them as 2R token halves, one per CTA: the kernel then ends
    // half a tile after the full waves instead of a whole tile (a 256-token
    // tile's time is mostly its MMAs, which halve).  Only when every tail
    // tile has at least 32 tokens, so that no half is nearly empty.
    const int G = (int)gridDim.x, N = sch.hi - sch.lo, R = N % G;
    if (R > 0 && 2 * R <= G) {
      const int F = sch.hi - R;
      bool big = true;
      for (int t = F + (int)threadIdx.x; t < sch.hi; t += (int)blockDim.x) {
        Tile tt;
        if (get_tile(sch, t, mtiles, mstep, tt)) big = big && tt.n >= 32;
      }
      if (__syncthreads_and(big)) {
        sch.split = true;
        sch.F = F;
        sch.vhi = F + 2 * R;
      }
    }
  }
  const int nacc = C::kAcc;
  // The epilogue of one tile for the calling warp's TMEM lane quarter, 32-column
  // chunks [ch0, ch1) of accumulator `ai`: gate/up -> h = SiLU(g) * u (FP16),
  // down -> y (FP16) of rows m0 + row (first accumulator half) and m0 + 128 +
  // row (second).  A single accumulator puts the epilogue on the MMA's
  // critical path: it is then split over the 4 epilogue warps and the 8
  // dequant warps (which wait for the MMA at that point anyway), a third each.
  auto epilogue_chunks = [&](const Tile& et, int ch0, int ch1, int ai) {
    const int qw = warp & 3, row = qw * 32 + lane;
    const uint32_t taddr = tmem + (uint32_t)(ai * 2 * C::kHalf) + ((uint32_t)(qw * 32) << 16);
    for (int col0 = ch0 * 32; col0 < ch1 * 32 && col0 < et.n; col0 += 32) {
      // the 32 columns' pair indices (down) or PRENORM row scales (gate/up):
      // one coalesced load per chunk, broadcast below
      int my_pair = 0;
      float my_rn = 1.f;
      if (col0 + lane < et.n) {
        if (!GU) my_pair = c.sorted[et.r0 + col0 + lane];
        else if (c.flags & 2u) my_rn = c.rnorm[c.sorted[et.r0 + col0 + lane] / c.k];
      }
      // 32 columns per TMEM load, or 2 x 16 in the narrow variant (whose 23
      // warps leave fewer registers per thread)
      constexpr int W = C::kThreads > 512 ? 16 : 32;
#pragma unroll
      for (int sub = 0; sub < 32; sub += W) {
        if (col0 + sub >= et.n) break;
        uint32_t va[W], vb[W];
        tmem_ld_cols(taddr + (uint32_t)(col0 + sub), va);
        tmem_ld_cols(taddr + (uint32_t)(C::kHalf + col0 + sub), vb);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < W; ++j) {
          const int nn = col0 + sub + j;
          const int pair = GU ? 0 : __shfl_sync(0xffffffffu, my_pair, sub + j);
          if (nn < et.n) {
            if (GU) {
              float gv = __uint_as_float(va[j]), uv = __uint_as_float(vb[j]);
              if (c.flags & 2u) {
                const float r = __shfl_sync(0xffffffffu, my_rn, sub + j);
                gv *= r;
                uv *= r;
              }
              c.hbuf[(size_t)(et.r0 + nn) * c.I + et.m0 + row] = __float2half_rn(silu_mul(gv, uv));
            } else {
              // the expert's output rounded once to FP16 (an activation), the
              // combine then sums the k ranks in FP32
              __half* yr = reinterpret_cast<__half*>(c.ybuf) + (size_t)pair * c.H + et.m0 + row;
              yr[0] = __float2half_rn(__uint_as_float(va[j]));
              yr[kMTile] = __float2half_rn(__uint_as_float(vb[j]));
            }
          }
        }
      }
    }
  };

  if (DENSE && warp == C::kWarpProd) {
    // ----------------------------------------- FP16 A producer (comparison)
    if (lane == 0) {
      Ring ra;
      for (int t = sch.lo + blockIdx.x;; t += gridDim.x) {
        Tile tl;
        if (!get_tile(sch, t, mtiles, mstep, tl)) break;
        bool ok = true;
        for (int ks = 0; ks < nks; ++ks) {
          if (!mbar_wait_bounded(&a_empty[ra.i], ra.ph ^ 1u, c.status)) {
            ok = false;
            break;
          }
          uint8_t* dst = smem + C::kOffA + ra.i * C::kABytes;
          mbar_expect_tx(&a_full[ra.i], (uint32_t)C::kABytes);
          tma_load_3d(dst, &tmA0, ks * kBK, tl.m0, tl.u - c.ub0, &a_full[ra.i]);
          tma_load_3d(dst + C::kAMat, &tmA1, ks * kBK, tl.m0 + m1off, tl.u - c.ub0, &a_full[ra.i]);
          ra.next(C::kStagesA);
        }
        if (!ok) break;
      }
    }
    __syncwarp();
  } else if (warp == C::kWarpProd) {
    // ------------------------------------------------- int4 chunk producer
    if (lane == 0) {
      Ring rr;
      for (int t = sch.lo + blockIdx.x;; t += gridDim.x) {
        Tile tl;
        if (!get_tile(sch, t, mtiles, mstep, tl)) break;
        bool ok = true;
        for (int ks = 0; ks < nst; ++ks) {
          if (!mbar_wait_bounded(&raw_empty[rr.i], rr.ph ^ 1u, c.status)) {
            ok = false;
            break;
          }
          uint8_t* dst = smem + C::kOffRaw + rr.i * C::kRawBytes;
          const int kc0 = ks * C::kCh;   // first K chunk of the stage
          // first K chunk of a scale block (or every stage): its scales come along
          const bool blk = C::kScalesEveryStage || (kc0 & 3) == 0;
          mbar_expect_tx(&raw_full[rr.i], blk ? (uint32_t)C::kRawBytes : (uint32_t)(C::kCh * C::kRawQ));
#pragma unroll
          for (int h = 0; h < C::kCh; ++h) {
            tma_load_4d(dst + h * C::kRawQ, &tmA0, 0, kc0 + h, tl.m0 / 16, tl.slot, &raw_full[rr.i]);
            tma_load_4d(dst + h * C::kRawQ + 8 * 512, &tmA1, 0, kc0 + h, (tl.m0 + m1off) / 16, tl.slot, &raw_full[rr.i]);
          }
          if (blk) {
            uint8_t* sdst = dst + C::kCh * C::kRawQ;
            tma_load_4d(sdst, &tmS0, 0, kc0 >> 2, tl.m0 / 16, tl.slot, &raw_full[rr.i]);
            tma_load_4d(sdst + 256, &tmS1, 0, kc0 >> 2, (tl.m0 + m1off) / 16, tl.slot, &raw_full[rr.i]);
          }
          rr.next(C::kStagesRaw);
        }
        if (!ok) break;
      }
    }
    __syncwarp();
  } else if (warp == C::kWarpProdB) {
    // ------------------------------------------------- token tile producer
    if (lane == 0) {
      Ring rb;
      for (int t = sch.lo + blockIdx.x;; t += gridDim.x) {
        Tile tl;
        if (!get_tile(sch, t, mtiles, mstep, tl)) break;
        constexpr int kBox = C::kBoxRows;
        const int nq = (tl.n + kBox - 1) / kBox;
        const int kpb = kb_per_stage<C>(tl.n);
        bool ok = true;
        for (int ks0 = 0; ks0 < nks; ks0 += kpb) {
          if (!mbar_wait_bounded(&b_empty[rb.i], rb.ph ^ 1u, c.status)) {
            ok = false;
            break;
          }
          const int nk = min(kpb, nks - ks0);
          uint8_t* bdst = smem + C::kOffB + rb.i * C::kBBytes;
          mbar_expect_tx(&b_full[rb.i], (uint32_t)(nk * nq * kBox * 128));
          for (int j = 0; j < nk; ++j)
            for (int q = 0; q < nq; ++q)
              tma_load_2d(bdst + (j * nq + q) * kBox * 128, &tmB, (ks0 + j) * kBK, tl.r0 + q * kBox, &b_full[rb.i]);
          rb.next(C::kStagesB);
        }
        if (!ok) break;
      }
    }
    __syncwarp();
  } else if (warp == C::kWarpMma || (C::kMmaWarps > 1 && warp == C::kWarpMma2)) {
    // ---------------------------------------------------------------- MMA
    const int mi = warp == C::kWarpMma ? 0 : 1;   // narrow: the A matrix this warp issues
    if (lane == 0) {
      Ring ra, rb, racc;
      bool ok = true;
      for (int t = sch.lo + blockIdx.x; ok; t += gridDim.x) {
        Tile tl;
        if (!get_tile(sch, t, mtiles, mstep, tl)) break;
        const int n16 = (tl.n + 15) & ~15;
        const uint32_t idesc = idesc_f16_f32(kMTile, n16);
        const int kpb = kb_per_stage<C>(tl.n);
        const uint32_t bsub = (uint32_t)(((tl.n + C::kBoxRows - 1) / C::kBoxRows) * C::kBoxRows * 128);
        if (!mbar_wait_bounded(&acc_empty[racc.i], racc.ph ^ 1u, c.status)) break;
        tc_fence_after();
        const uint32_t d0 = tmem + (uint32_t)(racc.i * 2 * C::kHalf);
        int kc = 0, j = 0;   // K chunk of the tile; K chunk inside the token stage
        for (int ks = 0; ks < nst && ok; ++ks) {
          if (!mbar_wait_bounded(&a_full[ra.i], ra.ph, c.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int h = 0; h < C::kCh; ++h, ++kc) {
            if (j == 0) {
              if (!mbar_wait_bounded(&b_full[rb.i], rb.ph, c.status)) {
                ok = false;
                break;
              }
              tc_fence_after();
            }
            const uint32_t b_base = smem_u32(smem + C::kOffB + rb.i * C::kBBytes) + (uint32_t)j * bsub;
            if constexpr (C::kTS) {
              // descriptors and TMEM addresses advance by constants within the
              // chunk (the descriptor's address field holds address / 16; no
              // carry: shared addresses stay below 2^18)
              const uint32_t a_t = tmem + (uint32_t)(C::kTmemA + ra.i * C::kTmemAStage + h * (kBK / 2));
              const uint64_t bd0 = sw128_desc(b_base);
              const uint32_t acc0 = kc != 0;
              const uint32_t dm = d0 + (uint32_t)(mi * C::kHalf), am = a_t + (uint32_t)(mi * C::kTmemAMat);
#pragma unroll
              for (int k16 = 0; k16 < kBK / 16; ++k16)
                umma_f16_ts(dm, am + (uint32_t)(k16 * 8), bd0 + (uint64_t)(k16 * 2), idesc, k16 == 0 ? acc0 : 1u);
            } else {
              const uint32_t a_base = smem_u32(smem + C::kOffA + ra.i * C::kABytes + mi * C::kAMat);
              const uint32_t dm = d0 + (uint32_t)(mi * C::kHalf);
#pragma unroll
              for (int k16 = 0; k16 < kBK / 16; ++k16)
                umma_f16_ss(dm, sw128_desc(a_base + k16 * 32), sw128_desc(b_base + k16 * 32), idesc, (kc | k16) != 0);
            }
            if (++j == kpb || kc == nks - 1) {   // the token stage's last K chunk
              umma_commit(&b_empty[rb.i]);
              rb.next(C::kStagesB);
              j = 0;
            }
          }
          if (!ok) break;
          umma_commit(&a_empty[ra.i]);
          ra.next(C::kStagesA);
        }
        if (!ok) break;
        umma_commit(&acc_full[racc.i]);
        racc.next(nacc);
      }
    }
    __syncwarp();
  } else if (warp >= C::kWarpDq) {
    // ------------------------------------------------------------ dequant
    const int g = lane >> 2, cq = lane & 3;
    const int dw = (warp - C::kWarpDq) % kDqWarps, grp = (warp - C::kWarpDq) / kDqWarps;   // 16-row tile, group
    int seq = 0;                                             // K steps of this CTA so far
    Ring rr, ra, racc;
    bool ok = true;
    Tile pend = {0, 0, 0, 0};   // gate/up: the tile whose epilogue share is still due
    bool have = false;
    // this warp's third of a gate/up tile's epilogue (dequant warps 0-3 the middle,
    // 4-7 the last third of the 32-column chunks)
    auto epilogue_share = [&]() -> bool {
      if (!mbar_wait_bounded(&acc_full[racc.i], racc.ph, c.status)) return false;
      tc_fence_after();
      const int nch = (pend.n + 31) / 32, part = 1 + (dw >> 2);
      epilogue_chunks(pend, part * nch / 3, (part + 1) * nch / 3, racc.i);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[racc.i]);
      racc.next(nacc);
      have = false;
      return true;
    };
    if (DENSE) {   // no dequantisation: the gate/up epilogue shares only
      for (int t = sch.lo + blockIdx.x;; t += gridDim.x) {
        if (!get_tile(sch, t, mtiles, mstep, pend) || !epilogue_share()) break;
      }
    }
    if constexpr (C::kTS) {
      // One row of one A matrix per thread, straight into tensor memory: warp
      // dw converts matrix dw / 4, rows 32 (warp % 4) + lane (its TMEM lane
      // quarter).  Row m of the 128-row matrix is row r = m % 16 of 16-row tile
      // m / 16; in a 512-byte int4 chunk its words sit in the 64 bytes of lane
      // group r % 8 (lanes 4 (r % 8) + c, c = 0..3), word j of lane c holding
      // K = 16c + 4j + {0, 1} in its bits 0-3 / 16-19 and K + {2, 3} in bits
      // 8-11 / 24-27 (rows 8-15 of the tile: the nibbles 4 bits higher).  The
      // FP16 pair of K = 2p, 2p + 1 goes to TMEM column p of the stage.
      const int mat = dw >> 2, qd = warp & 3;
      const int m = qd * 32 + lane, rt = m >> 4, r = m & 15;
      const uint32_t nshift = (uint32_t)(r >> 3) * 4u;
      const uint32_t trow = tmem + (uint32_t)(C::kTmemA + mat * C::kTmemAMat) + ((uint32_t)(qd * 32) << 16);
      for (int t = sch.lo + blockIdx.x; ok; t += gridDim.x) {
        Tile tl;
        if (!get_tile(sch, t, mtiles, mstep, tl)) break;
        for (int ks = 0; ks < nst; ++ks) {
          if ((seq++ % C::kDqGroups) != grp) {   // the other group's K step
            rr.next(C::kStagesRaw);
            ra.next(C::kStagesA);
            continue;
          }
          if (!mbar_wait_bounded(&raw_full[rr.i], rr.ph, c.status)) {
            ok = false;
            break;
          }
          const uint8_t* raw = smem + C::kOffRaw + rr.i * C::kRawBytes;
          const __half2 sc =
              __half2half2(reinterpret_cast<const __half*>(raw + C::kCh * C::kRawQ + mat * 256 + rt * 32)[r]);
          if (!mbar_wait_bounded(&a_empty[ra.i], ra.ph ^ 1u, c.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int h = 0; h < C::kCh; ++h) {
            const uint8_t* qp = raw + h * C::kRawQ + (mat * 8 + rt) * 512 + (r & 7) * 64;
            uint4 v[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) v[i] = *reinterpret_cast<const uint4*>(qp + 16 * i);
            uint32_t o[32];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const uint32_t wv[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const uint32_t w = wv[j] >> nshift;
                o[8 * i + 2 * j] = dequant_pair(w, sc);
                o[8 * i + 2 * j + 1] = dequant_pair(w >> 8, sc);
              }
            }
            tmem_st32(trow + (uint32_t)(ra.i * C::kTmemAStage + h * (kBK / 2)), o);
          }
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          // the int4 slot is released after its words were used (see below)
          if (lane == 0) {
            mbar_arrive(&a_full[ra.i]);
            mbar_arrive(&raw_empty[rr.i]);
          }
          rr.next(C::kStagesRaw);
          ra.next(C::kStagesA);
        }
      }
    }
    for (int t = sch.lo + blockIdx.x; ok && !DENSE && !C::kTS; t += gridDim.x) {
      Tile tl;
      if (!get_tile(sch, t, mtiles, mstep, tl)) break;
      // the scales of the thread's rows for the current block (read from the
      // raw stage that starts the block, or from every stage)
      __half2 slo[2][1], shi[2][1];
      for (int ks = 0; ks < nst; ++ks) {
        if (C::kDqGroups > 1 && (seq++ % C::kDqGroups) != grp) {   // the other group's K step
          rr.next(C::kStagesRaw);
          ra.next(C::kStagesA);
          continue;
        }
        // the previous tile's epilogue share first: the MMA waits for it
        // before it takes stage 0 of this tile
        if (C::kAcc == 1 && have && ks == 0 && !epilogue_share()) {
          ok = false;
          break;
        }
        if (!mbar_wait_bounded(&raw_full[rr.i], rr.ph, c.status)) {
          ok = false;
          break;
        }
        uint4 q[2][1];
        const uint8_t* raw = smem + C::kOffRaw + rr.i * C::kRawBytes;
        if (C::kScalesEveryStage || (ks & 3) == 0) {
#pragma unroll
          for (int m = 0; m < C::kMats; ++m) {
            const __half* sc = reinterpret_cast<const __half*>(raw + C::kRawQ + m * 256 + dw * 32);
            slo[m][0] = __half2half2(sc[g]);
            shi[m][0] = __half2half2(sc[g + 8]);
          }
        }
#pragma unroll
        for (int m = 0; m < C::kMats; ++m) q[m][0] = *reinterpret_cast<const uint4*>(raw + (m * 8 + dw) * 512 + lane * 16);
        if (!mbar_wait_bounded(&a_empty[ra.i], ra.ph ^ 1u, c.status)) {
          ok = false;
          break;
        }
        const uint32_t abase = smem_u32(smem + C::kOffA + ra.i * C::kABytes);
#pragma unroll
        for (int m = 0; m < C::kMats; ++m) {
#pragma unroll
          for (int tt = 0; tt < 1; ++tt) {
            const int row = dw * 16 + g;   // and row + 8 (same swizzle phase)
            const uint32_t rlo = abase + m * C::kAMat + row * 128;
            const uint32_t rhi = rlo + 8 * 128;
            const uint32_t sw = (uint32_t)(row & 7);
            const uint32_t w4[4] = {q[m][tt].x, q[m][tt].y, q[m][tt].z, q[m][tt].w};
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              // K values cq*16 + 8h .. + 7 of the chunk fill the 16-byte swizzle
              // unit 2 cq + h of rows g and g + 8 (words 2h, 2h + 1: 4 K each).
              // One 16-byte store per row: each 8-lane phase then covers the 8
              // units of its rows once (no bank conflicts).
              uint32_t a0[4], a1[4];
              dequant_word(w4[2 * h], slo[m][tt], shi[m][tt], a0);
              dequant_word(w4[2 * h + 1], slo[m][tt], shi[m][tt], a1);
              const uint32_t cu = ((uint32_t)(2 * cq + h) ^ sw) << 4;
              st_shared_v4_b32(rlo + cu, a0[0], a0[2], a1[0], a1[2]);
              st_shared_v4_b32(rhi + cu, a0[1], a0[3], a1[1], a1[3]);
            }
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        // The raw slot is released only now, after its words were consumed by
        // the arithmetic above: an arrive issued right behind the shared loads
        // let the next TMA fill overtake loads still queued behind the tensor
        // core's shared-memory traffic (seen as a few corrupt weight rows in
        // about one forward in twenty-five of the MMA-bound down projection).
        if (lane == 0) {
          mbar_arrive(&a_full[ra.i]);
          mbar_arrive(&raw_empty[rr.i]);
        }
        rr.next(C::kStagesRaw);
        ra.next(C::kStagesA);
      }
      if (ok && C::kAcc == 1) {
        pend = tl;
        have = true;
      }
    }
    if (!DENSE && ok && have) epilogue_share();   // the last tile
  } else {
    // ----------------------------------------------------------- epilogue
    // warps 3..6 -> TMEM lane quarters 3, 0, 1, 2
    Ring racc;
    for (int t = sch.lo + blockIdx.x;; t += gridDim.x) {
      Tile tl;
      if (!get_tile(sch, t, mtiles, mstep, tl)) break;
      if (!mbar_wait_bounded(&acc_full[racc.i], racc.ph, c.status)) break;
      tc_fence_after();
      const int nch = (tl.n + 31) / 32;
      epilogue_chunks(tl, 0, C::kAcc == 1 ? nch / 3 : nch, racc.i);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[racc.i]);
      racc.next(nacc);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == C::kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// out[t] = (x[t]) + sum_j w[t,j] y[t*k+j] in rank order j, FP32, then FP16.
// A CTA covers 512 hidden values of one token (8 per thread, 16-byte loads
// of the FP16 y rows: small CTAs, so that a few tokens still spread over
// the SMs); the token's weights (0 for an absent expert) are read once into
// shared memory so that the y loads of all ranks are independent.
constexpr int kCombineThreads = 64;
__global__ void __launch_bounds__(kCombineThreads) combine_kernel(FwdCtx c) {
  __shared__ float ws[32];
  pdl_wait();
  pdl_trigger();
  const int H = c.H, k = c.k;
  const int blocks_per_tok = (H / 8 + kCombineThreads - 1) / kCombineThreads;
  const int t = blockIdx.x / blocks_per_tok;
  const int v = (blockIdx.x % blocks_per_tok) * kCombineThreads + threadIdx.x;   // 8-value vector inside the row
  if (threadIdx.x < k) {
    const int p = t * k + threadIdx.x;
    ws[threadIdx.x] = c.table[c.ids[p]] >= 0 ? c.topw[p] : 0.f;
  }
  __syncthreads();
  if (v >= H / 8) return;
  float acc[8];
  if (c.flags & 1u) {
    const uint4 xv = *reinterpret_cast<const uint4*>(c.x + (size_t)t * H + v * 8);
    const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&xw[i]));
      acc[2 * i] = f.x;
      acc[2 * i + 1] = f.y;
    }
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.f;
  }
  const __half* yh = reinterpret_cast<const __half*>(c.ybuf);   // [pair][H] FP16
  for (int j0 = 0; j0 < k; j0 += 8) {
    uint4 y[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int j = j0 + u;
      y[u] = (j < k && ws[j] != 0.f) ? __ldcs(reinterpret_cast<const uint4*>(yh + ((size_t)t * k + j) * H) + v)
                                     : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int j = j0 + u;
      if (j < k && ws[j] != 0.f) {
        const float w = ws[j];
        const uint32_t yw[4] = {y[u].x, y[u].y, y[u].z, y[u].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&yw[i]));
          acc[2 * i] = fmaf(w, f.x, acc[2 * i]);
          acc[2 * i + 1] = fmaf(w, f.y, acc[2 * i + 1]);
        }
      }
    }
  }
  uint4 o;
  uint32_t* ow = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __half2 h2 = __floats2half2_rn(acc[2 * i], acc[2 * i + 1]);
    ow[i] = *reinterpret_cast<const uint32_t*>(&h2);
  }
  *reinterpret_cast<uint4*>(c.out + (size_t)t * H + v * 8) = o;
}

// xp[r] = x[sorted[r] / k]: activations in sorted-row order.  A CTA copies 8
// rows; each thread keeps its 16-byte loads of all 8 rows in flight at once.
constexpr int kGatherRows = 8;
__global__ void __launch_bounds__(256) gather_rows_kernel(FwdCtx c) {
  pdl_wait();
  pdl_trigger();
  const int P = c.T * c.k, vpr = c.H / 8;
  const int r0 = blockIdx.x * kGatherRows;
  for (int v = threadIdx.x; v < vpr; v += blockDim.x) {
    uint4 val[kGatherRows];
#pragma unroll
    for (int i = 0; i < kGatherRows; ++i) {
      const int r = r0 + i;
      if (r < P) val[i] = __ldg(reinterpret_cast<const uint4*>(c.x + (size_t)(c.sorted[r] / c.k) * c.H) + v);
    }
#pragma unroll
    for (int i = 0; i < kGatherRows; ++i) {
      const int r = r0 + i;
      if (r < P) reinterpret_cast<uint4*>(c.xp + (size_t)r * c.H)[v] = val[i];
    }
  }
}

// ------------------------------------------------------------ tensor maps
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    // the entry point as introduced in CUDA 12.0 (its signature since then)
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
    else
      cudaGetLastError();
  }
  return fn;
}

// Row-major FP16 matrix [rows][cols] (cols contiguous), box of box_rows x 64
// columns, 128-byte swizzle, zero fill out of range.
bool make_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {64, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool gemm_shapes_supported(int H, int I) { return H % (2 * kMTile) == 0 && I % kMTile == 0; }

PoolMaps make_pool_maps(const uint8_t* pool, const SlotLayout& lay, int num_slots) {
  PoolMaps pm;
  memset(&pm, 0, sizeof pm);
  pm.ok = false;
  EncodeTiledFn fn = encode_fn();
  if (!fn || !gemm_shapes_supported((int)lay.down.rows, (int)lay.gate.rows)) return pm;
  const MatLayout* mats[3] = {&lay.gate, &lay.up, &lay.down};
  for (int i = 0; i < 3; ++i) {
    const MatLayout& L = *mats[i];
    // [slot][row tile][K chunk][128 x u32 = 512 B], packed int4 part of each tile
    const cuuint64_t dims[4] = {128, L.k / 64, L.rows / 16, (cuuint64_t)num_slots};
    const cuuint64_t strides[3] = {512, L.tile_bytes, lay.bytes};
    const cuuint32_t box[4] = {128, 1, 8, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    if (fn(&pm.q[i], CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, const_cast<uint8_t*>(pool + L.off + L.scale_bytes), dims,
           strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return pm;
    // [slot][row tile][block][16 FP16 scales], the 16 scales of block b of 8 row tiles per load
    const cuuint64_t sdims[4] = {16, L.nb, L.rows / 16, (cuuint64_t)num_slots};
    const cuuint64_t sstrides[3] = {32, L.tile_bytes, lay.bytes};
    const cuuint32_t sbox[4] = {16, 1, 8, 1};
    if (fn(&pm.sc[i], CU_TENSOR_MAP_DATA_TYPE_UINT16, 4, const_cast<uint8_t*>(pool + L.off), sdims, sstrides, sbox,
           estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return pm;
  }
  pm.ok = true;
  return pm;
}

int gemm_tile_tokens(int T, int k, int E) {
  const long long P = (long long)T * k;
  return P <= 16ll * E ? 32 : P <= 64ll * E ? 128 : 256;
}

// gate/up and down grouped GEMMs of one token-tile variant (c.tile_tokens
// must equal NMAX: the routing kernels chunked the experts' rows with it)
template <int NMAX>
cudaError_t launch_gemm_pair(const FwdCtx& c, const PoolMaps& pm, cudaStream_t st, const StageEvents& se) {
  using CG = Cfg<true, NMAX>;
  using CD = Cfg<false, NMAX>;
  const uint64_t P = (uint64_t)c.T * c.k;
  CUtensorMap mx, mh;
  if (!make_map(&mx, c.xp, P, (uint64_t)c.H, CG::kBoxRows) || !make_map(&mh, c.hbuf, P, (uint64_t)c.I, CD::kBoxRows))
    return cudaErrorNotSupported;
  cudaError_t e = opt_in_smem((const void*)grouped_gemm_kernel<true, false, NMAX>, CG::kSmem);
  if (e == cudaSuccess) e = opt_in_smem((const void*)grouped_gemm_kernel<false, false, NMAX>, CD::kSmem);
  if (e != cudaSuccess) return e;
  const int grid = c.num_sms > 0 ? c.num_sms : 148;
  e = launch_pdl(grouped_gemm_kernel<true, false, NMAX>, dim3(grid), dim3(CG::kThreads), CG::kSmem, st, 1, c, mx, pm.q[0],
                 pm.q[1], pm.sc[0], pm.sc[1]);
  if (e == cudaSuccess) e = record_stage(se, 2, st);
  if (e == cudaSuccess)
    e = launch_pdl(grouped_gemm_kernel<false, false, NMAX>, dim3(grid), dim3(CD::kThreads), CD::kSmem, st, 1, c, mh,
                   pm.q[2], pm.q[2], pm.sc[2], pm.sc[2]);
  return e;
}

cudaError_t launch_gemm_experts(const FwdCtx& c, const PoolMaps& pm, bool gathered, cudaStream_t st,
                                const StageEvents& se) {
  if (!gemm_shapes_supported(c.H, c.I) || !pm.ok) return cudaErrorNotSupported;
  if (c.tile_tokens != 32 && c.tile_tokens != 128 && c.tile_tokens != 256) return cudaErrorInvalidValue;
  const uint64_t P = (uint64_t)c.T * c.k;
  cudaError_t e = cudaSuccess;
  if (!gathered)
    e = launch_pdl(gather_rows_kernel, dim3((unsigned)((P + kGatherRows - 1) / kGatherRows)), dim3(256), 0, st, 1, c);
  if (e == cudaSuccess) e = record_stage(se, 1, st);
  if (e == cudaSuccess)
    e = c.tile_tokens == 32    ? launch_gemm_pair<32>(c, pm, st, se)
        : c.tile_tokens == 128 ? launch_gemm_pair<128>(c, pm, st, se)
                               : launch_gemm_pair<256>(c, pm, st, se);
  if (e == cudaSuccess) e = record_stage(se, 3, st);
  if (e == cudaSuccess)
    e = launch_pdl(combine_kernel, dim3((unsigned)(c.T * ((c.H / 8 + kCombineThreads - 1) / kCombineThreads))),
                   dim3(kCombineThreads), 0, st, 1, c);
  if (e == cudaSuccess) e = record_stage(se, 4, st);
  return e;
}

DenseMaps make_dense_maps(const __half* xpool, int H, int I, int xslots) {
  DenseMaps dm;
  memset(&dm, 0, sizeof dm);
  dm.ok = false;
  EncodeTiledFn fn = encode_fn();
  if (!fn || !xpool || xslots < 1 || !gemm_shapes_supported(H, I)) return dm;
  const uint64_t slot_bytes = (uint64_t)3 * I * H * 2;
  // gate and up: [slot][I][H]; down: [slot][H][I]; 128 rows x 64 K per box, 128-byte swizzle
  const uint64_t off[3] = {0, (uint64_t)I * H, (uint64_t)2 * I * H};
  const uint64_t rows[3] = {(uint64_t)I, (uint64_t)I, (uint64_t)H}, ks[3] = {(uint64_t)H, (uint64_t)H, (uint64_t)I};
  for (int m = 0; m < 3; ++m) {
    const cuuint64_t dims[3] = {ks[m], rows[m], (cuuint64_t)xslots};
    const cuuint64_t strides[2] = {ks[m] * 2, slot_bytes};
    const cuuint32_t box[3] = {64, (cuuint32_t)kMTile, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    if (fn(&dm.a[m], CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<__half*>(xpool + off[m]), dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return dm;
  }
  dm.ok = true;
  return dm;
}

// The offload-qpacked comparison: the routed x rows gathered once, then per
// batch of at most xslots active experts an expansion into the FP16 execution
// slots and the dense gate/up and down grouped GEMMs, then the combine.  The
// number of batches is bounded by max_active on the host; a batch past the
// active experts exits on the device.
cudaError_t launch_offload_experts(const FwdCtx& c0, const DenseMaps& dm, bool gathered, cudaStream_t st,
                                   const StageEvents& se) {
  if (!gemm_shapes_supported(c0.H, c0.I) || !dm.ok || c0.xslots < 1) return cudaErrorNotSupported;
  const uint64_t P = (uint64_t)c0.T * c0.k;
  CUtensorMap mx, mh;
  if (!make_map(&mx, c0.xp, P, (uint64_t)c0.H, 64) || !make_map(&mh, c0.hbuf, P, (uint64_t)c0.I, 64))
    return cudaErrorNotSupported;
  using CG = Cfg<true, 256>;
  using CD = Cfg<false, 256>;
  if (c0.tile_tokens != 256) return cudaErrorInvalidValue;
  cudaError_t e = opt_in_smem((const void*)grouped_gemm_kernel<true, true, 256>, CG::kSmem);
  if (e == cudaSuccess) e = opt_in_smem((const void*)grouped_gemm_kernel<false, true, 256>, CD::kSmem);
  if (e != cudaSuccess) return e;
  const int grid = c0.num_sms > 0 ? c0.num_sms : 148;
  if (!gathered)
    e = launch_pdl(gather_rows_kernel, dim3((unsigned)((P + kGatherRows - 1) / kGatherRows)), dim3(256), 0, st, 1, c0);
  if (e == cudaSuccess) e = record_stage(se, 1, st);
  const int nb = (c0.max_active + c0.xslots - 1) / c0.xslots;
  for (int b = 0; b < nb && e == cudaSuccess; ++b) {
    FwdCtx c = c0;
    c.ub0 = b * c0.xslots;
    c.ub1 = c.ub0 + c0.xslots < c0.max_active ? c.ub0 + c0.xslots : c0.max_active;
    e = launch_expand(c, st);
    if (e == cudaSuccess)
      e = launch_pdl(grouped_gemm_kernel<true, true, 256>, dim3(grid), dim3(CG::kThreads), CG::kSmem, st, 1, c, mx,
                     dm.a[0], dm.a[1], dm.a[0], dm.a[1]);
    if (e == cudaSuccess)
      e = launch_pdl(grouped_gemm_kernel<false, true, 256>, dim3(grid), dim3(CD::kThreads), CD::kSmem, st, 1, c, mh,
                     dm.a[2], dm.a[2], dm.a[2], dm.a[2]);
  }
  if (e == cudaSuccess) e = record_stage(se, 2, st);
  if (e == cudaSuccess) e = record_stage(se, 3, st);
  if (e == cudaSuccess)
    e = launch_pdl(combine_kernel, dim3((unsigned)(c0.T * ((c0.H / 8 + kCombineThreads - 1) / kCombineThreads))),
                   dim3(kCombineThreads), 0, st, 1, c0);
  if (e == cudaSuccess) e = record_stage(se, 4, st);
  return e;
}
