// Fused decode-regime layer: one cooperative persistent launch per forward
// (router -> top-k -> permutation -> gate/up -> SiLU*up -> down -> combine),
// in the spirit of a fused small-batch executor ("top4-fused-v1" is named on
// "Horizon RunMap - architecture", "Regimes and executor boundaries"; its
// design is not published).
//
// Grid = one CTA per SM, all co-resident (cooperative launch).  A CTA has 12
// compute warps in NG groups of GW (6 x 2 for one token routed to >= 8
// experts, 3 x 4 for T <= 8, 2 x 6 above), one producer warp and one signaller
// warp.
//   routing  the grid's warps take the (token, expert, K half) dot products
//            of the router (and per-token sums of squares for PRENORM) ->
//            global; one bounded grid barrier; then every CTA reads the logits
//            and does softmax / top-k, the expert counts and the stable
//            permutation in shared memory (CTA 0 publishes them).
//   weights  each CTA owns a list of units (CtaUnits): gate/up items
//            (expert, 16-row tile of I) and down items (expert, 32 or 64 rows
//            of H), either a contiguous share of each kind (phase order) or
//            every G-th unit of one grid-wide order in which an expert's down
//            items trail its gate/up items by a fixed lag (interleaved
//            order).  The producer warp streams a CTA's units as a ring of
//            equal entries (a gate tile, an up tile, or the two row tiles of
//            a 32-row down block) with 1-D bulk copies, starting as soon as
//            the active experts are known; each consumer warp releases an
//            entry once it has read it.
//   gate/up  group q takes the CTA's units q, q + NG, ...: gate entry, then
//            up entry, K split over the group's warps, all (<= 16) tokens of
//            the expert at once from the x rows staged in shared memory; h = SiLU(g) * u
//            -> global (FP16); the group leader then leaves a note for the
//            signaller.
//   down     once every gate/up item of its expert has counted (a bounded
//            wait on that counter, usually already met thanks to the lag: no
//            grid-wide barrier), the group stages the expert's h rows and
//            multiplies its two row tiles -> y (FP32).
//   signal   the signaller warp turns batches of gate/up notes into GPU-wide
//            readiness counts behind one fence per batch, so no compute warp
//            waits on a fence or an atomic.
//   combine  a second bounded grid barrier; then the grid gathers
//            out[t] = (x[t]) + sum_j w[t, j] y[t k + j] in rank order j.
// Weights stay 4-bit until a warp dequantises a 16-byte chunk in registers
// for one MMA step (FP16 operands, FP32 accumulation).  Every wait is
// bounded: on a timeout the status word records it, the CTA stops waiting
// (its remaining arithmetic runs on whatever shared memory holds, and the
// status marks the forward void), and the producer lets its copies land
// before the CTA exits.
#include <atomic>

#include "gemv_dev.cuh"
#include "route_dev.cuh"

namespace {
using namespace gemv_dev;
using namespace route_dev;

constexpr int kCW = 12;                        // compute warps
constexpr int kNW = kCW + 2;                   // + producer warp + signaller warp
constexpr int kFThreads = kNW * 32;
constexpr int kMB = 16;                        // notes per group mailbox
constexpr int kDownRows = 32;                  // rows of H per down entry (2 row tiles)
constexpr int kMaxT = 16;                      // tokens of the fused path (all staged in smem)
constexpr int kMaxP = kMaxT * 32;
constexpr int kMaxSlots = 16;                  // ring entries
constexpr int kMinSlots = 4;
constexpr int kInFlight = 4;                   // ring entries in flight at once (bandwidth x latency per SM)
constexpr int kMaxExperts = 256;               // readiness counters per handle
constexpr uint32_t kSmemBudget = 226 * 1024;

// warps per compute group for a batch of T tokens
// (measured: 2-warp groups, the most items in flight, help only one token
// routed to 8 or more experts; otherwise fewer and wider groups spend less on
// the cross-warp reductions)
__host__ __device__ inline int fused_group_warps(int T, int k) { return T == 1 && k >= 8 ? 2 : T <= 8 ? 4 : 6; }

// The interleaved unit order (CtaUnits) for 4-warp groups when a gate/up item
// (16 H int4 values) and a 64-row down item (64 I) move about the same bytes
// (within 1/8): groups then take equal shares by count.  Measured on the
// OLMoE shape (H = 2 I): T = 4 35.1 against 38.0 us per layer in the phase
// order, T = 2 27.1 against 29.6; with 2- or 6-warp groups the phase order
// was faster (T = 1, 16), as it was on the Qwen shape (H = 2048, I = 1408),
// whose down items are larger.
inline int fused_interleaved(int H, int I, int gw) {
  const long long gu = 16ll * H, dn = 32ll * I, d = gu > dn ? gu - dn : dn - gu;
  return gw == 4 && 8 * d <= gu;
}

// The grid's unit order.  A unit is a gate/up item (expert, 16-row tile of I:
// a gate entry and an up entry) or a down item (expert, 64-row block of H:
// two entries of 2 row tiles); both move about the same bytes.  The units
// form blocks j = 0 .. U + L - 1: block j holds the down items of active
// expert j - L (when 0 <= j - L < U), then the gate/up items of active expert
// j (when j < U).  Unit x belongs to CTA x % G, whose groups take its units
// in turn, so the grid works through the order front to back: one expert's
// gate/up items run side by side in different CTAs, and its down items come
// L blocks later, when they are usually ready.  No grid-wide phase separates
// gate/up from down, and the weight stream does not pause between them.
// Every unit depends
// only on units earlier in the order, each CTA holds its units in that order
// and each group takes them in it, so the first unfinished unit of the grid
// can always proceed: no deadlock.
// L: the gate/up items of L - 1 experts (t1 each) span kLagQ quarters of one
// step of the grid's groups (G x NG units), so every expert's gate/up items
// have finished, and been counted, about that long before its first down item
// starts (the groups start together, so this covers the first experts too).
constexpr int kLagQ = 10;
struct UnitOrder {
  int U, L, t1, t2;
};
struct Unit {
  int down, u, idx;
};
__host__ __device__ inline UnitOrder unit_order(int U, int t1, int t2, int G, int NG) {
  return UnitOrder{U, 1 + (kLagQ * G * NG + 4 * t1 - 1) / (4 * t1), t1, t2};
}
__host__ __device__ inline Unit unit_at(const UnitOrder& o, int x) {
  const int r1 = (o.L < o.U ? o.L : o.U) * o.t1;   // blocks before L: gate/up items only
  if (x < r1) return Unit{0, x / o.t1, x % o.t1};
  x -= r1;
  const int nmix = o.U > o.L ? o.U - o.L : 0, bs = o.t1 + o.t2;
  if (x < nmix * bs) {
    const int jj = x / bs, r = x - jj * bs;
    return r < o.t2 ? Unit{1, jj, r} : Unit{0, o.L + jj, r - o.t2};
  }
  x -= nmix * bs;   // blocks from max(U, L): down items only
  return Unit{1, nmix + x / o.t2, x % o.t2};
}

// The units of CTA b, in the order its producer streams them and its groups
// (group q: units q, q + NG, ...) take them.  Two orders:
//   interleaved  x = b + j G of the unit order above; down items of 64 rows
//                of H (two entries), so both kinds move about the same bytes
//                when 16 H ~ 32 I;
//   phases       a contiguous share of the gate/up items, then a contiguous
//                share of the down items (32 rows of H: one entry); every
//                CTA reaches its down items about when the whole grid's
//                gate/up items finish, but a group's consecutive down items
//                mostly share an expert, whose h rows it stages once.
template <bool INTER>
struct CtaUnits {
  static constexpr bool inter = INTER;
  UnitOrder ord;
  int NU, b, G;                 // interleaved
  int a1, m1, a2, m2, t1, t2;   // phases (t2: 32-row down items per expert)
  DEV_INLINE int count() const { return inter ? (NU > b ? (NU - b + G - 1) / G : 0) : m1 + m2; }
  DEV_INLINE Unit at(int j) const {
    if (inter) return unit_at(ord, b + j * G);
    if (j < m1) return Unit{0, (a1 + j) / t1, (a1 + j) % t1};
    return Unit{1, (a2 + j - m1) / t2, (a2 + j - m1) % t2};
  }
  DEV_INLINE int first_entry(int j) const { return inter || j < m1 ? 2 * j : 2 * m1 + (j - m1); }
  DEV_INLINE int down_entries() const { return inter ? 2 : 1; }
  DEV_INLINE int down_block(const Unit& un, int sub) const { return inter ? 2 * un.idx + sub : un.idx; }   // 32-row block of H
};
template <bool INTER>
DEV_INLINE CtaUnits<INTER> cta_units(int U, int I, int H, int b, int G, int NG) {
  CtaUnits<INTER> cu;
  cu.b = b;
  cu.G = G;
  cu.t1 = I / 16;
  cu.t2 = H / kDownRows;
  cu.ord = unit_order(U, cu.t1, H / (2 * kDownRows), G, NG);
  cu.NU = U * (cu.t1 + H / (2 * kDownRows));
  const int n1 = U * cu.t1, n2 = U * cu.t2;
  cu.a1 = (int)((long long)b * n1 / G);
  cu.m1 = (int)((long long)(b + 1) * n1 / G) - cu.a1;
  cu.a2 = (int)((long long)b * n2 / G);
  cu.m2 = (int)((long long)(b + 1) * n2 / G) - cu.a2;
  return cu;
}

struct FusedSmem {
  uint32_t ns, slot_bytes, off_x, off_h, off_red, off_sb, off_route, total;
};

// Shared memory of the fused kernel for T tokens, top-k: the ring (as many
// entries as fit, at most kMaxSlots), the x rows [T][H + 8], per-group h rows
// [min(T, 8)][I + 8], the cross-warp reduction buffer and the routing state.
__host__ __device__ inline FusedSmem fused_smem(const SlotLayout& lay, int H, int I, int E, int T, int k, int gw) {
  const int NG = kCW / gw;
  FusedSmem f;
  const uint32_t sg = lay.gate.tile_bytes, sd = 2 * lay.down.tile_bytes;
  f.slot_bytes = ((sg > sd ? sg : sd) + 127) / 128 * 128;
  const int hrows = T < kTok ? T : kTok;
  const int ntok = T <= 8 ? 8 : 16;
  const uint32_t xa = ((uint32_t)T * (H + 8) * 2 + 127) / 128 * 128;
  const uint32_t ha = ((uint32_t)NG * hrows * (I + 8) * 2 + 127) / 128 * 128;
  const uint32_t red = (uint32_t)kCW * 2 * 16 * ntok * 4;
  // per-chunk prefix sums: x rows [T][H/64 + 1], per-group h rows [min(T, 8)][I/64 + 1]
  const uint32_t sbb = ((uint32_t)(T * (H / 64 + 1) + NG * hrows * (I / 64 + 1)) * 4 + 127) / 128 * 128;
  const int P = T * k;
  // logits [T][E] | ids, topw, sorted [P] | rnorm [T] | table, cnt, off [E + 1]
  // | active slot, start, count [E + 1] | chunk counts [ceil(P/32)][E] | misc
  const uint32_t route = (uint32_t)(T * E + 3 * P + T + 6 * (E + 1) + ((P + 31) / 32) * E + 8) * 4;
  const uint32_t rest = xa + ha + red + sbb + route;
  const uint32_t ns = rest < kSmemBudget ? (kSmemBudget - rest) / f.slot_bytes : 0u;
  f.ns = ns > (uint32_t)kMaxSlots ? (uint32_t)kMaxSlots : ns;
  f.off_x = f.ns * f.slot_bytes;
  f.off_h = f.off_x + xa;
  f.off_red = f.off_h + ha;
  f.off_sb = f.off_red + red;
  f.off_route = f.off_sb + sbb;
  f.total = f.off_route + route;
  return f;
}

DEV_INLINE unsigned long long ld_acquire_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

DEV_INLINE unsigned ld_acquire_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Bounded barrier over all CTAs of the grid, called by one thread per CTA:
// one arrival on a monotonic 64-bit counter, then a poll until it reaches the
// next multiple of the grid size (every launch leaves it at a multiple).
// Split into an arrival and a wait, so that a CTA can do local work between.
DEV_INLINE unsigned long long grid_arrive(unsigned long long* ctr, unsigned nblocks) {
  __threadfence();
  const unsigned long long old = atomicAdd(ctr, 1ull);
  return (old / nblocks + 1ull) * nblocks;
}

DEV_INLINE bool grid_wait(const unsigned long long* ctr, unsigned long long target, DevStatus* st) {
  const long long t0 = clock64();
  while (ld_acquire_u64(ctr) < target) {
    if (clock64() - t0 > MOE_WAIT_CYCLES) {
      atomicOr(&st->flags, STATUS_TIMEOUT);
      return false;
    }
    __nanosleep(32);
  }
  return true;
}

DEV_INLINE bool grid_barrier(unsigned long long* ctr, unsigned nblocks, DevStatus* st) {
  __threadfence();
  const unsigned long long old = atomicAdd(ctr, 1ull);
  const unsigned long long target = (old / nblocks + 1ull) * nblocks;
  const long long t0 = clock64();
  while (ld_acquire_u64(ctr) < target) {
    if (clock64() - t0 > MOE_WAIT_CYCLES) {
      atomicOr(&st->flags, STATUS_TIMEOUT);
      return false;
    }
    __nanosleep(32);
  }
  return true;
}

// Bounded wait on an mbarrier phase that also gives up as soon as the CTA's
// abort flag is set (by another wait that ran out); sets it on a timeout.
DEV_INLINE bool wait_phase(uint64_t* bar, uint32_t par, volatile int* abort, DevStatus* st) {
  if (mbar_try_wait(bar, par)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, par)) {
    if (*abort) return false;
    if (clock64() - t0 > MOE_WAIT_CYCLES) {
      atomicOr(&st->flags, STATUS_TIMEOUT);
      *abort = 1;
      return false;
    }
  }
  return true;
}

// Bounded poll until *ctr >= target (acquire), abort-aware like wait_phase.
DEV_INLINE bool wait_count(const unsigned* ctr, unsigned target, volatile int* abort, DevStatus* st) {
  if (ld_acquire_u32(ctr) >= target) return true;
  const long long t0 = clock64();
  while (ld_acquire_u32(ctr) < target) {
    if (*abort) return false;
    if (clock64() - t0 > MOE_WAIT_CYCLES) {
      atomicOr(&st->flags, STATUS_TIMEOUT);
      *abort = 1;
      return false;
    }
    __nanosleep(64);
  }
  return true;
}

// Bounded wait until ring slot e % NS holds entry e (seq, written by the
// producer once the slot is free for it) and the entry's bytes have landed.
// Checking the entry first keeps a consumer that runs ahead from waiting on
// a phase parity that an older, still pending phase of the slot aliases.
// Lane 0 waits (with back-off, so waiting warps leave the issue slots to the
// computing ones); __syncwarp then orders the other lanes' reads after it.
DEV_INLINE void warp_wait_entry(volatile int* seq, uint64_t* full, int e, int NS, volatile int* abort,
                                DevStatus* st, int lane) {
  if (lane == 0) {
    const int s = e % NS;
    bool ok = true;
    if (seq[s] != e) {
      const long long t0 = clock64();
      while (seq[s] != e) {
        if (*abort) {
          ok = false;
          break;
        }
        if (clock64() - t0 > MOE_WAIT_CYCLES) {
          atomicOr(&st->flags, STATUS_TIMEOUT);
          *abort = 1;
          ok = false;
          break;
        }
        __nanosleep(40);
      }
    }
    if (ok) wait_phase(&full[s], (uint32_t)((e / NS) & 1), abort, st);
  }
  __syncwarp();
}

DEV_INLINE void named_sync(int id, int nthreads) { asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory"); }

DEV_INLINE void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
DEV_INLINE void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Partial dot(x_t, w_e) over K in [k0, k1) (one warp, every load in flight
// together: at most 1024 wide).
DEV_INLINE float warp_dot_part(const __half* xt, const __half* we, int k0, int k1, int lane) {
  uint4 xv[4], wv[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int kk = k0 + i * 256 + lane * 8;
    if (kk < k1) {
      xv[i] = __ldg(reinterpret_cast<const uint4*>(xt + kk));
      wv[i] = __ldg(reinterpret_cast<const uint4*>(we + kk));
    }
  }
  float acc = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i)
    if (k0 + i * 256 + lane * 8 < k1) acc += dot8(xv[i], wv[i]);
  return warp_sum(acc);
}

// MMA of one 64-wide K chunk (four 16x8x16 steps) of a 16-row tile against
// NT n-tiles of 8 tokens, into c[nt] (which the caller zeroes per block).
// The int4 nibbles enter the MMA as FP16 bit patterns with no arithmetic:
//   row g     : 1024 + u          (u = q + 8 of row g)
//   row g + 8 : 1024 + u + 16 u'  (u' = q + 8 of row g + 8, the row-g nibble
//                                  of the same K left in place)
// block_epilogue() recovers the exact sum over K of q * b per row in FP32.
template <int NT>
DEV_INLINE void mma_chunk(float (&c)[NT][4], const uint4& q, const uint4 (&bl)[NT], const uint4 (&bh)[NT]) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t w = j == 0 ? q.x : j == 1 ? q.y : j == 2 ? q.z : q.w;
    uint32_t a[4];
    a[1] = __byte_perm(w, 0x64646464u, 0x7250);   // bytes 0, 2 under exponent 0x64
    a[3] = __byte_perm(w, 0x64646464u, 0x7351);   // bytes 1, 3
    a[0] = a[1] & 0xFF0FFF0Fu;
    a[2] = a[3] & 0xFF0FFF0Fu;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const uint4& bv = j < 2 ? bl[nt] : bh[nt];
      mma_16816(c[nt], a, (j & 1) ? bv.z : bv.x, (j & 1) ? bv.w : bv.y);
    }
  }
}

// For the chunks [k0, k1) of one 256-wide scale block: with c0..c3 the MMA
// sums and S the sum of b over those chunks for the column,
//   row g     : sum q b = c0 - 1032 S          (1024 + u = 1032 + q)
//   row g + 8 : sum q b = (c2 - c0 - 128 S) / 16
// times the row's block scale, accumulated in FP32 (q * s exact).
// pre[nt][h]: prefix sums over chunks of the B column (2 cc + h of n-tile nt).
template <int NT, int NC>
DEV_INLINE void block_epilogue(float (&acc)[2][4], const float (&c)[NC][NT][4], float sg, float sg8,
                               const float* const (&pre)[2][2], int k0, int k1) {
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const float s0 = pre[nt][0][k1] - pre[nt][0][k0], s1 = pre[nt][1][k1] - pre[nt][1][k0];
    float v0 = c[0][nt][0], v1 = c[0][nt][1], v2 = c[0][nt][2], v3 = c[0][nt][3];
#pragma unroll
    for (int i = 1; i < NC; ++i) {
      v0 += c[i][nt][0];
      v1 += c[i][nt][1];
      v2 += c[i][nt][2];
      v3 += c[i][nt][3];
    }
    acc[nt][0] = fmaf(sg, fmaf(-1032.f, s0, v0), acc[nt][0]);
    acc[nt][1] = fmaf(sg, fmaf(-1032.f, s1, v1), acc[nt][1]);
    acc[nt][2] = fmaf(sg8, fmaf(-128.f, s0, v2 - v0), acc[nt][2]);
    acc[nt][3] = fmaf(sg8, fmaf(-128.f, s1, v3 - v1), acc[nt][3]);
  }
}

// acc[nt] += tile (16 x K) x B over the warp's contiguous K chunks [c0, c1).
// brow[nt]: the lane's B row (token nt * 8 + lane / 4; any valid row for
// columns past the tokens) in shared memory, K contiguous; pre: see above.
// Generic: any range (the block epilogue runs at block ends and at c1).
template <int NT>
DEV_INLINE void mma_fold(float (&acc)[2][4], const uint8_t* tile, uint32_t scale_bytes,
                         const __half* const (&brow)[2], const float* const (&pre)[2][2], int lane, int c0, int c1) {
  const int g = lane >> 2, cc = lane & 3;
  const uint8_t* qp = tile + scale_bytes + lane * 16;
  const __half* scp = reinterpret_cast<const __half*>(tile) + g;
  int kc = c0;
  while (kc < c1) {
    const int bend = ((kc >> 2) + 1) * 4;
    const int e = bend < c1 ? bend : c1;
    float c[2][NT][4];   // two accumulator chains (even / odd chunks of the block)
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int r = 0; r < 4; ++r) c[i][nt][r] = 0.f;
    for (int k = kc; k < e; k += 2) {
      const bool two = k + 1 < e;
      uint4 q[2], bl[2][NT], bh[2][NT];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int k2 = (i == 0 || two) ? k + i : k;   // a missing odd chunk reloads the even one, unused
        q[i] = *reinterpret_cast<const uint4*>(qp + (size_t)k2 * 512);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          bl[i][nt] = *reinterpret_cast<const uint4*>(brow[nt] + k2 * 64 + cc * 16);
          bh[i][nt] = *reinterpret_cast<const uint4*>(brow[nt] + k2 * 64 + cc * 16 + 8);
        }
      }
      mma_chunk<NT>(c[0], q[0], bl[0], bh[0]);
      if (two) mma_chunk<NT>(c[1], q[1], bl[1], bh[1]);
    }
    const float sg = __half2float(scp[(kc >> 2) * 16]);
    const float sg8 = __half2float(scp[(kc >> 2) * 16 + 8]) * 0.0625f;
    block_epilogue<NT, 2>(acc, c, sg, sg8, pre, kc, e);
    kc = e;
  }
}

// The same for a range of CPW chunks (a multiple of 4) starting on a block
// boundary: fully unrolled, about 1.5x faster than the generic loop (the
// compiler schedules the loads of all CPW chunks ahead of their MMAs).
template <int NT, int CPW>
DEV_INLINE void mma_fold_static(float (&acc)[2][4], const uint8_t* tile, uint32_t scale_bytes,
                                const __half* const (&brow)[2], const float* const (&pre)[2][2], int lane,
                                int c0) {
  const int g = lane >> 2, cc = lane & 3;
  const uint8_t* qp = tile + scale_bytes + lane * 16 + (size_t)c0 * 512;
  const __half* scp = reinterpret_cast<const __half*>(tile) + g + (c0 >> 2) * 16;
  const __half* bp[NT];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) bp[nt] = brow[nt] + c0 * 64 + cc * 16;
#pragma unroll
  for (int bk = 0; bk < CPW / 4; ++bk) {
    float c[4][NT][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int r = 0; r < 4; ++r) c[i][nt][r] = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int ch = bk * 4 + i;
      const uint4 q = *reinterpret_cast<const uint4*>(qp + ch * 512);
      uint4 bl[NT], bh[NT];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        bl[nt] = *reinterpret_cast<const uint4*>(bp[nt] + ch * 64);
        bh[nt] = *reinterpret_cast<const uint4*>(bp[nt] + ch * 64 + 8);
      }
      mma_chunk<NT>(c[i], q, bl, bh);
    }
    const float sg = __half2float(scp[bk * 16]);
    const float sg8 = __half2float(scp[bk * 16 + 8]) * 0.0625f;
    block_epilogue<NT, 4>(acc, c, sg, sg8, pre, c0 + bk * 4, c0 + bk * 4 + 4);
  }
}

// Dispatch on the warp's chunk range.
template <int NT>
DEV_INLINE void mma_range(float (&acc)[2][4], const uint8_t* tile, uint32_t scale_bytes,
                          const __half* const (&brow)[2], const float* const (&pre)[2][2], int lane, int c0, int c1) {
  // one token tile over whole scale blocks (the OLMoE- and Qwen-shaped gate/up
  // and the OLMoE down at 4 warps per group): the unrolled form block by
  // block (a block's operands fit the 128 registers a thread has here); the
  // loop otherwise
  if (NT == 1 && (c0 & 3) == 0 && ((c1 - c0) & 3) == 0) {
    for (int b0 = c0; b0 < c1; b0 += 4) mma_fold_static<NT, 4>(acc, tile, scale_bytes, brow, pre, lane, b0);
  } else {
    mma_fold<NT>(acc, tile, scale_bytes, brow, pre, lane, c0, c1);
  }
}

// Prefix sums over K chunks of n FP16 rows [n][stride] (nk chunks of 64):
// out[row * (nk + 1) + j] = sum of the row's values in chunks < j.  Two steps
// separated by the caller's barrier: chunk_sums() then chunk_prefix().
DEV_INLINE void chunk_sums(float* out, const __half* rows, int stride, int n, int nk, int t0, int nthr) {
  for (int i = t0; i < n * nk; i += nthr) {
    const int r = i / nk, kc = i - r * nk;
    const uint4* p = reinterpret_cast<const uint4*>(rows + (size_t)r * stride + kc * 64);
    float s = 0.f;
#pragma unroll
    for (int v = 0; v < 8; ++v) {
      const uint4 u = p[v];
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[h]));
        s += f.x + f.y;
      }
    }
    out[r * (nk + 1) + kc + 1] = s;
  }
}

DEV_INLINE void chunk_prefix(float* out, int n, int nk, int t0, int nthr) {
  for (int r = t0; r < n; r += nthr) {
    float* o = out + r * (nk + 1);
    float s = 0.f;
    o[0] = 0.f;
    for (int j = 1; j <= nk; ++j) {
      s += o[j];
      o[j] = s;
    }
  }
}

// Group leader: posts a note (the active expert u of a finished gate/up
// item) to the signaller.  The group barrier before the call orders the
// item's h stores before the note.
DEV_INLINE void post_note(int* mbox, volatile int* head, volatile int* tail, int& my_head, int v,
                          volatile int* abort, DevStatus* st) {
  if (my_head - *tail >= kMB) {   // mailbox full: bounded wait for the signaller
    const long long t0 = clock64();
    while (my_head - *tail >= kMB) {
      if (*abort) return;
      if (clock64() - t0 > MOE_WAIT_CYCLES) {
        atomicOr(&st->flags, STATUS_TIMEOUT);
        *abort = 1;
        return;
      }
      __nanosleep(64);
    }
  }
  mbox[my_head % kMB] = v;
  __threadfence_block();
  *head = ++my_head;
}

template <int GW, bool INTER>
__global__ void __launch_bounds__(kFThreads, 1) fused_decode_kernel(FwdCtx c) {
  constexpr int NG = kCW / GW;
  constexpr int kMatUnroll = GW == 6 ? 2 : 1;
  extern __shared__ __align__(128) uint8_t sm[];
  __shared__ __align__(8) uint64_t full[kMaxSlots], empty[kMaxSlots], xbar;
  __shared__ int s_ok;
  __shared__ volatile int s_abort;   // a bounded wait ran out: stop waiting
  __shared__ volatile int s_seq[kMaxSlots];   // entry held by each ring slot
  __shared__ CtaUnits<INTER> s_cu;            // the CTA's units (compute warps and signaller)
  __shared__ int s_mbox[NG][kMB];             // group -> signaller notes
  __shared__ volatile int s_head[NG], s_tail[NG];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x, b = blockIdx.x;
  const int T = c.T, E = c.E, H = c.H, I = c.I, k = c.k, P = T * k;
  const FusedSmem L = fused_smem(c.lay, H, I, E, T, k, GW);
  __half* xcache = reinterpret_cast<__half*>(sm + L.off_x);
  __half* hstage = reinterpret_cast<__half*>(sm + L.off_h);
  float* red = reinterpret_cast<float*>(sm + L.off_red);
  float* sb_x = reinterpret_cast<float*>(sm + L.off_sb);        // [T][H/64 + 1] prefix sums
  float* sb_h = sb_x + T * (H / 64 + 1);                         // per group [min(T, 8)][I/64 + 1]
  float* lg = reinterpret_cast<float*>(sm + L.off_route);   // [T][E]
  int* r_ids = reinterpret_cast<int*>(lg + T * E);
  float* r_w = reinterpret_cast<float*>(r_ids + P);
  int* r_sorted = reinterpret_cast<int*>(r_w + P);
  float* r_rnorm = reinterpret_cast<float*>(r_sorted + P);
  int* r_table = reinterpret_cast<int*>(r_rnorm + T);
  int* r_cnt = r_table + (E + 1);
  int* r_off = r_cnt + (E + 1);
  int* r_aslot = r_off + (E + 1);
  int* r_astart = r_aslot + (E + 1);
  int* r_acount = r_astart + (E + 1);
  int* r_chunk = r_acount + (E + 1);            // [ceil(P/32)][E] per-32-pair counts
  int* r_misc = r_chunk + ((P + 31) / 32) * E;   // [0] = active experts

  const int NS = (int)L.ns;
  if (tid == 0) {
    s_ok = 1;
    s_abort = 0;
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], GW);   // one arrival per consumer warp
      s_seq[s] = -1;
    }
    for (int q = 0; q < NG; ++q) s_head[q] = s_tail[q] = 0;
    mbar_init(&xbar, 1);
    fence_mbar_init();
  }
  // everything above is CTA-local: it overlaps the tail of the preceding
  // kernel (programmatic dependent launch); x, the table and the counters are
  // read only after that kernel has completed
  pdl_wait();
  pdl_trigger();
  if (tid == 0) {
    // the T token rows of x, staged once (padded rows) for every gate/up item
    // of this CTA; the copies run while the router phase computes
    mbar_expect_tx(&xbar, (uint32_t)T * H * 2);
    for (int t = 0; t < T; ++t) bulk_g2s(xcache + (size_t)t * (H + 8), c.x + (size_t)t * H, (uint32_t)H * 2, &xbar);
  }
  for (int e = tid; e < E; e += blockDim.x) r_table[e] = c.table[e];
  // readiness counters start from zero: nothing counts before the routing barrier
  if (b == 0)
    for (int e = tid; e < E; e += blockDim.x) c.expert_ready[e] = 0u;

  // ---------------------------------------------------------------- routing
  {
    const int half = ((H / 2) + 255) / 256 * 256;   // K split point (multiple of 256)
    const int nt = 2 * T * E + ((c.flags & 2u) ? 2 * T : 0);
    for (int task = warp * G + b; task < nt; task += G * kNW) {
      const int part = task & 1, pair = task >> 1;
      const int k0 = part ? half : 0, k1 = part ? H : (half < H ? half : H);
      if (pair < T * E) {
        const int t = pair / E, e = pair % E;
        const float v = warp_dot_part(c.x + (size_t)t * H, c.router_w + (size_t)e * H, k0, k1, lane);
        if (lane == 0) c.logit_part[(size_t)part * T * E + pair] = v;
      } else {
        const int t = pair - T * E;
        const __half* xt = c.x + (size_t)t * H;
        const float v = warp_dot_part(xt, xt, k0, k1, lane);
        if (lane == 0) c.ss_part[(size_t)part * T + t] = v;
      }
    }
  }
  __syncthreads();
  // arrive at the routing barrier, then (while the other CTAs arrive) the
  // per-chunk prefix sums of the staged x rows, then wait
  unsigned long long bar_target = 0;
  if (tid == 0) {
    bar_target = grid_arrive(c.grid_bar, (unsigned)G);
    if (!mbar_wait_bounded(&xbar, 0, c.status)) s_ok = 0;   // x rows landed
  }
  __syncthreads();
  if (s_ok) {
    chunk_sums(sb_x, xcache, H + 8, T, H / 64, tid, kNW * 32);
    __syncthreads();
    chunk_prefix(sb_x, T, H / 64, tid, kNW * 32);
  }
  if (tid == 0 && s_ok && !grid_wait(c.grid_bar, bar_target, c.status)) s_ok = 0;
  __syncthreads();
  if (!s_ok) {
    if (tid == 0) mbar_wait_bounded(&xbar, 0, c.status);   // let the x copies land
    return;
  }

  // ------------------------------------------ routing in shared memory
  const int nchunk = (P + 31) / 32;
  for (int e = tid; e < nchunk * E; e += blockDim.x) r_chunk[e] = 0;
  {
    FwdCtx cl = c;   // top-k results go to shared memory
    cl.ids = r_ids;
    cl.topw = r_w;
    for (int t = warp; t < T; t += kNW) {
      // the token's logits: its two K-half partial sums, straight from global memory
      for (int e = lane; e < E; e += 32)
        lg[t * E + e] = __ldcg(&c.logit_part[t * E + e]) + __ldcg(&c.logit_part[T * E + t * E + e]);
      float r = 1.f;
      if (c.flags & 2u) {
        r = prenorm_scale(__ldcg(&c.ss_part[t]) + __ldcg(&c.ss_part[T + t]), H);
        if (lane == 0) r_rnorm[t] = r;
      }
      __syncwarp();
      topk_token(cl, t, lg + t * E, r, nullptr);
    }
  }
  __syncthreads();   // top-k ids and weights of every token
  const int tpe1 = I / 16;   // gate/up items per expert

  if (warp == kCW) {
    // ------------------------------------------------------------ producer
    // The active experts (routed and resident), ascending, straight from the
    // ids: a warp-wide union bitmask, so the weight stream starts while the
    // other warps count, scan and scatter.
    int U = 0;
    for (int w0 = 0; w0 < E; w0 += 32) {
      unsigned bits = 0;
      for (int p = lane; p < P; p += 32) {
        const int e = r_ids[p];
        if (e >= w0 && e < w0 + 32) bits |= 1u << (e - w0);
      }
      bits = __reduce_or_sync(kFull, bits);
      const int e = w0 + lane;
      const bool act = e < E && ((bits >> lane) & 1u) && r_table[e] >= 0;
      const unsigned am = __ballot_sync(kFull, act);
      if (act) r_aslot[U + __popc(am & ((1u << lane) - 1u))] = r_table[e];
      U += __popc(am);
    }
    __syncwarp();
    const CtaUnits<INTER> cu = cta_units<INTER>(U, I, H, b, G, NG);
    // the CTA's units in order: a gate/up item is a gate entry and an up
    // entry, a down item one or two entries of a 32-row block (2 row tiles);
    // entry e -> slot e % NS
    if (lane == 0) {
      int issued = 0;
      bool stop = false;
      const int nu = cu.count();
      for (int j = 0; j < nu && !stop; ++j) {
        const Unit un = cu.at(j);
        const uint8_t* base = c.pool + (size_t)r_aslot[un.u] * c.slot_bytes;
        for (int sub = 0; sub < (un.down ? cu.down_entries() : 2); ++sub) {
          const int e = issued, s = e % NS;
          if (!wait_phase(&empty[s], (uint32_t)((e / NS) & 1) ^ 1u, &s_abort, c.status)) {
            stop = true;
            break;
          }
          // at most kInFlight entries on their way: copies issued together share
          // the bandwidth and land together, so a bounded window lets the first
          // entries land (and compute start) early.  Entry e - kInFlight's slot
          // cannot hold a newer entry yet, so its parity is unambiguous.
          if (e >= kInFlight) {
            const int ep = e - kInFlight;
            if (!wait_phase(&full[ep % NS], (uint32_t)((ep / NS) & 1), &s_abort, c.status)) {
              stop = true;
              break;
            }
          }
          s_seq[s] = e;
          uint8_t* dst = sm + (size_t)s * L.slot_bytes;
          if (!un.down) {
            const MatLayout& M = sub ? c.lay.up : c.lay.gate;
            mbar_expect_tx(&full[s], M.tile_bytes);
            bulk_g2s(dst, tile_ptr(base, M, un.idx), M.tile_bytes, &full[s]);
          } else {
            const uint32_t bytes = 2 * c.lay.down.tile_bytes;   // the 2 row tiles of a block are contiguous
            mbar_expect_tx(&full[s], bytes);
            bulk_g2s(dst, tile_ptr(base, c.lay.down, 2 * cu.down_block(un, sub)), bytes, &full[s]);
          }
          issued = e + 1;
        }
      }
      // copies in flight land before the CTA (and its shared memory) ends:
      // only the last entry issued into a slot can still be pending
      for (int s = 0; s < NS && s < issued; ++s) {
        const int last = s + (issued - 1 - s) / NS * NS;
        mbar_wait_bounded(&full[s], (uint32_t)((last / NS) & 1), c.status);
      }
    }
    return;
  }

  // ---------------------------------------- counts, scan, active groups
  // (every warp but the producer: named barrier 6, 13 warps)
  const int wr = warp < kCW ? warp : kCW;   // the signaller takes the producer's turn
  for (int ch = wr; ch < nchunk; ch += kNW - 1) {
    // counts per 32-pair chunk: __match_any_sync groups equal ids (no atomics)
    const int p = ch * 32 + lane;
    const int e = p < P ? r_ids[p] : -1 - lane;
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    if (p < P && __popc(peers & ((1u << lane) - 1u)) == 0) r_chunk[ch * E + e] = __popc(peers);
  }
  named_sync(6, (kNW - 1) * 32);
  if (warp == 0) {
    // counts, exclusive scan and active groups (ascending experts) in one
    // compact loop of 32-expert rounds: this runs once per launch on one warp,
    // so its cost is mostly instruction fetch and grows with code size
    int n = 0, base = 0;
#pragma unroll 1
    for (int e0 = 0; e0 < E; e0 += 32) {
      const int e = e0 + lane;
      int ce = 0;
      if (e < E)
        for (int ch = 0; ch < nchunk; ++ch) ce += r_chunk[ch * E + e];
      int incl = ce;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += v;
      }
      const int off = base + incl - ce;
      if (e < E) r_off[e] = off;
      const int slot = ce > 0 ? r_table[e] : -1;
      const bool act = ce > 0 && slot >= 0;
      if (b == 0 && ce > 0 && slot < 0) {
        atomicAdd(&c.status->miss, (unsigned long long)ce);
        atomicOr(&c.status->flags, STATUS_MISS);
      }
      const unsigned am = __ballot_sync(kFull, act);
      const int pos = n + __popc(am & ((1u << lane) - 1u));
      if (act) {
        r_astart[pos] = off;
        r_acount[pos] = ce;
      }
      n += __popc(am);
      base += __shfl_sync(kFull, incl, 31);
    }
    if (lane == 0) {
      r_off[E] = base;
      r_misc[0] = n;
      s_cu = cta_units<INTER>(n, I, H, b, G, NG);
    }
  }
  named_sync(6, (kNW - 1) * 32);
  const int U = r_misc[0];
  const CtaUnits<INTER>& cu = s_cu;

  if (warp == kCW + 1) {
    // ----------------------------------------------------------- signaller
    // Turns the groups' gate/up notes into GPU-wide readiness counts, one
    // fence per batch of notes, the adds fire-and-forget.
    unsigned* ready = c.expert_ready;
    int m1 = 0;   // the CTA's gate/up items: one note each
    for (int j = lane; j < cu.count(); j += 32) m1 += 1 - cu.at(j).down;
    m1 = __reduce_add_sync(kFull, m1);
    int processed = 0, tails[NG];
#pragma unroll
    for (int q = 0; q < NG; ++q) tails[q] = 0;
    long long t0 = clock64();
    while (processed < m1) {
      int heads[NG], avail = 0;
#pragma unroll
      for (int q = 0; q < NG; ++q) {
        heads[q] = s_head[q];
        avail += heads[q] - tails[q];
      }
      __threadfence_block();   // notes read after the heads that announce them
      if (avail == 0) {
        if (s_abort) break;
        if (clock64() - t0 > MOE_WAIT_CYCLES) {
          if (lane == 0) atomicOr(&c.status->flags, STATUS_TIMEOUT);
          s_abort = 1;
          break;
        }
        __nanosleep(32);
        continue;
      }
      __threadfence();   // the h stores behind these notes are visible GPU-wide before the counts
      int n = 0;
#pragma unroll
      for (int q = 0; q < NG; ++q) {
        for (; tails[q] < heads[q]; ++tails[q], ++n) {
          const int u = reinterpret_cast<volatile int*>(s_mbox[q])[tails[q] % kMB];
          if (lane == (n & 31)) atomicAdd(&ready[u], 1u);
        }
      }
      __syncwarp();
      if (lane == 0)
#pragma unroll
        for (int q = 0; q < NG; ++q) s_tail[q] = tails[q];
      processed += n;
      t0 = clock64();
    }
    return;
  }

  // -------------------------------------------------------- compute warps
  // stable scatter: rank = same-expert pairs in earlier chunks + rank inside the chunk
  for (int ch = warp; ch < nchunk; ch += kCW) {
    const int p = ch * 32 + lane;
    const int e = p < P ? r_ids[p] : -1 - lane;
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    if (p < P) {
      int rank = __popc(peers & ((1u << lane) - 1u));
      for (int c2 = 0; c2 < ch; ++c2) rank += r_chunk[c2 * E + e];
      r_sorted[r_off[e] + rank] = p;
    }
  }
  named_sync(1, kCW * 32);
  if (b == 0) {   // publish the routing (debug outputs, rnorm)
    for (int i = tid; i < P; i += kCW * 32) {
      c.ids[i] = r_ids[i];
      c.topw[i] = r_w[i];
      c.sorted[i] = r_sorted[i];
    }
    for (int i = tid; i <= E; i += kCW * 32) c.offsets[i] = r_off[i];
    if (c.flags & 2u)
      for (int i = tid; i < T; i += kCW * 32) c.rnorm[i] = r_rnorm[i];
  }
  named_sync(1, kCW * 32);
  if (U == 0) {   // every routed expert is absent: out = residual or 0
    for (int i = b * kCW * 32 + tid; i < T * H; i += G * kCW * 32)
      c.out[i] = (c.flags & 1u) ? c.x[i] : __float2half_rn(0.f);
    return;
  }

  const int q = warp / GW, wq = warp % GW;   // group, warp in group
  const int gtid = tid - q * GW * 32;        // thread index inside the group
  const int g = lane >> 2, cc = lane & 3;
  const int gbar = 7 + q;                    // named barrier of group q (7 .. 12)
  const int ntok = T <= 8 ? 8 : 16;
  float* rg = red + q * GW * 2 * 16 * ntok;  // this group's reduction buffer
  __half* hs = hstage + (size_t)q * (T < kTok ? T : kTok) * (I + 8);   // this group's h rows
  const unsigned* ready = c.expert_ready;    // [u]: finished gate/up items of active expert u (this launch)
  int ready_u = -1, staged_u = -1, staged_p0 = -1;
  int my_head = 0;                           // leader: notes posted

  const int nu = cu.count();
  for (int j = q; j < nu; j += NG) {   // the CTA's units q, q + NG, ...
    const Unit un = cu.at(j);
    const int e0 = cu.first_entry(j);
    if (!un.down) {
      // ---------------------------------------------------- gate/up item
      const int u = un.u, rt = un.idx;
      const int start = r_astart[u], cnt = r_acount[u];   // cnt <= T <= 16
      const int ntl = cnt > 8 ? 2 : 1;
      const int tok0 = r_sorted[start] / k;
      const __half* brow[2];
      const float* pre[2][2];
      const int nkh = H / 64;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const int ti = nt * 8 + g;   // the lane's B row; rows past cnt feed discarded columns
        brow[nt] = xcache + (size_t)(ti < cnt ? r_sorted[start + ti] / k : tok0) * (H + 8);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int tc = nt * 8 + 2 * cc + h;   // the lane's output columns
          pre[nt][h] = sb_x + (size_t)(tc < cnt ? r_sorted[start + tc] / k : tok0) * (nkh + 1);
        }
      }
      const int kc0 = wq * nkh / GW, kc1 = (wq + 1) * nkh / GW;   // the warp's K chunks
      float* rw = rg + wq * 2 * 16 * ntok;   // K-split partials -> rg[warp][mat][row][token]
      // up to 4-warp groups not unrolled: one copy of the MMA loop serves gate
      // and up (a second copy doubles the instruction fetches); 6-warp groups
      // (T > 8, two token tiles) measured faster unrolled
#pragma unroll kMatUnroll
      for (int mat = 0; mat < 2; ++mat) {
        float acc[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int r = 0; r < 4; ++r) acc[nt][r] = 0.f;
        const int e = e0 + mat, s = e % NS;
        warp_wait_entry(s_seq, full, e, NS, &s_abort, c.status, lane);
        const uint8_t* tile = sm + (size_t)s * L.slot_bytes;
        if (ntl == 1)
          mma_range<1>(acc, tile, c.lay.gate.scale_bytes, brow, pre, lane, kc0, kc1);
        else
          mma_range<2>(acc, tile, c.lay.gate.scale_bytes, brow, pre, lane, kc0, kc1);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
          if (nt < ntl) {
            float* r0 = rw + (mat * 16 + g) * ntok + nt * 8 + 2 * cc;
            r0[0] = acc[nt][0];
            r0[1] = acc[nt][1];
            r0[8 * ntok] = acc[nt][2];
            r0[8 * ntok + 1] = acc[nt][3];
          }
        // The entry is released only after stores that depend on every word
        // read from it: the shared loads have completed before the bulk copy
        // that refills the slot can be issued.
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
      }
      named_sync(gbar, GW * 32);
      for (int idx = gtid; idx < 16 * cnt; idx += GW * 32) {
        const int tok = idx >> 4, row = idx & 15;
        float gs = 0.f, us = 0.f;
#pragma unroll
        for (int ww = 0; ww < GW; ++ww) {
          gs += rg[(ww * 2 + 0) * 16 * ntok + row * ntok + tok];
          us += rg[(ww * 2 + 1) * 16 * ntok + row * ntok + tok];
        }
        if (c.flags & 2u) {
          const float r = r_rnorm[r_sorted[start + tok] / k];
          gs *= r;
          us *= r;
        }
        c.hbuf[(size_t)(start + tok) * I + rt * 16 + row] = __float2half_rn(silu_mul(gs, us));
      }
      named_sync(gbar, GW * 32);   // h rows written, reduction buffer free
      if (gtid == 0) post_note(&s_mbox[q][0], &s_head[q], &s_tail[q], my_head, u, &s_abort, c.status);
    } else {
      // ------------------------------------------------------- down item
      const int u = un.u;
      const int start = r_astart[u], cnt = r_acount[u];
      if (u != ready_u) {   // h of expert u complete (every gate/up item counted)
        if (gtid == 0) wait_count(&ready[u], (unsigned)tpe1, &s_abort, c.status);
        ready_u = u;
      }
      const int tl = wq & 1, ks = wq >> 1;   // row tile of an entry, K part
#pragma unroll 1
      for (int sub = 0; sub < cu.down_entries(); ++sub) {   // the item's 32-row blocks, one entry each
        const int hb = cu.down_block(un, sub), e = e0 + sub, s = e % NS;
        const uint8_t* tile = sm + (size_t)s * L.slot_bytes + (size_t)tl * c.lay.down.tile_bytes;
        warp_wait_entry(s_seq, full, e, NS, &s_abort, c.status, lane);
        for (int p0 = 0; p0 < cnt; p0 += kTok) {
          const int np = min(kTok, cnt - p0);
          float* sbg = sb_h + (size_t)q * (T < kTok ? T : kTok) * (I / 64 + 1);   // this group's h prefix sums
          if (u != staged_u || p0 != staged_p0) {
            named_sync(gbar, GW * 32);   // readiness seen by the leader; the group is done with hs
            const int vpr = I / 8;       // the np rows are consecutive in hbuf
            const __half* src = c.hbuf + (size_t)(start + p0) * I;
            for (int v = gtid; v < np * vpr; v += GW * 32)
              cp_async16(hs + (size_t)(v / vpr) * (I + 8) + (v % vpr) * 8, src + (size_t)v * 8);
            cp_async_wait_all();
            named_sync(gbar, GW * 32);
            chunk_sums(sbg, hs, I + 8, np, I / 64, gtid, GW * 32);
            named_sync(gbar, GW * 32);
            chunk_prefix(sbg, np, I / 64, gtid, GW * 32);
            staged_u = u;
            staged_p0 = p0;
          }
          named_sync(gbar, GW * 32);   // staged rows and sums visible; previous pass done with rg
          float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
          const __half* const brow[2] = {hs + (size_t)(g < np ? g : 0) * (I + 8), hs};
          const int nki = I / 64, parts = GW / 2;
          const float* const pre[2][2] = {{sbg + (size_t)(2 * cc < np ? 2 * cc : 0) * (nki + 1),
                                           sbg + (size_t)(2 * cc + 1 < np ? 2 * cc + 1 : 0) * (nki + 1)},
                                          {sbg, sbg}};
          mma_range<1>(acc, tile, c.lay.down.scale_bytes, brow, pre, lane, ks * nki / parts, (ks + 1) * nki / parts);
          float* rw = rg + wq * 16 * kTok;
          rw[g * kTok + 2 * cc] = acc[0][0];
          rw[g * kTok + 2 * cc + 1] = acc[0][1];
          rw[(g + 8) * kTok + 2 * cc] = acc[0][2];
          rw[(g + 8) * kTok + 2 * cc + 1] = acc[0][3];
          named_sync(gbar, GW * 32);
          for (int idx = gtid; idx < kDownRows * np; idx += GW * 32) {
            const int tok = idx / kDownRows, row = idx % kDownRows, t16 = row >> 4, r16 = row & 15;
            float y = 0.f;
#pragma unroll
            for (int kp = 0; kp < GW / 2; ++kp) y += rg[(kp * 2 + t16) * 16 * kTok + r16 * kTok + tok];
            c.ybuf[(size_t)r_sorted[start + p0 + tok] * H + hb * kDownRows + row] = y;
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
      }
    }
  }

  // ---------------------------------------------------------------- combine
  // every y row of the layer is written once all CTAs pass this barrier;
  // out[t] = (x[t]) + sum_j w[t, j] y[t k + j], summed in rank order j
  named_sync(1, kCW * 32);
  if (tid == 0 && !grid_barrier(c.grid_bar, (unsigned)G, c.status)) s_abort = 1;
  named_sync(1, kCW * 32);
  const bool residual = c.flags & 1u;
  for (int idx = b * kCW * 32 + tid; idx < T * H; idx += G * kCW * 32) {
    const int t = idx / H, hr = idx - t * H;
    float acc = residual ? __half2float(c.x[idx]) : 0.f;
#pragma unroll 4
    for (int jj = 0; jj < k; ++jj) {
      const int pp = t * k + jj;
      if (r_table[r_ids[pp]] >= 0) acc = fmaf(r_w[pp], __ldcg(&c.ybuf[(size_t)pp * H + hr]), acc);
    }
    c.out[idx] = __float2half_rn(acc);
  }
}

template <int GW, bool INTER>
cudaError_t launch_fused(const FwdCtx& c, const FusedSmem& L, cudaStream_t st) {
  cudaError_t e = opt_in_smem((const void*)fused_decode_kernel<GW, INTER>, L.total);
  if (e != cudaSuccess) return e;
  int per_sm = 0;   // all CTAs of a cooperative launch must be co-resident
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fused_decode_kernel<GW, INTER>, kFThreads, L.total);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorNotSupported;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(c.num_sms);
  cfg.blockDim = dim3(kFThreads);
  cfg.dynamicSmemBytes = L.total;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  // programmatic dependent launch: the launch and the CTA-local prologue
  // overlap the preceding kernel (all CTAs still co-reside: the preceding
  // kernel never waits on this one)
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  static std::atomic<int> pdl_ok{1};   // cleared if the driver refuses the pair of attributes
  cfg.numAttrs = pdl_ok.load() ? 2 : 1;
  e = cudaLaunchKernelEx(&cfg, fused_decode_kernel<GW, INTER>, c);
  if (e != cudaSuccess && cfg.numAttrs == 2) {
    cudaGetLastError();
    pdl_ok.store(0);
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, fused_decode_kernel<GW, INTER>, c);
  }
  return e;
}

}  // namespace

// The fused kernel applies to small decode batches (every token row staged
// in shared memory) whose routing state leaves room for a ring of at least
// kMinSlots weight entries.
bool fused_decode_supported(const FwdCtx& c, int max_smem) {
  if (c.T > kMaxT || c.T * c.k > kMaxP || c.H % 64 || c.I % 64 || c.k > 32 || c.E > kMaxExperts) return false;
  const FusedSmem L = fused_smem(c.lay, c.H, c.I, c.E, c.T, c.k, fused_group_warps(c.T, c.k));
  return L.ns >= (uint32_t)kMinSlots && L.total <= kSmemBudget && (int)L.total <= max_smem;
}

cudaError_t launch_fused_decode(const FwdCtx& c, cudaStream_t st, const StageEvents& se) {
  const FusedSmem L = fused_smem(c.lay, c.H, c.I, c.E, c.T, c.k, fused_group_warps(c.T, c.k));
  const int gw = fused_group_warps(c.T, c.k);
  // the interleaved order is instantiated for 4-warp groups only
  cudaError_t e = gw == 2   ? launch_fused<2, false>(c, L, st)
                  : gw == 6 ? launch_fused<6, false>(c, L, st)
                  : fused_interleaved(c.H, c.I, gw) ? launch_fused<4, true>(c, L, st)
                                                    : launch_fused<4, false>(c, L, st);
  if (e == cudaSuccess) e = record_stage(se, 2, st);
  if (e == cudaSuccess) e = record_stage(se, 3, st);
  if (e == cudaSuccess) e = record_stage(se, 4, st);
  return e;
}
