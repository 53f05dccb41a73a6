// Router (FP16 x FP16 -> FP32 logits), softmax / top-k, and the stable
// token-to-expert permutation.
//
// Routing stays outside INT4 (Horizon RunMap landing page, "08 / Precision &
// quality"); it selects the experts of each routed layer ("06 / Follow a
// token").  Rule: softmax over all E logits, the k largest logits (ties to the
// lower expert index) listed largest first, weights = the softmax entries of
// those experts, not renormalised.
//
// Two launch shapes:
//   small T  : one launch of a thread-block cluster (up to 8 CTAs).  Each CTA
//              computes the logits of a slice of the experts and writes them
//              into CTA 0's shared memory (distributed shared memory); after
//              the cluster barrier CTA 0 finishes softmax/top-k and the
//              permutation entirely in shared memory.
//   larger T : one cooperative kernel (logits on the tensor cores, top-k,
//              scan, scatter and, for the grouped GEMM, the x rows in sorted
//              order: the forward's router; up to 64 tokens the same phases
//              on one 8-CTA thread-block cluster), or four launches (logits,
//              top-k, scan, scatter: the allocation-free router, which has
//              no barrier counter of its own).
#include "route_dev.cuh"

namespace {

using namespace route_dev;

// ------------------------------------------------------------ small T path
constexpr int kRouteTC = 8;       // tokens per staged x chunk

// Bytes of dynamic smem of route_cluster_kernel.
size_t route_cluster_smem(int T, int E, int H, int k) {
  return (size_t)2 * kRouteTC * H * 2 + (size_t)T * E * 4 + (size_t)T * 4 + (size_t)T * k * 4 +
         (size_t)(8 * E + 2 * E + 1) * 4;
}

// smem: xbuf [2][kRouteTC][H] f16 | logits [T][E] f32 (CTA 0) | ss [T] f32 (CTA 0)
//       | ids [T*k] i32 | permutation scratch
__global__ void __launch_bounds__(256) route_cluster_kernel(FwdCtx c) {
  extern __shared__ __align__(128) uint8_t rsm[];
  __shared__ __align__(8) uint64_t xbar[2];
  __shared__ int s_ok;
  pdl_wait();      // x may be the output of the preceding grid
  pdl_trigger();
  const int T = c.T, E = c.E, H = c.H;
  __half* xbuf = reinterpret_cast<__half*>(rsm);
  float* logits = reinterpret_cast<float*>(rsm + (size_t)2 * kRouteTC * H * 2);
  float* ss = logits + T * E;
  int* ids_s = reinterpret_cast<int*>(ss + T);
  int* scratch = ids_s + T * c.k;
  const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
  const int nch = (T + kRouteTC - 1) / kRouteTC;
  auto issue = [&](int ch) {
    const int ntok = min(kRouteTC, T - ch * kRouteTC);
    const uint32_t bytes = (uint32_t)ntok * H * 2;
    mbar_expect_tx(&xbar[ch & 1], bytes);
    bulk_g2s(xbuf + (size_t)(ch & 1) * kRouteTC * H, c.x + (size_t)ch * kRouteTC * H, bytes, &xbar[ch & 1]);
  };
  if (tid == 0) {
    s_ok = 1;
    mbar_init(&xbar[0], 1);
    mbar_init(&xbar[1], 1);
    fence_mbar_init();
    issue(0);
    if (nch > 1) issue(1);
  }
  cluster_sync();  // every CTA of the cluster is running; barrier init visible
  const uint32_t rank = cluster_rank(), C = gridDim.x;
  const int epc = (E + (int)C - 1) / (int)C;
  for (int ch = 0; ch < nch; ++ch) {
    const int b = ch & 1;
    if (!mbar_wait_bounded(&xbar[b], (ch >> 1) & 1, c.status)) s_ok = 0;
    __syncthreads();
    const int ntok = min(kRouteTC, T - ch * kRouteTC);
    const __half* xs = xbuf + (size_t)b * kRouteTC * H;
    if (s_ok) {
      for (int ei = w; ei < epc; ei += kLogitWarps) {
        const int e = (int)rank * epc + ei;
        if (e >= E) break;
        const __half* we = c.router_w + (size_t)e * H;
        float acc[kRouteTC];
#pragma unroll
        for (int t = 0; t < kRouteTC; ++t) acc[t] = 0.f;
        for (int kb = 0; kb < H; kb += 2048) {
          uint4 wr[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int kk = kb + i * 256 + lane * 8;
            wr[i] = kk < H ? __ldg(reinterpret_cast<const uint4*>(we + kk)) : make_uint4(0, 0, 0, 0);
          }
#pragma unroll
          for (int t = 0; t < kRouteTC; ++t) {
            if (t < ntok) {
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                const int kk = kb + i * 256 + lane * 8;
                if (kk < H) acc[t] += dot8(*reinterpret_cast<const uint4*>(xs + (size_t)t * H + kk), wr[i]);
              }
            }
          }
        }
#pragma unroll
        for (int t = 0; t < kRouteTC; ++t) {
          if (t < ntok) {
            const float v = warp_sum(acc[t]);
            if (lane == 0) st_cluster_f32(map_to_rank(&logits[(ch * kRouteTC + t) * E + e], 0), v);
          }
        }
      }
      if ((c.flags & 2u) && (int)rank == ch % (int)C && w < ntok) {   // PRENORM sums of squares
        const __half* xt = xs + (size_t)w * H;
        float s2 = 0.f;
        for (int kk = lane * 8; kk < H; kk += 256) {
          const uint4 v = *reinterpret_cast<const uint4*>(xt + kk);
          s2 += dot8(v, v);
        }
        s2 = warp_sum(s2);
        if (lane == 0) st_cluster_f32(map_to_rank(&ss[ch * kRouteTC + w], 0), s2);
      }
    }
    __syncthreads();   // every warp is done with xbuf[b]
    if (tid == 0 && ch + 2 < nch) issue(ch + 2);
  }
  cluster_sync();
  if (rank != 0) return;
  for (int t = w; t < T; t += blockDim.x >> 5) {
    float r = 1.f;
    if (c.flags & 2u) {
      r = prenorm_scale(ss[t], H);
      if (lane == 0) c.rnorm[t] = r;
    }
    topk_token(c, t, logits + t * E, r, ids_s);
  }
  __syncthreads();
  permute_block(c, ids_s, scratch);
}

// ------------------------------------------------------------ larger T path
constexpr int kRouteKC = 256;     // K slice of one logits CTA
constexpr int kRouteTile = 64;    // tokens x experts of one logits CTA

// Partial logits of a 64-token x 64-expert tile over one 256-wide K slice on
// the tensor cores (16x8x16 MMA, FP16 in, FP32 accumulate); the slices are
// summed in fixed order by the top-k step.  Threads [0, nthr) load (nthr a
// multiple of 128); warps 0-3 multiply.  sm: 2 x 64 x (256 + 8) halves.
constexpr int kLogitSmem = 2 * kRouteTile * (kRouteKC + 8) * 2;
DEV_INLINE void logits_tile(const FwdCtx& c, int tt, int et, int ks, uint8_t* sm, int nthr) {
  constexpr int S = kRouteKC + 8;   // padded row stride (halves): conflict-free fragment reads
  __half* xs = reinterpret_cast<__half*>(sm);
  __half* ws = xs + kRouteTile * S;
  const int T = c.T, E = c.E, H = c.H;
  const int t0 = tt * kRouteTile, e0 = et * kRouteTile;
  const int k0 = ks * kRouteKC, kc = min(kRouteKC, H - k0);
  const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31, g = lane >> 2, cq = lane & 3;
  const int vpr = kc / 8;   // 16-byte vectors per row
  const int nvec = kRouteTile * vpr;
  if (tid < nthr)
    for (int i0 = 0; i0 < nvec; i0 += 8 * nthr) {   // 16 independent loads in flight per thread
      uint4 xv[8], wv[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int i = i0 + u * nthr + tid;
        const int r = i / vpr, v = i % vpr;
        const uint4 z = make_uint4(0, 0, 0, 0);
        xv[u] = (i < nvec && t0 + r < T) ? __ldg(reinterpret_cast<const uint4*>(c.x + (size_t)(t0 + r) * H + k0) + v) : z;
        wv[u] = (i < nvec && e0 + r < E) ? __ldg(reinterpret_cast<const uint4*>(c.router_w + (size_t)(e0 + r) * H + k0) + v)
                                         : z;
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int i = i0 + u * nthr + tid;
        if (i < nvec) {
          const int r = i / vpr, v = i % vpr;
          *reinterpret_cast<uint4*>(xs + r * S + v * 8) = xv[u];
          *reinterpret_cast<uint4*>(ws + r * S + v * 8) = wv[u];
        }
      }
    }
  __syncthreads();
  if (w < 4) {
    float acc[8][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[nt][i] = 0.f;
    const __half* xa = xs + (w * 16 + g) * S + 2 * cq;
    for (int kk = 0; kk < kc; kk += 16) {
      uint32_t a[4];
      a[0] = *reinterpret_cast<const uint32_t*>(xa + kk);
      a[1] = *reinterpret_cast<const uint32_t*>(xa + 8 * S + kk);
      a[2] = *reinterpret_cast<const uint32_t*>(xa + kk + 8);
      a[3] = *reinterpret_cast<const uint32_t*>(xa + 8 * S + kk + 8);
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        const __half* wb = ws + (nt * 8 + g) * S + kk + 2 * cq;
        mma_16816(acc[nt], a, *reinterpret_cast<const uint32_t*>(wb), *reinterpret_cast<const uint32_t*>(wb + 8));
      }
    }
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int t = t0 + w * 16 + g + (i >= 2 ? 8 : 0), e = e0 + nt * 8 + 2 * cq + (i & 1);
        if (t < T && e < E) c.logit_part[((size_t)ks * T + t) * E + e] = acc[nt][i];
      }
    }
    if ((c.flags & 2u) && et == 0) {   // PRENORM: partial sums of squares
      for (int r = w; r < kRouteTile; r += 4) {
        float s2 = 0.f;
        for (int kk = lane * 2; kk < kc; kk += 64) {
          const float2 f = __half22float2(*reinterpret_cast<const __half2*>(xs + r * S + kk));
          s2 = fmaf(f.x, f.x, fmaf(f.y, f.y, s2));
        }
        s2 = warp_sum(s2);
        if (lane == 0 && t0 + r < T) c.ss_part[(size_t)ks * T + t0 + r] = s2;
      }
    }
  }
}

__global__ void __launch_bounds__(128) route_logits_mma_kernel(FwdCtx c) {
  extern __shared__ __align__(16) uint8_t lsm[];
  pdl_wait();
  pdl_trigger();
  logits_tile(c, blockIdx.x, blockIdx.y, blockIdx.z, lsm, 128);
}

// One warp per token: sums the K slices of its logits (fixed order), then
// softmax / top-k; then the CTA counts its 8 tokens' pairs per expert
// (route_hist row = blockIdx.x) for the parallel permutation.
__global__ void __launch_bounds__(256) route_topk_kernel(FwdCtx c) {
  __shared__ float lg[8][256];
  __shared__ int hcount[256];
  pdl_wait();
  pdl_trigger();
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + w;
  for (int e = threadIdx.x; e < c.E; e += blockDim.x) hcount[e] = 0;
  if (t < c.T) {
    for (int e = lane; e < c.E; e += 32) {
      float s = 0.f;
      for (int ks0 = 0; ks0 < c.ksplit; ks0 += 8) {   // 8 independent loads in flight, summed in order
        float v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
          v[i] = ks0 + i < c.ksplit ? c.logit_part[((size_t)(ks0 + i) * c.T + t) * c.E + e] : 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) s += v[i];
      }
      lg[w][e] = s;
    }
    float r = 1.f;
    if (c.flags & 2u) {
      float ss = 0.f;
      for (int ks = 0; ks < c.ksplit; ++ks) ss += c.ss_part[(size_t)ks * c.T + t];
      r = prenorm_scale(ss, c.H);
      if (lane == 0) c.rnorm[t] = r;
    }
    __syncwarp();
    topk_token(c, t, lg[w], r, nullptr);
  }
  __syncthreads();   // this CTA's ids (global) are visible to the whole CTA
  const int p0 = blockIdx.x * 8 * c.k, p1 = min(c.T, blockIdx.x * 8 + 8) * c.k;
  for (int p = p0 + (int)threadIdx.x; p < p1; p += blockDim.x) atomicAdd(&hcount[c.ids[p]], 1);   // counts: order-free
  __syncthreads();
  for (int e = threadIdx.x; e < c.E; e += blockDim.x) c.route_hist[(size_t)blockIdx.x * c.E + e] = hcount[e];
}

// One CTA per expert: exclusive scan of the expert's counts over the 8-token
// blocks (in place: route_hist becomes the block's first row inside the
// expert's group) and the expert's total in offsets[e].  The last CTA to
// finish (arrival counter) turns the totals into the exclusive offsets and
// the active-expert lists of the grouped GEMM, and resets the counter.
__global__ void __launch_bounds__(256) route_scan_kernel(FwdCtx c) {
  __shared__ int warp_tot[8];
  __shared__ int s_last;
  pdl_wait();
  pdl_trigger();
  const int e = blockIdx.x, nb = (c.T + 7) / 8;
  const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
  const int per = (nb + 255) / 256;   // consecutive blocks per thread
  const int b0 = min(nb, tid * per), b1 = min(nb, b0 + per);
  int loc = 0;
  for (int bb = b0; bb < b1; ++bb) loc += c.route_hist[(size_t)bb * c.E + e];
  int incl = loc;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) warp_tot[w] = incl;
  __syncthreads();
  int before = 0;
  for (int ww = 0; ww < w; ++ww) before += warp_tot[ww];
  int run = before + incl - loc;   // exclusive prefix of this thread's first block
  for (int bb = b0; bb < b1; ++bb) {
    const int v = c.route_hist[(size_t)bb * c.E + e];
    c.route_hist[(size_t)bb * c.E + e] = run;
    run += v;
  }
  if (tid == 255) c.offsets[e] = before + incl;   // the expert's total (the last thread holds it)
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    s_last = atomicAdd(c.route_counter, 1u) == (unsigned)c.E - 1u;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  if (w == 0) {   // totals -> exclusive offsets, active lists (ascending experts)
    int n = 0, tiles = 0, base = 0;
    for (int e0 = 0; e0 < c.E; e0 += 32) {
      const int ex = e0 + lane;
      const int ce = ex < c.E ? __ldcg(&c.offsets[ex]) : 0;
      int ci = ce;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(kFull, ci, o);
        if (lane >= o) ci += v;
      }
      const int off = base + ci - ce;
      const int slot = ce > 0 ? c.table[ex] : -1;
      const bool act = ce > 0 && slot >= 0;
      if (ce > 0 && slot < 0) {
        atomicAdd(&c.status->miss, (unsigned long long)ce);
        atomicOr(&c.status->flags, STATUS_MISS);
      }
      const unsigned am = __ballot_sync(kFull, act);
      const int pos = n + __popc(am & ((1u << lane) - 1u));
      const int ntl = act ? (ce + c.tile_tokens - 1) / c.tile_tokens : 0;
      int ti = ntl;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(kFull, ti, o);
        if (lane >= o) ti += v;
      }
      __syncwarp();
      if (ex < c.E) c.offsets[ex] = off;
      if (act) {
        c.act_expert[pos] = ex;
        c.act_slot[pos] = slot;
        c.act_start[pos] = off;
        c.act_count[pos] = ce;
        c.act_tile[pos] = tiles + ti - ntl;
      }
      n += __popc(am);
      tiles += __shfl_sync(kFull, ti, 31);
      base += __shfl_sync(kFull, ci, 31);
    }
    if (lane == 0) {
      c.offsets[c.E] = base;
      *c.n_active = n;
      c.act_tile[n] = tiles;
      *c.route_counter = 0u;
    }
  }
}

// One CTA per 8-token block: stable scatter of its pairs.  The rank of a pair
// inside its expert group = the block's base (route_hist) + the pairs of the
// same expert earlier in the block (__match_any_sync per 32 pairs, then the
// counts of the earlier 32-pair chunks).
__global__ void __launch_bounds__(256) route_scatter_kernel(FwdCtx c) {
  __shared__ int ccount[8][256];   // [32-pair chunk][expert]
  pdl_wait();
  pdl_trigger();
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int p0 = blockIdx.x * 8 * c.k, p1 = min(c.T, blockIdx.x * 8 + 8) * c.k;
  const int nch = (p1 - p0 + 31) / 32;   // <= 8 (k <= 32)
  for (int i = threadIdx.x; i < nch * c.E; i += blockDim.x) ccount[i / c.E][i % c.E] = 0;
  __syncthreads();
  int e = -1 - lane, rank = 0;
  unsigned peers = 0;
  const int p = p0 + w * 32 + lane;
  if (w < nch) {
    e = p < p1 ? c.ids[p] : -1 - lane;
    peers = __match_any_sync(kFull, e);
    rank = __popc(peers & ((1u << lane) - 1u));
    if (p < p1 && rank == 0) ccount[w][e] = __popc(peers);
  }
  __syncthreads();
  if (w < nch && p < p1) {
    int r = rank;
    for (int ch = 0; ch < w; ++ch) r += ccount[ch][e];
    const int pos = c.offsets[e] + c.route_hist[(size_t)blockIdx.x * c.E + e] + r;
    c.sorted[pos] = p;
    c.p2r[p] = pos;
  }
}

// ------------------------------------------- cooperative router
// One cooperative launch (every CTA co-resident) routes T > 8 tokens:
//   phase 0  the logits tiles of route_logits_mma_kernel (64 tokens x 64
//            experts x 256 K each), spread over the grid;
//   phase 1  per 8-token block: softmax / top-k (warp per token, the K slices
//            summed in order) and the block's pair count per expert
//            (route_hist row b);
//   phase 2  per expert: exclusive scan of its counts over the blocks, in
//            place, and its total (route_hist row nb); skipped for at most
//            kDirectBlocks blocks, where phase 3 sums the counts itself;
//   phase 3  every CTA turns the totals into the expert offsets; CTA 0 also
//            publishes them with the active-expert lists; per 8-token block,
//            the stable scatter of its pairs and (when xp is set: the
//            grouped-GEMM family) the copy of its tokens' x rows to their
//            sorted rows of xp (each x row read once, written k times).
// Bounded grid barriers separate the phases.  Same results as the separate
// logits, top-k, scan and scatter launches plus the gather kernel.

DEV_INLINE unsigned long long ld_acquire_u64_gpu(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

// Bounded barrier over the grid, called by thread 0 of each CTA: one arrival
// on a monotonic 64-bit counter, then a poll until it reaches the next
// multiple of the grid size.  Each counter is only ever used with one grid
// size, so every launch leaves it at a multiple.  False after about 1 s
// (STATUS_TIMEOUT set).
DEV_INLINE bool coop_grid_barrier(unsigned long long* ctr, unsigned nblocks, DevStatus* st) {
  __threadfence();
  const unsigned long long old = atomicAdd(ctr, 1ull);
  const unsigned long long target = (old / nblocks + 1ull) * nblocks;
  const long long t0 = clock64();
  while (ld_acquire_u64_gpu(ctr) < target) {
    if (clock64() - t0 > MOE_WAIT_CYCLES) {
      atomicOr(&st->flags, STATUS_TIMEOUT);
      return false;
    }
    __nanosleep(64);
  }
  __threadfence();
  return true;
}

// Up to this many 8-token blocks, every CTA sums the expert counts of the
// blocks itself (no per-expert scan phase, one grid barrier less), and the
// grid is one CTA per SM (barrier counter 0); above, two CTAs per SM where
// they fit (counter 1).
constexpr int kDirectBlocks = 64;

// CL: the same phases on one thread-block cluster of kRouteClusterCTAs CTAs
// (launched with programmatic dependent launch), the phase barriers being the
// hardware cluster barrier (release / acquire at cluster scope, which orders
// the global writes of one phase before the reads of the next): no grid-wide
// counter round trips, for the few token blocks of 16 < T <= 64.
constexpr int kRouteClusterCTAs = 8;
constexpr int kRouteClusterMaxT = 64;
static_assert(kDirectBlocks * 256 * 4 <= kLogitSmem, "block counts fit the logits tile's shared memory");

template <bool CL>
__global__ void __launch_bounds__(256) route_coop_kernel(FwdCtx c) {
  extern __shared__ __align__(16) uint8_t csm[];   // one logits tile (phase 0)
  __shared__ float lg[8][256];
  __shared__ int cnt[8][256];   // phase 1: row 0 = the block's counts; phase 3: per 32-pair chunk
  __shared__ int s_off[256];
  __shared__ int s_tot[256];    // per expert: pairs routed to it
  __shared__ int s_base[256];   // per expert: its pairs in blocks before the current one
  __shared__ int s_pos[256];
  __shared__ int warp_tot[8];
  __shared__ int s_ok;
  const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
  const int T = c.T, E = c.E, k = c.k, nb = (T + 7) / 8, G = (int)gridDim.x;
  const bool direct = nb <= kDirectBlocks;
  unsigned long long* bar = c.route_bar + (direct ? 0 : 1);   // one grid size per counter
  if (tid == 0) s_ok = 1;
  if (CL) {
    pdl_wait();      // x may be the output of the preceding grid
    pdl_trigger();
  }
  // every CTA of the grid (cluster) has finished the phase before; false after
  // a timed-out grid barrier (the cluster barrier has no time-out: every CTA
  // of a cluster is co-scheduled and arrives)
  auto phase_sync = [&]() -> bool {
    if (CL) {
      __syncthreads();
      cluster_sync();
      return true;
    }
    __syncthreads();
    if (tid == 0 && !coop_grid_barrier(bar, (unsigned)G, c.status)) s_ok = 0;
    __syncthreads();
    return s_ok != 0;
  };

  // ---------------------------------------------- phase 0: logits tiles
  {
    const int ntt = (T + kRouteTile - 1) / kRouteTile, net = (E + kRouteTile - 1) / kRouteTile;
    const int ntiles = ntt * net * c.ksplit;
    for (int ti = blockIdx.x; ti < ntiles; ti += G) {
      __syncthreads();   // the previous tile's shared memory is free
      const int ks = ti % c.ksplit, rest = ti / c.ksplit;
      logits_tile(c, rest / net, rest % net, ks, csm, 256);
    }
  }
  if (!phase_sync()) return;

  // ---------------------------------------------- phase 1: top-k, counts
  for (int b = blockIdx.x; b < nb; b += G) {
    __syncthreads();
    for (int e = tid; e < E; e += 256) cnt[0][e] = 0;
    const int t = b * 8 + w;
    if (t < T) {
      for (int e = lane; e < E; e += 32) {
        float sum = 0.f;
        for (int ks0 = 0; ks0 < c.ksplit; ks0 += 8) {   // 8 loads in flight, summed in slice order
          float v[8];
#pragma unroll
          for (int i = 0; i < 8; ++i)
            v[i] = ks0 + i < c.ksplit ? __ldcg(&c.logit_part[((size_t)(ks0 + i) * T + t) * E + e]) : 0.f;
#pragma unroll
          for (int i = 0; i < 8; ++i) sum += v[i];
        }
        lg[w][e] = sum;
      }
      float r = 1.f;
      if (c.flags & 2u) {
        float ss = 0.f;
        for (int ks = 0; ks < c.ksplit; ++ks) ss += __ldcg(&c.ss_part[(size_t)ks * T + t]);
        r = prenorm_scale(ss, c.H);
        if (lane == 0) c.rnorm[t] = r;
      }
      __syncwarp();
      topk_token(c, t, lg[w], r, nullptr);
    }
    __syncthreads();   // the block's ids (global) are visible to the whole CTA
    const int p0 = b * 8 * k, p1 = min(T, b * 8 + 8) * k;
    for (int p = p0 + tid; p < p1; p += 256) atomicAdd(&cnt[0][c.ids[p]], 1);   // counts: order-free
    __syncthreads();
    for (int e = tid; e < E; e += 256) c.route_hist[(size_t)b * E + e] = cnt[0][e];
  }
  if (!phase_sync()) return;

  // ---------------------------------------------- phase 2: per-expert scan
  // (many blocks only; up to kDirectBlocks, phase 3 sums the counts directly)
  const int per = (nb + 255) / 256;   // consecutive blocks per thread
  for (int e = blockIdx.x; !direct && e < E; e += G) {
    const int b0 = min(nb, tid * per), b1 = min(nb, b0 + per);
    int loc = 0;
    for (int bb = b0; bb < b1; ++bb) loc += __ldcg(&c.route_hist[(size_t)bb * E + e]);
    int incl = loc;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(kFull, incl, o);
      if (lane >= o) incl += n;
    }
    if (lane == 31) warp_tot[w] = incl;
    __syncthreads();
    int before = 0;
    for (int ww = 0; ww < w; ++ww) before += warp_tot[ww];
    int run = before + incl - loc;   // exclusive prefix of this thread's first block
    for (int bb = b0; bb < b1; ++bb) {
      const int v = __ldcg(&c.route_hist[(size_t)bb * E + e]);
      c.route_hist[(size_t)bb * E + e] = run;
      run += v;
    }
    if (tid == 255) c.route_hist[(size_t)nb * E + e] = before + incl;   // the expert's total
    __syncthreads();   // warp_tot reuse
  }
  if (!direct && !phase_sync()) return;
  // Up to kDirectBlocks blocks: every block's counts into shared memory (the
  // logits tile's space, free since phase 0) with one coalesced pass, so the
  // totals and each block's bases below are sums over shared memory.
  int* hist_s = reinterpret_cast<int*>(csm);   // [nb][E], nb * E * 4 <= kLogitSmem
  if (direct) {
    for (int i = tid; i < nb * E; i += 256) hist_s[i] = __ldcg(&c.route_hist[i]);
    __syncthreads();
  }
  for (int e = tid; e < E; e += 256) {   // the experts' totals
    int tot = 0;
    if (direct)
      for (int bb = 0; bb < nb; ++bb) tot += hist_s[bb * E + e];
    else
      tot = __ldcg(&c.route_hist[(size_t)nb * E + e]);
    s_tot[e] = tot;
  }
  __syncthreads();

  // ---------------------------------------------- phase 3: offsets, scatter, x rows
  if (w == 0) {   // totals -> exclusive offsets (every CTA); CTA 0 publishes them and the active lists
    const bool pub = blockIdx.x == 0;
    int n = 0, tiles = 0, base = 0;
    for (int e0 = 0; e0 < E; e0 += 32) {
      const int ex = e0 + lane;
      const int ce = ex < E ? s_tot[ex] : 0;
      int ci = ce;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(kFull, ci, o);
        if (lane >= o) ci += v;
      }
      const int off = base + ci - ce;
      if (ex < E) s_off[ex] = off;
      if (pub) {
        const int slot = ce > 0 ? c.table[ex] : -1;
        const bool act = ce > 0 && slot >= 0;
        if (ce > 0 && slot < 0) {
          atomicAdd(&c.status->miss, (unsigned long long)ce);
          atomicOr(&c.status->flags, STATUS_MISS);
        }
        const unsigned am = __ballot_sync(kFull, act);
        const int pos = n + __popc(am & ((1u << lane) - 1u));
        const int ntl = act ? (ce + c.tile_tokens - 1) / c.tile_tokens : 0;
        int ti = ntl;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int v = __shfl_up_sync(kFull, ti, o);
          if (lane >= o) ti += v;
        }
        if (ex < E) c.offsets[ex] = off;
        if (act) {
          c.act_expert[pos] = ex;
          c.act_slot[pos] = slot;
          c.act_start[pos] = off;
          c.act_count[pos] = ce;
          c.act_tile[pos] = tiles + ti - ntl;
        }
        n += __popc(am);
        tiles += __shfl_sync(kFull, ti, 31);
      }
      base += __shfl_sync(kFull, ci, 31);
    }
    if (pub && lane == 0) {
      c.offsets[E] = base;
      *c.n_active = n;
      c.act_tile[n] = tiles;
    }
  }
  const int vpr = c.H / 8;   // 16-byte vectors per x row
  for (int b = blockIdx.x; b < nb; b += G) {
    __syncthreads();   // s_off ready; cnt, s_pos reuse
    const int p0 = b * 8 * k, p1 = min(T, b * 8 + 8) * k;
    const int nch = (p1 - p0 + 31) / 32;   // <= 8 (k <= 32)
    for (int i = tid; i < nch * E; i += 256) cnt[i / E][i % E] = 0;
    for (int e = tid; e < E; e += 256) {   // the block's first row inside each expert's group
      int base = 0;
      if (direct)
        for (int bb = 0; bb < b; ++bb) base += hist_s[bb * E + e];
      else
        base = __ldcg(&c.route_hist[(size_t)b * E + e]);
      s_base[e] = base;
    }
    __syncthreads();
    int e = -1 - lane, rank = 0;
    const int p = p0 + w * 32 + lane;
    if (w < nch) {
      e = p < p1 ? c.ids[p] : -1 - lane;
      const unsigned peers = __match_any_sync(kFull, e);
      rank = __popc(peers & ((1u << lane) - 1u));
      if (p < p1 && rank == 0) cnt[w][e] = __popc(peers);
    }
    __syncthreads();
    if (w < nch && p < p1) {
      int r = rank;
      for (int ch = 0; ch < w; ++ch) r += cnt[ch][e];
      const int pos = s_off[e] + s_base[e] + r;
      c.sorted[pos] = p;
      c.p2r[p] = pos;
      s_pos[p - p0] = pos;
    }
    __syncthreads();
    const int ntok = min(8, T - b * 8);
    for (int v = tid; c.xp && v < vpr; v += 256) {
      uint4 xv[8];
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (j < ntok) xv[j] = __ldg(reinterpret_cast<const uint4*>(c.x + (size_t)(b * 8 + j) * c.H) + v);
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (j < ntok)
          for (int kk = 0; kk < k; ++kk) reinterpret_cast<uint4*>(c.xp + (size_t)s_pos[j * k + kk] * c.H)[v] = xv[j];
    }
  }
}

}  // namespace

bool route_single_launch(const FwdCtx& c) { return route_cluster_smem(c.T, c.E, c.H, c.k) <= 200 * 1024; }

cudaError_t launch_route(const FwdCtx& c, bool small, cudaStream_t st) {
  const size_t smem_small = route_cluster_smem(c.T, c.E, c.H, c.k);
  if (small && route_single_launch(c)) {
    int C = (c.E + kLogitWarps - 1) / kLogitWarps;
    if (C > kMaxCluster) C = kMaxCluster;
    cudaError_t e = opt_in_smem((const void*)route_cluster_kernel, smem_small);
    if (e != cudaSuccess) return e;
    return launch_pdl(route_cluster_kernel, dim3(C), dim3(256), smem_small, st, C, c);
  }
  FwdCtx cc = c;
  cc.ksplit = (c.H + kRouteKC - 1) / kRouteKC;
  const size_t lsmem = (size_t)2 * kRouteTile * (kRouteKC + 8) * sizeof(__half);
  cudaError_t e = opt_in_smem((const void*)route_logits_mma_kernel, lsmem);
  if (e != cudaSuccess) return e;
  const dim3 grid((c.T + kRouteTile - 1) / kRouteTile, (c.E + kRouteTile - 1) / kRouteTile, cc.ksplit);
  e = launch_pdl(route_logits_mma_kernel, grid, dim3(128), lsmem, st, 1, cc);
  if (e == cudaSuccess) e = launch_pdl(route_topk_kernel, dim3((c.T + 7) / 8), dim3(256), 0, st, 1, cc);
  if (e == cudaSuccess) e = launch_pdl(route_scan_kernel, dim3(c.E), dim3(256), 0, st, 1, cc);
  if (e == cudaSuccess) e = launch_pdl(route_scatter_kernel, dim3((c.T + 7) / 8), dim3(256), 0, st, 1, cc);
  return e;
}

cudaError_t launch_route_gather(const FwdCtx& c, bool gather, cudaStream_t st) {
  FwdCtx cc = c;
  if (!gather) cc.xp = nullptr;
  cc.ksplit = (c.H + kRouteKC - 1) / kRouteKC;
  if (c.T <= kRouteClusterMaxT) {
    cudaError_t e = opt_in_smem((const void*)route_coop_kernel<true>, kLogitSmem);
    if (e != cudaSuccess) return e;
    return launch_pdl(route_coop_kernel<true>, dim3(kRouteClusterCTAs), dim3(256), kLogitSmem, st, kRouteClusterCTAs,
                      cc);
  }
  cudaError_t e = opt_in_smem((const void*)route_coop_kernel<false>, kLogitSmem);
  if (e != cudaSuccess) return e;
  int per_sm = 0;   // all CTAs of the cooperative launch must be co-resident
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, route_coop_kernel<false>, 256, kLogitSmem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1 || c.num_sms < 1) return cudaErrorNotSupported;
  // the grid size belongs to the barrier counter the kernel picks (fixed per
  // counter); grid-stride loops cover any T
  const int nb = (c.T + 7) / 8;
  const int G = nb <= kDirectBlocks ? c.num_sms : c.num_sms * (per_sm >= 2 ? 2 : 1);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)G);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = kLogitSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, route_coop_kernel<false>, cc);
}
