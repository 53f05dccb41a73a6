// Fused decode-regime layer: one cooperative persistent launch per forward
// (router -> top-k -> permutation -> gate/up -> SiLU*up -> down -> combine),
// in the spirit of a fused small-batch executor ("top4-fused-v1" is named on
// "Horizon RunMap - architecture", "Regimes and executor boundaries"; its
// design is not published).
//
// Grid = one CTA per SM, all co-resident (cooperative launch).  A CTA has 12
// compute warps in 3 groups of 4 and one producer warp.
//   phase 0  the grid's warps take the (token, expert, K half) dot products of
//            the router (and per-token sums of squares for PRENORM) -> global;
//            bounded two-level grid barrier
//   phase 0b every CTA reads the logits and does softmax / top-k and the
//            stable permutation itself in shared memory (CTA 0 publishes it),
//            and stages the T token rows of x in shared memory
//   phase 1  the CTA's share of (expert, 16-row tile) gate/up items; the
//            producer streams their compact tiles and, right behind them, the
//            CTA's down tiles (independent of h) through 3 bulk-copy slots;
//            warp group q computes the items of slot q; h = SiLU(g) * u ->
//            global (FP16); bounded grid barrier among the compute warps
//   phase 2  the CTA's (expert, 64-row block) down items (a warp per 16-row
//            tile, whole K, the item's h rows staged by its group) -> y (FP32);
//            the last item to finish a 64-row block of H (arrival counter)
//            gathers the combine in rank order.
// Weights stay 4-bit until a warp dequantises a 16-byte chunk in registers
// for one MMA step (FP16 operands, FP32 accumulation).  Every wait is
// bounded: on timeout the status word records it and the CTA leaves.
#include "gemv_dev.cuh"
#include "route_dev.cuh"

namespace {
using namespace gemv_dev;
using namespace route_dev;

constexpr int kGroups = 3;                     // warp groups = ring slots
constexpr int kGW = 4;                         // warps per group
constexpr int kCW = kGroups * kGW;             // compute warps
constexpr int kFThreads = (kCW + 1) * 32;      // + producer warp
constexpr int kDownRows = 64;                  // rows of H per down item (4 tiles)
constexpr int kMaxT = 16;                      // tokens of the fused path (all staged in smem)
constexpr int kMaxP = kMaxT * 32;

constexpr uint32_t kSmemBudget = 226 * 1024;

struct FusedSmem {
  uint32_t ns, slot_bytes, off_x, x_bytes, off_red, off_route, total;
};

// Shared memory of the fused kernel for a batch of T tokens, top-k: ns weight
// slots (4 when they fit, else 3) feeding the 3 compute groups, the x rows /
// per-group h rows, the cross-warp reduction buffer, and the routing state.
__host__ __device__ inline FusedSmem fused_smem(const SlotLayout& lay, int H, int I, int E, int T, int k) {
  FusedSmem f;
  const uint32_t sg = 2 * lay.gate.tile_bytes, sd = (kDownRows / 16) * lay.down.tile_bytes;
  f.slot_bytes = ((sg > sd ? sg : sd) + 127) / 128 * 128;
  const int hrows = T < kTok ? T : kTok;
  // phase 1: x [T][H + 8]; phase 2: per group h [hrows][I + 8]
  const uint32_t xa = (uint32_t)T * (H + 8) * 2, ha = (uint32_t)kGroups * hrows * (I + 8) * 2;
  f.x_bytes = ((xa > ha ? xa : ha) + 127) / 128 * 128;
  const int P = T * k;
  // logits [T][E] | ids, topw, sorted [P] | rnorm [T] | table, cnt, off [E + 1]
  // | active slot, start, count [E + 1] | chunk counts [ceil(P/32)][E] | misc
  const uint32_t route = (uint32_t)(T * E + 3 * P + T + 6 * (E + 1) + ((P + 31) / 32) * E + 8) * 4;
  for (f.ns = 4; f.ns >= 3; --f.ns) {
    f.off_x = f.ns * f.slot_bytes;
    f.off_red = f.off_x + f.x_bytes;
    f.off_route = f.off_red + kGroups * kGW * 2 * 16 * kTok * 4;
    f.total = f.off_route + route;
    if (f.total <= kSmemBudget) break;
  }
  return f;
}

DEV_INLINE unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Bounded barrier over all CTAs of the grid, called by one thread per CTA.
// Arrivals go to one of 8 sub-counters; the last arrival of a sub-counter
// arrives on the top counter; the last top arrival resets both levels and
// bumps the generation word the others poll.  w: [10] = 8 sub-counters,
// top counter, generation.
DEV_INLINE bool grid_sync_one(unsigned* w, unsigned nblocks, DevStatus* st) {
  unsigned* gen = w + 9;
  const unsigned g0 = ld_acquire(gen);
  const unsigned grp = blockIdx.x & 7u;
  const unsigned in_grp = (nblocks - grp + 7u) / 8u;   // CTAs b with b % 8 == grp
  const unsigned ngrp = nblocks < 8u ? nblocks : 8u;
  __threadfence();
  if (atomicAdd(&w[grp], 1u) == in_grp - 1u) {
    w[grp] = 0u;
    if (atomicAdd(&w[8], 1u) == ngrp - 1u) {
      w[8] = 0u;
      __threadfence();
      atomicAdd(gen, 1u);
      return true;
    }
  }
  const long long t0 = clock64();
  while (ld_acquire(gen) == g0) {
    if (clock64() - t0 > MOE_WAIT_CYCLES) {
      atomicOr(&st->flags, STATUS_TIMEOUT);
      return false;
    }
    __nanosleep(20);
  }
  return true;
}

DEV_INLINE void named_sync(int id, int nthreads) { asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory"); }

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

// Stage rows (global, row pointers from rowptr(i)) into smem [n][stride] with
// nthr threads (this one is t0); 4 independent 16-byte loads in flight each.
template <typename RowFn>
DEV_INLINE void stage(__half* dst, int stride, int K, int n, RowFn rowptr, int t0, int nthr) {
  const int vpr = K / 8, tot = n * vpr;
  for (int i0 = 0; i0 < tot; i0 += 4 * nthr) {
    uint4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = i0 + u * nthr + t0;
      if (i < tot) v[u] = __ldg(reinterpret_cast<const uint4*>(rowptr(i / vpr)) + i % vpr);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = i0 + u * nthr + t0;
      if (i < tot) *(reinterpret_cast<uint4*>(dst + (i / vpr) * stride) + i % vpr) = v[u];
    }
  }
}

// acc[m] += rows of tile[m] (16 x K) x B, the lane's B row in smem (brow,
// NULL = zero row), over chunks kc0, kc0 + kstride, ... < nkc.
template <int NMAT>
DEV_INLINE void mma_tiles_s(float (&acc)[2][4], const uint8_t* const (&tile)[2], uint32_t scale_bytes,
                            const __half* brow, int lane, int kc0, int kstride, int nkc) {
  const int g = lane >> 2, c = lane & 3;
  for (int kc = kc0; kc < nkc; kc += kstride) {
    uint4 q[NMAT];
    __half2 slo[NMAT], shi[NMAT];
#pragma unroll
    for (int m = 0; m < NMAT; ++m) {
      q[m] = *reinterpret_cast<const uint4*>(tile[m] + scale_bytes + ((size_t)kc * 32 + lane) * 16);
      const __half* sc = reinterpret_cast<const __half*>(tile[m]) + (kc >> 2) * 16;
      slo[m] = __half2half2(sc[g]);
      shi[m] = __half2half2(sc[g + 8]);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int k0 = kc * 64 + j * 16 + 2 * c;
      const uint32_t b0 = brow ? *reinterpret_cast<const uint32_t*>(brow + k0) : 0u;
      const uint32_t b1 = brow ? *reinterpret_cast<const uint32_t*>(brow + k0 + 8) : 0u;
#pragma unroll
      for (int m = 0; m < NMAT; ++m) {
        const uint32_t w = j == 0 ? q[m].x : j == 1 ? q[m].y : j == 2 ? q[m].z : q[m].w;
        uint32_t a[4];
        dequant_word(w, slo[m], shi[m], a);
        mma_16816(acc[m], a, b0, b1);
      }
    }
  }
}

__global__ void __launch_bounds__(kFThreads, 1) fused_decode_kernel(FwdCtx c) {
  extern __shared__ __align__(128) uint8_t sm[];
  __shared__ __align__(8) uint64_t full[4], empty[4], xbar;
  __shared__ int s_ok;
  __shared__ int s_gok[kGroups];
  __shared__ unsigned s_last[kGroups];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x, b = blockIdx.x;
  const int T = c.T, E = c.E, H = c.H, I = c.I, k = c.k, P = T * k;
  const FusedSmem L = fused_smem(c.lay, H, I, E, T, k);
  __half* xcache = reinterpret_cast<__half*>(sm + L.off_x);
  float* red = reinterpret_cast<float*>(sm + L.off_red);
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
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(&xbar, 1);
    fence_mbar_init();
    // the T token rows of x, staged once (padded rows) for every gate/up item
    // of this CTA; the copies run while the router phase computes
    mbar_expect_tx(&xbar, (uint32_t)T * H * 2);
    for (int t = 0; t < T; ++t) bulk_g2s(xcache + (size_t)t * (H + 8), c.x + (size_t)t * H, (uint32_t)H * 2, &xbar);
  }
  for (int e = tid; e < E; e += blockDim.x) r_table[e] = c.table[e];

  // ---------------------------------------------------------------- phase 0
  {
    const int half = ((H / 2) + 255) / 256 * 256;   // K split point (multiple of 256)
    const int nt = 2 * T * E + ((c.flags & 2u) ? 2 * T : 0);
    for (int task = b * (kCW + 1) + warp; task < nt; task += G * (kCW + 1)) {
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
  if (tid == 0 && !grid_sync_one(c.grid_sync, G, c.status)) s_ok = 0;
  __syncthreads();
  if (!s_ok) return;

  // --------------------------------------------------------------- phase 0b
  for (int i = tid; i < T * E; i += blockDim.x) lg[i] = __ldcg(&c.logit_part[i]) + __ldcg(&c.logit_part[T * E + i]);
  if (c.flags & 2u)
    for (int t = tid; t < T; t += blockDim.x)
      r_rnorm[t] = prenorm_scale(__ldcg(&c.ss_part[t]) + __ldcg(&c.ss_part[T + t]), H);
  for (int e = tid; e < ((P + 31) / 32) * E; e += blockDim.x) r_chunk[e] = 0;
  __syncthreads();
  {
    FwdCtx cl = c;   // top-k results go to shared memory
    cl.ids = r_ids;
    cl.topw = r_w;
    for (int t = warp; t < T; t += kCW + 1)
      topk_token(cl, t, lg + t * E, (c.flags & 2u) ? r_rnorm[t] : 1.f, nullptr);
  }
  __syncthreads();
  // counts per 32-pair chunk: __match_any_sync groups equal ids (no atomics)
  const int nchunk = (P + 31) / 32;
  for (int ch = warp; ch < nchunk; ch += kCW + 1) {
    const int p = ch * 32 + lane;
    const int e = p < P ? r_ids[p] : -1 - lane;
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    if (p < P && __popc(peers & ((1u << lane) - 1u)) == 0) r_chunk[ch * E + e] = __popc(peers);
  }
  __syncthreads();
  if (warp == 0) {   // counts, exclusive scan, active list (ascending experts)
    const int per = (E + 31) / 32;
    int local[kMaxEPL];
    int s = 0;
#pragma unroll
    for (int i = 0; i < kMaxEPL; ++i) {
      const int e = lane * per + i;
      local[i] = s;
      if (i < per && e < E) {
        int ce = 0;
        for (int ch = 0; ch < nchunk; ++ch) ce += r_chunk[ch * E + e];
        r_cnt[e] = ce;
        s += ce;
      }
    }
    int incl = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(kFull, incl, o);
      if (lane >= o) incl += n;
    }
    const int excl = incl - s;
#pragma unroll
    for (int i = 0; i < kMaxEPL; ++i) {
      const int e = lane * per + i;
      if (i < per && e < E) r_off[e] = excl + local[i];
    }
    if (lane == 31) r_off[E] = incl;
    __syncwarp();
    int n = 0;
    for (int e0 = 0; e0 < E; e0 += 32) {
      const int e = e0 + lane;
      const int ce = e < E ? r_cnt[e] : 0;
      const int slot = ce > 0 ? r_table[e] : -1;
      const bool act = ce > 0 && slot >= 0;
      if (b == 0 && ce > 0 && slot < 0) {
        atomicAdd(&c.status->miss, (unsigned long long)ce);
        atomicOr(&c.status->flags, STATUS_MISS);
      }
      const unsigned am = __ballot_sync(kFull, act);
      const int pos = n + __popc(am & ((1u << lane) - 1u));
      if (act) {
        r_aslot[pos] = slot;
        r_astart[pos] = r_off[e];
        r_acount[pos] = ce;
      }
      n += __popc(am);
    }
    if (lane == 0) r_misc[0] = n;
  }
  __syncthreads();
  // stable scatter: rank = same-expert pairs in earlier chunks + rank inside the chunk
  for (int ch = warp; ch < nchunk; ch += kCW + 1) {
    const int p = ch * 32 + lane;
    const int e = p < P ? r_ids[p] : -1 - lane;
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    if (p < P) {
      int rank = __popc(peers & ((1u << lane) - 1u));
      for (int c2 = 0; c2 < ch; ++c2) rank += r_chunk[c2 * E + e];
      r_sorted[r_off[e] + rank] = p;
    }
  }
  __syncthreads();
  if (tid == 0 && !mbar_wait_bounded(&xbar, 0, c.status)) s_ok = 0;
  if (b == 0) {   // publish the routing (debug outputs, rnorm)
    for (int i = tid; i < P; i += blockDim.x) {
      c.ids[i] = r_ids[i];
      c.topw[i] = r_w[i];
      c.sorted[i] = r_sorted[i];
    }
    for (int i = tid; i <= E; i += blockDim.x) c.offsets[i] = r_off[i];
    if (c.flags & 2u)
      for (int i = tid; i < T; i += blockDim.x) c.rnorm[i] = r_rnorm[i];
  }

  // --------------------------------------------------------- phases 1 and 2
  __syncthreads();
  if (!s_ok) return;
  const int U = r_misc[0];
  if (U == 0) {   // every routed expert is absent: out = residual or 0
    for (int i = b * blockDim.x + tid; i < T * H; i += G * blockDim.x)
      c.out[i] = (c.flags & 1u) ? c.x[i] : __float2half_rn(0.f);
    return;
  }
  const int tpe1 = I / 16, tpe2 = H / kDownRows;
  const int n1 = U * tpe1, n2 = U * tpe2;
  const int a1 = (int)((long long)b * n1 / G), m1 = (int)((long long)(b + 1) * n1 / G) - a1;
  const int a2 = (int)((long long)b * n2 / G), m2 = (int)((long long)(b + 1) * n2 / G) - a2;

  if (warp == kCW) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      for (int j = 0; j < m1 + m2; ++j) {
        const int s = j % NS;
        const uint32_t par = (uint32_t)((j / NS) & 1);
        if (!mbar_wait_bounded(&empty[s], par ^ 1u, c.status)) break;
        uint8_t* dst = sm + (size_t)s * L.slot_bytes;
        if (j < m1) {
          const int it = a1 + j, u = it / tpe1, rt = it % tpe1;
          const uint8_t* base = c.pool + (size_t)r_aslot[u] * c.slot_bytes;
          const uint32_t TS = c.lay.gate.tile_bytes;
          mbar_expect_tx(&full[s], 2 * TS);
          bulk_g2s(dst, tile_ptr(base, c.lay.gate, rt), TS, &full[s]);
          bulk_g2s(dst + TS, tile_ptr(base, c.lay.up, rt), TS, &full[s]);
        } else {
          const int it = a2 + (j - m1), u = it / tpe2, hb = it % tpe2;
          const uint8_t* base = c.pool + (size_t)r_aslot[u] * c.slot_bytes;
          const uint32_t TS = c.lay.down.tile_bytes;   // the 4 row tiles of a block are contiguous
          mbar_expect_tx(&full[s], (kDownRows / 16) * TS);
          bulk_g2s(dst, tile_ptr(base, c.lay.down, hb * (kDownRows / 16)), (kDownRows / 16) * TS, &full[s]);
        }
      }
    }
    return;
  }

  // ---------------------------------------------------------------- compute
  const int q = warp / kGW, wq = warp % kGW;   // group, warp in group
  const int gtid = tid - q * kGW * 32;         // thread index inside the group
  const int g = lane >> 2, cc = lane & 3;
  const int gbar = 2 + q;                      // named barrier of group q
  bool ok = true;
  // phase 1: items j = q, q + 3, ... < m1 (slot q); B = token rows of xcache
  for (int j = q; j < m1 && ok; j += kGroups) {
    const int s = j % NS;
    const uint32_t par = (uint32_t)((j / NS) & 1);
    const int it = a1 + j, u = it / tpe1, rt = it % tpe1;
    const int start = r_astart[u], cnt = r_acount[u];
    const uint8_t* slot = sm + (size_t)s * L.slot_bytes;
    const uint8_t* const tiles[2] = {slot, slot + c.lay.gate.tile_bytes};
    // one thread per group waits (bounded); the group barrier shares the outcome
    if (gtid == 0) s_gok[q] = mbar_wait_bounded(&full[s], par, c.status) ? 1 : 0;
    named_sync(gbar, kGW * 32);
    if (!s_gok[q]) {
      ok = false;
      break;
    }
    float* rg = red + q * kGW * 2 * 16 * kTok;
    for (int p0 = 0; p0 < cnt; p0 += kTok) {
      const int np = min(kTok, cnt - p0);
      const __half* brow = g < np ? xcache + (size_t)(r_sorted[start + p0 + g] / k) * (H + 8) : nullptr;
      float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      mma_tiles_s<2>(acc, tiles, c.lay.gate.scale_bytes, brow, lane, wq, kGW, H / 64);
      float* rw = rg + wq * 2 * 16 * kTok;
#pragma unroll
      for (int m = 0; m < 2; ++m) {
        rw[(m * 16 + g) * kTok + 2 * cc] = acc[m][0];
        rw[(m * 16 + g) * kTok + 2 * cc + 1] = acc[m][1];
        rw[(m * 16 + g + 8) * kTok + 2 * cc] = acc[m][2];
        rw[(m * 16 + g + 8) * kTok + 2 * cc + 1] = acc[m][3];
      }
      named_sync(gbar, kGW * 32);
      {   // 128 threads = 16 rows x 8 tokens
        const int row = gtid / kTok, tok = gtid % kTok;
        if (tok < np) {
          float gs = 0.f, us = 0.f;
#pragma unroll
          for (int ww = 0; ww < kGW; ++ww) {
            gs += rg[(ww * 2 + 0) * 16 * kTok + row * kTok + tok];
            us += rg[(ww * 2 + 1) * 16 * kTok + row * kTok + tok];
          }
          if (c.flags & 2u) {
            const float r = r_rnorm[r_sorted[start + p0 + tok] / k];
            gs *= r;
            us *= r;
          }
          c.hbuf[(size_t)(start + p0 + tok) * I + rt * 16 + row] = __float2half_rn(silu_mul(gs, us));
        }
      }
      named_sync(gbar, kGW * 32);
    }
    if (gtid == 0) mbar_arrive(&empty[s]);
  }
  // every CTA passes here exactly once: all h written before any down item reads it
  __threadfence();
  named_sync(1, kCW * 32);
  if (tid == 0 && !grid_sync_one(c.grid_sync + 10, G, c.status)) s_ok = 0;
  named_sync(1, kCW * 32);
  if (!s_ok || !ok) return;
  // phase 2: items j in [m1, m1 + m2) sit in slot j % 3; group q takes j % 3 == q
  __half* hs = xcache + (size_t)q * (T < kTok ? T : kTok) * (I + 8);   // this group's h rows
  for (int j = m1 + ((q - m1 % kGroups + kGroups) % kGroups); j < m1 + m2 && ok; j += kGroups) {
    const int s = j % NS;
    const uint32_t par = (uint32_t)((j / NS) & 1);
    const int it = a2 + (j - m1), u = it / tpe2, hb = it % tpe2;
    const int start = r_astart[u], cnt = r_acount[u];
    const uint8_t* slot = sm + (size_t)s * L.slot_bytes;
    const uint8_t* const tiles[2] = {slot + (size_t)wq * c.lay.down.tile_bytes, nullptr};
    for (int p0 = 0; p0 < cnt; p0 += kTok) {
      const int np = min(kTok, cnt - p0);
      named_sync(gbar, kGW * 32);   // previous pass done with hs
      stage(hs, I + 8, I, np, [&](int r) { return c.hbuf + (size_t)(start + p0 + r) * I; }, gtid, kGW * 32);
      if (p0 == 0 && gtid == 0) s_gok[q] = mbar_wait_bounded(&full[s], par, c.status) ? 1 : 0;
      named_sync(gbar, kGW * 32);
      if (!s_gok[q]) {
        ok = false;
        break;
      }
      const __half* brow = g < np ? hs + (size_t)g * (I + 8) : nullptr;
      float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      mma_tiles_s<1>(acc, tiles, c.lay.down.scale_bytes, brow, lane, 0, 1, I / 64);
      // accumulator (row g / g+8 of tile wq, token 2cc / 2cc+1) -> y
      const int hrow = hb * kDownRows + wq * 16 + g;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int tok = 2 * cc + (i & 1);
        if (tok < np) c.ybuf[(size_t)r_sorted[start + p0 + tok] * H + hrow + (i >= 2 ? 8 : 0)] = acc[0][i];
      }
    }
    if (!ok) break;
    // the last of the U items of this 64-row block gathers the combine
    __threadfence();
    named_sync(gbar, kGW * 32);
    if (gtid == 0) {
      mbar_arrive(&empty[s]);
      s_last[q] = (atomicAdd(&c.down_counters[hb], 1u) == (unsigned)U - 1u) ? 1u : 0u;
    }
    named_sync(gbar, kGW * 32);
    if (s_last[q]) {
      __threadfence();
      const bool residual = c.flags & 1u;
      for (int i = gtid; i < T * kDownRows; i += kGW * 32) {
        const int t = i / kDownRows, hr = hb * kDownRows + (i % kDownRows);
        float acc = residual ? __half2float(c.x[(size_t)t * H + hr]) : 0.f;
        for (int jj = 0; jj < k; ++jj) {
          const int p = t * k + jj;
          if (r_table[r_ids[p]] >= 0) acc = fmaf(r_w[p], __ldcg(&c.ybuf[(size_t)p * H + hr]), acc);
        }
        c.out[(size_t)t * H + hr] = __float2half_rn(acc);
      }
      if (gtid == 0) c.down_counters[hb] = 0u;
    }
  }
}

}  // namespace

// The fused kernel applies to small decode batches (every token row staged
// in shared memory) whose routing state fits next to the weight slots.
bool fused_decode_supported(const FwdCtx& c, int max_smem) {
  if (c.T > kMaxT || c.T * c.k > kMaxP || c.H % kDownRows || c.I % 64 || c.k > 32) return false;
  const FusedSmem L = fused_smem(c.lay, c.H, c.I, c.E, c.T, c.k);
  return L.total <= kSmemBudget && (int)L.total <= max_smem;
}

cudaError_t launch_fused_decode(const FwdCtx& c, cudaStream_t st, const StageEvents& se) {
  const FusedSmem L = fused_smem(c.lay, c.H, c.I, c.E, c.T, c.k);
  cudaError_t e = opt_in_smem((const void*)fused_decode_kernel, L.total);
  if (e != cudaSuccess) return e;
  int per_sm = 0;   // all CTAs of a cooperative launch must be co-resident
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fused_decode_kernel, kFThreads, L.total);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorNotSupported;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(c.num_sms);
  cfg.blockDim = dim3(kFThreads);
  cfg.dynamicSmemBytes = L.total;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, fused_decode_kernel, c);
  if (e == cudaSuccess) e = record_stage(se, 2, st);
  if (e == cudaSuccess) e = record_stage(se, 3, st);
  if (e == cudaSuccess) e = record_stage(se, 4, st);
  return e;
}
