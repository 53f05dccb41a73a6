// Device routines of the router shared by the routing kernels and the fused
// decode kernel: FP16 dot products, softmax / top-k of one token, and the
// stable token-to-expert permutation of one CTA.
#pragma once
#include <float.h>
#include <limits.h>

#include "internal.h"

namespace route_dev {

constexpr int kLogitWarps = 8;    // experts per logits CTA (one warp each)
constexpr int kMaxEPL = 8;        // experts per lane in top-k: E <= 256
constexpr int kMaxCluster = 8;
constexpr unsigned kFull = 0xffffffffu;

DEV_INLINE float dot8(uint4 a, uint4 b) {
  const __half2* ha = reinterpret_cast<const __half2*>(&a);
  const __half2* hb = reinterpret_cast<const __half2*>(&b);
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 fa = __half22float2(ha[i]);
    const float2 fb = __half22float2(hb[i]);
    s = fmaf(fa.x, fb.x, s);
    s = fmaf(fa.y, fb.y, s);
  }
  return s;
}

// dot(x_t, w_e) over the whole hidden dimension (one warp).
DEV_INLINE float warp_dot(const __half* xt, const __half* we, int H, int lane) {
  float acc = 0.f;
  for (int kk = lane * 8; kk < H; kk += 256)
    acc += dot8(__ldg(reinterpret_cast<const uint4*>(xt + kk)), __ldg(reinterpret_cast<const uint4*>(we + kk)));
  return warp_sum(acc);
}

// Monotonic map of a (non-NaN) float to an unsigned key: a < b <=> key(a) < key(b).
DEV_INLINE uint32_t order_key(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Softmax + top-k of one token (one warp).  lg: the token's E logits (any
// address space), before bias and pre-norm scale r.  Each round picks the
// largest logit with two warp reductions (max of the order key, then min of
// the expert index among the lanes holding that key: ties -> lower index).
// Writes ids/weights to c.ids/c.topw and, when ids_s != NULL, the ids to ids_s.
template <int EPL>
DEV_INLINE void topk_token_epl(const FwdCtx& c, int t, const float* lg, float r, int* ids_s) {
  const int lane = threadIdx.x & 31;
  const int E = c.E;
  float v[EPL];
  uint32_t key[EPL];
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = lane + 32 * i;
    v[i] = e < E ? lg[e] * r + (c.bias ? c.bias[e] : 0.f) : -INFINITY;
    key[i] = e < E ? order_key(v[i]) : 0u;   // 0 = not a candidate (below -inf's key)
  }
  float m = -INFINITY, selv = -INFINITY;
  int sele = 0;
  for (int j = 0; j < c.k; ++j) {
    uint32_t bk = 0u;
    int be = 0;
    float bv = -INFINITY;
#pragma unroll
    for (int i = 0; i < EPL; ++i)
      if (key[i] > bk) { bk = key[i]; be = lane + 32 * i; bv = v[i]; }
    const uint32_t mk = __reduce_max_sync(kFull, bk);
    const uint32_t me = __reduce_min_sync(kFull, (bk == mk && bk != 0u) ? (uint32_t)be : 0xFFFFFFFFu);
    const float mv = __shfl_sync(kFull, bv, (int)(me & 31u));
    if (j == 0) m = mv;
    if (lane == j) { selv = mv; sele = (int)me; }
#pragma unroll
    for (int i = 0; i < EPL; ++i)
      if ((uint32_t)(lane + 32 * i) == me) key[i] = 0u;
  }
  float den = 0.f;
#pragma unroll
  for (int i = 0; i < EPL; ++i)
    if (lane + 32 * i < E && m != -INFINITY) den += expf(v[i] - m);
  den = warp_sum(den);
  if (lane < c.k) {
    c.ids[(size_t)t * c.k + lane] = sele;
    c.topw[(size_t)t * c.k + lane] = (m == -INFINITY) ? 0.f : expf(selv - m) / den;
    if (ids_s) ids_s[t * c.k + lane] = sele;
  }
}

DEV_INLINE void topk_token(const FwdCtx& c, int t, const float* lg, float r, int* ids_s) {
  if (c.E <= 32) topk_token_epl<1>(c, t, lg, r, ids_s);
  else if (c.E <= 64) topk_token_epl<2>(c, t, lg, r, ids_s);
  else if (c.E <= 128) topk_token_epl<4>(c, t, lg, r, ids_s);
  else topk_token_epl<8>(c, t, lg, r, ids_s);
}

DEV_INLINE float prenorm_scale(float ss, int H) { return 1.0f / sqrtf(ss / (float)H + 1e-6f); }

// Stable permutation of the T*k pairs by expert (block-wide; any blockDim that
// is a multiple of 32).  ids: the flat [T*k] expert ids (global or shared).
// smem: nwarps*E + 2E + 1 ints.  Each warp owns a contiguous run of pairs;
// per 32-pair round, __match_any_sync groups equal ids, so counts and ranks
// need no atomics (deterministic and contention-free).
template <typename IdT>
DEV_INLINE void permute_block(const FwdCtx& c, const IdT* ids, int* smem) {
  constexpr int kMaxRounds = 16;   // pairs per warp <= 16 * 32 in one sweep
  const int nw = blockDim.x >> 5, w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = c.E, P = c.T * c.k;
  int* hist = smem;            // [nw][E] counts, then running positions
  int* cnt = hist + nw * E;    // [E]
  int* off = cnt + E;          // [E+1]
  for (int i = threadIdx.x; i < nw * E; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  const int chunk = (P + nw - 1) / nw;
  const int p_beg = min(P, w * chunk), p_end = min(P, p_beg + chunk);
  const bool one_sweep = chunk <= kMaxRounds * 32;
  int my_er[kMaxRounds];   // (rank inside (warp, expert)) << 8 | expert of this lane's pairs
  // pass 1: per-warp counts (leaders add the size of their group) and ranks
#pragma unroll
  for (int rd = 0; rd < kMaxRounds; ++rd) {
    const int p = p_beg + rd * 32 + lane;
    if (p_beg + rd * 32 >= p_end) break;
    const bool valid = p < p_end;
    const int e = valid ? (int)ids[p] : -1 - lane;
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    int base = 0;
    if (valid) base = hist[w * E + e];
    __syncwarp();
    if (valid && rank == 0) hist[w * E + e] = base + __popc(peers);
    __syncwarp();
    my_er[rd] = ((base + rank) << 8) | (e & 0xFF);
  }
  if (!one_sweep) {   // long runs: count the rest (ranks recomputed in pass 2)
    for (int q = p_beg + kMaxRounds * 32; q < p_end; q += 32) {
      const int p = q + lane;
      const bool valid = p < p_end;
      const int e = valid ? (int)ids[p] : -1 - lane;
      const unsigned peers = __match_any_sync(0xffffffffu, e);
      if (valid && __popc(peers & ((1u << lane) - 1u)) == 0) hist[w * E + e] += __popc(peers);
      __syncwarp();
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int s = 0;
    for (int ww = 0; ww < nw; ++ww) s += hist[ww * E + e];
    cnt[e] = s;
  }
  __syncthreads();
  if (w == 0) {   // exclusive scan of cnt: lane owns experts lane*per .. lane*per+per-1
    const int per = (E + 31) / 32;
    int local[kMaxEPL];
    int s = 0;
#pragma unroll
    for (int i = 0; i < kMaxEPL; ++i) {
      const int e = lane * per + i;
      local[i] = s;
      if (i < per && e < E) s += cnt[e];
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
      if (i < per && e < E) off[e] = excl + local[i];
    }
    if (lane == 31) off[E] = incl;
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {   // hist -> first row of (warp, expert)
    int run = off[e];
    for (int ww = 0; ww < nw; ++ww) {
      const int hcount = hist[ww * E + e];
      hist[ww * E + e] = run;
      run += hcount;
    }
  }
  __syncthreads();
  // pass 2: scatter
#pragma unroll
  for (int rd = 0; rd < kMaxRounds; ++rd) {
    const int p = p_beg + rd * 32 + lane;
    if (p_beg + rd * 32 >= p_end) break;
    if (p < p_end) {
      const int pos = hist[w * E + (my_er[rd] & 0xFF)] + (my_er[rd] >> 8);
      c.sorted[pos] = p;
      c.p2r[p] = pos;
    }
  }
  if (!one_sweep) {
    // continue after the first kMaxRounds*32 pairs: running positions per expert
    __syncwarp();
    for (int rd = 0; rd < kMaxRounds; ++rd) {   // advance bases past pass-1 pairs
      const int q = p_beg + rd * 32;
      if (q >= p_end) break;
      const int p = q + lane;
      const bool valid = p < p_end;
      const int e = valid ? (my_er[rd] & 0xFF) : -1 - lane;
      const unsigned peers = __match_any_sync(0xffffffffu, e);
      if (valid && __popc(peers & ((1u << lane) - 1u)) == 0) hist[w * E + e] += __popc(peers);
      __syncwarp();
    }
    for (int q = p_beg + kMaxRounds * 32; q < p_end; q += 32) {
      const int p = q + lane;
      const bool valid = p < p_end;
      const int e = valid ? (int)ids[p] : -1 - lane;
      const unsigned peers = __match_any_sync(0xffffffffu, e);
      const int rank = __popc(peers & ((1u << lane) - 1u));
      if (valid) {
        const int pos = hist[w * E + e] + rank;
        c.sorted[pos] = p;
        c.p2r[p] = pos;
      }
      __syncwarp();
      if (valid && rank == 0) hist[w * E + e] += __popc(peers);
      __syncwarp();
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e <= E; e += blockDim.x) c.offsets[e] = off[e];
  if (w == 0) {   // active (routed and resident) experts in ascending order
    int n = 0, tiles = 0;
    for (int e0 = 0; e0 < E; e0 += 32) {
      const int e = e0 + lane;
      const int ce = e < E ? cnt[e] : 0;
      const int slot = ce > 0 ? c.table[e] : -1;
      const bool act = ce > 0 && slot >= 0;
      if (ce > 0 && slot < 0) {
        atomicAdd(&c.status->miss, (unsigned long long)ce);
        atomicOr(&c.status->flags, STATUS_MISS);
      }
      const unsigned am = __ballot_sync(kFull, act);
      const int pos = n + __popc(am & ((1u << lane) - 1u));
      const int nt = act ? (ce + c.tile_tokens - 1) / c.tile_tokens : 0;
      int incl = nt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int x = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += x;
      }
      if (act) {
        c.act_expert[pos] = e;
        c.act_slot[pos] = slot;
        c.act_start[pos] = off[e];
        c.act_count[pos] = ce;
        c.act_tile[pos] = tiles + incl - nt;
      }
      n += __popc(am);
      tiles += __shfl_sync(kFull, incl, 31);
    }
    if (lane == 0) {
      *c.n_active = n;
      c.act_tile[n] = tiles;
    }
  }
}


}  // namespace route_dev
