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
//   small T  : one launch.  CTAs compute split-K partial logits; the last CTA
//              to arrive (arrival counter, no waiting) finishes softmax/top-k
//              and the permutation for every token.
//   larger T : logits, top-k (warp per token) and permutation as three launches.
#include <float.h>
#include <limits.h>

#include "internal.h"

namespace {

constexpr int kLogitWarps = 8;    // experts per logits CTA (one warp each)
constexpr int kMaxEPL = 8;        // experts per lane in top-k: E <= 256
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

DEV_INLINE float sumsq8(uint4 a) { return dot8(a, a); }

// Softmax + top-k of token t (one warp).  Partial logits are read from L2
// (they may have been written by other CTAs of the same launch).
DEV_INLINE void topk_token(const FwdCtx& c, int t) {
  const int lane = threadIdx.x & 31;
  const int E = c.E, T = c.T;
  float r = 1.f;
  if (c.flags & 2u) {   // PRENORM
    float ss = 0.f;
    for (int ks = 0; ks < c.ksplit; ++ks) ss += __ldcg(&c.ss_part[(size_t)ks * T + t]);
    r = 1.0f / sqrtf(ss / (float)c.H + 1e-6f);
    if (lane == 0) c.rnorm[t] = r;
  }
  float v[kMaxEPL];
  bool live[kMaxEPL];
#pragma unroll
  for (int i = 0; i < kMaxEPL; ++i) {
    const int e = lane + 32 * i;
    live[i] = e < E;
    v[i] = -INFINITY;
    if (live[i]) {
      float s = 0.f;
      for (int ks = 0; ks < c.ksplit; ++ks) s += __ldcg(&c.logit_part[((size_t)ks * T + t) * E + e]);
      v[i] = s * r + (c.bias ? c.bias[e] : 0.f);
    }
  }
  float m = -INFINITY, selv = -INFINITY;
  int sele = 0;
  for (int j = 0; j < c.k; ++j) {
    float bv = -INFINITY;
    int be = INT_MAX;
#pragma unroll
    for (int i = 0; i < kMaxEPL; ++i)
      if (live[i] && (be == INT_MAX || v[i] > bv)) { bv = v[i]; be = lane + 32 * i; }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(kFull, bv, o);
      const int oe = __shfl_xor_sync(kFull, be, o);
      if (oe != INT_MAX && (be == INT_MAX || ov > bv || (ov == bv && oe < be))) { bv = ov; be = oe; }
    }
    if (j == 0) m = bv;
    if (lane == j) { selv = bv; sele = be; }
#pragma unroll
    for (int i = 0; i < kMaxEPL; ++i)
      if (be == lane + 32 * i) live[i] = false;
  }
  float den = 0.f;
#pragma unroll
  for (int i = 0; i < kMaxEPL; ++i)
    if (lane + 32 * i < E && m != -INFINITY) den += expf(v[i] - m);
  den = warp_sum(den);
  if (lane < c.k) {
    c.ids[(size_t)t * c.k + lane] = sele;
    c.topw[(size_t)t * c.k + lane] = (m == -INFINITY) ? 0.f : expf(selv - m) / den;
  }
}

// Stable permutation of the T*k pairs by expert (block-wide; any blockDim that
// is a multiple of 32).  smem: nwarps*E + 2E + 1 ints.
DEV_INLINE void permute_block(const FwdCtx& c, int* smem) {
  const int nw = blockDim.x >> 5, w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = c.E, P = c.T * c.k;
  int* hist = smem;            // [nw][E] counts, then running positions
  int* cnt = hist + nw * E;    // [E]
  int* off = cnt + E;          // [E+1]
  for (int i = threadIdx.x; i < nw * E; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  const int chunk = (P + nw - 1) / nw;
  const int p_beg = min(P, w * chunk), p_end = min(P, p_beg + chunk);
  for (int p = p_beg + lane; p < p_end; p += 32) atomicAdd(&hist[w * E + c.ids[p]], 1);
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
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int run = off[e];
    for (int ww = 0; ww < nw; ++ww) {
      const int hcount = hist[ww * E + e];
      hist[ww * E + e] = run;
      run += hcount;
    }
  }
  __syncthreads();
  for (int base = p_beg; base < p_end; base += 32) {
    const int p = base + lane;
    const bool valid = p < p_end;
    const int e = valid ? c.ids[p] : -1 - lane;
    const unsigned peers = __match_any_sync(kFull, e);
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

// Partial logits of experts [8*bx, 8*bx+8) over K slice by, tokens of bz.
__global__ void __launch_bounds__(256) route_logits_kernel(FwdCtx c, int tokens_per_cta, int fused) {
  extern __shared__ int route_smem[];
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = blockIdx.x * kLogitWarps + w;
  const int H = c.H, T = c.T;
  const int KC = H / c.ksplit;
  const int kbeg = blockIdx.y * KC, kend = kbeg + KC;
  const int t0 = blockIdx.z * tokens_per_cta, t1 = min(T, t0 + tokens_per_cta);
  if (e < c.E) {
    const __half* wr = c.router_w + (size_t)e * H;
    for (int t = t0; t < t1; ++t) {
      const __half* xt = c.x + (size_t)t * H;
      float acc = 0.f;
      for (int kk = kbeg + lane * 8; kk < kend; kk += 256)
        acc += dot8(__ldg(reinterpret_cast<const uint4*>(xt + kk)), __ldg(reinterpret_cast<const uint4*>(wr + kk)));
      acc = warp_sum(acc);
      if (lane == 0) c.logit_part[((size_t)blockIdx.y * T + t) * c.E + e] = acc;
    }
  }
  if ((c.flags & 2u) && blockIdx.x == 0) {   // PRENORM: partial sums of squares
    for (int t = t0 + w; t < t1; t += kLogitWarps) {
      const __half* xt = c.x + (size_t)t * H;
      float ss = 0.f;
      for (int kk = kbeg + lane * 8; kk < kend; kk += 256) ss += sumsq8(__ldg(reinterpret_cast<const uint4*>(xt + kk)));
      ss = warp_sum(ss);
      if (lane == 0) c.ss_part[(size_t)blockIdx.y * T + t] = ss;
    }
  }
  if (!fused) return;
  // Last CTA to arrive finishes the routing for every token.
  __threadfence();
  __syncthreads();
  __shared__ unsigned s_last;
  if (threadIdx.x == 0) {
    const unsigned total = gridDim.x * gridDim.y * gridDim.z;
    const unsigned old = atomicAdd(c.route_counter, 1u);
    s_last = (old == total - 1) ? 1u : 0u;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  for (int t = w; t < T; t += blockDim.x >> 5) topk_token(c, t);
  __syncthreads();
  permute_block(c, route_smem);
  if (threadIdx.x == 0) *c.route_counter = 0u;
}

__global__ void __launch_bounds__(256) route_topk_kernel(FwdCtx c) {
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t < c.T) topk_token(c, t);
}

__global__ void __launch_bounds__(1024) route_permute_kernel(FwdCtx c) {
  extern __shared__ int perm_smem[];
  permute_block(c, perm_smem);
}

}  // namespace

cudaError_t launch_route(const FwdCtx& c, bool fused, cudaStream_t st) {
  const dim3 block(256);
  if (fused) {
    const dim3 grid((c.E + kLogitWarps - 1) / kLogitWarps, c.ksplit, 1);
    const size_t smem = (size_t)(8 * c.E + 2 * c.E + 1) * sizeof(int);
    route_logits_kernel<<<grid, block, smem, st>>>(c, c.T, 1);
    return cudaGetLastError();
  }
  const int tpc = 16;
  const dim3 grid((c.E + kLogitWarps - 1) / kLogitWarps, c.ksplit, (c.T + tpc - 1) / tpc);
  route_logits_kernel<<<grid, block, 0, st>>>(c, tpc, 0);
  route_topk_kernel<<<(c.T + 7) / 8, block, 0, st>>>(c);
  const size_t smem = (size_t)(32 * c.E + 2 * c.E + 1) * sizeof(int);
  route_permute_kernel<<<1, 1024, smem, st>>>(c);
  return cudaGetLastError();
}
