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
//   larger T : logits, top-k (warp per token) and permutation as three launches.
#include <float.h>
#include <limits.h>

#include "internal.h"

namespace {

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

// Softmax + top-k of one token (one warp).  lg: the token's E logits (any
// address space), before bias and pre-norm scale r.  Writes ids/weights to
// global memory and, when ids_s != NULL, the ids to ids_s too.
DEV_INLINE void topk_token(const FwdCtx& c, int t, const float* lg, float r, int* ids_s) {
  const int lane = threadIdx.x & 31;
  const int E = c.E;
  float v[kMaxEPL];
  bool live[kMaxEPL];
#pragma unroll
  for (int i = 0; i < kMaxEPL; ++i) {
    const int e = lane + 32 * i;
    live[i] = e < E;
    v[i] = live[i] ? lg[e] * r + (c.bias ? c.bias[e] : 0.f) : -INFINITY;
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
    if (ids_s) ids_s[t * c.k + lane] = sele;
  }
}

DEV_INLINE float prenorm_scale(float ss, int H) { return 1.0f / sqrtf(ss / (float)H + 1e-6f); }

// Stable permutation of the T*k pairs by expert (block-wide; any blockDim that
// is a multiple of 32).  ids: the flat [T*k] expert ids (global or shared).
// smem: nwarps*E + 2E + 1 ints.
template <typename IdT>
DEV_INLINE void permute_block(const FwdCtx& c, const IdT* ids, int* smem) {
  const int nw = blockDim.x >> 5, w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = c.E, P = c.T * c.k;
  int* hist = smem;            // [nw][E] counts, then running positions
  int* cnt = hist + nw * E;    // [E]
  int* off = cnt + E;          // [E+1]
  for (int i = threadIdx.x; i < nw * E; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  const int chunk = (P + nw - 1) / nw;
  const int p_beg = min(P, w * chunk), p_end = min(P, p_beg + chunk);
  for (int p = p_beg + lane; p < p_end; p += 32) atomicAdd(&hist[w * E + (int)ids[p]], 1);
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
    const int e = valid ? (int)ids[p] : -1 - lane;
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
// summed in fixed order by the top-k kernel.
__global__ void __launch_bounds__(128) route_logits_mma_kernel(FwdCtx c) {
  extern __shared__ __align__(16) uint8_t lsm[];
  pdl_wait();
  pdl_trigger();
  constexpr int S = kRouteKC + 8;   // padded row stride (halves): conflict-free fragment reads
  __half* xs = reinterpret_cast<__half*>(lsm);
  __half* ws = xs + kRouteTile * S;
  const int T = c.T, E = c.E, H = c.H;
  const int t0 = blockIdx.x * kRouteTile, e0 = blockIdx.y * kRouteTile, ks = blockIdx.z;
  const int k0 = ks * kRouteKC, kc = min(kRouteKC, H - k0);
  const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31, g = lane >> 2, cq = lane & 3;
  const int vpr = kc / 8;   // 16-byte vectors per row
  for (int i = tid; i < kRouteTile * vpr; i += blockDim.x) {
    const int r = i / vpr, v = i % vpr;
    const uint4 z = make_uint4(0, 0, 0, 0);
    const int t = t0 + r, e = e0 + r;
    *reinterpret_cast<uint4*>(xs + r * S + v * 8) =
        t < T ? __ldg(reinterpret_cast<const uint4*>(c.x + (size_t)t * H + k0) + v) : z;
    *reinterpret_cast<uint4*>(ws + r * S + v * 8) =
        e < E ? __ldg(reinterpret_cast<const uint4*>(c.router_w + (size_t)e * H + k0) + v) : z;
  }
  __syncthreads();
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
  if ((c.flags & 2u) && blockIdx.y == 0) {   // PRENORM: partial sums of squares
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

// One warp per token: sums the K slices of its logits (fixed order), then
// softmax / top-k.
__global__ void __launch_bounds__(256) route_topk_kernel(FwdCtx c) {
  __shared__ float lg[8][256];
  pdl_wait();
  pdl_trigger();
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + w;
  if (t >= c.T) return;
  for (int e = lane; e < c.E; e += 32) {
    float s = 0.f;
    for (int ks = 0; ks < c.ksplit; ++ks) s += c.logit_part[((size_t)ks * c.T + t) * c.E + e];
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

// One CTA: the expert ids are staged in shared memory (one byte each), then
// histogram, scan and stable scatter run out of shared memory.
__global__ void __launch_bounds__(1024) route_permute_kernel(FwdCtx c, int ids_in_smem) {
  extern __shared__ __align__(16) int perm_smem[];
  pdl_wait();
  pdl_trigger();
  const int P = c.T * c.k;
  if (ids_in_smem) {
    uint8_t* ids8 = reinterpret_cast<uint8_t*>(perm_smem);
    int* scratch = perm_smem + (P + 15) / 16 * 4;
    for (int p = threadIdx.x; p < P; p += blockDim.x) ids8[p] = (uint8_t)c.ids[p];
    __syncthreads();
    permute_block(c, ids8, scratch);
  } else {
    permute_block(c, c.ids, perm_smem);
  }
}

}  // namespace

cudaError_t launch_route(const FwdCtx& c, bool small, cudaStream_t st) {
  const size_t smem_small = route_cluster_smem(c.T, c.E, c.H, c.k);
  if (small && smem_small <= 200 * 1024) {
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
  const int P = c.T * c.k;
  const size_t scratch = (size_t)(32 * c.E + 2 * c.E + 1) * sizeof(int);
  const size_t smem_ids = (size_t)(P + 15) / 16 * 16 + scratch;
  const int in_smem = smem_ids <= 200 * 1024;
  const size_t smem = in_smem ? smem_ids : scratch;
  if (e == cudaSuccess) e = opt_in_smem((const void*)route_permute_kernel, smem);
  if (e == cudaSuccess) e = launch_pdl(route_permute_kernel, dim3(1), dim3(1024), smem, st, 1, cc, in_smem);
  return e;
}
