// Decode regime: grouped split-K GEMV over compact int4 experts.
//
// Each CTA fetches its weight tiles (compact int4 + FP16 scales, layout.h)
// with 1-D bulk async copies (TMA) into shared memory, dequantises them in
// registers (nothing expanded is ever written anywhere) and multiplies on the
// tensor cores with FP16 operands and FP32 accumulation (Horizon RunMap
// landing page, "08 / Precision & quality": compact weights converted
// in-kernel, FP32 accumulation stages, explicit rounding).  Explicit FP16
// rounding points: h = SiLU(g) * u before the down projection, and the output.
//
//   gate/up : CTA = (16-row tile of I, active expert); 8 warps split K; the
//             SiLU*up epilogue writes h [sorted row][I] in FP16.
//   down    : CTA = (32-row block of H, active expert); 2 row tiles x 4-way K
//             split; writes the per-pair output y [pair][H] in FP32.  The last
//             CTA to finish a 32-row block (arrival counter, no waiting)
//             gathers out[t] = (x[t]) + sum_j w[t,j] y[t*k+j] for that block,
//             summing in rank order j (deterministic, no atomics on data).
// Launch chain: route -> gate/up -> down with programmatic dependent launch.
// The down CTAs start fetching their weight tiles as soon as they are
// resident (routing is complete by then) and wait for h only to multiply.
#include "gemv_dev.cuh"

namespace {
using namespace gemv_dev;

__global__ void __launch_bounds__(256) gemv_gateup_kernel(FwdCtx c, int xrows) {
  pdl_wait();      // routing results of the preceding grid
  pdl_trigger();
  const int u = blockIdx.y;
  if (u >= *c.n_active) return;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t bar;
  __shared__ int s_tok[kTok];
  __shared__ int s_ok;
  const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31, g = lane >> 2, cc = lane & 3;
  const int rt = blockIdx.x;
  const int slot = c.act_slot[u], start = c.act_start[u], cnt = c.act_count[u];
  const uint8_t* base = c.pool + (size_t)slot * c.slot_bytes;
  const MatLayout& LG = c.lay.gate;
  const int H = c.H, I = c.I, nkc = H / 64, stride = H + 8;
  const uint32_t TS = LG.tile_bytes;
  const uint8_t* const tiles[2] = {smem, smem + TS};
  __half* xs = reinterpret_cast<__half*>(smem + 2 * (size_t)TS);
  float* red = reinterpret_cast<float*>(smem + 2 * (size_t)TS + (size_t)xrows * stride * sizeof(__half));
  if (tid == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
    mbar_expect_tx(&bar, 2 * TS);
    bulk_g2s(smem, tile_ptr(base, LG, rt), TS, &bar);
    bulk_g2s(smem + TS, tile_ptr(base, c.lay.up, rt), TS, &bar);
  }
  for (int p0 = 0; p0 < cnt; p0 += kTok) {
    const int np = min(kTok, cnt - p0);
    __syncthreads();   // previous pass done with xs / red / s_tok; barrier init visible
    if (tid < np) s_tok[tid] = c.sorted[start + p0 + tid] / c.k;
    __syncthreads();
    stage_rows(xs, stride, H, c.x, s_tok, np);
    if (p0 == 0) {
      if (tid == 0) s_ok = 1;
      __syncthreads();
      if (!mbar_wait_bounded(&bar, 0, c.status)) s_ok = 0;
    }
    __syncthreads();
    if (!s_ok) return;   // timed out: give up (the status word records it)
    float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    mma_tiles<2>(acc, tiles, LG.scale_bytes, xs, stride, np, lane, w, 8, nkc);
    // accumulator (row g / g+8, token 2cc / 2cc+1) -> red[w][mat][row][tok]
    float* rw = red + w * 2 * 16 * kTok;
#pragma unroll
    for (int m = 0; m < 2; ++m) {
      rw[(m * 16 + g) * kTok + 2 * cc] = acc[m][0];
      rw[(m * 16 + g) * kTok + 2 * cc + 1] = acc[m][1];
      rw[(m * 16 + g + 8) * kTok + 2 * cc] = acc[m][2];
      rw[(m * 16 + g + 8) * kTok + 2 * cc + 1] = acc[m][3];
    }
    __syncthreads();
    if (tid < 16 * kTok) {
      const int row = tid / kTok, tok = tid % kTok;
      if (tok < np) {
        float gs = 0.f, us = 0.f;
#pragma unroll
        for (int ww = 0; ww < 8; ++ww) {
          gs += red[(ww * 2 + 0) * 16 * kTok + row * kTok + tok];
          us += red[(ww * 2 + 1) * 16 * kTok + row * kTok + tok];
        }
        if (c.flags & 2u) {
          const float r = c.rnorm[s_tok[tok]];
          gs *= r;
          us *= r;
        }
        c.hbuf[(size_t)(start + p0 + tok) * I + rt * 16 + row] = __float2half_rn(silu_mul(gs, us));
      }
    }
  }
}

__global__ void __launch_bounds__(256) gemv_down_kernel(FwdCtx c, int hrows) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t bar;
  __shared__ int s_rows[kTok];
  __shared__ int s_ok;
  __shared__ unsigned s_last;
  const int u = blockIdx.y, hb = blockIdx.x;
  const int tid = threadIdx.x;
  const int H = c.H, I = c.I;
  const MatLayout& LD = c.lay.down;
  const uint32_t TS = LD.tile_bytes;
  // Routing finished before the gate/up grid let this grid launch: read it
  // from L2 and start fetching this CTA's weight tiles before waiting for h.
  const int nact = __ldcg(c.n_active);
  const bool active = u < nact;
  int start = 0, cnt = 0;
  if (active) {
    const int slot = __ldcg(&c.act_slot[u]);
    start = __ldcg(&c.act_start[u]);
    cnt = __ldcg(&c.act_count[u]);
    if (tid == 0) {
      const uint8_t* base = c.pool + (size_t)slot * c.slot_bytes;
      mbar_init(&bar, 1);
      fence_mbar_init();
      mbar_expect_tx(&bar, 2 * TS);
      bulk_g2s(smem, tile_ptr(base, LD, 2 * hb), TS, &bar);
      bulk_g2s(smem + TS, tile_ptr(base, LD, 2 * hb + 1), TS, &bar);
    }
  }
  pdl_wait();      // h of the gate/up grid
  pdl_trigger();
  if (active) {
    const int w = tid >> 5, lane = tid & 31, g = lane >> 2, cc = lane & 3;
    const int half_sel = w >> 2, wk = w & 3;
    const int nkc = I / 64, stride = I + 8;
    const uint8_t* const tiles[2] = {smem + (size_t)half_sel * TS, nullptr};
    __half* hs = reinterpret_cast<__half*>(smem + 2 * (size_t)TS);
    float* red = reinterpret_cast<float*>(smem + 2 * (size_t)TS + (size_t)hrows * stride * sizeof(__half));
    for (int p0 = 0; p0 < cnt; p0 += kTok) {
      const int np = min(kTok, cnt - p0);
      __syncthreads();
      if (tid < np) s_rows[tid] = start + p0 + tid;
      __syncthreads();
      stage_rows(hs, stride, I, c.hbuf, s_rows, np);
      if (p0 == 0) {
        if (tid == 0) s_ok = 1;
        __syncthreads();
        if (!mbar_wait_bounded(&bar, 0, c.status)) s_ok = 0;
      }
      __syncthreads();
      if (!s_ok) break;
      float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      mma_tiles<1>(acc, tiles, LD.scale_bytes, hs, stride, np, lane, wk, 4, nkc);
      float* rw = red + w * 16 * kTok;
      rw[g * kTok + 2 * cc] = acc[0][0];
      rw[g * kTok + 2 * cc + 1] = acc[0][1];
      rw[(g + 8) * kTok + 2 * cc] = acc[0][2];
      rw[(g + 8) * kTok + 2 * cc + 1] = acc[0][3];
      __syncthreads();
      {   // 256 threads = 32 rows x 8 tokens
        const int row = tid / kTok, tok = tid % kTok;
        const int hsel = row >> 4, r16 = row & 15;
        if (tok < np) {
          float y = 0.f;
#pragma unroll
          for (int ww = 0; ww < 4; ++ww) y += red[(hsel * 4 + ww) * 16 * kTok + r16 * kTok + tok];
          const int pair = c.sorted[start + p0 + tok];
          c.ybuf[(size_t)pair * H + hb * 32 + row] = y;
        }
      }
    }
    __threadfence();
  }
  __syncthreads();
  if (tid == 0) {
    unsigned last = 0;
    if (active) last = (atomicAdd(&c.down_counters[hb], 1u) == (unsigned)nact - 1u) ? 1u : 0u;
    if (nact == 0 && u == 0) last = 1u;   // every routed expert absent: out = residual or 0
    s_last = last;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  // Gather-combine rows [hb*32, hb*32+32) of every token, rank order j.
  const bool residual = c.flags & 1u;
  for (int i = tid; i < c.T * 32; i += blockDim.x) {
    const int t = i >> 5, hrow = hb * 32 + (i & 31);
    float acc = residual ? __half2float(c.x[(size_t)t * H + hrow]) : 0.f;
    for (int j = 0; j < c.k; ++j) {
      const int p = t * c.k + j;
      if (c.table[c.ids[p]] >= 0) acc = fmaf(c.topw[p], __ldcg(&c.ybuf[(size_t)p * H + hrow]), acc);
    }
    c.out[(size_t)t * H + hrow] = __float2half_rn(acc);
  }
  if (tid == 0 && nact > 0) c.down_counters[hb] = 0u;
}

}  // namespace

size_t gemv_smem_gateup(int H, int I, int rows) {
  const SlotLayout L = moe_slot_layout(H, I);
  return 2 * (size_t)L.gate.tile_bytes + (size_t)rows * (H + 8) * sizeof(__half) + 8 * 2 * 16 * kTok * sizeof(float);
}

size_t gemv_smem_down(int H, int I, int rows) {
  const SlotLayout L = moe_slot_layout(H, I);
  return 2 * (size_t)L.down.tile_bytes + (size_t)rows * (I + 8) * sizeof(__half) + 8 * 16 * kTok * sizeof(float);
}

cudaError_t launch_gemv_experts(const FwdCtx& c, cudaStream_t st, const StageEvents& se) {
  const int rows = c.T < kTok ? c.T : kTok;
  const size_t smem_gu = gemv_smem_gateup(c.H, c.I, rows);
  const size_t smem_dn = gemv_smem_down(c.H, c.I, rows);
  cudaError_t e = opt_in_smem((const void*)gemv_gateup_kernel, smem_gu);
  if (e == cudaSuccess) e = opt_in_smem((const void*)gemv_down_kernel, smem_dn);
  if (e != cudaSuccess) return e;
  e = launch_pdl(gemv_gateup_kernel, dim3(c.I / 16, c.max_active), dim3(256), smem_gu, st, 1, c, rows);
  if (e == cudaSuccess) e = record_stage(se, 2, st);
  if (e == cudaSuccess) e = launch_pdl(gemv_down_kernel, dim3(c.H / 32, c.max_active), dim3(256), smem_dn, st, 1, c, rows);
  if (e == cudaSuccess) e = record_stage(se, 3, st);
  if (e == cudaSuccess) e = record_stage(se, 4, st);
  return e;
}
