// Decode regime: grouped split-K GEMV over compact int4 experts.
//
// Weights are streamed once from HBM with 128-bit loads in the internal
// fragment order (layout.h), dequantised in registers (never written back
// anywhere), and multiplied on the tensor cores with FP16 operands and FP32
// accumulation (Horizon RunMap landing page, "08 / Precision & quality":
// compact weights converted in-kernel, FP32 accumulation stages, explicit
// rounding).  Explicit FP16 rounding points: h = SiLU(g) * u before the down
// projection, and the final output.
//
//   gate/up : CTA = (16-row tile of I, active expert); 8 warps split K; the
//             SiLU*up epilogue writes h [sorted row][I] in FP16.
//   down    : CTA = (32-row block of H, active expert); 2 row tiles x 4-way K
//             split; writes the per-pair output y [pair][H] in FP32.  The last
//             CTA to finish a 32-row block (arrival counter, no waiting)
//             gathers out[t] = (x[t]) + sum_j w[t,j] y[t*k+j] for that block,
//             summing in rank order j (deterministic, no atomics on data).
#include "internal.h"

namespace {

constexpr int kTok = 8;           // tokens per pass (one MMA n-tile)
constexpr int kGroup = 4;         // 64-wide K chunks a warp holds in flight

struct ChunkRegs {
  uint4 q[kGroup];
  __half2 s_lo[kGroup], s_hi[kGroup];
};

DEV_INLINE void load_chunks(ChunkRegs& r, const uint8_t* base, const MatLayout& m, int rt, int lane,
                            int kc0, int kstride, int nkc) {
  const int g = lane >> 2;
  const __half* s = scale_ptr(base, m);
#pragma unroll
  for (int i = 0; i < kGroup; ++i) {
    const int kc = kc0 + i * kstride;
    if (kc < nkc) {
      r.q[i] = ld_stream(chunk_ptr(base, m, kc, rt, lane));
      const int b = kc >> 2;   // 256-wide scale block of this 64-wide chunk
      r.s_lo[i] = __half2half2(s[(size_t)b * m.rows + rt * 16 + g]);
      r.s_hi[i] = __half2half2(s[(size_t)b * m.rows + rt * 16 + g + 8]);
    }
  }
}

// acc += W[rt rows, chunks] * B, B read from an smem tile [kTok][stride] of FP16.
DEV_INLINE void mma_chunks(float (&acc)[4], const ChunkRegs& r, const __half* bs, int stride, int lane,
                           int kc0, int kstride, int nkc) {
  const int g = lane >> 2, c = lane & 3;
#pragma unroll
  for (int i = 0; i < kGroup; ++i) {
    const int kc = kc0 + i * kstride;
    if (kc < nkc) {
      const uint32_t words[4] = {r.q[i].x, r.q[i].y, r.q[i].z, r.q[i].w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        uint32_t a[4];
        dequant_word(words[j], r.s_lo[i], r.s_hi[i], a);
        const int k0 = kc * 64 + j * 16;
        const __half* brow = bs + g * stride + k0 + 2 * c;
        const uint32_t b0 = *reinterpret_cast<const uint32_t*>(brow);
        const uint32_t b1 = *reinterpret_cast<const uint32_t*>(brow + 8);
        mma_16816(acc, a, b0, b1);
      }
    }
  }
}

// Stage up to kTok FP16 rows (gathered by row index) into smem [kTok][stride].
DEV_INLINE void stage_rows(__half* dst, int stride, int K, const __half* src, const int32_t* rows, int nrows) {
  const int vec_per_row = K / 8;
  for (int i = threadIdx.x; i < kTok * vec_per_row; i += blockDim.x) {
    const int r = i / vec_per_row, v = i % vec_per_row;
    uint4 val = make_uint4(0, 0, 0, 0);
    if (r < nrows) val = __ldg(reinterpret_cast<const uint4*>(src + (size_t)rows[r] * K) + v);
    *(reinterpret_cast<uint4*>(dst + r * stride) + v) = val;
  }
}

__global__ void __launch_bounds__(256) gemv_gateup_kernel(FwdCtx c) {
  const int u = blockIdx.y;
  if (u >= *c.n_active) return;
  extern __shared__ __align__(16) uint8_t smem[];
  const int rt = blockIdx.x;
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, cc = lane & 3;
  const int slot = c.act_slot[u], start = c.act_start[u], cnt = c.act_count[u];
  const uint8_t* base = c.pool + (size_t)slot * c.slot_bytes;
  const int H = c.H, I = c.I, nkc = H / 64;
  const int stride = H + 8;
  __half* xs = reinterpret_cast<__half*>(smem);
  float* red = reinterpret_cast<float*>(smem + (size_t)kTok * stride * sizeof(__half));  // [8][2][16][8]
  __shared__ int s_tok[kTok];
  for (int p0 = 0; p0 < cnt; p0 += kTok) {
    const int np = min(kTok, cnt - p0);
    ChunkRegs rg, ru;
    load_chunks(rg, base, c.lay.gate, rt, lane, w, 8, nkc);
    load_chunks(ru, base, c.lay.up, rt, lane, w, 8, nkc);
    __syncthreads();   // previous pass is done with xs / red / s_tok
    if (threadIdx.x < kTok) s_tok[threadIdx.x] = threadIdx.x < np ? c.sorted[start + p0 + threadIdx.x] / c.k : 0;
    __syncthreads();
    stage_rows(xs, stride, H, c.x, s_tok, np);
    __syncthreads();
    float ag[4] = {0.f, 0.f, 0.f, 0.f}, au[4] = {0.f, 0.f, 0.f, 0.f};
    mma_chunks(ag, rg, xs, stride, lane, w, 8, nkc);
    mma_chunks(au, ru, xs, stride, lane, w, 8, nkc);
    for (int kc0 = w + 8 * kGroup; kc0 < nkc; kc0 += 8 * kGroup) {
      load_chunks(rg, base, c.lay.gate, rt, lane, kc0, 8, nkc);
      load_chunks(ru, base, c.lay.up, rt, lane, kc0, 8, nkc);
      mma_chunks(ag, rg, xs, stride, lane, kc0, 8, nkc);
      mma_chunks(au, ru, xs, stride, lane, kc0, 8, nkc);
    }
    // accumulator (row g / g+8, token 2cc / 2cc+1) -> red[w][mat][row][tok]
    float* rw = red + w * 2 * 16 * kTok;
    rw[(0 * 16 + g) * kTok + 2 * cc] = ag[0];
    rw[(0 * 16 + g) * kTok + 2 * cc + 1] = ag[1];
    rw[(0 * 16 + g + 8) * kTok + 2 * cc] = ag[2];
    rw[(0 * 16 + g + 8) * kTok + 2 * cc + 1] = ag[3];
    rw[(1 * 16 + g) * kTok + 2 * cc] = au[0];
    rw[(1 * 16 + g) * kTok + 2 * cc + 1] = au[1];
    rw[(1 * 16 + g + 8) * kTok + 2 * cc] = au[2];
    rw[(1 * 16 + g + 8) * kTok + 2 * cc + 1] = au[3];
    __syncthreads();
    if (threadIdx.x < 16 * kTok) {
      const int row = threadIdx.x / kTok, tok = threadIdx.x % kTok;
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

__global__ void __launch_bounds__(256) gemv_down_kernel(FwdCtx c) {
  const int u = blockIdx.y, hb = blockIdx.x;
  const int nact = *c.n_active;
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ unsigned s_last;
  const int H = c.H, I = c.I;
  const int tid = threadIdx.x;
  if (u < nact) {
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, cc = lane & 3;
    const int rt = hb * 2 + (w >> 2), wk = w & 3;
    const int slot = c.act_slot[u], start = c.act_start[u], cnt = c.act_count[u];
    const uint8_t* base = c.pool + (size_t)slot * c.slot_bytes;
    const int nkc = I / 64;
    const int stride = I + 8;
    __half* hs = reinterpret_cast<__half*>(smem);
    float* red = reinterpret_cast<float*>(smem + (size_t)kTok * stride * sizeof(__half));  // [8][16][8]
    __shared__ int s_rows[kTok];
    for (int p0 = 0; p0 < cnt; p0 += kTok) {
      const int np = min(kTok, cnt - p0);
      ChunkRegs rd;
      load_chunks(rd, base, c.lay.down, rt, lane, wk, 4, nkc);
      __syncthreads();
      if (tid < kTok) s_rows[tid] = start + p0 + (tid < np ? tid : 0);
      __syncthreads();
      stage_rows(hs, stride, I, c.hbuf, s_rows, np);
      __syncthreads();
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      mma_chunks(acc, rd, hs, stride, lane, wk, 4, nkc);
      for (int kc0 = wk + 4 * kGroup; kc0 < nkc; kc0 += 4 * kGroup) {
        load_chunks(rd, base, c.lay.down, rt, lane, kc0, 4, nkc);
        mma_chunks(acc, rd, hs, stride, lane, kc0, 4, nkc);
      }
      float* rw = red + w * 16 * kTok;
      rw[g * kTok + 2 * cc] = acc[0];
      rw[g * kTok + 2 * cc + 1] = acc[1];
      rw[(g + 8) * kTok + 2 * cc] = acc[2];
      rw[(g + 8) * kTok + 2 * cc + 1] = acc[3];
      __syncthreads();
      {   // 256 threads = 32 rows x 8 tokens
        const int row = tid / kTok, tok = tid % kTok;
        const int half_sel = row >> 4, r16 = row & 15;
        if (tok < np) {
          float y = 0.f;
#pragma unroll
          for (int ww = 0; ww < 4; ++ww) y += red[(half_sel * 4 + ww) * 16 * kTok + r16 * kTok + tok];
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
    if (u < nact) last = (atomicAdd(&c.down_counters[hb], 1u) == (unsigned)nact - 1u) ? 1u : 0u;
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
  if (tid == 0) c.down_counters[hb] = 0u;
}

}  // namespace

cudaError_t launch_gemv_experts(const FwdCtx& c, cudaStream_t st) {
  const size_t smem_gu = (size_t)kTok * (c.H + 8) * sizeof(__half) + 8 * 2 * 16 * kTok * sizeof(float);
  const size_t smem_dn = (size_t)kTok * (c.I + 8) * sizeof(__half) + 8 * 16 * kTok * sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(gemv_gateup_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_gu);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(gemv_down_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_dn);
  if (e != cudaSuccess) return e;
  gemv_gateup_kernel<<<dim3(c.I / 16, c.max_active), 256, smem_gu, st>>>(c);
  gemv_down_kernel<<<dim3(c.H / 32, c.max_active), 256, smem_dn, st>>>(c);
  return cudaGetLastError();
}
