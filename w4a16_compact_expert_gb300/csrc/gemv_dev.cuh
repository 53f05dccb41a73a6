// Device routines of the decode-regime GEMV shared by the GEMV kernels and
// the fused decode kernel: the int4 tile x token-rows MMA loop and row staging.
#pragma once
#include "internal.h"

namespace gemv_dev {

constexpr int kTok = 8;   // tokens per pass (one MMA n-tile)

DEV_INLINE uint32_t lds_b32_or0(const __half* p, bool valid) {
  return valid ? *reinterpret_cast<const uint32_t*>(p) : 0u;
}

// acc[m] += tile[m] rows x B over chunks kc = kc0, kc0 + kstride, ... (< nkc).
// B rows live in smem [np][stride] FP16; rows >= np read as zero.
template <int NMAT>
DEV_INLINE void mma_tiles(float (&acc)[2][4], const uint8_t* const (&tile)[2], uint32_t scale_bytes,
                          const __half* bs, int stride, int np, int lane, int kc0, int kstride, int nkc) {
  const int g = lane >> 2, c = lane & 3;
  const bool brow = g < np;
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
      const __half* bp = bs + g * stride + kc * 64 + c * 16 + j * 4;   // K slots of step j (layout.h)
      const uint32_t b0 = lds_b32_or0(bp, brow), b1 = lds_b32_or0(bp + 2, brow);
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

// Stage `nrows` FP16 rows (gathered by row index) into smem [*][stride].
// nthr threads (threadIdx.x < nthr) take part.
DEV_INLINE void stage_rows(__half* dst, int stride, int K, const __half* src, const int32_t* rows, int nrows,
                           int nthr = 256) {
  const int vec_per_row = K / 8;
  const int n = nrows * vec_per_row;
  for (int i0 = 0; i0 < n; i0 += 4 * nthr) {   // up to 4 independent loads in flight per thread
    uint4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = i0 + u * nthr + threadIdx.x;
      if (i < n) v[u] = __ldg(reinterpret_cast<const uint4*>(src + (size_t)rows[i / vec_per_row] * K) + i % vec_per_row);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = i0 + u * nthr + threadIdx.x;
      if (i < n) *(reinterpret_cast<uint4*>(dst + (i / vec_per_row) * stride) + i % vec_per_row) = v[u];
    }
  }
}

}  // namespace gemv_dev
