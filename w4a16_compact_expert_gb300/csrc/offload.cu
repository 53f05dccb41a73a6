// The offload-qpacked comparison: before a batch of active experts is
// multiplied, their compact int4 weights are expanded into bounded FP16
// execution slots, then a dense grouped GEMM reads the FP16 copies.  The pages
// name this as the historical profile that dequantises a low-bit source into
// bounded FP16/BF16 execution slots ("Horizon RunMap - architecture",
// "Representation and computation" and the profile list beside it); it is
// built here only as the baseline that the compact path is measured against.
//
// expand_kernel: one CTA per (16-row tile, matrix, active expert of the
// batch).  Each 16-byte chunk (kc, lane) of a compact tile holds rows g and
// g + 8 (g = lane / 4) at the 16 K values kc*64 + c*16 .. + 15 (c = lane % 4);
// word j covers kb = kc*64 + c*16 + 4j .. + 3 with the offset-binary nibbles
//   0: (g, kb)     1: (g+8, kb)     2: (g, kb+2)   3: (g+8, kb+2)
//   4: (g, kb+1)   5: (g+8, kb+1)   6: (g, kb+3)   7: (g+8, kb+3)
// and u = q + 8.  The slot gets w = q * s rounded to the nearest FP16 (the
// same value the grouped GEMM's dequant warps write into shared memory).
#include "internal.h"

namespace {

__global__ void __launch_bounds__(128) expand_kernel(FwdCtx c) {
  pdl_wait();
  pdl_trigger();
  const int u = c.ub0 + blockIdx.z;   // active expert
  if (u >= c.ub1 || u >= *c.n_active) return;
  const int mat = blockIdx.y;         // 0 gate, 1 up, 2 down
  const MatLayout& L = mat == 0 ? c.lay.gate : mat == 1 ? c.lay.up : c.lay.down;
  const int rt = blockIdx.x;          // 16-row tile
  if (rt >= (int)L.rows / 16) return;
  const int K = (int)L.k, nkc = K / 64;
  const uint8_t* tile = c.pool + (size_t)c.act_slot[u] * c.slot_bytes + L.off + (size_t)rt * L.tile_bytes;
  const __half* sc = reinterpret_cast<const __half*>(tile);   // [block][16 rows]
  const size_t mat_off = (size_t)mat * c.I * c.H;              // gate, up: I*H each; down follows
  __half* dst = c.xpool + (size_t)(u - c.ub0) * c.xslot_halves + mat_off + (size_t)rt * 16 * K;
  for (int idx = threadIdx.x; idx < nkc * 32; idx += blockDim.x) {
    const int kc = idx >> 5, lane = idx & 31, g = lane >> 2, cq = lane & 3;
    const uint4 qv = *reinterpret_cast<const uint4*>(tile + L.scale_bytes + (size_t)kc * 512 + lane * 16);
    const int kb0 = kc * 64 + cq * 16;   // 16 K values, inside one 256-wide block
    const float s_lo = __half2float(sc[(kb0 >> 8) * 16 + g]);
    const float s_hi = __half2float(sc[(kb0 >> 8) * 16 + g + 8]);
    const uint32_t w4[4] = {qv.x, qv.y, qv.z, qv.w};
    uint32_t lo[8], hi[8];   // rows g, g + 8: 16 FP16 values each, two per word
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t w = w4[j];
      auto q = [&](int p) { return (float)((int)((w >> (4 * p)) & 15u) - 8); };
      const __half2 r0 = __floats2half2_rn(q(0) * s_lo, q(4) * s_lo);   // (g, kb), (g, kb+1)
      const __half2 r1 = __floats2half2_rn(q(2) * s_lo, q(6) * s_lo);   // (g, kb+2), (g, kb+3)
      const __half2 h0 = __floats2half2_rn(q(1) * s_hi, q(5) * s_hi);   // (g+8, kb), (g+8, kb+1)
      const __half2 h1 = __floats2half2_rn(q(3) * s_hi, q(7) * s_hi);   // (g+8, kb+2), (g+8, kb+3)
      lo[2 * j] = *reinterpret_cast<const uint32_t*>(&r0);
      lo[2 * j + 1] = *reinterpret_cast<const uint32_t*>(&r1);
      hi[2 * j] = *reinterpret_cast<const uint32_t*>(&h0);
      hi[2 * j + 1] = *reinterpret_cast<const uint32_t*>(&h1);
    }
    uint4* pg = reinterpret_cast<uint4*>(dst + (size_t)g * K + kb0);
    uint4* ph = reinterpret_cast<uint4*>(dst + (size_t)(g + 8) * K + kb0);
    pg[0] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    pg[1] = make_uint4(lo[4], lo[5], lo[6], lo[7]);
    ph[0] = make_uint4(hi[0], hi[1], hi[2], hi[3]);
    ph[1] = make_uint4(hi[4], hi[5], hi[6], hi[7]);
  }
}

}  // namespace

cudaError_t launch_expand(const FwdCtx& c, cudaStream_t st) {
  const int rt = (c.H > c.I ? c.H : c.I) / 16;
  return launch_pdl(expand_kernel, dim3((unsigned)rt, 3, (unsigned)(c.ub1 - c.ub0)), dim3(128), 0, st, 1, c);
}
