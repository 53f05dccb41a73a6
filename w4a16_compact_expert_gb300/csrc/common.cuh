// Device helpers shared by the kernels: status word, int4 -> FP16 conversion,
// the 16x8x16 MMA step, warp reductions.
#pragma once
#include <cuda_fp16.h>
#include <stdint.h>

#include "layout.h"

// Device status word (one per handle).
struct DevStatus {
  unsigned long long miss;   // routed token-expert pairs whose expert had no slot
  unsigned int flags;        // STATUS_* bits
  unsigned int pad;
};
#define STATUS_MISS 1u
#define STATUS_TIMEOUT 2u

#define DEV_INLINE __device__ __forceinline__

DEV_INLINE uint32_t h2_as_u32(__half2 v) { return *reinterpret_cast<uint32_t*>(&v); }
DEV_INLINE __half2 u32_as_h2(uint32_t v) { return *reinterpret_cast<__half2*>(&v); }

// One word of the internal layout (eight offset-binary nibbles, see layout.h)
// -> the four FP16x2 A-operand registers, each the FP16 value nearest q*s.
// The conversion ORs a nibble into the mantissa of the FP16 number 1024
// (ulp 1 there), giving 1024 + u exactly; subtracting 1032 leaves q = u - 8.
// A nibble sitting 4 bits higher gives 1024 + 16u, undone by *1/16 - 72.
// (The "magic number" integer-to-float conversion, as used for int4 weights
// by e.g. Kim et al., "Who Says Elephants Can't Run", 2022.)  Every step up
// to q is exact; the only rounding is q*s -> FP16.
DEV_INLINE void dequant_word(uint32_t w, __half2 s_lo, __half2 s_hi, uint32_t (&a)[4]) {
  const uint32_t kMagic = 0x64006400u;                // (1024, 1024)
  const __half2 k1032 = u32_as_h2(0x64086408u);       // (1032, 1032)
  const __half2 kSixteenth = u32_as_h2(0x2C002C00u);  // (1/16, 1/16)
  const __half2 kMinus72 = u32_as_h2(0xD480D480u);    // (-72, -72)
  const uint32_t w8 = w >> 8;
  __half2 q0 = __hsub2(u32_as_h2((w & 0x000F000Fu) | kMagic), k1032);
  __half2 q1 = __hfma2(u32_as_h2((w & 0x00F000F0u) | kMagic), kSixteenth, kMinus72);
  __half2 q2 = __hsub2(u32_as_h2((w8 & 0x000F000Fu) | kMagic), k1032);
  __half2 q3 = __hfma2(u32_as_h2((w8 & 0x00F000F0u) | kMagic), kSixteenth, kMinus72);
  a[0] = h2_as_u32(__hmul2(q0, s_lo));   // (row g,   k 2c..2c+1)
  a[1] = h2_as_u32(__hmul2(q1, s_hi));   // (row g+8, k 2c..2c+1)
  a[2] = h2_as_u32(__hmul2(q2, s_lo));   // (row g,   k 2c+8..+9)
  a[3] = h2_as_u32(__hmul2(q3, s_hi));   // (row g+8, k 2c+8..+9)
}

// D += A(16x16, row) * B(16x8, col), FP16 inputs, FP32 accumulation.
DEV_INLINE void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

DEV_INLINE float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

DEV_INLINE float silu_mul(float g, float u) { return g / (1.0f + __expf(-g)) * u; }

// Pointer to the 16-byte chunk (kc, rt, lane) of a matrix in a slot row.
DEV_INLINE const uint4* chunk_ptr(const uint8_t* slot_base, const MatLayout& m, int kc, int rt, int lane) {
  const uint4* q = reinterpret_cast<const uint4*>(slot_base + m.q_off);
  return q + ((size_t)kc * (m.rows / 16) + rt) * 32 + lane;
}

DEV_INLINE const __half* scale_ptr(const uint8_t* slot_base, const MatLayout& m) {
  return reinterpret_cast<const __half*>(slot_base + m.s_off);
}

// 128-bit streaming load that does not allocate in L1 (weights are read once).
DEV_INLINE uint4 ld_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
