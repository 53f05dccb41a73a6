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

// D += A(16x16, row) * B(16x8, col), FP16 inputs, FP32 accumulation.  Not
// volatile: a pure register operation the compiler may schedule among the
// dequantisation arithmetic (volatile asm serialises them, about 3x slower).
DEV_INLINE void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm(
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

DEV_INLINE float silu_mul(float g, float u) { return __fdividef(g, 1.0f + __expf(-g)) * u; }

// Start of 16-row tile rt of a matrix in a slot row (layout.h).
DEV_INLINE const uint8_t* tile_ptr(const uint8_t* slot_base, const MatLayout& m, int rt) {
  return slot_base + m.off + (size_t)rt * m.tile_bytes;
}

// ---------------------------------------------------------------- mbarrier
DEV_INLINE uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

DEV_INLINE void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

DEV_INLINE void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }

DEV_INLINE void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

DEV_INLINE void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

DEV_INLINE bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait on an mbarrier phase: gives up after ~2^31 SM cycles (about
// one second), records STATUS_TIMEOUT and returns false.  No wait in this
// library is unbounded.
#define MOE_WAIT_CYCLES (1ll << 31)
DEV_INLINE bool mbar_wait_limit(uint64_t* bar, uint32_t parity, DevStatus* st, long long limit) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > limit) {
      atomicOr(&st->flags, STATUS_TIMEOUT);
      return false;
    }
  }
  return true;
}
DEV_INLINE bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, DevStatus* st) {
  return mbar_wait_limit(bar, parity, st, MOE_WAIT_CYCLES);
}

// Bounded poll until *flag >= target (acquire loads); same give-up rule.
DEV_INLINE bool flag_wait_limit(const unsigned* flag, unsigned target, DevStatus* st, long long limit) {
  const long long t0 = clock64();
  for (;;) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(flag) : "memory");
    if (v >= target) return true;
    if (clock64() - t0 > limit) {
      atomicOr(&st->flags, STATUS_TIMEOUT);
      return false;
    }
    __nanosleep(256);
  }
}

// 1-D bulk async copy global -> shared (TMA, no tensor map), completing on bar.
// dst, src 16-byte aligned; bytes a multiple of 16.
DEV_INLINE void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// ------------------------------------------- programmatic dependent launch
// wait: block until the preceding grid in the stream completed and its
// memory is visible (no-op when not launched with the PDL attribute).
DEV_INLINE void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// allow the next grid in the stream to start launching.
DEV_INLINE void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ------------------------------------------------------------------ cluster
DEV_INLINE uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

DEV_INLINE void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Shared-memory address of `p` (in this CTA's smem) mapped into CTA `rank`.
DEV_INLINE uint32_t map_to_rank(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
  return r;
}

DEV_INLINE void st_cluster_f32(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

// 128-bit streaming load that does not allocate in L1 (weights are read once).
DEV_INLINE uint4 ld_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// ------------------------------------------------------- tcgen05 / TMEM / TMA
DEV_INLINE void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
DEV_INLINE void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
DEV_INLINE void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }

DEV_INLINE void tmem_alloc(uint32_t* dst, uint32_t ncols) {   // whole warp
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)), "r"(ncols)
               : "memory");
}
DEV_INLINE void tmem_relinquish() { asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;"); }
DEV_INLINE void tmem_dealloc(uint32_t taddr, uint32_t ncols) {   // whole warp
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// Two int4 codes (offset binary, bits 0-3 and 16-19 of w) -> FP16x2 nearest
// (q * s): 1024 + u exactly (the conversion of dequant_word), minus 1032,
// times the scale.
DEV_INLINE uint32_t dequant_pair(uint32_t w, __half2 s) {
  const __half2 k1032 = u32_as_h2(0x64086408u);
  return h2_as_u32(__hmul2(__hsub2(u32_as_h2((w & 0x000F000Fu) | 0x64006400u), k1032), s));
}

// D[tmem] (+)= A[tmem] * B[smem desc], FP16 inputs, FP32 accumulate (A: M
// lanes, K / 2 columns of FP16 pairs, lower K in the low half).
DEV_INLINE void umma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(acc)
      : "memory");
}

// 32 consecutive 32-bit TMEM columns of this thread's lane <- r.
DEV_INLINE void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
      "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
      "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
DEV_INLINE void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// D[tmem] (+)= A[smem desc] * B[smem desc], FP16 inputs, FP32 accumulate.
DEV_INLINE void umma_f16_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(acc)
      : "memory");
}

// Arrives on `bar` once every tcgen05.mma issued so far by this thread completed.
DEV_INLINE void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// 32 consecutive 32-bit TMEM columns of this thread's lane (warp quarter rule applies).
DEV_INLINE void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
// 16 consecutive 32-bit TMEM columns of this thread's lane.
DEV_INLINE void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
DEV_INLINE void tmem_ld_cols(uint32_t taddr, uint32_t (&r)[32]) { tmem_ld32(taddr, r); }
DEV_INLINE void tmem_ld_cols(uint32_t taddr, uint32_t (&r)[16]) { tmem_ld16(taddr, r); }
DEV_INLINE void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, rows of
// 128 B (64 FP16), 8-row groups 1024 B apart.
DEV_INLINE uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);   // start address
  d |= (uint64_t)1 << 16;                      // leading byte offset (unused for swizzled K-major)
  d |= (uint64_t)(1024 >> 4) << 32;            // stride byte offset: 8 rows x 128 B
  d |= (uint64_t)1 << 46;                      // descriptor version
  d |= (uint64_t)2 << 61;                      // 128-byte swizzle
  return d;
}

// Instruction descriptor of kind::f16: FP16 A and B (K-major), FP32 D, M x N.
DEV_INLINE uint32_t idesc_f16_f32(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// TMA: one box at (c0, r0) of a 2-D tensor map.
DEV_INLINE void tma_load_2d(void* dst, const void* tmap, int c0, int r0, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cta.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_u32(dst)),
      "l"(tmap), "r"(c0), "r"(r0), "r"(smem_u32(bar))
      : "memory");
}

// TMA: one box at (c0, c1, c2, c3) of a 4-D tensor map (no swizzle).
DEV_INLINE void tma_load_4d(void* dst, const void* tmap, int c0, int c1, int c2, int c3, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cta.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(smem_u32(dst)),
      "l"(tmap), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_u32(bar))
      : "memory");
}
