// Prefill regime: persistent grouped GEMM on the 5th-generation tensor cores
// (tcgen05.mma, FP16 operands in shared memory, FP32 accumulators in TMEM).
//
// The compact int4 weights are the MMA A operand (M = 128 weight rows per
// tile); the tokens of one expert are the N dimension (N <= 256, padded only
// to a multiple of 16, so ragged expert loads waste little work).  Per 64-wide
// K step:
//   producer warp : one 4-D TMA load fetches the int4 chunks of the 8 row
//                   tiles of a matrix into a raw ring; the token rows of B come
//                   as 2-D TMA tiles, 128-byte swizzled (x gathered into
//                   sorted-row order by a small kernel for gate/up; h for down)
//   dequant warps : int4 -> FP16 (nearest q*s) written into a 128-byte
//                   swizzled K-major A ring (the only place an expanded value
//                   exists: one 64-wide K step of 128 rows, per CTA)
//   MMA warp      : one thread issues tcgen05.mma M128 x N x K16 (gate and up
//                   into two accumulators) and commits stage releases
//   epilogue warps: tcgen05.ld of the accumulators; gate/up: h = SiLU(g) * u
//                   rounded to FP16; down: y [pair][H] FP32
// A last kernel gathers out[t] = (x[t]) + sum_j w[t,j] y[t*k+j] in rank order.
// Every wait is bounded (status word + early exit), nothing spins forever.
// Sources: compact weights converted in-kernel with FP32 accumulation stages
// and explicit rounding (Horizon RunMap landing page, "08 / Precision &
// quality"); a grouped executor for the full-residency regime ("Horizon
// RunMap - architecture", "Regimes and executor boundaries").
#include <cuda.h>

#include "internal.h"

namespace {

constexpr int kMTile = 128;     // weight rows per tile (MMA M)
constexpr int kNMax = 256;      // tokens per tile (MMA N, max)
constexpr int kBK = 64;         // K per pipeline stage (one 128-byte swizzle row of FP16)
constexpr int kStagesRaw = 4;
constexpr int kStagesA = 2;
constexpr int kThreads = 320;   // warps 0-3 dequant, 4-7 epilogue, 8 producer, 9 MMA
constexpr uint32_t kTmemCols = 512;

template <bool GU>
struct Cfg {
  static constexpr int kMats = GU ? 2 : 1;
  static constexpr int kStagesB = GU ? 3 : 4;
  static constexpr int kAMat = kMTile * kBK * 2;          // 16 KB per matrix per stage
  static constexpr int kABytes = kMats * kAMat;
  static constexpr int kBBytes = kNMax * kBK * 2;         // 32 KB
  static constexpr int kRawBytes = kMats * 8 * 512;       // int4 chunks of 8 row tiles
  static constexpr int kOffA = 0;
  static constexpr int kOffB = kOffA + kStagesA * kABytes;
  static constexpr int kOffRaw = kOffB + kStagesB * kBBytes;
  static constexpr int kOffBar = kOffRaw + kStagesRaw * kRawBytes;
  static constexpr int kNumBars = 2 * kStagesRaw + 2 * kStagesA + 2 * kStagesB + 4;
  static constexpr int kSmem = kOffBar + kNumBars * 8 + 16 + 1024;   // + TMEM slot + alignment slack
};

struct Ring {
  int i = 0;
  uint32_t ph = 0;
  DEV_INLINE void next(int n) {
    if (++i == n) {
      i = 0;
      ph ^= 1u;
    }
  }
};

struct Tile {
  int slot, r0, n, m0;
};

// Tile t -> (active expert, token chunk, weight-row tile).  Chunks split an
// expert's rows into ceil(count / 256) near-equal parts.
DEV_INLINE bool get_tile(const FwdCtx& c, int t, int mtiles, Tile& out) {
  const int nact = *c.n_active;
  if (nact <= 0) return false;
  const int nchunks = c.act_tile[nact];
  if (t >= nchunks * mtiles) return false;
  const int mt = t % mtiles, ct = t / mtiles;
  int lo = 0, hi = nact - 1;
  while (lo < hi) {   // last u with act_tile[u] <= ct
    const int mid = (lo + hi + 1) >> 1;
    if (c.act_tile[mid] <= ct) lo = mid;
    else hi = mid - 1;
  }
  const int u = lo;
  const int nch = c.act_tile[u + 1] - c.act_tile[u], ch = ct - c.act_tile[u];
  const int cnt = c.act_count[u];
  const int b0 = (int)((long long)ch * cnt / nch), b1 = (int)((long long)(ch + 1) * cnt / nch);
  out.slot = c.act_slot[u];
  out.r0 = c.act_start[u] + b0;
  out.n = b1 - b0;
  out.m0 = mt * kMTile;
  return true;
}

DEV_INLINE void st_shared_b32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared.b32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

template <bool GU>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_kernel(FwdCtx c, const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmA0,
                        const __grid_constant__ CUtensorMap tmA1) {
  using C = Cfg<GU>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* raw_full = bars;
  uint64_t* raw_empty = raw_full + kStagesRaw;
  uint64_t* a_full = raw_empty + kStagesRaw;
  uint64_t* a_empty = a_full + kStagesA;
  uint64_t* b_full = a_empty + kStagesA;
  uint64_t* b_empty = b_full + C::kStagesB;
  uint64_t* acc_full = b_empty + C::kStagesB;   // [2]
  uint64_t* acc_empty = acc_full + 2;           // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  pdl_wait();      // routing (and, for down, h) of the preceding grids
  pdl_trigger();
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStagesRaw; ++s) {
      mbar_init(&raw_full[s], 1);
      mbar_init(&raw_empty[s], 4);
    }
    for (int s = 0; s < kStagesA; ++s) {
      mbar_init(&a_full[s], 4);
      mbar_init(&a_empty[s], 1);
    }
    for (int s = 0; s < C::kStagesB; ++s) {
      mbar_init(&b_full[s], 1);
      mbar_init(&b_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&acc_full[s], 1);
      mbar_init(&acc_empty[s], 4);
    }
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const MatLayout& LA = GU ? c.lay.gate : c.lay.down;
  const int K = (int)LA.k, nks = K / kBK, mtiles = (int)LA.rows / kMTile;
  const uint32_t TS = LA.tile_bytes, SB = LA.scale_bytes;
  const int nacc = GU ? 1 : 2;   // accumulator buffers (gate/up uses all 512 columns)

  if (warp == 8) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      Ring rr, rb;
      bool ok = true;
      for (int t = blockIdx.x; ok; t += gridDim.x) {
        Tile tl;
        if (!get_tile(c, t, mtiles, tl)) break;
        const int nq = (tl.n + 63) / 64;
        for (int ks = 0; ks < nks; ++ks) {
          if (!mbar_wait_bounded(&raw_empty[rr.i], rr.ph ^ 1u, c.status)) {
            ok = false;
            break;
          }
          uint8_t* dst = smem + C::kOffRaw + rr.i * C::kRawBytes;
          mbar_expect_tx(&raw_full[rr.i], C::kRawBytes);
          tma_load_4d(dst, &tmA0, 0, ks, tl.m0 / 16, tl.slot, &raw_full[rr.i]);
          if (GU) tma_load_4d(dst + 8 * 512, &tmA1, 0, ks, tl.m0 / 16, tl.slot, &raw_full[rr.i]);
          if (!mbar_wait_bounded(&b_empty[rb.i], rb.ph ^ 1u, c.status)) {
            ok = false;
            break;
          }
          uint8_t* bdst = smem + C::kOffB + rb.i * C::kBBytes;
          mbar_expect_tx(&b_full[rb.i], (uint32_t)nq * 64u * 128u);
          for (int q = 0; q < nq; ++q) tma_load_2d(bdst + q * 8192, &tmB, ks * kBK, tl.r0 + q * 64, &b_full[rb.i]);
          rr.next(kStagesRaw);
          rb.next(C::kStagesB);
        }
      }
    }
    __syncwarp();
  } else if (warp == 9) {
    // ---------------------------------------------------------------- MMA
    if (lane == 0) {
      Ring ra, rb, racc;
      bool ok = true;
      for (int t = blockIdx.x; ok; t += gridDim.x) {
        Tile tl;
        if (!get_tile(c, t, mtiles, tl)) break;
        const int n16 = (tl.n + 15) & ~15;
        const uint32_t idesc = idesc_f16_f32(kMTile, n16);
        if (!mbar_wait_bounded(&acc_empty[racc.i], racc.ph ^ 1u, c.status)) break;
        tc_fence_after();
        const uint32_t d0 = tmem + (GU ? 0u : (uint32_t)racc.i * 256u);
        for (int ks = 0; ks < nks; ++ks) {
          if (!mbar_wait_bounded(&a_full[ra.i], ra.ph, c.status) ||
              !mbar_wait_bounded(&b_full[rb.i], rb.ph, c.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_base = smem_u32(smem + C::kOffA + ra.i * C::kABytes);
          const uint32_t b_base = smem_u32(smem + C::kOffB + rb.i * C::kBBytes);
#pragma unroll
          for (int k16 = 0; k16 < kBK / 16; ++k16) {
            const uint64_t bdesc = sw128_desc(b_base + k16 * 32);
            const uint32_t acc = (ks | k16) != 0;
            umma_f16_ss(d0, sw128_desc(a_base + k16 * 32), bdesc, idesc, acc);
            if (GU) umma_f16_ss(tmem + 256u, sw128_desc(a_base + C::kAMat + k16 * 32), bdesc, idesc, acc);
          }
          umma_commit(&a_empty[ra.i]);
          umma_commit(&b_empty[rb.i]);
          ra.next(kStagesA);
          rb.next(C::kStagesB);
        }
        if (!ok) break;
        umma_commit(&acc_full[racc.i]);
        racc.next(nacc);
      }
    }
    __syncwarp();
  } else if (warp < 4) {
    // ------------------------------------------------------------ dequant
    const int g = lane >> 2, cq = lane & 3;
    Ring rr, ra;
    bool ok = true;
    for (int t = blockIdx.x; ok; t += gridDim.x) {
      Tile tl;
      if (!get_tile(c, t, mtiles, tl)) break;
      const uint8_t* base = c.pool + (size_t)tl.slot * c.slot_bytes;
      // Scales of the thread's rows: block b in use, block b+1 prefetched.
      __half2 slo[2][2], shi[2][2];
      __half nlo[2][2], nhi[2][2];
      auto load_scales = [&](int b, __half (&lo)[2][2], __half (&hi)[2][2]) {
#pragma unroll
        for (int m = 0; m < C::kMats; ++m) {
          const MatLayout& L = (GU && m == 1) ? c.lay.up : LA;
#pragma unroll
          for (int tt = 0; tt < 2; ++tt) {
            const __half* sc =
                reinterpret_cast<const __half*>(base + L.off + (size_t)(tl.m0 / 16 + warp * 2 + tt) * TS) + b * 16;
            lo[m][tt] = sc[g];
            hi[m][tt] = sc[g + 8];
          }
        }
      };
      load_scales(0, nlo, nhi);
      for (int ks = 0; ks < nks; ++ks) {
        if ((ks & 3) == 0) {
#pragma unroll
          for (int m = 0; m < C::kMats; ++m)
#pragma unroll
            for (int tt = 0; tt < 2; ++tt) {
              slo[m][tt] = __half2half2(nlo[m][tt]);
              shi[m][tt] = __half2half2(nhi[m][tt]);
            }
          if ((ks >> 2) + 1 < (int)LA.nb) load_scales((ks >> 2) + 1, nlo, nhi);
        }
        if (!mbar_wait_bounded(&raw_full[rr.i], rr.ph, c.status)) {
          ok = false;
          break;
        }
        uint4 q[2][2];
        const uint8_t* raw = smem + C::kOffRaw + rr.i * C::kRawBytes;
#pragma unroll
        for (int m = 0; m < C::kMats; ++m)
#pragma unroll
          for (int tt = 0; tt < 2; ++tt)
            q[m][tt] = *reinterpret_cast<const uint4*>(raw + (m * 8 + warp * 2 + tt) * 512 + lane * 16);
        __syncwarp();
        if (lane == 0) mbar_arrive(&raw_empty[rr.i]);
        if (!mbar_wait_bounded(&a_empty[ra.i], ra.ph ^ 1u, c.status)) {
          ok = false;
          break;
        }
        const uint32_t abase = smem_u32(smem + C::kOffA + ra.i * C::kABytes);
#pragma unroll
        for (int m = 0; m < C::kMats; ++m) {
#pragma unroll
          for (int tt = 0; tt < 2; ++tt) {
            const int row = (warp * 2 + tt) * 16 + g;   // and row + 8 (same swizzle phase)
            const uint32_t rlo = abase + m * C::kAMat + row * 128 + cq * 4;
            const uint32_t rhi = rlo + 8 * 128;
            const uint32_t sw = (uint32_t)(row & 7);
            const uint32_t w4[4] = {q[m][tt].x, q[m][tt].y, q[m][tt].z, q[m][tt].w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              uint32_t a[4];
              dequant_word(w4[j], slo[m][tt], shi[m][tt], a);
              const uint32_t c0 = ((uint32_t)(2 * j) ^ sw) << 4, c1 = ((uint32_t)(2 * j + 1) ^ sw) << 4;
              st_shared_b32(rlo + c0, a[0]);
              st_shared_b32(rhi + c0, a[1]);
              st_shared_b32(rlo + c1, a[2]);
              st_shared_b32(rhi + c1, a[3]);
            }
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&a_full[ra.i]);
        rr.next(kStagesRaw);
        ra.next(kStagesA);
      }
    }
  } else {
    // ----------------------------------------------------------- epilogue
    const int qw = warp & 3;
    const int row = qw * 32 + lane;
    Ring racc;
    for (int t = blockIdx.x;; t += gridDim.x) {
      Tile tl;
      if (!get_tile(c, t, mtiles, tl)) break;
      if (!mbar_wait_bounded(&acc_full[racc.i], racc.ph, c.status)) break;
      tc_fence_after();
      const uint32_t taddr = tmem + ((uint32_t)(qw * 32) << 16) + (GU ? 0u : (uint32_t)racc.i * 256u);
      for (int col0 = 0; col0 < tl.n; col0 += 32) {
        uint32_t va[32], vb[32];
        tmem_ld32(taddr + col0, va);
        if (GU) tmem_ld32(taddr + 256u + col0, vb);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int nn = col0 + j;
          if (nn < tl.n) {
            if (GU) {
              float gv = __uint_as_float(va[j]), uv = __uint_as_float(vb[j]);
              if (c.flags & 2u) {
                const float r = c.rnorm[c.sorted[tl.r0 + nn] / c.k];
                gv *= r;
                uv *= r;
              }
              c.hbuf[(size_t)(tl.r0 + nn) * c.I + tl.m0 + row] = __float2half_rn(silu_mul(gv, uv));
            } else {
              const int pair = c.sorted[tl.r0 + nn];
              c.ybuf[(size_t)pair * c.H + tl.m0 + row] = __uint_as_float(va[j]);
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[racc.i]);
      racc.next(nacc);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// out[t] = (x[t]) + sum_j w[t,j] y[t*k+j] in rank order j, FP32, then FP16.
__global__ void __launch_bounds__(256) combine_kernel(FwdCtx c) {
  pdl_wait();
  pdl_trigger();
  const int t = blockIdx.x;
  const int H = c.H;
  for (int v = threadIdx.x; v < H / 8; v += blockDim.x) {
    float acc[8];
    if (c.flags & 1u) {
      const uint4 xv = *reinterpret_cast<const uint4*>(c.x + (size_t)t * H + v * 8);
      const __half2* xh = reinterpret_cast<const __half2*>(&xv);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = __half22float2(xh[i]);
        acc[2 * i] = f.x;
        acc[2 * i + 1] = f.y;
      }
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = 0.f;
    }
    for (int j = 0; j < c.k; ++j) {
      const int p = t * c.k + j;
      if (c.table[c.ids[p]] < 0) continue;
      const float w = c.topw[p];
      const float4* yp = reinterpret_cast<const float4*>(c.ybuf + (size_t)p * H + v * 8);
      const float4 y0 = yp[0], y1 = yp[1];
      acc[0] = fmaf(w, y0.x, acc[0]);
      acc[1] = fmaf(w, y0.y, acc[1]);
      acc[2] = fmaf(w, y0.z, acc[2]);
      acc[3] = fmaf(w, y0.w, acc[3]);
      acc[4] = fmaf(w, y1.x, acc[4]);
      acc[5] = fmaf(w, y1.y, acc[5]);
      acc[6] = fmaf(w, y1.z, acc[6]);
      acc[7] = fmaf(w, y1.w, acc[7]);
    }
    uint4 o;
    __half2* oh = reinterpret_cast<__half2*>(&o);
#pragma unroll
    for (int i = 0; i < 4; ++i) oh[i] = __floats2half2_rn(acc[2 * i], acc[2 * i + 1]);
    *reinterpret_cast<uint4*>(c.out + (size_t)t * H + v * 8) = o;
  }
}

// xp[r] = x[sorted[r] / k]: activations in sorted-row order (one row per CTA).
__global__ void __launch_bounds__(256) gather_rows_kernel(FwdCtx c) {
  pdl_wait();
  pdl_trigger();
  const int r = blockIdx.x;
  const int tok = c.sorted[r] / c.k;
  const uint4* src = reinterpret_cast<const uint4*>(c.x + (size_t)tok * c.H);
  uint4* dst = reinterpret_cast<uint4*>(c.xp + (size_t)r * c.H);
  for (int v = threadIdx.x; v < c.H / 8; v += blockDim.x) dst[v] = __ldg(src + v);
}

// ------------------------------------------------------------ tensor maps
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPoint("cuTensorMapEncodeTiled", &p, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
    else
      cudaGetLastError();
  }
  return fn;
}

// Row-major FP16 matrix [rows][cols] (cols contiguous), box of box_rows x 64
// columns, 128-byte swizzle, zero fill out of range.
bool make_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {64, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool gemm_shapes_supported(int H, int I) { return H % kMTile == 0 && I % kMTile == 0; }

PoolMaps make_pool_maps(const uint8_t* pool, const SlotLayout& lay, int num_slots) {
  PoolMaps pm;
  memset(&pm, 0, sizeof pm);
  pm.ok = false;
  EncodeTiledFn fn = encode_fn();
  if (!fn || !gemm_shapes_supported((int)lay.down.rows, (int)lay.gate.rows)) return pm;
  const MatLayout* mats[3] = {&lay.gate, &lay.up, &lay.down};
  for (int i = 0; i < 3; ++i) {
    const MatLayout& L = *mats[i];
    // [slot][row tile][K chunk][128 x u32 = 512 B], packed int4 part of each tile
    const cuuint64_t dims[4] = {128, L.k / 64, L.rows / 16, (cuuint64_t)num_slots};
    const cuuint64_t strides[3] = {512, L.tile_bytes, lay.bytes};
    const cuuint32_t box[4] = {128, 1, 8, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    if (fn(&pm.q[i], CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, const_cast<uint8_t*>(pool + L.off + L.scale_bytes), dims,
           strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return pm;
  }
  pm.ok = true;
  return pm;
}

cudaError_t launch_gemm_experts(const FwdCtx& c, const PoolMaps& pm, cudaStream_t st, const StageEvents& se) {
  if (!gemm_shapes_supported(c.H, c.I) || !pm.ok) return cudaErrorNotSupported;
  const uint64_t P = (uint64_t)c.T * c.k;
  CUtensorMap mx, mh;
  if (!make_map(&mx, c.xp, P, (uint64_t)c.H, 64) || !make_map(&mh, c.hbuf, P, (uint64_t)c.I, 64))
    return cudaErrorNotSupported;
  cudaError_t e = opt_in_smem((const void*)grouped_gemm_kernel<true>, Cfg<true>::kSmem);
  if (e == cudaSuccess) e = opt_in_smem((const void*)grouped_gemm_kernel<false>, Cfg<false>::kSmem);
  if (e != cudaSuccess) return e;
  const int grid = c.num_sms > 0 ? c.num_sms : 148;
  e = launch_pdl(gather_rows_kernel, dim3((unsigned)P), dim3(256), 0, st, 1, c);
  if (e == cudaSuccess)
    e = launch_pdl(grouped_gemm_kernel<true>, dim3(grid), dim3(kThreads), Cfg<true>::kSmem, st, 1, c, mx, pm.q[0],
                   pm.q[1]);
  if (e == cudaSuccess) e = record_stage(se, 2, st);
  if (e == cudaSuccess)
    e = launch_pdl(grouped_gemm_kernel<false>, dim3(grid), dim3(kThreads), Cfg<false>::kSmem, st, 1, c, mh, pm.q[2],
                   pm.q[2]);
  if (e == cudaSuccess) e = record_stage(se, 3, st);
  if (e == cudaSuccess) e = launch_pdl(combine_kernel, dim3(c.T), dim3(256), 0, st, 1, c);
  if (e == cudaSuccess) e = record_stage(se, 4, st);
  return e;
}
