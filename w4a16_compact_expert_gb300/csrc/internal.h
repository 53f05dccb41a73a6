// Internal (non-ABI) declarations shared by the host runtime and the kernels.
#pragma once
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "layout.h"

// Everything one forward needs, resolved by the host runtime.
struct FwdCtx {
  // problem
  const __half* x;
  int T;
  const __half* router_w;
  const float* bias;
  uint32_t flags;
  __half* out;
  int H, I, E, k;
  // experts
  const uint8_t* pool;
  uint64_t slot_bytes;
  SlotLayout lay;
  const int32_t* table;        // [E] expert -> slot, -1 absent
  // routing workspaces
  int ksplit;                  // K split of the router logits
  float* logit_part;           // [ksplit][T][E]
  float* ss_part;              // [ksplit][T] partial sum of squares (PRENORM)
  float* rnorm;                // [T] 1/rms (PRENORM) else unused
  int32_t* ids;                // [T*k]
  float* topw;                 // [T*k]
  int32_t* offsets;            // [E+1]
  int32_t* sorted;             // [T*k] sorted row -> flat pair
  int32_t* p2r;                // [T*k] flat pair -> sorted row
  int32_t* act_expert;         // [E] active (routed and resident) experts, ascending
  int32_t* act_slot;           // [E]
  int32_t* act_start;          // [E] first sorted row of the group
  int32_t* act_count;          // [E] rows of the group
  int32_t* act_tile;           // [E+1] prefix of token tiles per active expert
  int32_t* n_active;           // [1]
  int tile_tokens;             // token tile of the grouped GEMM
  // expert workspaces
  __half* xp;                  // [T*k][H] activations gathered in sorted-row order (prefill)
  __half* hbuf;                // [T*k][I] SiLU*up in sorted-row order
  float* ybuf;                 // [T*k][H] per-pair expert output in flat pair order (FP32; FP16 on the grouped-GEMM path)
  int32_t* route_hist;         // [ceil(T/8) + 1][E] per 8-token block expert counts, then bases; last row: totals
  unsigned* route_counter;     // [1] arrival counter of the large-T router's scan (self-resetting)
  unsigned long long* route_bar;  // [2] grid-barrier counters of the cooperative router (monotonic; one grid size each)
  unsigned* down_counters;     // [H/32] arrival counters (self-resetting)
  unsigned long long* grid_bar;  // grid-barrier arrivals (monotonic, a multiple of the grid between uses)
  unsigned* expert_ready;      // [2][256]: [u] finished gate/up items of active expert u (the fused kernel); the rest unused
  DevStatus* status;
  int num_sms;
  int max_active;              // upper bound of active experts: min(E, T*k)
  // offload-qpacked comparison path: FP16 execution slots
  __half* xpool;               // [xslots][gate I*H | up I*H | down H*I], row-major, K contiguous
  uint64_t xslot_halves;       // halves per execution slot (3 I H)
  int xslots;                  // execution slots
  int ub0, ub1;                // the active experts [ub0, ub1) expanded into slots 0 .. ub1 - ub0 - 1
};

// Device counter block of a handle, in 32-bit words: [0, 2) the 64-bit grid
// barrier, [2, 2 + H/32) down arrival counters, then [2][256] per-expert
// readiness counters, the large-T router's arrival counter, the cooperative
// router's two 64-bit grid-barrier counters (8-byte aligned) and a last word
// that nothing writes.  Zero-initialised; every user leaves it zero (the
// grid barriers: a multiple of their grid size).
// the word after the readiness counters: the large-T router's arrival counter
inline size_t route_counter_word(int H) { return 2 + (size_t)H / 32 + 2 * 256; }
inline size_t route_bar_word(int H) { return (route_counter_word(H) + 2) & ~(size_t)1; }
inline size_t counter_words(int H) { return route_bar_word(H) + 5; }
// the last word of the counter block: never written by any kernel (the
// self-test waits on it)
inline size_t never_set_word(int H) { return counter_words(H) - 1; }

// selftest.cu: one kernel whose only wait can never be satisfied.
cudaError_t launch_selftest_wait(DevStatus* st, const unsigned* never_set, int which, long long limit,
                                 cudaStream_t s);

// repack.cu
cudaError_t launch_repack_matrix(const uint8_t* q, const uint16_t* s, uint8_t* slot_base,
                                 const MatLayout& m, cudaStream_t st);

// route.cu
cudaError_t launch_route(const FwdCtx& c, bool fused, cudaStream_t st);
bool route_single_launch(const FwdCtx& c);   // launch_route(small=true) is one kernel

// Records the optional stage event `i` of a forward (no-op when unset).
struct StageEvents {
  cudaEvent_t ev[5];
  bool on;
};
cudaError_t record_stage(const StageEvents& se, int i, cudaStream_t st);

// gemv.cu: decode regime (gate/up kernel, then down kernel with the combine)
cudaError_t launch_gemv_experts(const FwdCtx& c, cudaStream_t st, const StageEvents& se);

// decode_fused.cu: one cooperative launch per forward for small T
bool fused_decode_supported(const FwdCtx& c, int max_smem);
cudaError_t launch_fused_decode(const FwdCtx& c, cudaStream_t st, const StageEvents& se);

// gemm_tc.cu: prefill regime (gather, gate/up GEMM, down GEMM, combine)
bool gemm_shapes_supported(int H, int I);
// Token tile of the grouped GEMM for T tokens (routing chunks each expert's
// rows with it), by the average pairs per expert: 32 up to 16 (weights
// through tensor memory), 128 up to 64 (two accumulators), else 256.
int gemm_tile_tokens(int T, int k, int E);

// TMA maps over the whole slot pool for the grouped GEMM, built once per
// handle: q, the packed int4 chunks of gate, up and down ([slot][row tile][K
// chunk][512 B]), and sc, their block scales ([slot][row tile][block][16
// FP16]), boxes of 8 row tiles.
struct PoolMaps {
  CUtensorMap q[3];
  CUtensorMap sc[3];
  bool ok;
};
PoolMaps make_pool_maps(const uint8_t* pool, const SlotLayout& lay, int num_slots);
// gathered: c.xp already holds the x rows in sorted-row order (else the first
// launch gathers them).
cudaError_t launch_gemm_experts(const FwdCtx& c, const PoolMaps& pm, bool gathered, cudaStream_t st,
                                const StageEvents& se);

// The offload-qpacked comparison path: each batch of at most xslots active
// experts is expanded into FP16 execution slots (offload.cu), then the same
// grouped GEMM runs with dense FP16 A tiles loaded by TMA (gemm_tc.cu).
struct DenseMaps {
  CUtensorMap a[3];   // gate, up, down of the execution slots: [slot][rows][K] FP16, boxes of 128 rows x 64 K
  bool ok;
};
DenseMaps make_dense_maps(const __half* xpool, int H, int I, int xslots);
cudaError_t launch_expand(const FwdCtx& c, cudaStream_t st);   // active experts [c.ub0, c.ub1)
cudaError_t launch_offload_experts(const FwdCtx& c, const DenseMaps& dm, bool gathered, cudaStream_t st,
                                   const StageEvents& se);

// route.cu, above the single-launch cluster router: one cooperative kernel
// for the logits, softmax / top-k and the permutation, and with `gather` the
// copy of the routed x rows into sorted-row order (c.xp).
cudaError_t launch_route_gather(const FwdCtx& c, bool gather, cudaStream_t st);

// route: the largest T handled by the single-launch cluster router (its
// 8 CTAs take about 4 us per 8 tokens; the cooperative router is faster above)
#define ROUTE_FUSED_MAX_T 8

// gemv.cu: dynamic shared memory of the decode kernels for `rows` staged tokens.
size_t gemv_smem_gateup(int H, int I, int rows);
size_t gemv_smem_down(int H, int I, int rows);

// Sets the message returned by moe_w4a16_last_error(NULL) (calls without a handle).
void set_handle_free_error(const char* msg);

// Raises a kernel's dynamic shared-memory limit to at least `bytes` (once per
// device and value; thread-safe).
cudaError_t opt_in_smem(const void* func, size_t bytes);

// Launch with programmatic dependent launch allowed (the kernel must call
// griddepcontrol.wait before consuming the preceding grid's output) and an
// optional 1-D thread-block cluster.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       int cluster, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  int n = 0;
  attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  if (cluster > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = cluster;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}
