// moe_w4a16_route_noalloc: the routing launch sequence (logits, softmax/top-k,
// stable permutation) with every piece of scratch memory in one fixed,
// file-scope device array, for callers that may not allocate device memory.
//
// The array below is the only scratch these launches use.  Its host-side
// name is not a device address: host code obtains the device address with
// cudaGetSymbolAddress, once per device, with that device current, and passes
// the pointer to the kernels.  Every call shares the array, and it keeps the
// previous call's contents; the parts that must start cleared (the status
// word) are cleared by each call.
#include <mutex>

#include "moe_w4a16.h"
#include "internal.h"

#define MOE_NOALLOC_SCRATCH_BYTES (5u << 20)

static __device__ __align__(256) unsigned char g_route_scratch[MOE_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxTokens = MOE_W4A16_NOALLOC_MAX_TOKENS;
constexpr long long kMaxLogits = MOE_W4A16_NOALLOC_MAX_LOGITS;   // T * E * ceil(H / 256)
constexpr int kMaxHidden = MOE_W4A16_NOALLOC_MAX_HIDDEN;
constexpr int kMaxPairs = MOE_W4A16_NOALLOC_MAX_PAIRS;           // T * k
constexpr int kMaxE = 256;

// Byte offsets inside g_route_scratch.
constexpr size_t kOffLogits = 0;                                    // [H/256][T][E] f32 partial logits
constexpr size_t kOffSs = kOffLogits + (size_t)kMaxLogits * 4;      // [H/256][T] f32
constexpr size_t kOffRnorm = kOffSs + (size_t)kMaxTokens * (kMaxHidden / 256) * 4;   // [T] f32
constexpr size_t kOffSorted = kOffRnorm + (size_t)kMaxTokens * 4;   // [T*k] i32 (when the caller passes none)
constexpr size_t kOffP2r = kOffSorted + (size_t)kMaxPairs * 4;      // [T*k] i32
constexpr size_t kOffOffsets = kOffP2r + (size_t)kMaxPairs * 4;     // [E+1] i32 (when the caller passes none)
constexpr size_t kOffAct = kOffOffsets + 2048;                      // 5E+2 i32: active-expert lists
constexpr size_t kOffTable = kOffAct + 8192;                        // [E] i32 identity expert->slot
constexpr size_t kOffStatus = kOffTable + 1024;                     // DevStatus
constexpr size_t kOffCounter = kOffStatus + 256;                    // u32 arrival counter of the router scan
constexpr size_t kOffHist = kOffCounter + 256;                      // [ceil(T/8)][E] i32 block counts
constexpr size_t kMaxHist = (size_t)kMaxLogits / 8 + kMaxE;         // ceil(T/8) * E <= T*E/8 + E
constexpr size_t kOffEnd = kOffHist + kMaxHist * 4;
static_assert(kOffEnd <= MOE_NOALLOC_SCRATCH_BYTES, "scratch layout exceeds the static array");
static_assert((kMaxE + 1) * 4 <= 2048 && (5 * kMaxE + 2) * 4 <= 8192 && kMaxE * 4 <= 1024, "scratch slots");

std::mutex g_mu;
unsigned char* g_dev_ptr[128] = {};

// Identity expert->slot table (routing only: every expert counts as resident)
// and a cleared status word.  Device code names the array directly.
__global__ void noalloc_prepare_kernel(int E) {
  int32_t* table = reinterpret_cast<int32_t*>(g_route_scratch + kOffTable);
  for (int e = threadIdx.x; e < E; e += blockDim.x) table[e] = e;
  if (threadIdx.x == 0) {
    DevStatus* s = reinterpret_cast<DevStatus*>(g_route_scratch + kOffStatus);
    s->miss = 0;
    s->flags = 0;
    *reinterpret_cast<unsigned*>(g_route_scratch + kOffCounter) = 0u;
  }
}

moe_w4a16_status reject(const char* msg) {
  set_handle_free_error(msg);
  return MOE_W4A16_ERR_INVALID_ARG;
}

}  // namespace

extern "C" MOE_W4A16_API moe_w4a16_status moe_w4a16_route_noalloc(
    const void* x, int32_t T, int32_t hidden, int32_t num_experts, int32_t top_k, const void* router_w,
    const float* bias, uint32_t flags, int32_t* topk_ids, float* topk_w, int32_t* sorted_pairs,
    int32_t* expert_offsets, moe_w4a16_stream_t stream) {
  if (T < 0 || T > kMaxTokens) return reject("route_noalloc: T outside [0, MOE_W4A16_NOALLOC_MAX_TOKENS]");
  if (hidden < 64 || hidden % 64 || hidden > kMaxHidden)
    return reject("route_noalloc: hidden must be a multiple of 64 in [64, MOE_W4A16_NOALLOC_MAX_HIDDEN]");
  if (num_experts < 1 || num_experts > kMaxE) return reject("route_noalloc: num_experts outside [1, 256]");
  if (top_k < 1 || top_k > 32 || top_k > num_experts) return reject("route_noalloc: top_k outside [1, min(E, 32)]");
  const long long kslices = (hidden + 255) / 256;   // K slices of the router logits
  if ((long long)T * num_experts * kslices > kMaxLogits)
    return reject("route_noalloc: T * num_experts * ceil(hidden / 256) exceeds MOE_W4A16_NOALLOC_MAX_LOGITS");
  if ((long long)T * top_k > kMaxPairs) return reject("route_noalloc: T * top_k exceeds MOE_W4A16_NOALLOC_MAX_PAIRS");
  if (flags & ~(uint32_t)MOE_W4A16_PRENORM) return reject("route_noalloc: only the PRENORM flag applies");
  if (T == 0) return MOE_W4A16_OK;
  if (!x || !router_w || !topk_ids || !topk_w) return reject("route_noalloc: NULL x, router_w, topk_ids or topk_w");
  if (((uintptr_t)x | (uintptr_t)router_w) & 15u) return reject("route_noalloc: x and router_w must be 16-byte aligned");
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= 128) {
    cudaGetLastError();
    set_handle_free_error("route_noalloc: no current CUDA device");
    return MOE_W4A16_ERR_CUDA;
  }
  unsigned char* base = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_dev_ptr[dev]) {
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_route_scratch);
      if (e != cudaSuccess || !p) {
        cudaGetLastError();
        set_handle_free_error("route_noalloc: cudaGetSymbolAddress of the scratch array failed");
        return MOE_W4A16_ERR_CUDA;
      }
      g_dev_ptr[dev] = static_cast<unsigned char*>(p);
    }
    base = g_dev_ptr[dev];
  }
  FwdCtx c;
  memset(&c, 0, sizeof c);
  c.x = static_cast<const __half*>(x);
  c.T = T;
  c.router_w = static_cast<const __half*>(router_w);
  c.bias = bias;
  c.flags = flags;
  c.H = hidden;
  c.E = num_experts;
  c.k = top_k;
  c.table = reinterpret_cast<const int32_t*>(base + kOffTable);
  c.ksplit = 1;
  c.logit_part = reinterpret_cast<float*>(base + kOffLogits);
  c.ss_part = reinterpret_cast<float*>(base + kOffSs);
  c.rnorm = reinterpret_cast<float*>(base + kOffRnorm);
  c.ids = topk_ids;
  c.topw = topk_w;
  c.offsets = expert_offsets ? expert_offsets : reinterpret_cast<int32_t*>(base + kOffOffsets);
  c.sorted = sorted_pairs ? sorted_pairs : reinterpret_cast<int32_t*>(base + kOffSorted);
  c.p2r = reinterpret_cast<int32_t*>(base + kOffP2r);
  int32_t* act = reinterpret_cast<int32_t*>(base + kOffAct);
  c.act_expert = act;
  c.act_slot = act + num_experts;
  c.act_start = act + 2 * num_experts;
  c.act_count = act + 3 * num_experts;
  c.act_tile = act + 4 * num_experts;
  c.n_active = act + 5 * num_experts + 1;
  c.tile_tokens = 128;
  c.status = reinterpret_cast<DevStatus*>(base + kOffStatus);
  c.route_counter = reinterpret_cast<unsigned*>(base + kOffCounter);
  c.route_hist = reinterpret_cast<int32_t*>(base + kOffHist);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  noalloc_prepare_kernel<<<1, 256, 0, st>>>(num_experts);
  e = cudaGetLastError();
  if (e == cudaSuccess) e = launch_route(c, /*small=*/false, st);
  if (e != cudaSuccess) {
    cudaGetLastError();
    set_handle_free_error("route_noalloc: kernel launch failed");
    return MOE_W4A16_ERR_CUDA;
  }
  return MOE_W4A16_OK;
}
