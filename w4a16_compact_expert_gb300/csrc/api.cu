// Host runtime behind the C ABI (include/moe_w4a16.h): handle lifetime, slot
// pool, expert packing, slot table, forward dispatch and the status word.
//
// "Capacity is fixed before admission" (Horizon RunMap - architecture,
// section "Immutable authority and miss lifecycle"): create allocates the
// pool and every workspace; forward allocates nothing and never waits on the
// host.  "An expert being resident does not mean it is routed" (same page,
// "Regimes and executor boundaries"): slots and the expert->slot table are
// separate objects.
#include <algorithm>
#include <cstdio>
#include <mutex>
#include <cstring>
#include <string>
#include <vector>

#include "moe_w4a16.h"
#include "internal.h"
#include "handle.h"

namespace {

thread_local std::string g_create_err;

struct DeviceGuard {
  int prev = -1;
  bool ok = false;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
    ok = cudaSetDevice(dev) == cudaSuccess;
  }
  ~DeviceGuard() {
    if (prev >= 0) cudaSetDevice(prev);
  }
};

moe_w4a16_status fail(moe_w4a16_handle* h, moe_w4a16_status s, const std::string& msg) {
  if (h) h->err = msg;
  return s;
}

moe_w4a16_status cuda_fail(moe_w4a16_handle* h, cudaError_t e, const char* what) {
  cudaGetLastError();
  return fail(h, MOE_W4A16_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

template <typename T>
cudaError_t dalloc(moe_w4a16_handle* h, T** p, size_t count) {
  void* v = nullptr;
  cudaError_t e = cudaMalloc(&v, count * sizeof(T) > 0 ? count * sizeof(T) : 16);
  if (e == cudaSuccess) {
    h->allocs.push_back(v);
    *p = static_cast<T*>(v);
  }
  return e;
}

void free_all(moe_w4a16_handle* h) {
  for (void* p : h->allocs) cudaFree(p);
  h->allocs.clear();
}

bool is_device_ptr(const void* p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged;
}

int fused_ksplit(int H) {
  if (H % 256 != 0) return 1;
  const int nblk = H / 256;
  int ks = nblk < 8 ? nblk : 8;
  while (nblk % ks) --ks;
  return ks;
}

}  // namespace

void set_handle_free_error(const char* msg) { g_create_err = msg; }

cudaError_t opt_in_smem(const void* func, size_t bytes) {
  if (bytes <= 48 * 1024) return cudaSuccess;
  struct Entry {
    const void* f;
    int dev;
    size_t v;
  };
  static std::mutex mu;
  static std::vector<Entry> done;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  for (const Entry& x : done)
    if (x.f == func && x.dev == dev && x.v >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess) done.push_back({func, dev, bytes});
  return e;
}

cudaError_t record_stage(const StageEvents& se, int i, cudaStream_t st) {
  if (!se.on) return cudaSuccess;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(st, &cs);
  if (e != cudaSuccess) return e;
  if (cs == cudaStreamCaptureStatusActive) return cudaEventRecordWithFlags(se.ev[i], st, cudaEventRecordExternal);
  return cudaEventRecord(se.ev[i], st);
}

extern "C" {

moe_w4a16_status moe_w4a16_create(const moe_w4a16_config* cfg, moe_w4a16_handle** out) {
  if (!out) {
    g_create_err = "out is NULL";
    return MOE_W4A16_ERR_INVALID_ARG;
  }
  *out = nullptr;
  if (!cfg) {
    g_create_err = "cfg is NULL";
    return MOE_W4A16_ERR_INVALID_ARG;
  }
  const moe_w4a16_config c = *cfg;
  char buf[256];
  if (c.hidden < 2 || c.inter < 2 || (c.hidden & 1) || (c.inter & 1)) {
    snprintf(buf, sizeof buf, "hidden (%d) and inter (%d) must be even and >= 2", c.hidden, c.inter);
    g_create_err = buf;
    return MOE_W4A16_ERR_INVALID_ARG;
  }
  if (c.hidden % 64 || c.inter % 64) {
    snprintf(buf, sizeof buf, "hidden (%d) and inter (%d) must be multiples of 64 in this build", c.hidden, c.inter);
    g_create_err = buf;
    return MOE_W4A16_ERR_UNSUPPORTED;
  }
  if (c.num_experts < 1 || c.num_experts > 256 || c.top_k < 1 || c.top_k > 32 || c.top_k > c.num_experts ||
      c.num_slots < 1 || c.num_slots > 65535 || c.max_tokens < 1 || c.device < 0) {
    snprintf(buf, sizeof buf, "bad config: E=%d k=%d S=%d max_tokens=%d device=%d", c.num_experts, c.top_k,
             c.num_slots, c.max_tokens, c.device);
    g_create_err = buf;
    return MOE_W4A16_ERR_INVALID_ARG;
  }
  if (gemv_smem_gateup(c.hidden, c.inter, 8) > 220 * 1024 || gemv_smem_down(c.hidden, c.inter, 8) > 220 * 1024) {
    snprintf(buf, sizeof buf, "hidden %d / inter %d too large for the decode kernels' shared memory", c.hidden,
             c.inter);
    g_create_err = buf;
    return MOE_W4A16_ERR_UNSUPPORTED;
  }
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess || c.device >= ndev) {
    cudaGetLastError();
    snprintf(buf, sizeof buf, "CUDA device %d not available", c.device);
    g_create_err = buf;
    return MOE_W4A16_ERR_CUDA;
  }
  DeviceGuard dg(c.device);
  moe_w4a16_handle* h = new moe_w4a16_handle();
  h->cfg = c;
  h->lay = moe_slot_layout(c.hidden, c.inter);
  cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, c.device);
  cudaDeviceGetAttribute(&h->max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, c.device);
  h->ksplit_fused = fused_ksplit(c.hidden);
  h->gemv_max_tokens = 40;   // between the stack sweep's T = 32 (decode kernels faster) and T = 48 (GEMM faster)
  h->packed.assign(c.num_slots, 0);
  h->h_table.assign(c.num_experts, -1);
  const size_t H = c.hidden, I = c.inter, E = c.num_experts, T = c.max_tokens, P = T * c.top_k;
  const size_t nb_h = (H + 255) / 256, nb_i = (I + 255) / 256;
  h->stage_bytes = std::max(I * H / 2 + I * nb_h * 2, H * I / 2 + H * nb_i * 2) + 256;
  cudaError_t e = cudaSuccess;
#define ALLOC(ptr, n) \
  if (e == cudaSuccess) e = dalloc(h, &(ptr), (n))
  ALLOC(h->pool, (size_t)c.num_slots * h->lay.bytes);
  ALLOC(h->d_table, E);
  const size_t kslices = std::max<size_t>(8, (H + 255) / 256);   // router K slices
  ALLOC(h->logit_part, kslices * T * E);
  ALLOC(h->ss_part, kslices * T);
  ALLOC(h->rnorm, T);
  ALLOC(h->ids, P);
  ALLOC(h->topw, P);
  ALLOC(h->offsets, E + 1);
  ALLOC(h->sorted, P);
  ALLOC(h->p2r, P);
  ALLOC(h->act, 5 * E + 2 + 1);
  ALLOC(h->route_hist, (size_t)((T + 7) / 8 + 1) * E);   // + a row of expert totals (cooperative router)
  ALLOC(h->xp, P * H);
  ALLOC(h->hbuf, P * I);
  ALLOC(h->ybuf, P * H);
  ALLOC(h->counters, counter_words(H));
  ALLOC(h->status, 1);
  ALLOC(h->stage, h->stage_bytes);
  ALLOC(h->x_dev, T * H);
  ALLOC(h->out_dev, T * H);
#undef ALLOC
  if (e == cudaSuccess) e = cudaMemset(h->counters, 0, counter_words(H) * sizeof(unsigned));
  if (e == cudaSuccess) e = cudaMemset(h->status, 0, sizeof(DevStatus));
  if (e == cudaSuccess) e = cudaMemset(h->d_table, 0xff, E * sizeof(int32_t));
  h->cur_table = h->d_table;
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e == cudaSuccess) h->maps = make_pool_maps(h->pool, h->lay, c.num_slots);
  if (e != cudaSuccess) {
    const bool oom = e == cudaErrorMemoryAllocation;
    cudaGetLastError();
    g_create_err = std::string(oom ? "device allocation failed: " : "CUDA error at create: ") + cudaGetErrorString(e);
    free_all(h);
    delete h;
    return oom ? MOE_W4A16_ERR_OOM : MOE_W4A16_ERR_CUDA;
  }
  *out = h;
  return MOE_W4A16_OK;
}

moe_w4a16_status moe_w4a16_destroy(moe_w4a16_handle* h) {
  if (!h) return MOE_W4A16_OK;
  if (h->cache) return fail(h, MOE_W4A16_ERR_INVALID_ARG, "destroy the expert cache attached to this handle first");
  {
    DeviceGuard dg(h->cfg.device);
    cudaDeviceSynchronize();
    free_all(h);
  }
  delete h;
  return MOE_W4A16_OK;
}

moe_w4a16_status moe_w4a16_set_stage_events(moe_w4a16_handle* h, void* const* events) {
  if (!h) return MOE_W4A16_ERR_INVALID_ARG;
  if (!events) {
    h->events.on = false;
    return MOE_W4A16_OK;
  }
  for (int i = 0; i < 5; ++i) {
    if (!events[i]) return fail(h, MOE_W4A16_ERR_INVALID_ARG, "NULL stage event");
    h->events.ev[i] = static_cast<cudaEvent_t>(events[i]);
  }
  h->events.on = true;
  return MOE_W4A16_OK;
}

size_t moe_w4a16_slot_bytes(const moe_w4a16_handle* h) { return h ? (size_t)h->lay.bytes : 0; }

int32_t moe_w4a16_get_gemv_max_tokens(const moe_w4a16_handle* h) { return h ? h->gemv_max_tokens : -1; }

moe_w4a16_status moe_w4a16_set_gemv_max_tokens(moe_w4a16_handle* h, int32_t t_star) {
  if (!h) return MOE_W4A16_ERR_INVALID_ARG;
  if (t_star < 0) return fail(h, MOE_W4A16_ERR_INVALID_ARG, "gemv_max_tokens must be >= 0");
  h->gemv_max_tokens = t_star;
  return MOE_W4A16_OK;
}

moe_w4a16_status moe_w4a16_offload_enable(moe_w4a16_handle* h, int32_t n_slots) {
  if (!h) return MOE_W4A16_ERR_INVALID_ARG;
  if (n_slots < 1 || n_slots > 64) return fail(h, MOE_W4A16_ERR_INVALID_ARG, "n_slots outside [1, 64]");
  if (!gemm_shapes_supported(h->cfg.hidden, h->cfg.inter))
    return fail(h, MOE_W4A16_ERR_INVALID_ARG, "the grouped GEMM does not take these shapes");
  DeviceGuard dg(h->cfg.device);
  if (!dg.ok) return fail(h, MOE_W4A16_ERR_CUDA, "cudaSetDevice failed");
  if (h->xpool) {   // replace the previous execution slots
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(h, e, "synchronize before freeing the execution slots");
    for (size_t i = 0; i < h->allocs.size(); ++i)
      if (h->allocs[i] == h->xpool) {
        cudaFree(h->allocs[i]);
        h->allocs.erase(h->allocs.begin() + (long)i);
        break;
      }
    h->xpool = nullptr;
    h->xslots = 0;
  }
  const size_t halves = (size_t)n_slots * 3 * h->cfg.inter * h->cfg.hidden;
  cudaError_t e = dalloc(h, &h->xpool, halves);
  if (e != cudaSuccess) return cuda_fail(h, e, "execution slot allocation");
  h->dmaps = make_dense_maps(h->xpool, h->cfg.hidden, h->cfg.inter, n_slots);
  if (!h->dmaps.ok) return fail(h, MOE_W4A16_ERR_CUDA, "execution slot tensor maps");
  h->xslots = n_slots;
  return MOE_W4A16_OK;
}

moe_w4a16_status moe_w4a16_pack_experts(moe_w4a16_handle* h, int32_t slot0, int32_t n, const uint8_t* gate_q,
                                        const uint16_t* gate_s, const uint8_t* up_q, const uint16_t* up_s,
                                        const uint8_t* down_q, const uint16_t* down_s, moe_w4a16_stream_t stream) {
  if (!h) return MOE_W4A16_ERR_INVALID_ARG;
  if (h->cache) return fail(h, MOE_W4A16_ERR_INVALID_ARG, "an expert cache owns the slot rows of this handle");
  if (n < 0 || slot0 < 0 || (int64_t)slot0 + n > h->cfg.num_slots)
    return fail(h, MOE_W4A16_ERR_INVALID_ARG, "slot range [slot0, slot0+n) outside the pool");
  if (n == 0) return MOE_W4A16_OK;
  if (!gate_q || !gate_s || !up_q || !up_s || !down_q || !down_s)
    return fail(h, MOE_W4A16_ERR_INVALID_ARG, "NULL expert array");
  DeviceGuard dg(h->cfg.device);
  if (!dg.ok) return fail(h, MOE_W4A16_ERR_CUDA, "cudaSetDevice failed");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const MatLayout* mats[3] = {&h->lay.gate, &h->lay.up, &h->lay.down};
  const uint8_t* qs[3] = {gate_q, up_q, down_q};
  const uint16_t* ss[3] = {gate_s, up_s, down_s};
  bool on_dev_q[3], on_dev_s[3];
  for (int m = 0; m < 3; ++m) {
    on_dev_q[m] = is_device_ptr(qs[m]);
    on_dev_s[m] = is_device_ptr(ss[m]);
  }
  for (int i = 0; i < n; ++i) {
    uint8_t* slot_base = h->pool + (size_t)(slot0 + i) * h->lay.bytes;
    for (int m = 0; m < 3; ++m) {
      const MatLayout& L = *mats[m];
      const size_t qbytes = (size_t)L.rows * L.k / 2, sbytes = (size_t)L.rows * L.nb * 2;
      const uint8_t* q = qs[m] + (size_t)i * qbytes;
      const uint16_t* s = ss[m] + (size_t)i * L.rows * L.nb;
      cudaError_t e = cudaSuccess;
      if (!on_dev_q[m]) {
        e = cudaMemcpyAsync(h->stage, q, qbytes, cudaMemcpyHostToDevice, st);
        q = h->stage;
      }
      if (e == cudaSuccess && !on_dev_s[m]) {
        uint8_t* sdst = h->stage + ((qbytes + 255) / 256) * 256;
        e = cudaMemcpyAsync(sdst, s, sbytes, cudaMemcpyHostToDevice, st);
        s = reinterpret_cast<const uint16_t*>(sdst);
      }
      if (e == cudaSuccess) e = launch_repack_matrix(q, s, slot_base, L, st);
      if (e != cudaSuccess) return cuda_fail(h, e, "pack_experts");
    }
    h->packed[slot0 + i] = 1;
  }
  return MOE_W4A16_OK;
}

moe_w4a16_status moe_w4a16_set_slot_table(moe_w4a16_handle* h, const int32_t* expert_to_slot,
                                          moe_w4a16_stream_t stream) {
  if (!h) return MOE_W4A16_ERR_INVALID_ARG;
  if (!expert_to_slot) return fail(h, MOE_W4A16_ERR_INVALID_ARG, "expert_to_slot is NULL");
  if (h->cache) return fail(h, MOE_W4A16_ERR_INVALID_ARG, "an expert cache owns the slot table of this handle");
  const int E = h->cfg.num_experts, S = h->cfg.num_slots;
  std::vector<uint8_t> used(S, 0);
  for (int e = 0; e < E; ++e) {
    const int32_t s = expert_to_slot[e];
    if (s < -1 || s >= S) return fail(h, MOE_W4A16_ERR_INVALID_ARG, "slot index out of range for expert " + std::to_string(e));
    if (s < 0) continue;
    if (used[s]) return fail(h, MOE_W4A16_ERR_INVALID_ARG, "slot " + std::to_string(s) + " named twice");
    used[s] = 1;
    if (!h->packed[s]) return fail(h, MOE_W4A16_ERR_NOT_PACKED, "slot " + std::to_string(s) + " was never packed");
  }
  DeviceGuard dg(h->cfg.device);
  if (!dg.ok) return fail(h, MOE_W4A16_ERR_CUDA, "cudaSetDevice failed");
  h->h_table.assign(expert_to_slot, expert_to_slot + E);
  cudaError_t e = cudaMemcpyAsync(h->d_table, h->h_table.data(), E * sizeof(int32_t), cudaMemcpyHostToDevice,
                                  reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(h, e, "set_slot_table");
  h->table_set = true;
  h->cur_table = h->d_table;
  return MOE_W4A16_OK;
}

static void fill_ctx(moe_w4a16_handle* h, FwdCtx& c) {
  const int E = h->cfg.num_experts;
  c.H = h->cfg.hidden;
  c.I = h->cfg.inter;
  c.E = E;
  c.k = h->cfg.top_k;
  c.pool = h->pool;
  c.slot_bytes = h->lay.bytes;
  c.lay = h->lay;
  c.table = h->cur_table;
  c.logit_part = h->logit_part;
  c.ss_part = h->ss_part;
  c.rnorm = h->rnorm;
  c.ids = h->ids;
  c.topw = h->topw;
  c.offsets = h->offsets;
  c.sorted = h->sorted;
  c.p2r = h->p2r;
  c.act_expert = h->act;
  c.act_slot = h->act + E;
  c.act_start = h->act + 2 * E;
  c.act_count = h->act + 3 * E;
  c.act_tile = h->act + 4 * E;        // E + 1 entries
  c.n_active = h->act + 5 * E + 1;
  c.xp = h->xp;
  c.hbuf = h->hbuf;
  c.ybuf = h->ybuf;
  c.xpool = h->xpool;
  c.xslots = h->xslots;
  c.xslot_halves = (uint64_t)3 * h->cfg.inter * h->cfg.hidden;
  c.route_hist = h->route_hist;
  c.route_counter = h->counters + route_counter_word(h->cfg.hidden);
  c.route_bar = reinterpret_cast<unsigned long long*>(h->counters + route_bar_word(h->cfg.hidden));
  c.grid_bar = reinterpret_cast<unsigned long long*>(h->counters);
  c.down_counters = h->counters + 2;
  c.expert_ready = h->counters + 2 + h->cfg.hidden / 32;
  c.status = h->status;
  c.num_sms = h->num_sms;
}

moe_w4a16_status moe_w4a16_forward(moe_w4a16_handle* h, const void* x, int32_t T, const void* router_w,
                                   const float* bias, uint32_t flags, void* out, int32_t* topk_ids, float* topk_w,
                                   int32_t* sorted_pairs, int32_t* expert_offsets, moe_w4a16_stream_t stream) {
  if (!h) return MOE_W4A16_ERR_INVALID_ARG;
  if (T < 0 || T > h->cfg.max_tokens)
    return fail(h, MOE_W4A16_ERR_INVALID_ARG, "T=" + std::to_string(T) + " outside [0, max_tokens]");
  if (flags & ~63u) return fail(h, MOE_W4A16_ERR_INVALID_ARG, "unknown flag bits");
  if ((flags & MOE_W4A16_FORCE_GEMV) && (flags & MOE_W4A16_FORCE_GEMM))
    return fail(h, MOE_W4A16_ERR_INVALID_ARG, "FORCE_GEMV and FORCE_GEMM are exclusive");
  const bool offload = flags & MOE_W4A16_OFFLOAD;
  if (offload && (flags & MOE_W4A16_FORCE_GEMV))
    return fail(h, MOE_W4A16_ERR_INVALID_ARG, "OFFLOAD and FORCE_GEMV are exclusive");
  if (offload && h->xslots < 1) return fail(h, MOE_W4A16_ERR_INVALID_ARG, "OFFLOAD needs moe_w4a16_offload_enable");
  if (T == 0) {
    h->last_path = MOE_W4A16_PATH_NONE;
    h->last_launches = 0;
    return MOE_W4A16_OK;
  }
  if (!x || !router_w || !out) return fail(h, MOE_W4A16_ERR_INVALID_ARG, "NULL x, router_w or out");
  if (x == out) return fail(h, MOE_W4A16_ERR_INVALID_ARG, "out must not alias x");
  if (((uintptr_t)x | (uintptr_t)router_w | (uintptr_t)out) & 15u)
    return fail(h, MOE_W4A16_ERR_INVALID_ARG, "x, router_w and out must be 16-byte aligned");
  if (bias && ((uintptr_t)bias & 3u)) return fail(h, MOE_W4A16_ERR_INVALID_ARG, "bias must be 4-byte aligned");
  if (!h->table_set) return fail(h, MOE_W4A16_ERR_INVALID_ARG, "slot table not set");
  DeviceGuard dg(h->cfg.device);
  if (!dg.ok) return fail(h, MOE_W4A16_ERR_CUDA, "cudaSetDevice failed");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  FwdCtx c;
  memset(&c, 0, sizeof c);
  fill_ctx(h, c);
  c.x = static_cast<const __half*>(x);
  c.T = T;
  c.router_w = static_cast<const __half*>(router_w);
  c.bias = bias;
  c.flags = flags;
  c.out = static_cast<__half*>(out);
  const bool gemm = offload || (flags & MOE_W4A16_FORCE_GEMM) ||
                    (!(flags & MOE_W4A16_FORCE_GEMV) && T > h->gemv_max_tokens &&
                     gemm_shapes_supported(h->cfg.hidden, h->cfg.inter));
  const bool fused_route = T <= ROUTE_FUSED_MAX_T;
  c.ksplit = 1;
  c.tile_tokens = offload ? 256 : gemm_tile_tokens(T, c.k, c.E);   // token chunk of the grouped GEMM
  int ma = c.E;
  if ((long long)T * c.k < ma) ma = T * c.k;
  if (h->cfg.num_slots < ma) ma = h->cfg.num_slots;
  c.max_active = ma;
  const bool fused = !gemm && !(flags & MOE_W4A16_UNFUSED) && fused_decode_supported(c, h->max_smem);
  const bool single_route = fused_route && route_single_launch(c);
  // above the single-launch cluster router: one cooperative kernel, which on
  // the grouped-GEMM family also copies the x rows into sorted-row order
  const bool route_gathers = gemm && !single_route;
  const int route_launches = 1;
  int32_t path = offload ? MOE_W4A16_PATH_OFFLOAD : gemm ? MOE_W4A16_PATH_GEMM : MOE_W4A16_PATH_DECODE;
  cudaError_t e = record_stage(h->events, 0, st);
  if (e == cudaSuccess && !fused) e = single_route ? launch_route(c, true, st) : launch_route_gather(c, gemm, st);
  if (e == cudaSuccess && !gemm) e = record_stage(h->events, 1, st);   // the GEMM family records it after the gather
  if (e != cudaSuccess) return cuda_fail(h, e, "route launch");
  if (fused) {
    e = launch_fused_decode(c, st, h->events);
    path = MOE_W4A16_PATH_DECODE_FUSED;
    if (e == cudaErrorNotSupported) {   // cannot be co-resident here: separate launches
      path = MOE_W4A16_PATH_DECODE;
      e = launch_route(c, fused_route, st);
      if (e == cudaSuccess) e = launch_gemv_experts(c, st, h->events);
    }
  } else {
    e = offload ? launch_offload_experts(c, h->dmaps, route_gathers, st, h->events)
        : gemm  ? launch_gemm_experts(c, h->maps, route_gathers, st, h->events)
                : launch_gemv_experts(c, st, h->events);
  }
  if (e == cudaErrorNotSupported) return fail(h, MOE_W4A16_ERR_UNSUPPORTED, "grouped GEMM path not available");
  if (e != cudaSuccess) return cuda_fail(h, e, "expert launch");
  const size_t P = (size_t)T * c.k;
  if (e == cudaSuccess && topk_ids) e = cudaMemcpyAsync(topk_ids, c.ids, P * 4, cudaMemcpyDeviceToDevice, st);
  if (e == cudaSuccess && topk_w) e = cudaMemcpyAsync(topk_w, c.topw, P * 4, cudaMemcpyDeviceToDevice, st);
  if (e == cudaSuccess && sorted_pairs) e = cudaMemcpyAsync(sorted_pairs, c.sorted, P * 4, cudaMemcpyDeviceToDevice, st);
  if (e == cudaSuccess && expert_offsets)
    e = cudaMemcpyAsync(expert_offsets, c.offsets, (c.E + 1) * 4, cudaMemcpyDeviceToDevice, st);
  if (e != cudaSuccess) return cuda_fail(h, e, "debug output copy");
  h->last_path = path;
  const int batches = offload ? (c.max_active + h->xslots - 1) / h->xslots : 0;
  h->last_launches = path == MOE_W4A16_PATH_DECODE_FUSED ? 1
                     : path == MOE_W4A16_PATH_OFFLOAD ? route_launches + !route_gathers + 1 + 3 * batches
                     : path == MOE_W4A16_PATH_GEMM    ? route_launches + !route_gathers + 3
                                                      : route_launches + 2;
  return MOE_W4A16_OK;
}

int32_t moe_w4a16_last_path(const moe_w4a16_handle* h, int32_t* launches) {
  if (!h) return -1;
  if (launches) *launches = h->last_launches;
  return h->last_path;
}

moe_w4a16_status moe_w4a16_forward_host(moe_w4a16_handle* h, const void* x_host, int32_t T, const void* router_w,
                                        const float* bias, uint32_t flags, void* out_host, moe_w4a16_stream_t stream) {
  const moe_w4a16_status s = moe_w4a16_forward_host_async(h, x_host, T, router_w, bias, flags, out_host, stream);
  if (s != MOE_W4A16_OK || T == 0) return s;
  DeviceGuard dg(h->cfg.device);
  if (!dg.ok) return fail(h, MOE_W4A16_ERR_CUDA, "cudaSetDevice failed");
  const cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(h, e, "forward_host synchronize");
  return MOE_W4A16_OK;
}

moe_w4a16_status moe_w4a16_forward_host_async(moe_w4a16_handle* h, const void* x_host, int32_t T,
                                              const void* router_w, const float* bias, uint32_t flags, void* out_host,
                                              moe_w4a16_stream_t stream) {
  if (!h) return MOE_W4A16_ERR_INVALID_ARG;
  if (T < 0 || T > h->cfg.max_tokens) return fail(h, MOE_W4A16_ERR_INVALID_ARG, "T outside [0, max_tokens]");
  if (T == 0) return MOE_W4A16_OK;
  if (!x_host || !out_host) return fail(h, MOE_W4A16_ERR_INVALID_ARG, "NULL host buffer");
  DeviceGuard dg(h->cfg.device);
  if (!dg.ok) return fail(h, MOE_W4A16_ERR_CUDA, "cudaSetDevice failed");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const size_t bytes = (size_t)T * h->cfg.hidden * sizeof(__half);
  cudaError_t e = cudaMemcpyAsync(h->x_dev, x_host, bytes, cudaMemcpyHostToDevice, st);
  if (e != cudaSuccess) return cuda_fail(h, e, "forward_host H2D");
  moe_w4a16_status s = moe_w4a16_forward(h, h->x_dev, T, router_w, bias, flags, h->out_dev, nullptr, nullptr,
                                         nullptr, nullptr, stream);
  if (s != MOE_W4A16_OK) return s;
  e = cudaMemcpyAsync(out_host, h->out_dev, bytes, cudaMemcpyDeviceToHost, st);
  if (e != cudaSuccess) return cuda_fail(h, e, "forward_host D2H");
  return MOE_W4A16_OK;
}

moe_w4a16_status moe_w4a16_get_status(moe_w4a16_handle* h, int64_t* miss_count) {
  if (!h) return MOE_W4A16_ERR_INVALID_ARG;
  DeviceGuard dg(h->cfg.device);
  if (!dg.ok) return fail(h, MOE_W4A16_ERR_CUDA, "cudaSetDevice failed");
  DevStatus s;
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cudaMemcpy(&s, h->status, sizeof s, cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemset(h->status, 0, sizeof s);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(h, e, "get_status");
  if (miss_count) *miss_count = (int64_t)s.miss;
  if (s.flags & STATUS_TIMEOUT) {   // barriers and counters may be mid-use: start them afresh
    cudaMemset(h->counters, 0, counter_words(h->cfg.hidden) * sizeof(unsigned));
    cudaDeviceSynchronize();
    return fail(h, MOE_W4A16_ERR_TIMEOUT, "a bounded device wait gave up");
  }
  if (s.flags & STATUS_MISS) return fail(h, MOE_W4A16_ERR_NOT_RESIDENT, "a routed expert had no slot");
  return MOE_W4A16_OK;
}

const char* moe_w4a16_last_error(const moe_w4a16_handle* h) {
  return h ? h->err.c_str() : g_create_err.c_str();
}

}  // extern "C"

moe_w4a16_status moe_w4a16_selftest_timeout(moe_w4a16_handle* h, int32_t which, int64_t limit_cycles,
                                            moe_w4a16_stream_t stream) {
  if (!h) return MOE_W4A16_ERR_INVALID_ARG;
  if (which < 0 || which > 1) return fail(h, MOE_W4A16_ERR_INVALID_ARG, "which must be 0 or 1");
  if (limit_cycles < 1000 || limit_cycles > (1ll << 31))
    return fail(h, MOE_W4A16_ERR_INVALID_ARG, "limit_cycles outside [1000, 2^31]");
  DeviceGuard dg(h->cfg.device);
  if (!dg.ok) return fail(h, MOE_W4A16_ERR_CUDA, "cudaSetDevice failed");
  const cudaError_t e = launch_selftest_wait(h->status, h->counters + never_set_word(h->cfg.hidden), which,
                                             (long long)limit_cycles, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(h, e, "selftest launch");
  return MOE_W4A16_OK;
}
