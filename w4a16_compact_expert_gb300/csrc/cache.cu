// Expert cache: the partial-residency miss path of the C ABI
// (moe_w4a16_cache_*), after the resident-qpacked-cache-v1 lifecycle
// ("Horizon RunMap - architecture", sections "Immutable authority and miss
// lifecycle" and "Immutable cache — the scope of ADR 0009"):
//   immutable host backing -> bounded pinned staging -> unpublished spare
//   row (repacked on the device) -> one atomic publication of a complete
//   generation of the expert->slot table; leases keep evicted rows and old
//   tables from reuse until their consumers retire; eviction discards the
//   device copy (LRU, canonical initial placement); misses are serialised;
//   capacity is admitted at create; a failure before publication keeps the
//   previous generation, a failure during publication faults the cache.
// The state machine is the same for the CUDA transport and for the host-only
// simulation, which moves no bytes and whose lease events complete only when
// a test says so.
#include <algorithm>
#include <atomic>
#include <condition_variable>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <thread>
#include <vector>

#include "handle.h"
#include "internal.h"
#include "moe_w4a16.h"

namespace {

constexpr int kTableRing = 8;   // device tables of the last generations

struct Lease {
  uint64_t gen = 0;
  bool released = false;
  bool retired = false;
  cudaEvent_t ev = nullptr;   // release event (CUDA transport)
};

struct Retiring {
  int row;
  uint64_t gen_unmapped;   // the generation that stopped publishing the row
};

size_t align256(size_t v) { return (v + 255) / 256 * 256; }

// Host threads that copy a miss's canonical arrays from the backing into its
// pinned staging entry together: one host thread's copy rate (about 14 GB/s
// on the GB300's Grace host) would bound the whole miss path, well below
// what the host-to-device link carries.  The calling thread takes part; the
// bytes are cut into chunks that the threads claim from one counter.
class CopyPool {
 public:
  struct Seg {
    uint8_t* dst;
    const uint8_t* src;
    size_t bytes;
  };

  explicit CopyPool(int workers) {
    for (int i = 0; i < workers; ++i) th_.emplace_back([this] { loop(); });
  }
  ~CopyPool() {
    {
      std::lock_guard<std::mutex> lk(mu_);
      stop_ = true;
    }
    cv_.notify_all();
    for (auto& t : th_) t.join();
  }

  // Copies every segment; returns when all bytes are in place.
  void copy(const std::vector<Seg>& segs) {
    size_t total = 0;
    for (const Seg& sg : segs) total += sg.bytes;
    if (th_.empty() || total < 2 * kChunk) {
      for (const Seg& sg : segs) std::memcpy(sg.dst, sg.src, sg.bytes);
      return;
    }
    {
      std::lock_guard<std::mutex> lk(mu_);
      segs_ = &segs;
      nchunks_ = 0;
      for (const Seg& sg : segs) nchunks_ += (sg.bytes + kChunk - 1) / kChunk;
      next_.store(0);
      done_ = 0;
      ++job_;
    }
    cv_.notify_all();
    const size_t mine = work();
    std::unique_lock<std::mutex> lk(mu_);
    done_ += mine;
    done_cv_.wait(lk, [this] { return done_ == nchunks_; });
    segs_ = nullptr;
  }

 private:
  static constexpr size_t kChunk = 256 * 1024;

  // Claims chunks until none is left; returns how many this thread copied.
  size_t work() {
    size_t n = 0;
    for (;;) {
      size_t i = next_.fetch_add(1);
      if (i >= nchunks_) return n;
      for (const Seg& sg : *segs_) {   // chunk i -> (segment, offset)
        const size_t cs = (sg.bytes + kChunk - 1) / kChunk;
        if (i < cs) {
          const size_t off = i * kChunk, len = std::min(kChunk, sg.bytes - off);
          std::memcpy(sg.dst + off, sg.src + off, len);
          break;
        }
        i -= cs;
      }
      ++n;
    }
  }

  void loop() {
    uint64_t seen = 0;
    for (;;) {
      {
        std::unique_lock<std::mutex> lk(mu_);
        cv_.wait(lk, [&] { return stop_ || job_ != seen; });
        if (stop_) return;
        seen = job_;
      }
      const size_t mine = work();
      std::lock_guard<std::mutex> lk(mu_);
      done_ += mine;
      if (done_ == nchunks_) done_cv_.notify_all();
    }
  }

  std::vector<std::thread> th_;
  std::mutex mu_;
  std::condition_variable cv_, done_cv_;
  const std::vector<Seg>* segs_ = nullptr;
  size_t nchunks_ = 0, done_ = 0;
  std::atomic<size_t> next_{0};
  uint64_t job_ = 0;
  bool stop_ = false;
};

// Copy threads of a cache: half the host's cores, at most 8, counting the caller.
int copy_workers() {
  const unsigned hc = std::thread::hardware_concurrency();
  const int n = hc >= 2 ? (int)std::min(8u, hc / 2) : 1;
  return n - 1;
}

}  // namespace

struct moe_w4a16_cache {
  bool sim = false;
  moe_w4a16_handle* h = nullptr;
  int E = 0, S = 0;
  moe_w4a16_cache_config cfg{};
  uint64_t expert_bytes = 0;   // canonical qpacked bytes of one expert
  // immutable host backing (canonical arrays, leading axis = expert)
  const uint8_t* bq[3] = {nullptr, nullptr, nullptr};
  const uint16_t* bs[3] = {nullptr, nullptr, nullptr};
  size_t qbytes[3] = {0, 0, 0}, sbytes[3] = {0, 0, 0};
  size_t stage_entry = 0;      // bytes of one staging entry (six 256-aligned parts)
  // published state
  std::vector<int32_t> table;        // expert -> slot
  std::vector<int32_t> row_expert;   // slot -> published expert, -1 if none
  std::vector<uint64_t> last_use;
  uint64_t tick = 0, gen = 0;
  std::vector<int> free_rows;        // unpublished rows reusable now, ascending
  std::vector<Retiring> retiring;
  std::map<uint64_t, Lease> leases;
  uint64_t next_lease = 1;
  bool faulted = false;
  int sim_fail = 0;
  moe_w4a16_cache_stats st{};
  std::string err;
  // CUDA transport
  uint8_t* pinned = nullptr;          // staging_experts entries
  uint8_t* dstage = nullptr;          // device landing area of the staging entries
  std::vector<cudaEvent_t> stage_ev;  // transfer completion of each entry
  std::vector<bool> stage_live;
  int next_stage = 0;
  CopyPool* pool = nullptr;           // host threads of the backing -> staging copies
  int32_t* tables_dev = nullptr;      // kTableRing x E
  int32_t* tables_host = nullptr;     // pinned kTableRing x E
  cudaEvent_t table_ev[kTableRing] = {};
  uint64_t table_gen[kTableRing] = {};
};

namespace {

moe_w4a16_status cfail(moe_w4a16_cache* c, moe_w4a16_status s, const std::string& msg) {
  if (c) c->err = msg;
  return s;
}

moe_w4a16_status cuda_cfail(moe_w4a16_cache* c, cudaError_t e, const char* what) {
  return cfail(c, MOE_W4A16_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

// Marks released leases whose events completed as retired.
void refresh_leases(moe_w4a16_cache* c) {
  for (auto& kv : c->leases) {
    Lease& l = kv.second;
    if (!l.released || l.retired || c->sim) continue;
    if (cudaEventQuery(l.ev) == cudaSuccess) l.retired = true;
  }
  for (auto it = c->leases.begin(); it != c->leases.end();) {
    if (it->second.retired) {
      if (it->second.ev) cudaEventDestroy(it->second.ev);
      it = c->leases.erase(it);
    } else {
      ++it;
    }
  }
}

// Smallest generation any unretired lease holds (UINT64_MAX if none).
uint64_t oldest_lease_gen(const moe_w4a16_cache* c) {
  uint64_t m = UINT64_MAX;
  for (const auto& kv : c->leases) m = std::min(m, kv.second.gen);
  return m;
}

// Rows unmapped by generation g are reusable once no lease on a generation
// before g is left.
void reclaim_rows(moe_w4a16_cache* c) {
  const uint64_t oldest = oldest_lease_gen(c);
  for (auto it = c->retiring.begin(); it != c->retiring.end();) {
    if (oldest >= it->gen_unmapped) {
      c->free_rows.insert(std::lower_bound(c->free_rows.begin(), c->free_rows.end(), it->row), it->row);
      it = c->retiring.erase(it);
    } else {
      ++it;
    }
  }
}

// Waits for the oldest unretired lease: its release event on the CUDA
// transport; in the simulation (or if it was never released) this cannot
// make progress and fails.
moe_w4a16_status wait_oldest_lease(moe_w4a16_cache* c) {
  uint64_t id = 0, g = UINT64_MAX;
  for (const auto& kv : c->leases)
    if (kv.second.gen < g) {
      g = kv.second.gen;
      id = kv.first;
    }
  if (id == 0) return cfail(c, MOE_W4A16_ERR_TIMEOUT, "no lease to wait for");
  Lease& l = c->leases[id];
  if (!l.released)
    return cfail(c, MOE_W4A16_ERR_TIMEOUT,
                 "lease " + std::to_string(id) + " on generation " + std::to_string(g) +
                     " is still held: its rows cannot be reused yet");
  if (c->sim)
    return cfail(c, MOE_W4A16_ERR_TIMEOUT,
                 "lease " + std::to_string(id) + " has not retired (simulated event pending)");
  ++c->st.lease_waits;
  const cudaError_t e = cudaEventSynchronize(l.ev);
  if (e != cudaSuccess) return cuda_cfail(c, e, "waiting for a lease's release event");
  l.retired = true;
  refresh_leases(c);
  return MOE_W4A16_OK;
}

// Copies the canonical bytes of `expert` from the backing through a pinned
// staging entry to the device and repacks them into slot row `row`.
moe_w4a16_status transport_one(moe_w4a16_cache* c, int expert, int row, cudaStream_t st) {
  if (c->sim) {
    if (c->sim_fail == 1) {
      c->sim_fail = 0;
      return cfail(c, MOE_W4A16_ERR_CUDA, "simulated transport failure");
    }
    return MOE_W4A16_OK;
  }
  const int j = c->next_stage;
  c->next_stage = (c->next_stage + 1) % c->cfg.staging_experts;
  cudaError_t e = cudaSuccess;
  if (c->stage_live[j]) e = cudaEventSynchronize(c->stage_ev[j]);   // reuse only after its transfer retired
  if (e != cudaSuccess) return cuda_cfail(c, e, "staging entry event");
  uint8_t* hp = c->pinned + (size_t)j * c->stage_entry;
  uint8_t* dp = c->dstage + (size_t)j * c->stage_entry;
  size_t off = 0;
  size_t qoff[3], soff[3];
  std::vector<CopyPool::Seg> segs;
  for (int m = 0; m < 3; ++m) {
    qoff[m] = off;
    segs.push_back({hp + off, c->bq[m] + (size_t)expert * c->qbytes[m], c->qbytes[m]});
    off += align256(c->qbytes[m]);
    soff[m] = off;
    segs.push_back({hp + off, reinterpret_cast<const uint8_t*>(c->bs[m]) + (size_t)expert * c->sbytes[m],
                    c->sbytes[m]});
    off += align256(c->sbytes[m]);
  }
  c->pool->copy(segs);
  e = cudaMemcpyAsync(dp, hp, off, cudaMemcpyHostToDevice, st);
  const MatLayout* mats[3] = {&c->h->lay.gate, &c->h->lay.up, &c->h->lay.down};
  uint8_t* slot_base = c->h->pool + (size_t)row * c->h->lay.bytes;
  for (int m = 0; m < 3 && e == cudaSuccess; ++m)
    e = launch_repack_matrix(dp + qoff[m], reinterpret_cast<const uint16_t*>(dp + soff[m]), slot_base, *mats[m], st);
  if (e == cudaSuccess) e = cudaEventRecord(c->stage_ev[j], st);
  if (e != cudaSuccess) return cuda_cfail(c, e, "miss transport");
  c->stage_live[j] = true;
  c->h->packed[row] = 1;
  return MOE_W4A16_OK;
}

// Publishes `tab` as generation c->gen + 1 (ordered on st after the
// transfers); forwards enqueued from now on read it.
moe_w4a16_status publish(moe_w4a16_cache* c, const std::vector<int32_t>& tab, cudaStream_t st) {
  const uint64_t g = c->gen + 1;
  if (c->sim) {
    if (c->sim_fail == 2) {
      c->sim_fail = 0;
      c->faulted = true;
      return cfail(c, MOE_W4A16_ERR_CUDA, "simulated publication failure: cache faulted");
    }
    return MOE_W4A16_OK;
  }
  const int k = (int)(g % kTableRing);
  // the ring entry's previous generation must have no readers left
  while (c->table_gen[k] != 0 && oldest_lease_gen(c) <= c->table_gen[k]) {
    const moe_w4a16_status s = wait_oldest_lease(c);
    if (s != MOE_W4A16_OK) return s;   // before publication: previous generation stays
  }
  cudaError_t e = cudaSuccess;
  if (c->table_gen[k] != 0) e = cudaEventSynchronize(c->table_ev[k]);   // its host copy may be rewritten
  if (e != cudaSuccess) return cuda_cfail(c, e, "table ring event");
  int32_t* hostt = c->tables_host + (size_t)k * c->E;
  int32_t* devt = c->tables_dev + (size_t)k * c->E;
  std::memcpy(hostt, tab.data(), c->E * sizeof(int32_t));
  e = cudaMemcpyAsync(devt, hostt, c->E * sizeof(int32_t), cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess) e = cudaEventRecord(c->table_ev[k], st);
  if (e != cudaSuccess) {
    c->faulted = true;
    return cuda_cfail(c, e, "publication failed: cache faulted");
  }
  c->table_gen[k] = g;
  c->h->cur_table = devt;   // the atomic switch for every later forward
  c->h->table_set = true;
  return MOE_W4A16_OK;
}

moe_w4a16_status validate_config(int E, int S, const moe_w4a16_cache_config* cfg, const int32_t* initial,
                                 int32_t n_initial, std::string& why) {
  if (!cfg) {
    why = "NULL config";
    return MOE_W4A16_ERR_INVALID_ARG;
  }
  if (cfg->max_group < 1 || cfg->max_group > E) {
    why = "max_group must be in [1, num_experts]";
    return MOE_W4A16_ERR_INVALID_ARG;
  }
  if (cfg->spare_slots < cfg->max_group) {
    why = "spare_slots must be >= max_group (a group's misses need unpublished rows)";
    return MOE_W4A16_ERR_INVALID_ARG;
  }
  if (cfg->staging_experts < 1) {
    why = "staging_experts must be >= 1";
    return MOE_W4A16_ERR_INVALID_ARG;
  }
  if (n_initial < 0 || n_initial > E || (int64_t)n_initial + cfg->spare_slots > S) {
    why = "initial experts + spare_slots exceed the slot pool";
    return MOE_W4A16_ERR_INVALID_ARG;
  }
  if (S - cfg->spare_slots < cfg->max_group) {
    why = "the published rows (num_slots - spare_slots) cannot hold a whole group";
    return MOE_W4A16_ERR_INVALID_ARG;
  }
  if (n_initial > 0 && !initial) {
    why = "NULL initial list";
    return MOE_W4A16_ERR_INVALID_ARG;
  }
  std::vector<uint8_t> seen(E, 0);
  for (int i = 0; i < n_initial; ++i) {
    const int e = initial[i];
    if (e < 0 || e >= E || seen[e]) {
      why = "initial expert ids must be distinct and in range";
      return MOE_W4A16_ERR_INVALID_ARG;
    }
    seen[e] = 1;
  }
  return MOE_W4A16_OK;
}

void init_state(moe_w4a16_cache* c, const int32_t* initial, int32_t n_initial) {
  c->table.assign(c->E, -1);
  c->row_expert.assign(c->S, -1);
  c->last_use.assign(c->E, 0);
  for (int i = 0; i < n_initial; ++i) {
    c->table[initial[i]] = i;
    c->row_expert[i] = initial[i];
  }
  for (int r = n_initial; r < c->S; ++r) c->free_rows.push_back(r);
  c->gen = 1;
}

void free_transport(moe_w4a16_cache* c) {
  delete c->pool;
  c->pool = nullptr;
  for (auto& kv : c->leases)
    if (kv.second.ev) cudaEventDestroy(kv.second.ev);
  c->leases.clear();
  for (cudaEvent_t ev : c->stage_ev)
    if (ev) cudaEventDestroy(ev);
  c->stage_ev.clear();
  for (int k = 0; k < kTableRing; ++k)
    if (c->table_ev[k]) cudaEventDestroy(c->table_ev[k]);
  if (c->pinned) cudaFreeHost(c->pinned);
  if (c->tables_host) cudaFreeHost(c->tables_host);
  if (c->dstage) cudaFree(c->dstage);
  if (c->tables_dev) cudaFree(c->tables_dev);
  c->pinned = c->dstage = nullptr;
  c->tables_host = c->tables_dev = nullptr;
}

}  // namespace

// --------------------------------------------------------------------- ABI

moe_w4a16_status moe_w4a16_cache_create(moe_w4a16_handle* h, const moe_w4a16_cache_config* cfg,
                                        const uint8_t* gate_q, const uint16_t* gate_s, const uint8_t* up_q,
                                        const uint16_t* up_s, const uint8_t* down_q, const uint16_t* down_s,
                                        const int32_t* initial, int32_t n_initial, moe_w4a16_cache** out) {
  if (!h || !out) return MOE_W4A16_ERR_INVALID_ARG;
  *out = nullptr;
  if (h->cache) return MOE_W4A16_ERR_INVALID_ARG;
  if (!gate_q || !gate_s || !up_q || !up_s || !down_q || !down_s) {
    set_handle_free_error("NULL expert backing array");
    return MOE_W4A16_ERR_INVALID_ARG;
  }
  std::string why;
  const int E = h->cfg.num_experts, S = h->cfg.num_slots;
  moe_w4a16_status s = validate_config(E, S, cfg, initial, n_initial, why);
  if (s != MOE_W4A16_OK) {
    set_handle_free_error(why.c_str());
    return s;
  }
  moe_w4a16_cache* c = new moe_w4a16_cache();
  c->h = h;
  c->E = E;
  c->S = S;
  c->cfg = *cfg;
  const MatLayout* mats[3] = {&h->lay.gate, &h->lay.up, &h->lay.down};
  c->bq[0] = gate_q, c->bq[1] = up_q, c->bq[2] = down_q;
  c->bs[0] = gate_s, c->bs[1] = up_s, c->bs[2] = down_s;
  for (int m = 0; m < 3; ++m) {
    c->qbytes[m] = (size_t)mats[m]->rows * mats[m]->k / 2;
    c->sbytes[m] = (size_t)mats[m]->rows * mats[m]->nb * 2;
    c->expert_bytes += c->qbytes[m] + c->sbytes[m];
    c->stage_entry += align256(c->qbytes[m]) + align256(c->sbytes[m]);
  }
  int prev = -1;
  cudaGetDevice(&prev);
  cudaError_t e = cudaSetDevice(h->cfg.device);
  const int ns = cfg->staging_experts;
  if (e == cudaSuccess) e = cudaMallocHost(&c->pinned, (size_t)ns * c->stage_entry);
  if (e == cudaSuccess) e = cudaMalloc(&c->dstage, (size_t)ns * c->stage_entry);
  if (e == cudaSuccess) e = cudaMallocHost(&c->tables_host, (size_t)kTableRing * E * sizeof(int32_t));
  if (e == cudaSuccess) e = cudaMalloc(&c->tables_dev, (size_t)kTableRing * E * sizeof(int32_t));
  c->stage_ev.assign(ns, nullptr);
  c->stage_live.assign(ns, false);
  c->pool = new CopyPool(copy_workers());
  for (int j = 0; j < ns && e == cudaSuccess; ++j) e = cudaEventCreateWithFlags(&c->stage_ev[j], cudaEventDisableTiming);
  for (int k = 0; k < kTableRing && e == cudaSuccess; ++k)
    e = cudaEventCreateWithFlags(&c->table_ev[k], cudaEventDisableTiming);
  cudaStream_t st = nullptr;
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking);
  if (e != cudaSuccess) {
    set_handle_free_error((std::string("cache create: ") + cudaGetErrorString(e)).c_str());
    if (st) cudaStreamDestroy(st);
    free_transport(c);
    delete c;
    if (prev >= 0) cudaSetDevice(prev);
    return e == cudaErrorMemoryAllocation ? MOE_W4A16_ERR_OOM : MOE_W4A16_ERR_CUDA;
  }
  // canonical initial placement: initial[i] in slot i, published as generation 1
  init_state(c, initial, n_initial);
  s = MOE_W4A16_OK;
  for (int i = 0; i < n_initial && s == MOE_W4A16_OK; ++i) s = transport_one(c, initial[i], i, st);
  if (s == MOE_W4A16_OK) {
    c->gen = 0;
    s = publish(c, c->table, st);
    c->gen = 1;
  }
  if (s == MOE_W4A16_OK) {
    e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) s = cuda_cfail(c, e, "cache create");
  }
  cudaStreamDestroy(st);
  if (s != MOE_W4A16_OK) {
    set_handle_free_error(c->err.c_str());
    h->cur_table = h->d_table;
    free_transport(c);
    delete c;
    if (prev >= 0) cudaSetDevice(prev);
    return s;
  }
  h->cache = c;
  c->st.h2d_bytes = (uint64_t)n_initial * c->expert_bytes;
  if (prev >= 0) cudaSetDevice(prev);
  *out = c;
  return MOE_W4A16_OK;
}

moe_w4a16_status moe_w4a16_cache_create_sim(int32_t num_experts, int32_t num_slots, uint64_t expert_bytes,
                                            const moe_w4a16_cache_config* cfg, const int32_t* initial,
                                            int32_t n_initial, moe_w4a16_cache** out) {
  if (!out) return MOE_W4A16_ERR_INVALID_ARG;
  *out = nullptr;
  if (num_experts < 1 || num_experts > 4096 || num_slots < 1) {
    set_handle_free_error("num_experts must be in [1, 4096] and num_slots >= 1");
    return MOE_W4A16_ERR_INVALID_ARG;
  }
  std::string why;
  const moe_w4a16_status s = validate_config(num_experts, num_slots, cfg, initial, n_initial, why);
  if (s != MOE_W4A16_OK) {
    set_handle_free_error(why.c_str());
    return s;
  }
  moe_w4a16_cache* c = new moe_w4a16_cache();
  c->sim = true;
  c->E = num_experts;
  c->S = num_slots;
  c->cfg = *cfg;
  c->expert_bytes = expert_bytes;
  init_state(c, initial, n_initial);
  c->st.h2d_bytes = (uint64_t)n_initial * expert_bytes;
  *out = c;
  return MOE_W4A16_OK;
}

moe_w4a16_status moe_w4a16_cache_destroy(moe_w4a16_cache* c) {
  if (!c) return MOE_W4A16_OK;
  if (!c->sim) {
    int prev = -1;
    cudaGetDevice(&prev);
    cudaSetDevice(c->h->cfg.device);
    for (auto& kv : c->leases)
      if (kv.second.released && kv.second.ev) cudaEventSynchronize(kv.second.ev);
    for (size_t j = 0; j < c->stage_ev.size(); ++j)
      if (c->stage_live[j]) cudaEventSynchronize(c->stage_ev[j]);
    for (int k = 0; k < kTableRing; ++k)
      if (c->table_gen[k]) cudaEventSynchronize(c->table_ev[k]);
    // the handle keeps serving the last generation from its own table
    moe_w4a16_handle* h = c->h;
    h->h_table = c->table;
    cudaError_t e = cudaMemcpy(h->d_table, c->table.data(), c->E * sizeof(int32_t), cudaMemcpyHostToDevice);
    h->cur_table = h->d_table;
    h->table_set = e == cudaSuccess && !c->faulted;
    h->cache = nullptr;
    free_transport(c);
    if (prev >= 0) cudaSetDevice(prev);
  }
  delete c;
  return MOE_W4A16_OK;
}

moe_w4a16_status moe_w4a16_cache_acquire(moe_w4a16_cache* c, const int32_t* ids, int32_t n,
                                         moe_w4a16_stream_t stream, uint64_t* lease) {
  if (!c || !lease) return MOE_W4A16_ERR_INVALID_ARG;
  *lease = 0;
  if (c->faulted) return cfail(c, MOE_W4A16_ERR_CUDA, "the cache is faulted (a publication failed)");
  if (n < 0 || n > c->cfg.max_group) return cfail(c, MOE_W4A16_ERR_INVALID_ARG, "group size outside [0, max_group]");
  if (n > 0 && !ids) return cfail(c, MOE_W4A16_ERR_INVALID_ARG, "NULL ids");
  std::vector<uint8_t> in_group(c->E, 0);
  for (int i = 0; i < n; ++i) {
    if (ids[i] < 0 || ids[i] >= c->E || in_group[ids[i]])
      return cfail(c, MOE_W4A16_ERR_INVALID_ARG, "group ids must be distinct and in [0, num_experts)");
    in_group[ids[i]] = 1;
  }
  int prev = -1;
  if (!c->sim) {
    cudaGetDevice(&prev);
    cudaSetDevice(c->h->cfg.device);
  }
  struct Restore {
    int dev;
    ~Restore() {
      if (dev >= 0) cudaSetDevice(dev);
    }
  } restore{prev};
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  refresh_leases(c);
  reclaim_rows(c);
  ++c->tick;
  std::vector<int> misses;
  for (int e = 0; e < c->E; ++e)
    if (in_group[e] && c->table[e] < 0) misses.push_back(e);   // ascending expert order
  if (!misses.empty()) {
    // rows for the misses: spare rows reusable now, waiting for older leases if needed
    while ((int)c->free_rows.size() < (int)misses.size()) {
      const moe_w4a16_status s = wait_oldest_lease(c);
      if (s != MOE_W4A16_OK) return s;
      reclaim_rows(c);
    }
    std::vector<int> rows(c->free_rows.begin(), c->free_rows.begin() + misses.size());
    // victims: least recently used published experts outside the group, until
    // the published set fits num_slots - spare_slots again
    int resident = 0;
    for (int e = 0; e < c->E; ++e) resident += c->table[e] >= 0;
    const int excess = resident + (int)misses.size() - (c->S - c->cfg.spare_slots);
    std::vector<int> cand;
    for (int e = 0; e < c->E; ++e)
      if (c->table[e] >= 0 && !in_group[e]) cand.push_back(e);
    std::sort(cand.begin(), cand.end(), [&](int a, int b) {
      return c->last_use[a] != c->last_use[b] ? c->last_use[a] < c->last_use[b] : a < b;
    });
    std::vector<int> victims(cand.begin(), cand.begin() + std::max(0, std::min(excess, (int)cand.size())));
    // transport into the unpublished rows; a failure here keeps the published generation
    for (size_t i = 0; i < misses.size(); ++i) {
      const moe_w4a16_status s = transport_one(c, misses[i], rows[i], st);
      if (s != MOE_W4A16_OK) return s;   // rows stay in free_rows (never published)
    }
    std::vector<int32_t> tab = c->table;
    for (int v : victims) tab[v] = -1;
    for (size_t i = 0; i < misses.size(); ++i) tab[misses[i]] = rows[i];
    const moe_w4a16_status s = publish(c, tab, st);
    if (s != MOE_W4A16_OK) return s;   // faulted if the publication itself failed
    // the new generation is the published state
    ++c->gen;
    c->free_rows.erase(c->free_rows.begin(), c->free_rows.begin() + misses.size());
    for (int v : victims) {
      c->retiring.push_back({c->table[v], c->gen});
      c->row_expert[c->table[v]] = -1;
    }
    c->table = tab;
    for (size_t i = 0; i < misses.size(); ++i) c->row_expert[rows[i]] = misses[i];
    ++c->st.transactions;
    c->st.misses += misses.size();
    c->st.evictions += victims.size();
    c->st.h2d_bytes += (uint64_t)misses.size() * c->expert_bytes;
  }
  c->st.hits += (uint64_t)(n - (int)misses.size());
  for (int i = 0; i < n; ++i) c->last_use[ids[i]] = c->tick;
  const uint64_t id = c->next_lease++;
  c->leases[id].gen = c->gen;
  *lease = id;
  return MOE_W4A16_OK;
}

moe_w4a16_status moe_w4a16_cache_release(moe_w4a16_cache* c, uint64_t lease, moe_w4a16_stream_t stream) {
  if (!c) return MOE_W4A16_ERR_INVALID_ARG;
  auto it = c->leases.find(lease);
  if (it == c->leases.end() || it->second.released)
    return cfail(c, MOE_W4A16_ERR_INVALID_ARG, "unknown or already released lease");
  if (!c->sim) {
    int prev = -1;
    cudaGetDevice(&prev);
    cudaSetDevice(c->h->cfg.device);
    cudaError_t e = cudaEventCreateWithFlags(&it->second.ev, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventRecord(it->second.ev, reinterpret_cast<cudaStream_t>(stream));
    if (prev >= 0) cudaSetDevice(prev);
    if (e != cudaSuccess) return cuda_cfail(c, e, "lease release event");
  }
  it->second.released = true;
  return MOE_W4A16_OK;
}

moe_w4a16_status moe_w4a16_cache_get_stats(moe_w4a16_cache* c, moe_w4a16_cache_stats* out) {
  if (!c || !out) return MOE_W4A16_ERR_INVALID_ARG;
  refresh_leases(c);
  reclaim_rows(c);
  moe_w4a16_cache_stats s = c->st;
  s.generation = c->gen;
  s.d2h_bytes = 0;
  s.resident = 0;
  for (int e = 0; e < c->E; ++e) s.resident += c->table[e] >= 0;
  s.free_spares = (int32_t)c->free_rows.size();
  s.retiring = (int32_t)c->retiring.size();
  s.active_leases = (int32_t)c->leases.size();
  s.faulted = c->faulted ? 1 : 0;
  *out = s;
  return MOE_W4A16_OK;
}

int32_t moe_w4a16_cache_slot_of(const moe_w4a16_cache* c, int32_t expert) {
  if (!c || expert < 0 || expert >= c->E) return -1;
  return c->table[expert];
}

const char* moe_w4a16_cache_last_error(const moe_w4a16_cache* c) { return c ? c->err.c_str() : ""; }

moe_w4a16_status moe_w4a16_cache_sim_complete(moe_w4a16_cache* c, uint64_t lease) {
  if (!c || !c->sim) return MOE_W4A16_ERR_INVALID_ARG;
  auto it = c->leases.find(lease);
  if (it == c->leases.end() || !it->second.released)
    return cfail(c, MOE_W4A16_ERR_INVALID_ARG, "lease is unknown or not released");
  it->second.retired = true;
  return MOE_W4A16_OK;
}

moe_w4a16_status moe_w4a16_cache_sim_fail(moe_w4a16_cache* c, int32_t where) {
  if (!c || !c->sim || where < 0 || where > 2) return MOE_W4A16_ERR_INVALID_ARG;
  c->sim_fail = where;
  return MOE_W4A16_OK;
}
