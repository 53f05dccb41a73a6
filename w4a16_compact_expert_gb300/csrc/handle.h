// Definition of the library handle, shared by the host runtime (api.cu) and
// the expert cache (cache.cu).  Not part of the ABI.
#pragma once
#include <string>
#include <vector>

#include "moe_w4a16.h"
#include "internal.h"

struct moe_w4a16_handle {
  moe_w4a16_config cfg{};
  SlotLayout lay{};
  int num_sms = 0;
  int ksplit_fused = 1;
  int max_smem = 0;                  // opt-in shared memory per block
  int32_t gemv_max_tokens = 0;
  int32_t last_path = 0;             // MOE_W4A16_PATH_* of the last forward
  int32_t last_launches = 0;
  uint8_t* pool = nullptr;
  std::vector<uint8_t> packed;      // per slot: 1 once packed
  std::vector<int32_t> h_table;
  bool table_set = false;
  int32_t* d_table = nullptr;        // the table set_slot_table writes
  int32_t* cur_table = nullptr;      // the table forwards read: d_table, or the cache's published generation
  moe_w4a16_cache* cache = nullptr;  // attached expert cache (owns the table while attached)
  // workspaces
  float* logit_part = nullptr;
  float* ss_part = nullptr;
  float* rnorm = nullptr;
  int32_t* ids = nullptr;
  float* topw = nullptr;
  int32_t* offsets = nullptr;
  int32_t* sorted = nullptr;
  int32_t* p2r = nullptr;
  int32_t* act = nullptr;            // 5 arrays of E (+1) ints, see fill_ctx
  int32_t* route_hist = nullptr;     // [ceil(max_tokens/8)][E]
  __half* xp = nullptr;
  __half* hbuf = nullptr;
  float* ybuf = nullptr;
  __half* xpool = nullptr;           // offload-qpacked comparison: FP16 execution slots
  int xslots = 0;
  DenseMaps dmaps{};
  unsigned* counters = nullptr;      // counter_words(H): grid barrier, arrival and readiness counters
  DevStatus* status = nullptr;
  uint8_t* stage = nullptr;          // pack staging for host sources
  size_t stage_bytes = 0;
  __half* x_dev = nullptr;           // forward_host staging
  __half* out_dev = nullptr;
  StageEvents events{};
  PoolMaps maps{};
  std::vector<void*> allocs;
  std::string err;
};

