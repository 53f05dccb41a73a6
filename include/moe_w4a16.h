/*
 * moe_w4a16.h -- C ABI of the GB300 (sm_103a) W4A16 routed-expert MoE layer.
 *
 * One handle = one MoE FFN layer: a router [E, H] applied to FP16 activations,
 * top-k expert selection, and E experts whose gate/up [I, H] and down [H, I]
 * weights stay compact (signed int4, one FP16 scale per 256 consecutive K
 * values) in a fixed pool of GPU "slots".  No expanded FP16 copy of an expert
 * is ever kept: kernels dequantise the values they need while computing.
 *
 * Sources (Horizon RunMap pages):
 *  - "Horizon RunMap - architecture", section "Representation and
 *    computation": routed experts INT4 qpacked with 256-value blocks and FP16
 *    scales; compact weights on the GPU; FP16 activations; no persistent
 *    expanded expert (temporary kernel values and workspaces are separate).
 *  - same page, section "Immutable authority and miss lifecycle": capacity is
 *    fixed before admission (here: everything is sized at create).
 *  - same page, section "Regimes and executor boundaries": a resident expert
 *    need not be routed (slots and the expert->slot table are separate).
 *  - landing page (/en), section "08 / Precision & quality": values converted
 *    in-kernel, FP32 accumulation stages and explicit rounding; routing
 *    stays outside INT4.
 *
 * Canonical "qpacked" layout accepted by moe_w4a16_pack_experts, per expert,
 * experts concatenated along the leading axis:
 *   gate_q, up_q : uint8  [I][H/2]          gate_s, up_s : fp16 bits [I][ceil(H/256)]
 *   down_q       : uint8  [H][I/2]          down_s       : fp16 bits [H][ceil(I/256)]
 * Rows are output features, K (the reduction index) is contiguous; byte b of a
 * row holds K index 2b in its low nibble and 2b+1 in its high nibble; each
 * nibble is a two's-complement int4 in [-8, 7]; w[r][k] = q[r][k] * s[r][k/256]
 * (no zero-point; the last block of a row may be shorter than 256).
 *
 * Layer computed by moe_w4a16_forward for x [T][H] (FP16):
 *   xin   = PRENORM ? x / sqrt(mean_h x^2 + 1e-6) : x          (per token)
 *   l     = xin . W_r^T + bias                                 (FP32)
 *   p     = softmax(l) over all E;  ids = the k largest l (ties -> lower
 *           expert index), largest first;  w_j = p[ids_j] (not renormalised)
 *   y_j   = W_d (SiLU(W_g xin) * (W_u xin))   for expert ids_j
 *   out   = (RESIDUAL ? x : 0) + sum_{j=0..k-1} w_j y_j        (FP32, j order)
 * rounded to FP16 at two points: the SiLU*up product h (the A16 operand of the
 * down projection) and the final out; the grouped-GEMM path also rounds each
 * expert output y_j to FP16 before the FP32 combine.  How q*s enters the
 * multiply depends on the kernel family: the single-launch decode kernel
 * multiplies the exact integers q and applies s to each 64-wide partial sum
 * in FP32 (q*s exact); the separate-launch decode kernels and the grouped
 * GEMM multiply the FP16 value nearest q*s.  A routed expert whose slot is
 * absent contributes 0 and is counted as a miss (see moe_w4a16_get_status).
 *
 * Threading: a handle is not thread-safe; calls on one handle must be
 * serialised by the caller.  Forwards of one handle share its workspaces and
 * counters: enqueue them on one stream (or order them with events).  Different
 * handles may run on different streams at the same time, the single-launch
 * cooperative kernels included (each handle has its own counters).
 * Asynchrony: every call taking a cudaStream_t
 * only enqueues work on that stream (after synchronous argument checks);
 * device buffers passed in must stay valid until the stream reaches the call.
 * forward enqueues no allocation, no host synchronisation and no
 * host<->device copy, so it may be captured in a CUDA graph.
 *
 * Errors: argument, shape and state errors are returned synchronously and
 * nothing is enqueued.  Conditions only the device can see (a routed expert
 * that has no slot; a bounded wait that gave up) are recorded in a device
 * status word read by moe_w4a16_get_status.  The library never aborts or
 * traps.
 */
#ifndef MOE_W4A16_H
#define MOE_W4A16_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MOE_W4A16_API __attribute__((visibility("default")))
#else
#define MOE_W4A16_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* moe_w4a16_stream_t;   /* same type as cudaStream_t; NULL = legacy default stream */

typedef enum {
  MOE_W4A16_OK = 0,
  MOE_W4A16_ERR_INVALID_ARG = 1,   /* bad pointer, shape, index or flag */
  MOE_W4A16_ERR_CUDA = 2,          /* a CUDA runtime call failed (message in last_error) */
  MOE_W4A16_ERR_OOM = 3,           /* device allocation failed at create */
  MOE_W4A16_ERR_NOT_PACKED = 4,    /* the slot table names a slot never packed */
  MOE_W4A16_ERR_NOT_RESIDENT = 5,  /* get_status: a routed expert had no slot */
  MOE_W4A16_ERR_TIMEOUT = 6,       /* get_status: a bounded device wait gave up */
  MOE_W4A16_ERR_UNSUPPORTED = 7    /* valid request this build does not implement */
} moe_w4a16_status;

/* forward flags */
#define MOE_W4A16_RESIDUAL   1u   /* out = x + MoE(...) */
#define MOE_W4A16_PRENORM    2u   /* experts and router see x / rms(x) */
#define MOE_W4A16_FORCE_GEMV 4u   /* decode kernels whatever T is */
#define MOE_W4A16_FORCE_GEMM 8u   /* tensor-core grouped GEMM whatever T is */
#define MOE_W4A16_UNFUSED   16u   /* decode regime as separate route / gate-up / down launches
                                     instead of the single cooperative launch used for T <= 64 */
#define MOE_W4A16_OFFLOAD   32u   /* the offload-qpacked comparison path (see
                                     moe_w4a16_offload_enable); excludes FORCE_GEMV */

typedef struct {
  int32_t hidden;       /* H: multiple of 64, >= 64 */
  int32_t inter;        /* I: expert intermediate size, multiple of 64, >= 64 */
  int32_t num_experts;  /* E: 1..256 */
  int32_t top_k;        /* k: 1..min(E, 32) */
  int32_t num_slots;    /* S: GPU pool rows, 1..65535 */
  int32_t max_tokens;   /* upper bound on T for every forward, >= 1 */
  int32_t device;       /* CUDA device ordinal */
} moe_w4a16_config;

typedef struct moe_w4a16_handle moe_w4a16_handle;

/* Allocates the slot pool (S rows of the kernel-internal compact layout),
 * the expert->slot table and every forward workspace, sized from cfg.  No
 * slot is packed and the table maps every expert to "absent" until set.
 * On success *out receives the handle; on failure *out is NULL.  H or I that
 * is odd gives ERR_INVALID_ARG; even but not a multiple of 64 gives
 * ERR_UNSUPPORTED. */
MOE_W4A16_API moe_w4a16_status moe_w4a16_create(const moe_w4a16_config* cfg, moe_w4a16_handle** out);

/* Waits for the handle's device work, frees everything it owns.  NULL is OK. */
MOE_W4A16_API moe_w4a16_status moe_w4a16_destroy(moe_w4a16_handle* h);

/* Writes n experts, given in the canonical layout above, into slots
 * [slot0, slot0 + n).  The six arrays may be host or device pointers (the
 * kind is detected per array); host memory is copied synchronously through a
 * handle-owned device staging buffer, device memory is read on `stream`.
 * The pool keeps the compact 4-bit form (re-ordered for the kernels; still
 * 4 bits per weight plus the FP16 scales).  The caller's arrays may be freed
 * once the stream has passed this call. */
MOE_W4A16_API moe_w4a16_status moe_w4a16_pack_experts(moe_w4a16_handle* h, int32_t slot0, int32_t n,
                                        const uint8_t* gate_q, const uint16_t* gate_s,
                                        const uint8_t* up_q, const uint16_t* up_s,
                                        const uint8_t* down_q, const uint16_t* down_s,
                                        moe_w4a16_stream_t stream);

/* expert_to_slot: HOST array [E]; entry e is the slot holding expert e, or -1
 * if expert e is not resident.  Rejected (nothing changes): an entry outside
 * [-1, S), two experts on one slot (ERR_INVALID_ARG), or a slot that was
 * never packed (ERR_NOT_PACKED).  The table is uploaded on `stream`, so
 * forwards enqueued after this call on that stream see it. */
MOE_W4A16_API moe_w4a16_status moe_w4a16_set_slot_table(moe_w4a16_handle* h, const int32_t* expert_to_slot,
                                          moe_w4a16_stream_t stream);

/* One layer forward on `stream`.
 *   x        : device FP16 [T][H]        router_w : device FP16 [E][H]
 *   bias     : device FP32 [E] or NULL   (may hold -inf)
 *   out      : device FP16 [T][H]        (must not alias x)
 * Optional device outputs (NULL to skip), written in the same call:
 *   topk_ids [T][k] int32, topk_w [T][k] FP32,
 *   sorted_pairs [T*k] int32 (flat pair index p = t*k + j, grouped by expert
 *   ascending and by p ascending inside a group), expert_offsets [E+1] int32.
 * x, router_w and out must be 16-byte aligned (ERR_INVALID_ARG otherwise).
 * 0 <= T <= max_tokens; T == 0 enqueues nothing and returns OK.  FORCE_GEMV
 * and FORCE_GEMM are mutually exclusive. */
MOE_W4A16_API moe_w4a16_status moe_w4a16_forward(moe_w4a16_handle* h, const void* x, int32_t T,
                                   const void* router_w, const float* bias, uint32_t flags,
                                   void* out, int32_t* topk_ids, float* topk_w,
                                   int32_t* sorted_pairs, int32_t* expert_offsets,
                                   moe_w4a16_stream_t stream);

/* Same layer with HOST activations: copies x_host (FP16 [T][H]) into a
 * handle-owned device buffer, runs moe_w4a16_forward, copies the result into
 * out_host (FP16 [T][H]) and synchronises `stream` before returning.  Host
 * buffers should be page-locked for the copies to be asynchronous. */
MOE_W4A16_API moe_w4a16_status moe_w4a16_forward_host(moe_w4a16_handle* h, const void* x_host, int32_t T,
                                        const void* router_w, const float* bias, uint32_t flags,
                                        void* out_host, moe_w4a16_stream_t stream);

/* The same as moe_w4a16_forward_host without the final synchronisation: the
 * H2D copy, the forward and the D2H copy are enqueued on `stream` and the call
 * returns.  out_host holds the result once the stream has reached that point
 * (cudaStreamSynchronize or an event); x_host must stay unchanged until then.
 * Calls on one handle reuse its device staging buffers in stream order, so a
 * later call on the same stream may follow at once.  Host buffers must be
 * page-locked for the copies to run asynchronously (pageable buffers are
 * still correct, the driver then stages them synchronously).  Errors as for
 * moe_w4a16_forward; a failed copy enqueue returns ERR_CUDA. */
MOE_W4A16_API moe_w4a16_status moe_w4a16_forward_host_async(moe_w4a16_handle* h, const void* x_host, int32_t T,
                                                            const void* router_w, const float* bias,
                                                            uint32_t flags, void* out_host,
                                                            moe_w4a16_stream_t stream);

/* Synchronises the handle's device, reads and clears the device status word.
 * *miss_count (may be NULL) receives the number of routed token-expert pairs
 * whose expert had no slot since the last call.  Returns ERR_TIMEOUT if a
 * bounded wait gave up, else ERR_NOT_RESIDENT if there was a miss, else OK. */
MOE_W4A16_API moe_w4a16_status moe_w4a16_get_status(moe_w4a16_handle* h, int64_t* miss_count);

/* Message of the last error on this handle ("" if none).  With h == NULL,
 * the message of the last failed create. */
MOE_W4A16_API const char* moe_w4a16_last_error(const moe_w4a16_handle* h);

/* Limits of moe_w4a16_route_noalloc (its scratch is a fixed 5 MiB device array). */
#define MOE_W4A16_NOALLOC_MAX_TOKENS 4096
#define MOE_W4A16_NOALLOC_MAX_HIDDEN 4096
#define MOE_W4A16_NOALLOC_MAX_LOGITS 786432   /* T * num_experts * ceil(hidden / 256) */
#define MOE_W4A16_NOALLOC_MAX_PAIRS 65536     /* T * top_k */

/* Routing of one layer (router logits, softmax / top-k, stable permutation)
 * that allocates nothing and needs no handle.  It runs four launches
 * (tensor-core logits tiles over 256-wide K slices, top-k summing the slices
 * in order, per-expert scan, stable scatter); its ids, weights and
 * permutation equal bit for bit those of moe_w4a16_forward's cooperative
 * router (the forward's router above 8 tokens, outside the single-launch
 * decode kernel), which sums the same logits tiles in the same order.  The Horizon RunMap
 * pages have no counterpart to this entry point; it exists for callers that
 * cannot call cudaMalloc: code that runs inside a runtime whose allocator
 * already owns all device memory (plugins of serving engines that hand out
 * only pre-planned buffers), code that must not risk the implicit device
 * synchronisation or the failure of an allocation on a latency-critical
 * path, and code running while allocation is forbidden.  Creating a handle
 * allocates, so those callers cannot use moe_w4a16_forward's routing.
 *   x [T][H] FP16 and router_w [E][H] FP16: device, 16-byte aligned;
 *   bias [E] FP32 device or NULL; flags: 0 or MOE_W4A16_PRENORM;
 *   topk_ids [T][k] int32, topk_w [T][k] FP32: device outputs (required);
 *   sorted_pairs [T*k] int32, expert_offsets [E+1] int32: device outputs or NULL.
 * Work is enqueued on `stream` (the calling thread's current device).
 * Scratch lives in one file-scope device array of 5 MiB that every device
 * which loads the library keeps until the process exits.  The first call on
 * a device looks up that array's device address (cudaGetSymbolAddress) and
 * caches it for the life of the process; make that first call before any
 * stream capture on the device, and do not reset the device
 * (cudaDeviceReset) while the library is loaded: the cached address would
 * then point into a context that no longer exists.
 * Limits: T <= MOE_W4A16_NOALLOC_MAX_TOKENS, T*E*ceil(H/256) <=
 * ..._MAX_LOGITS, T*k <= ..._MAX_PAIRS, E <= 256, k <= min(E, 32), H a
 * multiple of 64 and <= ..._MAX_HIDDEN;
 * anything beyond returns ERR_INVALID_ARG with a message in
 * moe_w4a16_last_error(NULL), and nothing is enqueued.  All calls, on any
 * stream, share the one array: calls whose work overlaps on the GPU race and
 * give wrong results; serialise them (one stream, or events). */
MOE_W4A16_API moe_w4a16_status moe_w4a16_route_noalloc(const void* x, int32_t T, int32_t hidden,
                                                       int32_t num_experts, int32_t top_k, const void* router_w,
                                                       const float* bias, uint32_t flags, int32_t* topk_ids,
                                                       float* topk_w, int32_t* sorted_pairs,
                                                       int32_t* expert_offsets, moe_w4a16_stream_t stream);

/* Profiling aid.  With events != NULL (an array of 5 cudaEvent_t created by
 * the caller with timing enabled), every later forward on this handle records
 * them on its stream at the stage boundaries: [0] before routing, [1] after
 * routing (on the grouped-GEMM path: after the gather of the x rows that
 * follows routing), [2] after the gate/up kernel, [3] after the down kernel,
 * [4] after the combine ([4] == [3] on the separate-launch decode path, whose down
 * kernel also does the combine; on the single-launch decode path [1] == [0]
 * and [2] == [3] == [4] bracket the one fused kernel).  While the stream is
 * being captured they are recorded as external event nodes of the graph.
 * NULL turns recording off.  The handle keeps the five pointers, not the
 * array. */
MOE_W4A16_API moe_w4a16_status moe_w4a16_set_stage_events(moe_w4a16_handle* h, void* const* events);

/* Bytes of one slot row in the pool (compact weights + scales + padding). */
MOE_W4A16_API size_t moe_w4a16_slot_bytes(const moe_w4a16_handle* h);

/* The largest T the decode (GEMV) kernels take when no FORCE flag is given;
 * larger T runs the tensor-core grouped GEMM.  Settable for sweeps. */
MOE_W4A16_API int32_t moe_w4a16_get_gemv_max_tokens(const moe_w4a16_handle* h);
MOE_W4A16_API moe_w4a16_status moe_w4a16_set_gemv_max_tokens(moe_w4a16_handle* h, int32_t t_star);

/* Which kernel path the last successful forward on this handle enqueued, and
 * how many kernels it launched (debug-output copies not counted):
 *   MOE_W4A16_PATH_DECODE_FUSED  1 cooperative kernel (routing, permutation,
 *                                gate/up, down and combine in one launch)
 *   MOE_W4A16_PATH_DECODE        router (1 kernel) + gate/up + down
 *   MOE_W4A16_PATH_GEMM          router + gather (T <= 8: 1 + 1; above: 1
 *                                kernel that also gathers the x rows) +
 *                                gate/up GEMM + down GEMM + combine
 *   MOE_W4A16_PATH_OFFLOAD       router + gather (as above) + per batch of
 *                                execution slots (expand + dense gate/up GEMM
 *                                + dense down GEMM) + combine
 * PATH_NONE before any forward and after one with T == 0.  *launches may be
 * NULL.  Returns -1 for a NULL handle. */
enum {
  MOE_W4A16_PATH_NONE = 0,
  MOE_W4A16_PATH_DECODE_FUSED = 1,
  MOE_W4A16_PATH_DECODE = 2,
  MOE_W4A16_PATH_GEMM = 3,
  MOE_W4A16_PATH_OFFLOAD = 4
};
MOE_W4A16_API int32_t moe_w4a16_last_path(const moe_w4a16_handle* h, int32_t* launches);

/* The offload-qpacked comparison ("Horizon RunMap - architecture",
 * "Representation and computation" and its profile list: the historical
 * profile that dequantises a low-bit source into bounded FP16/BF16 execution
 * slots).  It is the baseline the compact path is measured against, not the
 * hot path.  Allocates n_slots FP16 execution slots on the handle's device
 * (each 3 * inter * hidden * 2 bytes: gate, up and down expanded, row-major;
 * owned by the handle, freed by destroy; a second call replaces them).  A
 * forward with MOE_W4A16_OFFLOAD then routes as usual, expands each batch of at
 * most n_slots active experts into the slots and runs the grouped GEMM on the
 * FP16 copies (w = q * s rounded to the nearest FP16, the same values the
 * compact GEMM dequantises in shared memory), so its outputs match the compact
 * GEMM path up to FP32 summation order.
 * Errors: INVALID_ARG (NULL handle, n_slots outside [1, 64], shapes the
 * grouped GEMM does not take), CUDA (allocation or tensor-map encoding). */
MOE_W4A16_API moe_w4a16_status moe_w4a16_offload_enable(moe_w4a16_handle* h, int32_t n_slots);


/* Failure-detection self-test (the pages have no counterpart).  Enqueues
 * one tiny kernel whose only wait can never be satisfied -- which = 0: an
 * mbarrier phase that nothing completes; 1: a device word that nothing
 * writes -- using the same bounded-wait helpers as every kernel of the
 * library, with limit_cycles (1000 .. 2^31 SM cycles) in place of the
 * library's limit of 2^31.  The wait gives up and records a timeout in the
 * handle's status word; moe_w4a16_get_status then returns ERR_TIMEOUT (and
 * clears it), and the context stays usable.  ERR_INVALID_ARG for a bad
 * `which` or limit. */
MOE_W4A16_API moe_w4a16_status moe_w4a16_selftest_timeout(moe_w4a16_handle* h, int32_t which,
                                                          int64_t limit_cycles, moe_w4a16_stream_t stream);

/* ======================================================================
 * Expert cache: the partial-residency miss path.
 *
 * Follows the lifecycle of the pages' resident-qpacked-cache-v1 contract
 * ("Horizon RunMap - architecture", section "Immutable authority and miss
 * lifecycle"; "Immutable cache — the scope of ADR 0009"):
 *   - the complete set of E experts stays in caller-owned host memory (the
 *     immutable backing, canonical qpacked layout as for pack_experts) for
 *     the cache's lifetime; it is never written;
 *   - a miss reserves a bounded pinned staging entry and an unpublished
 *     spare slot row; transport is backing -> pinned staging -> device
 *     (repacked into the spare row); a staging entry is reused only after
 *     its transfer-completion event has retired;
 *   - once every miss of the routed group has been transferred, one new
 *     complete generation of the expert->slot table is published
 *     atomically: forwards enqueued on this handle afterwards read it,
 *     forwards enqueued before keep reading the previous one;
 *   - a consumer holds a lease on the generation it read; the row of an
 *     evicted expert, and an old generation's table, are reused only after
 *     every lease on an older generation has retired (its release event
 *     completed);
 *   - eviction discards the device copy (least recently used resident
 *     expert outside the group, ties to the lower expert id); nothing is
 *     ever copied device -> host (d2h_bytes stays 0);
 *   - misses are serialised (one transaction at a time per cache);
 *   - capacity is fixed at create, which rejects insufficient staging or
 *     spare rows;
 *   - a failure before publication leaves the previous generation
 *     authoritative (the transaction's rows return to the spares); a
 *     failure during or after publication faults the cache: every later
 *     call returns MOE_W4A16_ERR_CUDA.
 * While a cache is attached to a handle it owns the handle's slot rows and
 * table: pack_experts and set_slot_table on the handle fail, and the handle
 * must outlive the cache.  Forwards must run between acquire and release of
 * a lease for the reuse guarantees to hold.
 * ==================================================================== */
typedef struct moe_w4a16_cache moe_w4a16_cache;

typedef struct {
  int32_t staging_experts; /* experts the pinned staging arena holds (>= 1) */
  int32_t spare_slots;     /* slot rows kept out of the published table (>= max_group) */
  int32_t max_group;       /* the most distinct experts one acquire may name (1..E) */
} moe_w4a16_cache_config;

typedef struct {
  uint64_t generation;    /* published generation (1 after create) */
  uint64_t transactions;  /* acquires that published a new generation */
  uint64_t hits;          /* experts named by acquires that were resident */
  uint64_t misses;        /* experts named by acquires that were transferred */
  uint64_t evictions;     /* resident experts discarded */
  uint64_t h2d_bytes;     /* expert bytes copied host -> device (canonical qpacked) */
  uint64_t d2h_bytes;     /* expert bytes copied device -> host: always 0 */
  uint64_t lease_waits;   /* times a transaction waited for older leases to retire */
  int32_t resident;       /* experts in the published generation */
  int32_t free_spares;    /* spare rows reusable now */
  int32_t retiring;       /* rows waiting for older leases to retire */
  int32_t active_leases;  /* leases not yet retired */
  int32_t faulted;        /* 1 once a failure after publication began */
} moe_w4a16_cache_stats;

/* Creates a cache over handle h (its slot pool: num_slots rows) with the
 * immutable host backing of all num_experts experts (six canonical arrays
 * as in pack_experts, leading axis = expert id; host memory, caller-owned,
 * unchanged until destroy) and places initial[0..n_initial) canonically in
 * slots 0..n_initial-1 (generation 1).  Admission (ERR_INVALID_ARG):
 * 1 <= max_group <= E, spare_slots >= max_group, staging_experts >= 1,
 * n_initial + spare_slots <= num_slots, distinct valid initial ids.
 * ERR_OOM when the staging arena cannot be allocated.  Synchronous. */
MOE_W4A16_API moe_w4a16_status moe_w4a16_cache_create(moe_w4a16_handle* h, const moe_w4a16_cache_config* cfg,
                                                      const uint8_t* gate_q, const uint16_t* gate_s,
                                                      const uint8_t* up_q, const uint16_t* up_s,
                                                      const uint8_t* down_q, const uint16_t* down_s,
                                                      const int32_t* initial, int32_t n_initial,
                                                      moe_w4a16_cache** out);

/* Waits for every outstanding lease and transfer, detaches and frees. */
MOE_W4A16_API moe_w4a16_status moe_w4a16_cache_destroy(moe_w4a16_cache* c);

/* Makes the distinct experts ids[0..n) (n <= max_group) resident and hands
 * out a lease on the generation that holds them.  All hits: no new
 * generation.  Misses: transfers on `stream`, then publishes a new
 * generation (the table copy is ordered on `stream` after the transfers).
 * May wait on the host for older leases to retire when no spare row is
 * reusable yet.  Errors: ERR_INVALID_ARG (bad ids, n > max_group),
 * ERR_CUDA (transport failed before publication: old generation kept; or
 * cache faulted), ERR_TIMEOUT (simulation: a needed lease never retires). */
MOE_W4A16_API moe_w4a16_status moe_w4a16_cache_acquire(moe_w4a16_cache* c, const int32_t* ids, int32_t n,
                                                       moe_w4a16_stream_t stream, uint64_t* lease);

/* Ends a lease once the work enqueued so far on `stream` completes (an
 * event is recorded; the lease retires when it has completed). */
MOE_W4A16_API moe_w4a16_status moe_w4a16_cache_release(moe_w4a16_cache* c, uint64_t lease,
                                                       moe_w4a16_stream_t stream);

MOE_W4A16_API moe_w4a16_status moe_w4a16_cache_get_stats(moe_w4a16_cache* c, moe_w4a16_cache_stats* out);

/* Slot of `expert` in the published generation, -1 if not resident (or bad
 * arguments). */
MOE_W4A16_API int32_t moe_w4a16_cache_slot_of(const moe_w4a16_cache* c, int32_t expert);

MOE_W4A16_API const char* moe_w4a16_cache_last_error(const moe_w4a16_cache* c);

/* Host-only simulation: the same cache logic with a transport that moves
 * no bytes and touches no GPU (no handle), for testing the lifecycle
 * without a device.  Lease release events complete only when
 * moe_w4a16_cache_sim_complete names them; a transaction that would have to
 * wait for one returns ERR_TIMEOUT before publication.
 * moe_w4a16_cache_sim_fail(c, 1) makes the next transaction's transport
 * fail (before publication), (c, 2) its publication fail. */
MOE_W4A16_API moe_w4a16_status moe_w4a16_cache_create_sim(int32_t num_experts, int32_t num_slots,
                                                          uint64_t expert_bytes,
                                                          const moe_w4a16_cache_config* cfg,
                                                          const int32_t* initial, int32_t n_initial,
                                                          moe_w4a16_cache** out);
MOE_W4A16_API moe_w4a16_status moe_w4a16_cache_sim_complete(moe_w4a16_cache* c, uint64_t lease);
MOE_W4A16_API moe_w4a16_status moe_w4a16_cache_sim_fail(moe_w4a16_cache* c, int32_t where);

#ifdef __cplusplus
}
#endif
#endif /* MOE_W4A16_H */
