// Kernel-internal compact layout of one expert slot (host + device).
//
// Each matrix W [R][K] (R output rows, K reduction) keeps 4 bits per weight.
// Packed int4: 16-byte chunks, one per (kc, rt, lane) with kc = K/64 chunk,
// rt = 16-row tile, lane = 0..31, at chunk index (kc * (R/16) + rt) * 32 + lane.
// Word j (0..3) of a chunk covers K values kc*64 + j*16 .. +15 of rows
// rt*16 + g and rt*16 + g + 8 (g = lane/4, c = lane%4): exactly the eight
// values one lane holds in the A operand of a 16x8x16 MMA step,
//   a0,a1 = (row g,   k 2c, 2c+1)   a2,a3 = (row g+8, k 2c, 2c+1)
//   a4,a5 = (row g,   k 2c+8, +9)   a6,a7 = (row g+8, k 2c+8, +9)
// stored as offset-binary nibbles u = q + 8 at nibble positions
//   a0->0, a2->1, a4->2, a6->3, a1->4, a3->5, a5->6, a7->7
// so that masking with 0x000F000F / 0x00F000F0 (after a shift by 0 or 8)
// yields the half2 pairs (a0,a1), (a2,a3), (a4,a5), (a6,a7).
// For a fixed kc, consecutive row tiles are contiguous, so a block of rows
// for one 64-wide K step is one contiguous range (bulk-copy friendly).
// Scales: FP16 [nb][R] (block-major), nb = ceil(K/256).
#pragma once
#include <stddef.h>
#include <stdint.h>

#define MOE_BLOCK_K 256
#define MOE_REGION_ALIGN 256

struct MatLayout {
  uint32_t rows;     // R
  uint32_t k;        // K
  uint32_t nb;       // ceil(K / 256)
  uint64_t q_off;    // byte offset of packed int4 within the slot
  uint64_t s_off;    // byte offset of FP16 scales within the slot
};

struct SlotLayout {
  MatLayout gate, up, down;
  uint64_t bytes;    // slot row size
};

static inline uint64_t moe_align_up(uint64_t v, uint64_t a) { return (v + a - 1) / a * a; }

static inline MatLayout moe_mat_layout(uint32_t rows, uint32_t k, uint64_t* cursor) {
  MatLayout m;
  m.rows = rows;
  m.k = k;
  m.nb = (k + MOE_BLOCK_K - 1) / MOE_BLOCK_K;
  m.q_off = *cursor;
  *cursor = moe_align_up(*cursor + (uint64_t)rows * k / 2, MOE_REGION_ALIGN);
  m.s_off = *cursor;
  *cursor = moe_align_up(*cursor + (uint64_t)m.nb * rows * 2, MOE_REGION_ALIGN);
  return m;
}

static inline SlotLayout moe_slot_layout(uint32_t hidden, uint32_t inter) {
  SlotLayout s;
  uint64_t cur = 0;
  s.gate = moe_mat_layout(inter, hidden, &cur);
  s.up = moe_mat_layout(inter, hidden, &cur);
  s.down = moe_mat_layout(hidden, inter, &cur);
  s.bytes = cur;
  return s;
}
