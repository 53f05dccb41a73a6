// Kernel-internal compact layout of one expert slot (host + device).
//
// Each matrix W [R][K] (R output rows, K reduction) keeps 4 bits per weight.
// It is stored as R/16 row tiles; a tile is one contiguous block of
//   [FP16 scales: nb x 16, block-major]  then  [packed int4: nkc x 32 x 16 B]
// (nb = ceil(K/256), nkc = K/64), so a kernel fetches a whole tile with a
// single bulk copy.  The 16-byte chunk (kc, lane) of a tile holds rows g and
// g + 8 of the tile (g = lane/4, c = lane%4) at the 16 K values
// kc*64 + c*16 .. kc*64 + c*16 + 15.  Its word j (0..3) holds the eight values
// the lane owns in the A operand of MMA step j (16x8x16) of the chunk, whose
// K slots 2c, 2c+1, 2c+8, 2c+9 stand for the K values kb, kb+1, kb+2, kb+3
// (kb = kc*64 + c*16 + 4j):
//   a0,a1 = (row g,   kb, kb+1)     a2,a3 = (row g+8, kb, kb+1)
//   a4,a5 = (row g,   kb+2, kb+3)   a6,a7 = (row g+8, kb+2, kb+3)
// so a lane's B operand for the whole chunk is the 16 consecutive activation
// values kc*64 + c*16 .. + 15 (two 16-byte loads).  Nibbles are offset binary
// u = q + 8 at nibble positions
//   a0->0, a2->1, a4->2, a6->3, a1->4, a3->5, a5->6, a7->7
// so that masking with 0x000F000F / 0x00F000F0 (after a shift by 0 or 8)
// yields the half2 pairs (a0,a1), (a2,a3), (a4,a5), (a6,a7), and the bytes
// 0, 2 (1, 3) of a word are the (row g, row g+8) nibble pairs of (a0..a3)
// ((a4..a7)).
#pragma once
#include <stddef.h>
#include <stdint.h>

#define MOE_BLOCK_K 256
#define MOE_REGION_ALIGN 256

struct MatLayout {
  uint32_t rows;        // R
  uint32_t k;           // K
  uint32_t nb;          // ceil(K / 256)
  uint32_t tile_bytes;  // nb * 32 + 8 * K  (one 16-row tile incl. its scales)
  uint32_t scale_bytes; // nb * 32
  uint64_t off;         // byte offset of the matrix within the slot
};

struct SlotLayout {
  MatLayout gate, up, down;
  uint64_t bytes;       // slot row size
};

static inline uint64_t moe_align_up(uint64_t v, uint64_t a) { return (v + a - 1) / a * a; }

static inline MatLayout moe_mat_layout(uint32_t rows, uint32_t k, uint64_t* cursor) {
  MatLayout m;
  m.rows = rows;
  m.k = k;
  m.nb = (k + MOE_BLOCK_K - 1) / MOE_BLOCK_K;
  m.scale_bytes = m.nb * 32;
  m.tile_bytes = m.scale_bytes + 8 * k;
  m.off = *cursor;
  *cursor = moe_align_up(*cursor + (uint64_t)(rows / 16) * m.tile_bytes, MOE_REGION_ALIGN);
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
