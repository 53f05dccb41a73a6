// Canonical qpacked matrix -> kernel-internal compact layout (layout.h).
// Still 4 bits per weight: this re-orders nibbles and scales, it expands nothing.
#include "internal.h"

namespace {

// One thread per output 32-bit word of the packed part of every tile.
__global__ void repack_q_kernel(const uint8_t* __restrict__ q, uint8_t* __restrict__ mat, MatLayout m) {
  const int half_k = m.k / 2;
  const int nkc = m.k / 64;
  const long long words_per_tile = (long long)nkc * 32 * 4;
  const long long n_words = words_per_tile * (m.rows / 16);
  for (long long wi = blockIdx.x * (long long)blockDim.x + threadIdx.x; wi < n_words;
       wi += (long long)gridDim.x * blockDim.x) {
    const int rt = (int)(wi / words_per_tile);
    const int in_tile = (int)(wi % words_per_tile);
    const int j = in_tile & 3;
    const int lane = (in_tile >> 2) & 31;
    const int kc = in_tile >> 7;
    const int g = lane >> 2, c = lane & 3;
    const int r_lo = rt * 16 + g, r_hi = r_lo + 8;
    const int kb = kc * 64 + c * 16 + j * 4;            // K of (a0, a1); (a4, a5) follow at kb + 2
    const uint32_t b_lo0 = q[(size_t)r_lo * half_k + kb / 2];        // (a0, a1)
    const uint32_t b_hi0 = q[(size_t)r_hi * half_k + kb / 2];        // (a2, a3)
    const uint32_t b_lo8 = q[(size_t)r_lo * half_k + (kb + 2) / 2];  // (a4, a5)
    const uint32_t b_hi8 = q[(size_t)r_hi * half_k + (kb + 2) / 2];  // (a6, a7)
    uint32_t w = (b_lo0 & 15u) | ((b_hi0 & 15u) << 4) | ((b_lo8 & 15u) << 8) | ((b_hi8 & 15u) << 12) |
                 ((b_lo0 >> 4) << 16) | ((b_hi0 >> 4) << 20) | ((b_lo8 >> 4) << 24) | ((b_hi8 >> 4) << 28);
    uint32_t* dst = reinterpret_cast<uint32_t*>(mat + (size_t)rt * m.tile_bytes + m.scale_bytes) + in_tile;
    *dst = w ^ 0x88888888u;   // two's complement nibble -> offset binary (q + 8)
  }
}

// tile rt, scale block b, tile row r16  <-  canonical s[rt*16 + r16][b]
__global__ void repack_s_kernel(const uint16_t* __restrict__ s, uint8_t* __restrict__ mat, MatLayout m) {
  const int n = m.rows * m.nb;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
    const int r = i / m.nb, b = i % m.nb;
    const int rt = r / 16, r16 = r % 16;
    uint16_t* dst = reinterpret_cast<uint16_t*>(mat + (size_t)rt * m.tile_bytes) + b * 16 + r16;
    *dst = s[i];
  }
}

}  // namespace

cudaError_t launch_repack_matrix(const uint8_t* q, const uint16_t* s, uint8_t* slot_base,
                                 const MatLayout& m, cudaStream_t st) {
  uint8_t* mat = slot_base + m.off;
  const long long n_words = (long long)m.rows * m.k / 8;
  int blocks = (int)((n_words + 255) / 256);
  if (blocks > 4096) blocks = 4096;
  repack_q_kernel<<<blocks, 256, 0, st>>>(q, mat, m);
  const int ns = m.rows * m.nb;
  repack_s_kernel<<<(ns + 255) / 256, 256, 0, st>>>(s, mat, m);
  return cudaGetLastError();
}
