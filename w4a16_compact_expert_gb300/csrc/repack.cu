// Canonical qpacked matrix -> kernel-internal compact layout (layout.h).
// Still 4 bits per weight: this re-orders nibbles, it expands nothing.
#include "internal.h"

namespace {

// One thread per output 32-bit word.
__global__ void repack_q_kernel(const uint8_t* __restrict__ q, uint32_t* __restrict__ out,
                                int rows, int k) {
  const long long n_words = (long long)rows * k / 8;
  const int half_k = k / 2;
  const int row_tiles = rows / 16;
  for (long long wi = blockIdx.x * (long long)blockDim.x + threadIdx.x; wi < n_words;
       wi += (long long)gridDim.x * blockDim.x) {
    const long long chunk = wi >> 2;
    const int j = (int)(wi & 3);
    const int lane = (int)(chunk & 31);
    const long long tile = chunk >> 5;
    const int rt = (int)(tile % row_tiles);
    const int kc = (int)(tile / row_tiles);
    const int g = lane >> 2, c = lane & 3;
    const int r_lo = rt * 16 + g, r_hi = r_lo + 8;
    const int kb = kc * 64 + j * 16 + 2 * c;            // even
    const uint32_t b_lo0 = q[(size_t)r_lo * half_k + kb / 2];        // (a0, a1)
    const uint32_t b_hi0 = q[(size_t)r_hi * half_k + kb / 2];        // (a2, a3)
    const uint32_t b_lo8 = q[(size_t)r_lo * half_k + (kb + 8) / 2];  // (a4, a5)
    const uint32_t b_hi8 = q[(size_t)r_hi * half_k + (kb + 8) / 2];  // (a6, a7)
    uint32_t w = (b_lo0 & 15u) | ((b_hi0 & 15u) << 4) | ((b_lo8 & 15u) << 8) | ((b_hi8 & 15u) << 12) |
                 ((b_lo0 >> 4) << 16) | ((b_hi0 >> 4) << 20) | ((b_lo8 >> 4) << 24) | ((b_hi8 >> 4) << 28);
    out[wi] = w ^ 0x88888888u;   // two's complement nibble -> offset binary (q + 8)
  }
}

// out[b][r] = in[r][b]
__global__ void repack_s_kernel(const uint16_t* __restrict__ s, uint16_t* __restrict__ out, int rows, int nb) {
  const int n = rows * nb;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
    const int b = i / rows, r = i % rows;
    out[i] = s[(size_t)r * nb + b];
  }
}

}  // namespace

cudaError_t launch_repack_matrix(const uint8_t* q, const uint16_t* s, uint8_t* slot_base,
                                 const MatLayout& m, cudaStream_t st) {
  const long long n_words = (long long)m.rows * m.k / 8;
  int blocks = (int)((n_words + 255) / 256);
  if (blocks > 4096) blocks = 4096;
  repack_q_kernel<<<blocks, 256, 0, st>>>(q, reinterpret_cast<uint32_t*>(slot_base + m.q_off), m.rows, m.k);
  const int ns = m.rows * m.nb;
  repack_s_kernel<<<(ns + 255) / 256, 256, 0, st>>>(s, reinterpret_cast<uint16_t*>(slot_base + m.s_off),
                                                    m.rows, m.nb);
  return cudaGetLastError();
}
