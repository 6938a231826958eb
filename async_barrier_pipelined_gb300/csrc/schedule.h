// Index and phase bookkeeping shared by the device roles and by host code
// (the planner, and the host-side replay of the pipeline protocol used in
// tests).  Plain integer arithmetic only, no CUDA types, so it compiles
// both under nvcc and a host C++ compiler.
#pragma once

#include <stdint.h>

#if defined(__CUDACC__)
#define GF16_HD __host__ __device__ __forceinline__
#else
#define GF16_HD inline
#endif

namespace gf16 {

// Position in a ring of `stages` shared-memory stages.  `phase` is the
// parity of the mbarrier phase the current lap uses: a fresh barrier is in
// phase 0, and every full lap of the ring moves each stage one phase on.
struct RingPos {
  uint32_t stage;
  uint32_t phase;
};

GF16_HD void ring_advance(RingPos& p, uint32_t stages) {
  p.stage += 1;
  const uint32_t wrap = (p.stage == stages) ? 1u : 0u;
  p.stage = wrap ? 0u : p.stage;
  p.phase ^= wrap;
}

// Step back one position (inverse of ring_advance).
GF16_HD void ring_retreat(RingPos& p, uint32_t stages) {
  const uint32_t wrap = (p.stage == 0) ? 1u : 0u;
  p.stage = wrap ? stages - 1u : p.stage - 1u;
  p.phase ^= wrap;
}

// Parity a producer waits on before refilling the stage at `p`: it needs
// the consumer's release of the previous lap.  On the first lap this is the
// parity of the phase "before" phase 0, which a fresh barrier reports as
// complete, so the first fill does not wait.
GF16_HD uint32_t producer_wait_parity(const RingPos& p) { return p.phase ^ 1u; }

// Parity a consumer waits on for the stage at `p` to be full.
GF16_HD uint32_t consumer_wait_parity(const RingPos& p) { return p.phase; }

// k-block range [kb0, kb1) of split `s` out of `split_k` over `kblocks`
// k-blocks: contiguous, non-empty when split_k <= kblocks, and covering
// [0, kblocks) exactly once over s = 0 .. split_k-1.
// (A kernel's first unit waits for this on one thread: one split needs no
// division, and while (s + 1) * kblocks fits in 31 bits a 32-bit division
// gives the same quotients as the 64-bit one, at a fraction of its cost.)
GF16_HD void split_range(int kblocks, int split_k, int s, int* kb0, int* kb1) {
  if (split_k == 1) {
    *kb0 = 0;
    *kb1 = kblocks;
  } else if (kblocks <= 46340) {  // s < split_k <= kblocks: (s + 1) * kblocks < 2^31
    *kb0 = (int)((uint32_t)(s * kblocks) / (uint32_t)split_k);
    *kb1 = (int)((uint32_t)((s + 1) * kblocks) / (uint32_t)split_k);
  } else {
    *kb0 = (int)(((int64_t)s * kblocks) / split_k);
    *kb1 = (int)(((int64_t)(s + 1) * kblocks) / split_k);
  }
}

// Work unit u -> (position in the tile order, split index).  The splits of
// one tile are adjacent units, so they run side by side.
GF16_HD void decode_unit(int u, int split_k, int* tile_pos, int* split) {
  *tile_pos = split_k == 1 ? u : u / split_k;
  *split = u - (*tile_pos) * split_k;
}

// Spread the low 16 bits of v to the even bit positions.
GF16_HD uint32_t morton_spread16(uint32_t v) {
  v &= 0xFFFFu;
  v = (v | (v << 8)) & 0x00FF00FFu;
  v = (v | (v << 4)) & 0x0F0F0F0Fu;
  v = (v | (v << 2)) & 0x33333333u;
  v = (v | (v << 1)) & 0x55555555u;
  return v;
}

// Gather the even bits of v into the low 16 bits (inverse of the spread).
GF16_HD uint32_t morton_compact16(uint32_t v) {
  v &= 0x55555555u;
  v = (v | (v >> 1)) & 0x33333333u;
  v = (v | (v >> 2)) & 0x0F0F0F0Fu;
  v = (v | (v >> 4)) & 0x00FF00FFu;
  v = (v | (v >> 8)) & 0x0000FFFFu;
  return v;
}

// Z-order code of tile (tm, tn): tm on the even bits, tn on the odd bits,
// so that tm = compact(code) and tn = compact(code >> 1) ("Xe2 ESIMD GEMM"
// page, "Tile walk order": row index from the even bits, column index from
// the odd bits).
GF16_HD uint32_t morton_code(uint32_t tm, uint32_t tn) {
  return morton_spread16(tm) | (morton_spread16(tn) << 1);
}

GF16_HD uint32_t pack_tile(uint32_t tm, uint32_t tn) { return tm | (tn << 16); }
GF16_HD uint32_t tile_m_of(uint32_t packed) { return packed & 0xFFFFu; }
GF16_HD uint32_t tile_n_of(uint32_t packed) { return packed >> 16; }

// The tile at position `rank` when the tiles of a tiles_m x tiles_n grid are
// listed by increasing morton_code, returned packed (pack_tile).  Z-order
// is the depth-first walk of the quadtree over the enclosing 2^L x 2^L
// square whose child digit is (tn bit, tm bit); descending it, and skipping
// each child by its number of in-grid tiles (the product of its clipped row
// and column extents), reaches the rank-th in-grid tile in 2 L steps with
// no table.  Requires rank < tiles_m * tiles_n and both sizes <= 65536.
GF16_HD uint32_t morton_tile_of_rank(uint32_t rank, uint32_t tiles_m, uint32_t tiles_n) {
  uint32_t side = 1;
  while (side < tiles_m || side < tiles_n) side <<= 1;
  uint32_t m0 = 0, n0 = 0;
  while (side > 1) {
    const uint32_t h = side >> 1;
    for (uint32_t digit = 0; digit < 4; ++digit) {
      const uint32_t cm = m0 + (digit & 1u) * h, cn = n0 + (digit >> 1) * h;
      const uint32_t rows = cm < tiles_m ? (tiles_m - cm < h ? tiles_m - cm : h) : 0u;
      const uint32_t cols = cn < tiles_n ? (tiles_n - cn < h ? tiles_n - cn : h) : 0u;
      const uint32_t count = rows * cols;
      if (rank < count || digit == 3) {
        m0 = cm;
        n0 = cn;
        break;
      }
      rank -= count;
    }
    side = h;
  }
  return pack_tile(m0, n0);
}

}  // namespace gf16
