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
GF16_HD void split_range(int kblocks, int split_k, int s, int* kb0, int* kb1) {
  *kb0 = (int)(((int64_t)s * kblocks) / split_k);
  *kb1 = (int)(((int64_t)(s + 1) * kblocks) / split_k);
}

// Work unit u -> (position in the tile order, split index).  The splits of
// one tile are adjacent units, so they run side by side.
GF16_HD void decode_unit(int u, int split_k, int* tile_pos, int* split) {
  *tile_pos = u / split_k;
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

}  // namespace gf16
