// Wide CTA-pair variant of the FP16 GEMM kernel (tcgen05 cta_group::2),
// instantiated for 512-column tiles (the 256-column pair kernel is
// gemm_pair.cuh).
//
// A cluster of two CTAs computes one 256-row output tile TN columns wide
// (TN = 256 or 512): CTA r (r = 0, 1) loads rows 128r .. 128r+127 of the A
// tile and its half of B's columns for every 256-column MMA of the tile
// into its own shared memory, and the even CTA ("leader") issues
// 256 x N x 16 MMAs that read both CTAs' shared memory and write both
// CTAs' tensor memory (rows 0-127 in the leader's, 128-255 in the peer's).
//
// Why two widths.  Per CTA and k-block a stage is 16 KB of A plus
// TN/2 x 64 halves of B.  Each SM can take in only about 64 bytes per clock
// from L2; a 256-wide tile needs 32 KB per 512 MMA cycles (64 B/clk, so the
// tensor core waits on loads about a fifth of the time), a 512-wide tile
// 48 KB per 1024 cycles (48 B/clk, tensor-core bound).  The 512-wide tile
// fills all 512 TMEM columns, so its epilogue cannot overlap the next
// tile's main loop; the 256-wide tile keeps two accumulators and overlaps.
// Tiles of a launch are TN wide, or TN/2 or TN/4 (>= 128) where that
// balances the last wave or covers a thin column remainder.
//
// Barrier protocol ("mbarrier State and Operations": phase completes when
// pending arrivals and transaction bytes are both zero):
//   full[s]        leader only, 1 arrival per phase: the leader's producer
//                  does arrive.expect_tx(bytes of both CTAs); both CTAs'
//                  copies complete their bytes on it (the peer's from the
//                  other SM).  The peer's producer never arrives, so no
//                  cross-SM fence sits on its path.  The MMA thread waits
//                  on it.
//   empty[s]       both CTAs, 1 arrival: the leader's tcgen05.commit,
//                  multicast to the pair, when the MMAs reading stage s end.
//   tmem_full[a]   both CTAs, 1 arrival: multicast commit after a tile.
//   tmem_empty[a]  leader only, 8 arrivals: 4 epilogue warps per CTA.
//   mma_done       leader only: last commit, waited before TMEM is freed.
// Every wait is bounded as in the single-CTA kernel.  After an abort the
// leader completes the phases of copies still in flight -- it arrives for
// fills its own producer never reached and takes off the bytes of fills the
// peer never issued (complete_tx) -- and waits (bounded) for the copies
// that were issued, before either CTA may exit.
#pragma once

namespace gf16 {
namespace pairw {

constexpr int PM = 256;         // rows per pair tile
constexpr int CM = 128;         // rows per CTA
constexpr int BK = 64;
constexpr int UMMA_K = 16;
constexpr int NUM_THREADS = 192;
constexpr int EPI_WARP0 = 2;
constexpr int EPI_WARPS = 4;
constexpr int MMA_N = 256;                      // widest single MMA
constexpr uint32_t A_STAGE = CM * BK * 2;       // 16 KB
constexpr uint32_t B_BOX_N = 64;                // columns per B copy (128-byte rows)
constexpr uint32_t B_BOX = B_BOX_N * BK * 2;    // 8 KB
constexpr uint32_t EPI_BUF = 32 * 64;
constexpr uint32_t TMEM_COLS = 512;

template <int TN>
struct Cfg {
  static_assert(TN == 256 || TN == 512, "pair tiles are 256 or 512 wide");
  static constexpr int ACCS = TN == 256 ? 2 : 1;              // TMEM accumulators
  static constexpr int STAGES = TN == 256 ? 6 : 4;
  static constexpr uint32_t STAGE = A_STAGE + (TN / 2) * BK * 2;  // bytes per CTA stage
  static constexpr uint32_t OFF_EPI = STAGES * STAGE;
  static constexpr uint32_t OFF_BAR = OFF_EPI + EPI_WARPS * 2 * EPI_BUF;
  static constexpr uint32_t NUM_BARS = 2 * STAGES + 2 * ACCS + 1;
  static constexpr uint32_t OFF_TMEM_SLOT = OFF_BAR + NUM_BARS * 8;
  static constexpr uint32_t OFF_ABORT = OFF_TMEM_SLOT + 4;
  static constexpr uint32_t OFF_PEER_ISSUED = OFF_ABORT + 4;
  static constexpr uint32_t SMEM_USED = OFF_PEER_ISSUED + 4;
  static constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;
  static_assert(SMEM_BYTES <= 232448, "over the 227 KB shared-memory limit per CTA");
  static_assert(STAGE % 1024 == 0 && OFF_EPI % 1024 == 0, "swizzled buffers need 1024-B alignment");
  static_assert(ACCS * TN <= (int)TMEM_COLS, "accumulators must fit in TMEM");
};

// Tile-table entry: bits 0-15 pair-row index (256 rows), bits 16-29 column
// offset in units of 128, bits 30-31 log2(width / 128): widths 128, 256, 512.
__host__ __device__ __forceinline__ uint32_t pack(uint32_t tpm, uint32_t n128, int width) {
  const uint32_t code = width == 512 ? 2u : width == 256 ? 1u : 0u;
  return tpm | (n128 << 16) | (code << 30);
}
__host__ __device__ __forceinline__ uint32_t tpm_of(uint32_t e) { return e & 0xFFFFu; }
__host__ __device__ __forceinline__ uint32_t n128_of(uint32_t e) { return (e >> 16) & 0x3FFFu; }
__host__ __device__ __forceinline__ int width_of(uint32_t e) { return 128 << (e >> 30); }

// kind::f16 instruction descriptor: D FP32, A/B FP16, A K-major, B MN-major,
// N >> 3 at bits 17-22, M >> 4 at bits 24-28 (M = 256 for the pair).
__host__ __device__ constexpr uint32_t idesc_for(int n) {
  return (1u << 4) | (1u << 16) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(PM >> 4) << 24);
}

struct Params {
  int M, N, K;
  int split_k, kblocks, num_units;
  const uint32_t* order;
  __half* C;
  int64_t ldc;
  int* status;
  unsigned long long timeout_ns;
  int fault_unit;
};

struct Bars {
  uint32_t full, empty, tfull, tempty, mma_done;
};

struct UnitGeom {
  int m0;        // first row of this CTA's half of the tile
  int n0;        // first column of the tile
  int width;     // 512, 256 or 128
  int split;
  int kb0, kb1;
};

__device__ __forceinline__ UnitGeom unit_geom(const Params& p, int u, uint32_t rank) {
  UnitGeom g;
  int tpos;
  decode_unit(u, p.split_k, &tpos, &g.split);
  split_range(p.kblocks, p.split_k, g.split, &g.kb0, &g.kb1);
  const uint32_t e = p.order[tpos];
  g.m0 = (int)tpm_of(e) * PM + (int)rank * CM;
  g.n0 = (int)n128_of(e) * 128;
  g.width = width_of(e);
  return g;
}

// A tile of width w is nmma = max(1, w/256) MMAs of N = min(w, 256); for
// each, this CTA holds half = N/2 of B's columns, half/64 copies of 64.
__device__ __forceinline__ uint32_t cta_stage_bytes(int width) {
  return A_STAGE + (uint32_t)(width / 2) * BK * 2;
}

__device__ __noinline__ bool wait_slow(uint32_t bar, uint32_t parity, uint64_t timeout_ns,
                                       int* status, volatile int* abort_flag) {
  const uint64_t t0 = ptx::globaltimer();
  while (true) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (ptx::globaltimer() - t0 > timeout_ns) {
      *abort_flag = 1;
      *(volatile int*)status = (int)GEMM_F16_ERR_TIMEOUT;
      __threadfence_system();
      return false;
    }
  }
}

__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, const Params& p,
                                           volatile int* abort_flag) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  return wait_slow(bar, parity, p.timeout_ns, p.status, abort_flag);
}

__device__ __noinline__ bool wait_drain(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = ptx::globaltimer();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (ptx::globaltimer() - t0 > limit_ns) return false;
  }
  return true;
}

// ------------------------------------------------------------------ roles
template <int TN>
__device__ __forceinline__ uint32_t producer_role(const CUtensorMap* tmA, const CUtensorMap* tmB,
                                                  const Params& p, uint32_t base, uint32_t rank,
                                                  uint32_t pair, uint32_t npairs, const Bars& b,
                                                  volatile int* abort_flag) {
  using C = Cfg<TN>;
  const uint32_t leader_full = ptx::map_to_cta(b.full, 0);
  RingPos pos{0, 0};
  uint32_t issued = 0;
  bool ok = true;
  for (int u = (int)pair; u < p.num_units && ok; u += (int)npairs) {
    const UnitGeom g = unit_geom(p, u, rank);
    const int mma_n = g.width < MMA_N ? g.width : MMA_N;
    const int nmma = g.width / mma_n;
    const int half = mma_n / 2;                  // B columns per CTA per MMA
    const int boxes = half / (int)B_BOX_N;
    const uint32_t bytes = cta_stage_bytes(g.width);
    const int skip_kb = (u == p.fault_unit && rank == 0) ? g.kb0 : -1;
    for (int kb = g.kb0; kb < g.kb1; ++kb) {
      if (!wait_phase(b.empty + 8 * pos.stage, producer_wait_parity(pos), p, abort_flag)) {
        ok = false;
        break;
      }
      if (rank == 0) ptx::mbar_arrive_expect_tx_relaxed(b.full + 8 * pos.stage, 2 * bytes);
      if (kb != skip_kb) {
        const uint32_t fb = leader_full + 8 * pos.stage;
        const int k0 = kb * BK;
        const uint32_t sa = base + pos.stage * C::STAGE;
        ptx::tma_load_2d_pair(sa, tmA, fb, k0, g.m0);
        uint32_t sb = sa + A_STAGE;
        for (int i = 0; i < nmma; ++i) {
          const int c0 = g.n0 + i * mma_n + (int)rank * half;
          for (int j = 0; j < boxes; ++j, sb += B_BOX)
            ptx::tma_load_2d_pair(sb, tmB, fb, c0 + j * (int)B_BOX_N, k0);
        }
      }
      ++issued;
      ring_advance(pos, C::STAGES);
    }
  }
  return issued;
}

template <int TN>
__device__ __forceinline__ void mma_role(const Params& p, uint32_t base, uint32_t tmem_base,
                                         uint32_t pair, uint32_t npairs, const Bars& b,
                                         volatile int* abort_flag) {
  using C = Cfg<TN>;
  RingPos pos{0, 0};
  uint32_t local = 0;
  for (int u = (int)pair; u < p.num_units; u += (int)npairs) {
    const UnitGeom g = unit_geom(p, u, 0);
    const int mma_n = g.width < MMA_N ? g.width : MMA_N;
    const int nmma = g.width / mma_n;
    const uint32_t b_step = (uint32_t)(mma_n / 2) * BK * 2;   // B bytes per MMA per CTA
    const uint32_t idesc = idesc_for(mma_n);
    const uint32_t acc = C::ACCS == 2 ? (local & 1u) : 0u;
    const uint32_t acc_phase = C::ACCS == 2 ? ((local >> 1) & 1u) : (local & 1u);
    if (!wait_phase(b.tempty + 8 * acc, acc_phase ^ 1u, p, abort_flag)) break;
    ptx::tc_fence_after();
    const uint32_t d_tmem = tmem_base + acc * (uint32_t)TN;
    bool ok = true;
    for (int kb = g.kb0; kb < g.kb1; ++kb) {
      if (!wait_phase(b.full + 8 * pos.stage, consumer_wait_parity(pos), p, abort_flag)) {
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      const uint32_t sa = base + pos.stage * C::STAGE;
      const uint64_t a_desc = smem_desc_sw128(sa, A_LBO, A_SBO);
      const uint32_t first = (kb == g.kb0) ? 1u : 0u;
      for (int i = 0; i < nmma; ++i) {
        const uint64_t b_desc = smem_desc_sw128(sa + A_STAGE + (uint32_t)i * b_step, B_BOX, 1024);
#pragma unroll
        for (int k = 0; k < BK / UMMA_K; ++k) {
          ptx::mma_f16_pair(d_tmem + (uint32_t)(i * MMA_N), a_desc + ((k * A_KSTEP) >> 4),
                            b_desc + ((k * B_KSTEP) >> 4), idesc, (first && k == 0) ? 0u : 1u);
        }
      }
      ptx::mma_commit_pair(b.empty + 8 * pos.stage, 0x3);
      ring_advance(pos, C::STAGES);
    }
    if (!ok) break;
    ptx::mma_commit_pair(b.tfull + 8 * acc, 0x3);
    ++local;
  }
  ptx::mma_commit_pair(b.mma_done, 0x1);
  wait_drain(b.mma_done, 0, p.timeout_ns);
}

__device__ __forceinline__ uint32_t pack_h2(uint32_t lo, uint32_t hi) {
  __half2 h = __floats2half2_rn(__uint_as_float(lo), __uint_as_float(hi));
  return *reinterpret_cast<uint32_t*>(&h);
}

template <int TN>
__device__ __forceinline__ void epilogue_role(const CUtensorMap* tmC, const CUtensorMap* tmW,
                                              const Params& p, uint32_t base, uint32_t tmem_base,
                                              uint32_t rank, uint32_t pair, uint32_t npairs,
                                              const Bars& b, uint32_t warp, uint32_t lane,
                                              volatile int* abort_flag) {
  using C = Cfg<TN>;
  const uint32_t quarter = warp & 3u;
  const uint32_t stage0 = base + C::OFF_EPI + (warp - EPI_WARP0) * 2 * EPI_BUF;
  const uint32_t row_off = lane * 64u;
  const uint32_t sw = (lane >> 1) & 3u;
  const uint32_t leader_tempty = ptx::map_to_cta(b.tempty, 0);
  uint32_t local = 0, nstore = 0;
  for (int u = (int)pair; u < p.num_units; u += (int)npairs) {
    const UnitGeom g = unit_geom(p, u, rank);
    const uint32_t acc = C::ACCS == 2 ? (local & 1u) : 0u;
    const uint32_t acc_phase = C::ACCS == 2 ? ((local >> 1) & 1u) : (local & 1u);
    bool got = wait_phase(b.tfull + 8 * acc, acc_phase, p, abort_flag);
    if (!__all_sync(0xffffffffu, got)) break;
    ptx::tc_fence_after();
    const int row0 = g.m0 + (int)quarter * 32;
    const uint32_t t_row = tmem_base + acc * (uint32_t)TN + ((quarter * 32u) << 16);
    if (row0 < p.M) {
      for (int c = 0; c < g.width / 32; ++c) {
        const int col0 = g.n0 + c * 32;
        if (col0 >= p.N) break;
        uint32_t r[32];
        ptx::tmem_ld_32x32b_x32(t_row + (uint32_t)c * 32u, r);
        ptx::tmem_ld_wait();
        ptx::reg_fence(r);
        if (p.split_k == 1 && col0 + 32 > p.N && (p.N & 7) != 0) {
          const int row = row0 + (int)lane;
          if (row < p.M) {
            __half* dst = p.C + (int64_t)row * p.ldc + col0;
            const int nvalid = p.N - col0;
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (j < nvalid) dst[j] = __float2half_rn(__uint_as_float(r[j]));
          }
        } else if (p.split_k == 1) {
          const uint32_t buf = stage0 + (nstore & 1u) * EPI_BUF;
          if (lane == 0) ptx::bulk_wait_group_read<1>();
          __syncwarp();
#pragma unroll
          for (uint32_t j = 0; j < 4; ++j) {
            ptx::st_shared_v4(buf + row_off + ((j ^ sw) << 4), pack_h2(r[8 * j + 0], r[8 * j + 1]),
                              pack_h2(r[8 * j + 2], r[8 * j + 3]),
                              pack_h2(r[8 * j + 4], r[8 * j + 5]),
                              pack_h2(r[8 * j + 6], r[8 * j + 7]));
          }
          ptx::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            ptx::tma_store_2d(tmC, buf, col0, row0);
            ptx::bulk_commit_group();
          }
          ++nstore;
        } else {
#pragma unroll
          for (uint32_t h = 0; h < 2; ++h) {
            if (col0 + 16 * (int)h >= p.N) break;
            const uint32_t buf = stage0 + (nstore & 1u) * EPI_BUF;
            if (lane == 0) ptx::bulk_wait_group_read<1>();
            __syncwarp();
#pragma unroll
            for (uint32_t j = 0; j < 4; ++j) {
              const uint32_t* v = &r[16 * h + 4 * j];
              ptx::st_shared_v4(buf + row_off + ((j ^ sw) << 4), v[0], v[1], v[2], v[3]);
            }
            ptx::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              ptx::tma_store_3d(tmW, buf, col0 + 16 * (int)h, row0, g.split);
              ptx::bulk_commit_group();
            }
            ++nstore;
          }
        }
      }
    }
    ptx::tc_fence_before();
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive_cluster(leader_tempty + 8 * acc);
    ++local;
  }
  // Only the shared-memory reads of the stores must end before the CTA
  // exits; their writes are complete when the grid is.
  if (lane == 0) ptx::bulk_wait_group_read<0>();
  __syncwarp();
}

// After both CTAs stopped: make every stage phase that a producer opened
// complete and wait (bounded) until the copies that were issued have
// landed.  Fill j used stage j % STAGES in phase parity (j / STAGES) & 1;
// its per-CTA byte count follows from the unit it belongs to.  A fill the
// leader never reached lacks its arrival: arrive expecting only the peer's
// bytes.  A fill the peer never issued leaves the peer's bytes expected:
// take them off with complete_tx.
template <int TN>
__device__ __noinline__ void leader_drain(const uint32_t* order, int num_units, int split_k,
                                          int kblocks, uint32_t full_bar, uint32_t pair,
                                          uint32_t npairs, uint32_t mine, uint32_t peer,
                                          uint64_t limit_ns) {
  using C = Cfg<TN>;
  const uint32_t hi = mine > peer ? mine : peer;
  const uint32_t lo = hi > (uint32_t)C::STAGES ? hi - (uint32_t)C::STAGES : 0u;
  uint32_t fill = 0;
  for (int u = (int)pair; u < num_units && fill < hi; u += (int)npairs) {
    int tpos, s, kb0, kb1;
    decode_unit(u, split_k, &tpos, &s);
    split_range(kblocks, split_k, s, &kb0, &kb1);
    const uint32_t bytes = cta_stage_bytes(width_of(order[tpos]));
    for (int kb = kb0; kb < kb1 && fill < hi; ++kb, ++fill) {
      if (fill < lo) continue;
      const uint32_t bar = full_bar + 8 * (fill % C::STAGES);
      if (fill >= mine) ptx::mbar_arrive_expect_tx_relaxed(bar, bytes);
      if (fill >= peer) ptx::mbar_complete_tx(bar, bytes);
      wait_drain(bar, (fill / C::STAGES) & 1u, limit_ns);
    }
  }
}

template <int TN>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NUM_THREADS, 1)
    gemm_f16_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                         const __grid_constant__ CUtensorMap tmB,
                         const __grid_constant__ CUtensorMap tmC,
                         const __grid_constant__ CUtensorMap tmW, const Params p) {
  using C = Cfg<TN>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  const uint32_t warp = __shfl_sync(0xffffffffu, threadIdx.x >> 5, 0);
  const uint32_t lane = threadIdx.x & 31u;
  const uint32_t rank = ptx::cluster_ctarank();
  const uint32_t pair = blockIdx.x >> 1;
  const uint32_t npairs = gridDim.x >> 1;

  Bars b;
  b.full = base + C::OFF_BAR;
  b.empty = b.full + 8 * C::STAGES;
  b.tfull = b.empty + 8 * C::STAGES;
  b.tempty = b.tfull + 8 * C::ACCS;
  b.mma_done = b.tempty + 8 * C::ACCS;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_ABORT);

  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&tmA);
    ptx::prefetch_tmap(&tmB);
    ptx::prefetch_tmap(&tmC);
    if (p.split_k > 1) ptx::prefetch_tmap(&tmW);
    for (int s = 0; s < C::STAGES; ++s) {
      ptx::mbar_init(b.full + 8 * s, 1);
      ptx::mbar_init(b.empty + 8 * s, 1);
    }
    for (int a = 0; a < C::ACCS; ++a) {
      ptx::mbar_init(b.tfull + 8 * a, 1);
      ptx::mbar_init(b.tempty + 8 * a, 2 * EPI_WARPS);
    }
    ptx::mbar_init(b.mma_done, 1);
    *abort_flag = 0;
    *reinterpret_cast<volatile uint32_t*>(smem + C::OFF_PEER_ISSUED) = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc_pair(base + C::OFF_TMEM_SLOT, TMEM_COLS);
    ptx::tmem_relinquish_pair();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();  // the peer's barriers exist before anyone signals them
  ptx::tc_fence_after();
  const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(smem + C::OFF_TMEM_SLOT);
  // A dependent launch (the split reduction) may be scheduled now; it waits
  // for this grid's completion before touching the partials.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // Launched as a programmatic dependent: everything above (barriers, TMEM,
  // tensor-map prefetch) may overlap the previous kernel's tail; no global
  // memory is touched before that kernel has completed.
  asm volatile("griddepcontrol.wait;" ::: "memory");

  uint32_t issued = 0;
  if (warp == 0) {
    if (lane == 0)
      issued = producer_role<TN>(&tmA, &tmB, p, base, rank, pair, npairs, b, abort_flag);
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) mma_role<TN>(p, base, tmem_base, pair, npairs, b, abort_flag);
    __syncwarp();
  } else {
    epilogue_role<TN>(&tmC, &tmW, p, base, tmem_base, rank, pair, npairs, b, warp, lane,
                      abort_flag);
  }

  if (warp == 0 && lane == 0 && rank == 1)
    ptx::st_cluster_u32(ptx::map_to_cta(base + C::OFF_PEER_ISSUED, 0), issued);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();  // both CTAs have stopped issuing
  // Only an aborted leader can have fills left incomplete: a producer that
  // stopped early starves this pair's MMA, whose bounded wait then aborts.
  if (warp == 0 && lane == 0 && rank == 0 && *abort_flag) {
    const uint32_t peer = *reinterpret_cast<volatile uint32_t*>(smem + C::OFF_PEER_ISSUED);
    leader_drain<TN>(p.order, p.num_units, p.split_k, p.kblocks, b.full, pair, npairs, issued, peer,
                     p.timeout_ns);
  }
  ptx::cluster_sync();  // no copy into either CTA is still in flight
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
}

}  // namespace pairw
}  // namespace gf16
