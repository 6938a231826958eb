// Cluster-of-four variant of the CTA-pair GEMM kernel: two CTA pairs share
// their A tiles through multicast copies.
//
// A cluster of four CTAs (ranks 0-3; CTAs 2j and 2j+1 form pair j, the even
// one its leader) computes a 256-row x 512-column cluster tile: pair j the
// 256 x 256 half at columns 256j .. 256j+255, exactly as the pair kernel
// does (tcgen05 cta_group::2, 256 x 256 x 16 MMAs issued by the leader, two
// TMEM accumulators, four epilogue warps per CTA).  CTA r holds rows
// 128(r & 1) .. +127 of the A tile -- the same rows as CTA r ^ 2 of the other
// pair -- so each of the two fetches one 64-row half of those rows and
// multicasts it into both (8 KB per CTA and stage instead of 16 KB).  B is
// per pair: each CTA fetches its pair's half of the 256 columns into its own
// shared memory.  Per SM and k-block the bytes it fetches from L2 drop from
// 32 KB to 24 KB for the same MMA work (an SM receives more through
// multicast than it can fetch alone), and an A whose rows straddle cache
// lines costs half as many extra line fetches.  The price: clusters of four
// fit on fewer SMs than pairs do (36 on 152 SMs), a tile is twice as wide,
// and there is no K-halves tail.  Row-major A and B only.
//
// Barrier protocol (the pair kernel's, plus the cross-pair release):
//   full[s]       pair leaders only, 1 arrival per phase: the leader's
//                 producer does arrive.expect_tx(64 KB: 2 x (16 KB A + 16 KB
//                 B)); the A halves from both pairs and the pair's own B
//                 copies complete their bytes on the leader of the pair they
//                 land in.
//   empty[s]      all four CTAs, 2 arrivals per phase: each pair leader's
//                 tcgen05.commit, multicast to all four CTAs, once the MMAs
//                 reading stage s have finished.  A producer refills stage s
//                 (in its own CTA and, for its A half, in the CTA of the other
//                 pair) only after both pairs have released it.
//   tmem_full[a]  both CTAs of a pair: the leader's multicast commit.
//   tmem_empty[a] pair leader, 8 arrivals (4 epilogue warps per CTA).
//   mma_done      pair leader: its last commit, waited before TMEM is freed.
// Every wait is bounded (GEMM_F16_OPT_TIMEOUT_NS).  After an abort, every CTA
// publishes how many fills it issued to both leaders, and each leader
// completes the phases its producers' stops left open: its own missing
// arrival, and the bytes of contributors that never issued a fill
// (complete_tx), then waits (bounded) until the copies that were issued have
// landed, before any CTA of the cluster may exit.
#pragma once

namespace gf16 {
namespace quad {

using pair::A_STAGE;
using pair::B_BOX;
using pair::B_BOX_N;
using pair::B_STAGE;
using pair::BK;
using pair::CM;
using pair::EPI_BUF;
using pair::EPI_WARP0;
using pair::EPI_WARPS;
using pair::NUM_THREADS;
using pair::Params;
using pair::PM;
using pair::STAGES;
using pair::TMEM_COLS;
using pair::UMMA_K;
using pair::WIDE;
using pair::wait_drain;
using pair::wait_phase;

constexpr int QN = 2 * WIDE;                      // columns of a cluster tile
constexpr uint32_t A_HALF = A_STAGE / 2;          // 64 rows x 64 K: one multicast box
constexpr uint32_t STAGE_TX = 2 * (A_STAGE + B_STAGE);  // bytes landing per pair and stage
constexpr uint32_t OWN_TX = A_HALF + B_STAGE;     // bytes one CTA issues per stage
constexpr uint32_t ACC_COLS = WIDE;

constexpr uint32_t OFF_A = 0;
constexpr uint32_t OFF_B = OFF_A + STAGES * A_STAGE;
constexpr uint32_t OFF_EPI = OFF_B + STAGES * B_STAGE;
constexpr uint32_t OFF_BAR = OFF_EPI + EPI_WARPS * 2 * EPI_BUF;
constexpr uint32_t NUM_BARS = 2 * STAGES + 2 + 2 + 1;
constexpr uint32_t OFF_TMEM_SLOT = OFF_BAR + NUM_BARS * 8;
constexpr uint32_t OFF_ABORT = OFF_TMEM_SLOT + 4;
constexpr uint32_t OFF_ISSUED = OFF_ABORT + 4;    // fills issued by each of the 4 CTAs
constexpr uint32_t SMEM_USED = OFF_ISSUED + 16;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;
static_assert(SMEM_BYTES <= 232448, "over the 227 KB shared-memory limit per CTA");
static_assert(OFF_B % 1024 == 0 && OFF_EPI % 1024 == 0, "swizzled buffers need 1024-B alignment");

struct Bars {
  uint32_t full, empty, tfull, tempty, mma_done;
};

struct UnitGeom {
  int m0;        // first row of this CTA's 128 rows of the tile
  int a_row;     // first row of the 64-row A half this CTA fetches
  int n0;        // first column of this pair's 256 columns
  int split;
  int kb0, kb1;
};

// Unit u = (cluster tile in `order`, split); `order` holds pack_tile(tm, tn)
// over 256-row x 512-column cluster tiles (Params::full_units and
// Params::tail_parts are not used).
__device__ __forceinline__ UnitGeom quad_geom(const Params& p, int u, uint32_t rank) {
  UnitGeom g;
  int tpos;
  decode_unit(u, p.split_k, &tpos, &g.split);
  split_range(p.kblocks, p.split_k, g.split, &g.kb0, &g.kb1);
  const uint32_t e = p.order[tpos];
  const uint32_t q = rank & 1u, pj = rank >> 1;
  g.m0 = (int)tile_m_of(e) * PM + (int)q * CM;
  g.a_row = g.m0 + (int)pj * (CM / 2);
  g.n0 = (int)tile_n_of(e) * QN + (int)pj * WIDE;
  return g;
}

// ------------------------------------------------------------------ roles
__device__ __forceinline__ uint32_t producer_role(const CUtensorMap* tmA, const CUtensorMap* tmB,
                                                  const Params& p, uint32_t base, uint32_t rank,
                                                  uint32_t cl, uint32_t ncl, const Bars& b,
                                                  volatile int* abort_flag) {
  const uint32_t leader_full = ptx::map_to_cta(b.full, rank & ~1u);
  const uint16_t a_mask = (uint16_t)((1u << rank) | (1u << (rank ^ 2u)));
  const uint32_t a_off = (rank >> 1) * A_HALF;  // where this CTA's A half lands in both
  RingPos pos{0, 0};
  uint32_t issued = 0;
  bool ok = true;
  for (int u = (int)cl; u < p.num_units && ok; u += (int)ncl) {
    const UnitGeom g = quad_geom(p, u, rank);
    const int nb0 = g.n0 + (int)(rank & 1u) * (WIDE / 2);  // this CTA's B columns
    const int skip_kb = (u == p.fault_unit && rank == 0) ? g.kb0 : -1;
    for (int kb = g.kb0; kb < g.kb1; ++kb) {
      if (!wait_phase(b.empty + 8 * pos.stage, producer_wait_parity(pos), p, abort_flag)) {
        ok = false;
        break;
      }
      if ((rank & 1u) == 0) ptx::mbar_arrive_expect_tx_relaxed(b.full + 8 * pos.stage, STAGE_TX);
      if (kb != skip_kb) {
        const uint32_t fb = leader_full + 8 * pos.stage;
        const int k0 = kb * BK;
        ptx::tma_load_2d_pair_mc(base + OFF_A + pos.stage * A_STAGE + a_off, tmA, fb, k0,
                                 g.a_row, a_mask);
        const uint32_t sb = base + OFF_B + pos.stage * B_STAGE;
        if (p.b3d) {
          ptx::tma_load_3d_pair(sb, tmB, fb, 0, k0, nb0 / (int)B_BOX_N);
        } else {
          ptx::tma_load_2d_pair(sb, tmB, fb, nb0, k0);
          ptx::tma_load_2d_pair(sb + B_BOX, tmB, fb, nb0 + (int)B_BOX_N, k0);
        }
      }
      ++issued;
      ring_advance(pos, STAGES);
    }
  }
  return issued;
}

// Pair leaders only (rank 0 or 2).
__device__ __forceinline__ void mma_role(const Params& p, uint32_t base, uint32_t tmem_base,
                                         uint32_t rank, uint32_t cl, uint32_t ncl, const Bars& b,
                                         volatile int* abort_flag) {
  const uint32_t idesc = pair::idesc_for(WIDE);
  const uint16_t pair_mask = (uint16_t)(0x3u << rank);
  RingPos pos{0, 0};
  uint32_t local = 0;
  for (int u = (int)cl; u < p.num_units; u += (int)ncl) {
    const UnitGeom g = quad_geom(p, u, rank);
    const uint32_t acc = local & 1u;
    const uint32_t acc_phase = (local >> 1) & 1u;
    if (!wait_phase(b.tempty + 8 * acc, acc_phase ^ 1u, p, abort_flag)) break;
    ptx::tc_fence_after();
    const uint32_t d_tmem = tmem_base + acc * ACC_COLS;
    bool ok = true;
    for (int kb = g.kb0; kb < g.kb1; ++kb) {
      if (!wait_phase(b.full + 8 * pos.stage, consumer_wait_parity(pos), p, abort_flag)) {
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      const uint64_t a_desc = smem_desc_sw128(base + OFF_A + pos.stage * A_STAGE, A_LBO, A_SBO);
      const uint64_t b_desc = smem_desc_sw128(base + OFF_B + pos.stage * B_STAGE, B_LBO, B_SBO);
      const uint32_t first = (kb == g.kb0) ? 1u : 0u;
#pragma unroll
      for (int k = 0; k < BK / UMMA_K; ++k) {
        ptx::mma_f16_pair(d_tmem, a_desc + ((k * A_KSTEP) >> 4), b_desc + ((k * B_KSTEP) >> 4),
                          idesc, (first && k == 0) ? 0u : 1u);
      }
      // both pairs' producers wait for this release (their A halves land here too)
      ptx::mma_commit_pair(b.empty + 8 * pos.stage, 0xF);
      ring_advance(pos, STAGES);
    }
    if (!ok) break;
    ptx::mma_commit_pair(b.tfull + 8 * acc, pair_mask);
    ++local;
  }
  ptx::mma_commit_pair(b.mma_done, (uint16_t)(1u << rank));
  wait_drain(b.mma_done, 0, p.timeout_ns);
}

__device__ __forceinline__ void epilogue_role(const CUtensorMap* tmC, const CUtensorMap* tmW,
                                              const Params& p, uint32_t base, uint32_t tmem_base,
                                              uint32_t rank, uint32_t cl, uint32_t ncl,
                                              const Bars& b, uint32_t warp, uint32_t lane,
                                              volatile int* abort_flag) {
  const uint32_t quarter = warp & 3u;
  pair::EpiStore st;
  st.stage0 = base + OFF_EPI + (warp - EPI_WARP0) * 2 * EPI_BUF;
  st.row_off = lane * 64u;
  st.sw = (lane >> 1) & 3u;
  st.nstore = 0;
  const uint32_t leader_tempty = ptx::map_to_cta(b.tempty, rank & ~1u);
  uint32_t local = 0;
  for (int u = (int)cl; u < p.num_units; u += (int)ncl) {
    const UnitGeom g = quad_geom(p, u, rank);
    const uint32_t acc = local & 1u;
    const uint32_t acc_phase = (local >> 1) & 1u;
    bool got = wait_phase(b.tfull + 8 * acc, acc_phase, p, abort_flag);
    if (!__all_sync(0xffffffffu, got)) break;
    ptx::tc_fence_after();
    const int row0 = g.m0 + (int)quarter * 32;
    const uint32_t t_row = tmem_base + acc * ACC_COLS + ((quarter * 32u) << 16);
    if (row0 < p.M) {
      for (int c = 0; c < WIDE / 32; ++c) {
        const int col0 = g.n0 + c * 32;
        if (col0 >= p.N) break;
        uint32_t r[32];
        ptx::tmem_ld_32x32b_x32(t_row + (uint32_t)c * 32u, r);
        ptx::tmem_ld_wait();
        ptx::reg_fence(r);
        // C (FP16), or a split's FP32 partial at [split][row][column]
        pair::store_chunk(tmC, tmW, p, r, row0, col0, p.split_k > 1, col0, row0, g.split, lane,
                          st);
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

// Pair leader (rank L = 0 or 2), after all four CTAs stopped issuing: make
// every stage phase of its full barriers that a producer opened complete, and
// wait (bounded) until the copies that were issued have landed.  Fill j used
// stage j % STAGES in phase parity (j / STAGES) & 1.  Per fill the pair
// receives 24 KB from each of its own CTAs (A half + B half) and 8 KB from
// each CTA of the other pair (its A half); fills before the last STAGES that
// any producer issued have completed on both leaders (a producer issues fill
// j only after both pairs released fill j - STAGES).
__device__ __noinline__ void leader_drain(const Bars& b, const volatile uint32_t* issued,
                                          uint32_t L, uint64_t limit_ns) {
  uint32_t n[4];
  uint32_t hi = 0;
  for (int c = 0; c < 4; ++c) {
    n[c] = issued[c];
    hi = n[c] > hi ? n[c] : hi;
  }
  const uint32_t lo = hi > (uint32_t)STAGES ? hi - (uint32_t)STAGES : 0u;
  for (uint32_t j = lo; j < hi; ++j) {
    const uint32_t bar = b.full + 8 * (j % STAGES);
    if (j >= n[L]) ptx::mbar_arrive_expect_tx_relaxed(bar, STAGE_TX - OWN_TX);
    if (j >= n[L ^ 1u]) ptx::mbar_complete_tx(bar, OWN_TX);
    if (j >= n[L ^ 2u]) ptx::mbar_complete_tx(bar, A_HALF);
    if (j >= n[L ^ 3u]) ptx::mbar_complete_tx(bar, A_HALF);
    wait_drain(bar, (j / STAGES) & 1u, limit_ns);
  }
}

__global__ void __cluster_dims__(4, 1, 1) __launch_bounds__(NUM_THREADS, 1)
    gemm_f16_quad_kernel(const __grid_constant__ CUtensorMap tmA,
                         const __grid_constant__ CUtensorMap tmB,
                         const __grid_constant__ CUtensorMap tmC,
                         const __grid_constant__ CUtensorMap tmW, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  const uint32_t warp = __shfl_sync(0xffffffffu, threadIdx.x >> 5, 0);
  const uint32_t lane = threadIdx.x & 31u;
  const uint32_t rank = ptx::cluster_ctarank();
  const uint32_t cl = blockIdx.x >> 2;
  const uint32_t ncl = gridDim.x >> 2;
  const bool leader = (rank & 1u) == 0;

  Bars b;
  b.full = base + OFF_BAR;
  b.empty = b.full + 8 * STAGES;
  b.tfull = b.empty + 8 * STAGES;
  b.tempty = b.tfull + 16;
  b.mma_done = b.tempty + 16;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_ABORT);
  volatile uint32_t* issued_by = reinterpret_cast<volatile uint32_t*>(smem + OFF_ISSUED);

  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&tmA);
    ptx::prefetch_tmap(&tmB);
    ptx::prefetch_tmap(&tmC);
    if (p.split_k > 1) ptx::prefetch_tmap(&tmW);
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(b.full + 8 * s, 1);
      ptx::mbar_init(b.empty + 8 * s, 2);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(b.tfull + 8 * a, 1);
      ptx::mbar_init(b.tempty + 8 * a, 2 * EPI_WARPS);
    }
    ptx::mbar_init(b.mma_done, 1);
    *abort_flag = 0;
    for (int c = 0; c < 4; ++c) issued_by[c] = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc_pair(base + OFF_TMEM_SLOT, TMEM_COLS);
    ptx::tmem_relinquish_pair();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();  // every CTA's barriers exist before anyone signals them
  ptx::tc_fence_after();
  const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(smem + OFF_TMEM_SLOT);
  // A dependent launch (the split reduction) may be scheduled now; it waits
  // for this grid's completion before touching the partials.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // The tile order was written by the host, not by the kernel this one
  // waits for: its first entry for this cluster can be on its way meanwhile.
  if (warp == 0 && lane == 0 && (int)cl < p.num_units) {
    int tpos, split;
    decode_unit((int)cl, p.split_k, &tpos, &split);
    ptx::prefetch_l1(p.order + tpos);
  }
  // Launched as a programmatic dependent: no global memory written by the
  // previous kernel is touched before it has completed.
  asm volatile("griddepcontrol.wait;" ::: "memory");

  uint32_t issued = 0;
  if (warp == 0) {
    if (lane == 0) issued = producer_role(&tmA, &tmB, p, base, rank, cl, ncl, b, abort_flag);
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0 && leader) mma_role(p, base, tmem_base, rank, cl, ncl, b, abort_flag);
    __syncwarp();
  } else {
    epilogue_role(&tmC, &tmW, p, base, tmem_base, rank, cl, ncl, b, warp, lane, abort_flag);
  }

  if (warp == 0 && lane == 0) {
    ptx::st_cluster_u32(ptx::map_to_cta(base + OFF_ISSUED + 4 * rank, 0), issued);
    ptx::st_cluster_u32(ptx::map_to_cta(base + OFF_ISSUED + 4 * rank, 2), issued);
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();  // all four CTAs have stopped issuing
  if (warp == 0 && lane == 0 && leader) leader_drain(b, issued_by, rank, p.timeout_ns);
  ptx::cluster_sync();  // no copy into any CTA of the cluster is still in flight
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
}

}  // namespace quad
}  // namespace gf16
