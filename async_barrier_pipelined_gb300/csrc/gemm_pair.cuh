// CTA-pair variant of the FP16 GEMM kernel (tcgen05 cta_group::2).
//
// A cluster of two CTAs computes one 256-row output tile: CTA r (r = 0, 1)
// loads rows 128r .. 128r+127 of the A tile and one half of the B tile's
// columns into its own shared memory, and the even CTA ("leader") issues
// 256 x W x 16 MMAs that read both CTAs' shared memory and write both CTAs'
// tensor memory (rows 0-127 in the leader's, 128-255 in the peer's).  Per
// CTA a k-block stage is 16 KB of A plus W/2 x 64 halves of B, so the ring
// is six stages deep and each SM pulls a third less data per MMA cycle than
// the single-CTA kernel.  Tiles are W = 256 columns wide, or 128 ("narrow")
// for a thin column remainder or, when K halves do not apply, to balance the
// last wave.  With one split, the tiles of a partial last wave may run as two
// K halves each (see Params::full_units) whose FP32 values a second kernel
// adds.
//
// Operand layouts are a template parameter (bit 0: A stored K x M, bit 1: B
// stored N x K): only the copies' boxes and the MMA descriptors differ.
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
// that were issued, before either CTA may exit.  Every stage carries the
// same bytes per CTA (narrow tiles load both B boxes too), so a fill's byte
// count never depends on its tile.
#pragma once

namespace gf16 {
namespace pair {

constexpr int PM = 256;         // rows per pair tile
constexpr int CM = 128;         // rows per CTA
constexpr int WIDE = 256;       // columns of a wide tile
constexpr int NARROW = 128;     // columns of a narrow tile
constexpr int BK = 64;
constexpr int UMMA_K = 16;
constexpr int STAGES = 6;
constexpr int NUM_THREADS = 192;
constexpr int EPI_WARP0 = 2;
constexpr int EPI_WARPS = 4;

constexpr uint32_t A_STAGE = CM * BK * 2;          // 16 KB
constexpr uint32_t B_BOX_N = 64;                   // columns per B copy (128 B rows)
constexpr uint32_t B_BOX = B_BOX_N * BK * 2;       // 8 KB
constexpr uint32_t B_STAGE = (WIDE / 2) * BK * 2;  // 16 KB (two boxes)
constexpr uint32_t CTA_STAGE_TX = A_STAGE + B_STAGE;  // bytes one CTA copies per stage
constexpr uint32_t EPI_BUF = 32 * 64;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t ACC_COLS = WIDE;

constexpr uint32_t OFF_A = 0;
constexpr uint32_t OFF_B = OFF_A + STAGES * A_STAGE;
constexpr uint32_t OFF_EPI = OFF_B + STAGES * B_STAGE;
constexpr uint32_t OFF_BAR = OFF_EPI + EPI_WARPS * 2 * EPI_BUF;
constexpr uint32_t NUM_BARS = 2 * STAGES + 2 + 2 + 1;
constexpr uint32_t OFF_TMEM_SLOT = OFF_BAR + NUM_BARS * 8;
constexpr uint32_t OFF_ABORT = OFF_TMEM_SLOT + 4;
constexpr uint32_t OFF_PEER_ISSUED = OFF_ABORT + 4;
constexpr uint32_t SMEM_USED = OFF_PEER_ISSUED + 4;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;
static_assert(SMEM_BYTES <= 232448, "over the 227 KB shared-memory limit per CTA");
static_assert(OFF_B % 1024 == 0 && OFF_EPI % 1024 == 0, "swizzled buffers need 1024-B alignment");

// Tile-table entry: bits 0-15 pair-row index (256 rows), bits 16-30 column
// offset in units of 128, bit 31 narrow (128 columns) instead of wide (256).
__host__ __device__ __forceinline__ uint32_t pack(uint32_t tpm, uint32_t n128, bool narrow) {
  return tpm | (n128 << 16) | (narrow ? 0x80000000u : 0u);
}
__host__ __device__ __forceinline__ uint32_t tpm_of(uint32_t e) { return e & 0xFFFFu; }
__host__ __device__ __forceinline__ uint32_t n128_of(uint32_t e) { return (e >> 16) & 0x7FFFu; }
__host__ __device__ __forceinline__ bool narrow_of(uint32_t e) { return (e >> 31) != 0; }

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
  int b3d;       // row-major B seen as 3-D (64 columns, K, column groups): one copy per stage
  // Units [0, full_units) are whole tiles (times the splits); units past it
  // are K halves (one split only): unit full_units + 2 t + q covers half q
  // of the k-blocks of tile order[full_units + t] ("tail" tile t) and stores
  // its FP32 values through tmW, which then maps a [2 t + q][256][256]
  // buffer; a second kernel adds the two halves (P0 + P1) and writes C.
  int full_units;
  int tail_parts;          // 2 with tail units, else 1
};

struct Bars {
  uint32_t full, empty, tfull, tempty, mma_done;
};

struct UnitGeom {
  int m0;        // first row of this CTA's half of the tile
  int n0;        // first column of the tile
  int width;     // 256 or 128
  int split;
  int kb0, kb1;
  int tail;      // tail tile index, or -1 for a whole tile
  int part;      // K part of a tail tile
};

__device__ __forceinline__ UnitGeom unit_geom(const Params& p, int u, uint32_t rank) {
  UnitGeom g;
  int tpos;
  if (u < p.full_units) {
    decode_unit(u, p.split_k, &tpos, &g.split);
    split_range(p.kblocks, p.split_k, g.split, &g.kb0, &g.kb1);
    g.tail = -1;
    g.part = 0;
  } else {
    const int v = u - p.full_units;
    g.tail = v / p.tail_parts;
    g.part = v - g.tail * p.tail_parts;
    g.split = 0;
    split_range(p.kblocks, p.tail_parts, g.part, &g.kb0, &g.kb1);
    tpos = p.full_units + g.tail;
  }
  const uint32_t e = p.order[tpos];
  g.m0 = (int)tpm_of(e) * PM + (int)rank * CM;
  g.n0 = (int)n128_of(e) * 128;
  g.width = narrow_of(e) ? NARROW : WIDE;
  return g;
}

__device__ __noinline__ bool wait_slow(uint32_t bar, uint32_t parity, const Params& p,
                                       volatile int* abort_flag) {
  const uint64_t t0 = ptx::globaltimer();
  while (true) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (ptx::globaltimer() - t0 > p.timeout_ns) {
      *abort_flag = 1;
      *(volatile int*)p.status = (int)GEMM_F16_ERR_TIMEOUT;
      __threadfence_system();
      return false;
    }
  }
}

__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, const Params& p,
                                           volatile int* abort_flag) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  return wait_slow(bar, parity, p, abort_flag);
}

__device__ __noinline__ bool wait_drain(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = ptx::globaltimer();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (ptx::globaltimer() - t0 > limit_ns) return false;
  }
  return true;
}

// ------------------------------------------------------------------ roles
template <int LAYOUT>
__device__ __forceinline__ uint32_t producer_role(const CUtensorMap* tmA, const CUtensorMap* tmB,
                                                  const Params& p, uint32_t base, uint32_t rank,
                                                  uint32_t pair, uint32_t npairs, const Bars& b,
                                                  volatile int* abort_flag) {
  const uint32_t leader_full = ptx::map_to_cta(b.full, 0);
  RingPos pos{0, 0};
  uint32_t issued = 0;
  bool ok = true;
  for (int u = (int)pair; u < p.num_units && ok; u += (int)npairs) {
    const UnitGeom g = unit_geom(p, u, rank);
    // This CTA's B columns: its half of the tile (two 64-column boxes are
    // always loaded; a narrow tile's MMA reads only the first).
    const int nb0 = g.n0 + (int)rank * (g.width / 2);
    const int skip_kb = (u == p.fault_unit && rank == 0) ? g.kb0 : -1;
    for (int kb = g.kb0; kb < g.kb1; ++kb) {
      if (!wait_phase(b.empty + 8 * pos.stage, producer_wait_parity(pos), p, abort_flag)) {
        ok = false;
        break;
      }
      if (rank == 0) ptx::mbar_arrive_expect_tx_relaxed(b.full + 8 * pos.stage, 2 * CTA_STAGE_TX);
      if (kb != skip_kb) {
        const uint32_t fb = leader_full + 8 * pos.stage;
        const int k0 = kb * BK;
        const uint32_t sa = base + OFF_A + pos.stage * A_STAGE;
        if constexpr ((LAYOUT & LAYOUT_AT) != 0) {   // A stored K x M
          ptx::tma_load_2d_pair(sa, tmA, fb, g.m0, k0);
          ptx::tma_load_2d_pair(sa + 8192, tmA, fb, g.m0 + 64, k0);
        } else {
          ptx::tma_load_2d_pair(sa, tmA, fb, k0, g.m0);
        }
        const uint32_t sb = base + OFF_B + pos.stage * B_STAGE;
        if constexpr ((LAYOUT & LAYOUT_BT) != 0) {   // B stored N x K: 128 rows of N
          ptx::tma_load_2d_pair(sb, tmB, fb, k0, nb0);
        } else if (p.b3d) {
          // both 64-column groups of this CTA's half in one copy
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

template <int LAYOUT>
__device__ __forceinline__ void mma_role(const Params& p, uint32_t base, uint32_t tmem_base,
                                         uint32_t pair, uint32_t npairs, const Bars& b,
                                         volatile int* abort_flag) {
  using D = OperandDesc<LAYOUT>;
  RingPos pos{0, 0};
  uint32_t local = 0;
  for (int u = (int)pair; u < p.num_units; u += (int)npairs) {
    const UnitGeom g = unit_geom(p, u, 0);
    const uint32_t idesc = idesc_for_layout(idesc_for(g.width), LAYOUT);
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
      const uint64_t a_desc = smem_desc_sw128(base + OFF_A + pos.stage * A_STAGE, D::a_lbo, D::a_sbo);
      const uint64_t b_desc = smem_desc_sw128(base + OFF_B + pos.stage * B_STAGE, D::b_lbo, D::b_sbo);
      const uint32_t first = (kb == g.kb0) ? 1u : 0u;
#pragma unroll
      for (int k = 0; k < BK / UMMA_K; ++k) {
        ptx::mma_f16_pair(d_tmem, a_desc + ((k * D::a_kstep) >> 4),
                          b_desc + ((k * D::b_kstep) >> 4), idesc, (first && k == 0) ? 0u : 1u);
      }
      ptx::mma_commit_pair(b.empty + 8 * pos.stage, 0x3);
      ring_advance(pos, STAGES);
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

// Per-warp state of the epilogue's FP16 (or split FP32) stores.
struct EpiStore {
  uint32_t stage0;   // this warp's two shared staging buffers
  uint32_t row_off;  // this lane's row in a staging buffer
  uint32_t sw;       // 16-byte-unit swizzle of that row
  uint32_t nstore;   // stores issued so far (selects the buffer)
};

// One 32-column chunk of accumulator values (lane = row) to C, or, with
// `fp32`, as FP32 values to tmW at (wx, wy, wz) (a split partial, or a tail
// tile's K half): rows past M and columns past N are clipped by the copy,
// except a ragged last chunk of an N that is not 16-byte aligned, which goes
// out to C with masked stores.
__device__ __forceinline__ void store_chunk(const CUtensorMap* tmC, const CUtensorMap* tmW,
                                            const Params& p, const uint32_t (&r)[32], int row0,
                                            int col0, bool fp32, int wx, int wy, int wz,
                                            uint32_t lane, EpiStore& st) {
  if (!fp32 && col0 + 32 > p.N && (p.N & 7) != 0) {
    const int row = row0 + (int)lane;
    if (row < p.M) {
      __half* dst = p.C + (int64_t)row * p.ldc + col0;
      const int nvalid = p.N - col0;
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (j < nvalid) dst[j] = __float2half_rn(__uint_as_float(r[j]));
    }
  } else if (!fp32) {
    const uint32_t buf = st.stage0 + (st.nstore & 1u) * EPI_BUF;
    if (lane == 0) ptx::bulk_wait_group_read<1>();
    __syncwarp();
#pragma unroll
    for (uint32_t j = 0; j < 4; ++j) {
      ptx::st_shared_v4(buf + st.row_off + ((j ^ st.sw) << 4), pack_h2(r[8 * j + 0], r[8 * j + 1]),
                        pack_h2(r[8 * j + 2], r[8 * j + 3]), pack_h2(r[8 * j + 4], r[8 * j + 5]),
                        pack_h2(r[8 * j + 6], r[8 * j + 7]));
    }
    ptx::fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      ptx::tma_store_2d(tmC, buf, col0, row0);
      ptx::bulk_commit_group();
    }
    ++st.nstore;
  } else {
#pragma unroll
    for (uint32_t h = 0; h < 2; ++h) {
      if (col0 + 16 * (int)h >= p.N) break;
      const uint32_t buf = st.stage0 + (st.nstore & 1u) * EPI_BUF;
      if (lane == 0) ptx::bulk_wait_group_read<1>();
      __syncwarp();
#pragma unroll
      for (uint32_t j = 0; j < 4; ++j) {
        const uint32_t* v = &r[16 * h + 4 * j];
        ptx::st_shared_v4(buf + st.row_off + ((j ^ st.sw) << 4), v[0], v[1], v[2], v[3]);
      }
      ptx::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        ptx::tma_store_3d(tmW, buf, wx + 16 * (int)h, wy, wz);
        ptx::bulk_commit_group();
      }
      ++st.nstore;
    }
  }
}

__device__ __forceinline__ void epilogue_role(const CUtensorMap* tmC, const CUtensorMap* tmW,
                                              const Params& p, uint32_t base, uint32_t tmem_base,
                                              uint32_t rank, uint32_t pair, uint32_t npairs,
                                              const Bars& b, uint32_t warp, uint32_t lane,
                                              volatile int* abort_flag) {
  const uint32_t quarter = warp & 3u;
  EpiStore st;
  st.stage0 = base + OFF_EPI + (warp - EPI_WARP0) * 2 * EPI_BUF;
  st.row_off = lane * 64u;
  st.sw = (lane >> 1) & 3u;
  st.nstore = 0;
  const uint32_t leader_tempty = ptx::map_to_cta(b.tempty, 0);
  uint32_t local = 0;
  for (int u = (int)pair; u < p.num_units; u += (int)npairs) {
    const UnitGeom g = unit_geom(p, u, rank);
    const uint32_t acc = local & 1u;
    const uint32_t acc_phase = (local >> 1) & 1u;
    bool got = wait_phase(b.tfull + 8 * acc, acc_phase, p, abort_flag);
    if (!__all_sync(0xffffffffu, got)) break;
    ptx::tc_fence_after();
    const int row0 = g.m0 + (int)quarter * 32;
    const uint32_t t_row = tmem_base + acc * ACC_COLS + ((quarter * 32u) << 16);
    // FP32 values for split partials ([split][M][ldw]) and tail halves
    // ([2 t + q][256][256], tile-relative coordinates).
    const bool fp32 = p.split_k > 1 || g.tail >= 0;
    const int wy = g.tail >= 0 ? (int)(rank * 128u + quarter * 32u) : row0;
    const int wz = g.tail >= 0 ? 2 * g.tail + g.part : g.split;
    if (row0 < p.M) {
      for (int c = 0; c < g.width / 32; ++c) {
        const int col0 = g.n0 + c * 32;
        if (col0 >= p.N) break;
        uint32_t r[32];
        ptx::tmem_ld_32x32b_x32(t_row + (uint32_t)c * 32u, r);
        ptx::tmem_ld_wait();
        ptx::reg_fence(r);
        store_chunk(tmC, tmW, p, r, row0, col0, fp32, g.tail >= 0 ? c * 32 : col0, wy, wz, lane,
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

// After both CTAs stopped: make every stage phase that a producer opened
// complete and wait (bounded) until the copies that were issued have
// landed.  Fill j used stage j % STAGES in phase parity (j / STAGES) & 1.
// A fill the leader never reached lacks its arrival: arrive expecting only
// the peer's bytes.  A fill the peer never issued leaves the peer's bytes
// expected: take them off with complete_tx.
__device__ __noinline__ void leader_drain(const Bars& b, uint32_t mine, uint32_t peer,
                                          uint64_t limit_ns) {
  const uint32_t hi = mine > peer ? mine : peer;
  const uint32_t lo = hi > (uint32_t)STAGES ? hi - (uint32_t)STAGES : 0u;
  for (uint32_t j = lo; j < hi; ++j) {
    const uint32_t bar = b.full + 8 * (j % STAGES);
    if (j >= mine) ptx::mbar_arrive_expect_tx_relaxed(bar, CTA_STAGE_TX);
    if (j >= peer) ptx::mbar_complete_tx(bar, CTA_STAGE_TX);
    wait_drain(bar, (j / STAGES) & 1u, limit_ns);
  }
}

template <int LAYOUT>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NUM_THREADS, 1)
    gemm_f16_pair_kernel(const __grid_constant__ CUtensorMap tmA,
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
  const uint32_t pair = blockIdx.x >> 1;
  const uint32_t npairs = gridDim.x >> 1;

  Bars b;
  b.full = base + OFF_BAR;
  b.empty = b.full + 8 * STAGES;
  b.tfull = b.empty + 8 * STAGES;
  b.tempty = b.tfull + 16;
  b.mma_done = b.tempty + 16;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_ABORT);

  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&tmA);
    ptx::prefetch_tmap(&tmB);
    ptx::prefetch_tmap(&tmC);
    if (p.split_k > 1 || p.tail_parts > 1) ptx::prefetch_tmap(&tmW);
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(b.full + 8 * s, 1);
      ptx::mbar_init(b.empty + 8 * s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(b.tfull + 8 * a, 1);
      ptx::mbar_init(b.tempty + 8 * a, 2 * EPI_WARPS);
    }
    ptx::mbar_init(b.mma_done, 1);
    *abort_flag = 0;
    *reinterpret_cast<volatile uint32_t*>(smem + OFF_PEER_ISSUED) = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc_pair(base + OFF_TMEM_SLOT, TMEM_COLS);
    ptx::tmem_relinquish_pair();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();  // the peer's barriers exist before anyone signals them
  ptx::tc_fence_after();
  const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(smem + OFF_TMEM_SLOT);
  // A dependent launch (the split reduction) may be scheduled now; it waits
  // for this grid's completion before touching the partials.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // The work list was written by the host before any launch of this shape,
  // not by the kernel this one waits for: its first entry for this pair can
  // be on its way while the wait lasts.
  if (warp == 0 && lane == 0 && (int)pair < p.num_units) {
    const int u = (int)pair;
    int tpos, split;
    if (u < p.full_units) decode_unit(u, p.split_k, &tpos, &split);
    else tpos = p.full_units + (u - p.full_units) / p.tail_parts;
    ptx::prefetch_l1(p.order + tpos);
  }
  // Launched as a programmatic dependent: everything above (barriers, TMEM,
  // tensor-map prefetch) may overlap the previous kernel's tail; no global
  // memory written by that kernel is touched before it has completed.
  asm volatile("griddepcontrol.wait;" ::: "memory");

  uint32_t issued = 0;
  if (warp == 0) {
    if (lane == 0)
      issued = producer_role<LAYOUT>(&tmA, &tmB, p, base, rank, pair, npairs, b, abort_flag);
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) mma_role<LAYOUT>(p, base, tmem_base, pair, npairs, b, abort_flag);
    __syncwarp();
  } else {
    epilogue_role(&tmC, &tmW, p, base, tmem_base, rank, pair, npairs, b, warp, lane, abort_flag);
  }

  if (warp == 0 && lane == 0 && rank == 1)
    ptx::st_cluster_u32(ptx::map_to_cta(base + OFF_PEER_ISSUED, 0), issued);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();  // both CTAs have stopped issuing
  if (warp == 0 && lane == 0 && rank == 0) {
    const uint32_t peer = *reinterpret_cast<volatile uint32_t*>(smem + OFF_PEER_ISSUED);
    leader_drain(b, issued, peer, p.timeout_ns);
  }
  ptx::cluster_sync();  // no copy into either CTA is still in flight
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
}

}  // namespace pair
}  // namespace gf16
