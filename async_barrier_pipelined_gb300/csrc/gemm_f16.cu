// Barrier-pipelined FP16 GEMM for GB300 (sm_103a): C = A * B, FP32 accumulate.
//
// One persistent CTA per SM, 192 threads in three roles:
//   warp 0      TMA producer: one elected lane fills a STAGES-deep ring of
//               shared-memory stages (A tile 128x64, B tile 64x256, 48 KB).
//               Per stage it arrives on full[s] with expect_tx(48 KB) and
//               issues the copies, which complete the transaction bytes.
//   warp 1      allocates 512 TMEM columns (two 128x256 FP32 accumulators)
//               and one lane issues tcgen05.mma (128x256x16, four per
//               k-block), releasing each stage with tcgen05.commit -> empty[s]
//               and handing a finished accumulator over with
//               tcgen05.commit -> tmem_full[acc].
//   warps 2..5  epilogue: tcgen05.ld of its 32-lane TMEM quarter, FP16
//               round-to-nearest-even, swizzled shared staging, TMA store.
//               (Split runs store FP32 partial tiles instead.)  Each warp
//               arrives on tmem_empty[acc] when it has read the accumulator,
//               so the MMA warp can start the next tile in the other one.
//
// This is the split-barrier pattern of the "Xe2 Nbarrier Pipelining" page
// ("Core Concept: Split Barrier"; "Producer-Consumer Pattern") carried over
// to mbarriers: the producer arrives (expect_tx) and moves on; consumers wait
// as late as possible.  The barrier rules followed are those of the
// "mbarrier State and Operations" page ("Phase Completion Condition", "Core
// APIs", "Three update paths").  One arrive per barrier phase per role, with
// no second arrive before the phase completes ("Xe2 Nbarrier Pipelining",
// "What Doesn't Work: Double-Arrive Deadlock"); every role walks the same
// work units and k-blocks, so arrivals and waits stay balanced on every path
// ("Xe2 ESIMD GEMM" page, "Hardware limits": equal barrier counts; "Insert
// Cluster Barrier Pass" page, Rules 4-5: handshakes balanced across tail
// and drain).  Ragged edges need no tail loop: the tensor copies fill
// out-of-bounds elements with zero and clip stores at the tensor bounds.
//
// Every barrier wait is bounded: past the plan's time limit the role records
// GEMM_F16_ERR_TIMEOUT, raises a CTA-wide abort flag, stops issuing, waits
// (bounded) for its own operations in flight, and the CTA frees its TMEM and
// exits.

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <utility>
#include <vector>

#include "host.h"
#include "ptx.cuh"
#include "schedule.h"
#include "common.cuh"

namespace gf16 {

// ------------------------------------------------------------------ tiling
constexpr int BM = 128;          // output tile rows (= MMA M, = TMEM lanes)
constexpr int BN = 256;          // widest output tile (= MMA N); a launch may use 128 or 64
constexpr int BK = 64;           // k-block: 64 halves = one 128-byte swizzle row
constexpr int UMMA_K = 16;       // K of one kind::f16 MMA
constexpr int STAGES = 4;          // stages of the widest tile; narrower tiles get more
constexpr int MAX_STAGES = 8;
constexpr int NUM_THREADS = 192;
constexpr int EPI_WARP0 = 2;
constexpr int EPI_WARPS = 4;

constexpr uint32_t A_STAGE = BM * BK * 2;        // 16 KB
constexpr uint32_t B_BOX_N = 64;                 // N extent of one B copy (128 B)
constexpr uint32_t B_BOX = B_BOX_N * BK * 2;     // 8 KB
constexpr uint32_t B_STAGE = BN * BK * 2;        // 32 KB (room for the widest tile)
constexpr uint32_t EPI_BUF = 32 * 64;            // 32 rows x 64 B staging box
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t ACC_COLS = BN;

// The ring: `stages` stages of (A tile, B tile) back to back, each stage
// A_STAGE + W*BK*2 bytes for a W-wide tile; 196,608 bytes hold 4 stages of
// 256-wide, 6 of 128-wide or 8 of 64-wide tiles.
constexpr uint32_t RING_BYTES = STAGES * (A_STAGE + B_STAGE);
constexpr uint32_t OFF_EPI = RING_BYTES;
constexpr uint32_t OFF_BAR = OFF_EPI + EPI_WARPS * 2 * EPI_BUF;
constexpr uint32_t NUM_BARS = 2 * MAX_STAGES + 2 + 2 + 1;  // full, empty, tmem_full, tmem_empty, mma_done
constexpr uint32_t OFF_TMEM_SLOT = OFF_BAR + NUM_BARS * 8;
constexpr uint32_t OFF_ABORT = OFF_TMEM_SLOT + 4;
constexpr uint32_t SMEM_USED = OFF_ABORT + 4;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;  // room to align the base to 1024
static_assert(SMEM_BYTES <= 232448, "over the 227 KB shared-memory limit per CTA");
static_assert(OFF_EPI % 1024 == 0 && A_STAGE % 1024 == 0, "swizzled buffers need 1024-B alignment");

// Stages of the ring for a W-wide tile.
__host__ __device__ constexpr int stages_for(int w) {
  return (int)(RING_BYTES / (A_STAGE + (uint32_t)w * BK * 2)) < MAX_STAGES
             ? (int)(RING_BYTES / (A_STAGE + (uint32_t)w * BK * 2))
             : MAX_STAGES;
}
static_assert(stages_for(256) == 4 && stages_for(128) == 6 && stages_for(64) == 8, "ring sizes");
static_assert(2 * ACC_COLS <= TMEM_COLS, "two accumulators must fit in TMEM");

// Operand layouts (the `layout` of gemm_f16_run_ex): bit 0 = A is stored
// K x M (M contiguous), bit 1 = B is stored N x K (K contiguous).  Row-major
// A is K-major for the MMA and row-major B is MN-major; a stored-transposed
// operand flips that.  Instruction-descriptor bits 15 / 16: A / B MN-major.
constexpr int LAYOUT_AT = 1, LAYOUT_BT = 2;
__host__ __device__ constexpr uint32_t idesc_for_layout(uint32_t idesc, int layout) {
  return (idesc & ~((1u << 15) | (1u << 16))) | ((layout & LAYOUT_AT) ? (1u << 15) : 0u) |
         ((layout & LAYOUT_BT) ? 0u : (1u << 16));
}

// A tile (K-major, 128-byte swizzle): 8-row groups 1024 B apart (SBO); the
// leading offset is unused for swizzled K-major operands.  One MMA K-slice
// of 16 halves is 32 bytes, so slice k starts 32*k bytes into the rows.
constexpr uint32_t A_LBO = 16, A_SBO = 1024, A_KSTEP = UMMA_K * 2;
// B tile (MN-major, 128-byte swizzle): 64-column groups 8 KB apart along N
// (LBO, one TMA box each), 8-row groups of K 1024 B apart (SBO).  Slice k
// covers rows 16k .. 16k+15, i.e. 2048 bytes further.
constexpr uint32_t B_LBO = B_BOX, B_SBO = 1024, B_KSTEP = UMMA_K * 128;
// Stored-transposed operands: an M-contiguous A tile is MN-major like
// row-major B (two 64-row copies 8 KB apart, 8-row groups of K 1 KB apart,
// 2048 bytes per K slice); an N x K (K-contiguous) B tile is K-major like
// row-major A (rows 128 B, 8-row groups 1 KB apart, 32 bytes per K slice).
constexpr uint32_t AT_LBO = 8192, AT_SBO = 1024, AT_KSTEP = UMMA_K * 128;
constexpr uint32_t BT_LBO = 16, BT_SBO = 1024, BT_KSTEP = UMMA_K * 2;
template <int LAYOUT>
struct OperandDesc {
  static constexpr uint32_t a_lbo = (LAYOUT & LAYOUT_AT) ? AT_LBO : A_LBO;
  static constexpr uint32_t a_sbo = (LAYOUT & LAYOUT_AT) ? AT_SBO : A_SBO;
  static constexpr uint32_t a_kstep = (LAYOUT & LAYOUT_AT) ? AT_KSTEP : A_KSTEP;
  static constexpr uint32_t b_lbo = (LAYOUT & LAYOUT_BT) ? BT_LBO : B_LBO;
  static constexpr uint32_t b_sbo = (LAYOUT & LAYOUT_BT) ? BT_SBO : B_SBO;
  static constexpr uint32_t b_kstep = (LAYOUT & LAYOUT_BT) ? BT_KSTEP : B_KSTEP;
};

struct Params {
  int M, N, K;
  int bn;                  // tile width of this launch: 256, 128 or 64
  int stages;              // ring depth for that width (stages_for(bn))
  uint32_t stage_bytes;    // A_STAGE + bn * BK * 2
  int tiles_m, tiles_n, split_k, kblocks, num_units;
  int row_major;           // tile order: 1 row-major, 0 Morton (morton_tile_of_rank)
  __half* C;               // output, for the masked stores of a ragged last chunk
  int64_t ldc;
  int* status;             // device-visible status word
  unsigned long long timeout_ns;
  int fault_unit;          // test only: unit whose first stage gets no copy
};

struct Bars {
  uint32_t full, empty, tfull, tempty, mma_done;  // shared addresses of the arrays
};

// Packed (tm, tn) of the tile at position `tpos` of the launch's tile order.
// With every unit in the first wave (one per CTA) the walk order cannot
// change what shares L2 at a time, and the quadtree descent (~1 us on one
// thread, before the first copy of a CTA's only tile) is not worth it: such
// launches take the row-major order.
__device__ __forceinline__ uint32_t tile_at(const Params& p, int tpos) {
  return (p.row_major || p.num_units <= (int)gridDim.x)
             ? pack_tile((uint32_t)tpos / (uint32_t)p.tiles_n, (uint32_t)tpos % (uint32_t)p.tiles_n)
             : morton_tile_of_rank((uint32_t)tpos, (uint32_t)p.tiles_m, (uint32_t)p.tiles_n);
}

// ------------------------------------------------------------------ waits
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

// Bounded phase wait; false if it timed out or another role aborted.
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, const Params& p,
                                           volatile int* abort_flag) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  return wait_slow(bar, parity, p, abort_flag);
}

// ------------------------------------------------------------------ roles
// Returns, through pos_out / issued_out, where the ring stands when the role
// stops, so that an aborted CTA can drain its copies in flight.
template <int LAYOUT>
__device__ __forceinline__ void producer_role(const CUtensorMap* tmA, const CUtensorMap* tmB,
                                              const Params& p, uint32_t base, const Bars& b,
                                              volatile int* abort_flag, RingPos* pos_out,
                                              uint32_t* issued_out) {
  RingPos pos{0, 0};
  uint32_t issued = 0;
  bool ok = true;
  const int boxes = p.bn / (int)B_BOX_N;
  const uint32_t stage_tx = A_STAGE + (uint32_t)p.bn * BK * 2;
  for (int u = blockIdx.x; u < p.num_units && ok; u += gridDim.x) {
    int tpos, s, kb0, kb1;
    decode_unit(u, p.split_k, &tpos, &s);
    split_range(p.kblocks, p.split_k, s, &kb0, &kb1);
    const uint32_t packed = tile_at(p, tpos);
    const int m0 = (int)tile_m_of(packed) * BM;
    const int n0 = (int)tile_n_of(packed) * p.bn;
    const int skip_kb = (u == p.fault_unit) ? kb0 : -1;
    for (int kb = kb0; kb < kb1; ++kb) {
      if (!wait_phase(b.empty + 8 * pos.stage, producer_wait_parity(pos), p, abort_flag)) {
        ok = false;
        break;
      }
      const uint32_t fb = b.full + 8 * pos.stage;
      ptx::mbar_arrive_expect_tx_relaxed(fb, stage_tx);
      if (kb != skip_kb) {
        const uint32_t sa = base + pos.stage * p.stage_bytes;
        const uint32_t sb = sa + A_STAGE;
        const int k0 = kb * BK;
        if constexpr ((LAYOUT & LAYOUT_AT) != 0) {
          ptx::tma_load_2d(sa, tmA, fb, m0, k0);            // 64 rows of M x 64 of K
          ptx::tma_load_2d(sa + 8192, tmA, fb, m0 + 64, k0);
        } else {
          ptx::tma_load_2d(sa, tmA, fb, k0, m0);
        }
        if constexpr ((LAYOUT & LAYOUT_BT) != 0) {
          ptx::tma_load_2d(sb, tmB, fb, k0, n0);            // bn rows of N x 64 of K
        } else {
          for (int j = 0; j < boxes; ++j)
            ptx::tma_load_2d(sb + j * B_BOX, tmB, fb, n0 + j * (int)B_BOX_N, k0);
        }
      }
      ++issued;
      ring_advance(pos, (uint32_t)p.stages);
    }
  }
  *pos_out = pos;
  *issued_out = issued;
}

// After an abort: wait (bounded) for the copies of the most recently issued
// stages, one per stage, so that no tensor copy still writes this CTA's
// shared memory when it exits.  A stage whose phase already completed
// returns at once.
__device__ __noinline__ void producer_drain(const Bars& b, RingPos pos, uint32_t issued,
                                            uint32_t stages, uint64_t limit_ns) {
  const uint32_t n = issued < stages ? issued : stages;
  for (uint32_t i = 0; i < n; ++i) {
    ring_retreat(pos, stages);
    wait_drain(b.full + 8 * pos.stage, consumer_wait_parity(pos), limit_ns);
  }
}

template <int LAYOUT>
__device__ __forceinline__ void mma_role(const Params& p, uint32_t base, uint32_t tmem_base,
                                         const Bars& b, volatile int* abort_flag) {
  using D = OperandDesc<LAYOUT>;
  RingPos pos{0, 0};
  uint32_t local = 0;
  const uint32_t idesc = idesc_for_layout(make_idesc(BM, p.bn), LAYOUT);
  for (int u = blockIdx.x; u < p.num_units; u += gridDim.x) {
    int tpos, s, kb0, kb1;
    decode_unit(u, p.split_k, &tpos, &s);
    split_range(p.kblocks, p.split_k, s, &kb0, &kb1);
    const uint32_t acc = local & 1u;
    const uint32_t acc_phase = (local >> 1) & 1u;
    if (!wait_phase(b.tempty + 8 * acc, acc_phase ^ 1u, p, abort_flag)) break;
    ptx::tc_fence_after();
    const uint32_t d_tmem = tmem_base + acc * ACC_COLS;
    bool ok = true;
    for (int kb = kb0; kb < kb1; ++kb) {
      if (!wait_phase(b.full + 8 * pos.stage, consumer_wait_parity(pos), p, abort_flag)) {
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      const uint32_t sa = base + pos.stage * p.stage_bytes;
      const uint64_t a_desc = smem_desc_sw128(sa, D::a_lbo, D::a_sbo);
      const uint64_t b_desc = smem_desc_sw128(sa + A_STAGE, D::b_lbo, D::b_sbo);
      const uint32_t first = (kb == kb0) ? 1u : 0u;
#pragma unroll
      for (int k = 0; k < BK / UMMA_K; ++k) {
        ptx::mma_f16(d_tmem, a_desc + ((k * D::a_kstep) >> 4), b_desc + ((k * D::b_kstep) >> 4),
                     idesc, (first && k == 0) ? 0u : 1u);
      }
      ptx::mma_commit(b.empty + 8 * pos.stage);
      ring_advance(pos, (uint32_t)p.stages);
    }
    if (!ok) break;
    ptx::mma_commit(b.tfull + 8 * acc);
    ++local;
  }
  // Every MMA issued so far must be finished before TMEM is freed.
  ptx::mma_commit(b.mma_done);
  wait_drain(b.mma_done, 0, p.timeout_ns);
}

__device__ __forceinline__ uint32_t pack_half2(uint32_t lo, uint32_t hi) {
  __half2 h = __floats2half2_rn(__uint_as_float(lo), __uint_as_float(hi));
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ void epilogue_role(const CUtensorMap* tmC, const CUtensorMap* tmW,
                                              const Params& p, uint32_t base, uint32_t tmem_base,
                                              const Bars& b, uint32_t warp, uint32_t lane,
                                              volatile int* abort_flag) {
  const uint32_t quarter = warp & 3u;  // TMEM lanes 32*quarter .. +31 are this warp's
  const uint32_t stage0 = base + OFF_EPI + (warp - EPI_WARP0) * 2 * EPI_BUF;
  // Staging layout = the tensor copy's 64-byte swizzle: row r at r*64, its
  // 16-byte chunk c at chunk position c ^ ((r >> 1) & 3).
  const uint32_t row_off = lane * 64u;
  const uint32_t sw = (lane >> 1) & 3u;
  uint32_t local = 0, nstore = 0;
  for (int u = blockIdx.x; u < p.num_units; u += gridDim.x) {
    int tpos, s;
    decode_unit(u, p.split_k, &tpos, &s);
    const uint32_t packed = tile_at(p, tpos);
    const int m0 = (int)tile_m_of(packed) * BM;
    const int n0 = (int)tile_n_of(packed) * p.bn;
    const uint32_t acc = local & 1u;
    const uint32_t acc_phase = (local >> 1) & 1u;
    bool got = wait_phase(b.tfull + 8 * acc, acc_phase, p, abort_flag);
    if (!__all_sync(0xffffffffu, got)) break;
    ptx::tc_fence_after();
    const int row0 = m0 + (int)quarter * 32;
    const uint32_t t_row = tmem_base + acc * ACC_COLS + ((quarter * 32u) << 16);
    if (row0 < p.M) {
      for (int c = 0; c < p.bn / 32; ++c) {
        const int col0 = n0 + c * 32;
        if (col0 >= p.N) break;
        uint32_t r[32];
        ptx::tmem_ld_32x32b_x32(t_row + (uint32_t)c * 32u, r);
        ptx::tmem_ld_wait();
        ptx::reg_fence(r);
        if (p.split_k == 1 && col0 + 32 > p.N && (p.N & 7) != 0) {
          // The chunk straddles a column bound that is not 16-byte aligned.
          // A tensor store would write on up to the next 16-byte boundary
          // past N, so this chunk goes out with masked plain stores.
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
            ptx::st_shared_v4(buf + row_off + ((j ^ sw) << 4), pack_half2(r[8 * j + 0], r[8 * j + 1]),
                              pack_half2(r[8 * j + 2], r[8 * j + 3]),
                              pack_half2(r[8 * j + 4], r[8 * j + 5]),
                              pack_half2(r[8 * j + 6], r[8 * j + 7]));
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
              ptx::tma_store_3d(tmW, buf, col0 + 16 * (int)h, row0, s);
              ptx::bulk_commit_group();
            }
            ++nstore;
          }
        }
      }
    }
    ptx::tc_fence_before();
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(b.tempty + 8 * acc);
    ++local;
  }
  // Only the shared-memory reads of the stores must end before the CTA
  // exits; their writes are complete when the grid is.
  if (lane == 0) ptx::bulk_wait_group_read<0>();
  __syncwarp();
}

// ------------------------------------------------------------------ kernels
template <int LAYOUT>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_f16_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmW,
                    const Params p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  const uint32_t warp = __shfl_sync(0xffffffffu, threadIdx.x >> 5, 0);
  const uint32_t lane = threadIdx.x & 31u;

  Bars b;
  b.full = base + OFF_BAR;
  b.empty = b.full + 8 * MAX_STAGES;
  b.tfull = b.empty + 8 * MAX_STAGES;
  b.tempty = b.tfull + 16;
  b.mma_done = b.tempty + 16;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_ABORT);

  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&tmA);
    ptx::prefetch_tmap(&tmB);
    ptx::prefetch_tmap(&tmC);
    if (p.split_k > 1) ptx::prefetch_tmap(&tmW);
    for (int s = 0; s < p.stages; ++s) {
      ptx::mbar_init(b.full + 8 * s, 1);   // the producer's arrive.expect_tx (+ tx bytes)
      ptx::mbar_init(b.empty + 8 * s, 1);  // one tcgen05.commit per use
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(b.tfull + 8 * a, 1);           // one tcgen05.commit per tile
      ptx::mbar_init(b.tempty + 8 * a, EPI_WARPS);  // one arrive per epilogue warp
    }
    ptx::mbar_init(b.mma_done, 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(base + OFF_TMEM_SLOT, TMEM_COLS);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(smem + OFF_TMEM_SLOT);
  // A dependent launch (the split reduction) may be scheduled now; it waits
  // for this grid's completion before touching the partials.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // Launched as a programmatic dependent: everything above (barriers, TMEM,
  // tensor-map prefetch) may overlap the previous kernel's tail; no global
  // memory is touched before that kernel has completed.
  asm volatile("griddepcontrol.wait;" ::: "memory");

  RingPos prod_pos{0, 0};
  uint32_t prod_issued = 0;
  if (warp == 0) {
    if (lane == 0)
      producer_role<LAYOUT>(&tmA, &tmB, p, base, b, abort_flag, &prod_pos, &prod_issued);
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) mma_role<LAYOUT>(p, base, tmem_base, b, abort_flag);
    __syncwarp();
  } else {
    epilogue_role(&tmC, &tmW, p, base, tmem_base, b, warp, lane, abort_flag);
  }

  ptx::tc_fence_before();
  __syncthreads();
  // Every role has stopped, so the abort flag is final here.
  if (warp == 0 && lane == 0 && *abort_flag)
    producer_drain(b, prod_pos, prod_issued, (uint32_t)p.stages, p.timeout_ns);
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// Row repack of an operand whose row pitch is not a multiple of 128 bytes:
// dst[r, c] = src[r, c] for r < rows, c < cols, with dst rows at a pitch of
// whole 128-byte lines.  A 128-byte copy-box row of such an operand spans two
// cache lines, which makes the operand copies of the GEMM kernels much
// slower than the lines they bring; the repacked copy is read instead.  Each
// thread moves 16-byte chunks (both pitches are multiples of 8 elements and
// both bases 16-byte aligned); a row's last chunk, if it ends past `cols`,
// is moved element by element so that nothing beyond the row is read.  The
// columns of dst past `cols` are never read (the tensor map's extent is
// `cols`).  Launched in stream order after whatever wrote src.
__global__ void __launch_bounds__(256)
    pack_rows_kernel(const __half* __restrict__ src, int64_t ld_src, __half* __restrict__ dst,
                     int64_t ld_dst, int64_t rows, int64_t cols) {
  // The product kernel that follows may start its set-up now; it waits for
  // this grid's completion (griddepcontrol.wait) before it reads dst.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int64_t chunks = (cols + 7) / 8;
  const int64_t total = rows * chunks;
  const int64_t step = (int64_t)gridDim.x * blockDim.x;
  for (int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; g < total; g += 4 * step) {
    uint4 v[4];
    int64_t r[4], c[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t gi = g + u * step;
      r[u] = gi / chunks;
      c[u] = (gi - r[u] * chunks) * 8;
      if (gi < total && c[u] + 8 <= cols)
        v[u] = __ldcs(reinterpret_cast<const uint4*>(src + r[u] * ld_src + c[u]));
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t gi = g + u * step;
      if (gi >= total) continue;
      if (c[u] + 8 <= cols) {
        *reinterpret_cast<uint4*>(dst + r[u] * ld_dst + c[u]) = v[u];
      } else {
        for (int64_t t = c[u]; t < cols; ++t) dst[r[u] * ld_dst + t] = src[r[u] * ld_src + t];
      }
    }
  }
}

// Fixed-order split reduction: C[i,j] = fp16_rn(P_0 + P_1 + ... + P_{S-1}),
// summed left to right in FP32.  Each thread owns 4 consecutive columns;
// the partial loads are issued sixteen splits at a time (independent loads,
// so a 16-way split waits for one round of loads, not sixteen), but the
// additions keep the order t = 0, 1, ..., S-1.
__device__ __forceinline__ void add4(float4& acc, const float4& v) {
  acc.x += v.x;
  acc.y += v.y;
  acc.z += v.z;
  acc.w += v.w;
}

__global__ void __launch_bounds__(256)
    splitk_reduce_kernel(const float* __restrict__ ws, int M, int N, int64_t ldw, int split_k,
                         int64_t split_stride, __half* __restrict__ C, int64_t ldc) {
  // Launched as a programmatic dependent of the GEMM kernel: wait here until
  // that grid has finished and its partials are visible.  (No early signal
  // to the next kernel: letting the next product start its set-up here made
  // 512 x 512 x 32768 in 16 splits 2 us slower per call.)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int64_t groups = (N + 3) / 4;
  const int64_t total = (int64_t)M * groups;
  for (int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; g < total;
       g += (int64_t)gridDim.x * blockDim.x) {
    const int64_t i = g / groups;
    const int j = (int)(g - i * groups) * 4;
    const float* src = ws + i * ldw + j;
    float4 acc = *reinterpret_cast<const float4*>(src);
    int s = 1;
    for (; s + 16 <= split_k; s += 16) {
      float4 v[16];
#pragma unroll
      for (int q = 0; q < 16; ++q)
        v[q] = *reinterpret_cast<const float4*>(src + (int64_t)(s + q) * split_stride);
#pragma unroll
      for (int q = 0; q < 16; ++q) add4(acc, v[q]);
    }
    if (s < split_k) {
      // the last 1..15 splits, also loaded together before they are added
      float4 v[15];
#pragma unroll
      for (int q = 0; q < 15; ++q)
        if (s + q < split_k)
          v[q] = *reinterpret_cast<const float4*>(src + (int64_t)(s + q) * split_stride);
#pragma unroll
      for (int q = 0; q < 15; ++q)
        if (s + q < split_k) add4(acc, v[q]);
    }
    const __half2 h0 = __floats2half2_rn(acc.x, acc.y), h1 = __floats2half2_rn(acc.z, acc.w);
    __half* dst = C + i * ldc + j;
    if (j + 4 <= N) {
      uint2 v;
      v.x = *reinterpret_cast<const uint32_t*>(&h0);
      v.y = *reinterpret_cast<const uint32_t*>(&h1);
      *reinterpret_cast<uint2*>(dst) = v;
    } else {
      const __half vals[4] = {__low2half(h0), __high2half(h0), __low2half(h1), __high2half(h1)};
      for (int t = 0; t < N - j; ++t) dst[t] = vals[t];
    }
  }
}

}  // namespace gf16

#include "gemm_pair.cuh"
#include "gemm_quad.cuh"

namespace gf16 {
// C of the pair kernel's tail tiles: C[i, j] = fp16_rn(P0[i, j] + P1[i, j]),
// P_q the FP32 values of K half q, stored as [2 t + q][256][256] for tail
// tile t = tiles[t] (pair-kernel table entries).  One thread per 4 columns;
// rows past M and columns past N are skipped.  Launched as a programmatic
// dependent of the pair kernel: waits for its completion first.
__global__ void __launch_bounds__(256)
    tail_reduce_kernel(const float* __restrict__ ws, const uint32_t* __restrict__ tiles,
                       int ntiles, int M, int N, __half* __restrict__ C, int64_t ldc) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int64_t total = (int64_t)ntiles * 256 * 64;
  for (int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; g < total;
       g += (int64_t)gridDim.x * blockDim.x) {
    const int t = (int)(g / (256 * 64));
    const int rem = (int)(g - (int64_t)t * 256 * 64);
    const int row = rem >> 6, col = (rem & 63) * 4;
    const uint32_t e = tiles[t];
    const int width = pair::narrow_of(e) ? pair::NARROW : pair::WIDE;
    const int i = (int)pair::tpm_of(e) * pair::PM + row;
    const int j = (int)pair::n128_of(e) * 128 + col;
    if (col >= width || i >= M || j >= N) continue;
    const float* p0 = ws + ((int64_t)(2 * t) * 256 + row) * 256 + col;
    const float4 a = *reinterpret_cast<const float4*>(p0);
    const float4 b = *reinterpret_cast<const float4*>(p0 + 256 * 256);
    const __half2 h0 = __floats2half2_rn(a.x + b.x, a.y + b.y);
    const __half2 h1 = __floats2half2_rn(a.z + b.z, a.w + b.w);
    __half* dst = C + (int64_t)i * ldc + j;
    if (j + 4 <= N && (ldc & 3) == 0) {
      uint2 v;
      v.x = *reinterpret_cast<const uint32_t*>(&h0);
      v.y = *reinterpret_cast<const uint32_t*>(&h1);
      *reinterpret_cast<uint2*>(dst) = v;
    } else {
      const __half vals[4] = {__low2half(h0), __high2half(h0), __low2half(h1), __high2half(h1)};
      for (int k = 0; k < 4 && j + k < N; ++k) dst[k] = vals[k];
    }
  }
}
}  // namespace gf16

// ====================================================================== host
using namespace gf16;
using namespace gf16::host;

namespace {

// Tile order of a tiles_m x tiles_n grid: row-major (order 1) or Morton
// (order 0, by increasing morton_code; the kernels derive the same order
// from a tile's rank with morton_tile_of_rank).
void build_tile_order(int tiles_m, int tiles_n, int order, std::vector<uint32_t>& out) {
  out.clear();
  out.reserve((size_t)tiles_m * tiles_n);
  const uint32_t n = (uint32_t)tiles_m * (uint32_t)tiles_n;
  for (uint32_t r = 0; r < n; ++r)
    out.push_back(order == 1 ? pack_tile(r / (uint32_t)tiles_n, r % (uint32_t)tiles_n)
                             : morton_tile_of_rank(r, (uint32_t)tiles_m, (uint32_t)tiles_n));
}

// Pair-kernel work-list entries as the host planner and gemm_f16_pair_tiles
// see them: pair row (256 rows) in bits 0-15, column offset in units of 128
// in bits 16-29, log2(width / 128) in bits 30-31 (width 128 or 256).
uint32_t ptile(uint32_t tpm, uint32_t n128, int width) {
  return tpm | (n128 << 16) | ((width == 256 ? 1u : 0u) << 30);
}
uint32_t ptile_tpm(uint32_t e) { return e & 0xFFFFu; }
uint32_t ptile_n128(uint32_t e) { return (e >> 16) & 0x3FFFu; }
int ptile_width(uint32_t e) { return 128 << (e >> 30); }

double pair_makespan(const std::vector<uint32_t>& tiles, int pairs) {
  std::vector<double> load((size_t)pairs, 0.0);
  for (size_t i = 0; i < tiles.size(); ++i)
    load[i % (size_t)pairs] += (double)ptile_width(tiles[i]) / pair::WIDE;
  return *std::max_element(load.begin(), load.end());
}

// K halves for the tiles of a partial last wave of 256-wide pair tiles (one
// split only).  A pair tile's k-blocks take about the same time whatever its
// width (measured at 4096^3: a 256 x 128 tile of the last wave 19 us, a
// 256 x 256 tile 18.8 us), so a half-width tile does not shorten the wave;
// two units of half the k-blocks each do.  Each half stores its FP32 values
// and a small kernel adds the two (in half order) and writes C.  Used when
// the 2 r halves of the r tiles of the partial wave fit in one wave and the
// tiles have at least 32 k-blocks (shorter ones gain less than the partial
// stores and the extra launch cost).  Returns 2, or 1 for no split.
int tail_parts_for(int64_t tiles, int pairs, int split_k, int kblocks) {
  if (split_k != 1 || pairs <= 0 || kblocks < 32) return 1;
  const int64_t r = tiles % pairs;
  return (r > 0 && 2 * r <= pairs) ? 2 : 1;
}

// Pair-kernel tile list: 256-wide tiles over the output in Morton order
// (pair-row on the even bits) while more than 128 columns remain, then the
// column remainder as 128-wide tiles.  With one split, if the tiles leave a
// partial last wave, the last (count % pairs) tiles get K halves (`*parts`
// = 2, see tail_parts_for); otherwise the full tiles of that wave are cut
// into 128-wide halves when that shortens the busiest pair's work.
void build_pair_tiles(int M, int N, int kblocks, int pairs, int split_k, int order,
                      std::vector<uint32_t>& out, int* parts) {
  *parts = 1;
  const int tn = pair::WIDE, w_half = pair::NARROW;
  const int tpms = (int)ceil_div(M, pair::PM);
  int full_cols = 0;
  while (N - full_cols * tn > w_half) ++full_cols;
  std::vector<uint32_t> grid;
  build_tile_order(tpms, std::max(full_cols, 1), order, grid);
  std::vector<uint32_t> full, rest;
  if (full_cols > 0)
    for (uint32_t e : grid) full.push_back(ptile(tile_m_of(e), tile_n_of(e) * 2, tn));
  if (N - full_cols * tn > 0)
    for (int t = 0; t < tpms; ++t) rest.push_back(ptile(t, full_cols * 2, w_half));
  out = full;
  out.insert(out.end(), rest.begin(), rest.end());
  if (split_k != 1 || pairs <= 0 || full.empty()) return;
  *parts = tail_parts_for((int64_t)out.size(), pairs, split_k, kblocks);
  if (*parts > 1) return;
  const size_t r = full.size() % (size_t)pairs;
  if (r == 0) return;
  std::vector<uint32_t> alt(full.begin(), full.end() - r);
  for (size_t i = full.size() - r; i < full.size(); ++i)
    for (int k = 0; k < 2; ++k) {
      const uint32_t n128 = ptile_n128(full[i]) + k;
      if ((int64_t)n128 * 128 < N) alt.push_back(ptile(ptile_tpm(full[i]), n128, w_half));
    }
  alt.insert(alt.end(), rest.begin(), rest.end());
  if (pair_makespan(alt, pairs) < pair_makespan(out, pairs)) out.swap(alt);
}
}  // namespace

namespace {

// Row-major B (K x N, N a multiple of 64) as a 3-D tensor (64 columns, K
// rows, N / 64 column groups; strides: row, 128 bytes), boxes of 64 x 64 x 2:
// one copy fetches both 64-column groups of a pair CTA's half of a B stage,
// in the same shared-memory layout as two 2-D boxes.  Cached in the plan.
int cached_encode_b3d(gemm_f16_plan_s* p, CUtensorMap* map, const void* ptr, uint64_t K,
                      uint64_t N, uint64_t ldb) {
  const uint64_t key[8] = {(uint64_t)(uintptr_t)ptr, K, N, ldb, 0, 0, 0, 0x3D00000000000000ull};
  if (tmap_lookup(p, key, map)) return GEMM_F16_OK;
  EncodeTiledFn fn = encode_fn();
  if (!fn) return GEMM_F16_ERR_CUDA;
  const cuuint64_t dims[3] = {64, K, N / 64};
  const cuuint64_t strides[2] = {ldb * 2, 128};
  const cuuint32_t box[3] = {64, (cuuint32_t)BK, 2};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(ptr), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    std::snprintf(g_last_cuda_error, sizeof(g_last_cuda_error),
                  "cuTensorMapEncodeTiled (3-D B) failed (CUresult %d)", (int)r);
    return GEMM_F16_ERR_CUDA;
  }
  tmap_remember(p, key, *map);
  return GEMM_F16_OK;
}

// Host <-> device copy of a row-strided matrix: one plain copy when both
// sides are contiguous, a pitched copy otherwise.
cudaError_t copy_rows(void* dst, int64_t dpitch, const void* src, int64_t spitch,
                      int64_t row_bytes, int64_t rows, cudaMemcpyKind kind, cudaStream_t stream) {
  if (dpitch == row_bytes && spitch == row_bytes)
    return cudaMemcpyAsync(dst, src, (size_t)(row_bytes * rows), kind, stream);
  return cudaMemcpy2DAsync(dst, (size_t)dpitch, src, (size_t)spitch, (size_t)row_bytes,
                           (size_t)rows, kind, stream);
}

}  // namespace

namespace gf16 {
namespace host {

int gemm_plan_init(gemm_f16_plan_s* p, const cudaDeviceProp& prop) {
  void* const single[4] = {(void*)gemm_f16_kernel<0>, (void*)gemm_f16_kernel<1>,
                           (void*)gemm_f16_kernel<2>, (void*)gemm_f16_kernel<3>};
  void* const pairs[4] = {(void*)pair::gemm_f16_pair_kernel<0>, (void*)pair::gemm_f16_pair_kernel<1>,
                          (void*)pair::gemm_f16_pair_kernel<2>, (void*)pair::gemm_f16_pair_kernel<3>};
  for (int l = 0; l < 4; ++l) {
    GF16_CUDA(cudaFuncSetAttribute(single[l], cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   (int)SMEM_BYTES),
              "cudaFuncSetAttribute(max dynamic smem)");
    GF16_CUDA(cudaFuncSetAttribute(pairs[l], cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   (int)pair::SMEM_BYTES),
              "cudaFuncSetAttribute(pair kernel smem)");
  }
  // Co-resident clusters of two for the pair kernel (0 if the query fails:
  // the pair kernel is then not used).
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(prop.multiProcessorCount / 2 * 2), 1, 1);
  cfg.blockDim = dim3(pair::NUM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = pair::SMEM_BYTES;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = 2;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  int clusters = 0;
  if (cudaOccupancyMaxActiveClusters(&clusters, pair::gemm_f16_pair_kernel<0>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    clusters = 0;
  }
  p->max_pairs = clusters;
  // ... and of four for the cluster-of-four kernel.
  GF16_CUDA(cudaFuncSetAttribute(quad::gemm_f16_quad_kernel,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)quad::SMEM_BYTES),
            "cudaFuncSetAttribute(cluster-of-four kernel smem)");
  cfg.gridDim = dim3((unsigned)(prop.multiProcessorCount / 4 * 4), 1, 1);
  cfg.blockDim = dim3(quad::NUM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = quad::SMEM_BYTES;
  attr.val.clusterDim.x = 4;
  int quads = 0;
  if (cudaOccupancyMaxActiveClusters(&quads, quad::gemm_f16_quad_kernel, &cfg) != cudaSuccess) {
    cudaGetLastError();
    quads = 0;
  }
  p->max_quads = clusters > 0 ? quads : 0;
  return GEMM_F16_OK;
}

void gemm_plan_release(gemm_f16_plan_s* p) {
  for (auto& t : p->orders) cudaFree(t.dev);
  p->orders.clear();
  if (p->apack) cudaFree(p->apack);
  if (p->tail_ws) cudaFree(p->tail_ws);
  for (int sl = 0; sl < 2; ++sl) {
    for (int i = 0; i < 3; ++i)
      if (p->hbuf[sl][i]) cudaFree(p->hbuf[sl][i]);
    if (p->in_done[sl]) cudaEventDestroy(p->in_done[sl]);
    if (p->gemm_done[sl]) cudaEventDestroy(p->gemm_done[sl]);
  }
}

}  // namespace host
}  // namespace gf16

extern "C" {

int gemm_f16_tile_shape(int* bm, int* bn, int* bk, int* stages) {
  if (bm) *bm = BM;
  if (bn) *bn = BN;
  if (bk) *bk = BK;
  if (stages) *stages = STAGES;
  return GEMM_F16_OK;
}

int gemm_f16_validate_ex(int layout, int M, int N, int K, const void* A, int64_t lda,
                         const void* B, int64_t ldb, const void* C, int64_t ldc, int split_k) {
  if (layout < 0 || layout > 3) return GEMM_F16_ERR_INVALID_ARG;
  if (M <= 0 || N <= 0 || K <= 0) return GEMM_F16_ERR_INVALID_ARG;
  if (ceil_div(M, BM) > 65535 || ceil_div(N, BN) > 65535) return GEMM_F16_ERR_INVALID_ARG;
  if (!A || !B || !C) return GEMM_F16_ERR_INVALID_ARG;
  const int64_t a_row = (layout & LAYOUT_AT) ? M : K;   // elements in a stored row of A
  const int64_t b_row = (layout & LAYOUT_BT) ? K : N;   // ... of B
  if (lda < a_row || ldb < b_row || ldc < N) return GEMM_F16_ERR_INVALID_ARG;
  if (split_k < 1 || split_k > ceil_div(K, BK)) return GEMM_F16_ERR_INVALID_ARG;
  if (((uintptr_t)A | (uintptr_t)B | (uintptr_t)C) & 15u) return GEMM_F16_ERR_MISALIGNED;
  if ((lda | ldb | ldc) & 7) return GEMM_F16_ERR_MISALIGNED;
  return GEMM_F16_OK;
}

int gemm_f16_validate(int M, int N, int K, const void* A, int64_t lda, const void* B, int64_t ldb,
                      const void* C, int64_t ldc, int split_k) {
  return gemm_f16_validate_ex(0, M, N, K, A, lda, B, ldb, C, ldc, split_k);
}

int64_t gemm_f16_tile_order(int tiles_m, int tiles_n, int order, uint32_t* out, int64_t cap) {
  if (tiles_m < 1 || tiles_n < 1 || tiles_m > 65535 || tiles_n > 65535) return GEMM_F16_ERR_INVALID_ARG;
  if (order != 0 && order != 1) return GEMM_F16_ERR_INVALID_ARG;
  if (cap < 0 || (cap > 0 && !out)) return GEMM_F16_ERR_INVALID_ARG;
  std::vector<uint32_t> v;
  build_tile_order(tiles_m, tiles_n, order, v);
  const int64_t n = (int64_t)v.size();
  if (cap > 0) std::memcpy(out, v.data(), sizeof(uint32_t) * (size_t)std::min<int64_t>(n, cap));
  return n;
}

int64_t gemm_f16_pair_tiles(int M, int N, int K, int pairs, int split_k, int order,
                            int tile_width, uint32_t* out, int64_t cap, int* tail_parts) {
  if (M <= 0 || N <= 0 || K <= 0 || pairs < 1 || split_k < 1 || (order != 0 && order != 1))
    return GEMM_F16_ERR_INVALID_ARG;
  if (tile_width != 256) return GEMM_F16_ERR_INVALID_ARG;
  if (ceil_div(M, pair::PM) > 65535 || (N + 127) / 128 >= 0x3FFF) return GEMM_F16_ERR_INVALID_ARG;
  if (cap < 0 || (cap > 0 && !out)) return GEMM_F16_ERR_INVALID_ARG;
  std::vector<uint32_t> v;
  int parts = 1;
  build_pair_tiles(M, N, (int)ceil_div(K, BK), pairs, split_k, order, v, &parts);
  const int64_t n = (int64_t)v.size();
  if (cap > 0) std::memcpy(out, v.data(), sizeof(uint32_t) * (size_t)std::min<int64_t>(n, cap));
  if (tail_parts) *tail_parts = parts;
  return n;
}

}  // extern "C"

namespace {

int upload_table(gemm_f16_plan_s* p, const int64_t (&key)[6], const std::vector<uint32_t>& host,
                 const uint32_t** out, int parts = 1) {
  uint32_t* dev = nullptr;
  GF16_CUDA(cudaMalloc(&dev, host.size() * sizeof(uint32_t)), "cudaMalloc(tile order)");
  cudaError_t e = cudaMemcpy(dev, host.data(), host.size() * sizeof(uint32_t), cudaMemcpyHostToDevice);
  if (e != cudaSuccess) {
    cudaFree(dev);
    return cuda_fail(e, "cudaMemcpy(tile order)");
  }
  OrderTable t;
  std::memcpy(t.key, key, sizeof(key));
  t.dev = dev;
  t.count = (int64_t)host.size();
  t.parts = parts;
  p->orders.push_back(t);
  *out = dev;
  return GEMM_F16_OK;
}

const OrderTable* find_table(gemm_f16_plan_s* p, const int64_t (&key)[6]) {
  for (auto& t : p->orders)
    if (std::memcmp(t.key, key, sizeof(key)) == 0) return &t;
  return nullptr;
}

int get_pair_table(gemm_f16_plan_s* p, int M, int N, int kblocks, int split_k,
                   const uint32_t** out, int64_t* count, int* parts) {
  const int64_t key[6] = {1, M, N, p->max_pairs,
                          (int64_t)split_k | ((int64_t)kblocks << 32), p->tile_order};
  if (const OrderTable* t = find_table(p, key)) {
    *out = t->dev;
    *count = t->count;
    *parts = t->parts;
    return GEMM_F16_OK;
  }
  std::vector<uint32_t> host;
  build_pair_tiles(M, N, kblocks, p->max_pairs, split_k, p->tile_order, host, parts);
  for (uint32_t& e : host)  // the kernel's entry format: narrow flag in bit 31
    e = pair::pack(ptile_tpm(e), ptile_n128(e), ptile_width(e) == pair::NARROW);
  *count = (int64_t)host.size();
  return upload_table(p, key, host, out, *parts);
}

// The cluster-of-four kernel's tile order (256 x 512 cluster tiles, packed
// pack_tile(tm, tn)), built and uploaded on first use.
int get_quad_table(gemm_f16_plan_s* p, int tiles_m, int tiles_n, const uint32_t** out) {
  const int64_t key[6] = {2, tiles_m, tiles_n, 0, 0, p->tile_order};
  if (const OrderTable* t = find_table(p, key)) {
    *out = t->dev;
    return GEMM_F16_OK;
  }
  std::vector<uint32_t> host;
  build_tile_order(tiles_m, tiles_n, p->tile_order, host);
  return upload_table(p, key, host, out);
}

// Tile width of the single-CTA kernel: 256, 128 or 64 columns.  Estimated
// time = waves x (k-blocks per unit x cycles per k-block + fixed cost per
// tile), with cycles per k-block max(W/2, 32 + W/4) for a 128 x W x 64
// k-block (tensor-core time vs. shared-memory operand reads) and ~2000
// cycles of pipeline fill and epilogue per tile.  Narrow tiles win when
// wide ones leave SMs idle.
int pick_tile_width(int M, int N, int kblocks, int split_k, int num_sms) {
  const int64_t kb_unit = ceil_div(kblocks, split_k);
  int best = BN;
  int64_t best_cost = -1;
  for (int w : {256, 128, 64}) {
    if (ceil_div(N, w) > 65535) continue;
    const int64_t units = ceil_div(M, BM) * ceil_div(N, w) * split_k;
    const int64_t waves = ceil_div(units, std::max(num_sms, 1));
    const int64_t per_kb = std::max<int64_t>(w / 2, 32 + w / 4);
    const int64_t cost = waves * (kb_unit * per_kb + 2000);
    if (best_cost < 0 || cost < best_cost) {
      best = w;
      best_cost = cost;
    }
  }
  return best;
}

// Kernel instance for a layout (template parameter 0..3).
template <typename F0, typename F1, typename F2, typename F3>
inline void* pick_instance(int layout, F0 f0, F1 f1, F2 f2, F3 f3) {
  switch (layout) {
    case 1: return (void*)f1;
    case 2: return (void*)f2;
    case 3: return (void*)f3;
    default: return (void*)f0;
  }
}

// What a run of this shape does with the plan's current options: which
// kernel, the single-CTA tile width, and whether A is repacked first.
struct RunChoice {
  bool use_quad;  // cluster-of-four kernel (two CTA pairs sharing A)
  bool use_pair;  // CTA-pair kernel (else single-CTA kernel; also set with use_quad)
  int bn;         // single-CTA tile width: 256, 128 or 64
  bool pack_a;    // A copied to whole-line rows before the product
};

RunChoice choose_run(const gemm_f16_plan_s* p, int layout, int M, int N, int K, int64_t lda,
                     int split_k) {
  RunChoice c;
  const int kblocks = (int)ceil_div(K, BK);
  c.bn = (p->tile_width != 0 && ceil_div(N, p->tile_width) <= 65535)
             ? p->tile_width
             : pick_tile_width(M, N, kblocks, split_k, p->num_sms);
  // Automatic choice: the pair kernel once its 256 x 256 tiles (times the
  // splits) fill at least half a wave of pairs; below that the single-CTA
  // kernel's smaller tiles spread the work over more SMs.
  const bool pair_fits = (N + 127) / 128 < 0x3FFF && p->max_pairs > 0;
  const int64_t pair_work = ceil_div(M, 256) * ceil_div(N, 256) * (int64_t)split_k;
  c.use_pair = pair_fits && (p->kernel == 2 || p->kernel == 3 ||
                             (p->kernel == 0 && M > BM && 2 * pair_work >= p->max_pairs));
  // A whose row pitch is not a multiple of 128 bytes: every 128-byte row of
  // an A copy box spans two cache lines.  On large products the automatic
  // choice either runs the cluster-of-four kernel, which fetches half as
  // many A rows per SM (so half the extra lines), or copies A to rows of
  // whole lines first (see pack_rows_kernel) for the pair kernel.  Measured
  // at 4000 x 4104 x 3000 (lda 3000): clusters of four without the copy
  // 68-71 us, the pair kernel after the copy 77 us, clusters of four after
  // the copy 75-77 us.  Clusters of four are taken when their waves (36
  // clusters of 256 x 512 tiles on 152 SMs) are no more than the pair
  // kernel's.
  const int64_t a_elems = (int64_t)M * K;
  const bool a_off_lines = (lda * 2) % 128 != 0;
  const bool large = N >= 2048 && a_elems >= ((int64_t)1 << 22);
  const bool quad_fits = c.use_pair && layout == 0 && p->max_quads > 0 &&
                         ceil_div(N, quad::QN) <= 0xFFFF && ceil_div(M, pair::PM) <= 0xFFFF;
  const int64_t quad_waves =
      ceil_div(ceil_div(M, pair::PM) * ceil_div(N, quad::QN) * (int64_t)split_k,
               std::max(p->max_quads, 1));
  const int64_t pair_waves = ceil_div(pair_work, std::max(p->max_pairs, 1));
  c.use_quad = quad_fits && (p->kernel == 3 || (p->kernel == 0 && a_off_lines && large &&
                                                p->a_repack != 2 && quad_waves <= pair_waves));
  c.pack_a = a_off_lines && (p->a_repack == 2 ||
                             (p->a_repack == 0 && c.use_pair && !c.use_quad && large));
  return c;
}

int run_device(gemm_f16_plan_s* p, int layout, int M, int N, int K, const void* A, int64_t lda,
               const void* B, int64_t ldb, void* C, int64_t ldc, int split_k,
               cudaStream_t stream) {
  const RunChoice choice = choose_run(p, layout, M, N, K, lda, split_k);
  const int tiles_m = (int)ceil_div(M, BM);
  const int kblocks = (int)ceil_div(K, BK);
  const int bn = choice.bn;
  const int tiles_n = (int)ceil_div(N, bn);
  const int64_t units = (int64_t)tiles_m * tiles_n * split_k;
  if (units > 0x7fffffff) return GEMM_F16_ERR_INVALID_ARG;
  const bool use_pair = choice.use_pair;
  const bool use_quad = choice.use_quad;
  const int quad_tm = (int)ceil_div(M, pair::PM), quad_tn = (int)ceil_div(N, quad::QN);
  const uint32_t* order = nullptr;
  int64_t pair_tiles = 0;
  int tail_parts = 1;
  int rc = GEMM_F16_OK;
  if (use_quad) {
    rc = get_quad_table(p, quad_tm, quad_tn, &order);
    if (rc) return rc;
  } else if (use_pair) {
    rc = get_pair_table(p, M, N, kblocks, split_k, &order, &pair_tiles, &tail_parts);
    if (rc) return rc;
  }

  const int64_t a_rows = (layout & LAYOUT_AT) ? K : M, a_cols = (layout & LAYOUT_AT) ? M : K;
  if (choice.pack_a) {
    const int64_t ldp = (a_cols + 63) / 64 * 64;
    rc = ensure_buffer(&p->apack, &p->apack_bytes, (size_t)(a_rows * ldp * 2), stream,
                       "A repack allocation");
    if (rc) return rc;
    const int64_t total = a_rows * ((a_cols + 7) / 8);
    const int pgrid = (int)std::max<int64_t>(
        1, std::min<int64_t>(ceil_div(total, 256 * 4), (int64_t)p->num_sms * 8));
    pack_rows_kernel<<<pgrid, 256, 0, stream>>>(static_cast<const __half*>(A), lda,
                                                static_cast<__half*>(p->apack), ldp, a_rows,
                                                a_cols);
    GF16_CUDA(cudaGetLastError(), "launch pack_rows_kernel");
    A = p->apack;
    lda = ldp;
  }

  alignas(64) CUtensorMap tmA, tmB, tmC, tmW;
  std::memset(&tmW, 0, sizeof(tmW));
  // A: row-major M x K -> boxes of 64 K x 128 rows; stored K x M -> boxes
  // of 64 M x 64 K (two per tile).  B: row-major K x N -> boxes of 64 N x
  // 64 K; stored N x K -> one box of 64 K x the tile's (or, in the pair
  // kernel, the CTA's) columns.
  if (layout & LAYOUT_AT)
    rc = cached_encode_2d(p, &tmA, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, A, (uint64_t)M, (uint64_t)K,
                          (uint64_t)lda * 2, 64, BK, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
  else
    rc = cached_encode_2d(p, &tmA, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, A, (uint64_t)K, (uint64_t)M,
                          (uint64_t)lda * 2, BK, use_quad ? BM / 2 : BM,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
  if (rc) return rc;
  const bool b3d = use_pair && !(layout & LAYOUT_BT) && (N % 64) == 0;
  if (layout & LAYOUT_BT)
    rc = cached_encode_2d(p, &tmB, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, B, (uint64_t)K, (uint64_t)N,
                          (uint64_t)ldb * 2, BK, use_pair ? 128u : (uint32_t)bn,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
  else if (b3d)
    rc = cached_encode_b3d(p, &tmB, B, (uint64_t)K, (uint64_t)N, (uint64_t)ldb);
  else
    rc = cached_encode_2d(p, &tmB, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, B, (uint64_t)N, (uint64_t)K,
                          (uint64_t)ldb * 2, B_BOX_N, BK, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
  if (rc) return rc;
  rc = cached_encode_2d(p, &tmC, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, C, (uint64_t)N, (uint64_t)M,
                 (uint64_t)ldc * 2, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B,
                 CU_TENSOR_MAP_L2_PROMOTION_NONE);
  if (rc) return rc;

  const int64_t ldw = (N + 7) / 8 * 8;
  const int64_t split_stride = (int64_t)M * ldw;
  if (split_k > 1) {
    const size_t bytes = (size_t)split_k * (size_t)split_stride * sizeof(float);
    rc = ensure_buffer(&p->ws, &p->ws_bytes, bytes, stream, "workspace allocation");
    if (rc) return rc;
    rc = encode_3d_f32(&tmW, p->ws, (uint64_t)N, (uint64_t)M, (uint64_t)split_k,
                       (uint64_t)ldw * 4, (uint64_t)split_stride * 4);
    if (rc) return rc;
  }

  if (use_quad) {
    const int64_t qunits = (int64_t)quad_tm * quad_tn * split_k;
    if (qunits > 0x7fffffff) return GEMM_F16_ERR_INVALID_ARG;
    pair::Params pp;
    pp.M = M;
    pp.N = N;
    pp.K = K;
    pp.split_k = split_k;
    pp.kblocks = kblocks;
    pp.num_units = (int)qunits;
    pp.order = order;
    pp.C = static_cast<__half*>(C);
    pp.ldc = ldc;
    pp.status = p->status_dev;
    pp.timeout_ns = p->timeout_ns;
    pp.fault_unit = p->fault_unit;
    pp.b3d = b3d ? 1 : 0;
    pp.full_units = (int)qunits;
    pp.tail_parts = 1;
    int64_t cap = std::max(p->max_quads, 1);
    if (p->sm_limit > 0) cap = std::max<int64_t>(1, std::min<int64_t>(cap, p->sm_limit / 4));
    const int64_t nquads = std::min<int64_t>(qunits, cap);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(4 * nquads), 1, 1);
    cfg.blockDim = dim3(quad::NUM_THREADS, 1, 1);
    cfg.dynamicSmemBytes = quad::SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute pdl;
    pdl.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &pdl;
    cfg.numAttrs = 1;
    void* args[] = {(void*)&tmA, (void*)&tmB, (void*)&tmC, (void*)&tmW, (void*)&pp};
    cudaEvent_t t0;
    if ((rc = timing_begin(p, stream, &t0))) return rc;
    const cudaError_t le = cudaLaunchKernelExC(&cfg, (void*)quad::gemm_f16_quad_kernel, args);
    rc = timing_end(p, stream, t0, le == cudaSuccess);
    GF16_CUDA(le, "launch gemm_f16_quad_kernel");
    if (rc) return rc;
  } else if (use_pair) {
    int64_t pair_cap = std::max(p->max_pairs, 1);
    if (p->sm_limit > 0) pair_cap = std::max<int64_t>(1, std::min<int64_t>(pair_cap, p->sm_limit / 2));
    // The last (pair_tiles % pairs) tiles run as two K halves each (one
    // split, 256-wide tiles; see tail_parts_for), planned for all pairs.
    const int64_t tail_tiles = tail_parts > 1 ? pair_tiles % std::max(p->max_pairs, 1) : 0;
    const int64_t full_units = (pair_tiles - tail_tiles) * split_k;
    const int64_t punits = full_units + tail_tiles * tail_parts;
    if (punits > 0x7fffffff) return GEMM_F16_ERR_INVALID_ARG;
    pair::Params pp;
    pp.full_units = (int)full_units;
    pp.tail_parts = tail_tiles > 0 ? tail_parts : 1;
    if (tail_tiles > 0) {
      // [2 t + q][256][256] FP32 values of the halves; tmW maps it instead
      // of the split workspace (one split, so that is unused).
      const int64_t planes = tail_tiles * 2;
      rc = ensure_buffer(&p->tail_ws, &p->tail_ws_bytes, (size_t)planes * 256 * 256 * sizeof(float),
                         stream, "tail partial allocation");
      if (rc) return rc;
      rc = encode_3d_f32(&tmW, p->tail_ws, 256, 256, (uint64_t)planes, 256 * sizeof(float),
                         256 * 256 * sizeof(float));
      if (rc) return rc;
    }
    pp.M = M;
    pp.N = N;
    pp.K = K;
    pp.split_k = split_k;
    pp.kblocks = kblocks;
    pp.num_units = (int)punits;
    pp.order = order;
    pp.C = static_cast<__half*>(C);
    pp.ldc = ldc;
    pp.status = p->status_dev;
    pp.timeout_ns = p->timeout_ns;
    pp.fault_unit = p->fault_unit;
    pp.b3d = b3d ? 1 : 0;
    const int64_t npairs = std::min<int64_t>(punits, pair_cap);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(2 * npairs), 1, 1);
    cfg.blockDim = dim3(pair::NUM_THREADS, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute pdl;
    pdl.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &pdl;
    cfg.numAttrs = 1;
    cfg.dynamicSmemBytes = pair::SMEM_BYTES;
    void* fn = pick_instance(layout, pair::gemm_f16_pair_kernel<0>, pair::gemm_f16_pair_kernel<1>,
                             pair::gemm_f16_pair_kernel<2>, pair::gemm_f16_pair_kernel<3>);
    void* args[] = {(void*)&tmA, (void*)&tmB, (void*)&tmC, (void*)&tmW, (void*)&pp};
    cudaEvent_t t0;
    if ((rc = timing_begin(p, stream, &t0))) return rc;
    const cudaError_t le = cudaLaunchKernelExC(&cfg, fn, args);
    rc = timing_end(p, stream, t0, le == cudaSuccess);
    GF16_CUDA(le, "launch gemm_f16_pair_kernel");
    if (rc) return rc;
    if (tail_tiles > 0) {
      // P0 + P1 of each tail tile into C (a programmatic dependent launch).
      const int64_t groups = tail_tiles * 256 * 64;
      cudaLaunchConfig_t tcfg = {};
      tcfg.gridDim = dim3((unsigned)std::min<int64_t>(ceil_div(groups, 256), (int64_t)p->num_sms * 8),
                          1, 1);
      tcfg.blockDim = dim3(256, 1, 1);
      tcfg.stream = stream;
      tcfg.attrs = &pdl;
      tcfg.numAttrs = 1;
      GF16_CUDA(cudaLaunchKernelEx(&tcfg, tail_reduce_kernel, (const float*)p->tail_ws,
                                   order + full_units, (int)tail_tiles, M, N,
                                   static_cast<__half*>(C), (int64_t)ldc),
                "launch tail_reduce_kernel");
    }
  } else {
  Params prm;
  prm.M = M;
  prm.N = N;
  prm.K = K;
  prm.bn = bn;
  prm.stages = stages_for(bn);
  prm.stage_bytes = A_STAGE + (uint32_t)bn * BK * 2;
  prm.tiles_m = tiles_m;
  prm.tiles_n = tiles_n;
  prm.split_k = split_k;
  prm.kblocks = kblocks;
  prm.num_units = (int)units;
  prm.row_major = p->tile_order;
  prm.C = static_cast<__half*>(C);
  prm.ldc = ldc;
  prm.status = p->status_dev;
  prm.timeout_ns = p->timeout_ns;
  prm.fault_unit = p->fault_unit;

  const int sm_cap = p->sm_limit > 0 ? std::min(p->sm_limit, p->num_sms) : p->num_sms;
  const int grid = (int)std::min<int64_t>(units, sm_cap);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(NUM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute pdl;
  pdl.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &pdl;
  cfg.numAttrs = 1;
  {
    void* fn = pick_instance(layout, gemm_f16_kernel<0>, gemm_f16_kernel<1>, gemm_f16_kernel<2>,
                             gemm_f16_kernel<3>);
    void* args[] = {(void*)&tmA, (void*)&tmB, (void*)&tmC, (void*)&tmW, (void*)&prm};
    cudaEvent_t t0;
    if ((rc = timing_begin(p, stream, &t0))) return rc;
    const cudaError_t le = cudaLaunchKernelExC(&cfg, fn, args);
    rc = timing_end(p, stream, t0, le == cudaSuccess);
    GF16_CUDA(le, "launch gemm_f16_kernel");
    if (rc) return rc;
  }
  }

  if (split_k > 1) {
    const int64_t groups = (int64_t)M * ((N + 3) / 4);
    const int rgrid = (int)std::min<int64_t>(ceil_div(groups, 256), (int64_t)p->num_sms * 8);
    cudaLaunchConfig_t rcfg = {};
    rcfg.gridDim = dim3(rgrid, 1, 1);
    rcfg.blockDim = dim3(256, 1, 1);
    rcfg.stream = stream;
    cudaLaunchAttribute pdl;
    pdl.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl.val.programmaticStreamSerializationAllowed = 1;
    rcfg.attrs = &pdl;
    rcfg.numAttrs = 1;
    GF16_CUDA(cudaLaunchKernelEx(&rcfg, splitk_reduce_kernel, (const float*)p->ws, M, N, ldw,
                                 split_k, split_stride, (__half*)C, (int64_t)ldc),
              "launch splitk_reduce_kernel");
  }
  return GEMM_F16_OK;
}

// What a run of these sizes would enqueue with the plan's options and
// device facts (gemm_f16_run_info, gemm_f16_run_choice).
int run_info_impl(const gemm_f16_plan_s* p, int layout, int M, int N, int K, int64_t lda,
                  int split_k, int info[4]) {
  if (!info || M <= 0 || N <= 0 || K <= 0 || split_k < 1 || layout < 0 || layout > 3 ||
      lda < ((layout & LAYOUT_AT) ? M : K))
    return GEMM_F16_ERR_INVALID_ARG;
  const RunChoice c = choose_run(p, layout, M, N, K, lda, split_k);
  // a partial last wave of 256-wide pair tiles in K halves adds their merge
  int parts = 1;
  if (c.use_pair && !c.use_quad && split_k == 1) {
    std::vector<uint32_t> tiles;
    build_pair_tiles(M, N, (int)ceil_div(K, BK), p->max_pairs, split_k, p->tile_order, tiles, &parts);
  }
  info[0] = c.use_quad ? 3 : c.use_pair ? 2 : 1;
  info[1] = 1 + (split_k > 1 ? 1 : 0) + (c.pack_a ? 1 : 0) + (parts > 1 ? 1 : 0);
  info[2] = c.pack_a ? 1 : 0;
  info[3] = c.use_pair ? pair::WIDE : c.bn;
  return GEMM_F16_OK;
}

}  // namespace

extern "C" {

int gemm_f16_run(gemm_f16_plan_t p, int M, int N, int K, const void* A, int64_t lda,
                 const void* B, int64_t ldb, void* C, int64_t ldc, int split_k,
                 gemm_f16_stream_t stream) {
  if (!p) return GEMM_F16_ERR_INVALID_ARG;
  int rc = gemm_f16_validate(M, N, K, A, lda, B, ldb, C, ldc, split_k);
  if (rc) return rc;
  DeviceGuard g(p->device);
  return run_device(p, 0, M, N, K, A, lda, B, ldb, C, ldc, split_k, (cudaStream_t)stream);
}

int gemm_f16_run_ex(gemm_f16_plan_t p, int layout, int M, int N, int K, const void* A,
                    int64_t lda, const void* B, int64_t ldb, void* C, int64_t ldc, int split_k,
                    gemm_f16_stream_t stream) {
  if (!p) return GEMM_F16_ERR_INVALID_ARG;
  int rc = gemm_f16_validate_ex(layout, M, N, K, A, lda, B, ldb, C, ldc, split_k);
  if (rc) return rc;
  DeviceGuard g(p->device);
  return run_device(p, layout, M, N, K, A, lda, B, ldb, C, ldc, split_k, (cudaStream_t)stream);
}

int gemm_f16_run_info(gemm_f16_plan_t p, int layout, int M, int N, int K, int64_t lda,
                      int split_k, int info[4]) {
  if (!p) return GEMM_F16_ERR_INVALID_ARG;
  return run_info_impl(p, layout, M, N, K, lda, split_k, info);
}

int gemm_f16_run_choice(int layout, int M, int N, int K, int64_t lda, int split_k, int num_sms,
                        int max_pairs, int max_quads, int info[4]) {
  if (num_sms < 1 || max_pairs < 0 || max_quads < 0 || 2 * max_pairs > num_sms ||
      4 * max_quads > num_sms)
    return GEMM_F16_ERR_INVALID_ARG;
  gemm_f16_plan_s facts;  // default options; only the device facts are set
  facts.num_sms = num_sms;
  facts.max_pairs = max_pairs;
  facts.max_quads = max_quads;
  return run_info_impl(&facts, layout, M, N, K, lda, split_k, info);
}

int gemm_f16_run_host(gemm_f16_plan_t p, int M, int N, int K, const void* hA, int64_t lda,
                      const void* hB, int64_t ldb, void* hC, int64_t ldc, int split_k,
                      gemm_f16_stream_t stream_) {
  if (!p) return GEMM_F16_ERR_INVALID_ARG;
  if (M <= 0 || N <= 0 || K <= 0 || !hA || !hB || !hC) return GEMM_F16_ERR_INVALID_ARG;
  if (lda < K || ldb < N || ldc < N) return GEMM_F16_ERR_INVALID_ARG;
  // Staging rows at the 16-byte minimum pitch: a contiguous host matrix then
  // moves in one plain copy (a pitched copy is several times slower); an A
  // whose pitch is then off 128-byte lines is repacked on the device.
  const int64_t dlda = (K + 7) / 8 * 8, dldb = (N + 7) / 8 * 8, dldc = dldb;
  int rc = gemm_f16_validate(M, N, K, (const void*)16, dlda, (const void*)16, dldb, (const void*)16,
                             dldc, split_k);
  if (rc) return rc;
  cudaStream_t stream = (cudaStream_t)stream_;
  DeviceGuard g(p->device);
  // The input-copy stream is shared with attn_f16_fwd_host; each entry point
  // creates its own events, each one once.
  if (!p->in_stream)
    GF16_CUDA(cudaStreamCreateWithFlags(&p->in_stream, cudaStreamNonBlocking),
              "create input-copy stream");
  for (int sl = 0; sl < 2; ++sl) {
    if (!p->in_done[sl])
      GF16_CUDA(cudaEventCreateWithFlags(&p->in_done[sl], cudaEventDisableTiming), "create event");
    if (!p->gemm_done[sl])
      GF16_CUDA(cudaEventCreateWithFlags(&p->gemm_done[sl], cudaEventDisableTiming),
                "create event");
  }
  const int slot = p->host_slot;
  p->host_slot ^= 1;
  void** buf = p->hbuf[slot];
  const size_t bytes[3] = {(size_t)M * dlda * 2, (size_t)K * dldb * 2, (size_t)M * dldc * 2};
  if (p->hcap[slot][0] < bytes[0] || p->hcap[slot][1] < bytes[1] || p->hcap[slot][2] < bytes[2]) {
    // Growing a slot: let everything that may still use it finish first.
    GF16_CUDA(cudaDeviceSynchronize(), "synchronise before growing run_host staging");
    for (int i = 0; i < 3; ++i) {
      if (p->hcap[slot][i] >= bytes[i]) continue;
      if (buf[i]) cudaFree(buf[i]);
      buf[i] = nullptr;
      p->hcap[slot][i] = 0;
      GF16_CUDA(cudaMalloc(&buf[i], bytes[i]), "run_host staging allocation");
      p->hcap[slot][i] = bytes[i];
    }
  }
  // Input copies on the plan's own stream, once the call that last used
  // this slot (two calls ago) has finished its product and its result copy;
  // the product on `stream` waits for them; the result copy follows the
  // product on `stream`.
  GF16_CUDA(cudaStreamWaitEvent(p->in_stream, p->gemm_done[slot], 0), "order input copies");
  GF16_CUDA(copy_rows(buf[0], dlda * 2, hA, lda * 2, (int64_t)K * 2, M, cudaMemcpyHostToDevice,
                      p->in_stream),
            "copy A to device");
  GF16_CUDA(copy_rows(buf[1], dldb * 2, hB, ldb * 2, (int64_t)N * 2, K, cudaMemcpyHostToDevice,
                      p->in_stream),
            "copy B to device");
  GF16_CUDA(cudaEventRecord(p->in_done[slot], p->in_stream), "record input copies");
  GF16_CUDA(cudaStreamWaitEvent(stream, p->in_done[slot], 0), "order product after inputs");
  rc = run_device(p, 0, M, N, K, buf[0], dlda, buf[1], dldb, buf[2], dldc, split_k, stream);
  if (rc) return rc;
  GF16_CUDA(copy_rows(hC, ldc * 2, buf[2], dldc * 2, (int64_t)N * 2, M, cudaMemcpyDeviceToHost,
                      stream),
            "copy C to host");
  // The slot is free again once C has left it, whatever stream the next
  // call that uses it runs on.
  GF16_CUDA(cudaEventRecord(p->gemm_done[slot], stream), "record product and result copy");
  return GEMM_F16_OK;
}

}  // extern "C"

// ====================================================== no-allocation entry
// gemm_f16_run_noalloc: the plan-free variant for callers that must not
// allocate device memory (see gemm_f16.h).  Its scratch is one file-scope
// device array, laid out as
//   [0, 256)              status word used when the caller passes none
//   [256, 256 + 32 MiB)   FP32 split partials [split][M][ldw]
// The kernel derives its tiles from the unit index (morton_tile_of_rank),
// so no tile table is kept between calls.  Host code must not use the
// array's name as an address: the per-device set-up below asks the runtime
// for its device address.
namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[GEMM_F16_NOALLOC_SCRATCH_BYTES];

constexpr size_t NOALLOC_STATUS_OFF = 0;
constexpr size_t NOALLOC_WS_OFF = 256;
static_assert(NOALLOC_WS_OFF + GEMM_F16_NOALLOC_WS_BYTES == GEMM_F16_NOALLOC_SCRATCH_BYTES,
              "scratch layout");

constexpr int NOALLOC_MAX_DEVICES = 64;
struct NoallocDevice {
  bool ready = false;
  unsigned char* scratch = nullptr;  // device address of g_noalloc_scratch on this device
  int num_sms = 0;
};
NoallocDevice g_noalloc_devices[NOALLOC_MAX_DEVICES];
std::mutex g_noalloc_mutex;

// One-time set-up on the current device `dev` (that device is current).
int noalloc_setup(int dev, NoallocDevice* d) {
  int major = 0, minor = 0, sms = 0;
  GF16_CUDA(cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev),
            "cudaDeviceGetAttribute(major)");
  GF16_CUDA(cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev),
            "cudaDeviceGetAttribute(minor)");
  if (major != 10 || minor != 3) return GEMM_F16_ERR_UNSUPPORTED_DEVICE;
  GF16_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev),
            "cudaDeviceGetAttribute(SM count)");
  GF16_CUDA(cudaFuncSetAttribute(gemm_f16_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)SMEM_BYTES),
            "cudaFuncSetAttribute(max dynamic smem)");
  void* ptr = nullptr;
  GF16_CUDA(cudaGetSymbolAddress(&ptr, g_noalloc_scratch), "cudaGetSymbolAddress(scratch)");
  d->scratch = static_cast<unsigned char*>(ptr);
  d->num_sms = sms;
  d->ready = true;
  return GEMM_F16_OK;
}

// The current device's entry, set up on first use (mutex held by the caller).
int noalloc_device(NoallocDevice** out) {
  int dev = 0;
  GF16_CUDA(cudaGetDevice(&dev), "cudaGetDevice");
  if (dev < 0 || dev >= NOALLOC_MAX_DEVICES) return GEMM_F16_ERR_UNSUPPORTED_DEVICE;
  NoallocDevice* d = &g_noalloc_devices[dev];
  if (!d->ready) {
    const int rc = noalloc_setup(dev, d);
    if (rc) return rc;
  }
  *out = d;
  return GEMM_F16_OK;
}

}  // namespace

extern "C" int gemm_f16_run_noalloc(int M, int N, int K, const void* A, int64_t lda,
                                    const void* B, int64_t ldb, void* C, int64_t ldc,
                                    int split_k, int* status, gemm_f16_stream_t stream_) {
  int rc = gemm_f16_validate(M, N, K, A, lda, B, ldb, C, ldc, split_k);
  if (rc) return rc;
  const int tiles_m = (int)ceil_div(M, BM);
  const int tiles_n = (int)ceil_div(N, BN);
  const int64_t tiles = (int64_t)tiles_m * tiles_n;
  const int64_t ldw = (N + 7) / 8 * 8;
  const int64_t split_stride = (int64_t)M * ldw;
  if (split_k > 1 &&
      (uint64_t)split_k * (uint64_t)split_stride * sizeof(float) > GEMM_F16_NOALLOC_WS_BYTES)
    return GEMM_F16_ERR_SCRATCH_TOO_SMALL;
  const int64_t units = tiles * split_k;
  if (units > 0x7fffffff) return GEMM_F16_ERR_INVALID_ARG;
  cudaStream_t stream = (cudaStream_t)stream_;

  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  NoallocDevice* d = nullptr;
  rc = noalloc_device(&d);
  if (rc) return rc;

  alignas(64) CUtensorMap tmA, tmB, tmC, tmW;
  std::memset(&tmW, 0, sizeof(tmW));
  rc = encode_2d(&tmA, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, A, (uint64_t)K, (uint64_t)M,
                 (uint64_t)lda * 2, BK, BM, CU_TENSOR_MAP_SWIZZLE_128B,
                 CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
  if (rc) return rc;
  rc = encode_2d(&tmB, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, B, (uint64_t)N, (uint64_t)K,
                 (uint64_t)ldb * 2, B_BOX_N, BK, CU_TENSOR_MAP_SWIZZLE_128B,
                 CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
  if (rc) return rc;
  rc = encode_2d(&tmC, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, C, (uint64_t)N, (uint64_t)M,
                 (uint64_t)ldc * 2, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B,
                 CU_TENSOR_MAP_L2_PROMOTION_NONE);
  if (rc) return rc;
  float* ws = reinterpret_cast<float*>(d->scratch + NOALLOC_WS_OFF);
  if (split_k > 1) {
    rc = encode_3d_f32(&tmW, ws, (uint64_t)N, (uint64_t)M, (uint64_t)split_k, (uint64_t)ldw * 4,
                       (uint64_t)split_stride * 4);
    if (rc) return rc;
  }

  Params prm;
  prm.M = M;
  prm.N = N;
  prm.K = K;
  prm.bn = BN;
  prm.stages = stages_for(BN);
  prm.stage_bytes = A_STAGE + (uint32_t)BN * BK * 2;
  prm.tiles_m = tiles_m;
  prm.tiles_n = tiles_n;
  prm.split_k = split_k;
  prm.kblocks = (int)ceil_div(K, BK);
  prm.num_units = (int)units;
  prm.row_major = 0;
  prm.C = static_cast<__half*>(C);
  prm.ldc = ldc;
  prm.status = status ? status : reinterpret_cast<int*>(d->scratch + NOALLOC_STATUS_OFF);
  prm.timeout_ns = 1000000000ull;
  prm.fault_unit = -1;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)std::min<int64_t>(units, d->num_sms), 1, 1);
  cfg.blockDim = dim3(NUM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.stream = stream;
  GF16_CUDA(cudaLaunchKernelEx(&cfg, gemm_f16_kernel<0>, tmA, tmB, tmC, tmW, prm),
            "launch gemm_f16_kernel (no-alloc)");
  if (split_k > 1) {
    const int64_t groups = (int64_t)M * ((N + 3) / 4);
    cudaLaunchConfig_t rcfg = {};
    rcfg.gridDim = dim3((unsigned)std::min<int64_t>(ceil_div(groups, 256), (int64_t)d->num_sms * 8), 1, 1);
    rcfg.blockDim = dim3(256, 1, 1);
    rcfg.stream = stream;
    GF16_CUDA(cudaLaunchKernelEx(&rcfg, splitk_reduce_kernel, (const float*)ws, M, N, ldw, split_k,
                                 split_stride, (__half*)C, (int64_t)ldc),
              "launch splitk_reduce_kernel (no-alloc)");
  }
  return GEMM_F16_OK;
}

extern "C" int gemm_f16_noalloc_status(void) {
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  NoallocDevice* d = nullptr;
  int rc = noalloc_device(&d);
  if (rc) return rc;
  int v = 0;
  GF16_CUDA(cudaMemcpyFromSymbol(&v, g_noalloc_scratch, sizeof(int), NOALLOC_STATUS_OFF,
                                 cudaMemcpyDeviceToHost),
            "read no-alloc status word");
  if (v != 0) {
    const int zero = 0;
    GF16_CUDA(cudaMemcpyToSymbol(g_noalloc_scratch, &zero, sizeof(int), NOALLOC_STATUS_OFF,
                                 cudaMemcpyHostToDevice),
              "clear no-alloc status word");
  }
  return v;
}
