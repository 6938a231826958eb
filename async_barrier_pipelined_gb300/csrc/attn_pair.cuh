// CTA-pair variant of the attention forward kernel (tcgen05 cta_group::2),
// head dimension 256, blocks of 128 keys; persistent over work items.
//
// A work item is 256 query rows of one (batch, head).  A cluster of two CTAs
// takes items cluster, cluster + C, cluster + 2C, ... (C clusters, one per
// pair of SMs; query tiles vary fastest, so clusters running at the same
// time share a head's keys and values in L2).  For an item, CTA r holds rows
// 128r .. 128r+127 (its Q tile in shared memory, its rows of S, P and O in
// its tensor memory) and the even CTA ("leader") issues the MMAs for both:
//   S = Q K^T   256 x 128 x 16, 16 per key block; B (the key block) is split
//               by keys: CTA r holds keys 64r .. 64r+63 of the block.
//   O += P V    256 x 256 x 16, 8 per key block; A (P, FP16) is read from
//               each CTA's tensor memory, B (the value block) is split by
//               columns: CTA r holds d = 128r .. 128r+127.
// Each SM so takes in 32 KB of K and 32 KB of V per 128 keys -- half of
// what the single-CTA kernel needs for the same work -- and the S MMAs are
// 128 keys wide (a 64-wide S MMA runs at two thirds of the tensor rate).
// P never passes through shared memory: per block and CTA that saves 32 KB
// of softmax stores and 32 KB of MMA operand reads.
//
// Roles per CTA (320 threads): warp 0 copies (Q per item, then K and V
// halves through a 4-slot ring), warp 1 issues the MMAs (leader only),
// warps 2-5 run the softmax (one query row per thread), warps 6-9 write O.
// Per key block j the softmax loads S_j into registers and says so (s_free),
// which lets the leader issue S_{j+1} into the one S buffer while O += P V of
// block j-1 runs; it then writes P_j into one of two P buffers in tensor
// memory and publishes it (the split barrier's ARRIVE); the leader's MMA
// thread WAITs for both CTAs before O += P V.  Between items nothing drains:
// the producer reloads Q as soon as the item's last S MMA has read it, the
// leader issues the last O += P V of item k and then S_0 of item k+1, and
// while the softmax warps already work on item k+1 the epilogue warps read
// O of item k out of tensor memory (O += P V of item k+1's first block
// waits for that), scale it by 1/l and store it with tensor copies.
//
// Barriers ("mbarrier State and Operations" page):
//   q_full, full[s]  leader only: its producer's arrive.expect_tx for both
//                    CTAs' bytes; both CTAs' copies complete them.
//   q_empty          both: multicast commit after an item's last S MMA.
//   empty[s]         both: the leader's commit, multicast to the pair.
//   s_full           both: multicast commit when S is written.
//   s_free, p_full[b], o_free
//                    leader only: one arrival per leader softmax (epilogue)
//                    warp, each expecting 16 bytes; each peer warp signals
//                    with a 16-byte shared-memory copy into the leader that
//                    completes 16 bytes on it.  (A release arrival across
//                    the cluster took ~0.8 us; the copy lands in a fraction
//                    of that.)  s_free: S is in registers in both CTAs;
//                    p_full[b]: P buffer b is written in both CTAs; o_free:
//                    both CTAs' epilogue warps have read O.
//   o_done[b]        both: multicast commit when O += P V from P buffer b ends.
//   l_ready, l_free  per CTA: the softmax warps hand an item's row sums to
//                    the epilogue warps through shared memory.
//   mma_done         leader only: the last commit, waited before TMEM is freed.
// Phases count key blocks (and items) over the whole run of a cluster.
// Every wait is bounded; after an abort the leader completes the phases of
// copies in flight (as the pair GEMM kernel does) before either CTA exits.

#pragma once

namespace gf16 {
namespace attnp {

using attn::block_offset;
using attn::block_weights;
using attn::HD;
using attn::pack_half2;

constexpr int CQ = 128;                 // query rows per CTA
constexpr int PQ = 2 * CQ;              // query rows per pair (one work item)
constexpr int BKV = 128;                // keys per block
constexpr int RING = 4;                 // K / V half-tiles in flight per CTA
constexpr int SM_WARPS = 4;             // softmax warps 2..5
constexpr int EP_WARPS = 4;             // epilogue warps 6..9
constexpr int NUM_THREADS = 32 * (2 + SM_WARPS + EP_WARPS);

constexpr uint32_t CHUNK_Q = CQ * 128;                 // 64 d x 128 rows: 16 KB
constexpr uint32_t Q_BYTES = (HD / 64) * CHUNK_Q;      // 64 KB
constexpr uint32_t K_CHUNK = (BKV / 2) * 128;          // 64 d x 64 keys: 8 KB
constexpr uint32_t V_CHUNK = BKV * 128;                // 64 d x 128 keys: 16 KB
constexpr uint32_t SLOT_BYTES = 32768;                 // a K half (4 chunks) or a V half (2)
constexpr uint32_t O_BOX = 32 * 128;                   // 32 rows x 64 d of O: 4 KB
constexpr uint32_t OFF_Q = 0;
constexpr uint32_t OFF_RING = OFF_Q + Q_BYTES;
constexpr uint32_t OFF_STAGE = OFF_RING + RING * SLOT_BYTES;  // two O boxes per epilogue warp
constexpr uint32_t OFF_L = OFF_STAGE + EP_WARPS * 2 * O_BOX;  // row sums and offsets, softmax -> epilogue
constexpr uint32_t OFF_BAR = OFF_L + 2 * CQ * 4;
// q_full, q_empty, full[RING], empty[RING], s_full, s_free, p_full[2],
// o_done[2], o_free, l_ready, l_free, mma_done
constexpr uint32_t NUM_BARS = 2 + 2 * RING + 2 + 2 + 2 + 3 + 1;
constexpr uint32_t OFF_TMEM_SLOT = OFF_BAR + NUM_BARS * 8;
constexpr uint32_t OFF_ABORT = OFF_TMEM_SLOT + 4;
constexpr uint32_t OFF_PEER_FILLS = OFF_ABORT + 4;       // ring fills the peer issued
constexpr uint32_t OFF_PEER_QLOADS = OFF_PEER_FILLS + 4;  // Q tiles the peer issued
// Signalling copies, 16 bytes each: destinations in the leader (per
// signalling warp: p_full, s_free, o_free), then the sources read in the
// peer (one per softmax or epilogue warp).
constexpr uint32_t OFF_SIG = (OFF_PEER_QLOADS + 4 + 15) / 16 * 16;
constexpr uint32_t SIG_BYTES = 16;
constexpr uint32_t SIG_P = 0;
constexpr uint32_t SIG_S = SIG_P + SM_WARPS * SIG_BYTES;
constexpr uint32_t SIG_O = SIG_S + SM_WARPS * SIG_BYTES;
constexpr uint32_t SIG_SRC = SIG_O + EP_WARPS * SIG_BYTES;
constexpr uint32_t SMEM_BYTES = OFF_SIG + SIG_SRC + (SM_WARPS + EP_WARPS) * SIG_BYTES + 1024;
static_assert(SMEM_BYTES <= 232448, "over the 227 KB shared-memory limit per CTA");
static_assert(OFF_RING % 1024 == 0 && OFF_STAGE % 1024 == 0,
              "swizzled buffers need 1024-B alignment");
static_assert((HD / 64) * K_CHUNK == SLOT_BYTES && 2 * V_CHUNK == SLOT_BYTES, "slot sizes");

constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t S_COL = 0;     // S: columns 0 .. 127 (FP32)
constexpr uint32_t P_COL = 128;   // P buffers: columns 128 and 192, 64 each (FP16 pairs)
constexpr uint32_t O_COL = 256;   // O: columns 256 .. 511

// kind::f16, FP32 accumulate, M = 256 (the pair): S = Q K^T with both
// operands K-major; O += P V with P K-major (tensor memory) and V MN-major.
constexpr uint32_t IDESC_QK = (1u << 4) | ((uint32_t)(BKV >> 3) << 17) | ((uint32_t)(PQ >> 4) << 24);
constexpr uint32_t IDESC_PV =
    (1u << 4) | (1u << 16) | ((uint32_t)(HD >> 3) << 17) | ((uint32_t)(PQ >> 4) << 24);

struct Params {
  int seq_q, seq_kv;
  int nkv;                      // key blocks: ceil(seq_kv / 128)
  int n_qt;                     // query tiles of 256 rows: ceil(seq_q / 256)
  int heads;
  int n_items;                  // batch * heads * n_qt
  int n_split;                  // key ranges per item (1: O is written directly)
  int bps;                      // key blocks per range (the last range may have fewer)
  int n_units;                  // n_items * n_split
  float* part_ml;               // n_split > 1: per unit and row, the offset m and the sum l
  float scale_log2;
  int* status;
  unsigned long long timeout_ns;
  int fault_unit;               // test only: unit whose first ring fill gets no leader copy
};

struct Bars {
  uint32_t q_full, q_empty, full, empty, s_full, s_free, p_full, o_done, o_free, l_ready, l_free,
      mma_done;
};

// Work unit -> first query row, head, batch (query tiles vary fastest) and
// the unit's key blocks j0 .. j0 + nb - 1 (a unit is one key range of an
// item; without a split, the whole item).
struct Item {
  int q0, h, bz, j0, nb;
};
__device__ __forceinline__ Item decode_unit(int u, const Params& p) {
  const int it = u / p.n_split;
  const int j0 = (u - it * p.n_split) * p.bps;
  const int bh = it / p.n_qt;
  const int nb = p.nkv - j0 < p.bps ? p.nkv - j0 : p.bps;
  return Item{(it - bh * p.n_qt) * PQ, bh % p.heads, bh / p.heads, j0, nb};
}

__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, const Params& p,
                                           volatile int* abort_flag) {
  if (ptx::mbar_try_wait_poll(bar, parity)) return true;
  return attn::wait_slow(bar, parity, p.status, p.timeout_ns, abort_flag);
}

// The same wait suspending in hardware between checks (copy and MMA threads).
__device__ __forceinline__ bool wait_phase_suspend(uint32_t bar, uint32_t parity, const Params& p,
                                                   volatile int* abort_flag) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  return attn::wait_slow<true>(bar, parity, p.status, p.timeout_ns, abort_flag);
}

// A wait that sleeps between polls (256 ns), for the epilogue warps, which
// wait most of an item for its row sums: polling at full rate would take
// issue slots from the softmax, MMA and copy warps on the same schedulers.
__device__ __noinline__ bool wait_sleepy(uint32_t bar, uint32_t parity, const Params& p,
                                         volatile int* abort_flag) {
  const uint64_t t0 = ptx::globaltimer();
  while (true) {
    if (ptx::mbar_try_wait_poll(bar, parity)) return true;
    if (*abort_flag) return false;
    if (ptx::globaltimer() - t0 > p.timeout_ns) {
      *abort_flag = 1;
      *(volatile int*)p.status = (int)GEMM_F16_ERR_TIMEOUT;
      __threadfence_system();
      return false;
    }
    __nanosleep(256);
  }
}

// The same wait taken by a whole warp; true only if every lane saw the phase.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const Params& p,
                                          volatile int* abort_flag) {
  const bool got = wait_phase(bar, parity, p, abort_flag);
  return __all_sync(0xffffffffu, got);
}

// One arrival per warp on a leader barrier: the leader's warps arrive
// expecting 16 bytes, the peer's send them with a signalling copy.
__device__ __forceinline__ void signal_leader(uint32_t rank, uint32_t lane, uint32_t local_bar,
                                              uint32_t leader_bar, uint32_t dst, uint32_t src) {
  ptx::tc_fence_before();
  __syncwarp();
  if (lane == 0) {
    if (rank == 0)
      ptx::mbar_arrive_expect_tx(local_bar, SIG_BYTES);
    else
      ptx::bulk_copy_to_cluster(dst, src, SIG_BYTES, leader_bar);
  }
}

// ------------------------------------------------------------------ producer
// Both CTAs, per item: this CTA's Q rows, then its halves of the K and V
// blocks in the order the MMA thread consumes them (K_0, then per block j:
// K_{j+1}, V_j), crediting the leader's barriers; the leader also arrives
// (expect_tx) for the pair.  Q of the next item waits for q_empty.
struct Issued {
  uint32_t fills, qloads;
};
__device__ __forceinline__ Issued producer_role(const CUtensorMap* tmQ, const CUtensorMap* tmK,
                                                const CUtensorMap* tmV, const Params& p,
                                                uint32_t base, const Bars& b, uint32_t rank,
                                                int cluster, int nclusters,
                                                volatile int* abort_flag) {
  const uint32_t leader_q = ptx::map_to_cta(b.q_full, 0);
  const uint32_t leader_full = ptx::map_to_cta(b.full, 0);
  RingPos pos{0, 0};
  Issued n{0, 0};
  bool ok = true;
  for (int u = cluster; u < p.n_units && ok; u += nclusters) {
    const Item w = decode_unit(u, p);
    if (n.qloads > 0 && !wait_phase_suspend(b.q_empty, (n.qloads - 1) & 1u, p, abort_flag)) break;
    if (rank == 0) ptx::mbar_arrive_expect_tx_relaxed(b.q_full, 2 * Q_BYTES);
#pragma unroll
    for (int c = 0; c < HD / 64; ++c)
      ptx::tma_load_4d_pair(base + OFF_Q + c * CHUNK_Q, tmQ, leader_q, 64 * c,
                            w.q0 + (int)rank * CQ, w.h, w.bz);
    ++n.qloads;
    bool first = true;
    auto fill = [&](bool is_k, int j) -> bool {
      if (!wait_phase_suspend(b.empty + 8 * pos.stage, producer_wait_parity(pos), p, abort_flag))
        return false;
      if (rank == 0) ptx::mbar_arrive_expect_tx_relaxed(b.full + 8 * pos.stage, 2 * SLOT_BYTES);
      if (!(first && u == p.fault_unit && rank == 0)) {
        const uint32_t dst = base + OFF_RING + pos.stage * SLOT_BYTES;
        const uint32_t fb = leader_full + 8 * pos.stage;
        if (is_k) {
#pragma unroll
          for (int c = 0; c < HD / 64; ++c)
            ptx::tma_load_4d_pair(dst + c * K_CHUNK, tmK, fb, 64 * c,
                                  (w.j0 + j) * BKV + (int)rank * (BKV / 2), w.h, w.bz);
        } else {
#pragma unroll
          for (int c = 0; c < 2; ++c)
            ptx::tma_load_4d_pair(dst + c * V_CHUNK, tmV, fb, (int)rank * 128 + 64 * c,
                                  (w.j0 + j) * BKV, w.h, w.bz);
        }
      }
      first = false;
      ++n.fills;
      ring_advance(pos, RING);
      return true;
    };
    ok = fill(true, 0);
    for (int j = 0; j < w.nb && ok; ++j) {
      if (j + 1 < w.nb) ok = fill(true, j + 1);
      if (ok) ok = fill(false, j);
    }
  }
  return n;
}

// ------------------------------------------------------------------ MMA issuer (leader)
__device__ __forceinline__ void mma_role(const Params& p, uint32_t base, uint32_t tmem_base,
                                         const Bars& b, int cluster, int nclusters,
                                         volatile int* abort_flag) {
  RingPos pos{0, 0};
  const uint32_t q_addr = base + OFF_Q;
  const uint32_t o_tmem = tmem_base + O_COL;

  // S of global block gs into the S buffer, once both CTAs hold S of block
  // gs - 1 in registers; after an item's last S, q_empty hands Q back.
  auto issue_qk = [&](uint32_t gs, bool last_of_item) -> bool {
    if (gs > 0) {
      if (!wait_phase_suspend(b.s_free, (gs - 1) & 1u, p, abort_flag)) return false;
    }
    if (!wait_phase_suspend(b.full + 8 * pos.stage, consumer_wait_parity(pos), p, abort_flag))
      return false;
    ptx::tc_fence_after();
    const uint32_t k_addr = base + OFF_RING + pos.stage * SLOT_BYTES;
#pragma unroll
    for (int kk = 0; kk < HD / 16; ++kk) {
      const uint32_t off_q = (uint32_t)(kk >> 2) * CHUNK_Q + (uint32_t)(kk & 3) * 32u;
      const uint32_t off_k = (uint32_t)(kk >> 2) * K_CHUNK + (uint32_t)(kk & 3) * 32u;
      ptx::mma_f16_pair(tmem_base + S_COL, smem_desc_sw128(q_addr + off_q, 16, 1024),
                        smem_desc_sw128(k_addr + off_k, 16, 1024), IDESC_QK, kk > 0 ? 1u : 0u);
    }
    ptx::mma_commit_pair(b.empty + 8 * pos.stage, 0x3);
    ptx::mma_commit_pair(b.s_full, 0x3);
    if (last_of_item) ptx::mma_commit_pair(b.q_empty, 0x3);
    ring_advance(pos, RING);
    return true;
  };

  uint32_t g0 = 0;   // global index of the unit's first key block
  uint32_t ki = 0;   // units done
  bool ok = true;
  for (int u = cluster; u < p.n_units && ok; u += nclusters, ++ki) {
    const int nb = decode_unit(u, p).nb;
    if (!wait_phase_suspend(b.q_full, ki & 1u, p, abort_flag)) break;
    ptx::tc_fence_after();
    ok = issue_qk(g0, nb == 1);
    for (int j = 0; j < nb && ok; ++j) {
      const uint32_t gj = g0 + (uint32_t)j;
      if (j + 1 < nb && !issue_qk(gj + 1, j + 2 == nb)) {
        ok = false;
        break;
      }
      // The split barrier's WAIT: both CTAs' P rows are in tensor memory.
      const uint32_t pb = gj & 1u;
      if (!wait_phase_suspend(b.p_full + 8 * pb, (gj >> 1) & 1u, p, abort_flag) ||
          !wait_phase_suspend(b.full + 8 * pos.stage, consumer_wait_parity(pos), p, abort_flag)) {
        ok = false;
        break;
      }
      // The unit's first O += P V overwrites O: both CTAs' epilogue warps
      // must have read the previous unit's O.
      if (j == 0 && ki > 0 && !wait_phase_suspend(b.o_free, (ki - 1) & 1u, p, abort_flag)) {
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      const uint32_t v_addr = base + OFF_RING + pos.stage * SLOT_BYTES;
      const uint32_t p_tmem = tmem_base + P_COL + pb * (BKV / 2);
#pragma unroll
      for (int kk = 0; kk < BKV / 16; ++kk)   // 16 keys = 8 columns of P per MMA
        ptx::mma_f16_pair_tmem_a(o_tmem, p_tmem + (uint32_t)kk * 8u,
                                 smem_desc_sw128(v_addr + (uint32_t)kk * 2048u, V_CHUNK, 1024),
                                 IDESC_PV, (j > 0 || kk > 0) ? 1u : 0u);
      ptx::mma_commit_pair(b.empty + 8 * pos.stage, 0x3);
      ptx::mma_commit_pair(b.o_done + 8 * pb, 0x3);
      ring_advance(pos, RING);
    }
    g0 += (uint32_t)nb;
  }
}

// ------------------------------------------------------------------ softmax
__device__ __forceinline__ void softmax_role(const Params& p, uint32_t base, uint32_t tmem_base,
                                             const Bars& b, float* l_rows, uint32_t rank,
                                             uint32_t warp, uint32_t lane, int cluster,
                                             int nclusters, volatile int* abort_flag) {
  const uint32_t quarter = warp & 3u;
  const uint32_t t_lane = (quarter * 32u) << 16;
  const uint32_t leader_p_full = ptx::map_to_cta(b.p_full, 0);
  const uint32_t leader_s_free = ptx::map_to_cta(b.s_free, 0);
  const uint32_t sig_p = ptx::map_to_cta(base + OFF_SIG + SIG_P + (warp - 2) * SIG_BYTES, 0);
  const uint32_t sig_s = ptx::map_to_cta(base + OFF_SIG + SIG_S + (warp - 2) * SIG_BYTES, 0);
  const uint32_t sig_src = base + OFF_SIG + SIG_SRC + (warp - 2) * SIG_BYTES;
  const float sl2 = p.scale_log2;
  uint32_t g = 0;    // global key block
  uint32_t ki = 0;   // units done
  bool ok = true;
  for (int u = cluster; u < p.n_units && ok; u += nclusters, ++ki) {
    const bool more_units = u + nclusters < p.n_units;
    const Item w = decode_unit(u, p);
    float m = -INFINITY;
    float l = 0.f;
    for (int j = 0; j < w.nb; ++j, ++g) {
      if (!warp_wait(b.s_full, g & 1u, p, abort_flag)) {
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      uint32_t s[BKV];
#pragma unroll
      for (int c = 0; c < BKV / 32; ++c)
        ptx::tmem_ld_32x32b_x32(tmem_base + t_lane + S_COL + 32u * c,
                                *reinterpret_cast<uint32_t(*)[32]>(&s[32 * c]));
      ptx::tmem_ld_wait();
      ptx::reg_fence(s);
      // S is in registers: the next S may overwrite it.
      if (j + 1 < w.nb || more_units)
        signal_leader(rank, lane, b.s_free, leader_s_free, sig_s, sig_src);
      const int valid = p.seq_kv - (w.j0 + j) * BKV;
      float alpha;
      const float m_new = block_offset<BKV>(s, sl2, valid, m, &alpha);
      uint32_t pk[BKV / 2];
      const float lsum = valid < BKV ? block_weights<BKV, true>(s, sl2, -m_new, valid, pk)
                                     : block_weights<BKV, false>(s, sl2, -m_new, valid, pk);
      const uint32_t pb = g & 1u;
      if (g >= 2) {
        // P buffer pb was last read by O += P V of global block g-2.
        if (!warp_wait(b.o_done + 8 * pb, ((g - 2) >> 1) & 1u, p, abort_flag)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
      }
      // P row -> tensor memory: column c of the buffer holds keys 2c, 2c+1.
      const uint32_t p_tmem = tmem_base + t_lane + P_COL + pb * (BKV / 2);
      ptx::tmem_st_32x32b_x32(p_tmem, *reinterpret_cast<const uint32_t(*)[32]>(&pk[0]));
      ptx::tmem_st_32x32b_x32(p_tmem + 32u, *reinterpret_cast<const uint32_t(*)[32]>(&pk[32]));
      if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
        // Compensation: O *= alpha once O += P V of the item's previous
        // block has landed.
        const uint32_t ob = (g - 1) & 1u;
        if (!warp_wait(b.o_done + 8 * ob, ((g - 1) >> 1) & 1u, p, abort_flag)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < HD / 32; ++c) {
          uint32_t o[32];
          const uint32_t ta = tmem_base + t_lane + O_COL + (uint32_t)c * 32u;
          ptx::tmem_ld_32x32b_x32(ta, o);
          ptx::tmem_ld_wait();
          ptx::reg_fence(o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
          ptx::tmem_st_32x32b_x32(ta, o);
        }
      }
      ptx::tmem_st_wait();
      // The split barrier's ARRIVE (one per warp, on the leader's barrier) ...
      signal_leader(rank, lane, b.p_full + 8 * pb, leader_p_full + 8 * pb, sig_p, sig_src);
      // ... and the window: the deferred sum update.
      l = l * alpha + lsum;
      m = m_new;
    }
    if (!ok) break;
    // Hand the row's sum and offset to the epilogue warps (once they took
    // the last ones).
    if (ki > 0 && !warp_wait(b.l_free, (ki - 1) & 1u, p, abort_flag)) break;
    l_rows[quarter * 32u + lane] = l;
    l_rows[CQ + quarter * 32u + lane] = m;
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(b.l_ready);
  }
}

// ------------------------------------------------------------------ epilogue
// Per unit, once its last O += P V has landed: O (FP32, tensor memory) * 1/l.
// Without a key split -> FP16, staged per warp in two 32-row x 64-column
// boxes (128-byte swizzle) and stored into O with tensor copies.  With a
// split -> FP32 partial, staged in 32-row x 32-column boxes and stored into
// the workspace (row u * 256 + r of the partial tensor), with the row's
// offset m and sum l beside it; the combine kernel merges the ranges.
__device__ __forceinline__ void epilogue_role(const CUtensorMap* tmO, const CUtensorMap* tmP,
                                              const Params& p, uint32_t base, uint32_t tmem_base,
                                              const Bars& b, const float* l_rows, uint32_t rank,
                                              uint32_t warp, uint32_t lane, int cluster,
                                              int nclusters, volatile int* abort_flag) {
  const uint32_t quarter = warp & 3u;
  const uint32_t t_lane = (quarter * 32u) << 16;
  const uint32_t e = warp - (2 + SM_WARPS);
  const uint32_t leader_o_free = ptx::map_to_cta(b.o_free, 0);
  const uint32_t sig_o = ptx::map_to_cta(base + OFF_SIG + SIG_O + e * SIG_BYTES, 0);
  const uint32_t sig_src = base + OFF_SIG + SIG_SRC + (SM_WARPS + e) * SIG_BYTES;
  const uint32_t stage = base + OFF_STAGE + e * 2u * O_BOX;
  const uint32_t lsw = lane & 7u;
  const uint32_t row = quarter * 32u + lane;   // row within this CTA's 128
  const bool split = p.n_split > 1;
  uint32_t ki = 0;
  uint32_t g_end = 0;  // global key blocks up to and including this unit's
  for (int u = cluster; u < p.n_units; u += nclusters, ++ki) {
    const Item w = decode_unit(u, p);
    const bool more_units = u + nclusters < p.n_units;
    g_end += (uint32_t)w.nb;
    const uint32_t g_last = g_end - 1;
    if (!__all_sync(0xffffffffu, wait_sleepy(b.l_ready, ki & 1u, p, abort_flag))) break;
    const float l = l_rows[row];
    const float m = l_rows[CQ + row];
    __syncwarp();
    if (more_units && lane == 0) ptx::mbar_arrive(b.l_free);
    if (!warp_wait(b.o_done + 8 * (g_last & 1u), (g_last >> 1) & 1u, p, abort_flag)) break;
    ptx::tc_fence_after();
    const float inv_l = 1.f / l;
    if (!split) {
      const int r0 = w.q0 + (int)rank * CQ + (int)quarter * 32;
#pragma unroll 1
      for (int c = 0; c < HD / 64; ++c) {
        uint32_t o[64];
        const uint32_t ta = tmem_base + t_lane + O_COL + (uint32_t)c * 64u;
        ptx::tmem_ld_32x32b_x32(ta, *reinterpret_cast<uint32_t(*)[32]>(&o[0]));
        ptx::tmem_ld_32x32b_x32(ta + 32u, *reinterpret_cast<uint32_t(*)[32]>(&o[32]));
        ptx::tmem_ld_wait();
        ptx::reg_fence(o);
        // O is in registers: the next unit's first O += P V may overwrite it.
        if (c == HD / 64 - 1 && more_units)
          signal_leader(rank, lane, b.o_free, leader_o_free, sig_o, sig_src);
        // Box c & 1 is free once the store that used it two boxes ago read it.
        if (lane == 0) ptx::bulk_wait_group_read<1>();
        __syncwarp();
        const uint32_t box = stage + (uint32_t)(c & 1) * O_BOX;
#pragma unroll
        for (uint32_t i = 0; i < 8; ++i) {
          const float* f = reinterpret_cast<const float*>(&o[8 * i]);
          ptx::st_shared_v4(box + lane * 128u + ((i ^ lsw) << 4),
                            pack_half2(f[0] * inv_l, f[1] * inv_l),
                            pack_half2(f[2] * inv_l, f[3] * inv_l),
                            pack_half2(f[4] * inv_l, f[5] * inv_l),
                            pack_half2(f[6] * inv_l, f[7] * inv_l));
        }
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0 && r0 < p.seq_q) {
          ptx::tma_store_4d(tmO, box, 64 * c, r0, w.h, w.bz);
          ptx::bulk_commit_group();
        }
        __syncwarp();
      }
    } else {
      const int prow = u * PQ + (int)rank * CQ + (int)quarter * 32;  // first partial row
      float2* ml = reinterpret_cast<float2*>(p.part_ml) + (size_t)prow + lane;
      *ml = make_float2(m, l);
#pragma unroll 1
      for (int c = 0; c < HD / 32; ++c) {
        uint32_t o[32];
        ptx::tmem_ld_32x32b_x32(tmem_base + t_lane + O_COL + (uint32_t)c * 32u, o);
        ptx::tmem_ld_wait();
        ptx::reg_fence(o);
        if (c == HD / 32 - 1 && more_units)
          signal_leader(rank, lane, b.o_free, leader_o_free, sig_o, sig_src);
        if (lane == 0) ptx::bulk_wait_group_read<1>();
        __syncwarp();
        const uint32_t box = stage + (uint32_t)(c & 1) * O_BOX;
#pragma unroll
        for (uint32_t i = 0; i < 8; ++i)
          ptx::st_shared_v4(box + lane * 128u + ((i ^ lsw) << 4),
                            __float_as_uint(__uint_as_float(o[4 * i]) * inv_l),
                            __float_as_uint(__uint_as_float(o[4 * i + 1]) * inv_l),
                            __float_as_uint(__uint_as_float(o[4 * i + 2]) * inv_l),
                            __float_as_uint(__uint_as_float(o[4 * i + 3]) * inv_l));
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          ptx::tma_store_2d(tmP, box, 32 * c, prow);
          ptx::bulk_commit_group();
        }
        __syncwarp();
      }
    }
  }
  if (lane == 0) ptx::bulk_wait_group<0>();
  __syncwarp();
}

// After both CTAs stopped issuing: complete every phase a producer opened
// and wait (bounded) for the copies that were issued.  Ring fill f used slot
// f % RING in phase parity (f / RING) & 1; Q load q is phase q of q_full
// (at most the last one can be open).  A fill or Q load the leader never
// reached lacks its arrival: arrive expecting only the peer's bytes.  One
// the peer never issued leaves its bytes expected: take them off with
// complete_tx.
__device__ __noinline__ void leader_drain(const Bars& b, Issued mine, Issued peer,
                                          uint64_t limit_ns) {
  const uint32_t hi = mine.fills > peer.fills ? mine.fills : peer.fills;
  const uint32_t lo = hi > (uint32_t)RING ? hi - (uint32_t)RING : 0u;
  for (uint32_t f = lo; f < hi; ++f) {
    const uint32_t bar = b.full + 8 * (f % RING);
    if (f >= mine.fills) ptx::mbar_arrive_expect_tx_relaxed(bar, SLOT_BYTES);
    if (f >= peer.fills) ptx::mbar_complete_tx(bar, SLOT_BYTES);
    wait_drain(bar, (f / RING) & 1u, limit_ns);
  }
  const uint32_t qhi = mine.qloads > peer.qloads ? mine.qloads : peer.qloads;
  if (qhi > 0) {
    const uint32_t q = qhi - 1;
    if (q >= mine.qloads) ptx::mbar_arrive_expect_tx_relaxed(b.q_full, Q_BYTES);
    if (q >= peer.qloads) ptx::mbar_complete_tx(b.q_full, Q_BYTES);
    wait_drain(b.q_full, q & 1u, limit_ns);
  }
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NUM_THREADS, 1)
    attn_f16_fwd_pair_kernel(const __grid_constant__ CUtensorMap tmQ,
                             const __grid_constant__ CUtensorMap tmK,
                             const __grid_constant__ CUtensorMap tmV,
                             const __grid_constant__ CUtensorMap tmO,
                             const __grid_constant__ CUtensorMap tmP, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  const uint32_t warp = __shfl_sync(0xffffffffu, threadIdx.x >> 5, 0);
  const uint32_t lane = threadIdx.x & 31u;
  const uint32_t rank = ptx::cluster_ctarank();
  const int cluster = (int)(blockIdx.x >> 1);
  const int nclusters = (int)(gridDim.x >> 1);
  float* l_rows = reinterpret_cast<float*>(smem + OFF_L);

  Bars b;
  b.q_full = base + OFF_BAR;
  b.q_empty = b.q_full + 8;
  b.full = b.q_empty + 8;
  b.empty = b.full + 8 * RING;
  b.s_full = b.empty + 8 * RING;
  b.s_free = b.s_full + 8;
  b.p_full = b.s_free + 8;
  b.o_done = b.p_full + 16;
  b.o_free = b.o_done + 16;
  b.l_ready = b.o_free + 8;
  b.l_free = b.l_ready + 8;
  b.mma_done = b.l_free + 8;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_ABORT);

  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&tmQ);
    ptx::prefetch_tmap(&tmK);
    ptx::prefetch_tmap(&tmV);
    ptx::prefetch_tmap(p.n_split > 1 ? &tmP : &tmO);
    ptx::mbar_init(b.q_full, 1);
    ptx::mbar_init(b.q_empty, 1);
    for (int s = 0; s < RING; ++s) {
      ptx::mbar_init(b.full + 8 * s, 1);
      ptx::mbar_init(b.empty + 8 * s, 1);
    }
    ptx::mbar_init(b.s_full, 1);
    ptx::mbar_init(b.s_free, SM_WARPS);  // leader warps (+ the peer's bytes)
    for (int k = 0; k < 2; ++k) {
      ptx::mbar_init(b.p_full + 8 * k, SM_WARPS);  // leader warps (+ the peer's bytes)
      ptx::mbar_init(b.o_done + 8 * k, 1);
    }
    ptx::mbar_init(b.o_free, EP_WARPS);  // leader warps (+ the peer's bytes)
    ptx::mbar_init(b.l_ready, SM_WARPS);
    ptx::mbar_init(b.l_free, EP_WARPS);
    ptx::mbar_init(b.mma_done, 1);
    *abort_flag = 0;
    *reinterpret_cast<volatile uint32_t*>(smem + OFF_PEER_FILLS) = 0;
    *reinterpret_cast<volatile uint32_t*>(smem + OFF_PEER_QLOADS) = 0;
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
  // The next kernel in the stream may be scheduled now (it waits for this
  // grid before touching memory); and this one, launched as a programmatic
  // dependent, touches no global memory before the previous kernel has
  // completed.  Only the set-up above overlaps that kernel's tail.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");

  Issued issued{0, 0};
  if (warp == 0) {
    if (lane == 0)
      issued = producer_role(&tmQ, &tmK, &tmV, p, base, b, rank, cluster, nclusters, abort_flag);
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      mma_role(p, base, tmem_base, b, cluster, nclusters, abort_flag);
      // Every MMA issued must be finished before TMEM is freed.
      ptx::mma_commit_pair(b.mma_done, 0x1);
      wait_drain(b.mma_done, 0, p.timeout_ns);
    }
    __syncwarp();
  } else if (warp < 2 + SM_WARPS) {
    softmax_role(p, base, tmem_base, b, l_rows, rank, warp, lane, cluster, nclusters, abort_flag);
  } else {
    epilogue_role(&tmO, &tmP, p, base, tmem_base, b, l_rows, rank, warp, lane, cluster,
                  nclusters, abort_flag);
  }

  if (warp == 0 && lane == 0 && rank == 1) {
    ptx::st_cluster_u32(ptx::map_to_cta(base + OFF_PEER_FILLS, 0), issued.fills);
    ptx::st_cluster_u32(ptx::map_to_cta(base + OFF_PEER_QLOADS, 0), issued.qloads);
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();  // both CTAs have stopped issuing
  if (warp == 0 && lane == 0 && rank == 0) {
    const Issued peer{*reinterpret_cast<volatile uint32_t*>(smem + OFF_PEER_FILLS),
                      *reinterpret_cast<volatile uint32_t*>(smem + OFF_PEER_QLOADS)};
    leader_drain(b, issued, peer, p.timeout_ns);
  }
  ptx::cluster_sync();  // no copy into either CTA is still in flight
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
}

// Merges the key ranges of a split run.  Per query row, with M the largest
// range offset: O = sum_s w_s O_s / sum_s w_s, w_s = l_s 2^(m_s - M), O_s the
// range's normalised partial (FP32), ranges in order, one RN rounding to
// FP16.  One warp per row, eight columns per lane; launched as a
// programmatic dependent of the attention kernel.
__global__ void __launch_bounds__(256)
    attn_combine_kernel(const float* __restrict__ part, const float2* __restrict__ ml,
                        const Params p, __half* __restrict__ O, int64_t os_b, int64_t os_h,
                        int64_t os_r) {
  // The next kernel of the stream may start its set-up at once; it waits
  // for this grid before it touches memory.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int64_t gw = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = (int)(threadIdx.x & 31u);
  if (gw >= (int64_t)p.n_items * PQ) return;
  const int it = (int)(gw / PQ);
  const int r = (int)(gw - (int64_t)it * PQ);
  const int bh = it / p.n_qt;
  const int q = (it - bh * p.n_qt) * PQ + r;
  if (q >= p.seq_q) return;
  const int64_t u0 = (int64_t)it * p.n_split;
  float mmax = -INFINITY;
  for (int s = 0; s < p.n_split; ++s) mmax = fmaxf(mmax, ml[(u0 + s) * PQ + r].x);
  float wsum = 0.f;
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  for (int s = 0; s < p.n_split; ++s) {
    const float2 v = ml[(u0 + s) * PQ + r];
    const float wgt = v.y * exp2f(v.x - mmax);
    wsum += wgt;
    const float4* src =
        reinterpret_cast<const float4*>(part + ((u0 + s) * PQ + r) * HD + lane * 8);
    const float4 a0 = src[0], a1 = src[1];
    acc[0] = fmaf(wgt, a0.x, acc[0]);
    acc[1] = fmaf(wgt, a0.y, acc[1]);
    acc[2] = fmaf(wgt, a0.z, acc[2]);
    acc[3] = fmaf(wgt, a0.w, acc[3]);
    acc[4] = fmaf(wgt, a1.x, acc[4]);
    acc[5] = fmaf(wgt, a1.y, acc[5]);
    acc[6] = fmaf(wgt, a1.z, acc[6]);
    acc[7] = fmaf(wgt, a1.w, acc[7]);
  }
  const float inv = 1.f / wsum;
  uint4 out;
  out.x = pack_half2(acc[0] * inv, acc[1] * inv);
  out.y = pack_half2(acc[2] * inv, acc[3] * inv);
  out.z = pack_half2(acc[4] * inv, acc[5] * inv);
  out.w = pack_half2(acc[6] * inv, acc[7] * inv);
  __half* dst = O + (int64_t)(bh / p.heads) * os_b + (int64_t)(bh % p.heads) * os_h +
                (int64_t)q * os_r + lane * 8;
  *reinterpret_cast<uint4*>(dst) = out;
}

}  // namespace attnp
}  // namespace gf16
