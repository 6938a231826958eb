// Scaled dot-product attention forward for head dimension 256 on GB300
// (sm_103a): O = softmax(scale * Q K^T) V per batch and head, binary16 in and
// out, FP32 scores, accumulator and softmax statistics.
//
// The schedule is the "SDP Kernel Split Barrier B" pattern of the "Xe2
// Nbarrier Pipelining" page, carried over to mbarriers and tensor memory.
// Per block of 64 keys: S = Q K^T (tensor core) -> softmax with a running
// row maximum -> P stored to shared memory -> ARRIVE -> [window: the deferred
// sum update; the next K and V tiles arrive through the copy ring; the next
// S = Q K^T runs on the tensor core] -> the MMA thread WAITS -> O += P V.
// P is double-buffered, so the softmax of block j+1 overlaps P V of block j.
//
// The output rescale ("compensation") is applied to the TMEM accumulator
// before P is published.  Here it is lazy: the exponent offset m a row uses
// only moves when the block maximum exceeds it by more than RESCALE_LOG2
// (base-2 units), so weights stay <= 2^RESCALE_LOG2 and the accumulator is
// touched only when some row of a warp moved its offset.  Numerator and
// denominator use the same offset, so the result is the same softmax.
//
// One CTA per (128 query rows, head, batch), 192 threads:
//   warp 0      TMA producer: Q once (128 x 256, four 64-column boxes), then
//               K and V tiles (64 x 256, 32 KB) into a 4-slot ring in the
//               order the MMA thread consumes them: K0, K1, K2, V0, K3, V1, ...
//   warp 1      allocates 512 TMEM columns (three 64-column S buffers, O in
//               256) and one lane issues the MMAs: S_j+2 = Q K_j+2^T
//               (128x64x16, x16) two blocks ahead of O += P_j V_j
//               (128x256x16, x4), releasing ring slots with tcgen05.commit.
//   warps 2..5  softmax + epilogue: one query row per thread (its TMEM
//               lane).  Row max / exp2 / row sum in FP32, P rounded to
//               binary16 into shared memory, final O / l rounded to binary16
//               and written with tensor stores.
//
// Barriers ("mbarrier State and Operations" page): q_full and full[s] (one
// arrive.expect_tx + the copies' bytes), empty[s] (one commit), s_full[b]
// (one commit per S block), p_full[b] (128 softmax threads), o_done[b] (one
// commit per P V block) for P buffer b, mma_done.  Every wait is bounded as
// in the GEMM kernels: past the time limit the role records
// GEMM_F16_ERR_TIMEOUT, raises the CTA's abort flag and stops; the CTA
// drains its copies and MMAs in flight and frees its TMEM before it exits.

#pragma once

namespace gf16 {
namespace attn {

constexpr int HD = 256;                 // head dimension
constexpr int BQ = 128;                 // query rows per CTA (MMA M, TMEM lanes)
constexpr int BKV = 64;                 // keys per block
constexpr int RING = 4;                 // K / V tiles in flight
constexpr int NUM_THREADS = 192;
constexpr int SM_THREADS = 128;

constexpr uint32_t CHUNK_Q = BQ * 128;            // 64 d-columns x 128 rows: 16 KB
constexpr uint32_t CHUNK_KV = BKV * 128;          // 64 d-columns x 64 rows: 8 KB
constexpr uint32_t Q_BYTES = (HD / 64) * CHUNK_Q;       // 64 KB
constexpr uint32_t TILE_BYTES = (HD / 64) * CHUNK_KV;   // 32 KB
constexpr uint32_t P_BYTES = BQ * BKV * 2;              // 16 KB per P buffer
constexpr uint32_t OFF_Q = 0;
constexpr uint32_t OFF_RING = OFF_Q + Q_BYTES;
constexpr uint32_t OFF_P = OFF_RING + RING * TILE_BYTES;  // two P buffers
constexpr uint32_t OFF_BAR = OFF_P + 2 * P_BYTES;
// q_full, full[RING], empty[RING], s_full[3], p_full[2], o_done[2], mma_done
constexpr uint32_t NUM_BARS = 1 + 2 * RING + 3 + 2 + 2 + 1;
constexpr uint32_t OFF_TMEM_SLOT = OFF_BAR + NUM_BARS * 8;
constexpr uint32_t OFF_ABORT = OFF_TMEM_SLOT + 4;
constexpr uint32_t SMEM_BYTES = OFF_ABORT + 4 + 1024;  // + room to align the base to 1024
static_assert(SMEM_BYTES <= 232448, "over the 227 KB shared-memory limit per CTA");
static_assert(OFF_RING % 1024 == 0 && OFF_P % 1024 == 0, "swizzled buffers need 1024-B alignment");

// S = Q K^T runs LOOKAHEAD key blocks ahead of the softmax, so S needs
// LOOKAHEAD + 1 buffers in TMEM.
constexpr int LOOKAHEAD = 2;
constexpr int S_BUFS = LOOKAHEAD + 1;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t S_COL = 0;     // S buffers at columns 0, 64, 128
constexpr uint32_t O_COL = 256;   // O: columns 256 .. 511
static_assert(S_COL + S_BUFS * BKV <= O_COL, "S buffers overlap O in TMEM");

// Lazy rescale threshold: a row's exponent offset moves only when its block
// maximum (base-2 units) exceeds the offset by more than this.
constexpr float RESCALE_LOG2 = 8.f;

// Instruction descriptors (kind::f16, FP32 accumulate): S = Q K^T has both
// operands K-major (Q rows and K rows both run along d); O += P V has A
// (P) K-major and B (V, rows along d = N) MN-major.
constexpr uint32_t IDESC_QK = make_idesc(BQ, BKV) & ~(1u << 16);
constexpr uint32_t IDESC_PV = make_idesc(BQ, HD);

struct Params {
  int seq_q, seq_kv;
  int nkv;                      // key blocks: ceil(seq_kv / 64)
  float scale_log2;             // scale * log2(e): scores go to base 2
  int* status;
  unsigned long long timeout_ns;
  int fault_cta;                // test only: CTA whose first K tile gets no copy
};

struct Bars {
  uint32_t q_full, full, empty, s_full, p_full, o_done, mma_done;
};

// Bounded wait loop.  SUSPEND: try_wait with the suspend-time hint (the
// thread waits in hardware); otherwise it polls.  The pair kernel's copy and
// MMA threads suspend; its softmax and epilogue warps, whose waits sit on
// the critical path of every key block, poll (all waits suspending measured
// 1.5 % slower on 4 x 16 x 4096^2, copy and MMA threads alone 0.7 % faster).
template <bool SUSPEND = false>
__device__ __noinline__ bool wait_slow(uint32_t bar, uint32_t parity, int* status,
                                       unsigned long long timeout_ns, volatile int* abort_flag) {
  const uint64_t t0 = ptx::globaltimer();
  while (true) {
    if (SUSPEND ? ptx::mbar_try_wait(bar, parity) : ptx::mbar_try_wait_poll(bar, parity))
      return true;
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
  if (ptx::mbar_try_wait_poll(bar, parity)) return true;
  return wait_slow(bar, parity, p.status, p.timeout_ns, abort_flag);
}

// ------------------------------------------------------------------ producer
// Issues the copies in consumption order; returns how many ring slots it
// filled (for the drain after an abort) through `issued`, and its ring
// position through `pos_out`.
__device__ __forceinline__ void producer_role(const CUtensorMap* tmQ, const CUtensorMap* tmK,
                                              const CUtensorMap* tmV, const Params& p,
                                              uint32_t base, const Bars& b, int q0, int h,
                                              int bz, bool fault, volatile int* abort_flag,
                                              RingPos* pos_out, uint32_t* issued_out) {
  ptx::mbar_arrive_expect_tx_relaxed(b.q_full, Q_BYTES);
#pragma unroll
  for (int c = 0; c < HD / 64; ++c)
    ptx::tma_load_4d(base + OFF_Q + c * CHUNK_Q, tmQ, b.q_full, 64 * c, q0, h, bz);

  RingPos pos{0, 0};
  uint32_t issued = 0;
  // One K or V tile into the next ring slot.
  auto load = [&](const CUtensorMap* tm, int j) -> bool {
    if (!wait_phase(b.empty + 8 * pos.stage, producer_wait_parity(pos), p, abort_flag))
      return false;
    const uint32_t fb = b.full + 8 * pos.stage;
    ptx::mbar_arrive_expect_tx_relaxed(fb, TILE_BYTES);
    if (!(fault && issued == 0)) {
      const uint32_t dst = base + OFF_RING + pos.stage * TILE_BYTES;
#pragma unroll
      for (int c = 0; c < HD / 64; ++c)
        ptx::tma_load_4d(dst + c * CHUNK_KV, tm, fb, 64 * c, j * BKV, h, bz);
    }
    ++issued;
    ring_advance(pos, RING);
    return true;
  };
  // The MMA thread's consumption order: K_0 .. K_{LOOKAHEAD-1}, then for
  // each block j: K_{j+LOOKAHEAD}, V_j.
  bool ok = true;
  for (int t = 0; t < LOOKAHEAD && t < p.nkv && ok; ++t) ok = load(tmK, t);
  for (int j = 0; j < p.nkv && ok; ++j) {
    if (j + LOOKAHEAD < p.nkv) ok = load(tmK, j + LOOKAHEAD);
    if (ok) ok = load(tmV, j);
  }
  *pos_out = pos;
  *issued_out = issued;
}

// ------------------------------------------------------------------ MMA issuer
__device__ __forceinline__ void mma_role(const Params& p, uint32_t base, uint32_t tmem_base,
                                         const Bars& b, volatile int* abort_flag) {
  if (!wait_phase(b.q_full, 0, p, abort_flag)) return;
  ptx::tc_fence_after();
  RingPos pos{0, 0};
  const uint32_t q_addr = base + OFF_Q;
  const uint32_t o_tmem = tmem_base + O_COL;

  // S_j = Q K_j^T into S buffer `sb`: 16 MMAs of K = 16 along d.
  auto issue_qk = [&](uint32_t sb) -> bool {
    if (!wait_phase(b.full + 8 * pos.stage, consumer_wait_parity(pos), p, abort_flag))
      return false;
    ptx::tc_fence_after();
    const uint32_t k_addr = base + OFF_RING + pos.stage * TILE_BYTES;
#pragma unroll
    for (int kk = 0; kk < HD / 16; ++kk) {
      const uint32_t off_q = (uint32_t)(kk >> 2) * CHUNK_Q + (uint32_t)(kk & 3) * 32u;
      const uint32_t off_k = (uint32_t)(kk >> 2) * CHUNK_KV + (uint32_t)(kk & 3) * 32u;
      ptx::mma_f16(tmem_base + S_COL + sb * BKV, smem_desc_sw128(q_addr + off_q, 16, 1024),
                   smem_desc_sw128(k_addr + off_k, 16, 1024), IDESC_QK, kk > 0 ? 1u : 0u);
    }
    ptx::mma_commit(b.empty + 8 * pos.stage);
    ptx::mma_commit(b.s_full + 8 * sb);
    ring_advance(pos, RING);
    return true;
  };

  bool ok = true;
  for (int t = 0; t < LOOKAHEAD && t < p.nkv && ok; ++t) ok = issue_qk((uint32_t)t % S_BUFS);
  for (int j = 0; j < p.nkv && ok; ++j) {
    // S two blocks ahead: it runs on the tensor core while the softmax
    // warps work on block j and P V of block j-1 drains.
    if (j + LOOKAHEAD < p.nkv && !issue_qk((uint32_t)(j + LOOKAHEAD) % S_BUFS)) break;
    // The split barrier's WAIT: P_j is in shared memory and O is rescaled.
    const uint32_t pb = (uint32_t)j & 1u;
    if (!wait_phase(b.p_full + 8 * pb, ((uint32_t)j >> 1) & 1u, p, abort_flag)) break;
    ptx::tc_fence_after();
    if (!wait_phase(b.full + 8 * pos.stage, consumer_wait_parity(pos), p, abort_flag)) break;
    ptx::tc_fence_after();
    const uint32_t v_addr = base + OFF_RING + pos.stage * TILE_BYTES;
#pragma unroll
    for (int kk = 0; kk < BKV / 16; ++kk) {
      ptx::mma_f16(o_tmem,
                   smem_desc_sw128(base + OFF_P + pb * P_BYTES + (uint32_t)kk * 32u, 16, 1024),
                   smem_desc_sw128(v_addr + (uint32_t)kk * 2048u, CHUNK_KV, 1024), IDESC_PV,
                   (j > 0 || kk > 0) ? 1u : 0u);
    }
    ptx::mma_commit(b.empty + 8 * pos.stage);
    ptx::mma_commit(b.o_done + 8 * pb);
    ring_advance(pos, RING);
  }
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Sum of a packed pair of binary16 values, in FP32.
__device__ __forceinline__ float half2_sum(uint32_t v) {
  const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&v));
  return f.x + f.y;
}

// P = 2^(scale*log2(e)*s - m) for one row of a key block of NCOL keys,
// packed to binary16 pairs; returns the FP32 sum of the weights (four
// partial sums).  MASK: keys from `valid` on are past the sequence end and
// get weight 0.
template <int NCOL, bool MASK>
__device__ __forceinline__ float block_weights(const uint32_t (&s)[NCOL], float sl2, float neg_m,
                                               int valid, uint32_t (&pk)[NCOL / 2]) {
  float l4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int c = 0; c < NCOL / 2; ++c) {
    float p0 = ptx::ex2_approx(fmaf(__uint_as_float(s[2 * c]), sl2, neg_m));
    float p1 = ptx::ex2_approx(fmaf(__uint_as_float(s[2 * c + 1]), sl2, neg_m));
    if (MASK) {
      p0 = (2 * c < valid) ? p0 : 0.f;
      p1 = (2 * c + 1 < valid) ? p1 : 0.f;
    }
    pk[c] = pack_half2(p0, p1);
    l4[c & 3] += p0 + p1;
  }
  return (l4[0] + l4[1]) + (l4[2] + l4[3]);
}

// Exponent offset update of one row for a key block (base-2 units):
// `s` holds the raw scores, keys from `valid` on excluded.  Returns the new
// offset (moved only when the block maximum passes m + RESCALE_LOG2) and
// sets `alpha` = 2^(m - m_new), exactly 1 when the offset stays.
template <int NCOL>
__device__ __forceinline__ float block_offset(uint32_t (&s)[NCOL], float sl2, int valid, float m,
                                              float* alpha) {
  if (valid < NCOL) {  // keep padded keys out of the maximum
    const float fill = sl2 >= 0.f ? -INFINITY : INFINITY;
#pragma unroll
    for (int c = 0; c < NCOL; ++c)
      if (c >= valid) s[c] = __float_as_uint(fill);
  }
  // eight independent chains over the raw scores (the minimum when the
  // scale is negative), scaled once
  float r8[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) r8[k] = __uint_as_float(s[k]);
  if (sl2 >= 0.f) {
#pragma unroll
    for (int c = 8; c < NCOL; ++c) r8[c & 7] = fmaxf(r8[c & 7], __uint_as_float(s[c]));
#pragma unroll
    for (int k = 1; k < 8; ++k) r8[0] = fmaxf(r8[0], r8[k]);
  } else {
#pragma unroll
    for (int c = 8; c < NCOL; ++c) r8[c & 7] = fminf(r8[c & 7], __uint_as_float(s[c]));
#pragma unroll
    for (int k = 1; k < 8; ++k) r8[0] = fminf(r8[0], r8[k]);
  }
  const float mx = (sl2 == 0.f) ? 0.f : r8[0] * sl2;
  const float m_new = (mx > m + RESCALE_LOG2) ? mx : m;
  *alpha = (m_new == m) ? 1.f : ptx::ex2_approx(m - m_new);
  return m_new;
}

// ------------------------------------------------------------------ softmax + epilogue
__device__ __forceinline__ void softmax_role(const CUtensorMap* tmO, const Params& p,
                                             uint32_t base, uint32_t tmem_base, const Bars& b,
                                             uint32_t warp, uint32_t lane, int q0, int h, int bz,
                                             volatile int* abort_flag) {
  const uint32_t quarter = warp & 3u;             // TMEM lanes 32*quarter .. +31
  const uint32_t row = quarter * 32u + lane;      // query row within the tile
  const uint32_t t_lane = (quarter * 32u) << 16;
  const uint32_t sw = row & 7u;
  const float sl2 = p.scale_log2;
  float m = -INFINITY;                            // exponent offset in use (base-2 units)
  float l = 0.f;                                  // running row sum
  bool ok = true;
  for (int j = 0; j < p.nkv; ++j) {
    const uint32_t sb = (uint32_t)j % S_BUFS;     // S buffer
    const uint32_t pb = (uint32_t)j & 1u;         // P buffer
    bool got = wait_phase(b.s_full + 8 * sb, ((uint32_t)j / S_BUFS) & 1u, p, abort_flag);
    if (!__all_sync(0xffffffffu, got)) {
      ok = false;
      break;
    }
    ptx::tc_fence_after();
    uint32_t s[64];
    ptx::tmem_ld_32x32b_x32(tmem_base + t_lane + S_COL + sb * BKV,
                            *reinterpret_cast<uint32_t(*)[32]>(&s[0]));
    ptx::tmem_ld_32x32b_x32(tmem_base + t_lane + S_COL + sb * BKV + 32,
                            *reinterpret_cast<uint32_t(*)[32]>(&s[32]));
    ptx::tmem_ld_wait();
    ptx::reg_fence(s);
    const int valid = p.seq_kv - j * BKV;  // keys of this block inside the sequence
    float alpha;
    const float m_new = block_offset<BKV>(s, sl2, valid, m, &alpha);
    uint32_t pk[32];
    const float lsum = valid < BKV ? block_weights<BKV, true>(s, sl2, -m_new, valid, pk)
                                   : block_weights<BKV, false>(s, sl2, -m_new, valid, pk);
    // P buffer pb was last read by P V of block j-2.
    if (j >= 2) {
      got = wait_phase(b.o_done + 8 * pb, ((uint32_t)(j - 2) >> 1) & 1u, p, abort_flag);
      if (!__all_sync(0xffffffffu, got)) {
        ok = false;
        break;
      }
    }
    // P row -> shared memory, 128-byte swizzle (16-byte chunk g of row r at
    // chunk position g ^ (r mod 8)), the K-major layout the MMA reads.
    const uint32_t p_row = base + OFF_P + pb * P_BYTES + row * 128u;
#pragma unroll
    for (uint32_t g = 0; g < 8; ++g)
      ptx::st_shared_v4(p_row + ((g ^ sw) << 4), pk[4 * g], pk[4 * g + 1], pk[4 * g + 2],
                        pk[4 * g + 3]);
    if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
      // Compensation: O *= alpha once P V of block j-1 has landed in O.
      const uint32_t ob = (uint32_t)(j - 1) & 1u;
      got = wait_phase(b.o_done + 8 * ob, ((uint32_t)(j - 1) >> 1) & 1u, p, abort_flag);
      if (!__all_sync(0xffffffffu, got)) {
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
      ptx::tmem_st_wait();
    }
    ptx::fence_proxy_async_smem();
    ptx::tc_fence_before();
    // The split barrier's ARRIVE ...
    ptx::mbar_arrive(b.p_full + 8 * pb);
    // ... and the window: the deferred sum update.
    l = l * alpha + lsum;
    m = m_new;
  }
  if (ok) {
    const uint32_t ob = (uint32_t)(p.nkv - 1) & 1u;
    const bool got = wait_phase(b.o_done + 8 * ob, ((uint32_t)(p.nkv - 1) >> 1) & 1u, p, abort_flag);
    ok = __all_sync(0xffffffffu, got);
  }
  if (ok) {
    ptx::tc_fence_after();
    const float inv_l = 1.f / l;
    // Staging in the Q buffer (every MMA has completed): per warp 4 boxes of
    // 32 rows x 64 columns, 128-byte swizzle.
    const uint32_t stage = base + OFF_Q + quarter * 4u * 4096u;
    const uint32_t lsw = lane & 7u;
#pragma unroll 1
    for (int c = 0; c < HD / 32; ++c) {
      uint32_t o[32];
      ptx::tmem_ld_32x32b_x32(tmem_base + t_lane + O_COL + (uint32_t)c * 32u, o);
      ptx::tmem_ld_wait();
      ptx::reg_fence(o);
      const uint32_t box = stage + (uint32_t)(c >> 1) * 4096u + lane * 128u;
#pragma unroll
      for (uint32_t i = 0; i < 4; ++i) {
        const uint32_t g = (uint32_t)(c & 1) * 4u + i;
        const float* f = reinterpret_cast<const float*>(&o[8 * i]);
        ptx::st_shared_v4(box + ((g ^ lsw) << 4), pack_half2(f[0] * inv_l, f[1] * inv_l),
                          pack_half2(f[2] * inv_l, f[3] * inv_l),
                          pack_half2(f[4] * inv_l, f[5] * inv_l),
                          pack_half2(f[6] * inv_l, f[7] * inv_l));
      }
    }
    ptx::fence_proxy_async_smem();
    __syncwarp();
    const int r0 = q0 + (int)quarter * 32;
    if (lane == 0 && r0 < p.seq_q) {
#pragma unroll
      for (int bx = 0; bx < HD / 64; ++bx)
        ptx::tma_store_4d(tmO, stage + (uint32_t)bx * 4096u, 64 * bx, r0, h, bz);
      ptx::bulk_commit_group();
      ptx::bulk_wait_group_read<0>();
    }
    __syncwarp();
  }
}

// After an abort: wait (bounded) for the copies still in flight into the
// ring (at most the last RING slots) and for Q.
__device__ __noinline__ void producer_drain(const Bars& b, RingPos pos, uint32_t issued,
                                            uint64_t limit_ns) {
  const uint32_t n = issued < (uint32_t)RING ? issued : (uint32_t)RING;
  for (uint32_t i = 0; i < n; ++i) {
    ring_retreat(pos, RING);
    wait_drain(b.full + 8 * pos.stage, consumer_wait_parity(pos), limit_ns);
  }
  wait_drain(b.q_full, 0, limit_ns);
}

__global__ void __launch_bounds__(NUM_THREADS, 1)
    attn_f16_fwd_kernel(const __grid_constant__ CUtensorMap tmQ,
                        const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV,
                        const __grid_constant__ CUtensorMap tmO, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  const uint32_t warp = __shfl_sync(0xffffffffu, threadIdx.x >> 5, 0);
  const uint32_t lane = threadIdx.x & 31u;
  const int q0 = (int)blockIdx.x * BQ;
  const int h = (int)blockIdx.y;
  const int bz = (int)blockIdx.z;
  const int cta = (int)(blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z));

  Bars b;
  b.q_full = base + OFF_BAR;
  b.full = b.q_full + 8;
  b.empty = b.full + 8 * RING;
  b.s_full = b.empty + 8 * RING;
  b.p_full = b.s_full + 8 * S_BUFS;
  b.o_done = b.p_full + 16;
  b.mma_done = b.o_done + 16;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_ABORT);

  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&tmQ);
    ptx::prefetch_tmap(&tmK);
    ptx::prefetch_tmap(&tmV);
    ptx::prefetch_tmap(&tmO);
    ptx::mbar_init(b.q_full, 1);
    for (int s = 0; s < RING; ++s) {
      ptx::mbar_init(b.full + 8 * s, 1);
      ptx::mbar_init(b.empty + 8 * s, 1);
    }
    for (int k = 0; k < S_BUFS; ++k) ptx::mbar_init(b.s_full + 8 * k, 1);
    for (int k = 0; k < 2; ++k) {
      ptx::mbar_init(b.p_full + 8 * k, SM_THREADS);
      ptx::mbar_init(b.o_done + 8 * k, 1);
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
  // The next kernel in the stream may be scheduled now (it waits for this
  // grid before touching memory); and this one, launched as a programmatic
  // dependent, touches no global memory before the previous kernel has
  // completed.  Only the set-up above overlaps that kernel's tail.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");

  RingPos prod_pos{0, 0};
  uint32_t prod_issued = 0;
  if (warp == 0) {
    if (lane == 0)
      producer_role(&tmQ, &tmK, &tmV, p, base, b, q0, h, bz, cta == p.fault_cta, abort_flag,
                    &prod_pos, &prod_issued);
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      mma_role(p, base, tmem_base, b, abort_flag);
      // Every MMA issued must be finished before TMEM is freed.
      ptx::mma_commit(b.mma_done);
      wait_drain(b.mma_done, 0, p.timeout_ns);
    }
    __syncwarp();
  } else {
    softmax_role(&tmO, p, base, tmem_base, b, warp, lane, q0, h, bz, abort_flag);
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 0 && lane == 0 && *abort_flag)
    producer_drain(b, prod_pos, prod_issued, p.timeout_ns);
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

}  // namespace attn
}  // namespace gf16
