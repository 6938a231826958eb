// Attention forward pass entry points (attn_f16_fwd, attn_f16_fwd_host,
// attn_f16_validate, attn_f16_key_ranges) and the two attention kernels:
// the persistent CTA-pair kernel (attn_pair.cuh) and the single-CTA kernel
// (attn_f16.cuh).  The plan object and the shared host helpers come from
// host.h; the plan's status word, time limit, SM limit and test fault
// option are shared with the GEMM.

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdio>
#include <cstring>

#include "host.h"
#include "ptx.cuh"
#include "schedule.h"
#include "common.cuh"

#include "attn_f16.cuh"
#include "attn_pair.cuh"

using namespace gf16;
using namespace gf16::host;

namespace gf16 {
namespace host {

int attn_plan_init(gemm_f16_plan_s* p, const cudaDeviceProp& prop) {
  GF16_CUDA(cudaFuncSetAttribute(attn::attn_f16_fwd_kernel,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)attn::SMEM_BYTES),
            "cudaFuncSetAttribute(attention kernel smem)");
  GF16_CUDA(cudaFuncSetAttribute(attnp::attn_f16_fwd_pair_kernel,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)attnp::SMEM_BYTES),
            "cudaFuncSetAttribute(pair attention kernel smem)");
  // Co-resident clusters of two for the pair kernel (0 if the query fails:
  // the single-CTA kernel is then used).
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(prop.multiProcessorCount / 2 * 2), 1, 1);
  cfg.blockDim = dim3(attnp::NUM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = attnp::SMEM_BYTES;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = 2;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  int clusters = 0;
  if (cudaOccupancyMaxActiveClusters(&clusters, attnp::attn_f16_fwd_pair_kernel, &cfg) !=
      cudaSuccess) {
    cudaGetLastError();
    clusters = 0;
  }
  p->attn_pairs = clusters;
  return GEMM_F16_OK;
}

void attn_plan_release(gemm_f16_plan_s* p) {
  for (int sl = 0; sl < 2; ++sl) {
    if (p->attn_in_done[sl]) cudaEventDestroy(p->attn_in_done[sl]);
    if (p->attn_done[sl]) cudaEventDestroy(p->attn_done[sl]);
    for (int i = 0; i < 4; ++i)
      if (p->abuf[sl][i]) cudaFree(p->abuf[sl][i]);
  }
}

}  // namespace host
}  // namespace gf16

namespace {

// [batch, head, row, 256] binary16 view as a 4-D tensor map: dims (d, row,
// head, batch), box (64, box_rows, 1, 1), 128-byte swizzle.
int encode_bhsd(CUtensorMap* map, const void* ptr, int batch, int heads, int rows,
                const int64_t st[3], uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return fail_msg("cuTensorMapEncodeTiled entry point not available");
  // A stride of an extent-1 dimension is never used; give the map a valid one.
  const int64_t row_st = st[2];
  const int64_t head_st = heads > 1 ? st[1] : row_st * rows;
  const int64_t batch_st = batch > 1 ? st[0] : head_st * heads;
  const cuuint64_t dims[4] = {(cuuint64_t)attn::HD, (cuuint64_t)rows, (cuuint64_t)heads,
                              (cuuint64_t)batch};
  const cuuint64_t strides[3] = {(cuuint64_t)row_st * 2, (cuuint64_t)head_st * 2,
                                 (cuuint64_t)batch_st * 2};
  const cuuint32_t box[4] = {64, box_rows, 1, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4, const_cast<void*>(ptr), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    std::snprintf(g_last_cuda_error, sizeof(g_last_cuda_error),
                  "cuTensorMapEncodeTiled (attention operand) failed (CUresult %d)", (int)r);
    return GEMM_F16_ERR_CUDA;
  }
  return GEMM_F16_OK;
}

// encode_bhsd through the plan's tensor-map cache (keys tagged apart from
// the 2-D GEMM maps).
int cached_encode_bhsd(gemm_f16_plan_s* p, CUtensorMap* map, const void* ptr, int batch,
                       int heads, int rows, const int64_t st[3], uint32_t box_rows) {
  const uint64_t key[8] = {(uint64_t)(uintptr_t)ptr, ((uint64_t)(uint32_t)batch << 32) | (uint32_t)heads,
                           (uint64_t)(uint32_t)rows, (uint64_t)st[0], (uint64_t)st[1],
                           (uint64_t)st[2], (uint64_t)box_rows, 0x4D00000000000000ull};
  if (tmap_lookup(p, key, map)) return GEMM_F16_OK;
  const int rc = encode_bhsd(map, ptr, batch, heads, rows, st, box_rows);
  if (rc) return rc;
  tmap_remember(p, key, *map);
  return GEMM_F16_OK;
}

bool strides_ok(const int64_t* st) {
  if (!st) return false;
  for (int i = 0; i < 3; ++i)
    if (st[i] <= 0 || st[i] >= ((int64_t)1 << 38)) return false;
  return st[2] >= attn::HD;
}

}  // namespace

// Co-resident CTA pairs the pair attention kernel may use (SM limit applied).
static int64_t attn_pair_slots(const gemm_f16_plan_s* p) {
  int64_t slots = p->attn_pairs;
  if (p->sm_limit > 0) slots = std::max<int64_t>(1, std::min<int64_t>(slots, p->sm_limit / 2));
  return slots;
}

// Key ranges per item of the pair attention kernel and the blocks per range
// (none empty): the option if set (capped at the block count), else a split
// when the items fill less than half of the pair slots and there are at
// least four key blocks.
static int64_t attn_key_ranges(const gemm_f16_plan_s* p, int64_t items, int64_t nkv,
                               int* bps) {
  const int64_t slots = attn_pair_slots(p);
  int64_t n = 1;
  if (p->attn_split > 0)
    n = std::min<int64_t>(p->attn_split, nkv);
  else if (2 * items <= slots && nkv >= 4)
    n = std::min<int64_t>(slots / items, nkv / 2);
  n = std::max<int64_t>(n, 1);
  *bps = (int)ceil_div(nkv, n);
  return ceil_div(nkv, *bps);
}

extern "C" {

int attn_f16_validate(int batch, int heads, int seq_q, int seq_kv, int head_dim, const void* Q,
                      const int64_t q_strides[3], const void* K, const int64_t k_strides[3],
                      const void* V, const int64_t v_strides[3], const void* O,
                      const int64_t o_strides[3], float scale) {
  if (batch < 1 || heads < 1 || batch > 65535 || heads > 65535) return GEMM_F16_ERR_INVALID_ARG;
  if (seq_q < 1 || seq_kv < 1) return GEMM_F16_ERR_INVALID_ARG;
  if (head_dim != attn::HD) return GEMM_F16_ERR_INVALID_ARG;
  if (!Q || !K || !V || !O) return GEMM_F16_ERR_INVALID_ARG;
  if (!(scale == scale) || scale > 3.0e38f || scale < -3.0e38f) return GEMM_F16_ERR_INVALID_ARG;
  const int64_t* sts[4] = {q_strides, k_strides, v_strides, o_strides};
  for (const int64_t* st : sts)
    if (!strides_ok(st)) return GEMM_F16_ERR_INVALID_ARG;
  const void* ptrs[4] = {Q, K, V, O};
  for (const void* ptr : ptrs)
    if ((uintptr_t)ptr & 15) return GEMM_F16_ERR_MISALIGNED;
  for (const int64_t* st : sts)
    if ((st[0] | st[1] | st[2]) & 7) return GEMM_F16_ERR_MISALIGNED;
  return GEMM_F16_OK;
}

int attn_f16_key_ranges(gemm_f16_plan_t p, int batch, int heads, int seq_q, int seq_kv,
                        int* ranges) {
  if (!p || !ranges || batch < 1 || heads < 1 || seq_q < 1 || seq_kv < 1)
    return GEMM_F16_ERR_INVALID_ARG;
  *ranges = 1;
  if (p->attn_kernel == 1 || p->attn_pairs <= 0) return GEMM_F16_OK;
  const int64_t items = (int64_t)batch * heads * ceil_div(seq_q, attnp::PQ);
  int bps = 0;
  *ranges = (int)attn_key_ranges(p, items, ceil_div(seq_kv, attnp::BKV), &bps);
  return GEMM_F16_OK;
}

int attn_f16_fwd(gemm_f16_plan_t p, int batch, int heads, int seq_q, int seq_kv, int head_dim,
                 const void* Q, const int64_t q_strides[3], const void* K,
                 const int64_t k_strides[3], const void* V, const int64_t v_strides[3], void* O,
                 const int64_t o_strides[3], float scale, gemm_f16_stream_t stream) {
  if (!p) return GEMM_F16_ERR_INVALID_ARG;
  int rc = attn_f16_validate(batch, heads, seq_q, seq_kv, head_dim, Q, q_strides, K, k_strides,
                             V, v_strides, O, o_strides, scale);
  if (rc) return rc;
  DeviceGuard g(p->device);
  const bool use_pair = p->attn_kernel != 1 && p->attn_pairs > 0;
  CUtensorMap tmQ, tmK, tmV, tmO;
  if ((rc = cached_encode_bhsd(p, &tmQ, Q, batch, heads, seq_q, q_strides, attn::BQ))) return rc;
  if ((rc = cached_encode_bhsd(p, &tmK, K, batch, heads, seq_kv, k_strides, 64))) return rc;
  if ((rc = cached_encode_bhsd(p, &tmV, V, batch, heads, seq_kv, v_strides, use_pair ? 128u : 64u)))
    return rc;
  if ((rc = cached_encode_bhsd(p, &tmO, O, batch, heads, seq_q, o_strides, 32))) return rc;
  if (use_pair) {
    attnp::Params prm;
    prm.seq_q = seq_q;
    prm.seq_kv = seq_kv;
    prm.nkv = (int)ceil_div(seq_kv, attnp::BKV);
    prm.n_qt = (int)ceil_div(seq_q, attnp::PQ);
    prm.heads = heads;
    const int64_t items = (int64_t)batch * heads * prm.n_qt;
    if (items > INT32_MAX - 65536) return GEMM_F16_ERR_INVALID_ARG;  // unit + clusters fits
    prm.n_items = (int)items;
    prm.scale_log2 = scale * 1.4426950408889634f;  // log2(e)
    prm.status = p->status_dev;
    prm.timeout_ns = p->timeout_ns;
    prm.fault_unit = p->fault_unit;
    // Persistent: one cluster per co-resident pair slot (fewer under an SM
    // limit), never more than there are units.
    const int64_t slots = attn_pair_slots(p);
    int64_t n_split = attn_key_ranges(p, items, prm.nkv, &prm.bps);
    const int64_t units = items * n_split;
    if (units > INT32_MAX - 65536) return GEMM_F16_ERR_INVALID_ARG;
    prm.n_split = (int)n_split;
    prm.n_units = (int)units;
    prm.part_ml = nullptr;
    CUtensorMap tmP = tmO;
    const size_t part_bytes = (size_t)units * attnp::PQ * attn::HD * sizeof(float);
    if (n_split > 1) {
      const size_t bytes = part_bytes + (size_t)units * attnp::PQ * 2 * sizeof(float);
      if ((rc = ensure_buffer(&p->ws, &p->ws_bytes, bytes, (cudaStream_t)stream,
                              "attention workspace allocation")))
        return rc;
      prm.part_ml = reinterpret_cast<float*>(static_cast<char*>(p->ws) + part_bytes);
      // The partial O: units * 256 rows of 256 FP32, stored in 32 x 32 boxes.
      if ((rc = cached_encode_2d(p, &tmP, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, p->ws, attn::HD,
                                 (uint64_t)units * attnp::PQ, attn::HD * sizeof(float), 32, 32,
                                 CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B)))
        return rc;
    }
    const int64_t clusters = std::min<int64_t>(slots, units);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(2 * clusters), 1, 1);
    cfg.blockDim = dim3(attnp::NUM_THREADS, 1, 1);
    cfg.dynamicSmemBytes = attnp::SMEM_BYTES;
    cfg.stream = (cudaStream_t)stream;
    cudaLaunchAttribute pdl;
    pdl.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &pdl;
    cfg.numAttrs = 1;
    cudaEvent_t t0;
    if ((rc = timing_begin(p, cfg.stream, &t0))) return rc;
    const cudaError_t le =
        cudaLaunchKernelEx(&cfg, attnp::attn_f16_fwd_pair_kernel, tmQ, tmK, tmV, tmO, tmP, prm);
    rc = timing_end(p, cfg.stream, t0, le == cudaSuccess);
    GF16_CUDA(le, "launch attn_f16_fwd_pair_kernel");
    if (rc) return rc;
    if (n_split > 1) {
      // One warp per query row of every item.
      cudaLaunchConfig_t ccfg = {};
      ccfg.gridDim = dim3((unsigned)(items * attnp::PQ / 8), 1, 1);
      ccfg.blockDim = dim3(256, 1, 1);
      ccfg.stream = (cudaStream_t)stream;
      ccfg.attrs = &pdl;
      ccfg.numAttrs = 1;
      GF16_CUDA(cudaLaunchKernelEx(&ccfg, attnp::attn_combine_kernel,
                                   static_cast<const float*>(p->ws),
                                   static_cast<const float2*>(static_cast<const void*>(prm.part_ml)),
                                   prm, static_cast<__half*>(O), o_strides[0], o_strides[1],
                                   o_strides[2]),
                "launch attn_combine_kernel");
    }
    return GEMM_F16_OK;
  }
  attn::Params prm;
  prm.seq_q = seq_q;
  prm.seq_kv = seq_kv;
  prm.nkv = (int)ceil_div(seq_kv, attn::BKV);
  prm.scale_log2 = scale * 1.4426950408889634f;  // log2(e)
  prm.status = p->status_dev;
  prm.timeout_ns = p->timeout_ns;
  prm.fault_cta = p->fault_unit;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)ceil_div(seq_q, attn::BQ), (unsigned)heads, (unsigned)batch);
  cfg.blockDim = dim3(attn::NUM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = attn::SMEM_BYTES;
  cfg.stream = (cudaStream_t)stream;
  cudaLaunchAttribute pdl;
  pdl.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &pdl;
  cfg.numAttrs = 1;
  cudaEvent_t t0;
  if ((rc = timing_begin(p, cfg.stream, &t0))) return rc;
  const cudaError_t le = cudaLaunchKernelEx(&cfg, attn::attn_f16_fwd_kernel, tmQ, tmK, tmV, tmO, prm);
  rc = timing_end(p, cfg.stream, t0, le == cudaSuccess);
  GF16_CUDA(le, "launch attn_f16_fwd_kernel");
  if (rc) return rc;
  return GEMM_F16_OK;
}

int attn_f16_fwd_host(gemm_f16_plan_t p, int batch, int heads, int seq_q, int seq_kv,
                      int head_dim, const void* hQ, const void* hK, const void* hV, void* hO,
                      float scale, gemm_f16_stream_t stream_) {
  if (!p || !hQ || !hK || !hV || !hO) return GEMM_F16_ERR_INVALID_ARG;
  // device copies are contiguous [batch, head, row, 256]
  const int64_t qs[3] = {(int64_t)heads * seq_q * 256, (int64_t)seq_q * 256, 256};
  const int64_t ks[3] = {(int64_t)heads * seq_kv * 256, (int64_t)seq_kv * 256, 256};
  const void* probe = reinterpret_cast<const void*>(static_cast<uintptr_t>(256));
  int rc = attn_f16_validate(batch, heads, seq_q, seq_kv, head_dim, probe, qs, probe, ks, probe, ks,
                             probe, qs, scale);
  if (rc) return rc;
  cudaStream_t stream = (cudaStream_t)stream_;
  DeviceGuard g(p->device);
  if (!p->in_stream)
    GF16_CUDA(cudaStreamCreateWithFlags(&p->in_stream, cudaStreamNonBlocking),
              "create input-copy stream");
  for (int sl = 0; sl < 2; ++sl) {
    if (!p->attn_in_done[sl])
      GF16_CUDA(cudaEventCreateWithFlags(&p->attn_in_done[sl], cudaEventDisableTiming),
                "create event");
    if (!p->attn_done[sl])
      GF16_CUDA(cudaEventCreateWithFlags(&p->attn_done[sl], cudaEventDisableTiming),
                "create event");
  }
  const int slot = p->attn_slot;
  p->attn_slot ^= 1;
  void** buf = p->abuf[slot];
  const size_t qbytes = (size_t)batch * heads * seq_q * 256 * 2;
  const size_t kbytes = (size_t)batch * heads * seq_kv * 256 * 2;
  const size_t bytes[4] = {qbytes, kbytes, kbytes, qbytes};
  bool grow = false;
  for (int i = 0; i < 4; ++i) grow = grow || p->acap[slot][i] < bytes[i];
  if (grow) {
    // Growing a slot: let everything that may still use it finish first.
    GF16_CUDA(cudaDeviceSynchronize(), "synchronise before growing attention staging");
    for (int i = 0; i < 4; ++i) {
      if (p->acap[slot][i] >= bytes[i]) continue;
      if (buf[i]) cudaFree(buf[i]);
      buf[i] = nullptr;
      p->acap[slot][i] = 0;
      GF16_CUDA(cudaMalloc(&buf[i], bytes[i]), "attention staging allocation");
      p->acap[slot][i] = bytes[i];
    }
  }
  // Q, K, V go in on the plan's input stream once the call that last used
  // this slot (two calls ago) has finished its pass and its output copy; the
  // pass on `stream` waits for them; O comes back on `stream` after the pass.
  GF16_CUDA(cudaStreamWaitEvent(p->in_stream, p->attn_done[slot], 0), "order input copies");
  GF16_CUDA(cudaMemcpyAsync(buf[0], hQ, qbytes, cudaMemcpyHostToDevice, p->in_stream), "copy Q");
  GF16_CUDA(cudaMemcpyAsync(buf[1], hK, kbytes, cudaMemcpyHostToDevice, p->in_stream), "copy K");
  GF16_CUDA(cudaMemcpyAsync(buf[2], hV, kbytes, cudaMemcpyHostToDevice, p->in_stream), "copy V");
  GF16_CUDA(cudaEventRecord(p->attn_in_done[slot], p->in_stream), "record input copies");
  GF16_CUDA(cudaStreamWaitEvent(stream, p->attn_in_done[slot], 0), "order pass after inputs");
  rc = attn_f16_fwd(p, batch, heads, seq_q, seq_kv, head_dim, buf[0], qs, buf[1], ks, buf[2], ks,
                    buf[3], qs, scale, stream_);
  if (rc) return rc;
  GF16_CUDA(cudaMemcpyAsync(hO, buf[3], qbytes, cudaMemcpyDeviceToHost, stream), "copy O to host");
  // The slot is free again once O has left it, whatever stream the next call uses.
  GF16_CUDA(cudaEventRecord(p->attn_done[slot], stream), "record pass and output copy");
  return GEMM_F16_OK;
}

}  // extern "C"
