// The plan object (gemm_f16_plan / destroy / status / options), error
// reporting, and the host helpers shared by the GEMM and attention entry
// points: tensor-map encoding with a per-plan cache and stream-ordered
// buffer growth.  No device code lives here.

#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>

#include "host.h"

namespace gf16 {
namespace host {

thread_local char g_last_cuda_error[512] = "no CUDA error recorded";

int cuda_fail(cudaError_t e, const char* what) {
  std::snprintf(g_last_cuda_error, sizeof(g_last_cuda_error), "%s: %s (%s)", what,
                cudaGetErrorName(e), cudaGetErrorString(e));
  return (e == cudaErrorMemoryAllocation) ? GEMM_F16_ERR_OOM : GEMM_F16_ERR_CUDA;
}

int fail_msg(const char* msg) {
  std::snprintf(g_last_cuda_error, sizeof(g_last_cuda_error), "%s", msg);
  return GEMM_F16_ERR_CUDA;
}

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

int encode_2d(CUtensorMap* map, CUtensorMapDataType dt, const void* ptr, uint64_t inner,
              uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
              CUtensorMapSwizzle swz, CUtensorMapL2promotion promo) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return fail_msg("cuTensorMapEncodeTiled entry point not available");
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, dt, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swz, promo, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    std::snprintf(g_last_cuda_error, sizeof(g_last_cuda_error),
                  "cuTensorMapEncodeTiled failed (CUresult %d)", (int)r);
    return GEMM_F16_ERR_CUDA;
  }
  return GEMM_F16_OK;
}

int encode_3d_f32(CUtensorMap* map, const void* ptr, uint64_t n, uint64_t m, uint64_t s,
                  uint64_t row_bytes, uint64_t plane_bytes) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return fail_msg("cuTensorMapEncodeTiled entry point not available");
  const cuuint64_t dims[3] = {n, m, s};
  const cuuint64_t strides[2] = {row_bytes, plane_bytes};
  const cuuint32_t box[3] = {16, 32, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(ptr), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                  CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    std::snprintf(g_last_cuda_error, sizeof(g_last_cuda_error),
                  "cuTensorMapEncodeTiled (workspace) failed (CUresult %d)", (int)r);
    return GEMM_F16_ERR_CUDA;
  }
  return GEMM_F16_OK;
}

int ensure_buffer(void** buf, size_t* cap, size_t bytes, cudaStream_t stream, const char* what) {
  if (*cap >= bytes) return GEMM_F16_OK;
  if (*buf) {
    GF16_CUDA(cudaFreeAsync(*buf, stream), what);
    *buf = nullptr;
    *cap = 0;
  }
  GF16_CUDA(cudaMallocAsync(buf, bytes, stream), what);
  *cap = bytes;
  return GEMM_F16_OK;
}

bool tmap_lookup(const gemm_f16_plan_s* p, const uint64_t (&key)[8], CUtensorMap* map) {
  for (int i = 0; i < p->tmap_used; ++i) {
    if (std::memcmp(p->tmaps[i].key, key, sizeof(key)) == 0) {
      *map = p->tmaps[i].map;
      return true;
    }
  }
  return false;
}

void tmap_remember(gemm_f16_plan_s* p, const uint64_t (&key)[8], const CUtensorMap& map) {
  TmapEntry& e = p->tmaps[p->tmap_next];
  std::memcpy(e.key, key, sizeof(key));
  e.map = map;
  p->tmap_next = (p->tmap_next + 1) % TMAP_CACHE;
  if (p->tmap_used < TMAP_CACHE) ++p->tmap_used;
}

int cached_encode_2d(gemm_f16_plan_s* p, CUtensorMap* map, CUtensorMapDataType dt, const void* ptr,
                     uint64_t inner, uint64_t outer, uint64_t row_bytes, uint32_t box_inner,
                     uint32_t box_outer, CUtensorMapSwizzle swz, CUtensorMapL2promotion promo) {
  const uint64_t key[8] = {(uint64_t)(uintptr_t)ptr, inner, outer, row_bytes,
                           ((uint64_t)box_inner << 32) | box_outer,
                           ((uint64_t)dt << 32) | (uint64_t)swz, (uint64_t)promo, 0};
  if (tmap_lookup(p, key, map)) return GEMM_F16_OK;
  const int rc = encode_2d(map, dt, ptr, inner, outer, row_bytes, box_inner, box_outer, swz, promo);
  if (rc) return rc;
  tmap_remember(p, key, *map);
  return GEMM_F16_OK;
}

constexpr size_t MAX_TIMING_PAIRS = 65536;

static int timing_event(gemm_f16_plan_s* p, cudaEvent_t* ev) {
  if (!p->timing_pool.empty()) {
    *ev = p->timing_pool.back();
    p->timing_pool.pop_back();
    return GEMM_F16_OK;
  }
  GF16_CUDA(cudaEventCreate(ev), "cudaEventCreate(kernel timing)");
  return GEMM_F16_OK;
}

int timing_begin(gemm_f16_plan_s* p, cudaStream_t stream, cudaEvent_t* start) {
  *start = nullptr;
  if (!p->kernel_timing || p->timing_marks.size() >= 2 * MAX_TIMING_PAIRS) return GEMM_F16_OK;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  GF16_CUDA(cudaStreamIsCapturing(stream, &cs), "cudaStreamIsCapturing");
  if (cs != cudaStreamCaptureStatusNone) return GEMM_F16_OK;
  cudaEvent_t ev;
  int rc = timing_event(p, &ev);
  if (rc) return rc;
  const cudaError_t e = cudaEventRecord(ev, stream);
  if (e != cudaSuccess) {
    p->timing_pool.push_back(ev);
    return cuda_fail(e, "cudaEventRecord(kernel timing)");
  }
  *start = ev;
  return GEMM_F16_OK;
}

int timing_end(gemm_f16_plan_s* p, cudaStream_t stream, cudaEvent_t start, bool launched) {
  if (!start) return GEMM_F16_OK;
  if (!launched) {
    p->timing_pool.push_back(start);
    return GEMM_F16_OK;
  }
  cudaEvent_t ev;
  int rc = timing_event(p, &ev);
  if (rc) {
    p->timing_pool.push_back(start);
    return rc;
  }
  const cudaError_t e = cudaEventRecord(ev, stream);
  if (e != cudaSuccess) {
    p->timing_pool.push_back(start);
    p->timing_pool.push_back(ev);
    return cuda_fail(e, "cudaEventRecord(kernel timing)");
  }
  p->timing_marks.push_back(start);
  p->timing_marks.push_back(ev);
  return GEMM_F16_OK;
}

}  // namespace host
}  // namespace gf16

using namespace gf16::host;

extern "C" {

const char* gemm_f16_strerror(int code) {
  switch (code) {
    case GEMM_F16_OK: return "ok";
    case GEMM_F16_ERR_INVALID_ARG: return "invalid argument";
    case GEMM_F16_ERR_MISALIGNED: return "pointer not 16-byte aligned or leading dimension not a multiple of 8";
    case GEMM_F16_ERR_UNSUPPORTED_DEVICE: return "device is not compute capability 10.3 (sm_103a)";
    case GEMM_F16_ERR_OOM: return "out of memory";
    case GEMM_F16_ERR_CUDA: return "CUDA call failed";
    case GEMM_F16_ERR_TIMEOUT: return "an in-kernel barrier wait timed out";
    case GEMM_F16_ERR_SCRATCH_TOO_SMALL: return "problem too large for the fixed no-alloc scratch";
    default: return "unknown error code";
  }
}

const char* gemm_f16_last_cuda_error(void) { return g_last_cuda_error; }

int gemm_f16_plan(gemm_f16_plan_t* out, int device) {
  if (!out) return GEMM_F16_ERR_INVALID_ARG;
  *out = nullptr;
  int ndev = 0;
  GF16_CUDA(cudaGetDeviceCount(&ndev), "cudaGetDeviceCount");
  if (device < 0 || device >= ndev) return GEMM_F16_ERR_INVALID_ARG;
  cudaDeviceProp prop;
  GF16_CUDA(cudaGetDeviceProperties(&prop, device), "cudaGetDeviceProperties");
  if (prop.major != 10 || prop.minor != 3) return GEMM_F16_ERR_UNSUPPORTED_DEVICE;
  DeviceGuard g(device);
  gemm_f16_plan_s* p = new (std::nothrow) gemm_f16_plan_s();
  if (!p) return GEMM_F16_ERR_OOM;
  p->device = device;
  p->num_sms = prop.multiProcessorCount;
  int rc = gemm_plan_init(p, prop);
  if (!rc) rc = attn_plan_init(p, prop);
  if (rc) {
    delete p;
    return rc;
  }
  cudaError_t e = cudaHostAlloc(&p->status_host, sizeof(int), cudaHostAllocMapped);
  if (e != cudaSuccess) {
    delete p;
    return cuda_fail(e, "cudaHostAlloc(status)");
  }
  *p->status_host = 0;
  e = cudaHostGetDevicePointer(reinterpret_cast<void**>(&p->status_dev), p->status_host, 0);
  if (e != cudaSuccess) {
    cudaFreeHost(p->status_host);
    delete p;
    return cuda_fail(e, "cudaHostGetDevicePointer(status)");
  }
  *out = p;
  return GEMM_F16_OK;
}

int gemm_f16_destroy(gemm_f16_plan_t p) {
  if (!p) return GEMM_F16_OK;
  {
    DeviceGuard g(p->device);
    cudaDeviceSynchronize();
    gemm_plan_release(p);
    attn_plan_release(p);
    if (p->ws) cudaFree(p->ws);
    if (p->in_stream) cudaStreamDestroy(p->in_stream);
    for (cudaEvent_t ev : p->timing_marks) cudaEventDestroy(ev);
    for (cudaEvent_t ev : p->timing_pool) cudaEventDestroy(ev);
    if (p->status_host) cudaFreeHost(p->status_host);
  }
  delete p;
  return GEMM_F16_OK;
}

int gemm_f16_status(gemm_f16_plan_t p) {
  if (!p) return GEMM_F16_ERR_INVALID_ARG;
  volatile int* s = p->status_host;
  const int v = *s;
  *s = 0;
  return v;
}

int gemm_f16_set_option(gemm_f16_plan_t p, int option, int64_t value) {
  if (!p) return GEMM_F16_ERR_INVALID_ARG;
  switch (option) {
    case GEMM_F16_OPT_TIMEOUT_NS:
      if (value <= 0) return GEMM_F16_ERR_INVALID_ARG;
      p->timeout_ns = (unsigned long long)value;
      return GEMM_F16_OK;
    case GEMM_F16_OPT_TILE_ORDER:
      if (value != 0 && value != 1) return GEMM_F16_ERR_INVALID_ARG;
      p->tile_order = (int)value;
      return GEMM_F16_OK;
    case GEMM_F16_OPT_FAULT_UNIT:
      if (value < -1 || value > 0x7fffffff) return GEMM_F16_ERR_INVALID_ARG;
      p->fault_unit = (int)value;
      return GEMM_F16_OK;
    case GEMM_F16_OPT_SM_LIMIT:
      if (value < 0 || value > 0x7fffffff) return GEMM_F16_ERR_INVALID_ARG;
      p->sm_limit = (int)value;
      return GEMM_F16_OK;
    case GEMM_F16_OPT_ATTN_KERNEL:
      if (value < 0 || value > 2) return GEMM_F16_ERR_INVALID_ARG;
      p->attn_kernel = (int)value;
      return GEMM_F16_OK;
    case GEMM_F16_OPT_ATTN_SPLIT:
      if (value < 0 || value > 65536) return GEMM_F16_ERR_INVALID_ARG;
      p->attn_split = (int)value;
      return GEMM_F16_OK;
    case GEMM_F16_OPT_A_REPACK:
      if (value < 0 || value > 2) return GEMM_F16_ERR_INVALID_ARG;
      p->a_repack = (int)value;
      return GEMM_F16_OK;
    case GEMM_F16_OPT_TILE_WIDTH:
      if (value != 0 && value != 64 && value != 128 && value != 256) return GEMM_F16_ERR_INVALID_ARG;
      p->tile_width = (int)value;
      return GEMM_F16_OK;
    case GEMM_F16_OPT_KERNEL_TIMING:
      if (value != 0 && value != 1) return GEMM_F16_ERR_INVALID_ARG;
      p->kernel_timing = (int)value;
      return GEMM_F16_OK;
    case GEMM_F16_OPT_KERNEL:
      if (value < 0 || value > 3) return GEMM_F16_ERR_INVALID_ARG;
      if (value >= 2 && p->max_pairs <= 0) return GEMM_F16_ERR_UNSUPPORTED_DEVICE;
      if (value == 3 && p->max_quads <= 0) return GEMM_F16_ERR_UNSUPPORTED_DEVICE;
      p->kernel = (int)value;
      return GEMM_F16_OK;
    default:
      return GEMM_F16_ERR_INVALID_ARG;
  }
}

int gemm_f16_get_option(gemm_f16_plan_t p, int option, int64_t* value) {
  if (!p || !value) return GEMM_F16_ERR_INVALID_ARG;
  switch (option) {
    case GEMM_F16_OPT_TIMEOUT_NS: *value = (int64_t)p->timeout_ns; return GEMM_F16_OK;
    case GEMM_F16_OPT_TILE_ORDER: *value = p->tile_order; return GEMM_F16_OK;
    case GEMM_F16_OPT_FAULT_UNIT: *value = p->fault_unit; return GEMM_F16_OK;
    case GEMM_F16_OPT_KERNEL: *value = p->kernel; return GEMM_F16_OK;
    case GEMM_F16_OPT_TILE_WIDTH: *value = p->tile_width; return GEMM_F16_OK;
    case GEMM_F16_OPT_SM_LIMIT: *value = p->sm_limit; return GEMM_F16_OK;
    case GEMM_F16_OPT_ATTN_KERNEL: *value = p->attn_kernel; return GEMM_F16_OK;
    case GEMM_F16_OPT_ATTN_SPLIT: *value = p->attn_split; return GEMM_F16_OK;
    case GEMM_F16_OPT_A_REPACK: *value = p->a_repack; return GEMM_F16_OK;
    case GEMM_F16_OPT_KERNEL_TIMING: *value = p->kernel_timing; return GEMM_F16_OK;
    case GEMM_F16_INFO_NUM_SMS: *value = p->num_sms; return GEMM_F16_OK;
    case GEMM_F16_INFO_MAX_PAIRS: *value = p->max_pairs; return GEMM_F16_OK;
    case GEMM_F16_INFO_MAX_QUADS: *value = p->max_quads; return GEMM_F16_OK;
    default: return GEMM_F16_ERR_INVALID_ARG;
  }
}

int gemm_f16_kernel_time(gemm_f16_plan_t p, double* total_ms, int64_t* launches) {
  if (!p || !total_ms || !launches) return GEMM_F16_ERR_INVALID_ARG;
  *total_ms = 0.0;
  *launches = 0;
  DeviceGuard g(p->device);
  int rc = GEMM_F16_OK;
  double sum = 0.0;
  int64_t n = 0;
  for (size_t i = 0; i + 1 < p->timing_marks.size(); i += 2) {
    cudaEvent_t a = p->timing_marks[i], b = p->timing_marks[i + 1];
    float ms = 0.0f;
    cudaError_t e = cudaEventSynchronize(b);
    if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, a, b);
    if (e != cudaSuccess) {
      if (!rc) rc = cuda_fail(e, "kernel timing event");
    } else {
      sum += ms;
      ++n;
    }
  }
  for (cudaEvent_t ev : p->timing_marks) p->timing_pool.push_back(ev);
  p->timing_marks.clear();
  if (rc) return rc;
  *total_ms = sum;
  *launches = n;
  return GEMM_F16_OK;
}

}  // extern "C"
