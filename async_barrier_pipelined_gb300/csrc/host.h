// Host-side pieces shared by the library's translation units: the plan
// object behind gemm_f16_plan_t, CUDA error bookkeeping, tensor-map
// encoding (with the plan's cache) and stream-ordered buffer growth.
//
// plan.cu defines these; gemm_f16.cu (GEMM kernels and entry points) and
// attn_f16.cu (attention kernels and entry points) use them.  Each of the
// two adds its own part of plan creation and destruction through the
// *_plan_init / *_plan_release hooks below.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <vector>

#include "attn_f16.h"
#include "gemm_f16.h"

namespace gf16 {
namespace host {

// Text of the most recent CUDA failure on this host thread
// (gemm_f16_last_cuda_error).
extern thread_local char g_last_cuda_error[512];

// Record `e` with `what` and map it to a library error code
// (GEMM_F16_ERR_OOM for an allocation failure, else GEMM_F16_ERR_CUDA).
int cuda_fail(cudaError_t e, const char* what);
// Record a failure that has no cudaError_t (e.g. a driver entry point).
int fail_msg(const char* msg);

#define GF16_CUDA(call, what)                                         \
  do {                                                                \
    cudaError_t e_ = (call);                                          \
    if (e_ != cudaSuccess) return ::gf16::host::cuda_fail(e_, what);  \
  } while (0)

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
// cuTensorMapEncodeTiled through the runtime's driver entry-point query
// (NULL if the driver does not provide it).
EncodeTiledFn encode_fn();

// 2-D tiled tensor map: `inner` x `outer` elements, rows `row_bytes` apart,
// boxes of box_inner x box_outer, zero fill out of range.
int encode_2d(CUtensorMap* map, CUtensorMapDataType dt, const void* ptr, uint64_t inner,
              uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
              CUtensorMapSwizzle swz, CUtensorMapL2promotion promo);
// 3-D FP32 tensor map (n, m, s) with boxes of 16 x 32 x 1 and the 64-byte
// swizzle: the split partials [s][m][n] written by the epilogues.
int encode_3d_f32(CUtensorMap* map, const void* ptr, uint64_t n, uint64_t m, uint64_t s,
                  uint64_t row_bytes, uint64_t plane_bytes);

// Makes `dev` current for the guard's lifetime.
struct DeviceGuard {
  int prev = -1;
  bool switched = false;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) == cudaSuccess && prev != dev) switched = (cudaSetDevice(dev) == cudaSuccess);
  }
  ~DeviceGuard() {
    if (switched) cudaSetDevice(prev);
  }
};

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Grow a stream-ordered device buffer to at least `bytes` (free the old one
// and allocate on `stream`).
int ensure_buffer(void** buf, size_t* cap, size_t bytes, cudaStream_t stream, const char* what);

// Device tile tables cached per plan (pair-kernel work lists), keyed by the
// shape and options they were built for.
struct OrderTable {
  int64_t key[6];
  uint32_t* dev;
  int64_t count;
  int parts;  // K parts of the last (count % pairs) tiles (1: none)
};

// Recently encoded tensor maps, keyed by everything the encoding depends on,
// so that repeated runs on the same buffers skip cuTensorMapEncodeTiled.
struct TmapEntry {
  uint64_t key[8];
  CUtensorMap map;
};
constexpr int TMAP_CACHE = 32;

}  // namespace host
}  // namespace gf16

struct gemm_f16_plan_s {
  int device = 0;
  int num_sms = 0;
  int* status_host = nullptr;  // mapped pinned host memory
  int* status_dev = nullptr;
  unsigned long long timeout_ns = 1000000000ull;
  int tile_order = 0;
  int fault_unit = -1;
  int kernel = 0;      // 0 auto, 1 single CTA, 2 CTA pair
  int tile_width = 0;  // single-CTA tile width: 0 auto, else 256 / 128 / 64
  int sm_limit = 0;    // most SMs a launch may use (0: all)
  int attn_kernel = 0; // attention: 0 auto (CTA pair), 1 single CTA, 2 CTA pair
  int attn_split = 0;  // pair attention key ranges: 0 auto, n >= 1 forced
  int a_repack = 0;    // repack A with a pitch off 128-byte lines: 0 auto, 1 never, 2 always
  int max_pairs = 0;   // co-resident clusters of two for the pair kernel
  int max_quads = 0;   // co-resident clusters of four for the cluster-of-four kernel
  int attn_pairs = 0;  // co-resident clusters of two for the pair attention kernel
  void* ws = nullptr;
  size_t ws_bytes = 0;
  void* apack = nullptr;  // repacked copy of A (see pack_rows_kernel)
  size_t apack_bytes = 0;
  // FP32 values of the K halves of the pair kernel's last-wave tiles.
  void* tail_ws = nullptr;
  size_t tail_ws_bytes = 0;
  std::vector<gf16::host::OrderTable> orders;
  // run_host: two slots of device staging (A, B, C) used by alternate calls,
  // a stream for the input copies and the events that order the slots.
  void* hbuf[2][3] = {{nullptr, nullptr, nullptr}, {nullptr, nullptr, nullptr}};
  size_t hcap[2][3] = {{0, 0, 0}, {0, 0, 0}};
  cudaStream_t in_stream = nullptr;
  cudaEvent_t in_done[2] = {nullptr, nullptr};
  cudaEvent_t gemm_done[2] = {nullptr, nullptr};
  int host_slot = 0;
  // attn_f16_fwd_host: two slots of device Q, K, V, O and their events.
  void* abuf[2][4] = {{nullptr, nullptr, nullptr, nullptr}, {nullptr, nullptr, nullptr, nullptr}};
  size_t acap[2][4] = {{0, 0, 0, 0}, {0, 0, 0, 0}};
  cudaEvent_t attn_in_done[2] = {nullptr, nullptr};
  cudaEvent_t attn_done[2] = {nullptr, nullptr};
  int attn_slot = 0;
  gf16::host::TmapEntry tmaps[gf16::host::TMAP_CACHE];
  int tmap_used = 0, tmap_next = 0;
  // GEMM_F16_OPT_KERNEL_TIMING: recorded (start, end) event pairs around
  // product / attention kernel launches, and the idle events they reuse.
  int kernel_timing = 0;
  std::vector<cudaEvent_t> timing_marks;  // start, end, start, end, ...
  std::vector<cudaEvent_t> timing_pool;
};

namespace gf16 {
namespace host {

// The plan's tensor-map cache: look a key up (true and *map filled on a
// hit) or remember a freshly encoded map (oldest entry replaced).
bool tmap_lookup(const gemm_f16_plan_s* p, const uint64_t (&key)[8], CUtensorMap* map);
void tmap_remember(gemm_f16_plan_s* p, const uint64_t (&key)[8], const CUtensorMap& map);

// encode_2d through the plan's cache.
int cached_encode_2d(gemm_f16_plan_s* p, CUtensorMap* map, CUtensorMapDataType dt, const void* ptr,
                     uint64_t inner, uint64_t outer, uint64_t row_bytes, uint32_t box_inner,
                     uint32_t box_outer, CUtensorMapSwizzle swz, CUtensorMapL2promotion promo);

// Kernel timing records (GEMM_F16_OPT_KERNEL_TIMING).  timing_begin records
// a start event on `stream` and returns it in *start (nullptr when timing is
// off, the stream is capturing, or 65536 pairs are waiting); timing_end
// records the matching end event after a successful launch, or returns the
// start event to the pool when the launch failed (nothing for a nullptr
// start).
int timing_begin(gemm_f16_plan_s* p, cudaStream_t stream, cudaEvent_t* start);
int timing_end(gemm_f16_plan_s* p, cudaStream_t stream, cudaEvent_t start, bool launched);

// Per-translation-unit parts of gemm_f16_plan / gemm_f16_destroy, called
// with the plan's device current.  init: kernel attributes and co-resident
// cluster counts; release: device buffers and events of that part.
int gemm_plan_init(gemm_f16_plan_s* p, const cudaDeviceProp& prop);
void gemm_plan_release(gemm_f16_plan_s* p);
int attn_plan_init(gemm_f16_plan_s* p, const cudaDeviceProp& prop);
void attn_plan_release(gemm_f16_plan_s* p);

}  // namespace host
}  // namespace gf16
