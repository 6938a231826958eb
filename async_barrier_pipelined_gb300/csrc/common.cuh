// Device helpers shared by the GEMM and attention kernels: the tcgen05
// descriptor builders and the bounded wait used while draining.
//
// The descriptor bit layouts follow the public PTX ISA description of
// tcgen05.mma (instruction descriptor of kind::f16; shared-memory matrix
// descriptor).
#pragma once

#include <stdint.h>

#include "ptx.cuh"

namespace gf16 {

// Instruction descriptor of tcgen05.mma kind::f16: D FP32 (bits 4-5 = 1),
// A and B FP16 (bits 7-9, 10-12 = 0), A K-major (bit 15 = 0), B MN-major
// (bit 16 = 1, row-major B is N-contiguous), N >> 3 at bits 17-22,
// M >> 4 at bits 24-28.
__host__ __device__ constexpr uint32_t make_idesc(int m, int n) {
  return (1u << 4) | (0u << 7) | (0u << 10) | (0u << 15) | (1u << 16) |
         ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

// Shared-memory matrix descriptor (tcgen05): start address >> 4 (bits 0-13),
// leading byte offset >> 4 (16-29), stride byte offset >> 4 (32-45), fixed
// 0b001 at bits 46-48, base offset 0, swizzle mode 2 = 128-byte (bits 61-63).
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// Bounded wait used while draining after an abort (ignores the abort flag):
// true once the phase of parity `parity` of the barrier at shared address
// `bar` has completed, false after `limit_ns` nanoseconds.
static __device__ __noinline__ bool wait_drain(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = ptx::globaltimer();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (ptx::globaltimer() - t0 > limit_ns) return false;
  }
  return true;
}

}  // namespace gf16
