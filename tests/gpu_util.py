"""Helpers for the GPU parity tests: move seeded binary16 inputs to the
device, call the C ABI through the binding, bring the result back."""
from __future__ import annotations

import numpy as np

SENTINEL_BITS = 0x7E00  # a binary16 NaN used to detect writes outside C


def to_device(bits: np.ndarray, ld: int | None = None, pad_bits: int = SENTINEL_BITS):
    """binary16 bit matrix -> (padded) CUDA float16 tensor view, row stride ld."""
    import torch
    rows, cols = bits.shape
    ld = (cols + 7) // 8 * 8 if ld is None else ld
    host = np.full((rows, ld), pad_bits, dtype=np.uint16)
    host[:, :cols] = bits
    t = torch.from_numpy(host.view(np.float16)).cuda()
    return t[:, :cols]


def run(plan, A_bits, B_bits, split_k=1, lda=None, ldb=None, ldc=None,
        guard_rows=0, stream=None):
    """Run C = A*B on the GPU.  Returns (C as float64, full C buffer bits).

    The C buffer has ldc columns and guard_rows extra rows, all pre-filled
    with a NaN sentinel, so that writes outside the M x N result show up.
    """
    import torch
    import async_barrier_pipelined_gb300 as g
    M, K = A_bits.shape
    N = B_bits.shape[1]
    A = to_device(A_bits, lda)
    B = to_device(B_bits, ldb)
    ldc = (N + 7) // 8 * 8 if ldc is None else ldc
    cbuf = torch.from_numpy(
        np.full((M + guard_rows, ldc), SENTINEL_BITS, np.uint16).view(np.float16)).cuda()
    C = cbuf[:M, :N]
    s = torch.cuda.current_stream() if stream is None else stream
    g.gemm_f16_run(plan.handle, M, N, K, A.data_ptr(), A.stride(0), B.data_ptr(), B.stride(0),
                   C.data_ptr(), C.stride(0), split_k, int(s.cuda_stream))
    s.synchronize()
    st = plan.status()
    if st != 0:
        raise AssertionError(f"device status {st}: {g.gemm_f16_strerror(st)}")
    full = cbuf.cpu().numpy().view(np.uint16)
    return full[:M, :N].view(np.float16).astype(np.float64), full


def run_layout(plan, A_bits, B_bits, layout, split_k=1, lda=None, ldb=None, ldc=None,
               guard_rows=0):
    """Like run(), for an operand layout: A_bits is M x K and B_bits K x N
    (the logical operands); an operand whose layout bit is set is stored
    transposed on the device (A as K rows of M, B as N rows of K) with row
    stride lda / ldb, and passed to gemm_f16_run_ex."""
    import torch
    import async_barrier_pipelined_gb300 as g
    M, K = A_bits.shape
    N = B_bits.shape[1]
    A = to_device(np.ascontiguousarray(A_bits.T) if layout & g.LAYOUT_TN else A_bits, lda)
    B = to_device(np.ascontiguousarray(B_bits.T) if layout & g.LAYOUT_NT else B_bits, ldb)
    ldc = (N + 7) // 8 * 8 if ldc is None else ldc
    cbuf = torch.from_numpy(
        np.full((M + guard_rows, ldc), SENTINEL_BITS, np.uint16).view(np.float16)).cuda()
    C = cbuf[:M, :N]
    s = torch.cuda.current_stream()
    g.gemm_f16_run_ex(plan.handle, layout, M, N, K, A.data_ptr(), A.stride(0), B.data_ptr(),
                      B.stride(0), C.data_ptr(), C.stride(0), split_k, int(s.cuda_stream))
    s.synchronize()
    st = plan.status()
    if st != 0:
        raise AssertionError(f"device status {st}: {g.gemm_f16_strerror(st)}")
    full = cbuf.cpu().numpy().view(np.uint16)
    return full[:M, :N].view(np.float16).astype(np.float64), full


def assert_untouched_outside(full_bits: np.ndarray, M: int, N: int):
    """Everything outside the M x N result must still be the sentinel."""
    pad_cols = full_bits[:M, N:]
    extra_rows = full_bits[M:, :]
    assert np.all(pad_cols == SENTINEL_BITS), "write past column N"
    assert np.all(extra_rows == SENTINEL_BITS), "write past row M"
