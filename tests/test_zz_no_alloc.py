"""The plan-free, allocation-free entry point gemm_f16_run_noalloc.

Some callers cannot call cudaMalloc: their device memory is owned by another
allocator (a framework's caching pool that has already reserved the free
HBM, so a direct cudaMalloc may fail), or they run in latency-critical loops
where the device-wide synchronisation of cudaMalloc/cudaFree would stall
every other stream.  gemm_f16_run_noalloc serves them from one fixed scratch
array compiled into the library instead of plan-owned buffers.

These tests call it through the C ABI and compare its output with the FP64
oracle (the parity criteria used everywhere else) and with the regular entry
point's (gemm_f16_run with a plan), which runs the same kernels in the same
order and so must agree bit for bit, on two calls in a row, so that a second
call that finds the scratch holding the first call's data still gets it
right.  A call without a status pointer reports through
gemm_f16_noalloc_status.

This file is collected last on purpose; it passes both alone in a fresh
process (where its first call performs the per-device set-up) and after
the other tests.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
import synthetic_inputs as si
from tests import gpu_util, parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def plan():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import async_barrier_pipelined_gb300 as g
    from async_barrier_pipelined_gb300 import build
    build.build()
    p = g.Plan(0)
    # gemm_f16_run_noalloc runs the single-CTA kernel; compare it with the
    # plan entry point running that same kernel.
    p.set_option(g.OPT_KERNEL, 1)
    yield p
    p.close()


def _noalloc(A_bits, B_bits, split_k, status_ptr):
    import torch
    import async_barrier_pipelined_gb300 as g
    M, K = A_bits.shape
    N = B_bits.shape[1]
    A = gpu_util.to_device(A_bits)
    B = gpu_util.to_device(B_bits)
    ldc = (N + 7) // 8 * 8
    cbuf = torch.from_numpy(np.full((M, ldc), gpu_util.SENTINEL_BITS, np.uint16)
                            .view(np.float16)).cuda()
    C = cbuf[:, :N]
    s = torch.cuda.current_stream()
    g.gemm_f16_run_noalloc(M, N, K, A.data_ptr(), A.stride(0), B.data_ptr(), B.stride(0),
                           C.data_ptr(), C.stride(0), split_k, status_ptr,
                           int(s.cuda_stream))
    s.synchronize()
    full = cbuf.cpu().numpy().view(np.uint16)
    return full[:, :N].view(np.float16).astype(np.float64), full


CASES = [
    ("gemm_splitk", None),                                   # 512x512x32768, 16 splits: 16 MiB scratch
    ("split_ragged", si.custom(200, 300, 1000, seed=77, split_k=3)),
    ("no_split_ragged", si.custom(385, 513, 1000, seed=78)),
    ("two_waves", si.custom(2000, 3000, 256, seed=80)),     # 16 x 12 tiles on 152 SMs
]


@pytest.mark.parametrize("name,w", CASES, ids=[c[0] for c in CASES])
def test_noalloc_matches_oracle_and_plan_entry_point_twice(plan, name, w):
    import torch
    w = si.WORKLOADS[name] if w is None else w
    A, B = w.pair_bits(0)
    want = oracle.gemm_f16(A, B)
    ref, _ = gpu_util.run(plan, A, B, split_k=w.split_k)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for call in range(2):
        got, full = _noalloc(A, B, w.split_k, status.data_ptr())
        assert int(status.item()) == 0, f"call {call}: device status {int(status.item())}"
        parity.check(got, want, f"{name} no-alloc call {call} vs oracle")
        assert np.array_equal(got, ref), f"{name} call {call}: not bit-identical to the plan path"
        gpu_util.assert_untouched_outside(full, w.M, w.N)


def test_noalloc_without_status_pointer(plan):
    """status = NULL: the kernel's status goes to the library's own word,
    read (and cleared) by gemm_f16_noalloc_status."""
    import async_barrier_pipelined_gb300 as g
    w = si.custom(300, 600, 700, seed=79, split_k=2)
    A, B = w.pair_bits(0)
    want = oracle.gemm_f16(A, B)
    for call in range(2):
        got, full = _noalloc(A, B, w.split_k, 0)
        assert g.gemm_f16_noalloc_status() == 0
        parity.check(got, want, f"no status pointer, call {call}")
        gpu_util.assert_untouched_outside(full, w.M, w.N)


def test_noalloc_rejects_problems_beyond_its_scratch(plan):
    import torch
    import async_barrier_pipelined_gb300 as g
    buf = torch.empty(16, dtype=torch.float16, device="cuda")
    p = buf.data_ptr()
    # 16 splits x 4096 x 4096 FP32 partials = 1 GiB > 32 MiB of scratch
    with pytest.raises(g.GemmError) as e:
        g.gemm_f16_run_noalloc(4096, 4096, 4096, p, 4096, p, 4096, p, 4096, 16, 0, 0)
    assert e.value.code == g.ERR_SCRATCH_TOO_SMALL
