"""Failure detection on the GPU without a GPU fault.

Every barrier wait in the kernels is bounded.  The test-only plan option
GEMM_F16_OPT_FAULT_UNIT makes the producer of one work unit expect a stage's
bytes but issue no copy for it, so that stage's barrier phase never
completes and the MMA role's wait must run out.  No copy is left in flight
and no memory is touched that a normal run would not touch.  The kernel
must then record GEMM_F16_ERR_TIMEOUT in the plan's status word, free its
tensor memory and return; the next run on the same context must be correct.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from tests import gpu_util

pytestmark = pytest.mark.gpu


def _f16(x):
    return np.asarray(x, dtype=np.float64).astype(np.float16).view(np.uint16)


@pytest.mark.parametrize("kernel", [1, 2, 3], ids=["cta1", "pair256", "quad"])
def test_bounded_wait_reports_timeout_and_context_survives(kernel):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import async_barrier_pipelined_gb300 as g
    from async_barrier_pipelined_gb300 import build
    build.build()
    rng = np.random.default_rng(5)
    M = N = K = 256
    A = _f16(rng.integers(-2, 3, (M, K)))
    B = _f16(rng.integers(-2, 3, (K, N)))
    want = oracle.gemm_f16(A, B)
    with g.Plan(0) as plan:
        plan.set_option(g.OPT_KERNEL, kernel)
        plan.set_option(g.OPT_TIMEOUT_NS, 20_000_000)      # 20 ms per wait
        plan.set_option(g.OPT_FAULT_UNIT, 0)
        At, Bt = gpu_util.to_device(A), gpu_util.to_device(B)
        C = torch.zeros((M, N), dtype=torch.float16, device="cuda")
        s = torch.cuda.current_stream()
        g.gemm_f16_run(plan.handle, M, N, K, At.data_ptr(), K, Bt.data_ptr(), N,
                       C.data_ptr(), N, 1, int(s.cuda_stream))
        s.synchronize()                                     # returns: the waits are bounded
        assert plan.status() == g.ERR_TIMEOUT
        assert plan.status() == g.OK                        # read-and-clear

        plan.set_option(g.OPT_FAULT_UNIT, -1)
        for _ in range(2):                                  # the context and TMEM are fine
            c, _ = gpu_util.run(plan, A, B)
            assert np.array_equal(c, want)
            assert plan.status() == g.OK


@pytest.mark.parametrize("kernel", [1, 2], ids=["cta1", "pair"])
def test_attention_bounded_wait_reports_timeout_and_context_survives(kernel):
    """The attention kernels: the first key tile of CTA (or CTA pair) 1 gets
    no copy, so the MMA thread's wait runs out; the run must return with
    ERR_TIMEOUT and the next run on the same context must be correct."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import async_barrier_pipelined_gb300 as g
    import synthetic_inputs as si
    from tests import parity
    from async_barrier_pipelined_gb300 import build
    build.build()
    w = si.attn_custom(1, 2, 512, 300, seed=9)
    Qb, Kb, Vb = w.bits()
    Q, K, V = (torch.from_numpy(x.view(np.float16)).cuda() for x in (Qb, Kb, Vb))
    with g.Plan(0) as plan:
        plan.set_option(g.OPT_ATTN_KERNEL, kernel)
        plan.set_option(g.OPT_TIMEOUT_NS, 20_000_000)
        plan.set_option(g.OPT_FAULT_UNIT, 1)
        g.attention(plan, Q, K, V)
        torch.cuda.synchronize()
        assert plan.status() == g.ERR_TIMEOUT
        assert plan.status() == g.OK
        plan.set_option(g.OPT_FAULT_UNIT, -1)
        want = oracle.attention_f16(Qb, Kb, Vb, w.scale)
        for _ in range(2):
            O = g.attention(plan, Q, K, V)
            torch.cuda.synchronize()
            assert plan.status() == g.OK
            parity.check(O.cpu().numpy().astype(np.float64), want, "after timeout")
