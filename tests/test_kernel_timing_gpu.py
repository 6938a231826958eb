"""Kernel timing records (GEMM_F16_OPT_KERNEL_TIMING, gemm_f16_kernel_time).

With the option on, each GEMM call records a CUDA event pair around its
product kernel (not the repack, the K-halves merge or the split reduction)
and each attention call around its attention kernel; the getter returns the
summed durations and the number of launches, then forgets them.  The
records must not change any result, must not be taken while the stream is
being captured into a graph, and cost nothing when the option is off.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
import synthetic_inputs as si
from tests import gpu_util, parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def g():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import async_barrier_pipelined_gb300 as g
    from async_barrier_pipelined_gb300 import build
    build.build()
    return g


# (M, N, K, split_k, kernel): single CTA, pair with a K-halved last wave and
# its merge, pair with split partials and the reduction, cluster of four
CASES = [(384, 640, 512, 1, 1), (1024, 1024, 2048, 1, 2), (512, 768, 4096, 4, 2),
         (700, 1296, 1000, 1, 3)]


def test_off_by_default_records_nothing(g):
    w = si.custom(256, 384, 320, seed=5)
    A_bits, B_bits = w.pair_bits(0)
    with g.Plan(0) as plan:
        assert plan.get_option(g.OPT_KERNEL_TIMING) == 0
        gpu_util.run(plan, A_bits, B_bits)
        assert plan.kernel_time() == (0.0, 0)


def test_one_record_per_product_kernel_and_results_unchanged(g):
    with g.Plan(0) as plan:
        plan.set_option(g.OPT_KERNEL_TIMING, 1)
        for M, N, K, split, kernel in CASES:
            w = si.custom(M, N, K, seed=M + N + K)
            A_bits, B_bits = w.pair_bits(0)
            plan.set_option(g.OPT_KERNEL, kernel)
            got, _ = gpu_util.run(plan, A_bits, B_bits, split_k=split)
            parity.check(got, oracle.gemm_f16(A_bits, B_bits), f"{M}x{N}x{K}/{split} k{kernel}")
            ms, n = plan.kernel_time()
            assert n == 1, (M, N, K, split, kernel, n)
            assert 0.0 < ms < 1000.0
            assert plan.kernel_time() == (0.0, 0)        # read once, then forgotten


def test_attention_records_its_kernel(g):
    import torch
    w = si.attn_custom(1, 4, 700, 900, seed=17)
    Qb, Kb, Vb = w.bits()
    Q, K, V = (torch.from_numpy(x.view(np.float16)).cuda() for x in (Qb, Kb, Vb))
    with g.Plan(0) as plan:
        plan.set_option(g.OPT_KERNEL_TIMING, 1)
        for kernel in (1, 2):
            plan.set_option(g.OPT_ATTN_KERNEL, kernel)
            O = g.attention(plan, Q, K, V)
            torch.cuda.synchronize()
            assert plan.status() == g.OK
            parity.check(O.cpu().numpy().astype(np.float64),
                         oracle.attention_f16(Qb, Kb, Vb, w.scale), f"attention k{kernel}")
        ms, n = plan.kernel_time()
        assert n == 2 and ms > 0.0


def test_many_launches_sum_and_count(g):
    import torch
    M = N = K = 512
    w = si.custom(M, N, K, seed=3)
    A_bits, B_bits = w.pair_bits(0)
    A, B = gpu_util.to_device(A_bits), gpu_util.to_device(B_bits)
    C = torch.empty((M, N), dtype=torch.float16, device="cuda")
    with g.Plan(0) as plan:
        plan.set_option(g.OPT_KERNEL_TIMING, 1)
        for _ in range(50):
            g.matmul(plan, A, B, C=C)
        plan.set_option(g.OPT_KERNEL_TIMING, 0)
        for _ in range(5):
            g.matmul(plan, A, B, C=C)                # not recorded
        ms, n = plan.kernel_time()
        assert n == 50
        assert 0.0 < ms / n < 1.0                    # a 512^3 product takes microseconds
        torch.cuda.synchronize()
        assert plan.status() == g.OK


def test_nothing_recorded_under_graph_capture(g):
    import torch
    M, N, K = 384, 640, 512
    w = si.custom(M, N, K, seed=9)
    A_bits, B_bits = w.pair_bits(0)
    A, B = gpu_util.to_device(A_bits), gpu_util.to_device(B_bits)
    C = torch.empty((M, N), dtype=torch.float16, device="cuda")
    with g.Plan(0) as plan:
        side = torch.cuda.Stream()
        with torch.cuda.stream(side):
            g.matmul(plan, A, B, C=C)                # builds what the run needs
        side.synchronize()
        plan.set_option(g.OPT_KERNEL_TIMING, 1)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            g.matmul(plan, A, B, C=C)
        C.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert plan.kernel_time() == (0.0, 0)
        parity.check(C.cpu().numpy().astype(np.float64), oracle.gemm_f16(A_bits, B_bits),
                     "graph replay with timing on")


def test_option_values(g):
    with g.Plan(0) as plan:
        for bad in (-1, 2):
            with pytest.raises(g.GemmError):
                plan.set_option(g.OPT_KERNEL_TIMING, bad)
        plan.set_option(g.OPT_KERNEL_TIMING, 1)
        assert plan.get_option(g.OPT_KERNEL_TIMING) == 1


def test_layout_and_host_entry_points_record_their_product(g):
    import torch
    M, N, K = 640, 384, 704
    w = si.custom(M, N, K, seed=21)
    A_bits, B_bits = w.pair_bits(0)
    want = oracle.gemm_f16(A_bits, B_bits)
    with g.Plan(0) as plan:
        plan.set_option(g.OPT_KERNEL_TIMING, 1)
        # transposed A and B through gemm_f16_run_ex (matmul passes .t() views)
        A = gpu_util.to_device(np.ascontiguousarray(A_bits.T)).t()
        B = gpu_util.to_device(np.ascontiguousarray(B_bits.T)).t()
        C = g.matmul(plan, A, B)
        torch.cuda.synchronize()
        parity.check(C.cpu().numpy().astype(np.float64), want, "TT with timing on")
        ms, n = plan.kernel_time()
        assert n == 1 and ms > 0.0
        # host operands: the copies are not timed, the product is
        hA = torch.from_numpy(A_bits.view(np.float16)).pin_memory()
        hB = torch.from_numpy(B_bits.view(np.float16)).pin_memory()
        hC = torch.empty((M, N), dtype=torch.float16).pin_memory()
        s = torch.cuda.current_stream()
        for _ in range(3):
            g.gemm_f16_run_host(plan.handle, M, N, K, hA.data_ptr(), K, hB.data_ptr(), N,
                                hC.data_ptr(), N, 1, int(s.cuda_stream))
        s.synchronize()
        assert plan.status() == g.OK
        parity.check(hC.numpy().astype(np.float64), want, "host operands with timing on")
        ms, n = plan.kernel_time()
        assert n == 3 and ms > 0.0
