"""The GEMM and attention entry points inside a captured CUDA graph.

After one run of each shape (which builds and uploads what the run needs:
the CTA-pair work list, grown workspaces, tensor maps), a run enqueues only
kernel launches, so it can be captured into a CUDA graph and replayed.
Replays must give the eager run's bits, and be correct against the FP64
oracle, for the single-CTA kernel, the CTA pair with its K-halves merge, a
split run with its reduction, the A repack, and the attention pair kernel.
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


# (M, N, K, split_k, kernel, lda): what one call enqueues
CASES = [
    (384, 640, 512, 1, 1, None),       # single-CTA kernel
    (1024, 1024, 2048, 1, 2, None),    # pair kernel, last wave in K halves + merge
    (512, 768, 4096, 4, 2, None),      # pair kernel, split partials + reduction
    (2000, 2048, 1000, 1, 2, 1000),    # A repack (2000-byte rows) + pair kernel
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c[:4])) + f"-k{c[4]}")
def test_gemm_replays_from_a_captured_graph(g, case):
    import torch
    M, N, K, split, kernel, lda = case
    w = si.custom(M, N, K, seed=M + N + K + split)
    A_bits, B_bits = w.pair_bits(0)
    want = oracle.gemm_f16(A_bits, B_bits)
    A = gpu_util.to_device(A_bits, lda)
    B = gpu_util.to_device(B_bits)
    with g.Plan(0) as plan:
        plan.set_option(g.OPT_KERNEL, kernel)
        side = torch.cuda.Stream()
        C = torch.empty((M, N), dtype=torch.float16, device="cuda")
        with torch.cuda.stream(side):
            g.matmul(plan, A, B, C=C, split_k=split)      # eager: builds what the run needs
        side.synchronize()
        assert plan.status() == g.OK
        eager = C.cpu().numpy().astype(np.float64)
        parity.check(eager, want, f"eager {case}")
        C.zero_()
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            g.matmul(plan, A, B, C=C, split_k=split)
        for _ in range(2):
            C.zero_()
            graph.replay()
            torch.cuda.synchronize()
            assert plan.status() == g.OK
            got = C.cpu().numpy().astype(np.float64)
            assert np.array_equal(got.view(np.uint64), eager.view(np.uint64)), f"replay {case}"


def test_attention_replays_from_a_captured_graph(g):
    import torch
    w = si.attn_custom(1, 4, 700, 900, seed=17)
    Qb, Kb, Vb = w.bits()
    want = oracle.attention_f16(Qb, Kb, Vb, w.scale)
    Q, K, V = (torch.from_numpy(x.view(np.float16)).cuda() for x in (Qb, Kb, Vb))
    with g.Plan(0) as plan:
        O = torch.empty_like(Q)
        side = torch.cuda.Stream()
        with torch.cuda.stream(side):
            g.attention(plan, Q, K, V, O=O)
        side.synchronize()
        assert plan.status() == g.OK
        eager = O.cpu().numpy().astype(np.float64)
        parity.check(eager, want, "attention eager")
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            g.attention(plan, Q, K, V, O=O)
        for _ in range(2):
            O.zero_()
            graph.replay()
            torch.cuda.synchronize()
            assert plan.status() == g.OK
            got = O.cpu().numpy().astype(np.float64)
            assert np.array_equal(got.view(np.uint64), eager.view(np.uint64)), "attention replay"
