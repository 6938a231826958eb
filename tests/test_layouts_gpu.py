"""GPU parity of the transposed-operand layouts (gemm_f16_run_ex).

Layout TN stores A as K rows of M, NT stores B as N rows of K, TT both.
The kernels read a transposed operand with the other dimension innermost
and give the tensor core the other major mode, so a wrong descriptor
stride, k-step or box order shows up as a wrong product.  Small-integer
and permutation inputs must come out bit-exact; random inputs follow the
criteria of the "Xe2 ESIMD GEMM" page ("Correctness testing"), as in
test_gemm_gpu.py.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
import synthetic_inputs as si
from tests import gpu_util, oracle_cache, parity

pytestmark = pytest.mark.gpu

LAYOUTS = [0, 1, 2, 3]
LAYOUT_IDS = ["NN", "TN", "NT", "TT"]


@pytest.fixture(scope="module", params=[1, 2, 3], ids=["cta1", "pair256", "quad"])
def plan(request):
    """A plan pinned to the single-CTA kernel (1), the CTA-pair kernel (2) or
    the cluster-of-four kernel (3; row-major layouts only, others run 2)."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import async_barrier_pipelined_gb300 as g
    from async_barrier_pipelined_gb300 import build
    build.build()
    p = g.Plan(0)
    p.set_option(g.OPT_KERNEL, request.param)
    yield p
    p.close()


def _f16(x):
    return np.asarray(x, dtype=np.float64).astype(np.float16).view(np.uint16)


@pytest.mark.parametrize("layout", LAYOUTS, ids=LAYOUT_IDS)
def test_permutations_exact(plan, layout):
    """P * X and Y * Q with permutation matrices P, Q: every output element
    is one input element, so any misplaced row, column or k-slice shows."""
    rng = np.random.default_rng(11 + layout)
    n = 320
    P = _f16(np.eye(n)[rng.permutation(n)])
    Q = _f16(np.eye(n)[rng.permutation(n)])
    X = _f16(rng.integers(-8, 9, (n, 264)))
    Y = _f16(rng.integers(-8, 9, (136, n)))
    to64 = lambda b: b.view(np.float16).astype(np.float64)
    c, _ = gpu_util.run_layout(plan, P, X, layout)
    assert np.array_equal(c, to64(P) @ to64(X))
    c, _ = gpu_util.run_layout(plan, Y, Q, layout)
    assert np.array_equal(c, to64(Y) @ to64(Q))


@pytest.mark.parametrize("layout", LAYOUTS, ids=LAYOUT_IDS)
@pytest.mark.parametrize("shape", [(128, 256, 64), (256, 512, 384), (300, 520, 200),
                                   (129, 257, 1000)], ids=lambda s: "x".join(map(str, s)))
def test_small_integers_bit_exact(plan, layout, shape):
    M, N, K = shape
    rng = np.random.default_rng(M + N + K + layout)
    A = _f16(rng.integers(-2, 3, (M, K)))
    B = _f16(rng.integers(-2, 3, (K, N)))
    c, full = gpu_util.run_layout(plan, A, B, layout, guard_rows=2,
                                  ldc=(N + 7) // 8 * 8 + 8)
    assert np.array_equal(c, oracle.gemm_f16(A, B))
    gpu_util.assert_untouched_outside(full, M, N)


SWEEP = [(1, 1, 1), (7, 9, 13), (33, 65, 17), (127, 255, 63), (200, 300, 100),
         (64, 1000, 72), (1000, 64, 200), (385, 513, 1000)]


@pytest.mark.parametrize("layout", [1, 2, 3], ids=LAYOUT_IDS[1:])
@pytest.mark.parametrize("shape", SWEEP, ids=lambda s: "x".join(map(str, s)))
def test_shape_sweep(plan, layout, shape):
    M, N, K = shape
    w = si.custom(M, N, K, seed=M * 7919 + N * 31 + K + layout)
    A, B = w.pair_bits(0)
    c, full = gpu_util.run_layout(plan, A, B, layout, guard_rows=2,
                                  ldc=(N + 7) // 8 * 8 + 8)
    parity.check(c, oracle.gemm_f16(A, B), f"layout {layout} {M}x{N}x{K}")
    gpu_util.assert_untouched_outside(full, M, N)


@pytest.mark.parametrize("layout", [1, 2, 3], ids=LAYOUT_IDS[1:])
def test_strided_transposed_operands(plan, layout):
    """Leading dimensions above the stored row length; the padding is NaN."""
    M, N, K = 257, 300, 520
    w = si.custom(M, N, K, seed=77 + layout)
    A, B = w.pair_bits(0)
    lda = ((M if layout & 1 else K) + 7) // 8 * 8 + 24
    ldb = ((K if layout & 2 else N) + 7) // 8 * 8 + 40
    c, full = gpu_util.run_layout(plan, A, B, layout, lda=lda, ldb=ldb,
                                  ldc=(N + 7) // 8 * 8 + 16, guard_rows=1)
    parity.check(c, oracle.gemm_f16(A, B), f"strided layout {layout}")
    gpu_util.assert_untouched_outside(full, M, N)


@pytest.mark.parametrize("layout", [1, 2, 3], ids=LAYOUT_IDS[1:])
@pytest.mark.parametrize("shape,split", [((256, 256, 256), 4), ((200, 300, 1000), 3),
                                         ((130, 520, 4096), 16)])
def test_split_k_layouts_match_nn_bitwise(plan, layout, shape, split):
    """Same partial sums in the same order whatever the storage: a split
    run in any layout equals the NN run bit for bit, and is correct."""
    M, N, K = shape
    w = si.custom(M, N, K, seed=K + split)
    A, B = w.pair_bits(0)
    c0, _ = gpu_util.run_layout(plan, A, B, 0, split_k=split)
    c1, _ = gpu_util.run_layout(plan, A, B, layout, split_k=split)
    parity.check(c1, oracle.gemm_f16(A, B), f"split {split} layout {layout}")
    assert np.array_equal(c0.view(np.uint64), c1.view(np.uint64))


def test_gemm_4096_tt_full(plan):
    """The 4096^3 workload with both operands stored transposed, every
    element against the oracle."""
    A, B = oracle_cache.gemm_inputs("gemm_4096", 1)
    c, _ = gpu_util.run_layout(plan, A, B, 3)
    parity.check(c, oracle_cache.gemm_ref("gemm_4096", 1), "gemm_4096 TT")


def test_matmul_takes_transposed_views(plan):
    """matmul passes A.t() / B.t() views as layouts TN / NT, no copies."""
    import torch
    import async_barrier_pipelined_gb300 as g
    w = si.custom(200, 264, 136, seed=3)
    A, B = w.pair_bits(0)
    want = oracle.gemm_f16(A, B)
    At = gpu_util.to_device(np.ascontiguousarray(A.T))        # K x M storage
    Bt = gpu_util.to_device(np.ascontiguousarray(B.T))        # N x K storage
    An, Bn = gpu_util.to_device(A), gpu_util.to_device(B)
    for a, b in ((An, Bn), (At.t(), Bn), (An, Bt.t()), (At.t(), Bt.t())):
        c = g.matmul(plan, a, b)
        torch.cuda.synchronize()
        assert plan.status() == g.OK
        parity.check(c.cpu().numpy().astype(np.float64), want, "matmul view")
