"""GPU tests of the A repack (option GEMM_F16_OPT_A_REPACK).

When A's row pitch is not a multiple of 128 bytes, the library may first
copy A into rows of whole 128-byte lines and run the product on that copy.
The copy moves binary16 values unchanged, so the product must be bit for bit
the one computed from the original A (same kernel, same tiles, same order),
and it must meet the parity criteria of the "Xe2 ESIMD GEMM" page
("Correctness testing") against the FP64 oracle.  The source rows are padded
with a NaN sentinel past K (past M for A stored K x M): a repack that read or
kept anything beyond a row would turn the product into NaN.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
import synthetic_inputs as si
from tests import gpu_util, oracle_cache, parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", params=[1, 2, 3], ids=["cta1", "pair256", "quad"])
def plan(request):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import async_barrier_pipelined_gb300 as g
    from async_barrier_pipelined_gb300 import build
    build.build()
    p = g.Plan(0)
    p.set_option(g.OPT_KERNEL, request.param)
    yield p
    p.set_option(g.OPT_A_REPACK, 0)
    p.close()


def _both(plan, A, B, layout, lda, split_k=1):
    """(product with the repack forced off, product with it forced on, twice)."""
    import async_barrier_pipelined_gb300 as g
    out = []
    for opt in (1, 2, 2):
        plan.set_option(g.OPT_A_REPACK, opt)
        c, full = gpu_util.run_layout(plan, A, B, layout, split_k=split_k, lda=lda,
                                      guard_rows=1)
        gpu_util.assert_untouched_outside(full, A.shape[0], B.shape[1])
        out.append(c)
    plan.set_option(g.OPT_A_REPACK, 0)
    return out


# (M, N, K, split_k); lda is the stored row length rounded up to 8, plus 8 when
# that happens to land on a whole line, so that every pitch is off by 16-112 bytes.
CASES = [(300, 520, 200, 1), (385, 513, 1000, 1), (256, 256, 72, 1), (129, 300, 13, 1),
         (700, 1100, 520, 1), (200, 300, 1000, 3),
         (1000, 1104, 2048, 1)]   # on the pair kernel: a last wave in K halves


def _off_line_ld(cols):
    ld = (cols + 7) // 8 * 8
    return ld + 8 if (ld * 2) % 128 == 0 else ld


@pytest.mark.parametrize("layout", [0, 1], ids=["NN", "TN"])
@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c)))
def test_repack_bit_identical_and_correct(plan, layout, case):
    M, N, K, split = case
    w = si.custom(M, N, K, seed=M + 3 * N + 7 * K + layout)
    A, B = w.pair_bits(0)
    lda = _off_line_ld(M if layout else K)
    assert (lda * 2) % 128 != 0
    never, once, again = _both(plan, A, B, layout, lda, split)
    parity.check(once, oracle.gemm_f16(A, B), f"repacked A {M}x{N}x{K} layout {layout}")
    assert np.array_equal(never.view(np.uint64), once.view(np.uint64))
    assert np.array_equal(once.view(np.uint64), again.view(np.uint64))


def test_repack_grows_and_shrinks_between_shapes(plan):
    """The plan keeps one repack buffer: a larger A grows it, a smaller one
    reuses it; each product is still exact on small-integer inputs."""
    import async_barrier_pipelined_gb300 as g
    rng = np.random.default_rng(5)
    plan.set_option(g.OPT_A_REPACK, 2)
    try:
        for M, N, K in [(130, 140, 60), (520, 300, 1000), (130, 140, 60)]:
            a = rng.integers(-1, 2, size=(M, K)).astype(np.float16)
            b = rng.integers(-1, 2, size=(K, N)).astype(np.float16)
            want = a.astype(np.float64) @ b.astype(np.float64)   # |entries| <= K < 2048: exact
            c, _ = gpu_util.run(plan, a.view(np.uint16), b.view(np.uint16),
                                lda=_off_line_ld(K))
            assert np.array_equal(c, want), (M, N, K)
    finally:
        plan.set_option(g.OPT_A_REPACK, 0)


def test_repack_option_values(plan):
    import async_barrier_pipelined_gb300 as g
    for v in (0, 1, 2):
        plan.set_option(g.OPT_A_REPACK, v)
        assert plan.get_option(g.OPT_A_REPACK) == v
    plan.set_option(g.OPT_A_REPACK, 0)
    with pytest.raises(g.GemmError):
        plan.set_option(g.OPT_A_REPACK, 3)


def test_ragged_workload_auto_repack_matches_plain(plan):
    """4000 x 4104 x 3000 with lda = 3000 (6000-byte rows): on the pair
    kernel the automatic setting repacks A.  Same bits as without the
    repack, and correct on every element against the oracle."""
    import async_barrier_pipelined_gb300 as g
    w = si.WORKLOADS["gemm_ragged"]
    A, B = oracle_cache.gemm_inputs("gemm_ragged")
    plan.set_option(g.OPT_A_REPACK, 1)
    plain, _ = gpu_util.run(plan, A, B, lda=w.K)
    plan.set_option(g.OPT_A_REPACK, 0)
    auto, _ = gpu_util.run(plan, A, B, lda=w.K)
    assert np.array_equal(plain.view(np.uint64), auto.view(np.uint64))
    parity.check(auto, oracle_cache.gemm_ref("gemm_ragged"), "ragged workload")


def test_run_info_reports_the_launches(plan):
    """gemm_f16_run_info names the kernel and counts the launches one call
    enqueues: the product, the split reduction and the repack of A."""
    import async_barrier_pipelined_gb300 as g
    h = plan.handle
    kernel = plan.get_option(g.OPT_KERNEL)
    info = g.gemm_f16_run_info(h, 0, 4000, 4104, 3000, 3000)
    assert info["kernel"] == kernel
    assert info["repack_a"] == (kernel == 2) and info["launches"] == 1 + (kernel == 2)
    assert g.gemm_f16_run_info(h, 0, 4000, 4104, 3000, 3008)["launches"] == 1
    assert g.gemm_f16_run_info(h, 0, 512, 512, 32768, 32768, 16)["launches"] == 2
    plan.set_option(g.OPT_A_REPACK, 2)
    try:
        i2 = g.gemm_f16_run_info(h, 1, 300, 520, 200, 304, 3)   # A stored 200 x 300
        assert i2["repack_a"] and i2["launches"] == 3
        plan.set_option(g.OPT_A_REPACK, 1)
        assert not g.gemm_f16_run_info(h, 0, 4000, 4104, 3000, 3000)["repack_a"]
    finally:
        plan.set_option(g.OPT_A_REPACK, 0)
    assert g.gemm_f16_run_info(h, 0, 128, 128, 128, 128)["tile_width"] in (64, 128, 256)
    with pytest.raises(g.GemmError):
        g.gemm_f16_run_info(h, 0, 128, 128, 128, 100)   # lda < K
    with pytest.raises(g.GemmError):
        g.gemm_f16_run_info(h, 4, 128, 128, 128, 128)


def test_automatic_choice_for_an_off_line_a():
    """The automatic kernel choice for large products whose A rows are off
    128-byte lines: the cluster-of-four kernel on A as it lies when its
    waves of clusters are no more than the pair kernel's waves, else the
    pair kernel after a repack of A; whole-line A keeps the pair kernel.
    The expectations follow the documented rule from the plan's own cluster
    counts, and every product is checked on every element."""
    import math
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import async_barrier_pipelined_gb300 as g
    from async_barrier_pipelined_gb300 import build
    build.build()
    with g.Plan(0) as plan:
        pairs = plan.get_option(g.INFO_MAX_PAIRS)
        quads = plan.get_option(g.INFO_MAX_QUADS)
        if pairs <= 0 or quads <= 0:
            pytest.skip("no clusters of two or four on this device")
        for M, N, K, lda in [(4000, 4104, 3000, 3000), (4864, 2048, 1000, 1000),
                             (2048, 2048, 2048, 2048)]:
            tm = math.ceil(M / 256)
            off_line = (lda * 2) % 128 != 0
            quad_ok = math.ceil(tm * math.ceil(N / 512) / quads) <= math.ceil(tm * math.ceil(N / 256) / pairs)
            want_quad = off_line and quad_ok
            info = g.gemm_f16_run_info(plan.handle, 0, M, N, K, lda)
            assert info["kernel"] == (3 if want_quad else 2), (M, N, K, info)
            assert info["repack_a"] == (off_line and not want_quad), (M, N, K, info)
            if (M, N, K) == (4000, 4104, 3000):
                A, B = oracle_cache.gemm_inputs("gemm_ragged")
                want = oracle_cache.gemm_ref("gemm_ragged")
            else:
                w = si.custom(M, N, K, seed=M + N + K)
                A, B = w.pair_bits(0)
                want = oracle.gemm_f16(A, B)
            c, full = gpu_util.run(plan, A, B, lda=lda, guard_rows=1)
            gpu_util.assert_untouched_outside(full, M, N)
            parity.check(c, want, f"automatic choice {M}x{N}x{K} lda={lda}")
