"""GPU parity: the CUDA path through the C ABI against the FP64 oracle.

Criteria ("Xe2 ESIMD GEMM" page, "Correctness testing"): no NaN/Inf in the
output, checked first; relative RMS error < 0.5%; and every element within
1e-2 * (|ref| + 1).  Small-integer inputs whose exact products fit binary16
must come out bit-exact (they localise layout and descriptor errors).
Split runs must be bitwise reproducible.
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
    """A plan pinned to one kernel: 1 = single-CTA, 2 = CTA pair with
    256-wide tiles, 3 = two CTA pairs in a cluster of four sharing A by
    multicast.  Every test in this file runs once per kernel."""
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


def _small_int_bits(rng, shape, lo=-2, hi=3):
    return _f16(rng.integers(lo, hi, size=shape))


# ---------------------------------------------------------------- exact cases
def test_identity_single_tile(plan):
    rng = np.random.default_rng(1)
    A = _small_int_bits(rng, (128, 64), -8, 9)
    c, _ = gpu_util.run(plan, A, _f16(np.eye(64)))
    assert np.array_equal(c, A.view(np.float16).astype(np.float64))


def test_identity_left_multi_tile(plan):
    rng = np.random.default_rng(2)
    B = _small_int_bits(rng, (256, 512), -8, 9)
    c, _ = gpu_util.run(plan, _f16(np.eye(256)), B)
    assert np.array_equal(c, B.view(np.float16).astype(np.float64))


def test_permutations_exact(plan):
    rng = np.random.default_rng(3)
    m, k, n = 256, 192, 320
    A = _small_int_bits(rng, (m, k), -8, 9)
    pc = rng.permutation(k)
    Q = np.zeros((k, k))
    Q[pc, np.arange(k)] = 1.0
    c, _ = gpu_util.run(plan, A, _f16(Q))
    assert np.array_equal(c, A.view(np.float16).astype(np.float64)[:, pc])


@pytest.mark.parametrize("shape", [(128, 256, 64), (256, 256, 256), (384, 512, 320),
                                   (300, 700, 200)])
def test_small_integers_bit_exact(plan, shape):
    """Entries in {-2..2}: |R| <= 4K <= 2048 is exact in FP32 and binary16."""
    M, N, K = shape
    rng = np.random.default_rng(M + N + K)
    A = _small_int_bits(rng, (M, K))
    B = _small_int_bits(rng, (K, N))
    c, full = gpu_util.run(plan, A, B, guard_rows=3, ldc=(N + 7) // 8 * 8 + 8)
    assert np.array_equal(c, oracle.gemm_f16(A, B))
    gpu_util.assert_untouched_outside(full, M, N)


# ---------------------------------------------------------------- workloads
def test_gemm_256(plan):
    w = si.WORKLOADS["gemm_256"]
    A, B = w.pair_bits(0)
    c, _ = gpu_util.run(plan, A, B)
    parity.check(c, oracle.gemm_f16(A, B), "gemm_256")


def test_gemm_1024(plan):
    w = si.WORKLOADS["gemm_1024"]
    A, B = w.pair_bits(0)
    c, _ = gpu_util.run(plan, A, B)
    parity.check(c, oracle.gemm_f16(A, B), "gemm_1024")


def test_gemm_4096_pairs_full(plan):
    """Full 4096^3 in the benchmark's launch configuration, two of the eight
    rotating pairs (the first and the last), every element against the
    oracle."""
    for p in (0, 7):
        A, B = oracle_cache.gemm_inputs("gemm_4096", p)
        c, _ = gpu_util.run(plan, A, B)
        parity.check(c, oracle_cache.gemm_ref("gemm_4096", p), f"gemm_4096 pair {p}")


def test_gemm_ragged_full(plan):
    """4000 x 4104 x 3000 (ragged in M, N and K), every element."""
    w = si.WORKLOADS["gemm_ragged"]
    A, B = oracle_cache.gemm_inputs("gemm_ragged")
    c, full = gpu_util.run(plan, A, B, guard_rows=5, ldc=w.N + 8)
    parity.check(c, oracle_cache.gemm_ref("gemm_ragged"), "gemm_ragged")
    gpu_util.assert_untouched_outside(full, w.M, w.N)


def test_gemm_splitk_full_and_reproducible(plan):
    w = si.WORKLOADS["gemm_splitk"]
    A, B = w.pair_bits(0)
    ref = oracle.gemm_f16(A, B)
    c0, full0 = gpu_util.run(plan, A, B, split_k=w.split_k)
    parity.check(c0, ref, "gemm_splitk")
    for _ in range(10):
        _, full = gpu_util.run(plan, A, B, split_k=w.split_k)
        assert np.array_equal(full, full0)
    # and on a freshly created plan (new workspace, new tile tables)
    import async_barrier_pipelined_gb300 as g
    with g.Plan(0) as fresh:
        fresh.set_option(g.OPT_KERNEL, plan.get_option(g.OPT_KERNEL))
        _, full = gpu_util.run(fresh, A, B, split_k=w.split_k)
    assert np.array_equal(full, full0)


# ---------------------------------------------------------------- shape sweep
SWEEP = [
    (1, 1, 1), (1, 8, 8), (8, 1, 16), (7, 9, 13), (16, 16, 16), (33, 65, 17),
    (127, 255, 63), (129, 257, 65), (128, 256, 64), (200, 300, 100),
    (64, 1000, 72), (1000, 64, 200), (385, 513, 1000), (256, 264, 8),
    # extreme aspect ratios at larger sizes: one row across nine column
    # tiles of the cluster-of-four kernel, eight columns down many row
    # tiles, K = 1, long K on thin outputs, a K one past a k-block
    (1, 4104, 3000), (4000, 8, 3000), (2048, 2048, 1), (3, 1030, 4100),
    (1030, 24, 4100), (520, 1536, 65),
]


@pytest.mark.parametrize("shape", SWEEP, ids=lambda s: "x".join(map(str, s)))
def test_shape_sweep(plan, shape):
    M, N, K = shape
    w = si.custom(M, N, K, seed=M * 7919 + N * 31 + K)
    A, B = w.pair_bits(0)
    c, full = gpu_util.run(plan, A, B, guard_rows=2, ldc=(N + 7) // 8 * 8 + 8)
    parity.check(c, oracle.gemm_f16(A, B), f"{M}x{N}x{K}")
    gpu_util.assert_untouched_outside(full, M, N)


@pytest.mark.parametrize("shape", [(100, 130, 70), (257, 300, 1000)])
def test_strided_operands(plan, shape):
    """lda, ldb, ldc larger than the matrix; the padding holds NaN."""
    M, N, K = shape
    w = si.custom(M, N, K, seed=5)
    A, B = w.pair_bits(0)
    lda = (K + 7) // 8 * 8 + 24
    ldb = (N + 7) // 8 * 8 + 40
    c, full = gpu_util.run(plan, A, B, lda=lda, ldb=ldb, ldc=(N + 7) // 8 * 8 + 16,
                           guard_rows=1)
    parity.check(c, oracle.gemm_f16(A, B), "strided")
    gpu_util.assert_untouched_outside(full, M, N)


@pytest.mark.parametrize("shape,split", [((256, 256, 256), 2), ((256, 256, 256), 4),
                                         ((200, 300, 1000), 3), ((129, 40, 640), 10),
                                         ((1, 1, 128), 2), ((130, 520, 4096), 64)])
def test_split_k_sweep(plan, shape, split):
    M, N, K = shape
    w = si.custom(M, N, K, seed=K + split)
    A, B = w.pair_bits(0)
    c, full = gpu_util.run(plan, A, B, split_k=split, guard_rows=2,
                           ldc=(N + 7) // 8 * 8 + 8)
    parity.check(c, oracle.gemm_f16(A, B), f"split {split}")
    gpu_util.assert_untouched_outside(full, M, N)
    _, full2 = gpu_util.run(plan, A, B, split_k=split, guard_rows=2, ldc=(N + 7) // 8 * 8 + 8)
    assert np.array_equal(full, full2)


def test_row_major_tile_order_same_result(plan):
    import async_barrier_pipelined_gb300 as g
    w = si.custom(700, 900, 300, seed=9)
    A, B = w.pair_bits(0)
    c0, _ = gpu_util.run(plan, A, B)
    plan.set_option(g.OPT_TILE_ORDER, 1)
    try:
        c1, _ = gpu_util.run(plan, A, B)
    finally:
        plan.set_option(g.OPT_TILE_ORDER, 0)
    assert np.array_equal(c0, c1)


def test_run_host_matches_device_path(plan):
    import torch
    import async_barrier_pipelined_gb300 as g
    w = si.custom(300, 260, 200, seed=21)
    A, B = w.pair_bits(0)
    c_dev, _ = gpu_util.run(plan, A, B)
    hA = torch.from_numpy(A.view(np.float16)).pin_memory()
    hB = torch.from_numpy(B.view(np.float16)).pin_memory()
    hC = torch.empty((w.M, w.N), dtype=torch.float16).pin_memory()
    s = torch.cuda.current_stream()
    g.gemm_f16_run_host(plan.handle, w.M, w.N, w.K, hA.data_ptr(), w.K, hB.data_ptr(), w.N,
                        hC.data_ptr(), w.N, 1, int(s.cuda_stream))
    s.synchronize()
    assert plan.status() == 0
    assert np.array_equal(hC.numpy().astype(np.float64), c_dev)


def test_invalid_arguments_enqueue_nothing(plan):
    import torch
    import async_barrier_pipelined_gb300 as g
    A = torch.zeros((64, 64), dtype=torch.float16, device="cuda")
    with pytest.raises(g.GemmError) as e:
        g.gemm_f16_run(plan.handle, 64, 64, 64, A.data_ptr() + 2, 64, A.data_ptr(), 64,
                       A.data_ptr(), 64, 1, 0)
    assert e.value.code == g.ERR_MISALIGNED
    with pytest.raises(g.GemmError) as e:
        g.gemm_f16_run(plan.handle, 64, 64, 64, A.data_ptr(), 64, A.data_ptr(), 64,
                       A.data_ptr(), 64, 2, 0)
    assert e.value.code == g.ERR_INVALID_ARG


def test_kernels_agree(plan):
    """The other kernel on the same inputs agrees within the parity bounds."""
    import async_barrier_pipelined_gb300 as g
    w = si.custom(1000, 1300, 700, seed=31)
    A, B = w.pair_bits(0)
    c0, _ = gpu_util.run(plan, A, B)
    mine = plan.get_option(g.OPT_KERNEL)
    plan.set_option(g.OPT_KERNEL, 2 if mine == 1 else 1)
    try:
        c1, _ = gpu_util.run(plan, A, B)
    finally:
        plan.set_option(g.OPT_KERNEL, mine)
    parity.check(c1, c0, "kernel 1 vs kernel 2")


@pytest.mark.parametrize("width", [64, 128, 256])
@pytest.mark.parametrize("shape,split", [((300, 700, 200), 1), ((129, 257, 1000), 3),
                                         ((1000, 64, 72), 1)])
def test_single_cta_tile_widths(plan, width, shape, split):
    """Every tile width of the single-CTA kernel (and its ring depth) against
    the oracle; the pair kernel ignores the option."""
    import async_barrier_pipelined_gb300 as g
    M, N, K = shape
    w = si.custom(M, N, K, seed=width + M)
    A, B = w.pair_bits(0)
    plan.set_option(g.OPT_TILE_WIDTH, width)
    try:
        c, full = gpu_util.run(plan, A, B, split_k=split, guard_rows=1, ldc=(N + 7) // 8 * 8 + 8)
    finally:
        plan.set_option(g.OPT_TILE_WIDTH, 0)
    parity.check(c, oracle.gemm_f16(A, B), f"width {width}")
    gpu_util.assert_untouched_outside(full, M, N)


def test_run_host_back_to_back_calls(plan):
    """Consecutive run_host calls overlap (input copies of call i+1 during the
    product of call i, two alternating device slots): every result must still
    be its own product, including when a slot grows mid-sequence."""
    import torch
    import async_barrier_pipelined_gb300 as g
    shapes = [(300, 260, 200), (300, 260, 200), (520, 300, 330), (300, 260, 200),
              (129, 64, 1000), (520, 300, 330)]
    s = torch.cuda.current_stream()
    side = torch.cuda.Stream()
    jobs = []
    for t, (M, N, K) in enumerate(shapes):
        w = si.custom(M, N, K, seed=100 + t)
        A, B = w.pair_bits(0)
        hA = torch.from_numpy(A.view(np.float16)).pin_memory()
        hB = torch.from_numpy(B.view(np.float16)).pin_memory()
        hC = torch.full((M, N), float("nan"), dtype=torch.float16).pin_memory()
        # Call 2 runs on another stream, ordered between its neighbours; call
        # 4 reuses its slot (without growing it) and must not overwrite that
        # slot's C before call 2's result copy there has finished.
        st = side if t == 2 else s
        if t == 2:
            side.wait_stream(s)
        g.gemm_f16_run_host(plan.handle, M, N, K, hA.data_ptr(), K, hB.data_ptr(), N,
                            hC.data_ptr(), N, 1, int(st.cuda_stream))
        if t == 2:
            s.wait_stream(side)
        jobs.append((A, B, hA, hB, hC))
    torch.cuda.synchronize()
    assert plan.status() == 0
    for A, B, _, _, hC in jobs:
        parity.check(hC.numpy().astype(np.float64), oracle.gemm_f16(A, B), "run_host chain")


@pytest.mark.parametrize("shape", [(1024, 1024, 2048), (300, 600, 2048), (1300, 1024, 2048),
                                   (256, 256, 2048)])
def test_tail_k_halves_exact_and_repeatable(plan, shape):
    """With one split, the pair kernel runs the tiles of a partial last wave
    as two K halves whose FP32 values a second kernel adds (P0 + P1).
    Small-integer products stay exact; random inputs meet the parity bounds
    and repeat bit for bit, also on fewer SMs (the halves are planned for
    the device, not for the launch).  The other kernels run the same checks."""
    import async_barrier_pipelined_gb300 as g
    M, N, K = shape
    if plan.get_option(g.OPT_KERNEL) == 2:
        _, parts = g.gemm_f16_pair_tiles(M, N, plan.get_option(g.INFO_MAX_PAIRS), 1, K=K,
                                         with_parts=True)
        assert parts == 2
        assert g.gemm_f16_run_info(plan.handle, 0, M, N, K, K)["launches"] == 2
    rng = np.random.default_rng(M + N + K)
    A = _small_int_bits(rng, (M, K), -1, 2)
    B = _small_int_bits(rng, (K, N), -1, 2)
    c, full = gpu_util.run(plan, A, B, guard_rows=1, ldc=(N + 7) // 8 * 8 + 8)
    assert np.array_equal(c, oracle.gemm_f16(A, B))      # |entries| <= K < 2^24, |C| < 2048
    gpu_util.assert_untouched_outside(full, M, N)
    w = si.custom(M, N, K, seed=K + 5)
    A, B = w.pair_bits(0)
    outs = []
    try:
        for limit in (0, 0, 24, 8):
            plan.set_option(g.OPT_SM_LIMIT, limit)
            outs.append(gpu_util.run(plan, A, B)[0])
    finally:
        plan.set_option(g.OPT_SM_LIMIT, 0)
    parity.check(outs[0], oracle.gemm_f16(A, B), f"tail halves {shape}")
    for o in outs[1:]:
        assert np.array_equal(o.view(np.uint64), outs[0].view(np.uint64))


def _random_cases(n, seed):
    """Seeded random products: sizes from 1 up to ~1300 (several tiles of
    every kernel, with ragged edges), K up to ~2300, split_k up to 6, and
    operand / output strides padded by 0-120 elements (multiples of 8)."""
    rng = np.random.default_rng(seed)
    cases = []
    for _ in range(n):
        M = int(rng.integers(1, 1300))
        N = int(rng.integers(1, 1300))
        K = int(rng.integers(1, 2300))
        kb = (K + 63) // 64
        split = int(rng.integers(1, min(6, kb) + 1))
        pad = [int(rng.integers(0, 16)) * 8 for _ in range(3)]
        cases.append((M, N, K, split, pad))
    return cases


@pytest.mark.parametrize("case", _random_cases(24, 2024),
                         ids=lambda c: "x".join(map(str, c[:4])) + "-p" + "_".join(map(str, c[4])))
def test_random_shapes_against_oracle(plan, case):
    """Random shapes, splits and padded strides, every element against the
    oracle, with NaN sentinels around C and in the operands' padding."""
    M, N, K, split, (pa, pb, pc) = case
    w = si.custom(M, N, K, seed=M * 7 + N * 13 + K)
    A, B = w.pair_bits(0)
    lda = (K + 7) // 8 * 8 + pa
    ldb = (N + 7) // 8 * 8 + pb
    ldc = (N + 7) // 8 * 8 + pc
    c, full = gpu_util.run(plan, A, B, split_k=split, lda=lda, ldb=ldb, ldc=ldc, guard_rows=1)
    gpu_util.assert_untouched_outside(full, M, N)
    parity.check(c, oracle.gemm_f16(A, B), f"random {case}")
