"""Pins for the FP64 oracle: checks against things other than the oracle.

Each test ties the oracle to a fact fixed by the mathematics or by an
independent implementation, so that a plausible slip in it (a dropped term, a
wrong sign or index, a transposed operand, a stride mix-up, a bad binary16
decode) fails at least one of them:

* binary16 widening vs numpy's own float16 -> float64 conversion, all 65536
  bit patterns (independent library routine);
* hand-worked products from tests/golden/ (worked on paper);
* identity and permutation matrices (exact);
* rank-1 closed form R = K * u_i * v_j (exact);
* brute force in exact rational arithmetic for every M, N, K <= 8
  (exact equality on a narrow exponent range, the recursive-summation error
  bound on the full binary16 range including subnormals);
* the transpose identity (B^T A^T)^T = A B, bit for bit (same k order);
* linearity in A, to FP64 round-off;
* strided operands whose padding holds NaN (a stride slip shows as NaN);
* empty sums and empty shapes.
"""
from __future__ import annotations

import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from tests import parity

GOLDEN = os.path.join(os.path.dirname(__file__), "golden",
                      "hand_worked_products.txt")


def _f16(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float64).astype(np.float16).view(np.uint16)


def _rand_f16_bits(rng, shape, lo_exp=-4, hi_exp=4):
    """Random finite binary16 values with exponents in [lo_exp, hi_exp)."""
    mant = rng.integers(1024, 2048, size=shape).astype(np.float64)
    e = rng.integers(lo_exp, hi_exp, size=shape)
    sign = rng.choice([-1.0, 1.0], size=shape)
    return _f16(sign * np.ldexp(mant / 1024.0, e))


def _rand_any_finite_f16_bits(rng, shape):
    """Random finite binary16 patterns over the whole range, incl. subnormals."""
    bits = rng.integers(0, 1 << 16, size=shape, dtype=np.uint32).astype(np.uint16)
    exp = (bits >> 10) & 0x1F
    bits[exp == 31] &= 0xBBFF  # turn inf/NaN patterns into finite ones
    return bits


def _exact(A_bits, B_bits):
    """Exact rational product via Fractions over the binary16 values."""
    a = A_bits.view(np.float16).astype(np.float64)
    b = B_bits.view(np.float16).astype(np.float64)
    M, K = a.shape
    N = b.shape[1]
    fa = [[Fraction(float(a[i, k])) for k in range(K)] for i in range(M)]
    fb = [[Fraction(float(b[k, j])) for j in range(N)] for k in range(K)]
    return [[sum((fa[i][k] * fb[k][j] for k in range(K)), Fraction(0))
             for j in range(N)] for i in range(M)]


# --------------------------------------------------------------------------
def test_widening_matches_numpy_for_every_bit_pattern():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ours = oracle.widen_f16(bits)
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    # signed zeros and infinities keep their sign
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(ref[~nan]))
    assert oracle.f16_to_f64_scalar(0x0001) == 2.0 ** -24  # smallest subnormal
    assert oracle.f16_to_f64_scalar(0x7BFF) == 65504.0     # largest finite


def _read_golden():
    cases = []
    with open(GOLDEN) as fh:
        lines = [ln.strip() for ln in fh if ln.strip() and not ln.startswith("#")]
    i = 0
    while i < len(lines):
        head = lines[i].split()
        assert head[0] == "case", head
        name, M, N, K = head[1], int(head[2]), int(head[3]), int(head[4])
        rows = [[float(t) for t in ln.split()] for ln in lines[i + 1:i + 1 + M + K + M]]
        assert lines[i + 1 + M + K + M] == "end"
        cases.append((name, np.array(rows[:M]), np.array(rows[M:M + K]),
                      np.array(rows[M + K:])))
        i += 2 + M + K + M
    return cases


@pytest.mark.parametrize("case", _read_golden(), ids=lambda c: c[0])
def test_hand_worked_products(case):
    _, a, b, r = case
    got = oracle.gemm_f16(_f16(a), _f16(b))
    assert np.array_equal(got, r)


def test_identity_is_exact():
    rng = np.random.default_rng(11)
    for (m, n) in [(1, 1), (5, 7), (33, 17), (64, 128)]:
        A = _rand_any_finite_f16_bits(rng, (m, n))
        I_n = _f16(np.eye(n))
        I_m = _f16(np.eye(m))
        a = oracle.widen_f16(A)
        assert np.array_equal(oracle.gemm_f16(A, I_n), a)
        assert np.array_equal(oracle.gemm_f16(I_m, A), a)


def test_permutations_move_rows_and_columns():
    rng = np.random.default_rng(12)
    m, n = 23, 31
    A = _rand_f16_bits(rng, (m, n))
    a = oracle.widen_f16(A)
    pr = rng.permutation(m)
    pc = rng.permutation(n)
    P = np.zeros((m, m))
    P[np.arange(m), pr] = 1.0          # (P A)[i] = A[pr[i]]
    Q = np.zeros((n, n))
    Q[pc, np.arange(n)] = 1.0          # (A Q)[:, j] = A[:, pc[j]]
    assert np.array_equal(oracle.gemm_f16(_f16(P), A), a[pr])
    assert np.array_equal(oracle.gemm_f16(A, _f16(Q)), a[:, pc])


def test_rank_one_closed_form():
    rng = np.random.default_rng(13)
    M, N, K = 9, 13, 1000
    u = _rand_f16_bits(rng, (M,))
    v = _rand_f16_bits(rng, (N,))
    A = np.repeat(u[:, None], K, axis=1)
    B = np.repeat(v[None, :], K, axis=0)
    uf = u.view(np.float16).astype(np.float64)
    vf = v.view(np.float16).astype(np.float64)
    want = K * np.outer(uf, vf)          # exact: 22-bit products times K <= 2^10
    assert np.array_equal(oracle.gemm_f16(A, B), want)


@pytest.mark.parametrize("K", range(1, 9))
def test_brute_force_exact_small(K):
    """Every M, N <= 8 for this K: equality with exact rational arithmetic.

    Values have exponents in [-4, 4), so each product has <= 22 significant
    bits within a 16-octave window and every partial sum is exact in binary64.
    """
    rng = np.random.default_rng(100 + K)
    for M in range(1, 9):
        for N in range(1, 9):
            A = _rand_f16_bits(rng, (M, K))
            B = _rand_f16_bits(rng, (K, N))
            got = oracle.gemm_f16(A, B)
            ex = _exact(A, B)
            want = np.array([[float(x) for x in row] for row in ex])
            assert np.array_equal(got, want), (M, N, K)


@pytest.mark.parametrize("K", [1, 3, 8])
def test_brute_force_full_range_within_summation_bound(K):
    """Full binary16 range incl. subnormals: |oracle - exact| <= gamma * sum|ab|.

    Recursive summation of K exactly-formed products in binary64 has error at
    most (K-1) u / (1 - (K-1) u) * sum_k |a_ik b_kj|, u = 2^-53.
    """
    rng = np.random.default_rng(200 + K)
    u = 2.0 ** -53
    gamma = (K - 1) * u / (1 - (K - 1) * u) if K > 1 else 0.0
    for M in range(1, 9):
        for N in range(1, 9):
            A = _rand_any_finite_f16_bits(rng, (M, K))
            B = _rand_any_finite_f16_bits(rng, (K, N))
            got = oracle.gemm_f16(A, B)
            ex = _exact(A, B)
            a = np.abs(A.view(np.float16).astype(np.float64))
            b = np.abs(B.view(np.float16).astype(np.float64))
            absprod = a @ b
            for i in range(M):
                for j in range(N):
                    err = abs(Fraction(got[i, j]) - ex[i][j])
                    assert err <= Fraction(gamma) * Fraction(absprod[i, j]) * Fraction(1.0000001), (M, N, K, i, j)


def test_transpose_identity_bitwise():
    rng = np.random.default_rng(14)
    A = _rand_any_finite_f16_bits(rng, (37, 53))
    B = _rand_any_finite_f16_bits(rng, (53, 29))
    R = oracle.gemm_f16(A, B)
    Rt = oracle.gemm_f16(np.ascontiguousarray(B.T), np.ascontiguousarray(A.T))
    assert np.array_equal(R, Rt.T)


def test_linearity_in_A():
    rng = np.random.default_rng(15)
    A1 = oracle.widen_f16(_rand_f16_bits(rng, (20, 40)))
    A2 = oracle.widen_f16(_rand_f16_bits(rng, (20, 40)))
    B = oracle.widen_f16(_rand_f16_bits(rng, (40, 30)))
    lhs = oracle.gemm_f64(A1 + A2, B)
    rhs = oracle.gemm_f64(A1, B) + oracle.gemm_f64(A2, B)
    scale = oracle.gemm_f64(np.abs(A1) + np.abs(A2), np.abs(B))
    assert np.all(np.abs(lhs - rhs) <= 64 * 2.0 ** -53 * scale)


def test_strided_operands_ignore_nan_padding():
    rng = np.random.default_rng(16)
    M, N, K = 12, 10, 14
    A = _rand_f16_bits(rng, (M, K))
    B = _rand_f16_bits(rng, (K, N))
    a = oracle.widen_f16(A)
    b = oracle.widen_f16(B)
    Ap = np.full((M, K + 5), np.nan)
    Ap[:, :K] = a
    Bp = np.full((K, N + 3), np.nan)
    Bp[:, :N] = b
    R = oracle.gemm_f64(Ap[:, :K], Bp[:, :N])
    assert np.isfinite(R).all()
    assert np.array_equal(R, oracle.gemm_f64(a, b))


def test_empty_sum_and_empty_shapes():
    assert np.array_equal(oracle.gemm_f64(np.zeros((3, 0)), np.zeros((0, 4))),
                          np.zeros((3, 4)))
    assert oracle.gemm_f64(np.zeros((0, 5)), np.zeros((5, 4))).shape == (0, 4)


def test_oracle_against_independent_library_product():
    """Cross-check with numpy's BLAS product on a mid-size case (rounding differs)."""
    rng = np.random.default_rng(17)
    A = _rand_f16_bits(rng, (70, 300))
    B = _rand_f16_bits(rng, (300, 50))
    a = oracle.widen_f16(A)
    b = oracle.widen_f16(B)
    R = oracle.gemm_f64(a, b)
    ref = a @ b
    assert np.all(np.abs(R - ref) <= 600 * 2.0 ** -53 * (np.abs(a) @ np.abs(b)))


# ---- the comparison rules themselves --------------------------------------
def test_parity_rules_catch_nan_first():
    r = np.ones((4, 4))
    c = r.copy()
    c[1, 2] = np.nan
    with pytest.raises(parity.ParityError, match="non-finite"):
        parity.check(c, r)


def test_parity_rules_thresholds():
    r = np.full((100,), 10.0)
    parity.check(r * (1 + 4e-3), r)          # rel_rms 4e-3 passes
    with pytest.raises(parity.ParityError, match="rel_rms"):
        parity.check(r * (1 + 6e-3), r)
    c = r.copy()
    c[0] += 0.2                               # one element off by 0.2 > 0.11
    with pytest.raises(parity.ParityError, match="per-element"):
        parity.check(c, r)
