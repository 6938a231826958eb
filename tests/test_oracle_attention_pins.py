"""Pins for the FP64 attention oracle: checks against things other than it.

Each test ties oracle.attention_f64 / attention_f16 to a fact fixed by the
mathematics or by an independent implementation, so that a plausible slip
(a dropped scale, a missing max shift, a wrong normaliser, K and V mixed up,
a stride or head mix-up) fails at least one of them:

* hand-worked cases from tests/golden/attention_worked.txt;
* one key: the output is that value row, exactly;
* equal scores: the output is the mean of the value rows (exact rational
  mean, rounded once);
* two keys: the logistic closed form sigma(s1 - s2), with the score
  difference computed in exact rational arithmetic;
* the textbook formula exp(s_j) / sum_k exp(s_k) evaluated with 50 decimal
  digits (mpmath) on tiny random cases;
* scipy.special.softmax followed by a matrix product (independent library
  routines) on random cases;
* invariance to a common shift of every key, to permuting key/value pairs,
  linearity in V;
* scores near 1e3 stay finite and match the closed form;
* batch, head and row strides; a subset of rows equals those rows of the
  full result.
"""
from __future__ import annotations

import os
from fractions import Fraction

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "attention_worked.txt")


def _f16_vals(rng, shape, lo=-4, hi=5, scale=1.0):
    """Values exactly representable in binary16 (small integers times 2^-k)."""
    return (rng.integers(lo, hi, size=shape) * scale).astype(np.float16).astype(np.float64)


def _read_golden():
    cases, cur = [], None
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, *vals = line.split()
        if key == "scale":
            cur = {"scale": float(vals[0]), "k": [], "v": []}
        elif key == "q":
            cur["q"] = [float(x) for x in vals]
        elif key in ("k", "v"):
            cur[key].append([float(x) for x in vals])
        elif key == "o":
            cur["o"] = [float(x) for x in vals]
        elif key == "end":
            cases.append(cur)
    return cases


def test_golden_worked_cases():
    cases = _read_golden()
    assert len(cases) == 4
    for c in cases:
        Q = np.array(c["q"], dtype=np.float64).reshape(1, 1, 1, -1)
        K = np.array(c["k"], dtype=np.float64)[None, None]
        V = np.array(c["v"], dtype=np.float64)[None, None]
        o = oracle.attention_f64(Q, K, V, c["scale"])[0, 0, 0]
        np.testing.assert_allclose(o, c["o"], rtol=1e-15, atol=1e-15)


def test_single_key_returns_value_row_exactly():
    rng = np.random.default_rng(1)
    Q = _f16_vals(rng, (2, 3, 5, 16))
    K = _f16_vals(rng, (2, 3, 1, 16))
    V = _f16_vals(rng, (2, 3, 1, 16), scale=0.125)
    O = oracle.attention_f64(Q, K, V, 0.0625)
    assert np.array_equal(O, np.broadcast_to(V, O.shape))


@pytest.mark.parametrize("skv", [1, 3, 64, 100])
def test_equal_scores_give_the_mean(skv):
    rng = np.random.default_rng(skv)
    Q = _f16_vals(rng, (1, 2, 4, 8))
    K = np.zeros((1, 2, skv, 8))
    V = _f16_vals(rng, (1, 2, skv, 8), scale=0.25)
    O = oracle.attention_f64(Q, K, V, 1.0)
    for h in range(2):
        mean = [float(sum(Fraction(x) for x in V[0, h, :, d]) / skv) for d in range(8)]
        for i in range(4):
            np.testing.assert_allclose(O[0, h, i], mean, rtol=4e-16, atol=0)
    # scale 0 gives the same whatever the keys
    O0 = oracle.attention_f64(Q, _f16_vals(rng, (1, 2, skv, 8)), V, 0.0)
    np.testing.assert_allclose(O0, O, rtol=4e-16, atol=0)


def test_two_keys_logistic_closed_form():
    rng = np.random.default_rng(7)
    D = 32
    for trial in range(20):
        q = _f16_vals(rng, (D,), scale=0.5)
        k1, k2 = _f16_vals(rng, (D,), scale=0.25), _f16_vals(rng, (D,), scale=0.25)
        v1, v2 = _f16_vals(rng, (D,)), _f16_vals(rng, (D,))
        scale = 0.0625
        ds = Fraction(scale) * sum(Fraction(a) * (Fraction(b) - Fraction(c))
                                   for a, b, c in zip(q, k1, k2))
        sig = 1.0 / (1.0 + np.exp(-float(ds)))
        want = sig * v1 + (1.0 - sig) * v2
        Q = q.reshape(1, 1, 1, D)
        K = np.stack([k1, k2])[None, None]
        V = np.stack([v1, v2])[None, None]
        got = oracle.attention_f64(Q, K, V, scale)[0, 0, 0]
        np.testing.assert_allclose(got, want, rtol=1e-13, atol=1e-14)


def test_textbook_formula_in_high_precision():
    mp = pytest.importorskip("mpmath")
    mp.mp.dps = 50
    rng = np.random.default_rng(11)
    B, H, Sq, Skv, D = 1, 2, 3, 5, 6
    Q = _f16_vals(rng, (B, H, Sq, D), scale=0.5)
    K = _f16_vals(rng, (B, H, Skv, D), scale=0.5)
    V = _f16_vals(rng, (B, H, Skv, D))
    scale = 0.3
    O = oracle.attention_f64(Q, K, V, scale)
    for h in range(H):
        for i in range(Sq):
            s = [mp.mpf(scale) * mp.fsum(mp.mpf(Q[0, h, i, d]) * mp.mpf(K[0, h, j, d])
                                          for d in range(D)) for j in range(Skv)]
            e = [mp.exp(x) for x in s]
            tot = mp.fsum(e)
            for d in range(D):
                want = mp.fsum(e[j] * mp.mpf(V[0, h, j, d]) for j in range(Skv)) / tot
                assert abs(O[0, h, i, d] - float(want)) <= 1e-14 * (abs(float(want)) + 1)


def test_against_scipy_softmax():
    sp = pytest.importorskip("scipy.special")
    rng = np.random.default_rng(3)
    B, H, Sq, Skv, D = 2, 3, 17, 29, 16
    Q = rng.standard_normal((B, H, Sq, D)).astype(np.float16).astype(np.float64)
    K = rng.standard_normal((B, H, Skv, D)).astype(np.float16).astype(np.float64)
    V = rng.standard_normal((B, H, Skv, D)).astype(np.float16).astype(np.float64)
    scale = 1.0 / np.sqrt(D)
    S = scale * np.einsum("bhid,bhjd->bhij", Q, K)
    want = np.einsum("bhij,bhjd->bhid", sp.softmax(S, axis=-1), V)
    np.testing.assert_allclose(oracle.attention_f64(Q, K, V, scale), want, rtol=1e-12,
                               atol=1e-14)


def test_invariances():
    rng = np.random.default_rng(5)
    B, H, Sq, Skv, D = 1, 2, 6, 40, 16
    Q = _f16_vals(rng, (B, H, Sq, D), scale=0.25)
    K = _f16_vals(rng, (B, H, Skv, D), scale=0.25)
    V1 = _f16_vals(rng, (B, H, Skv, D))
    V2 = _f16_vals(rng, (B, H, Skv, D))
    scale = 0.125
    O = oracle.attention_f64(Q, K, V1, scale)
    # a common shift c of every key adds scale * q.c to all scores of a row
    c = _f16_vals(rng, (D,))
    np.testing.assert_allclose(oracle.attention_f64(Q, K + c, V1, scale), O, rtol=1e-12,
                               atol=1e-13)
    # permuting key/value pairs together
    perm = rng.permutation(Skv)
    np.testing.assert_allclose(oracle.attention_f64(Q, K[:, :, perm], V1[:, :, perm], scale), O,
                               rtol=1e-13, atol=1e-14)
    # but permuting only the values changes the result
    assert not np.allclose(oracle.attention_f64(Q, K, V1[:, :, perm], scale), O)
    # linear in V
    np.testing.assert_allclose(oracle.attention_f64(Q, K, V1 + V2, scale),
                               O + oracle.attention_f64(Q, K, V2, scale), rtol=1e-12, atol=1e-13)


def test_large_scores_stay_finite():
    D = 8
    q = np.zeros(D)
    q[0] = 64.0
    k = np.zeros((3, D))
    k[0, 0], k[1, 0], k[2, 0] = 15.625, 15.640625, 0.0   # scores 1000, 1001, 0
    v = np.eye(3, D)
    got = oracle.attention_f64(q.reshape(1, 1, 1, D), k[None, None], v[None, None], 1.0)[0, 0, 0]
    e = np.e
    want = np.zeros(D)
    want[0], want[1] = 1 / (1 + e), e / (1 + e)           # exp(-1000) is far below FP64's eps
    assert np.all(np.isfinite(got))
    np.testing.assert_allclose(got, want, rtol=1e-15, atol=1e-300)


def test_strides_heads_and_row_subsets():
    rng = np.random.default_rng(9)
    B, H, Sq, Skv, D = 2, 3, 9, 11, 8
    # [B, S, H, D] storage seen as [B, H, S, D]: head stride D, row stride H*D
    Qs = _f16_vals(rng, (B, Sq, H, D))
    Ks = _f16_vals(rng, (B, Skv, H, D))
    Vs = _f16_vals(rng, (B, Skv, H, D))
    Q, K, V = (x.transpose(0, 2, 1, 3) for x in (Qs, Ks, Vs))
    O = oracle.attention_f64(Q, K, V, 0.25)
    Oc = oracle.attention_f64(*(np.ascontiguousarray(x) for x in (Q, K, V)), 0.25)
    assert np.array_equal(O, Oc)
    for b in range(B):
        for h in range(H):
            one = oracle.attention_f64(Q[b:b + 1, h:h + 1], K[b:b + 1, h:h + 1],
                                       V[b:b + 1, h:h + 1], 0.25)
            assert np.array_equal(one[0, 0], O[b, h])
    rows = np.array([8, 0, 3])
    assert np.array_equal(oracle.attention_f64(Q, K, V, 0.25, rows=rows), O[:, :, rows])


def test_f16_entry_widens_bits():
    rng = np.random.default_rng(4)
    Q = rng.standard_normal((1, 1, 3, 8)).astype(np.float16)
    K = rng.standard_normal((1, 1, 4, 8)).astype(np.float16)
    V = rng.standard_normal((1, 1, 4, 8)).astype(np.float16)
    a = oracle.attention_f16(Q.view(np.uint16), K.view(np.uint16), V.view(np.uint16), 0.5)
    b = oracle.attention_f64(Q.astype(np.float64), K.astype(np.float64), V.astype(np.float64), 0.5)
    assert np.array_equal(a, b)


def test_rejects_zero_keys_and_bad_shapes():
    with pytest.raises(ValueError):
        oracle.attention_f64(np.zeros((1, 1, 2, 4)), np.zeros((1, 1, 0, 4)),
                             np.zeros((1, 1, 0, 4)), 1.0)
    with pytest.raises(ValueError):
        oracle.attention_f64(np.zeros((1, 1, 2, 4)), np.zeros((1, 1, 3, 4)),
                             np.zeros((1, 1, 2, 4)), 1.0)
