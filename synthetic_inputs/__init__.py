"""Seeded synthetic FP16 inputs for the GEMM and attention workloads.

This module only draws numbers; it holds none of the GEMM's arithmetic, and
both the oracle side (tests) and the GPU side (tests, bench) take their
inputs from it.

Generator: SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014), used counter-style: draw t of a stream with
key ``s`` is mix64(s + (t + 1) * 0x9E3779B97F4A7C15), where mix64 is the
published finaliser (xor-shift 30, multiply 0xBF58476D1CE4E5B9, xor-shift 27,
multiply 0x94D049BB133111EB, xor-shift 31).  A matrix pair is one stream: A
takes draws 0 .. M*K-1 (row-major), B the next K*N draws (row-major).

Distributions (values are rounded to binary16 by round-to-nearest-even, via
numpy's float64 -> float16 conversion):

* ``uniform_nonzero(r, eps)``: uniform on [-r, -eps] U [eps, r].  The sign
  is the top bit of the draw, the magnitude eps + (r - eps) * u with u the
  next 24 bits / 2^24.  This is the distribution that rejecting |x| < eps
  from uniform[-r, r] would give, drawn without a rejection loop.  With
  eps >= 1e-3 * r no value rounds to zero in binary16.
* ``normal(sigma)``: Box-Muller over two consecutive draws, cos branch only:
  sigma * sqrt(-2 ln u1) * cos(2 pi u2), u1 = (top 24 bits + 1) / 2^24 in
  (0, 1], u2 = next 24 bits / 2^24.  Two draws per value.

Workloads: see ``WORKLOADS`` below.  Each has a fixed stream key; the 4096^3
case has eight A/B pairs for cache busting, pair p keyed (2 << 32) + p.

Attention workloads (``ATTN_WORKLOADS``): Q, K, V of shape [batch, heads,
seq, 256] in one stream: Q takes the first B*H*Sq*256 draws (row-major over
b, h, i, d), K the next B*H*Skv*256, V the next.  Q and K are normal with
sigma 1 (so a score q.k / 16 has unit variance), V uniform on
[-1, -1e-3] U [1e-3, 1].
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


def splitmix64(key: int, start: int, count: int) -> np.ndarray:
    """Draws start .. start+count-1 of the SplitMix64 stream with ``key``."""
    z = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    tmp = np.empty_like(z)
    with np.errstate(over="ignore"):
        np.multiply(z, _GOLDEN, out=z)
        np.add(z, np.uint64(key & 0xFFFFFFFFFFFFFFFF), out=z)
        for shift, mult in ((30, _M1), (27, _M2), (31, None)):
            np.right_shift(z, np.uint64(shift), out=tmp)
            np.bitwise_xor(z, tmp, out=z)
            if mult is not None:
                np.multiply(z, mult, out=z)
    return z


def _to_f16_bits(x: np.ndarray) -> np.ndarray:
    return x.astype(np.float16).view(np.uint16)


def uniform_nonzero_bits(key: int, start: int, count: int, r: float,
                         eps: float) -> np.ndarray:
    """binary16 bit patterns of uniform values on [-r,-eps] U [eps,r]."""
    z = splitmix64(key, start, count)
    neg = (z >> np.uint64(63)).astype(np.float64)
    np.right_shift(z, np.uint64(39), out=z)
    np.bitwise_and(z, np.uint64(0xFFFFFF), out=z)
    mag = z.astype(np.float64)
    del z
    mag *= 1.0 / 16777216.0
    mag *= (r - eps)
    mag += eps
    neg *= -2.0
    neg += 1.0
    mag *= neg
    return _to_f16_bits(mag)


def normal_bits(key: int, start: int, count: int, sigma: float) -> np.ndarray:
    """binary16 bit patterns of N(0, sigma^2) values (Box-Muller)."""
    z = splitmix64(key, 2 * start, 2 * count)
    top = (z >> np.uint64(40)).astype(np.float64)
    u1 = (top[0::2] + 1.0) / 16777216.0
    u2 = top[1::2] / 16777216.0
    x = sigma * np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)
    return _to_f16_bits(x)


@dataclass(frozen=True)
class Workload:
    """One GEMM workload: shape, split, value distribution and seeds."""
    name: str
    M: int
    N: int
    K: int
    split_k: int
    dist: str            # "uniform_nonzero" or "normal"
    scale: float         # r for uniform, sigma for normal
    eps: float           # excluded magnitude for uniform (unused for normal)
    keys: tuple          # one stream key per A/B pair

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K

    def pair_bits(self, p: int = 0, rows=None):
        """(A_bits, B_bits) as uint16 arrays, shapes (M, K) and (K, N).

        ``rows`` restricts A to those rows (their draws are taken from the
        same positions of the stream, so the values equal the full matrix's).
        """
        key = self.keys[p]
        M, N, K = self.M, self.N, self.K
        if rows is None:
            a = self._draw(key, 0, M * K).reshape(M, K)
        else:
            rows = np.asarray(rows, dtype=np.int64)
            a = np.stack([self._draw(key, int(i) * K, K) for i in rows]) \
                if len(rows) else np.zeros((0, K), np.uint16)
        b = self._draw(key, M * K, K * N).reshape(K, N)
        return a, b

    def _draw(self, key, start, count):
        if self.dist == "uniform_nonzero":
            return uniform_nonzero_bits(key, start, count, self.scale, self.eps)
        if self.dist == "normal":
            return normal_bits(key, start, count, self.scale)
        raise ValueError(self.dist)


def _w(name, M, N, K, split_k, dist, scale, eps, keys):
    return Workload(name, M, N, K, split_k, dist, scale, eps, tuple(keys))


#: The five workloads: a 256^3 correctness case, 1024^3, 4096^3 with eight
#: rotating pairs, a ragged 4000 x 4104 x 3000 case and a long-K split case.
WORKLOADS = {
    "gemm_256": _w("gemm_256", 256, 256, 256, 1, "uniform_nonzero", 1.0, 1e-3, [0]),
    "gemm_1024": _w("gemm_1024", 1024, 1024, 1024, 1, "uniform_nonzero", 1.0, 1e-3, [1]),
    "gemm_4096": _w("gemm_4096", 4096, 4096, 4096, 1, "uniform_nonzero", 1.0, 1e-3,
                    [(2 << 32) + p for p in range(8)]),
    "gemm_ragged": _w("gemm_ragged", 4000, 4104, 3000, 1, "normal", 0.5, 0.0, [3]),
    "gemm_splitk": _w("gemm_splitk", 512, 512, 32768, 16, "uniform_nonzero", 0.25,
                      2.5e-4, [4]),
}


def custom(M: int, N: int, K: int, seed: int, split_k: int = 1,
           dist: str = "uniform_nonzero", scale: float = 1.0,
           eps: float = 1e-3) -> Workload:
    """A workload of any shape with the same generator (for shape sweeps).

    For the uniform distribution ``eps`` is relative to ``scale``.
    """
    return _w(f"custom_{M}x{N}x{K}_s{seed}", M, N, K, split_k, dist, scale,
              eps * scale if dist == "uniform_nonzero" else 0.0, [seed])


@dataclass(frozen=True)
class AttnWorkload:
    """One attention workload: [B, H, S, D] shapes, distributions, seed."""
    name: str
    B: int
    H: int
    Sq: int
    Skv: int
    D: int
    key: int
    qk_sigma: float = 1.0

    @property
    def scale(self) -> float:
        return 1.0 / float(np.sqrt(self.D))

    @property
    def flops(self) -> int:
        """Two products per head: S = Q K^T and O = P V."""
        return 4 * self.B * self.H * self.Sq * self.Skv * self.D

    def _q0(self):
        return 0

    def _k0(self):
        return self.B * self.H * self.Sq * self.D

    def _v0(self):
        return self._k0() + self.B * self.H * self.Skv * self.D

    def bits(self):
        """(Q, K, V) as uint16 arrays of shape [B, H, S, D]."""
        B, H, D = self.B, self.H, self.D
        q = normal_bits(self.key, self._q0(), B * H * self.Sq * D, self.qk_sigma)
        k = normal_bits(self.key, self._k0(), B * H * self.Skv * D, self.qk_sigma)
        v = uniform_nonzero_bits(self.key, self._v0(), B * H * self.Skv * D, 1.0, 1e-3)
        return (q.reshape(B, H, self.Sq, D), k.reshape(B, H, self.Skv, D),
                v.reshape(B, H, self.Skv, D))

    def head_bits(self, b: int, h: int, rows=None):
        """(Q rows, K, V) of one (batch, head), each [1, 1, S, D]; ``rows``
        selects query rows (same values as in the full tensor)."""
        D, H = self.D, self.H
        bh = b * H + h
        if rows is None:
            rows = np.arange(self.Sq)
        rows = np.asarray(rows, dtype=np.int64)
        q = np.stack([normal_bits(self.key, self._q0() + (bh * self.Sq + int(i)) * D, D,
                                  self.qk_sigma) for i in rows]) if len(rows) else \
            np.zeros((0, D), np.uint16)
        k = normal_bits(self.key, self._k0() + bh * self.Skv * D, self.Skv * D, self.qk_sigma)
        v = uniform_nonzero_bits(self.key, self._v0() + bh * self.Skv * D, self.Skv * D, 1.0,
                                 1e-3)
        return (q.reshape(1, 1, len(rows), D), k.reshape(1, 1, self.Skv, D),
                v.reshape(1, 1, self.Skv, D))


#: Attention forward at head dimension 256 (the pages' HD=256 kernel; they
#: state no batch, head count or sequence length): a small case the oracle
#: finishes at once, a ragged case (query and key counts not multiples of
#: the 128 / 64 blocks) and a throughput case, 4 x 16 heads x 4096 x 4096.
ATTN_WORKLOADS = {
    "attn_256": AttnWorkload("attn_256", 1, 2, 256, 256, 256, 10),
    "attn_ragged": AttnWorkload("attn_ragged", 2, 3, 1000, 1500, 256, 11),
    "attn_4096": AttnWorkload("attn_4096", 4, 16, 4096, 4096, 256, 12),
}


def attn_custom(B: int, H: int, Sq: int, Skv: int, seed: int, qk_sigma: float = 1.0,
                D: int = 256) -> AttnWorkload:
    """An attention workload of any shape with the same generator."""
    return AttnWorkload(f"attn_{B}x{H}x{Sq}x{Skv}_s{seed}", B, H, Sq, Skv, D, seed, qk_sigma)
