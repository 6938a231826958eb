"""Full-size FP64 oracle results shared by the GPU parity tests of one
pytest session.

The benchmark's workloads are compared with the oracle on every output
element.  A 4096^3 product costs the oracle a few seconds on the host's
cores, so each result is computed once per session and reused by every
test (and kernel variant) that checks the same inputs.  The arrays are
read-only.
"""
from __future__ import annotations

import functools

import numpy as np

import oracle
import synthetic_inputs as si


def _frozen(x: np.ndarray) -> np.ndarray:
    x.flags.writeable = False
    return x


@functools.lru_cache(maxsize=None)
def gemm_inputs(name: str, pair: int = 0):
    """(A bits, B bits) of pair `pair` of GEMM workload `name`."""
    A, B = si.WORKLOADS[name].pair_bits(pair)
    return _frozen(A), _frozen(B)


@functools.lru_cache(maxsize=None)
def gemm_ref(name: str, pair: int = 0) -> np.ndarray:
    """Oracle C (float64, M x N) of pair `pair` of GEMM workload `name`."""
    A, B = gemm_inputs(name, pair)
    return _frozen(oracle.gemm_f16(A, B))


@functools.lru_cache(maxsize=None)
def attn_inputs(name: str):
    """(Q, K, V) bits of attention workload `name`."""
    return tuple(_frozen(x) for x in si.ATTN_WORKLOADS[name].bits())


@functools.lru_cache(maxsize=None)
def attn_ref(name: str) -> np.ndarray:
    """Oracle O (float64, [batch, head, row, 256]) of attention workload
    `name`, computed one batch entry at a time to bound the host memory."""
    w = si.ATTN_WORKLOADS[name]
    Qb, Kb, Vb = attn_inputs(name)
    out = np.empty(Qb.shape, np.float64)
    for b in range(Qb.shape[0]):
        out[b:b + 1] = oracle.attention_f16(Qb[b:b + 1], Kb[b:b + 1], Vb[b:b + 1], w.scale)
    return _frozen(out)
