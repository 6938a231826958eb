"""FP64 CPU oracles: the FP16 GEMM C = A*B and the attention forward pass.

TEST INFRASTRUCTURE ONLY.  Only the test suite, ``__graft_entry__.smoke()``
and the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import
this package.  The product path (the C-ABI library and its Python binding)
never imports, links or runs it, and this package never imports the product.

The arithmetic lives in ``gemm_oracle.c`` and ``attn_oracle.c`` (plain C, compiled with gcc and
OpenMP); this module only builds it and marshals numpy arrays through ctypes.

What it computes: R[i, j] = sum_k double(a_ik) * double(b_kj) over the
binary16 inputs widened exactly to binary64, summed in increasing k
("Xe2 ESIMD GEMM" page, section "Correctness testing": a CPU reference for
the half-precision product; FP64 here instead of the page's FP32).

Pins (tests/test_oracle_pins.py): widening checked against numpy's own
binary16 conversion for all 65536 bit patterns; hand-worked 2x2 and 3x3
products (tests/golden/); identity and permutation matrices; rank-1 closed
form; brute force in exact rational arithmetic for every M, N, K <= 8;
transpose identity; strided inputs whose padding is NaN.

The attention oracle (``attn_oracle.c``, ``attention_f16``) is the plain
definition of softmax(scale * Q K^T) V per batch and head, written out in
FP64 (the streaming "SDP" kernel of the "Xe2 Nbarrier Pipelining" page
reaches it up to rounding).  Pins (tests/test_oracle_attention_pins.py):
one key (output = that value row), equal scores (output = mean of the value
rows), two keys against the logistic closed form, an exact 50-digit
evaluation of the textbook softmax formula on tiny cases, scipy's softmax on
random cases, invariance to a common shift of the keys and to permuting
key/value pairs, linearity in V, overflow-free large scores, and batch /
head / stride independence.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gemm_oracle.c")
_SRCS = [_SRC, os.path.join(_HERE, "attn_oracle.c")]
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle C sources into one shared library with gcc + OpenMP."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and all(os.path.getmtime(_LIB_PATH) >= os.path.getmtime(f) for f in _SRCS)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-ffp-contract=off", *_SRCS, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.oracle_f16_to_f64.argtypes = [ctypes.c_uint16]
            lib.oracle_f16_to_f64.restype = ctypes.c_double
            lib.oracle_widen_f16.argtypes = [ctypes.c_int64, ctypes.c_void_p,
                                             ctypes.c_void_p]
            lib.oracle_widen_f16.restype = None
            lib.oracle_gemm_f64.argtypes = [
                ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                ctypes.c_void_p, ctypes.c_int64,
                ctypes.c_void_p, ctypes.c_int64,
                ctypes.c_void_p, ctypes.c_int64]
            lib.oracle_gemm_f64.restype = None
            lib.oracle_attention_f64.argtypes = [
                ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_double, ctypes.c_void_p,
                ctypes.c_int64, ctypes.c_void_p]
            lib.oracle_attention_f64.restype = ctypes.c_int
            lib.oracle_num_threads.argtypes = []
            lib.oracle_num_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def num_threads() -> int:
    """OpenMP threads the oracle's GEMM runs on."""
    return int(_load().oracle_num_threads())


def f16_to_f64_scalar(bits: int) -> float:
    """Widen one binary16 bit pattern (0..65535) to a Python float."""
    return float(_load().oracle_f16_to_f64(int(bits) & 0xFFFF))


def widen_f16(bits: np.ndarray) -> np.ndarray:
    """Widen an array of binary16 bit patterns (uint16) to float64."""
    src = np.ascontiguousarray(bits, dtype=np.uint16)
    dst = np.empty(src.shape, dtype=np.float64)
    _load().oracle_widen_f16(src.size, src.ctypes.data, dst.ctypes.data)
    return dst


def gemm_f64(A: np.ndarray, B: np.ndarray) -> np.ndarray:
    """R = A @ B by the plain triple loop, for float64 A (M x K), B (K x N).

    A and B may be row-strided views (inner stride 1 is required); R is a
    fresh contiguous M x N float64 array.
    """
    A = np.asarray(A)
    B = np.asarray(B)
    if A.dtype != np.float64 or B.dtype != np.float64:
        raise TypeError("oracle.gemm_f64 takes float64 operands")
    if A.ndim != 2 or B.ndim != 2 or A.shape[1] != B.shape[0]:
        raise ValueError(f"shape mismatch {A.shape} x {B.shape}")
    if A.strides[1] != 8:
        A = np.ascontiguousarray(A)
    if B.strides[1] != 8:
        B = np.ascontiguousarray(B)
    M, K = A.shape
    N = B.shape[1]
    R = np.empty((M, N), dtype=np.float64)
    if M and N:
        _load().oracle_gemm_f64(M, N, K, A.ctypes.data, A.strides[0] // 8,
                                B.ctypes.data, B.strides[0] // 8,
                                R.ctypes.data, N)
    return R


def gemm_f16(A_bits: np.ndarray, B_bits: np.ndarray, rows=None) -> np.ndarray:
    """Exact-input FP64 product of binary16 matrices given as uint16 bits.

    ``rows`` (optional index array) restricts the result to those rows of A,
    in the order given: R[t] = A[rows[t]] @ B.
    """
    A_bits = np.asarray(A_bits, dtype=np.uint16)
    if rows is not None:
        A_bits = A_bits[np.asarray(rows, dtype=np.int64)]
    return gemm_f64(widen_f16(A_bits), widen_f16(B_bits))


def _bhsd_strides(X: np.ndarray) -> np.ndarray:
    if X.ndim != 4 or X.strides[3] != X.itemsize:
        raise ValueError("attention operands are [batch, head, row, d] with d contiguous")
    return np.array([X.strides[0], X.strides[1], X.strides[2]], dtype=np.int64) // X.itemsize


def attention_f64(Q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float,
                  rows=None) -> np.ndarray:
    """softmax(scale * Q K^T) V for float64 [B, H, S, D] arrays (d contiguous,
    other strides free).  ``rows`` restricts the result to those query rows:
    the output is [B, H, len(rows) or Sq, D]."""
    for X in (Q, K, V):
        if X.dtype != np.float64:
            raise TypeError("oracle.attention_f64 takes float64 operands")
    B, H, Sq, D = Q.shape
    Skv = K.shape[2]
    if K.shape != (B, H, Skv, D) or V.shape != (B, H, Skv, D):
        raise ValueError(f"shape mismatch {Q.shape} {K.shape} {V.shape}")
    qs, ks, vs = _bhsd_strides(Q), _bhsd_strides(K), _bhsd_strides(V)
    r = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    nr = Sq if r is None else len(r)
    O = np.empty((B, H, nr, D), dtype=np.float64)
    if O.size == 0:
        return O
    if Skv == 0:
        raise ValueError("attention over zero keys is undefined")
    rc = _load().oracle_attention_f64(
        B, H, Sq, Skv, D, Q.ctypes.data, qs.ctypes.data, K.ctypes.data, ks.ctypes.data,
        V.ctypes.data, vs.ctypes.data, float(scale),
        None if r is None else r.ctypes.data, nr, O.ctypes.data)
    if rc != 0:
        raise MemoryError("oracle_attention_f64: out of memory")
    return O


def attention_f16(Q_bits: np.ndarray, K_bits: np.ndarray, V_bits: np.ndarray,
                  scale: float, rows=None) -> np.ndarray:
    """Attention over binary16 inputs given as uint16 bits [B, H, S, D],
    widened exactly; ``scale`` is used as given (a float)."""
    return attention_f64(widen_f16(Q_bits), widen_f16(K_bits), widen_f16(V_bits), scale, rows)
