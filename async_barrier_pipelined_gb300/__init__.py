"""Python binding of the gemm_f16 C ABI (include/gemm_f16.h).

Argument marshalling only: every step of the product runs in the CUDA
kernels of ``csrc/gemm_f16.cu``.  The functions keep the C names; raw
pointers are Python ints.  ``matmul`` is a convenience that takes torch
tensors (PyTorch is used only for device memory and streams).

The library is built in-tree by ``async_barrier_pipelined_gb300.build.build()``
(``__graft_entry__.build()`` calls it).  If it is missing, loading fails
loudly; there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
import threading

from .build import LIB_PATH

__all__ = [
    "GemmError", "load", "gemm_f16_plan", "gemm_f16_run", "gemm_f16_run_host",
    "gemm_f16_destroy", "gemm_f16_status", "gemm_f16_set_option",
    "gemm_f16_strerror", "gemm_f16_last_cuda_error", "gemm_f16_validate",
    "gemm_f16_tile_order", "gemm_f16_tile_shape", "Plan", "matmul",
    "OK", "ERR_INVALID_ARG", "ERR_MISALIGNED", "ERR_UNSUPPORTED_DEVICE",
    "ERR_OOM", "ERR_CUDA", "ERR_TIMEOUT", "ERR_SCRATCH_TOO_SMALL", "gemm_f16_run_noalloc", "gemm_f16_noalloc_status",
    "OPT_TIMEOUT_NS", "OPT_TILE_ORDER", "OPT_FAULT_UNIT", "OPT_KERNEL", "OPT_TILE_WIDTH", "OPT_SM_LIMIT", "OPT_ATTN_KERNEL", "OPT_ATTN_SPLIT", "OPT_A_REPACK", "OPT_KERNEL_TIMING", "INFO_NUM_SMS", "INFO_MAX_PAIRS", "INFO_MAX_QUADS",
    "gemm_f16_get_option", "gemm_f16_pair_tiles", "EXPORTED_SYMBOLS",
    "gemm_f16_run_ex", "gemm_f16_validate_ex", "attn_f16_fwd", "attn_f16_validate",
    "attn_f16_key_ranges", "gemm_f16_run_info", "gemm_f16_run_choice", "attn_f16_fwd_host", "attention_host",
    "attention", "ATTN_HEAD_DIM", "gemm_f16_kernel_time",
    "LAYOUT_NN", "LAYOUT_TN", "LAYOUT_NT", "LAYOUT_TT",
]

OK = 0
ERR_INVALID_ARG = -1
ERR_MISALIGNED = -2
ERR_UNSUPPORTED_DEVICE = -3
ERR_OOM = -4
ERR_CUDA = -5
ERR_TIMEOUT = -6
ERR_SCRATCH_TOO_SMALL = -7

OPT_TIMEOUT_NS = 1
OPT_TILE_ORDER = 2
OPT_FAULT_UNIT = 3
OPT_KERNEL = 4
OPT_TILE_WIDTH = 5
OPT_SM_LIMIT = 6
OPT_ATTN_KERNEL = 7
OPT_ATTN_SPLIT = 8
OPT_A_REPACK = 9
OPT_KERNEL_TIMING = 10
INFO_NUM_SMS = 100
INFO_MAX_PAIRS = 101
INFO_MAX_QUADS = 102

ATTN_HEAD_DIM = 256

LAYOUT_NN = 0
LAYOUT_TN = 1   # A stored K x M
LAYOUT_NT = 2   # B stored N x K
LAYOUT_TT = 3

_c_int, _c_i64, _vp = ctypes.c_int, ctypes.c_int64, ctypes.c_void_p

#: name -> (restype, argtypes) for every entry point of include/gemm_f16.h
_SIGNATURES = {
    "gemm_f16_plan": (_c_int, [ctypes.POINTER(_vp), _c_int]),
    "gemm_f16_run": (_c_int, [_vp, _c_int, _c_int, _c_int, _vp, _c_i64, _vp, _c_i64,
                              _vp, _c_i64, _c_int, _vp]),
    "gemm_f16_run_ex": (_c_int, [_vp, _c_int, _c_int, _c_int, _c_int, _vp, _c_i64, _vp,
                                 _c_i64, _vp, _c_i64, _c_int, _vp]),
    "gemm_f16_run_host": (_c_int, [_vp, _c_int, _c_int, _c_int, _vp, _c_i64, _vp, _c_i64,
                                   _vp, _c_i64, _c_int, _vp]),
    "gemm_f16_destroy": (_c_int, [_vp]),
    "gemm_f16_status": (_c_int, [_vp]),
    "gemm_f16_set_option": (_c_int, [_vp, _c_int, _c_i64]),
    "gemm_f16_get_option": (_c_int, [_vp, _c_int, ctypes.POINTER(_c_i64)]),
    "gemm_f16_strerror": (ctypes.c_char_p, [_c_int]),
    "gemm_f16_last_cuda_error": (ctypes.c_char_p, []),
    "gemm_f16_validate": (_c_int, [_c_int, _c_int, _c_int, _vp, _c_i64, _vp, _c_i64,
                                   _vp, _c_i64, _c_int]),
    "gemm_f16_validate_ex": (_c_int, [_c_int, _c_int, _c_int, _c_int, _vp, _c_i64, _vp,
                                      _c_i64, _vp, _c_i64, _c_int]),
    "gemm_f16_tile_order": (_c_i64, [_c_int, _c_int, _c_int,
                                     ctypes.POINTER(ctypes.c_uint32), _c_i64]),
    "gemm_f16_tile_shape": (_c_int, [ctypes.POINTER(_c_int)] * 4),
    "gemm_f16_pair_tiles": (_c_i64, [_c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int,
                                     ctypes.POINTER(ctypes.c_uint32), _c_i64,
                                     ctypes.POINTER(_c_int)]),
    "gemm_f16_run_noalloc": (_c_int, [_c_int, _c_int, _c_int, _vp, _c_i64, _vp, _c_i64,
                                      _vp, _c_i64, _c_int, _vp, _vp]),
    "gemm_f16_noalloc_status": (_c_int, []),
    "attn_f16_fwd": (_c_int, [_vp, _c_int, _c_int, _c_int, _c_int, _c_int,
                              _vp, ctypes.POINTER(_c_i64), _vp, ctypes.POINTER(_c_i64),
                              _vp, ctypes.POINTER(_c_i64), _vp, ctypes.POINTER(_c_i64),
                              ctypes.c_float, _vp]),
    "attn_f16_validate": (_c_int, [_c_int, _c_int, _c_int, _c_int, _c_int,
                                   _vp, ctypes.POINTER(_c_i64), _vp, ctypes.POINTER(_c_i64),
                                   _vp, ctypes.POINTER(_c_i64), _vp, ctypes.POINTER(_c_i64),
                                   ctypes.c_float]),
    "attn_f16_key_ranges": (_c_int, [_vp, _c_int, _c_int, _c_int, _c_int,
                                     ctypes.POINTER(_c_int)]),
    "gemm_f16_run_info": (_c_int, [_vp, _c_int, _c_int, _c_int, _c_int, _c_i64, _c_int,
                                   ctypes.POINTER(_c_int)]),
    "gemm_f16_run_choice": (_c_int, [_c_int, _c_int, _c_int, _c_int, _c_i64, _c_int, _c_int,
                                     _c_int, _c_int, ctypes.POINTER(_c_int)]),
    "attn_f16_fwd_host": (_c_int, [_vp, _c_int, _c_int, _c_int, _c_int, _c_int, _vp, _vp, _vp,
                                   _vp, ctypes.c_float, _vp]),
    "gemm_f16_kernel_time": (_c_int, [_vp, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(_c_i64)]),
}
EXPORTED_SYMBOLS = tuple(_SIGNATURES)

_lock = threading.Lock()
_lib = None


class GemmError(RuntimeError):
    """A negative gemm_f16 return code."""

    def __init__(self, code: int, where: str):
        self.code = code
        msg = gemm_f16_strerror(code)
        if code == ERR_CUDA:
            msg += f" [{gemm_f16_last_cuda_error()}]"
        super().__init__(f"{where}: {msg} (code {code})")


def load() -> ctypes.CDLL:
    """Load the in-tree library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise ImportError(
                    f"gemm_f16 library not built ({LIB_PATH} missing); run "
                    "async_barrier_pipelined_gb300.build.build() first. "
                    "There is no fallback implementation.")
            lib = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in _SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def _check(rc: int, where: str) -> int:
    if rc < 0:
        raise GemmError(rc, where)
    return rc


def gemm_f16_strerror(code: int) -> str:
    return load().gemm_f16_strerror(code).decode()


def gemm_f16_last_cuda_error() -> str:
    return load().gemm_f16_last_cuda_error().decode()


def gemm_f16_plan(device: int = 0) -> int:
    """Create a plan on ``device``; returns the opaque handle as an int."""
    h = _vp()
    _check(load().gemm_f16_plan(ctypes.byref(h), device), "gemm_f16_plan")
    return h.value


def gemm_f16_destroy(plan: int) -> None:
    _check(load().gemm_f16_destroy(plan), "gemm_f16_destroy")


def gemm_f16_status(plan: int) -> int:
    """Device-reported status since the last call (0 or ERR_TIMEOUT); clears it."""
    return load().gemm_f16_status(plan)


def gemm_f16_set_option(plan: int, option: int, value: int) -> None:
    _check(load().gemm_f16_set_option(plan, option, value), "gemm_f16_set_option")


def gemm_f16_get_option(plan: int, option: int) -> int:
    v = _c_i64()
    _check(load().gemm_f16_get_option(plan, option, ctypes.byref(v)), "gemm_f16_get_option")
    return v.value


def gemm_f16_run(plan: int, M: int, N: int, K: int, A: int, lda: int, B: int, ldb: int,
                 C: int, ldc: int, split_k: int = 1, stream: int = 0) -> None:
    """Enqueue C = A*B (device pointers) on ``stream`` (a cudaStream_t as int)."""
    _check(load().gemm_f16_run(plan, M, N, K, A, lda, B, ldb, C, ldc, split_k, stream),
           "gemm_f16_run")


def gemm_f16_run_ex(plan: int, layout: int, M: int, N: int, K: int, A: int, lda: int, B: int,
                    ldb: int, C: int, ldc: int, split_k: int = 1, stream: int = 0) -> None:
    """gemm_f16_run with an operand layout (LAYOUT_NN / TN / NT / TT)."""
    _check(load().gemm_f16_run_ex(plan, layout, M, N, K, A, lda, B, ldb, C, ldc, split_k,
                                  stream), "gemm_f16_run_ex")


def gemm_f16_run_host(plan: int, M: int, N: int, K: int, hA: int, lda: int, hB: int,
                      ldb: int, hC: int, ldc: int, split_k: int = 1, stream: int = 0) -> None:
    """Enqueue copy-in, C = A*B and copy-out for HOST pointers on ``stream``."""
    _check(load().gemm_f16_run_host(plan, M, N, K, hA, lda, hB, ldb, hC, ldc, split_k,
                                    stream), "gemm_f16_run_host")


def gemm_f16_run_noalloc(M: int, N: int, K: int, A: int, lda: int, B: int, ldb: int,
                         C: int, ldc: int, split_k: int = 1, status: int = 0,
                         stream: int = 0) -> None:
    """Enqueue C = A*B without a plan and without allocating device memory.

    For callers that may not call cudaMalloc (their device memory belongs to
    another allocator, or they cannot afford its device-wide sync).  Uses the
    library's fixed scratch array; ``status`` is 0 or the address of a
    device-visible int that receives ERR_TIMEOUT if a wait runs out.  Calls
    that overlap on the GPU race on the shared scratch.
    """
    _check(load().gemm_f16_run_noalloc(M, N, K, A, lda, B, ldb, C, ldc, split_k, status,
                                       stream), "gemm_f16_run_noalloc")


def gemm_f16_noalloc_status() -> int:
    """Read and clear the status word of no-alloc calls made with status 0
    on the current device (0, or ERR_TIMEOUT).  Call after their stream has
    been synchronised."""
    rc = int(load().gemm_f16_noalloc_status())
    if rc not in (0, ERR_TIMEOUT):
        _check(rc, "gemm_f16_noalloc_status")
    return rc


def gemm_f16_validate(M, N, K, A, lda, B, ldb, C, ldc, split_k) -> int:
    return load().gemm_f16_validate(M, N, K, A, lda, B, ldb, C, ldc, split_k)


def gemm_f16_validate_ex(layout, M, N, K, A, lda, B, ldb, C, ldc, split_k) -> int:
    return load().gemm_f16_validate_ex(layout, M, N, K, A, lda, B, ldb, C, ldc, split_k)


def _strides3(st):
    if st is None or len(st) != 3:
        raise ValueError("strides are (batch, head, row) in elements")
    return (_c_i64 * 3)(*[int(x) for x in st])


def attn_f16_fwd(plan: int, batch: int, heads: int, seq_q: int, seq_kv: int, head_dim: int,
                 Q: int, q_strides, K: int, k_strides, V: int, v_strides, O: int, o_strides,
                 scale: float, stream: int = 0) -> None:
    """Enqueue attention forward (device pointers; strides (batch, head, row))."""
    _check(load().attn_f16_fwd(plan, batch, heads, seq_q, seq_kv, head_dim,
                               Q, _strides3(q_strides), K, _strides3(k_strides),
                               V, _strides3(v_strides), O, _strides3(o_strides),
                               float(scale), stream), "attn_f16_fwd")


def attn_f16_validate(batch, heads, seq_q, seq_kv, head_dim, Q, q_strides, K, k_strides,
                      V, v_strides, O, o_strides, scale) -> int:
    return load().attn_f16_validate(batch, heads, seq_q, seq_kv, head_dim,
                                    Q, _strides3(q_strides), K, _strides3(k_strides),
                                    V, _strides3(v_strides), O, _strides3(o_strides),
                                    float(scale))


def gemm_f16_run_info(plan: int, layout: int, M: int, N: int, K: int, lda: int,
                      split_k: int = 1) -> dict:
    """What gemm_f16_run_ex would enqueue for these sizes (nothing is run)."""
    info = (_c_int * 4)()
    _check(load().gemm_f16_run_info(plan, layout, M, N, K, lda, split_k, info),
           "gemm_f16_run_info")
    return {"kernel": info[0], "launches": info[1], "repack_a": bool(info[2]),
            "tile_width": info[3]}


def gemm_f16_run_choice(layout: int, M: int, N: int, K: int, lda: int, split_k: int = 1,
                        num_sms: int = 152, max_pairs: int = 76, max_quads: int = 36) -> dict:
    """gemm_f16_run_info for default options on a device with these facts
    (host only; the defaults are a GB300's)."""
    info = (_c_int * 4)()
    _check(load().gemm_f16_run_choice(layout, M, N, K, lda, split_k, num_sms, max_pairs,
                                      max_quads, info), "gemm_f16_run_choice")
    return {"kernel": info[0], "launches": info[1], "repack_a": bool(info[2]),
            "tile_width": info[3]}


def gemm_f16_kernel_time(plan: int) -> tuple:
    """(total milliseconds, launches) of the kernels timed since the last
    read (OPT_KERNEL_TIMING); waits for the recorded events."""
    ms = ctypes.c_double(0.0)
    n = _c_i64(0)
    _check(load().gemm_f16_kernel_time(plan, ctypes.byref(ms), ctypes.byref(n)),
           "gemm_f16_kernel_time")
    return ms.value, n.value


def attn_f16_key_ranges(plan: int, batch: int, heads: int, seq_q: int, seq_kv: int) -> int:
    """Key ranges attn_f16_fwd would use for these sizes (1: no split)."""
    n = _c_int(0)
    _check(load().attn_f16_key_ranges(plan, batch, heads, seq_q, seq_kv, ctypes.byref(n)),
           "attn_f16_key_ranges")
    return n.value


def gemm_f16_tile_order(tiles_m: int, tiles_n: int, order: int = 0) -> list:
    """Tile order as a list of (tile_m, tile_n)."""
    n = _check(load().gemm_f16_tile_order(tiles_m, tiles_n, order, None, 0),
               "gemm_f16_tile_order")
    buf = (ctypes.c_uint32 * n)()
    _check(load().gemm_f16_tile_order(tiles_m, tiles_n, order, buf, n), "gemm_f16_tile_order")
    return [(v & 0xFFFF, v >> 16) for v in buf]


def gemm_f16_pair_tiles(M: int, N: int, pairs: int, split_k: int = 1, order: int = 0,
                        tile_width: int = 256, K: int = 4096, with_parts: bool = False):
    """CTA-pair work list as (row0, col0, width) tuples; with ``with_parts``
    also the K parts of the last (len % pairs) tiles: (tiles, parts)."""
    parts = _c_int(1)
    n = _check(load().gemm_f16_pair_tiles(M, N, K, pairs, split_k, order, tile_width, None, 0,
                                          ctypes.byref(parts)), "gemm_f16_pair_tiles")
    buf = (ctypes.c_uint32 * n)()
    _check(load().gemm_f16_pair_tiles(M, N, K, pairs, split_k, order, tile_width, buf, n, None),
           "gemm_f16_pair_tiles")
    tiles = [((v & 0xFFFF) * 256, ((v >> 16) & 0x3FFF) * 128, 128 << (v >> 30)) for v in buf]
    return (tiles, parts.value) if with_parts else tiles


def gemm_f16_tile_shape() -> tuple:
    """(BM, BN, BK, STAGES) of the compiled kernel."""
    vals = [_c_int() for _ in range(4)]
    load().gemm_f16_tile_shape(*[ctypes.byref(v) for v in vals])
    return tuple(v.value for v in vals)


class Plan:
    """Owning wrapper of a plan handle."""

    def __init__(self, device: int = 0):
        self.device = device
        self.handle = gemm_f16_plan(device)

    def close(self):
        if self.handle:
            gemm_f16_destroy(self.handle)
            self.handle = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def status(self) -> int:
        return gemm_f16_status(self.handle)

    def set_option(self, option: int, value: int) -> None:
        gemm_f16_set_option(self.handle, option, value)

    def get_option(self, option: int) -> int:
        return gemm_f16_get_option(self.handle, option)

    def kernel_time(self) -> tuple:
        """(total milliseconds, launches) of the product / attention kernels
        timed since the last read (see OPT_KERNEL_TIMING)."""
        return gemm_f16_kernel_time(self.handle)


def _stream_handle(stream) -> int:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _operand(X, rows: int, cols: int, name: str):
    """(transposed, leading dimension) of a rows x cols view, or raise."""
    if X.stride(1) == 1 and (rows == 1 or X.stride(0) >= cols):
        return False, X.stride(0) if rows > 1 else cols
    if X.stride(0) == 1 and (cols == 1 or X.stride(1) >= rows):
        return True, X.stride(1) if cols > 1 else rows
    raise ValueError(f"{name} must be row-major or a transposed row-major view")


def matmul(plan: Plan, A, B, C=None, split_k: int = 1, stream=None):
    """C = A @ B for float16 CUDA tensors (C allocated if None).

    A and B may each be row-major or the transpose of a row-major tensor
    (``X.t()``); the matching operand layout is passed to the kernel, so no
    copy is made.  C must be row-major.
    """
    import torch
    if A.dtype != torch.float16 or B.dtype != torch.float16:
        raise TypeError("A and B must be torch.float16")
    if A.dim() != 2 or B.dim() != 2 or A.shape[1] != B.shape[0]:
        raise ValueError(f"shape mismatch {tuple(A.shape)} x {tuple(B.shape)}")
    M, K = A.shape
    N = B.shape[1]
    at, lda = _operand(A, M, K, "A")
    bt, ldb = _operand(B, K, N, "B")
    if C is None:
        C = torch.empty((M, N), dtype=torch.float16, device=A.device)
    elif C.dtype != torch.float16 or tuple(C.shape) != (M, N) or C.stride(1) != 1:
        raise ValueError("C must be a row-major float16 M x N tensor")
    layout = (LAYOUT_TN if at else 0) | (LAYOUT_NT if bt else 0)
    gemm_f16_run_ex(plan.handle, layout, M, N, K, A.data_ptr(), lda, B.data_ptr(), ldb,
                    C.data_ptr(), C.stride(0) if M > 1 else N, split_k, _stream_handle(stream))
    return C


def attention(plan: Plan, Q, K, V, O=None, scale=None, stream=None):
    """softmax(scale * Q K^T) V for float16 CUDA tensors of shape
    [batch, heads, seq, 256] (the last dimension contiguous; other strides
    free, so ``x.transpose(1, 2)`` of a [batch, seq, heads, 256] tensor works).
    ``scale`` defaults to 1/sqrt(256).  O is allocated if None."""
    import torch
    for name, X in (("Q", Q), ("K", K), ("V", V)):
        if X.dtype != torch.float16 or X.dim() != 4 or X.stride(3) != 1:
            raise ValueError(f"{name} must be a float16 [B, H, S, D] tensor with D contiguous")
    B, H, Sq, D = Q.shape
    Skv = K.shape[2]
    if tuple(K.shape) != (B, H, Skv, D) or tuple(V.shape) != (B, H, Skv, D):
        raise ValueError(f"shape mismatch {tuple(Q.shape)} {tuple(K.shape)} {tuple(V.shape)}")
    if O is None:
        O = torch.empty((B, H, Sq, D), dtype=torch.float16, device=Q.device)
    elif O.dtype != torch.float16 or tuple(O.shape) != (B, H, Sq, D) or O.stride(3) != 1:
        raise ValueError("O must be a float16 [B, H, Sq, D] tensor with D contiguous")
    if scale is None:
        scale = 1.0 / (D ** 0.5)
    st = lambda X: (X.stride(0), X.stride(1), X.stride(2))
    attn_f16_fwd(plan.handle, B, H, Sq, Skv, D, Q.data_ptr(), st(Q), K.data_ptr(), st(K),
                 V.data_ptr(), st(V), O.data_ptr(), st(O), scale, _stream_handle(stream))
    return O


def attn_f16_fwd_host(plan: int, batch: int, heads: int, seq_q: int, seq_kv: int, head_dim: int,
                      hQ: int, hK: int, hV: int, hO: int, scale: float, stream: int = 0) -> None:
    """The forward pass on contiguous host buffers (see attn_f16.h)."""
    _check(load().attn_f16_fwd_host(plan, batch, heads, seq_q, seq_kv, head_dim, hQ, hK, hV, hO,
                                    float(scale), stream), "attn_f16_fwd_host")


def attention_host(plan: Plan, hQ, hK, hV, hO, scale=None, stream=None):
    """attention() for contiguous float16 CPU tensors (pinned for asynchronous
    copies): Q, K, V are copied in and O out by the library, overlapping
    consecutive calls.  Synchronise the stream before reading hO."""
    import torch
    for name, X in (("Q", hQ), ("K", hK), ("V", hV), ("O", hO)):
        if X.dtype != torch.float16 or X.dim() != 4 or X.is_cuda or not X.is_contiguous():
            raise ValueError(f"{name} must be a contiguous float16 CPU tensor [B, H, S, D]")
    B, H, Sq, D = hQ.shape
    Skv = hK.shape[2]
    if (tuple(hK.shape) != (B, H, Skv, D) or tuple(hV.shape) != (B, H, Skv, D)
            or tuple(hO.shape) != (B, H, Sq, D)):
        raise ValueError("shape mismatch")
    if scale is None:
        scale = 1.0 / (D ** 0.5)
    attn_f16_fwd_host(plan.handle, B, H, Sq, Skv, D, hQ.data_ptr(), hK.data_ptr(), hV.data_ptr(),
                      hO.data_ptr(), scale, _stream_handle(stream))
    return hO
