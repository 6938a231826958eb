"""CPU-only checks of the C-ABI library: it loads, exports every entry point
that include/gemm_f16.h and include/attn_f16.h declare, and its host-side logic (argument
validation, tile order) behaves as documented.  No compute call is made.
"""
from __future__ import annotations

import ctypes
import os
import re

import pytest

import async_barrier_pipelined_gb300 as g
from async_barrier_pipelined_gb300 import build as gbuild

HEADER = os.path.join(gbuild.INCLUDE, "gemm_f16.h")
HEADERS = [HEADER, os.path.join(gbuild.INCLUDE, "attn_f16.h")]


@pytest.fixture(scope="module")
def lib():
    gbuild.build()
    return g.load()


def _declared_functions():
    names = set()
    for h in HEADERS:
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names |= set(re.findall(r"\b((?:gemm|attn)_f16_\w+)\s*\(", text))
    return sorted(names)


def test_header_and_binding_agree():
    assert _declared_functions() == sorted(g.EXPORTED_SYMBOLS)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_strerror_covers_codes(lib):
    for code in (0, -1, -2, -3, -4, -5, -6, -7):
        assert g.gemm_f16_strerror(code) != "unknown error code"
    assert g.gemm_f16_strerror(-99) == "unknown error code"


def test_tile_shape(lib):
    assert g.gemm_f16_tile_shape() == (128, 256, 64, 4)


P = 1 << 20  # a 16-byte-aligned fake address (never dereferenced)


@pytest.mark.parametrize("args,code", [
    ((256, 256, 256, P, 256, P, 256, P, 256, 1), g.OK),
    ((4000, 4104, 3000, P, 3000, P, 4104, P, 4104, 1), g.OK),
    ((512, 512, 32768, P, 32768, P, 512, P, 512, 16), g.OK),
    ((1, 1, 1, P, 8, P, 8, P, 8, 1), g.OK),
    ((0, 8, 8, P, 8, P, 8, P, 8, 1), g.ERR_INVALID_ARG),
    ((8, 0, 8, P, 8, P, 8, P, 8, 1), g.ERR_INVALID_ARG),
    ((8, 8, 0, P, 8, P, 8, P, 8, 1), g.ERR_INVALID_ARG),
    ((8, 8, 8, 0, 8, P, 8, P, 8, 1), g.ERR_INVALID_ARG),
    ((8, 8, 8, P, 8, 0, 8, P, 8, 1), g.ERR_INVALID_ARG),
    ((8, 8, 8, P, 8, P, 8, 0, 8, 1), g.ERR_INVALID_ARG),
    ((8, 8, 16, P, 8, P, 8, P, 8, 1), g.ERR_INVALID_ARG),     # lda < K
    ((8, 16, 8, P, 8, P, 8, P, 16, 1), g.ERR_INVALID_ARG),    # ldb < N
    ((8, 16, 8, P, 8, P, 16, P, 8, 1), g.ERR_INVALID_ARG),    # ldc < N
    ((8, 8, 8, P, 8, P, 8, P, 8, 0), g.ERR_INVALID_ARG),      # split_k < 1
    ((8, 8, 128, P, 128, P, 8, P, 8, 3), g.ERR_INVALID_ARG),  # split_k > ceil(K/64)
    ((8, 8, 128, P, 128, P, 8, P, 8, 2), g.OK),
    ((8, 8, 8, P + 8, 8, P, 8, P, 8, 1), g.ERR_MISALIGNED),
    ((8, 8, 8, P, 8, P + 2, 8, P, 8, 1), g.ERR_MISALIGNED),
    ((8, 8, 8, P, 8, P, 8, P + 4, 8, 1), g.ERR_MISALIGNED),
    ((8, 8, 8, P, 12, P, 8, P, 8, 1), g.ERR_MISALIGNED),
    ((8, 8, 8, P, 8, P, 12, P, 8, 1), g.ERR_MISALIGNED),
    ((8, 8, 8, P, 8, P, 8, P, 12, 1), g.ERR_MISALIGNED),
])
def test_validate(lib, args, code):
    assert g.gemm_f16_validate(*args) == code


def test_null_plan_is_rejected(lib):
    assert lib.gemm_f16_run(None, 8, 8, 8, P, 8, P, 8, P, 8, 1, None) == g.ERR_INVALID_ARG
    assert lib.gemm_f16_status(None) == g.ERR_INVALID_ARG
    assert lib.gemm_f16_set_option(None, 1, 5) == g.ERR_INVALID_ARG
    ms, n = ctypes.c_double(1.0), ctypes.c_int64(1)
    assert lib.gemm_f16_kernel_time(None, ctypes.byref(ms), ctypes.byref(n)) == g.ERR_INVALID_ARG
    assert lib.gemm_f16_destroy(None) == g.OK


def test_plan_without_gpu_fails_cleanly(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    h = ctypes.c_void_p()
    rc = lib.gemm_f16_plan(ctypes.byref(h), 0)
    assert rc in (g.ERR_CUDA, g.ERR_INVALID_ARG)
    assert h.value is None


def _deinterleave_even(code):
    out = 0
    for b in range(16):
        out |= ((code >> (2 * b)) & 1) << b
    return out


@pytest.mark.parametrize("tm,tn", [(1, 1), (2, 1), (8, 4), (32, 16), (32, 17), (4, 2),
                                   (3, 50), (64, 64)])
def test_tile_order_is_a_permutation(lib, tm, tn):
    for order in (0, 1):
        tiles = g.gemm_f16_tile_order(tm, tn, order)
        assert len(tiles) == tm * tn
        assert sorted(tiles) == [(i, j) for i in range(tm) for j in range(tn)]


def test_row_major_order(lib):
    assert g.gemm_f16_tile_order(2, 3, 1) == [(0, 0), (0, 1), (0, 2), (1, 0), (1, 1), (1, 2)]


def test_morton_order_on_square_grid_is_z_order(lib):
    """On a 2^p x 2^p grid tile number t is (even bits of t, odd bits of t)."""
    tiles = g.gemm_f16_tile_order(16, 16, 0)
    for t, (m, n) in enumerate(tiles):
        assert m == _deinterleave_even(t)
        assert n == _deinterleave_even(t >> 1)


def test_morton_order_rectangular_keeps_z_order(lib):
    """Ragged grids: the order is the square grid's order with the
    out-of-range tiles removed (codes strictly increasing)."""
    def code(m, n):
        c = 0
        for b in range(16):
            c |= ((m >> b) & 1) << (2 * b) | ((n >> b) & 1) << (2 * b + 1)
        return c
    tiles = g.gemm_f16_tile_order(32, 17, 0)
    codes = [code(m, n) for m, n in tiles]
    assert codes == sorted(codes) and len(set(codes)) == len(codes)


def test_tile_order_rejects_bad_grid(lib):
    assert lib.gemm_f16_tile_order(0, 4, 0, None, 0) == g.ERR_INVALID_ARG
    assert lib.gemm_f16_tile_order(4, 65536, 0, None, 0) == g.ERR_INVALID_ARG
    assert lib.gemm_f16_tile_order(4, 4, 2, None, 0) == g.ERR_INVALID_ARG


def _covered(tiles, M, N):
    """Count how often each output element is covered by the pair tiles."""
    import numpy as np
    cov = np.zeros((M, N), np.int32)
    for r0, c0, w in tiles:
        cov[r0:min(r0 + 256, M), c0:min(c0 + w, N)] += 1
    return cov


@pytest.mark.parametrize("M,N", [(4096, 4096), (4000, 4104), (1024, 1024), (512, 512),
                                 (129, 300), (256, 129), (300, 384), (1, 1), (2000, 100),
                                 (777, 5000)])
@pytest.mark.parametrize("pairs", [76, 7, 1])
def test_pair_tiles_cover_output_exactly_once(lib, M, N, pairs):
    import numpy as np
    tiles = g.gemm_f16_pair_tiles(M, N, pairs, 1, 0)
    cov = _covered(tiles, M, N)
    assert np.all(cov == 1)
    for r0, c0, w in tiles:            # no tile starts outside the output
        assert r0 < M and c0 < N and w in (128, 256)


def _makespan(tiles, pairs):
    load = [0.0] * pairs
    for i, (_, _, w) in enumerate(tiles):
        load[i % pairs] += w / 256
    return max(load)


def _tail_makespan(tiles, parts, pairs):
    """Busiest pair's work in tile times when the last len % pairs tiles run
    as `parts` K parts each (units handed out round-robin)."""
    r = len(tiles) % pairs if parts > 1 else 0
    units = [w / 256 for *_, w in tiles[:len(tiles) - r]]
    for *_, w in tiles[len(tiles) - r:]:
        units += [w / 256 / parts] * parts
    load = [0.0] * pairs
    for i, x in enumerate(units):
        load[i % pairs] += x
    return max(load)


def test_pair_tiles_balance_the_last_wave(lib):
    # 4096^3: 256 wide tiles on 76 pairs = 3 full waves + 28; the 28 run as
    # two K halves each (56 units), so the busiest pair does 3.5 tiles' work
    t, parts = g.gemm_f16_pair_tiles(4096, 4096, 76, 1, K=4096, with_parts=True)
    assert len(t) == 256 and all(w == 256 for *_, w in t) and parts == 2
    assert _tail_makespan(t, parts, 76) == 3.5
    # ragged 4000 x 4104 x 3000: 256 tiles + 16 narrow remainder tiles = 3
    # waves + 44; 88 halves would not fit in one wave, so the 44 are cut
    # into narrow tiles instead (3.5 tiles' work for the busiest pair)
    t, parts = g.gemm_f16_pair_tiles(4000, 4104, 76, 1, K=3000, with_parts=True)
    assert parts == 1 and _makespan(t, 76) == 3.5
    # 1024 x 1024 x 4096: 16 tiles on 76 pairs, 32 halves; with K = 1024
    # (16 k-blocks) the halves would save less than their merge costs
    t, parts = g.gemm_f16_pair_tiles(1024, 1024, 76, 1, K=4096, with_parts=True)
    assert len(t) == 16 and parts == 2 and _tail_makespan(t, parts, 76) == 0.5
    assert g.gemm_f16_pair_tiles(1024, 1024, 76, 1, K=1024, with_parts=True)[1] == 1
    # a whole last wave: no parts
    assert g.gemm_f16_pair_tiles(4864, 4096, 76, 1, K=4096, with_parts=True)[1] == 1
    # too few k-blocks for parts of two: the 28 tiles become 56 narrow ones
    t, parts = g.gemm_f16_pair_tiles(4096, 4096, 76, 1, K=64, with_parts=True)
    assert parts == 1
    assert sum(w == 256 for *_, w in t) == 228 and sum(w == 128 for *_, w in t) == 56
    assert _makespan(t, 76) == 3.5
    # splits keep whole tiles (the split units are the parallelism)
    t, parts = g.gemm_f16_pair_tiles(512, 512, 76, 16, K=32768, with_parts=True)
    assert len(t) == 4 and all(w == 256 for *_, w in t) and parts == 1


def test_pair_tiles_reject_bad_arguments(lib):
    assert lib.gemm_f16_pair_tiles(0, 8, 8, 76, 1, 0, 256, None, 0, None) == g.ERR_INVALID_ARG
    assert lib.gemm_f16_pair_tiles(8, 8, 0, 76, 1, 0, 256, None, 0, None) == g.ERR_INVALID_ARG
    assert lib.gemm_f16_pair_tiles(8, 8, 8, 0, 1, 0, 256, None, 0, None) == g.ERR_INVALID_ARG
    assert lib.gemm_f16_pair_tiles(8, 8, 8, 76, 0, 0, 256, None, 0, None) == g.ERR_INVALID_ARG
    assert lib.gemm_f16_pair_tiles(8, 8, 8, 76, 1, 0, 384, None, 0, None) == g.ERR_INVALID_ARG
    assert lib.gemm_f16_pair_tiles(8, 8, 8, 76, 1, 0, 512, None, 0, None) == g.ERR_INVALID_ARG
    assert lib.gemm_f16_pair_tiles(8, 8, 8, 76, 1, 0, 256, None, 0, None) == 1


@pytest.mark.parametrize("layout,args,code", [
    (0, (16, 32, 64, P, 64, P, 32, P, 32, 1), g.OK),
    (1, (16, 32, 64, P, 16, P, 32, P, 32, 1), g.OK),       # A stored K x M: lda >= M
    (1, (16, 32, 64, P, 8, P, 32, P, 32, 1), g.ERR_INVALID_ARG),
    (1, (24, 32, 64, P, 24, P, 32, P, 32, 1), g.OK),       # lda need not reach K
    (2, (16, 32, 64, P, 64, P, 64, P, 32, 1), g.OK),       # B stored N x K: ldb >= K
    (2, (16, 32, 64, P, 64, P, 32, P, 32, 1), g.ERR_INVALID_ARG),
    (3, (16, 32, 64, P, 16, P, 64, P, 32, 1), g.OK),
    (3, (16, 32, 64, P, 64, P, 32, P, 32, 1), g.ERR_INVALID_ARG),
    (3, (16, 32, 64, P, 20, P, 64, P, 32, 1), g.ERR_MISALIGNED),
    (4, (16, 32, 64, P, 64, P, 32, P, 32, 1), g.ERR_INVALID_ARG),
    (-1, (16, 32, 64, P, 64, P, 32, P, 32, 1), g.ERR_INVALID_ARG),
])
def test_validate_layouts(lib, layout, args, code):
    assert g.gemm_f16_validate_ex(layout, *args) == code
    if layout == 0:
        assert g.gemm_f16_validate(*args) == code


_ST = (64 * 256, 64 * 256, 256)


@pytest.mark.parametrize("args,code", [
    ((1, 1, 64, 64, 256, P, _ST, P, _ST, P, _ST, P, _ST, 0.0625), g.OK),
    ((4, 16, 4096, 4096, 256, P, _ST, P, _ST, P, _ST, P, _ST, 0.0625), g.OK),
    ((1, 1, 64, 64, 128, P, _ST, P, _ST, P, _ST, P, _ST, 0.0625), g.ERR_INVALID_ARG),
    ((0, 1, 64, 64, 256, P, _ST, P, _ST, P, _ST, P, _ST, 0.0625), g.ERR_INVALID_ARG),
    ((1, 0, 64, 64, 256, P, _ST, P, _ST, P, _ST, P, _ST, 0.0625), g.ERR_INVALID_ARG),
    ((1, 1, 0, 64, 256, P, _ST, P, _ST, P, _ST, P, _ST, 0.0625), g.ERR_INVALID_ARG),
    ((1, 1, 64, 0, 256, P, _ST, P, _ST, P, _ST, P, _ST, 0.0625), g.ERR_INVALID_ARG),
    ((65536, 1, 64, 64, 256, P, _ST, P, _ST, P, _ST, P, _ST, 0.0625), g.ERR_INVALID_ARG),
    ((1, 1, 64, 64, 256, 0, _ST, P, _ST, P, _ST, P, _ST, 0.0625), g.ERR_INVALID_ARG),
    ((1, 1, 64, 64, 256, P, _ST, P, _ST, P, _ST, 0, _ST, 0.0625), g.ERR_INVALID_ARG),
    ((1, 1, 64, 64, 256, P, (64 * 256, 64 * 256, 128), P, _ST, P, _ST, P, _ST, 0.0625),
     g.ERR_INVALID_ARG),                                   # row stride < 256
    ((1, 1, 64, 64, 256, P, (0, 64 * 256, 256), P, _ST, P, _ST, P, _ST, 0.0625),
     g.ERR_INVALID_ARG),                                   # zero stride
    ((1, 1, 64, 64, 256, P, _ST, P, _ST, P, _ST, P, _ST, float("inf")), g.ERR_INVALID_ARG),
    ((1, 1, 64, 64, 256, P + 8, _ST, P, _ST, P, _ST, P, _ST, 0.0625), g.ERR_MISALIGNED),
    ((1, 1, 64, 64, 256, P, _ST, P, (64 * 256, 64 * 256, 260), P, _ST, P, _ST, 0.0625),
     g.ERR_MISALIGNED),
    ((1, 2, 64, 64, 256, P, (64 * 256, 64 * 256 + 4, 256), P, _ST, P, _ST, P, _ST, 0.0625),
     g.ERR_MISALIGNED),
    # [B, S, H, D] storage: head stride 256, row stride H * 256
    ((2, 8, 100, 300, 256, P, (100 * 8 * 256, 256, 8 * 256), P, (300 * 8 * 256, 256, 8 * 256),
      P, (300 * 8 * 256, 256, 8 * 256), P, (100 * 8 * 256, 256, 8 * 256), 0.0625), g.OK),
])
def test_attn_validate(lib, args, code):
    assert g.attn_f16_validate(*args) == code


@pytest.mark.parametrize("tiles,kblocks,want", [
    (76 + 38, 32, 2),    # 38 tiles left over: 76 halves fill one wave exactly
    (76 + 39, 32, 1),    # 39 left: 78 halves would need a second wave
    (76 + 38, 31, 1),    # fewer than 32 k-blocks: the halves would not pay
    (76, 64, 1),         # whole waves only
    (1, 32, 2),          # a single tile on 76 pairs
])
def test_pair_tail_halves_rule(lib, tiles, kblocks, want):
    """K halves for the tiles of a partial last wave: only with one split,
    256-wide tiles, at least 32 k-blocks, and all halves in one wave."""
    M, N = 256 * tiles, 256          # one pair-tile column: `tiles` tiles
    _, parts = g.gemm_f16_pair_tiles(M, N, 76, 1, K=64 * kblocks, with_parts=True)
    assert parts == want
    # never with a split
    assert g.gemm_f16_pair_tiles(M, N, 76, 2, K=64 * kblocks, with_parts=True)[1] == 1


@pytest.mark.parametrize("args,want", [
    # the benchmark's workloads on a GB300 (152 SMs, 76 pairs, 36 clusters of four)
    ((0, 256, 256, 256, 256, 1), (1, 1, False, 64)),         # single CTA, 64-wide tiles
    ((0, 1024, 1024, 1024, 1024, 1), (1, 1, False, 64)),
    ((0, 4096, 4096, 4096, 4096, 1), (2, 2, False, 256)),    # pair + K-halves merge
    ((0, 4000, 4104, 3000, 3000, 1), (3, 1, False, 256)),    # off-line A: cluster of four
    ((0, 512, 512, 32768, 32768, 16), (2, 2, False, 256)),   # pair + split reduction
    # the same ragged product with whole-line A rows: the pair kernel
    ((0, 4000, 4104, 3000, 3008, 1), (2, 1, False, 256)),
    # off-line A, but clusters of four would take more waves (3 of 36 vs 2 of 76)
    ((0, 4864, 2048, 1000, 1000, 1), (2, 2, True, 256)),
    # off-line A stored transposed: only the pair kernel, after a repack
    ((1, 4000, 4104, 3000, 4000, 1), (2, 2, True, 256)),
    # off-line A on a product too small for either
    ((0, 1000, 1000, 1000, 1000, 1), (1, 1, False, 64)),
])
def test_automatic_choice_on_a_gb300(lib, args, want):
    """The automatic kernel choice, pinned for the benchmark's workloads and
    the boundaries of the off-line-A rule, without a GPU."""
    info = g.gemm_f16_run_choice(*args)
    assert (info["kernel"], info["launches"], info["repack_a"], info["tile_width"]) == want


def test_automatic_choice_follows_the_device_facts(lib):
    ragged = (0, 4000, 4104, 3000, 3000, 1)
    # no clusters of four: the pair kernel after a repack of A
    info = g.gemm_f16_run_choice(*ragged, num_sms=152, max_pairs=76, max_quads=0)
    assert info["kernel"] == 2 and info["repack_a"] and info["launches"] == 2
    # fewer SMs: still 4 waves either way, clusters of four
    info = g.gemm_f16_run_choice(*ragged, num_sms=148, max_pairs=74, max_quads=36)
    assert info["kernel"] == 3 and not info["repack_a"]
    # no pairs at all: the single-CTA kernel
    info = g.gemm_f16_run_choice(0, 4096, 4096, 4096, 4096, 1, num_sms=152, max_pairs=0,
                                 max_quads=0)
    assert info["kernel"] == 1


@pytest.mark.parametrize("facts", [(0, 0, 0), (152, 77, 36), (152, 76, 39), (152, -1, 0)])
def test_automatic_choice_rejects_impossible_device_facts(lib, facts):
    with pytest.raises(g.GemmError):
        g.gemm_f16_run_choice(0, 256, 256, 256, 256, 1, *facts)
    with pytest.raises(g.GemmError):     # lda below K, like gemm_f16_run_info
        g.gemm_f16_run_choice(0, 256, 256, 256, 100, 1)
