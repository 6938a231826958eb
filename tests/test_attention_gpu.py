"""GPU parity of the attention forward kernel (attn_f16_fwd) against the FP64
oracle (oracle.attention_f16).

Criteria as for the GEMM ("Xe2 ESIMD GEMM" page, "Correctness testing"):
no NaN/Inf first, then relative RMS error < 0.5% and every element within
1e-2 * (|ref| + 1).  Exact cases pin the data paths: with all keys equal
the output is the mean of the value rows (exact for small integers and a
power-of-two key count), and with one-hot keys and a dominant score each
query copies one value row (exact).  Ramps of scores make the running
maximum move from block to block, so the output rescale runs (in every
block for the steep ramp).
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
import synthetic_inputs as si
from tests import oracle_cache, parity

pytestmark = pytest.mark.gpu

D = 256


@pytest.fixture(scope="module", params=[1, 2], ids=["cta1", "pair"])
def plan(request):
    """A plan pinned to one attention kernel: 1 = single CTA (128 query
    rows, 64-key blocks), 2 = CTA pair (256 query rows, 128-key blocks).
    Every test in this file runs on both."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import async_barrier_pipelined_gb300 as g
    from async_barrier_pipelined_gb300 import build
    build.build()
    p = g.Plan(0)
    p.set_option(g.OPT_ATTN_KERNEL, request.param)
    yield p
    p.close()


def _dev(bits, layout="bhsd", pad=0):
    """uint16 [B, H, S, D] bits -> CUDA float16 [B, H, S, D] view.

    layout "bhsd": rows of one head contiguous (row stride D + pad);
    "bshd": [B, S, H, D] storage seen as [B, H, S, D]."""
    import torch
    B, H, S, Dd = bits.shape
    if layout == "bhsd":
        host = np.full((B, H, S, Dd + pad), 0x7E00, np.uint16)
        host[..., :Dd] = bits
        t = torch.from_numpy(host.view(np.float16)).cuda()
        return t[..., :Dd]
    host = np.full((B, S, H, Dd + pad), 0x7E00, np.uint16)
    host[..., :Dd] = bits.transpose(0, 2, 1, 3)
    t = torch.from_numpy(host.view(np.float16)).cuda()
    return t[..., :Dd].transpose(1, 2)


def _run(plan, Qb, Kb, Vb, scale=None, layout="bhsd", pad=0, o_layout=None):
    import torch
    import async_barrier_pipelined_gb300 as g
    Q, K, V = _dev(Qb, layout, pad), _dev(Kb, layout, pad), _dev(Vb, layout, pad)
    B, H, Sq, _ = Qb.shape
    O = _dev(np.full((B, H, Sq, D), 0x7E00, np.uint16), o_layout or layout, pad)
    g.attention(plan, Q, K, V, O, scale=scale)
    torch.cuda.synchronize()
    st = plan.status()
    assert st == g.OK, g.gemm_f16_strerror(st)
    return O.cpu().numpy().astype(np.float64)


def _f16(x):
    return np.asarray(x, dtype=np.float64).astype(np.float16).view(np.uint16)


# ---------------------------------------------------------------- exact cases
@pytest.mark.parametrize("shape", [(1, 1, 128, 64), (2, 3, 200, 256), (1, 2, 1, 512)],
                         ids=lambda s: "x".join(map(str, s)))
def test_equal_keys_give_the_exact_mean(plan, shape):
    """K = 0: every score is 0, every weight 1, the output the mean of V.
    Small integers over a power-of-two key count: exact in binary16."""
    B, H, Sq, Skv = shape
    rng = np.random.default_rng(Skv)
    Q = _f16(rng.standard_normal((B, H, Sq, D)))
    K = np.zeros((B, H, Skv, D), np.uint16)
    Vv = rng.integers(-8, 9, (B, H, Skv, D)).astype(np.float64)
    o = _run(plan, Q, K, _f16(Vv))
    # the exact mean (an integer sum over a power of two), rounded once
    want = np.broadcast_to(Vv.mean(axis=2, keepdims=True), o.shape)
    assert np.array_equal(o, want.astype(np.float16).astype(np.float64))


@pytest.mark.parametrize("skv", [1, 63, 100, 1000])
def test_equal_keys_ragged_key_count_masks_the_tail(plan, skv):
    """A key count that is not a multiple of the 64-key block: the padded
    keys must get weight 0 (else the mean is taken over too many rows)."""
    rng = np.random.default_rng(skv + 1)
    Q = _f16(rng.standard_normal((1, 2, 130, D)))
    K = np.zeros((1, 2, skv, D), np.uint16)
    Vb = _f16(rng.integers(-8, 9, (1, 2, skv, D)))
    o = _run(plan, Q, K, Vb)
    ref = oracle.attention_f16(Q, K, Vb, 1 / 16)
    parity.check(o, ref, f"equal keys skv={skv}")
    # the mean rounded once to binary16, up to one unit in the last place
    assert np.max(np.abs(o - ref)) <= np.max(np.abs(ref)) * 2 ** -10 + 1e-7


@pytest.mark.parametrize("sq,skv", [(256, 256), (300, 200), (129, 65)])
def test_one_hot_keys_select_value_rows_exactly(plan, sq, skv):
    """Key j = e_(j mod 256); query i = 320 e_(pi(i)): the matching score is
    20, every other 0, so every other key's weight is below exp(-20) ~ 2e-9
    of the match's.  Their total pull on the output is then far below half
    a binary16 unit of any value row entry of magnitude >= 1/8, so each query
    returns value row pi(i) exactly (entries are nonzero multiples of 1/8)."""
    rng = np.random.default_rng(sq * skv)
    pi = rng.integers(0, skv, sq)
    Q = np.zeros((1, 1, sq, D))
    Q[0, 0, np.arange(sq), pi % D] = 320.0
    K = np.zeros((1, 1, skv, D))
    K[0, 0, np.arange(skv), np.arange(skv) % D] = 1.0      # skv <= 256: distinct keys
    Vv = rng.integers(1, 101, (1, 1, skv, D)) * rng.choice([-1.0, 1.0], (1, 1, skv, D)) / 8.0
    o = _run(plan, _f16(Q), _f16(K), _f16(Vv))
    assert np.array_equal(o[0, 0], Vv[0, 0, pi])


# ---------------------------------------------------------------- workloads
@pytest.mark.parametrize("name", ["attn_256", "attn_ragged"])
def test_workloads_full(plan, name):
    w = si.ATTN_WORKLOADS[name]
    Qb, Kb, Vb = w.bits()
    o = _run(plan, Qb, Kb, Vb)
    parity.check(o, oracle.attention_f16(Qb, Kb, Vb, w.scale), name)


def test_attn_4096_full(plan):
    """The throughput workload (4 x 16 x 4096 x 4096) in the launch
    configuration the benchmark times; every element of O against the
    oracle."""
    import torch
    import async_barrier_pipelined_gb300 as g
    Qb, Kb, Vb = oracle_cache.attn_inputs("attn_4096")
    # the cached inputs are read-only arrays: copy before handing them to torch
    Q, K, V = (torch.from_numpy(x.view(np.float16).copy()).cuda() for x in (Qb, Kb, Vb))
    O = g.attention(plan, Q, K, V)
    torch.cuda.synchronize()
    assert plan.status() == g.OK
    got = O.cpu().numpy().astype(np.float64)
    parity.check(got, oracle_cache.attn_ref("attn_4096"), "attn_4096")


SHAPES = [(1, 1, 1, 1), (1, 1, 1, 1000), (1, 1, 129, 65), (2, 2, 64, 64), (1, 3, 513, 127),
          (3, 1, 257, 2049),
          # one query row against many keys (key split with a single row),
          # many rows against one key, and many small heads
          (1, 2, 1, 6000), (1, 1, 3000, 1), (4, 24, 33, 70)]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_shape_sweep(plan, shape):
    B, H, Sq, Skv = shape
    w = si.attn_custom(B, H, Sq, Skv, seed=Sq * 31 + Skv)
    Qb, Kb, Vb = w.bits()
    parity.check(_run(plan, Qb, Kb, Vb), oracle.attention_f16(Qb, Kb, Vb, w.scale),
                 f"{shape}")


@pytest.mark.parametrize("top", [24.0, 160.0])
def test_running_max_moves(plan, top):
    """Scores ramp up along the keys (to about `top`), so the row maximum
    grows block after block: with top = 160 by ~13 (base 2) per 64-key
    block, more than the lazy-rescale threshold, so the accumulator is
    rescaled in every block; with top = 24 a few times."""
    rng = np.random.default_rng(2)
    Sq, Skv = 200, 1100
    Q = rng.standard_normal((1, 2, Sq, D))
    Q[..., 0] = 16.0
    K = rng.standard_normal((1, 2, Skv, D)) * 0.5
    K[..., 0] = np.linspace(0, top, Skv)
    Vb = _f16(rng.uniform(-1, 1, (1, 2, Skv, D)))
    Qb, Kb = _f16(Q), _f16(K)
    parity.check(_run(plan, Qb, Kb, Vb), oracle.attention_f16(Qb, Kb, Vb, 1 / 16), "ramp")


@pytest.mark.parametrize("sigma,scale", [(3.0, 1 / 16), (1.0, 0.2), (1.0, -0.05), (1.0, 0.0)])
def test_peaked_and_odd_scales(plan, sigma, scale):
    w = si.attn_custom(1, 2, 300, 700, seed=int(sigma * 10 + scale * 100), qk_sigma=sigma)
    Qb, Kb, Vb = w.bits()
    parity.check(_run(plan, Qb, Kb, Vb, scale=scale),
                 oracle.attention_f16(Qb, Kb, Vb, np.float32(scale)), f"sigma {sigma} scale {scale}")


@pytest.mark.parametrize("layout,pad", [("bshd", 0), ("bhsd", 40), ("bshd", 8)])
def test_strided_layouts(plan, layout, pad):
    """[B, S, H, D] storage and padded rows (padding holds NaN)."""
    w = si.attn_custom(2, 3, 150, 333, seed=17 + pad)
    Qb, Kb, Vb = w.bits()
    o = _run(plan, Qb, Kb, Vb, layout=layout, pad=pad)
    parity.check(o, oracle.attention_f16(Qb, Kb, Vb, w.scale), f"{layout} pad {pad}")


def test_output_rows_outside_untouched(plan):
    """O with padded rows: the NaN padding and the rows of other heads stay
    as they were (a ragged last query block must not spill over)."""
    import torch
    import async_barrier_pipelined_gb300 as g
    w = si.attn_custom(1, 2, 100, 80, seed=5)
    Qb, Kb, Vb = w.bits()
    Q, K, V = (_dev(x) for x in (Qb, Kb, Vb))
    big = torch.from_numpy(np.full((1, 2, 100, D + 16), 0x7E00, np.uint16).view(np.float16)).cuda()
    O = big[..., :D]
    g.attention(plan, Q, K, V, O)
    torch.cuda.synchronize()
    full = big.cpu().numpy().view(np.uint16)
    assert np.all(full[..., D:] == 0x7E00)
    parity.check(full[..., :D].view(np.float16).astype(np.float64),
                 oracle.attention_f16(Qb, Kb, Vb, w.scale), "padded O")


def test_repeat_runs_bitwise_identical(plan):
    w = si.attn_custom(1, 4, 384, 1024, seed=3)
    Qb, Kb, Vb = w.bits()
    o0 = _run(plan, Qb, Kb, Vb)
    for _ in range(5):
        assert np.array_equal(_run(plan, Qb, Kb, Vb).view(np.uint64), o0.view(np.uint64))


def test_invalid_arguments_enqueue_nothing(plan):
    import torch
    import async_barrier_pipelined_gb300 as g
    Q = torch.zeros((1, 1, 64, D), dtype=torch.float16, device="cuda")
    st = (64 * D, 64 * D, D)
    ptr = Q.data_ptr()
    cases = [
        ((1, 1, 64, 64, 128, ptr, st, ptr, st, ptr, st, ptr, st, 1.0), g.ERR_INVALID_ARG),
        ((0, 1, 64, 64, D, ptr, st, ptr, st, ptr, st, ptr, st, 1.0), g.ERR_INVALID_ARG),
        ((1, 1, 0, 64, D, ptr, st, ptr, st, ptr, st, ptr, st, 1.0), g.ERR_INVALID_ARG),
        ((1, 1, 64, 64, D, ptr + 2, st, ptr, st, ptr, st, ptr, st, 1.0), g.ERR_MISALIGNED),
        ((1, 1, 64, 64, D, ptr, (64 * D, 64 * D, D + 4), ptr, st, ptr, st, ptr, st, 1.0),
         g.ERR_MISALIGNED),
        ((1, 1, 64, 64, D, ptr, st, ptr, st, ptr, st, ptr, st, float("nan")), g.ERR_INVALID_ARG),
    ]
    for args, code in cases:
        with pytest.raises(g.GemmError) as e:
            g.attn_f16_fwd(plan.handle, *args, stream=0)
        assert e.value.code == code
    torch.cuda.synchronize()
    assert plan.status() == g.OK


@pytest.mark.parametrize("skv", [100, 200, 333])
def test_many_items_per_cluster(plan, skv):
    """The pair kernel is persistent: under an SM limit a few clusters walk
    many work items (256 query rows of one batch and head), reloading Q and
    handing O to the epilogue warps between items.  One to three key blocks
    per item make the item boundaries come fast.  The output must match the
    oracle and be bitwise the same for every number of clusters (the
    single-CTA kernel ignores the limit)."""
    import async_barrier_pipelined_gb300 as g
    w = si.attn_custom(2, 3, 600, skv, seed=skv + 7)   # 18 items, ragged last query tile
    Qb, Kb, Vb = w.bits()
    want = oracle.attention_f16(Qb, Kb, Vb, w.scale)
    outs = []
    try:
        for limit in (0, 6, 4, 2):
            plan.set_option(g.OPT_SM_LIMIT, limit)
            outs.append(_run(plan, Qb, Kb, Vb))
    finally:
        plan.set_option(g.OPT_SM_LIMIT, 0)
    parity.check(outs[0], want, f"skv {skv}")
    for o in outs[1:]:
        assert np.array_equal(o.view(np.uint64), outs[0].view(np.uint64))


@pytest.mark.parametrize("splits", [2, 3, 8, 64])
def test_key_split_matches_oracle(plan, splits):
    """The pair kernel cuts each item's keys into ranges, writes normalised
    FP32 partials with their row offsets and sums, and a second kernel merges
    them.  1000 keys are 8 blocks, the last one ragged (104 keys): 2 and 3
    ranges leave a short last range, 8 ranges are one block each, 64 is
    capped at 8.  The single-CTA kernel ignores the option."""
    import async_barrier_pipelined_gb300 as g
    w = si.attn_custom(1, 3, 300, 1000, seed=splits + 40)
    Qb, Kb, Vb = w.bits()
    try:
        plan.set_option(g.OPT_ATTN_SPLIT, splits)
        o = _run(plan, Qb, Kb, Vb)
    finally:
        plan.set_option(g.OPT_ATTN_SPLIT, 0)
    parity.check(o, oracle.attention_f16(Qb, Kb, Vb, w.scale), f"{splits} key ranges")


def test_key_split_bitwise_repeatable_and_strided(plan):
    """A split run with [B, S, H, D] storage and padded rows matches the
    oracle and repeats bit for bit."""
    import torch
    import async_barrier_pipelined_gb300 as g
    w = si.attn_custom(2, 2, 260, 700, seed=77)
    Qb, Kb, Vb = w.bits()
    want = oracle.attention_f16(Qb, Kb, Vb, w.scale)
    try:
        plan.set_option(g.OPT_ATTN_SPLIT, 3)
        outs = [_run(plan, Qb, Kb, Vb, layout="bshd", pad=8) for _ in range(3)]
    finally:
        plan.set_option(g.OPT_ATTN_SPLIT, 0)
    parity.check(outs[0], want, "split, bshd")
    for o in outs[1:]:
        assert np.array_equal(o.view(np.uint64), outs[0].view(np.uint64))


def test_key_ranges_query(plan):
    """attn_f16_key_ranges reports the split attn_f16_fwd uses: for the pair
    kernel the option capped at the block count and rounded to non-empty
    ranges, no split when the items fill the GPU and a split when they fill
    less than half of it; always 1 for the single-CTA kernel."""
    import async_barrier_pipelined_gb300 as g
    h = plan.handle
    single = plan.get_option(g.OPT_ATTN_KERNEL) == 1
    try:
        # 1000 keys = 8 blocks of 128; 5 ranges of 2 blocks would leave one empty
        for opt, want in ((3, 3), (64, 8), (5, 4)):
            plan.set_option(g.OPT_ATTN_SPLIT, opt)
            assert g.attn_f16_key_ranges(h, 1, 3, 300, 1000) == (1 if single else want)
        plan.set_option(g.OPT_ATTN_SPLIT, 0)
        assert g.attn_f16_key_ranges(h, 4, 16, 4096, 4096) == 1
        n = g.attn_f16_key_ranges(h, 1, 2, 256, 16384)   # 2 items, 128 blocks
        assert n == 1 if single else 2 <= n <= 64
    finally:
        plan.set_option(g.OPT_ATTN_SPLIT, 0)
    with pytest.raises(g.GemmError):
        g.attn_f16_key_ranges(h, 0, 1, 1, 1)


def test_host_entry_matches_device_path(plan):
    """attn_f16_fwd_host with pinned host Q, K, V, O: five calls in a row
    with different inputs and sizes, one of them on another stream (the two
    device sets alternate, the second and third calls grow theirs) give the
    device path's bits and meet the oracle's bounds."""
    import torch
    import async_barrier_pipelined_gb300 as g
    shapes = [(1, 2, 300, 500), (2, 1, 256, 256), (1, 3, 520, 700), (1, 2, 300, 500),
              (1, 1, 400, 600)]
    side = torch.cuda.Stream()
    calls = []
    for i, (B, H, Sq, Skv) in enumerate(shapes):
        w = si.attn_custom(B, H, Sq, Skv, seed=100 + i)
        qb, kb, vb = w.bits()
        hQ, hK, hV = (torch.from_numpy(x.view(np.float16).copy()).pin_memory()
                      for x in (qb, kb, vb))
        hO = torch.empty((B, H, Sq, D), dtype=torch.float16).pin_memory()
        # The third call runs on another stream, ordered between its
        # neighbours (a plan's workspace serves one pass at a time); the
        # plan's input copies for the fifth call reuse its set (without
        # growing it) only once its pass and output copy there are done.
        if i == 2:
            side.wait_stream(torch.cuda.current_stream())
        g.attention_host(plan, hQ, hK, hV, hO, scale=w.scale, stream=side if i == 2 else None)
        if i == 2:
            torch.cuda.current_stream().wait_stream(side)
        calls.append((hO, hQ, hK, hV, qb, kb, vb, w))
    torch.cuda.synchronize()
    assert plan.status() == g.OK
    for hO, hQ, hK, hV, qb, kb, vb, w in calls:
        got = hO.numpy().astype(np.float64)
        want_dev = _run(plan, qb, kb, vb, scale=w.scale)
        assert np.array_equal(got.view(np.uint64), want_dev.view(np.uint64))
        parity.check(got, oracle.attention_f16(qb, kb, vb, w.scale), f"host entry {qb.shape}")
    with pytest.raises(g.GemmError):
        g.attn_f16_fwd_host(plan.handle, 1, 1, 1, 1, 128, 1, 1, 1, 1, 0.0625, 0)


def test_host_entries_share_a_plan():
    """attn_f16_fwd_host and gemm_f16_run_host on one fresh plan, attention
    first: both entry points share the plan's input-copy stream and each
    keeps its own events and device sets."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import async_barrier_pipelined_gb300 as g
    from async_barrier_pipelined_gb300 import build
    build.build()
    with g.Plan(0) as p:
        w = si.attn_custom(1, 2, 300, 500, seed=7)
        qb, kb, vb = w.bits()
        hQ, hK, hV = (torch.from_numpy(x.view(np.float16).copy()).pin_memory()
                      for x in (qb, kb, vb))
        hO = torch.empty((1, 2, 300, D), dtype=torch.float16).pin_memory()
        g.attention_host(p, hQ, hK, hV, hO, scale=w.scale)
        gw = si.custom(300, 260, 200, seed=8)
        A, B = gw.pair_bits(0)
        hA = torch.from_numpy(A.view(np.float16)).pin_memory()
        hB = torch.from_numpy(B.view(np.float16)).pin_memory()
        hC = torch.full((300, 260), float("nan"), dtype=torch.float16).pin_memory()
        s = torch.cuda.current_stream()
        g.gemm_f16_run_host(p.handle, 300, 260, 200, hA.data_ptr(), 200, hB.data_ptr(), 260,
                            hC.data_ptr(), 260, 1, int(s.cuda_stream))
        hO2 = torch.empty_like(hO).pin_memory()
        g.attention_host(p, hQ, hK, hV, hO2, scale=w.scale)
        s.synchronize()
        assert p.status() == g.OK
        parity.check(hC.numpy().astype(np.float64), oracle.gemm_f16(A, B), "gemm host after attention")
        ref = oracle.attention_f16(qb, kb, vb, w.scale)
        parity.check(hO.numpy().astype(np.float64), ref, "attention host, first")
        assert np.array_equal(hO.numpy().view(np.uint16), hO2.numpy().view(np.uint16))
