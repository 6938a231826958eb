"""Host replay of the kernel's barrier protocol (tests/mbarrier_model/).

The model implements the mbarrier operations as the "mbarrier State and
Operations" page defines them and drives the producer / MMA / epilogue role
loops with the kernel's own index and parity helpers (schedule.h) under
seeded random interleavings of roles, copy completions and tensor-core
completions.  See model.cpp for the invariants checked.  attn_pair_model.cpp
replays the persistent CTA-pair attention kernel's protocol for one cluster
over several items (copy ring, Q reloads, S / P / O hand-over between the
MMA thread, the softmax warps and the epilogue warps of both CTAs, the
peer's signalling copies) and also checks that every parity wait returns
with exactly the phase it waited for; planted mistakes (a wait left out)
must make it fail.  quad_model.cpp replays the cluster-of-four GEMM
kernel (two CTA pairs multicasting A halves into each other's shared
memory, stages released by both pairs' commits) with its abort drains;
planted mistakes there must fail too.
"""
from __future__ import annotations

import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "mbarrier_model", "model.cpp")
PAIR_SRC = os.path.join(HERE, "mbarrier_model", "pair_model.cpp")
ATTN_SRC = os.path.join(HERE, "mbarrier_model", "attn_pair_model.cpp")
QUAD_SRC = os.path.join(HERE, "mbarrier_model", "quad_model.cpp")
CSRC = os.path.join(os.path.dirname(HERE), "async_barrier_pipelined_gb300", "csrc")
BUILD = os.path.join(HERE, "mbarrier_model", "_build")
EXE = os.path.join(BUILD, "model")
PAIR_EXE = os.path.join(BUILD, "pair_model")
ATTN_EXE = os.path.join(BUILD, "attn_pair_model")
QUAD_EXE = os.path.join(BUILD, "quad_model")


def _build(src, exe, defines=()):
    if shutil.which("g++") is None:
        pytest.skip("g++ not available")
    os.makedirs(BUILD, exist_ok=True)
    deps = [src, os.path.join(CSRC, "schedule.h"),
            os.path.join(HERE, "mbarrier_model", "mbar_model.h")]
    if not os.path.exists(exe) or any(os.path.getmtime(d) > os.path.getmtime(exe) for d in deps):
        tmp = exe + f".tmp{os.getpid()}"
        subprocess.run(["g++", "-std=c++17", "-O2", "-pthread", *[f"-D{d}" for d in defines],
                        "-I", CSRC, src, "-o", tmp], check=True)
        os.replace(tmp, exe)
    return exe


@pytest.fixture(scope="module")
def model():
    return _build(SRC, EXE)


@pytest.fixture(scope="module")
def pair_model():
    return _build(PAIR_SRC, PAIR_EXE)


@pytest.fixture(scope="module")
def attn_model():
    return _build(ATTN_SRC, ATTN_EXE)


@pytest.fixture(scope="module")
def quad_model():
    return _build(QUAD_SRC, QUAD_EXE)


def _run(exe, *args):
    r = subprocess.run([exe, *map(str, args)], capture_output=True, text=True, timeout=300)
    return r.returncode, r.stdout.strip()


# (stages, units, grid, cta, split_k, kblocks, seeds)
CASES = [
    (4, 2, 2, 0, 1, 4, 200),        # 256^3: 2 tiles, 4 k-blocks
    (4, 32, 32, 5, 1, 16, 200),     # 1024^3: 32 tiles on 32 CTAs
    (4, 512, 152, 0, 1, 64, 30),    # 4096^3, first CTA (4 tiles)
    (4, 512, 152, 151, 1, 64, 30),  # 4096^3, last CTA (3 tiles)
    (4, 544, 152, 7, 1, 47, 30),    # ragged 4000x4104x3000
    (4, 128, 128, 3, 16, 512, 10),  # split-K 512x512x32768, 16 splits of 32
    (1, 5, 2, 0, 1, 3, 200),        # one stage
    (2, 9, 4, 1, 3, 7, 200),        # uneven split ranges (7 k-blocks in 3)
    (3, 6, 1, 0, 2, 2, 200),        # one k-block per split
    (5, 3, 1, 0, 1, 1, 200),        # single k-block, more stages than fills
    (4, 1, 1, 0, 1, 1, 200),        # one unit, one k-block
    (8, 128, 128, 9, 1, 16, 100),   # 1024^3 with 64-wide tiles: 8-stage ring
    (6, 64, 64, 2, 1, 16, 100),     # 128-wide tiles: 6-stage ring
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(map(str, c)))
def test_protocol_interleavings(model, case):
    rc, out = _run(model, *case)
    assert rc == 0 and out.startswith("OK"), out


def test_fault_leaves_mma_blocked_on_the_starved_stage(model):
    # unit 2 belongs to CTA 0 of a 2-CTA grid; its first stage gets no copy
    rc, out = _run(model, 4, 8, 2, 0, 1, 4, 3, 2)
    assert rc == 0 and out.startswith("DEADLOCK-AS-EXPECTED"), out


def test_fault_on_other_cta_does_not_affect_this_one(model):
    rc, out = _run(model, 4, 8, 2, 1, 1, 4, 20, 2)
    assert rc == 0 and out.startswith("OK"), out


# CTA-pair protocol: (stages, units, pairs, pair, split_k, kblocks, seeds, mode[, arg])
PAIR_CASES = [
    (6, 284, 76, 0, 1, 64, 10, "normal"),     # 4096^2: 228 wide + 56 narrow units, first pair
    (6, 284, 76, 75, 1, 64, 10, "normal"),    # last pair (3 units)
    (6, 272, 76, 5, 1, 47, 10, "normal"),     # ragged 4000 x 4104 x 3000
    (6, 64, 64, 3, 16, 512, 4, "normal"),     # split-K units
    (2, 9, 4, 1, 3, 7, 100, "normal"),        # uneven split ranges
    (1, 5, 2, 0, 1, 3, 100, "normal"),        # one stage
    (6, 3, 1, 0, 1, 1, 100, "normal"),        # one k-block per unit
]


@pytest.mark.parametrize("case", PAIR_CASES, ids=lambda c: "-".join(map(str, c)))
def test_pair_protocol_interleavings(pair_model, case):
    rc, out = _run(pair_model, *case)
    assert rc == 0 and out.startswith("OK") and "deadlocks=0" in out, out


@pytest.mark.parametrize("case", [
    (6, 8, 2, 0, 1, 4, 50, "fault", 2),          # leader skips one fill's copies
    (6, 8, 2, 0, 1, 9, 50, "fault", 0),
    (6, 8, 2, 0, 1, 20, 100, "stop_leader", 5),  # leader producer times out early
    (3, 8, 2, 0, 1, 20, 100, "stop_leader", 0),
    (6, 8, 2, 0, 1, 20, 100, "stop_peer", 7),    # peer producer times out early
    (3, 8, 2, 0, 1, 20, 100, "stop_peer", 0),
    (4, 8, 1, 0, 2, 20, 100, "stop_peer", 13),
], ids=lambda c: "-".join(map(str, c)))
def test_pair_abort_drain_completes_issued_phases(pair_model, case):
    """Every seed deadlocks (the state the kernel's bounded waits escape);
    the leader's drain then completes every phase whose copies were issued,
    and only the faulted fill (whose bytes never come) stays open."""
    rc, out = _run(pair_model, *case)
    seeds = case[6]
    assert rc == 0 and out.startswith("OK") and f"deadlocks={seeds}" in out, out


def test_pair_fault_on_other_pair_does_not_affect_this_one(pair_model):
    rc, out = _run(pair_model, 6, 8, 2, 1, 1, 4, 20, "fault", 2)
    assert rc == 0 and "deadlocks=0" in out, out


# (ring slots, key blocks, seeds): 1 and 2 blocks (no reuse), odd / even
# counts, the kernel's 3-slot ring and others
# (ring, key blocks per item, items per cluster, key ranges per item, seeds);
# with ranges the units have ceil(blocks / ranges) blocks and the last fewer
ATTN_CASES = [(4, 1, 1, 1, 100), (4, 2, 3, 1, 60), (4, 5, 2, 1, 40), (4, 1, 5, 1, 60),
              (2, 3, 4, 1, 40), (3, 2, 3, 1, 60), (1, 2, 3, 1, 40),
              (4, 5, 2, 3, 40), (4, 8, 1, 8, 40), (3, 7, 2, 2, 40)]


@pytest.mark.parametrize("case", ATTN_CASES, ids=lambda c: "-".join(map(str, c)))
def test_attention_pair_protocol_interleavings(attn_model, case):
    rc, out = _run(attn_model, *case)
    assert rc == 0 and out.startswith("OK"), out


def test_attention_pair_fault_blocks_the_mma_on_the_starved_fill(attn_model):
    rc, out = _run(attn_model, 4, 3, 2, 1, 20, "fault")
    assert rc == 0 and out.startswith("DEADLOCK-AS-EXPECTED"), out


@pytest.mark.parametrize("plant,case,expect", [
    # the MMA thread does not wait for s_free: S of the next block may land
    # before every softmax warp has read S (needs two blocks per item; with
    # one, the wait for P of the block orders it anyway)
    ("PLANT_SKIP_S_FREE_WAIT", (4, 2, 4, 1, 200), "overwrites the S buffer"),
    # the item's first O += P V does not wait for o_free: it may overwrite O
    # before the epilogue warps read the previous item's O
    ("PLANT_SKIP_O_FREE_WAIT", (4, 1, 6, 1, 300), "overwrites O before the epilogue"),
    # the softmax does not wait for l_free: it may overwrite the row sums
    # before the epilogue warps read them
    ("PLANT_SKIP_L_FREE_WAIT", (4, 1, 6, 1, 300), "row sums overwritten"),
])
def test_attention_pair_model_catches_planted_mistakes(plant, case, expect):
    exe = _build(ATTN_SRC, ATTN_EXE + "_" + plant.lower(), defines=(plant,))
    rc, out = _run(exe, *case)
    assert rc != 0 and expect in out, out


# Cluster-of-four protocol: (stages, units, clusters, cluster, split_k,
# kblocks, seeds, mode[, args])
QUAD_CASES = [
    (6, 144, 36, 0, 1, 47, 10, "normal"),     # ragged 4000 x 4104 x 3000: 16 x 9 cluster tiles
    (6, 144, 36, 35, 1, 47, 10, "normal"),    # ... last cluster
    (6, 128, 36, 20, 1, 64, 10, "normal"),    # 4096^3: 16 x 8 cluster tiles
    (6, 32, 36, 3, 16, 512, 4, "normal"),     # 512 x 512 x 32768, 16 splits
    (2, 9, 4, 1, 3, 7, 50, "normal"),         # uneven split ranges
    (1, 5, 2, 0, 1, 3, 50, "normal"),         # one stage
    (6, 3, 1, 0, 1, 1, 50, "normal"),         # one k-block per unit
]


@pytest.mark.parametrize("case", QUAD_CASES, ids=lambda c: "-".join(map(str, c)))
def test_quad_protocol_interleavings(quad_model, case):
    rc, out = _run(quad_model, *case)
    assert rc == 0 and out.startswith("OK") and "deadlocks=0" in out, out


@pytest.mark.parametrize("case", [
    (6, 8, 2, 0, 1, 4, 50, "fault", 2),           # CTA 0 skips one fill's copies
    (6, 8, 2, 0, 1, 9, 50, "fault", 0),
    (6, 8, 2, 0, 1, 20, 50, "stop", 0, 5),        # a pair leader's producer times out
    (3, 8, 2, 0, 1, 20, 50, "stop", 1, 0),        # a pair peer's
    (6, 8, 2, 0, 1, 20, 50, "stop", 2, 7),        # the other pair's leader
    (3, 8, 2, 0, 1, 20, 50, "stop", 3, 4),        # the other pair's peer
    (4, 8, 1, 0, 2, 20, 50, "stop", 3, 13),
], ids=lambda c: "-".join(map(str, c)))
def test_quad_abort_drains_complete_issued_phases(quad_model, case):
    """Every seed deadlocks (the state the kernel's bounded waits escape);
    both leaders' drains then complete every phase whose copies were issued,
    and only the faulted fill (whose bytes never come, in both pairs) stays
    open."""
    rc, out = _run(quad_model, *case)
    seeds = case[6]
    assert rc == 0 and out.startswith("OK") and f"deadlocks={seeds}" in out, out


def test_quad_fault_on_other_cluster_does_not_affect_this_one(quad_model):
    rc, out = _run(quad_model, 6, 8, 2, 1, 1, 4, 20, "fault", 2)
    assert rc == 0 and "deadlocks=0" in out, out


@pytest.mark.parametrize("plant,case,expect", [
    # each leader's commit releases only its own pair's stages: the other
    # pair's producers multicast into a stage still being read
    ("PLANT_OWN_PAIR_RELEASE", (2, 6, 1, 0, 1, 8, 300, "normal"), "still being read"),
    # a leader's drain forgets the other pair's A halves
    ("PLANT_DRAIN_OWN_PAIR_ONLY", (6, 8, 2, 0, 1, 20, 100, "stop", 2, 7), "incomplete"),
    ("PLANT_DRAIN_OWN_PAIR_ONLY", (6, 8, 2, 0, 1, 20, 100, "stop", 0, 5), "incomplete"),
])
def test_quad_model_catches_planted_mistakes(plant, case, expect):
    exe = _build(QUAD_SRC, QUAD_EXE + "_" + plant.lower(), defines=(plant,))
    rc, out = _run(exe, *case)
    assert rc != 0 and expect in out, out
