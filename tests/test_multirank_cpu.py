"""The benchmark's multi-rank path on CPU (two gloo ranks, no GPU).

With N GPUs each rank runs an independent replica (the GEMM and attention
paths have no exchange step, so no collective touches the data path); only
the timing is combined: every rank's event time goes through a MAX
all-reduce, and the whole-job value is the work of all ranks over that
slowest time.  The reference arm runs on rank 0 only; other ranks exit 0
without work.
"""
from __future__ import annotations

import contextlib
import io
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = 10.0 + 5.0 * rank                    # rank 1 is the slow one
    worst = bench.max_over_ranks(ms, world)
    value = bench.whole_job_tflops(1e12, 10, world, worst)
    with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
        f.write(f"{worst} {value}\n")
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_value_with_two_gloo_ranks(tmp_path):
    mp = pytest.importorskip("torch.multiprocessing")
    port = _free_port()
    mp.spawn(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True)
    for rank in range(2):
        worst, value = map(float, open(tmp_path / f"rank{rank}.txt").read().split())
        assert worst == 15.0                   # both ranks see the slowest time
        assert value == pytest.approx(1e12 * 10 * 2 / 0.015 / 1e12)


def test_single_process_needs_no_collective():
    import bench
    assert bench.max_over_ranks(12.5, 1) == 12.5
    assert bench.whole_job_tflops(2e12, 4, 1, 8.0) == pytest.approx(2e12 * 4 / 0.008 / 1e12)


@pytest.mark.parametrize("workload", ["gemm_256", "attn_256"])
def test_reference_arm_runs_on_rank_zero_only(monkeypatch, workload):
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("LOCAL_RANK", "1")
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference", "--gpus", "2",
                                      "--steps", "1", "--warmup", "0", "--workload", workload])
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        rc = bench.main()
    assert rc == 0 and buf.getvalue() == ""
