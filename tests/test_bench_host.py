"""Host arithmetic of the benchmark's roofline record (no GPU).

The roofline divides a kernel's algorithmic work by its duration per
launch.  Both the event-pair time of the product kernel and the step time
bound that duration from above, so the smaller one is used and named; the
algorithmic bytes of an HBM-bound product kernel are A and B once plus C in
FP16, or the FP32 partial tiles when the K range is split.
"""
from __future__ import annotations

import os
import sys

import pytest

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402
import synthetic_inputs as si  # noqa: E402


def test_kernel_duration_takes_the_smaller_bound():
    assert bench.kernel_duration(0.080, 0.083) == (0.080, "kernel events")
    assert bench.kernel_duration(0.0102, 0.0067) == (0.0067, "timed-region step time")
    assert bench.kernel_duration(0.05, 0.05) == (0.05, "kernel events")


def test_kernel_and_compulsory_bytes():
    w = si.WORKLOADS["gemm_splitk"]           # 512 x 512 x 32768, 16 splits
    ab = 2 * (512 * 32768 + 32768 * 512)
    assert bench.compulsory_bytes(w) == ab + 2 * 512 * 512
    assert bench.kernel_bytes(w) == ab + 16 * 512 * 512 * 4
    w = si.WORKLOADS["gemm_4096"]
    assert bench.kernel_bytes(w) == bench.compulsory_bytes(w) == 2 * 3 * 4096 * 4096


@pytest.mark.parametrize("name", ["gemm_256", "gemm_1024", "gemm_4096", "gemm_ragged",
                                  "gemm_splitk"])
def test_bound_follows_the_ridge_point(name):
    """The benchmark's bound: tensor when FLOP per compulsory byte is at or
    above the ridge point of the measured peaks, else HBM."""
    w = si.WORKLOADS[name]
    peak, _, peak_hbm, _ = bench.load_peaks()
    ridge = peak * 1e12 / (peak_hbm * 1e9)
    fpb = w.flops / bench.compulsory_bytes(w)
    want_tensor = {"gemm_256": False, "gemm_1024": True, "gemm_4096": True,
                   "gemm_ragged": True, "gemm_splitk": False}[name]
    assert (fpb >= ridge) == want_tensor
