"""bench.py's host-side accounting, without a GPU: the credited FLOPs of the five workloads
(the pages' convention: forward 2·B·H·T²·d, backward 2.5x), the launch list per head
dimension, the renamed workload variants and the spread statistics."""
from __future__ import annotations

import argparse
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402
import seeded_inputs as si  # noqa: E402

# (workload, forward GFLOP, backward GFLOP) as the metric credits them
CREDITED = [("tiny", 0.000524288, 0.00131072), ("gpt12m", 0.402653184, 1.00663296),
            ("gpt100m", 12.884901888, 32.21225472), ("gpt205m", 34.359738368, 85.89934592),
            ("long8k", 274.877906944, 687.19476736)]


@pytest.mark.parametrize("name,fwd,bwd", CREDITED)
def test_credited_flops(name, fwd, bwd):
    w = si.WORKLOADS[name]
    f, b = bench.credited_flops(*w.shape)
    assert abs(f / 1e9 - fwd) < 1e-9 and abs(b / 1e9 - bwd) < 1e-9


def test_kernel_flops_add_up_to_the_algorithmic_gemms():
    w = si.WORKLOADS["gpt205m"]
    kf = bench.kernel_flops(w)
    g = w.B * w.H * w.T * w.T * w.d  # one causal T x T GEMM
    assert kf["fwd"] == 2 * g and kf["bwd_dkdv"] == 4 * g and kf["bwd_dq"] == 3 * g
    assert kf["bwd"] == kf["bwd_dkdv"] + kf["bwd_dq"]


@pytest.mark.parametrize("d,fused,expect", [
    (32, False, ("fwd", "bwd_dq", "bwd_dkdv")), (64, False, ("fwd", "bwd_dq", "bwd_dkdv")),
    (80, False, ("fwd", "bwd_preprocess", "bwd_dkdv", "bwd_dq")),
    (128, False, ("fwd", "bwd_preprocess", "bwd_dkdv", "bwd_dq")),
    (64, True, ("fwd", "bwd_preprocess", "bwd_dkdv_dq", "bwd_dq_finish")),
    (128, True, ("fwd", "bwd_preprocess", "bwd_dkdv", "bwd_dq")),
])
def test_launch_list(d, fused, expect):
    assert bench.kernels_for(d, fused) == expect


def test_variants_are_renamed():
    w = si.WORKLOADS["long8k"]
    ns = argparse.Namespace(non_causal=True, head_dim=80)
    v = bench.variant(w, ns)
    assert v.name == "long8k_noncausal_d80" and not v.causal and v.d == 80 and v.T == w.T
    same = bench.variant(w, argparse.Namespace(non_causal=False, head_dim=128))
    assert same.name == "long8k" and same.d == 128


def test_spread():
    s = bench.spread([5.0, 1.0, 3.0, 2.0, 4.0])
    assert s == {"ms_min": 1.0, "ms_median": 3.0, "ms_p95": 5.0}


def test_default_line_is_the_largest_configuration(monkeypatch):
    """Without flags the bench runs long8k (B1 H16 T8192 d128), the largest single-GPU
    configuration, at N = 1."""
    import sys
    import bench
    import seeded_inputs as si
    monkeypatch.setattr(sys, "argv", ["bench.py"])
    args = bench.parse()
    assert args.workload == "long8k" and args.gpus == 1 and args.impl == "ours"
    big = max(si.WORKLOADS.values(), key=lambda w: sum(bench.credited_flops(*w.shape)))
    assert big.name == args.workload


def test_every_traffic_record_matches_its_kernel_source():
    """Each DRAM-traffic record under profiles/ was captured from the kernel source as it
    stands: a record whose source hash no longer matches would make the bench line's
    roofline.traffic null for that workload."""
    import json
    import os
    recs = json.load(open(os.path.join(bench.ROOT, "profiles", "traffic.json")))
    stale = [k for k in recs if bench.captured_traffic(*k.split(":", 1)) is None]
    assert not stale, f"records captured from other kernel sources: {stale}"
    for k in ("long8k:bwd_dkdv", "long8k:fwd", "gpt205m:bwd_dkdv"):
        assert k in recs


def test_sustained_peak_is_the_measured_one():
    """The second denominator is the measured seconds-long bf16 rate, below the burst peak."""
    import json
    import os
    peaks = json.load(open(os.path.join(bench.ROOT, "MEASURED_PEAKS.json")))
    sust, kind = bench.sustained_peak()
    assert kind == "measured" and sust == peaks["bf16_tflops_sustained"]
    assert sust < bench.load_peaks()[0]
