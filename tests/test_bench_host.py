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
    kv = bench.variant(w, argparse.Namespace(non_causal=False, head_dim=None, kv_heads=1))
    assert kv.name == "long8k_kv1" and kv.H == w.H and kv.seed == w.seed
    assert bench.variant(w, argparse.Namespace(non_causal=False, head_dim=None, kv_heads=16)).name == "long8k"


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


def _heads(seed, H, H_kv, T=40, d=8, bad=None):
    """Oracle outputs of every head of a tiny problem, as oracle_sample returns them, and
    the same as 'GPU' outputs (key/value-head dK, dV), optionally with one value wrong."""
    import numpy as np
    import oracle
    rng = np.random.default_rng(seed)
    q, do = rng.standard_normal((2, H, T, d))
    k, v = rng.standard_normal((2, H_kv, T, d))
    G = H // H_kv
    ref, dk, dv = {}, np.zeros_like(k), np.zeros_like(v)
    for h in range(H):
        o, lse, _ = oracle.head_forward(q[h], k[h // G], v[h // G], 0.3, True)
        dq, dkh, dvh, _ = oracle.head_backward(q[h], k[h // G], v[h // G], do[h], 0.3, True)
        ref[(0, h)] = (o, lse, dq, dkh, dvh)
        dk[h // G] += dkh
        dv[h // G] += dvh
    gpu = {(0, h): (r[0].copy(), r[1].copy(), r[2].copy(), dk[h // G].copy(), dv[h // G].copy())
           for (_, h), r in ref.items()}
    if bad is not None:
        i, delta = bad
        gpu[(0, 1)][i][5] += delta
    return gpu, ref


def test_parity_receipt_passes_exact_outputs_and_fails_planted_errors():
    gpu, ref = _heads(1, 4, 4)
    r = bench.parity_receipt(gpu, ref)
    assert r["pass"] and r["heads"] == 4 and r["o_max_abs"] == 0.0 and r["dk_rel_rms"] == 0.0
    for i, delta in ((0, 0.05), (1, 0.01), (2, 5.0), (3, 5.0), (4, 5.0)):  # O, LSE, dQ, dK, dV
        g, rf = _heads(1, 4, 4, bad=(i, delta))
        assert not bench.parity_receipt(g, rf)["pass"], i


def test_parity_receipt_sums_grouped_heads():
    """With 2 query heads per key/value head, dK and dV are compared as the group's sum,
    and only for groups whose query heads were all sampled."""
    gpu, ref = _heads(2, 4, 2)
    r = bench.parity_receipt(gpu, ref, G=2)
    assert r["pass"] and r["dk_rel_rms"] < 1e-12 and r["dv_rel_rms"] < 1e-12
    part = {key: ref[key] for key in [(0, 0)]}  # group 0 incomplete: no dK / dV comparison
    r = bench.parity_receipt({key: gpu[key] for key in part}, part, G=2)
    assert r["pass"] and "dk_rel_rms" not in r


def test_oracle_sample_maps_grouped_heads():
    """Under grouped key/value heads the CPU sample reads key/value head h // (H / H_kv)."""
    import numpy as np
    import seeded_inputs as si
    w = si.Workload("gqa_sample", 1, 4, 32, 8, seed=5)
    x = si.make_inputs(w)
    x = dict(x, k=np.ascontiguousarray(x["k"][:, :2]), v=np.ascontiguousarray(x["v"][:, :2]))
    f, s, n, outs = bench.oracle_sample(w, 4, x, H_kv=2)
    assert n == 4 and sorted(outs) == [(0, 0), (0, 1), (0, 2), (0, 3)] and f > 0


def test_gpu_lock_is_exclusive(tmp_path, monkeypatch):
    import fcntl
    monkeypatch.setattr(bench.tempfile, "gettempdir", lambda: str(tmp_path))
    with bench.GpuLock(7) as lk:
        with open(lk.path, "w") as other:
            with pytest.raises(BlockingIOError):
                fcntl.flock(other, fcntl.LOCK_EX | fcntl.LOCK_NB)
    with open(lk.path, "w") as other:  # released on exit
        fcntl.flock(other, fcntl.LOCK_EX | fcntl.LOCK_NB)
