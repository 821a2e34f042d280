"""bench.py's JSON line on a small workload: every key of the line's contract is present and
consistent, in both launch orders, and --order is refused where it does not apply."""
from __future__ import annotations

import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench(*args, timeout=600):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], capture_output=True, text=True,
                       timeout=timeout, cwd=ROOT)
    return r


def _line(r):
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    return json.loads(lines[0])


@pytest.mark.gpu
@pytest.mark.parametrize("order", ["fwd-bwd", "bwd-fwd"])
def test_bench_line_keys(order):
    d = _line(_bench("--workload", "gpt12m", "--steps", "5", "--warmup", "3", "--e2e-steps", "3",
                     "--no-cpu-baseline", "--order", order))
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "roofline", "e2e", "gpu_launches", "clocks", "kernels"):
        assert k in d, k
    assert d["value"] > 0 and d["unit"] == "TFLOP/s" and d["n_gpus"] == 1 and d["steps"] == 5 and d["warmup"] == 3
    assert d["higher_is_better"] is True and d["dtype"] == "bf16" and d["data"] == "synthetic"
    c = d["config"]
    assert c["workload"] == "gpt12m" and (c["B"], c["H"], c["T"], c["d"]) == (8, 6, 256, 64) and c["order"] == order
    rf = d["roofline"]
    assert rf["bound"] == "tensor" and rf["unit"] == "TFLOP/s" and rf["peak"] > 0
    assert abs(rf["frac"] - rf["achieved"] / rf["peak"]) < 1e-3
    sp = d["vs_sustained_peak"]  # the same rates against the seconds-long (power-capped) bf16 rate
    assert 0 < sp["peak"] <= rf["peak"] and abs(sp["frac"] - d["value"] / sp["peak"]) < 1e-3
    assert abs(sp["fwd_frac"] - d["fwd_tflops"] / sp["peak"]) < 1e-3
    e = d["e2e"]
    n = 8 * 6 * 256 * 64 * 2
    assert e["value"] > 0 and e["h2d_bytes_per_step"] == 4 * n and e["d2h_bytes_per_step"] == 4 * n + 8 * 6 * 256 * 4
    # three launches a step at d = 64: forward, dQ (which forms D), dK/dV
    assert d["gpu_launches"] == 3 * 5 and set(d["kernels"]) == {"fwd", "bwd_dq", "bwd_dkdv"}
    assert d["ms_per_step"] > 0 and all(k["ms"] > 0 for k in d["kernels"].values())
    # the forward and backward rates come from their own kernels' times, whatever the order
    from oracle import credited_flops
    fwd_f, bwd_f = credited_flops(8, 6, 256, 64)
    ks = d["kernels"]
    assert abs(d["fwd_tflops"] - fwd_f / (ks["fwd"]["ms"] * 1e-3) / 1e12) <= 0.01 * d["fwd_tflops"] + 0.01
    bwd_ms = ks["bwd_dq"]["ms"] + ks["bwd_dkdv"]["ms"]
    assert abs(d["bwd_tflops"] - bwd_f / (bwd_ms * 1e-3) / 1e12) <= 0.01 * d["bwd_tflops"] + 0.01


def test_order_is_refused_for_the_block():
    r = _bench("--block", "--order", "bwd-fwd", timeout=120)
    assert r.returncode != 0 and "--order applies to the attention line" in r.stderr


@pytest.mark.gpu
def test_bench_block_line_keys():
    d = _line(_bench("--block", "--workload", "gpt12m", "--steps", "4", "--warmup", "3", "--e2e-steps", "3"))
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "config", "roofline", "e2e",
              "gpu_launches", "clocks", "stages"):
        assert k in d, k
    c = d["config"]
    assert c["workload"] == "gpt12m_block" and c["C"] == 6 * 64 and c["rope"] is True
    assert set(d["stages"]) == {"qkv_proj", "attn_fwd", "out_proj", "out_proj_bwd", "attn_bwd", "qkv_proj_bwd"}
    assert d["value"] > 0 and d["e2e"]["value"] > 0 and d["e2e"]["h2d_bytes_per_step"] > 0
    assert d["e2e"]["d2h_bytes_per_step"] > 0 and d["gpu_launches"] > 0
    rf = d["roofline"]
    assert rf["peak"] > 0 and abs(rf["frac"] - rf["achieved"] / rf["peak"]) < 1e-3


@pytest.mark.gpu
@pytest.mark.parametrize("extra", [(), ("--kv-heads", "2")])
def test_bench_line_carries_a_passing_parity_receipt(extra):
    """With the CPU leg on, the line carries the receipt of a step at the same shape checked
    against the oracle before timing (every head of gpt12m fits the sample), and the
    cpu_baseline from that oracle run; with grouped key/value heads too."""
    d = _line(_bench("--workload", "gpt12m", "--steps", "5", "--warmup", "3", "--e2e-steps", "3", *extra))
    r = d["parity_receipt"]
    assert r["pass"] and r["heads"] == 8 * 6, r
    assert all(k in r for k in ("o_max_abs", "o_rel_rms", "lse_max_abs", "dq_rel_rms", "dk_rel_rms", "dv_rel_rms"))
    assert r["o_rel_rms"] <= 5e-3 and r["dk_rel_rms"] <= 1e-2
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] > 0 and cb["cores"] >= 1 and "48 of 48 heads" in cb["sample"]
