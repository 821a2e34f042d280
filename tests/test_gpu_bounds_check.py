"""The bounds-checked build of the library (libattn_debug.so, compiled with
-DATTN_DEBUG_BOUNDS=1): every TMA coordinate, bulk-copy range and global store index of
the attention kernels is checked on the device before the access, and a failed check
skips the access, records itself in the device error word and makes check_device_error
raise ATTN_ERR_DEVICE_BOUNDS. This runs the edge shapes (T = 1, tile boundaries, ragged
tails, d = 32 / 64 / 80 / 128, causal and not), grouped key/value heads, persistent
multi-item launches, work items dealt in two groups of slices, tensors of more than 2^31
elements and a 131072-token sequence through it, in a process of its own: the outputs
must match the oracle (or, for the largest cases, be finite and repeat across identical
heads) and no check may fire. It stands in for a run under compute-sanitizer."""
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = r"""
import causal_attention_gb300 as ca
assert ca._dll._name.endswith("libattn_debug.so"), ca._dll._name
import numpy as np
import seeded_inputs as si
from tests import gpu_util as gu
from tests.test_gpu_parity import EDGE

cases = [si.Workload(f"edge{B}x{H}x{T}x{d}", B, H, T, d, causal=c, seed=77 + T + d) for B, H, T, d, c in EDGE]
cases += [si.Workload("multi64", 4, 16, 640, 64, seed=3), si.Workload("multi128", 2, 8, 640, 128, seed=4)]
for w in cases:
    x = si.make_inputs(w)
    heads = None if w.B * w.H <= 8 else [(0, 0), (w.B - 1, w.H - 1)]
    err = gu.compare(gu.run_gpu(w, x), gu.run_oracle(w, x, heads=heads), heads)  # raises on a fired check
    gu.assert_within_tolerance(err, w.name)
# grouped key/value heads (the split dK/dV with partial sums at MQA)
for B, H, Hkv, T, d in ((1, 8, 1, 257, 64), (1, 4, 2, 385, 128), (2, 4, 1, 300, 80)):
    seed = 600 + H + Hkv + d
    bits = {"q": si.normal_bf16_bits(seed, 0, (B, H, T, d)), "k": si.normal_bf16_bits(seed, 1, (B, Hkv, T, d)),
            "v": si.normal_bf16_bits(seed, 2, (B, Hkv, T, d)), "do": si.normal_bf16_bits(seed, 3, (B, H, T, d))}
    q, k, v, do = (gu.to_device(bits[n]) for n in ("q", "k", "v", "do"))
    o, lse = ca.forward(q, k, v, 1.0 / np.sqrt(d), True)
    dq, dk, dv = ca.backward(q, k, v, o, do, lse, 1.0 / np.sqrt(d), True)
    ca.check_device_error()
    for t in (o, lse, dq, dk, dv):
        assert bool(t.isfinite().all())
# slices dealt in two groups of three (their K and V exceed the kernels' L2 budget)
q, k, v, do = (gu.to_device(si.normal_bf16_bits(4300, i, (1, 6, 16384, 128))) for i in range(4))
o, lse = ca.forward(q, k, v, 1.0 / np.sqrt(128), True)
dq, dk, dv = ca.backward(q, k, v, o, do, lse, 1.0 / np.sqrt(128), True)
ca.check_device_error()
for t in (o, lse, dq, dk, dv):
    assert bool(t.isfinite().all())
del q, k, v, do, o, lse, dq, dk, dv
# tensors of more than 2^31 elements: the last heads' offsets pass every 32-bit index;
# four seeded heads repeated, so the last heads' outputs equal the first heads'
import torch
base = [gu.to_device(si.normal_bf16_bits(4400, i, (1, 4, 256, 128))) for i in range(4)]
q, k, v, do = (t.repeat(128, 129, 1, 1) for t in base)
o, lse = ca.forward(q, k, v, 1.0 / np.sqrt(128), True)
dq, dk, dv = ca.backward(q, k, v, o, do, lse, 1.0 / np.sqrt(128), True)
ca.check_device_error()
for t in (o, lse, dq, dk, dv):
    assert torch.equal(t[-1, -4:], t[0, :4])
del q, k, v, do, o, lse, dq, dk, dv
torch.cuda.empty_cache()
# one long sequence, T = 131072 (1024 key tiles)
q, k, v, do = (gu.to_device(si.normal_bf16_bits(4500, i, (1, 1, 131072, 64))) for i in range(4))
o, lse = ca.forward(q, k, v, 1.0 / np.sqrt(64), True)
dq, dk, dv = ca.backward(q, k, v, o, do, lse, 1.0 / np.sqrt(64), True)
ca.check_device_error()
for t in (o, lse, dq, dk, dv):
    assert bool(t.isfinite().all())
print("bounds-checked build: no check fired on", len(cases) + 6, "cases")
"""


def test_edge_shapes_under_device_bounds_checks():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from causal_attention_gb300 import _lib
    assert os.path.exists(_lib.DEBUG_LIB_PATH), "build() makes libattn_debug.so"
    env = dict(os.environ, ATTN_BOUNDS_CHECK="1", PYTHONPATH=ROOT)
    r = subprocess.run([sys.executable, "-c", SCRIPT], cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    print(r.stdout[-2000:], r.stderr[-4000:])
    assert r.returncode == 0, r.stderr[-4000:]
    assert "no check fired" in r.stdout
