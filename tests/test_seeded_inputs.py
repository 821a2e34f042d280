"""The shared input generator: bf16 rounding against torch, determinism, moments."""
import numpy as np
import torch

import seeded_inputs as si


def test_bf16_rounding_matches_torch():
    x = (si.normal_f64(5, 0, 100000) * 3.0).astype(np.float32)
    # include exact ties and values near bf16 boundaries
    ties = np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -1.0 - 2 ** -8, 448.0, 0.0625, 1e-30], np.float32)
    x = np.concatenate([x, ties])
    ours = si.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    back = si.bf16_bits_to_f64(ours)
    assert np.array_equal(back, torch.from_numpy(x).to(torch.bfloat16).double().numpy())


def test_deterministic_and_counter_based():
    a = si.uniform_u64(1, 2, 1000)
    b = si.uniform_u64(1, 2, 10, start=500)
    assert np.array_equal(a[500:510], b)
    assert not np.array_equal(si.uniform_u64(1, 3, 1000), a)


def test_normal_moments():
    z = si.normal_f64(9, 1, 400000)
    assert abs(z.mean()) < 0.01 and abs(z.std() - 1.0) < 0.01


def test_workloads_shapes():
    w = si.WORKLOADS["long8k"]
    assert w.shape == (1, 16, 8192, 128) and abs(w.scale - 128 ** -0.5) < 1e-15
    x = si.make_inputs(si.WORKLOADS["tiny"])
    assert x["q"].dtype == np.uint16 and x["q"].shape == (1, 2, 64, 32)
    q = si.bf16_bits_to_f64(si.normal_bf16_bits(1004, 0, (1, 1, 4096, 128), 3.0))
    assert 2.9 < q.std() < 3.1
