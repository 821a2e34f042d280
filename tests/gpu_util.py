"""Helpers shared by the GPU tests: device tensors from the seeded bf16 bytes, the
oracle on the same bytes, and the error metrics with the tolerances they use."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import seeded_inputs as si

# Tolerances of the GPU path against the fp64 oracle.
TOL_O_MAX_ABS = 2e-2
TOL_O_REL_RMS = 5e-3
TOL_LSE_MAX_ABS = 1e-3
TOL_GRAD_REL_RMS = 1e-2


def to_device(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def max_abs(a, b):
    return float(np.max(np.abs(a - b))) if a.size else 0.0


def rel_rms(a, b):
    den = float(np.linalg.norm(b))
    return float(np.linalg.norm(a - b)) / den if den > 0 else float(np.linalg.norm(a - b))


def run_gpu(w: si.Workload, x=None):
    """fwd + bwd through the binding. Returns a dict of device tensors."""
    import causal_attention_gb300 as ca
    x = x or si.make_inputs(w)
    q, k, v, do = (to_device(x[n]) for n in ("q", "k", "v", "do"))
    o, lse = ca.forward(q, k, v, w.scale, w.causal)
    dq, dk, dv = ca.backward(q, k, v, o, do, lse, w.scale, w.causal)
    ca.check_device_error()
    return dict(o=o, lse=lse, dq=dq, dk=dk, dv=dv)


def run_oracle(w: si.Workload, x, heads=None):
    q, k, v, do = (si.bf16_bits_to_f64(x[n]) for n in ("q", "k", "v", "do"))
    o, lse = oracle.forward(q, k, v, w.scale, w.causal, heads=heads)
    dq, dk, dv, _ = oracle.backward(q, k, v, do, w.scale, w.causal, heads=heads)
    return dict(o=o, lse=lse, dq=dq, dk=dk, dv=dv)


def run_oracle_all_heads(w: si.Workload, x, workers: int = 8):
    """The oracle over every head of a workload, spread over a process pool."""
    from tests import oracle_pool
    return oracle_pool.all_heads(w.scale, w.causal, x, workers)


def compare(gpu, ref, heads=None):
    """Error metrics over the compared heads (all heads if None)."""
    out = {}
    for name in ("o", "lse", "dq", "dk", "dv"):
        g = to_f64(gpu[name])
        r = ref[name]
        if heads is not None:
            g = np.stack([g[b, h] for b, h in heads])
            r = np.stack([r[b, h] for b, h in heads])
        out[name] = (max_abs(g, r), rel_rms(g, r))
    return out


# Per-tile bar of the gradients: the whole-tensor bar applied to every 128-row tile of every
# head, with a factor 2 for tiles whose norm is below the tensor's average. A tile with one
# row wrong by about that row's own size has rel-RMS near sqrt(1/128) = 0.088 and fails it.
TOL_GRAD_TILE_REL_RMS = 2 * TOL_GRAD_REL_RMS


def tile_errors(gpu, ref, tile=128):
    """The worst 128-row tile of dQ, dK and dV over every head: {name: (rel-RMS of that
    tile, (b, h, first row), its max-abs error / the tile's max |ref|)}."""
    out = {}
    for name in ("dq", "dk", "dv"):
        g, r = to_f64(gpu[name]), ref[name]
        B, H, T, _ = r.shape
        worst = (-1.0, None, 0.0)
        for b in range(B):
            for h in range(H):
                for t0 in range(0, T, tile):
                    gt, rt = g[b, h, t0:t0 + tile], r[b, h, t0:t0 + tile]
                    e = rel_rms(gt, rt)
                    if e > worst[0]:
                        worst = (e, (b, h, t0), max_abs(gt, rt) / max(float(np.max(np.abs(rt))), 1e-30))
        out[name] = worst
    return out


def assert_tiles_within_tolerance(terr, label=""):
    for name, (e, where, rel_max) in terr.items():
        assert e <= TOL_GRAD_TILE_REL_RMS, f"{label} {name} tile {where}: rel-RMS {e:.3e} (max-abs / max {rel_max:.3e})"


def assert_within_tolerance(err, label=""):
    o_max, o_rms = err["o"]
    assert o_max <= TOL_O_MAX_ABS, f"{label} O max-abs {o_max:.3e}"
    assert o_rms <= TOL_O_REL_RMS, f"{label} O rel-RMS {o_rms:.3e}"
    assert err["lse"][0] <= TOL_LSE_MAX_ABS, f"{label} LSE max-abs {err['lse'][0]:.3e}"
    for g in ("dq", "dk", "dv"):
        assert err[g][1] <= TOL_GRAD_REL_RMS, f"{label} {g} rel-RMS {err[g][1]:.3e}"
