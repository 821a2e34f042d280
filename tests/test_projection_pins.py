"""The projection oracle against its pins (CPU only), and planted mistakes that the
pins must catch."""
from __future__ import annotations

import os
import types

import numpy as np
import pytest

from oracle import projections
from tests import projection_pins as pins

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle", "projections.py")


@pytest.mark.parametrize("check", pins.ALL_CHECKS, ids=lambda c: c.__name__)
def test_pin(check):
    check(projections)


MUTATIONS = {
    "nt computes A B": ('        return a @ b.T', '        return a @ b'),
    "tn computes A B^T": ('        return a.T @ b', '        return a @ b.T'),
    "heads split token-major": ("return y.reshape(B, T, n_heads, d).transpose(0, 2, 1, 3).copy()",
                                "return y.reshape(B, n_heads, T, d).copy()"),
    "K and V blocks swapped": ("    k = split_heads(y[:, H * d: (H + H_kv) * d], B, T, H_kv, d)\n"
                               "    v = split_heads(y[:, (H + H_kv) * d:], B, T, H_kv, d)",
                               "    v = split_heads(y[:, H * d: (H + H_kv) * d], B, T, H_kv, d)\n"
                               "    k = split_heads(y[:, (H + H_kv) * d:], B, T, H_kv, d)"),
    "RoPE pairs by halves": ("    x0, x1 = x[..., 0::2], x[..., 1::2]",
                             "    x0, x1 = x[..., : d // 2], x[..., d // 2:]"),
    "RoPE frequency exponent sign": ("theta = base ** (-2.0 * k / d)", "theta = base ** (2.0 * k / d)"),
    "RoPE positions from 1": ("np.arange(T, dtype=np.float64)[:, None]", "np.arange(1, T + 1, dtype=np.float64)[:, None]"),
    "RoPE rotation sense": ("    out[..., 0::2] = x0 * c - x1 * s\n    out[..., 1::2] = x0 * s + x1 * c",
                            "    out[..., 0::2] = x0 * c + x1 * s\n    out[..., 1::2] = -x0 * s + x1 * c"),
    "RoPE backward not inverted": ("dq, dk = rope(dq, inverse=True), rope(dk, inverse=True)",
                                   "dq, dk = rope(dq), rope(dk)"),
    "RoPE on v too": ("        q, k = rope(q), rope(k)\n", "        q, k, v = rope(q), rope(k), rope(v)\n"),
    "dO with W_o transposed": ('do = split_heads(gemm(dy2, w_o, "nn"), B, T, H, d)',
                               'do = split_heads(gemm(dy2, w_o.T, "nn"), B, T, H, d)'),
    "dW_qkv with X in time-major token order": ('dw = gemm(dy, x.reshape(B * T, C), "tn")',
                                                'dw = gemm(dy, x.transpose(1, 0, 2).reshape(B * T, C), "tn")'),
    "dX without the V block": ("dy = np.concatenate([merge_heads(dq), merge_heads(dk), merge_heads(dv)], axis=1)",
                               "dy = np.concatenate([merge_heads(dq), merge_heads(dk), 0 * merge_heads(dv)], axis=1)"),
}


def _mutant(old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor not found once: {old!r}"
    mod = types.ModuleType("projections_mutant")
    exec(compile(src.replace(old, new), "projections_mutant", "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name):
    mod = _mutant(*MUTATIONS[name])
    caught = []
    for check in pins.ALL_CHECKS:
        try:
            with np.errstate(all="ignore"):
                check(mod)
        except Exception as e:  # AssertionError, or a shape / NaN failure
            caught.append((check.__name__, type(e).__name__))
    assert caught, f"planted mistake '{name}' passed every pin"
