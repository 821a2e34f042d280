"""The CPU oracle against brute force, finite differences, closed forms, invariants,
a library routine and the pages' printed accumulator cell; then the same checks
against copies of the oracle with planted mistakes, each of which must be caught."""
from __future__ import annotations

import importlib.util
import json
import os
import types

import numpy as np
import pytest

import oracle
import seeded_inputs as si
from tests import oracle_pins as pins

ORACLE_SRC = os.path.join(os.path.dirname(oracle.__file__), "attention.py")


@pytest.mark.parametrize("T", [1, 2, 3, 17])
@pytest.mark.parametrize("causal", [True, False])
def test_brute_force_small(T, causal):
    pins.check_brute_force(oracle, T=T, d=8, seed=100 + T, causal=causal)


def test_brute_force_tiny_workload():
    """The tiny workload (B1 H2 T64 d32), head by head, against pure-Python loops."""
    w = si.WORKLOADS["tiny"]
    x = si.make_inputs(w)
    q, k, v, do = (si.bf16_bits_to_f64(x[n]) for n in ("q", "k", "v", "do"))
    o, lse = oracle.forward(q, k, v, w.scale, True)
    dq, dk, dv, _ = oracle.backward(q, k, v, do, w.scale, True)
    for h in range(w.H):
        O, L, dQ, dK, dV = pins.brute_head(q[0, h].tolist(), k[0, h].tolist(), v[0, h].tolist(),
                                           do[0, h].tolist(), w.scale, True)
        for a, b in ((o[0, h], O), (lse[0, h], L), (dq[0, h], dQ), (dk[0, h], dK), (dv[0, h], dV)):
            assert np.max(np.abs(a - b)) <= 1e-12


@pytest.mark.parametrize("causal", [True, False])
def test_finite_differences(causal):
    pins.check_finite_differences(oracle, causal=causal)


def test_finite_differences_tiny_workload_head():
    """Central differences over every Q, K, V element of one head of the tiny workload."""
    w = si.WORKLOADS["tiny"]
    x = si.make_inputs(w)
    q, k, v, do = (si.bf16_bits_to_f64(x[n])[0, 1].copy() for n in ("q", "k", "v", "do"))
    dq, dk, dv, _ = oracle.head_backward(q, k, v, do, w.scale, True)
    for xx, g in ((q, dq), (k, dk), (v, dv)):
        fd = np.zeros_like(xx)
        for i in range(xx.shape[0]):
            for c in range(xx.shape[1]):
                x0 = xx[i, c]
                h = 1e-6 * max(1.0, abs(x0))
                xx[i, c] = x0 + h
                lp = np.sum(do * oracle.head_forward(q, k, v, w.scale, True)[0])
                xx[i, c] = x0 - h
                lm = np.sum(do * oracle.head_forward(q, k, v, w.scale, True)[0])
                xx[i, c] = x0
                fd[i, c] = (lp - lm) / (2 * h)
        assert np.linalg.norm(fd - g) / np.linalg.norm(g) <= 1e-6


def test_lse_gradient():
    pins.check_lse_gradient(oracle)


@pytest.mark.parametrize("causal", [True, False])
def test_row_sums(causal):
    pins.check_row_sums(oracle, causal=causal)


def test_t1():
    pins.check_t1(oracle)


def test_q_zero():
    pins.check_q_zero(oracle)


def test_first_row():
    pins.check_first_row(oracle)


@pytest.mark.parametrize("causal", [True, False])
def test_gradient_sums(causal):
    pins.check_gradient_sums(oracle, causal=causal)


def test_prefix_locality():
    pins.check_prefix_locality(oracle)


def test_accumulator_cell():
    pins.check_accumulator_cell(oracle)


@pytest.mark.parametrize("causal", [True, False])
def test_against_torch_sdpa(causal):
    pins.check_against_torch_sdpa(oracle, causal=causal)


@pytest.mark.parametrize("name", ["tiny", "gpt12m"])
def test_fp32_instantiation(name):
    pins.check_fp32_instantiation(oracle, si.WORKLOADS[name])


def test_fp32_instantiation_long_context_head():
    """One head of the long-context stress shape (T=8192, d=128, Q,K ~ N(0, 9))."""
    w = si.WORKLOADS["long8k"].with_(H=1, T=2048)
    pins.check_fp32_instantiation(oracle, w)


def test_flop_convention_matches_pages():
    g = json.load(open(os.path.join(pins.GOLDEN, "flop_convention.json")))
    for r in g["rows"]:
        fwd, bwd = oracle.credited_flops(r["B"], r["H"], r["T"], r["d"])
        assert round(fwd / (r["ms"] * 1e-3) / 1e12, 1) == r["tflops_printed"]
        assert bwd == 2.5 * fwd


@pytest.mark.parametrize("causal", [True, False])
def test_gqa_finite_differences(causal):
    pins.check_gqa_finite_differences(oracle, causal=causal)


@pytest.mark.parametrize("H,H_kv", [(6, 2), (4, 1), (3, 3)])
def test_gqa_against_torch_sdpa(H, H_kv):
    pins.check_gqa_against_torch_sdpa(oracle, H=H, H_kv=H_kv)


def test_gqa_heads_subset():
    """dK / dV of a key/value head are NaN unless all its query heads are computed."""
    q = np.random.default_rng(5).standard_normal((1, 4, 8, 4))
    k = np.random.default_rng(6).standard_normal((1, 2, 8, 4))
    do = np.random.default_rng(7).standard_normal((1, 4, 8, 4))
    full = oracle.backward(q, k, k, do, 0.5)
    part = oracle.backward(q, k, k, do, 0.5, heads=[(0, 0), (0, 1), (0, 2)])
    assert np.array_equal(part[1][0, 0], full[1][0, 0]) and np.isnan(part[1][0, 1]).all()
    with pytest.raises(ValueError):
        oracle.forward(q, k[:, :1].repeat(3, axis=1), k[:, :1].repeat(3, axis=1), 0.5)


def test_heads_subset_matches_full():
    w = si.WORKLOADS["gpt12m"].with_(B=2, H=3, T=40)
    x = si.make_inputs(w)
    q, k, v, do = (si.bf16_bits_to_f64(x[n]) for n in ("q", "k", "v", "do"))
    o, lse = oracle.forward(q, k, v, w.scale)
    o2, lse2 = oracle.forward(q, k, v, w.scale, heads=[(1, 2)])
    assert np.array_equal(o[1, 2], o2[1, 2]) and np.isnan(o2[0, 0]).all()
    dq, dk, dv, D = oracle.backward(q, k, v, do, w.scale)
    assert np.allclose(D, oracle.preprocess_D(o, do), rtol=0, atol=1e-13)


# ---------------------------------------------------------------------------
# planted mistakes: each must make at least one pin fail
# ---------------------------------------------------------------------------

MUTATIONS = {
    "dK without scale": ("dk = (ds.T @ q) * dtype(scale)", "dk = (ds.T @ q)"),
    "dQ without scale": ("dq = (ds @ k) * dtype(scale)", "dq = (ds @ k)"),
    "dQ with transposed dS": ("dq = (ds @ k) * dtype(scale)", "dq = (ds.T @ k) * dtype(scale)"),
    "dV with untransposed P": ("dv = p.T @ do", "dv = p @ do"),
    "dS without the D term": ("ds = p * (dp - D[:, None])", "ds = p * dp"),
    "dS with D added": ("ds = p * (dp - D[:, None])", "ds = p * (dp + D[:, None])"),
    "dP with an extra scale": ("dp = do @ v.T", "dp = (do @ v.T) * dtype(scale)"),
    "mask excludes the diagonal": ("return j <= i", "return j < i"),
    "mask is anti-causal": ("return j <= i", "return j >= i"),
    "log base 2 in LSE": ("lse = m + np.log(l)", "lse = m + np.log2(l)"),
    "LSE without the max": ("lse = m + np.log(l)", "lse = np.log(l)"),
    "forward without scale": ("s = (q @ k.T) * dtype(scale)                       # S = Q K^T * scale",
                              "s = (q @ k.T)"),
    "P from the max, not LSE": ("p = np.exp(s - lse[:, None])                        # softmax",
                                "p = np.exp(s - m[:, None])  # softmax"),
    "D over the wrong axis": ("D = (do * np.asarray(o, dtype=dtype)).sum(axis=1)",
                              "D = (do * np.asarray(o, dtype=dtype)).sum(axis=1) * 0.5"),
    "GQA head mapping modulo": ("return h // (H // H_kv)", "return h % H_kv"),
    "GQA dK not summed over the group": ("dk[b, g] += dk_h", "dk[b, g] = dk_h"),
    "GQA dV not summed over the group": ("dv[b, g] += dv_h", "dv[b, g] = dv_h"),
}


def _mutant(old, new):
    src = open(ORACLE_SRC).read()
    assert src.count(old) >= 1, f"mutation anchor not found: {old!r}"
    src = src.replace(old, new, 1)
    mod = types.ModuleType("oracle_mutant")
    exec(compile(src, "oracle_mutant", "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name):
    mod = _mutant(*MUTATIONS[name])
    caught = []
    for check in pins.ALL_FAST_CHECKS:
        try:
            with np.errstate(all="ignore"):
                check(mod)
        except Exception as e:  # AssertionError or a shape/NaN failure
            caught.append((check.__name__, type(e).__name__))
    assert caught, f"planted mistake '{name}' passed every pin"
