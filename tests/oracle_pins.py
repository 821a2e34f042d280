"""Checks that pin the CPU oracle to facts other than itself.

Each ``check_*`` takes an oracle module (the real one, or a copy with a planted
mistake) and raises AssertionError when the oracle disagrees with:
  * a brute-force restatement in pure-Python loops that uses the textbook softmax
    Jacobian (no D = rowsum(dO * O) identity, no saved logsumexp);
  * central finite differences of L = sum(dO * O);
  * closed forms (T = 1, Q = 0, the first causal row) and invariants (row sums,
    gradient sums, D = sum_j P dP);
  * a library routine (torch scaled_dot_product_attention in float64 with autograd);
  * a value the pages print (the Rigel accumulator cell).
"""
from __future__ import annotations

import json
import math
import os

import numpy as np

import seeded_inputs as si

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rand(seed, shape, sigma=1.0):
    return si.bf16_bits_to_f64(si.normal_bf16_bits(seed, 7, shape, sigma))


# ---------------------------------------------------------------------------
# brute force in pure Python (tiny inputs)
# ---------------------------------------------------------------------------

def brute_head(q, k, v, do, scale, causal):
    """Textbook attention and its gradient by explicit loops, for one head."""
    T, d = len(q), len(q[0])
    P = [[0.0] * T for _ in range(T)]
    for i in range(T):
        row = []
        for j in range(T):
            if causal and j > i:
                row.append(None)
            else:
                row.append(scale * sum(q[i][c] * k[j][c] for c in range(d)))
        mx = max(x for x in row if x is not None)
        e = [0.0 if x is None else math.exp(x - mx) for x in row]
        z = sum(e)
        for j in range(T):
            P[i][j] = e[j] / z
    O = [[sum(P[i][j] * v[j][c] for j in range(T)) for c in range(d)] for i in range(T)]
    lse = []
    for i in range(T):
        xs = [scale * sum(q[i][c] * k[j][c] for c in range(d))
              for j in range(T) if not (causal and j > i)]
        mx = max(xs)
        lse.append(mx + math.log(sum(math.exp(x - mx) for x in xs)))
    # gradient of L = sum(dO * O) through the softmax Jacobian
    dP = [[sum(do[i][c] * v[j][c] for c in range(d)) for j in range(T)] for i in range(T)]
    dS = [[0.0] * T for _ in range(T)]
    for i in range(T):
        for j in range(T):
            # dL/ds_ij = sum_k dP_ik * P_ik * (delta_kj - P_ij)
            dS[i][j] = sum(dP[i][kk] * P[i][kk] * ((1.0 if kk == j else 0.0) - P[i][j])
                           for kk in range(T))
    dV = [[sum(P[i][j] * do[i][c] for i in range(T)) for c in range(d)] for j in range(T)]
    dQ = [[scale * sum(dS[i][j] * k[j][c] for j in range(T)) for c in range(d)] for i in range(T)]
    dK = [[scale * sum(dS[i][j] * q[i][c] for i in range(T)) for c in range(d)] for j in range(T)]
    return (np.array(O), np.array(lse), np.array(dQ), np.array(dK), np.array(dV))


def check_brute_force(orc, T=17, d=8, seed=11, causal=True, tol=1e-12):
    q, k, v, do = (_rand(seed + i, (T, d)) for i in range(4))
    scale = 1.0 / math.sqrt(d)
    O, lse, dQ, dK, dV = brute_head(q.tolist(), k.tolist(), v.tolist(), do.tolist(), scale, causal)
    o2, lse2, _ = orc.head_forward(q, k, v, scale, causal)
    dq2, dk2, dv2, _ = orc.head_backward(q, k, v, do, scale, causal)
    for name, a, b in (("O", o2, O), ("LSE", lse2, lse), ("dQ", dq2, dQ), ("dK", dk2, dK), ("dV", dv2, dV)):
        err = float(np.max(np.abs(a - b))) if a.size else 0.0
        assert err <= tol * max(1.0, float(np.max(np.abs(b)))), f"brute force {name}: {err}"


# ---------------------------------------------------------------------------
# finite differences
# ---------------------------------------------------------------------------

def _loss(orc, q, k, v, do, scale, causal):
    o, _, _ = orc.head_forward(q, k, v, scale, causal)
    return float(np.sum(do * o))


def check_finite_differences(orc, T=24, d=8, seed=21, causal=True, tol=1e-6, stride=1):
    """Central differences of L = sum(dO * O) w.r.t. every element of Q, K, V."""
    q, k, v, do = (_rand(seed + i, (T, d)) for i in range(4))
    scale = 1.0 / math.sqrt(d)
    dq, dk, dv, _ = orc.head_backward(q, k, v, do, scale, causal)
    for name, x, g in (("Q", q, dq), ("K", k, dk), ("V", v, dv)):
        fd = np.zeros_like(x)
        flat = x.reshape(-1)
        idx = range(0, flat.size, stride)
        for n in idx:
            x0 = flat[n]
            h = 1e-6 * max(1.0, abs(x0))
            flat[n] = x0 + h
            lp = _loss(orc, q, k, v, do, scale, causal)
            flat[n] = x0 - h
            lm = _loss(orc, q, k, v, do, scale, causal)
            flat[n] = x0
            fd.reshape(-1)[n] = (lp - lm) / (2 * h)
        sel = np.zeros(flat.size, dtype=bool)
        sel[list(idx)] = True
        a, b = g.reshape(-1)[sel], fd.reshape(-1)[sel]
        rel = np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300)
        assert rel <= tol, f"finite differences d{name}: rel {rel:.3e}"


def check_lse_gradient(orc, T=16, d=8, seed=31, causal=True, tol=1e-6):
    """FD of sum_i w_i LSE_i w.r.t. Q against scale * w_i * sum_j P_ij k_j."""
    q, k, v = (_rand(seed + i, (T, d)) for i in range(3))
    w = _rand(seed + 9, (T,))
    scale = 1.0 / math.sqrt(d)
    _, _, p = orc.head_forward(q, k, v, scale, causal)
    analytic = scale * w[:, None] * (p @ k)
    fd = np.zeros_like(q)
    for i in range(T):
        for c in range(d):
            x0 = q[i, c]
            h = 1e-6 * max(1.0, abs(x0))
            q[i, c] = x0 + h
            lp = float(np.sum(w * orc.head_forward(q, k, v, scale, causal)[1]))
            q[i, c] = x0 - h
            lm = float(np.sum(w * orc.head_forward(q, k, v, scale, causal)[1]))
            q[i, c] = x0
            fd[i, c] = (lp - lm) / (2 * h)
    rel = np.linalg.norm(fd - analytic) / np.linalg.norm(analytic)
    assert rel <= tol, f"LSE gradient rel {rel:.3e}"


# ---------------------------------------------------------------------------
# closed forms and invariants
# ---------------------------------------------------------------------------

def check_row_sums(orc, T=40, d=16, seed=41, causal=True):
    q, k, v = (_rand(seed + i, (T, d), 2.0) for i in range(3))
    _, _, p = orc.head_forward(q, k, v, 0.25, causal)
    assert np.all(np.abs(p.sum(axis=1) - 1.0) <= 1e-12), "softmax rows do not sum to 1"
    if causal:
        assert np.all(p[~orc.causal_mask(T)] == 0.0), "masked probabilities are not 0"


def check_t1(orc, d=32, seed=51):
    q, k, v, do = (_rand(seed + i, (1, d)) for i in range(4))
    scale = 0.3
    o, lse, _ = orc.head_forward(q, k, v, scale, True)
    assert np.array_equal(o, v), "T=1: O != V"
    assert abs(lse[0] - scale * float(q[0] @ k[0])) <= 1e-14 * max(1, abs(lse[0])), "T=1: LSE"
    dq, dk, dv, _ = orc.head_backward(q, k, v, do, scale, True)
    # one key: softmax is constant 1, so dQ = dK = 0 and dV = dO
    assert np.max(np.abs(dq)) <= 1e-14 and np.max(np.abs(dk)) <= 1e-14, "T=1: dQ/dK != 0"
    assert np.allclose(dv, do, rtol=0, atol=1e-15), "T=1: dV != dO"


def check_q_zero(orc, T=33, d=16, seed=61):
    q = np.zeros((T, d))
    k, v = _rand(seed, (T, d)), _rand(seed + 1, (T, d))
    o, lse, _ = orc.head_forward(q, k, v, 0.125, True)
    prefix_mean = np.cumsum(v, axis=0) / np.arange(1, T + 1)[:, None]
    assert np.max(np.abs(o - prefix_mean)) <= 1e-13, "Q=0: O is not the causal prefix mean"
    assert np.max(np.abs(lse - np.log(np.arange(1, T + 1)))) <= 1e-13, "Q=0: LSE != ln(i+1)"


def check_first_row(orc, T=20, d=16, seed=71):
    q, k, v = (_rand(seed + i, (T, d)) for i in range(3))
    o, lse, _ = orc.head_forward(q, k, v, 0.25, True)
    assert np.array_equal(o[0], v[0]), "causal row 0: O_0 != V_0"
    assert abs(lse[0] - 0.25 * float(q[0] @ k[0])) <= 1e-14 * max(1, abs(lse[0])), "row 0 LSE"


def check_gradient_sums(orc, T=48, d=16, seed=81, causal=True):
    q, k, v, do = (_rand(seed + i, (T, d)) for i in range(4))
    dq, dk, dv, D = orc.head_backward(q, k, v, do, 0.25, causal)
    # softmax is invariant to shifting all keys: sum_j dK_j = 0
    assert np.max(np.abs(dk.sum(axis=0))) <= 1e-12 * max(1, np.max(np.abs(dk))), "sum_j dK_j != 0"
    # rows of P sum to 1: sum_j dV_j = sum_i dO_i
    assert np.max(np.abs(dv.sum(axis=0) - do.sum(axis=0))) <= 1e-12 * T, "sum dV != sum dO"
    # D_i = sum_j P_ij dP_ij
    _, _, p = orc.head_forward(q, k, v, 0.25, causal)
    dp = do @ v.T
    assert np.max(np.abs(D - (p * dp).sum(axis=1))) <= 1e-12 * T, "D != sum_j P dP"


def check_prefix_locality(orc, T=40, n=12, d=8, seed=131, tol=1e-12):
    """Causal attention is local to prefixes: rows i < n of O and LSE equal those of the
    problem cut to its first n rows; with dO zero past row n the whole backward equals the
    backward of that prefix (a later query has dP = 0 and D = 0, so dS = 0), zero on every
    later row; and row i alone is non-causal attention of query i over keys 0..i."""
    q, k, v, do = (_rand(seed + i, (T, d)) for i in range(4))
    do[n:] = 0.0
    o, lse, _ = orc.head_forward(q, k, v, 0.3, True)
    po, plse, _ = orc.head_forward(q[:n], k[:n], v[:n], 0.3, True)
    assert np.max(np.abs(o[:n] - po)) <= tol and np.max(np.abs(lse[:n] - plse)) <= tol, "prefix forward"
    dq, dk, dv, _ = orc.head_backward(q, k, v, do, 0.3, True)
    pdq, pdk, pdv, _ = orc.head_backward(q[:n], k[:n], v[:n], do[:n], 0.3, True)
    for name, full, pre in (("dQ", dq, pdq), ("dK", dk, pdk), ("dV", dv, pdv)):
        assert np.max(np.abs(full[:n] - pre)) <= tol, f"prefix {name}"
        assert not np.any(full[n:]), f"{name} nonzero past the prefix"
    for i in (0, n, T - 1):
        oi, li, _ = orc.head_forward(q[i:i + 1], k[:i + 1], v[:i + 1], 0.3, False)
        assert np.max(np.abs(oi[0] - o[i])) <= tol and abs(li[0] - lse[i]) <= tol, f"row {i} alone"


def check_accumulator_cell(orc):
    g = json.load(open(os.path.join(GOLDEN, "accumulator_cell.json")))
    d = g["d"]
    q = np.ones((1, d))
    k = np.full((1, d), g["k_rest"])
    k[0, 0] = g["k_first"]
    v = _rand(91, (1, d))
    o, lse, _ = orc.head_forward(q, k, v, 1.0, True)
    assert lse[0] == g["expected_score"], f"accumulator cell LSE {lse[0]}"
    assert np.array_equal(o, v)


def check_against_torch_sdpa(orc, B=1, H=2, T=64, d=32, seed=1000, causal=True):
    """torch scaled_dot_product_attention in float64 on the CPU, with autograd."""
    import torch
    rng = [si.bf16_bits_to_f64(si.normal_bf16_bits(seed, s, (B, H, T, d))) for s in range(4)]
    q, k, v, do = rng
    scale = 1.0 / math.sqrt(d)
    o, lse = orc.forward(q, k, v, scale, causal)
    dq, dk, dv, _ = orc.backward(q, k, v, do, scale, causal)
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    to = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=causal, scale=scale)
    to.backward(torch.tensor(do))
    s = torch.tensor(q) @ torch.tensor(k).transpose(-1, -2) * scale
    if causal:
        s = s.masked_fill(~torch.ones(T, T, dtype=torch.bool).tril(), float("-inf"))
    tlse = torch.logsumexp(s, dim=-1)
    for name, a, b in (("O", o, to.detach()), ("LSE", lse, tlse), ("dQ", dq, tq.grad),
                       ("dK", dk, tk.grad), ("dV", dv, tv.grad)):
        err = float(np.max(np.abs(a - b.numpy())))
        assert err <= 1e-12, f"torch sdpa {name}: {err}"


def check_fp32_instantiation(orc, w, tol=1e-4, heads=None):
    """The fp32 build of the oracle stays within the pages' 1e-4 of the fp64 one."""
    x = si.make_inputs(w)
    q, k, v, do = (si.bf16_bits_to_f64(x[n]) for n in ("q", "k", "v", "do"))
    res = {}
    for dt in (np.float64, np.float32):
        o, lse = orc.forward(q, k, v, w.scale, w.causal, dtype=dt, heads=heads)
        dq, dk, dv, _ = orc.backward(q, k, v, do, w.scale, w.causal, dtype=dt, heads=heads)
        res[dt] = (o, lse, dq, dk, dv)
    for name, a, b in zip(("O", "LSE", "dQ", "dK", "dV"), res[np.float32], res[np.float64]):
        m = ~np.isnan(b)
        err = float(np.max(np.abs(a[m].astype(np.float64) - b[m])))
        assert err <= tol, f"fp32 vs fp64 {name}: {err:.3e}"


def check_gqa_finite_differences(orc, B=1, H=4, H_kv=2, T=10, d=4, seed=301, causal=True, tol=1e-6):
    """Grouped key/value heads: central differences of L = sum(dO * O) w.r.t. every
    element of the shared K and V (each feeds H / H_kv query heads) and of Q, against
    the backward's dK, dV (sums over the group) and dQ."""
    q = _rand(seed, (B, H, T, d))
    k, v = _rand(seed + 1, (B, H_kv, T, d)), _rand(seed + 2, (B, H_kv, T, d))
    do = _rand(seed + 3, (B, H, T, d))
    scale = 1.0 / math.sqrt(d)
    dq, dk, dv, _ = orc.backward(q, k, v, do, scale, causal)

    def loss():
        o, _ = orc.forward(q, k, v, scale, causal)
        return float(np.sum(do * o))

    for name, x, g in (("Q", q, dq), ("K", k, dk), ("V", v, dv)):
        flat, fd = x.reshape(-1), np.zeros(x.size)
        for n in range(flat.size):
            x0 = flat[n]
            h = 1e-6 * max(1.0, abs(x0))
            flat[n] = x0 + h
            lp = loss()
            flat[n] = x0 - h
            lm = loss()
            flat[n] = x0
            fd[n] = (lp - lm) / (2 * h)
        rel = np.linalg.norm(g.reshape(-1) - fd) / max(np.linalg.norm(fd), 1e-300)
        assert rel <= tol, f"GQA finite differences d{name}: rel {rel:.3e}"


def check_gqa_against_torch_sdpa(orc, B=1, H=6, H_kv=2, T=24, d=8, seed=311, causal=True):
    """torch scaled_dot_product_attention with enable_gqa (query head h reads key/value
    head h // (H / H_kv)), float64 on the CPU, with autograd."""
    import torch
    q = _rand(seed, (B, H, T, d))
    k, v = _rand(seed + 1, (B, H_kv, T, d)), _rand(seed + 2, (B, H_kv, T, d))
    do = _rand(seed + 3, (B, H, T, d))
    scale = 1.0 / math.sqrt(d)
    o, lse = orc.forward(q, k, v, scale, causal)
    dq, dk, dv, _ = orc.backward(q, k, v, do, scale, causal)
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    to = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=causal, scale=scale,
                                                          enable_gqa=True)
    to.backward(torch.tensor(do))
    for name, a, b in (("O", o, to.detach()), ("dQ", dq, tq.grad), ("dK", dk, tk.grad), ("dV", dv, tv.grad)):
        err = float(np.max(np.abs(a - b.numpy())))
        assert err <= 1e-12, f"torch sdpa (GQA) {name}: {err}"


ALL_FAST_CHECKS = (
    check_brute_force,
    check_finite_differences,
    check_lse_gradient,
    check_row_sums,
    check_t1,
    check_q_zero,
    check_first_row,
    check_gradient_sums,
    check_prefix_locality,
    check_accumulator_cell,
    check_gqa_finite_differences,
    check_gqa_against_torch_sdpa,
)
