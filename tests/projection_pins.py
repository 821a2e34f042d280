"""Checks that pin the projection oracle (``oracle.projections``) to facts other than
itself. Each ``check_*`` takes the module (the real one, or a copy with a planted
mistake) and raises when it disagrees with:
  * pure-Python loops over the index definitions (the three GEMM orientations, the
    head split, the Q / K / V column ranges of the QKV weight);
  * the closed forms the pages' RoPE formulas give for one-hot inputs (interleaved
    pairs; theta_0 = 1 and theta_1 = base^(-2/d)) and the rotation's invariants
    (pair norms, inverse, dot products depending only on the position difference);
  * central finite differences of L = sum(G * outputs) through the forward;
  * a library routine (torch.nn.functional.linear in float64 with autograd).
"""
from __future__ import annotations

import math

import numpy as np

import seeded_inputs as si


def _rand(seed, shape, sigma=1.0):
    return si.bf16_bits_to_f64(si.normal_bf16_bits(seed, 9, shape, sigma))


def check_gemm_brute_force(mod):
    M, N, K = 3, 4, 5
    a_mk, a_km = _rand(1, (M, K)), _rand(2, (K, M))
    b_nk, b_kn = _rand(3, (N, K)), _rand(4, (K, N))
    cases = {"nt": (a_mk, b_nk, lambda i, j, k: a_mk[i, k] * b_nk[j, k]),
             "nn": (a_mk, b_kn, lambda i, j, k: a_mk[i, k] * b_kn[k, j]),
             "tn": (a_km, b_kn, lambda i, j, k: a_km[k, i] * b_kn[k, j])}
    for layout, (a, b, term) in cases.items():
        c = mod.gemm(a, b, layout)
        assert c.shape == (M, N), layout
        for i in range(M):
            for j in range(N):
                want = math.fsum(term(i, j, k) for k in range(K))
                assert abs(c[i, j] - want) <= 1e-12 * (1 + abs(want)), (layout, i, j)


def check_split_merge(mod):
    B, T, nh, d = 2, 3, 2, 4
    y = _rand(5, (B * T, nh * d))
    s = mod.split_heads(y, B, T, nh, d)
    assert s.shape == (B, nh, T, d)
    for b in range(B):
        for h in range(nh):
            for t in range(T):
                for c in range(d):
                    assert s[b, h, t, c] == y[b * T + t, h * d + c]
    assert np.array_equal(mod.merge_heads(s), y)


def check_qkv_columns(mod):
    """q / k / v element (b, h, t, c) is the dot product of token (b, t) with weight row
    h*d + c of its block (Q rows first, then K, then V)."""
    B, T, C, H, H_kv, d = 1, 2, 3, 2, 1, 2
    x, w = _rand(6, (B, T, C)), _rand(7, ((H + 2 * H_kv) * d, C))
    q, k, v = mod.qkv_projection(x, w, H, H_kv, d, use_rope=False)
    assert q.shape == (B, H, T, d) and k.shape == (B, H_kv, T, d) and v.shape == (B, H_kv, T, d)
    for name, t_, row0, nh in (("q", q, 0, H), ("k", k, H * d, H_kv), ("v", v, (H + H_kv) * d, H_kv)):
        for h in range(nh):
            for t in range(T):
                for c in range(d):
                    want = math.fsum(x[0, t, j] * w[row0 + h * d + c, j] for j in range(C))
                    assert abs(t_[0, h, t, c] - want) <= 1e-12, (name, h, t, c)
    # the output projection: y[b, t, n] = sum over heads and columns of O[b, h, t, c] W_o[n, h*d + c]
    o, w_o = _rand(8, (B, H, T, d)), _rand(9, (C, H * d))
    y = mod.out_projection(o, w_o)
    for t in range(T):
        for n in range(C):
            want = math.fsum(o[0, h, t, c] * w_o[n, h * d + c] for h in range(H) for c in range(d))
            assert abs(y[0, t, n] - want) <= 1e-12


def check_rope_closed_forms(mod):
    # one-hot at column 0 (pair k = 0, theta_0 = 1): position t is rotated by t radians,
    # into columns 0 and 1 only (interleaved pairs)
    T, d = 3, 4
    x = np.zeros((T, d))
    x[:, 0] = 1.0
    r = mod.rope(x)
    for t in range(T):
        want = [math.cos(t), math.sin(t), 0.0, 0.0]
        assert np.allclose(r[t], want, rtol=0, atol=1e-14), (t, r[t])
    # one-hot at column 3 (the odd member of pair k = 1, theta_1 = 10000^(-2/4) = 0.01):
    # (0, 1) rotated by 0.01 t is (-sin, cos)
    x = np.zeros((T, d))
    x[:, 3] = 1.0
    r = mod.rope(x)
    for t in range(T):
        want = [0.0, 0.0, -math.sin(0.01 * t), math.cos(0.01 * t)]
        assert np.allclose(r[t], want, rtol=0, atol=1e-14), (t, r[t])


def check_rope_invariants(mod):
    T, d = 9, 8
    x = _rand(10, (2, T, d))
    r = mod.rope(x)
    # pair norms kept; the inverse rotation undoes it
    assert np.allclose(r[..., 0::2] ** 2 + r[..., 1::2] ** 2, x[..., 0::2] ** 2 + x[..., 1::2] ** 2, rtol=1e-12)
    assert np.allclose(mod.rope(r, inverse=True), x, rtol=0, atol=1e-12)
    # <rope(q)_m, rope(k)_n> depends only on m - n: the same vectors placed at (m, n)
    # and at (m + s, n + s)
    qv, kv = _rand(11, (d,)), _rand(12, (d,))
    for m, n, s in ((5, 2, 3), (1, 4, 4), (0, 0, 8)):
        q1, k1 = np.zeros((T, d)), np.zeros((T, d))
        q1[m], k1[n] = qv, kv
        q2, k2 = np.zeros((T, d)), np.zeros((T, d))
        q2[m + s], k2[n + s] = qv, kv
        a = mod.rope(q1)[m] @ mod.rope(k1)[n]
        b = mod.rope(q2)[m + s] @ mod.rope(k2)[n + s]
        assert abs(a - b) <= 1e-12 * (1 + abs(a)), (m, n, s)


def _fd_check(loss, params, grads, n_probe=12, seed=0):
    """Central differences of loss() at n_probe entries of each parameter."""
    rng = np.random.default_rng(seed)
    for p, g in zip(params, grads):
        flat = p.reshape(-1)
        for idx in rng.choice(flat.size, size=min(n_probe, flat.size), replace=False):
            h = 1e-6 * max(1.0, abs(flat[idx]))
            old = flat[idx]
            flat[idx] = old + h
            lp = loss()
            flat[idx] = old - h
            lm = loss()
            flat[idx] = old
            fd = (lp - lm) / (2 * h)
            ga = g.reshape(-1)[idx]
            assert abs(fd - ga) <= 1e-6 * max(1.0, abs(fd)), (idx, fd, ga)


def check_projection_finite_differences(mod):
    B, T, C, H, H_kv, d = 2, 5, 8, 2, 1, 4
    for use_rope in (False, True):
        x, w = _rand(13, (B, T, C)), _rand(14, ((H + 2 * H_kv) * d, C))
        gq, gk, gv = _rand(15, (B, H, T, d)), _rand(16, (B, H_kv, T, d)), _rand(17, (B, H_kv, T, d))

        def loss():
            q, k, v = mod.qkv_projection(x, w, H, H_kv, d, use_rope)
            return float((gq * q).sum() + (gk * k).sum() + (gv * v).sum())

        dx, dw = mod.qkv_projection_backward(gq, gk, gv, x, w, use_rope)
        assert dx.shape == x.shape and dw.shape == w.shape
        _fd_check(loss, [x, w], [dx, dw], seed=int(use_rope))
    # output projection with C = H d (a transposed W_o would still have the right shape)
    o, w_o, g = _rand(18, (B, H, T, d)), _rand(19, (C, H * d)), _rand(20, (B, T, C))

    def loss_o():
        return float((g * mod.out_projection(o, w_o)).sum())

    do, dw_o = mod.out_projection_backward(g, o, w_o)
    assert do.shape == o.shape and dw_o.shape == w_o.shape
    _fd_check(loss_o, [o, w_o], [do, dw_o], seed=2)


def check_against_torch_linear(mod):
    import torch
    B, T, C, N = 2, 7, 16, 24
    x, w, g = _rand(21, (B, T, C)), _rand(22, (N, C)), _rand(23, (B, T, N))
    xt = torch.tensor(x, dtype=torch.float64, requires_grad=True)
    wt = torch.tensor(w, dtype=torch.float64, requires_grad=True)
    y = torch.nn.functional.linear(xt, wt)
    (y * torch.tensor(g)).sum().backward()
    x2, g2 = x.reshape(B * T, C), g.reshape(B * T, N)
    assert np.allclose(mod.gemm(x2, w, "nt"), y.detach().numpy().reshape(B * T, N), rtol=1e-12, atol=1e-12)
    assert np.allclose(mod.gemm(g2, w, "nn"), xt.grad.numpy().reshape(B * T, C), rtol=1e-12, atol=1e-12)
    assert np.allclose(mod.gemm(g2, x2, "tn"), wt.grad.numpy(), rtol=1e-12, atol=1e-12)


ALL_CHECKS = (
    check_gemm_brute_force,
    check_split_merge,
    check_qkv_columns,
    check_rope_closed_forms,
    check_rope_invariants,
    check_projection_finite_differences,
    check_against_torch_linear,
)
