"""The projections around the attention on the GPU against the fp64 oracle
(``oracle.projections``) on the same seeded bf16 inputs: the three GEMM orientations at
exact, ragged and split-K sizes, the QKV / output projections forward and backward (with
grouped key/value heads and RoPE), bitwise determinism, and the B4 T2048 C1024 block.

Tolerances (derived from the arithmetic): a bf16 output is the fp32 sum rounded once, so
each element is within one bf16 ulp (2^-8 relative) of the exact value plus the fp32
summation error, and the relative RMS error is about 2^-9 / sqrt(3) = 1.1e-3 (bound 3e-3).
An fp32 output (weight gradients) carries only the fp32 summation error over K terms of
exact bf16 products, ~sqrt(K) 2^-24 relative (bound 1e-4); with RoPE the backward first
rounds the rotated-back dQ, dK to bf16, which adds the 1.1e-3 of a bf16 rounding to the
Q / K rows of dW_qkv and to dX (bound 4e-3)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import seeded_inputs as si
from oracle import projections as orc
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

TOL_BF16_REL_RMS = 3e-3
TOL_F32_REL_RMS = 1e-4
TOL_ROPE_BWD_REL_RMS = 4e-3


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _bits(seed, stream, shape, sigma=1.0):
    return si.normal_bf16_bits(seed, stream, shape, sigma)


def _pair(seed, stream, shape, sigma=1.0):
    b = _bits(seed, stream, shape, sigma)
    return gu.to_device(b), si.bf16_bits_to_f64(b)


def _check_bf16(g, r, label, tol=TOL_BF16_REL_RMS):
    g = gu.to_f64(g)
    assert g.shape == r.shape, label
    assert np.isfinite(g).all(), label
    err = gu.rel_rms(g, r)
    # element-wise: within two bf16 ulps of the exact value, plus a floor for values near 0
    floor = 1e-3 * float(np.abs(r).max())
    bad = np.abs(g - r) > 2.0 ** -7 * np.abs(r) + floor
    print(label, f"rel-RMS {err:.2e}", f"max-abs {gu.max_abs(g, r):.2e}")
    assert err <= tol, f"{label} rel-RMS {err:.3e}"
    assert not bad.any() or tol > TOL_BF16_REL_RMS, f"{label}: {int(bad.sum())} elements beyond 2 ulps"


def _check_f32(g, r, label, tol=TOL_F32_REL_RMS):
    g = gu.to_f64(g)
    assert g.shape == r.shape, label
    err = gu.rel_rms(g, r)
    print(label, f"rel-RMS {err:.2e}")
    assert err <= tol, f"{label} rel-RMS {err:.3e}"


GEMMS = [
    # (layout, M, N, K): one tile, ragged edges in every dimension, several tiles, K
    # shorter than one K-step, and tn products that are split over K
    ("nt", 128, 256, 64), ("nt", 200, 136, 72), ("nt", 384, 520, 1000), ("nt", 8, 8, 8),
    ("nn", 128, 256, 64), ("nn", 200, 136, 72), ("nn", 640, 264, 520),
    ("tn", 128, 256, 64), ("tn", 200, 136, 72), ("tn", 64, 64, 1280), ("tn", 1024, 1024, 4096),
    ("tn", 136, 264, 2056),
]


@pytest.mark.parametrize("layout,M,N,K", GEMMS)
def test_gemm_parity(layout, M, N, K):
    import causal_attention_gb300 as ca
    seed = 300 + M + N + K
    a_shape = (K, M) if layout == "tn" else (M, K)
    b_shape = (N, K) if layout == "nt" else (K, N)
    a, a64 = _pair(seed, 0, a_shape)
    b, b64 = _pair(seed, 1, b_shape, 0.05)
    c = ca.gemm(a, b, layout)
    ca.check_device_error()
    ref = orc.gemm(a64, b64, layout)
    if layout == "tn":
        _check_f32(c, ref, f"gemm {layout} {M}x{N}x{K}")
    else:
        _check_bf16(c, ref, f"gemm {layout} {M}x{N}x{K}")
    again = ca.gemm(a, b, layout)
    assert torch.equal(c, again), "not deterministic"


PROJ = [
    # (B, T, C, H, H_kv, d, rope)
    (2, 300, 256, 4, 4, 64, False), (2, 300, 256, 4, 2, 64, True), (1, 129, 128, 2, 1, 128, True),
    (3, 64, 192, 2, 2, 64, True), (1, 1000, 512, 8, 2, 64, False),
    # one token per sequence (every token tile and K-step is one row); one head, d = 128
    (3, 1, 64, 1, 1, 64, True), (2, 77, 136, 1, 1, 128, True),
]


def _proj_inputs(B, T, C, H, H_kv, d, seed):
    x, x64 = _pair(seed, 0, (B, T, C))
    w, w64 = _pair(seed, 1, ((H + 2 * H_kv) * d, C), 0.02)
    w_o, w_o64 = _pair(seed, 2, (C, H * d), 0.02)
    return x, x64, w, w64, w_o, w_o64


@pytest.mark.parametrize("B,T,C,H,H_kv,d,rope", PROJ)
def test_projection_forward_parity(B, T, C, H, H_kv, d, rope):
    import causal_attention_gb300 as ca
    seed = 700 + T + C + H + H_kv + d
    x, x64, w, w64, w_o, w_o64 = _proj_inputs(B, T, C, H, H_kv, d, seed)
    tab = ca.rope_table(T, d) if rope else None
    q, k, v = ca.qkv_projection(x, w, H, H_kv, d, tab)
    ca.check_device_error()
    rq, rk, rv = orc.qkv_projection(x64, w64, H, H_kv, d, use_rope=rope)
    for name, g, r in (("q", q, rq), ("k", k, rk), ("v", v, rv)):
        _check_bf16(g, r, f"qkv {name}")
    # the output projection, on an O of the attention's shape
    o, o64 = _pair(seed, 3, (B, H, T, d))
    y = ca.out_projection(o, w_o)
    ca.check_device_error()
    _check_bf16(y, orc.out_projection(o64, w_o64), "out y")


@pytest.mark.parametrize("B,T,C,H,H_kv,d,rope", PROJ)
def test_projection_backward_parity(B, T, C, H, H_kv, d, rope):
    import causal_attention_gb300 as ca
    seed = 900 + T + C + H + H_kv + d
    x, x64, w, w64, w_o, w_o64 = _proj_inputs(B, T, C, H, H_kv, d, seed)
    o, o64 = _pair(seed, 3, (B, H, T, d))
    dy, dy64 = _pair(seed, 4, (B, T, C))
    d_o, dw_o = ca.out_projection_backward(dy, o, w_o)
    ca.check_device_error()
    r_do, r_dwo = orc.out_projection_backward(dy64, o64, w_o64)
    _check_bf16(d_o, r_do, "out dO")
    _check_f32(dw_o, r_dwo, "out dW_o")
    dq, dq64 = _pair(seed, 5, (B, H, T, d))
    dk, dk64 = _pair(seed, 6, (B, H_kv, T, d))
    dv, dv64 = _pair(seed, 7, (B, H_kv, T, d))
    tab = ca.rope_table(T, d) if rope else None
    dx, dw = ca.qkv_projection_backward(dq, dk, dv, x, w, tab)
    ca.check_device_error()
    r_dx, r_dw = orc.qkv_projection_backward(dq64, dk64, dv64, x64, w64, use_rope=rope)
    _check_bf16(dx, r_dx, "qkv dX", TOL_ROPE_BWD_REL_RMS if rope else TOL_BF16_REL_RMS)
    _check_f32(dw, r_dw, "qkv dW", TOL_ROPE_BWD_REL_RMS if rope else TOL_F32_REL_RMS)
    # repeated runs give the same bits
    dx2, dw2 = ca.qkv_projection_backward(dq, dk, dv, x, w, tab)
    d_o2, dw_o2 = ca.out_projection_backward(dy, o, w_o)
    assert torch.equal(dx, dx2) and torch.equal(dw, dw2) and torch.equal(d_o, d_o2) and torch.equal(dw_o, dw_o2)


def test_rope_kernel_round_trip():
    """attn_rope forward then inverse on the device, against the oracle's rotation."""
    import causal_attention_gb300 as ca
    B, H, T, d = 2, 3, 77, 128
    x, x64 = _pair(41, 0, (B, H, T, d))
    tab = ca.rope_table(T, d)
    y = torch.empty_like(x)
    ca.attn_rope(x, y, tab)
    _check_bf16(y, orc.rope(x64), "rope")
    z = torch.empty_like(x)
    ca.attn_rope(y, z, tab, inverse=True)
    _check_bf16(z, orc.rope(gu.to_f64(y), inverse=True), "rope inverse")
    # the table itself: cos / sin of t * 10000^(-2k/d) to fp32 rounding
    ang = orc.rope_angles(T, d)
    t64 = tab.double().cpu().numpy()
    assert np.abs(t64[..., 0] - np.cos(ang)).max() <= 1e-7
    assert np.abs(t64[..., 1] - np.sin(ang)).max() <= 1e-7


def test_block_shapes_of_the_b4_t2048_workload():
    """The attention block of B4 H16 T2048 d64 (C = H d = 1024) with RoPE: QKV projection,
    output projection and both backward passes, whole tensors against the oracle."""
    import causal_attention_gb300 as ca
    B, T, C, H, H_kv, d = 4, 2048, 1024, 16, 16, 64
    x, x64, w, w64, w_o, w_o64 = _proj_inputs(B, T, C, H, H_kv, d, 4242)
    tab = ca.rope_table(T, d)
    q, k, v = ca.qkv_projection(x, w, H, H_kv, d, tab)
    rq, rk, rv = orc.qkv_projection(x64, w64, H, H_kv, d, use_rope=True)
    for name, g, r in (("q", q, rq), ("k", k, rk), ("v", v, rv)):
        _check_bf16(g, r, f"block {name}")
    del rq, rk, rv
    o, o64 = _pair(4243, 3, (B, H, T, d))
    _check_bf16(ca.out_projection(o, w_o), orc.out_projection(o64, w_o64), "block y")
    dy, dy64 = _pair(4243, 4, (B, T, C))
    d_o, dw_o = ca.out_projection_backward(dy, o, w_o)
    r_do, r_dwo = orc.out_projection_backward(dy64, o64, w_o64)
    _check_bf16(d_o, r_do, "block dO")
    _check_f32(dw_o, r_dwo, "block dW_o")
    dq, dq64 = _pair(4243, 5, (B, H, T, d))
    dk, dk64 = _pair(4243, 6, (B, H_kv, T, d))
    dv, dv64 = _pair(4243, 7, (B, H_kv, T, d))
    dx, dw = ca.qkv_projection_backward(dq, dk, dv, x, w, tab)
    ca.check_device_error()
    r_dx, r_dw = orc.qkv_projection_backward(dq64, dk64, dv64, x64, w64, use_rope=True)
    _check_bf16(dx, r_dx, "block dX", TOL_ROPE_BWD_REL_RMS)
    _check_f32(dw, r_dw, "block dW_qkv", TOL_ROPE_BWD_REL_RMS)


def test_block_cuda_graph_matches_eager():
    """The projection entry points are capturable into a CUDA graph too: QKV projection
    with RoPE, attention, output projection and the backward of all three, replayed into
    NaN-poisoned buffers, give the eager bits."""
    import causal_attention_gb300 as ca
    B, T, C, H, H_kv, d = 2, 300, 256, 4, 2, 64
    x, _, w, _, w_o, _ = _proj_inputs(B, T, C, H, H_kv, d, 555)
    dy, _ = _pair(556, 4, (B, T, C))
    tab = ca.rope_table(T, d)
    out = {"q": torch.empty((B, H, T, d), dtype=torch.bfloat16, device="cuda")}
    for n in ("k", "v", "dk", "dv"):
        out[n] = torch.empty((B, H_kv, T, d), dtype=torch.bfloat16, device="cuda")
    for n in ("o", "do", "dq"):
        out[n] = torch.empty_like(out["q"])
    out["lse"] = torch.empty((B, H, T), dtype=torch.float32, device="cuda")
    out["y"], out["dx"] = torch.empty_like(x), torch.empty_like(x)
    out["dw_o"] = torch.empty((C, H * d), dtype=torch.float32, device="cuda")
    out["dw"] = torch.empty(tuple(w.shape), dtype=torch.float32, device="cuda")
    ws = ca.new_workspace(B, H, T, d, kv_heads=H_kv)
    wsp = ca.new_proj_workspace(B, T, C, H, H_kv, d)
    scale = 1.0 / np.sqrt(d)
    st = torch.cuda.Stream()

    def step():
        ca.attn_qkv_proj(x, w, out["q"], out["k"], out["v"], tab, st)
        ca.attn_fwd(out["q"], out["k"], out["v"], out["o"], out["lse"], scale, True, st)
        ca.attn_out_proj(out["o"], w_o, out["y"], st)
        ca.attn_out_proj_bwd(dy, out["o"], w_o, out["do"], out["dw_o"], wsp, st)
        ca.attn_bwd(out["q"], out["k"], out["v"], out["o"], out["do"], out["lse"], out["dq"], out["dk"], out["dv"], ws,
                    scale, True, st)
        ca.attn_qkv_proj_bwd(out["dq"], out["dk"], out["dv"], x, w, out["dx"], out["dw"], wsp, tab, st)
    with torch.cuda.stream(st):
        step()
    torch.cuda.synchronize()
    ca.check_device_error()
    eager = {n: t.clone() for n, t in out.items()}
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=st):
        step()
    for t in out.values():
        t.fill_(float("nan"))
    with torch.cuda.stream(st):
        g.replay()
    torch.cuda.synchronize()
    ca.check_device_error()
    for n in out:
        assert torch.equal(out[n], eager[n]), n
