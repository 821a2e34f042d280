"""CPU oracle for the projections around the fused attention: the training GEMMs, the
head split / merge, rotary position embedding, and the QKV / output projections with
their backward.

TEST INFRASTRUCTURE ONLY. Nothing in the library imports this module; only the test
suite and ``bench.py``'s reference leg use it. It shares no code with the CUDA path.

Plain fp64 numpy: every product is one library matmul of whole matrices; there is no
tiling, no split-K and no fusion. Heads are split and merged with reshapes.

Definitions followed (page, section):

* GEMM orientations of a training step: forward ``Y = X W^T`` ("nt"), backward
  ``dX = dY W`` ("nn") and ``dW = dY^T X`` ("tn"). Forge RESEARCH.md, section 5 "GEMM
  design" (the transpose-variants item: training needs nt, nn and tn), and the Forge
  paper, section "Results" (the GEMM table: forward MLP X W1^T, backward dX = dY W,
  dW = dY^T X).
* Rotary position embedding: Forge RESEARCH.md, section 7 "Training loop", model
  formulas: interleaved pairs (2k, 2k+1) of each head row at sequence position m are
  rotated by the angle m * theta_k, theta_k = 10000^(-2k / d_head), applied to q and k
  only; the backward is the rotation by -m * theta_k.

Readings where the pages leave a step open:

* The attention block around the fused kernel is the nanoGPT / llm.c one that section
  7 distils: one QKV weight ``W_qkv`` of shape [(H + 2 H_kv) d, C] whose output
  features are Q (H heads), then K, then V (H_kv heads each), each head's d features
  contiguous; one output weight ``W_o`` of shape [C, H d] applied to the heads
  concatenated in head order. No biases.
* The rotation's position m is the token's index t within its sequence (0-based).
* RoPE is applied after the projection and before attention, so the backward applies
  the inverse rotation to dQ and dK before the projection's own backward (the
  rotation is orthogonal: its adjoint is its inverse).
* Weight gradients are returned in fp64 here; the GPU writes them in fp32 (the pages
  keep gradients in f32, RESEARCH.md section 7 "Mixed precision").
"""
from __future__ import annotations

import numpy as np

ROPE_BASE = 10000.0


def gemm(a: np.ndarray, b: np.ndarray, layout: str) -> np.ndarray:
    """C = op(A) op(B) for the three training orientations: "nt" C = A B^T (A [M, K],
    B [N, K]); "nn" C = A B (A [M, K], B [K, N]); "tn" C = A^T B (A [K, M], B [K, N])."""
    if layout == "nt":
        return a @ b.T
    if layout == "nn":
        return a @ b
    if layout == "tn":
        return a.T @ b
    raise ValueError(layout)


def split_heads(y: np.ndarray, B: int, T: int, n_heads: int, d: int) -> np.ndarray:
    """[B*T, n_heads*d] (token rows, head-major features) -> [B, n_heads, T, d]."""
    return y.reshape(B, T, n_heads, d).transpose(0, 2, 1, 3).copy()


def merge_heads(x: np.ndarray) -> np.ndarray:
    """[B, n_heads, T, d] -> [B*T, n_heads*d]: the inverse of split_heads."""
    B, nh, T, d = x.shape
    return x.transpose(0, 2, 1, 3).reshape(B * T, nh * d).copy()


def rope_angles(T: int, d: int, base: float = ROPE_BASE) -> np.ndarray:
    """[T, d/2] angles m * theta_k with theta_k = base^(-2k/d)."""
    k = np.arange(d // 2, dtype=np.float64)
    theta = base ** (-2.0 * k / d)
    return np.arange(T, dtype=np.float64)[:, None] * theta[None, :]


def rope(x: np.ndarray, inverse: bool = False, base: float = ROPE_BASE) -> np.ndarray:
    """Rotates the interleaved pairs (x[..., t, 2k], x[..., t, 2k+1]) by the angle
    t * theta_k (by -t * theta_k when inverse). x: [..., T, d]."""
    T, d = x.shape[-2], x.shape[-1]
    ang = rope_angles(T, d, base)
    if inverse:
        ang = -ang
    c, s = np.cos(ang), np.sin(ang)
    x0, x1 = x[..., 0::2], x[..., 1::2]
    out = np.empty_like(x)
    out[..., 0::2] = x0 * c - x1 * s
    out[..., 1::2] = x0 * s + x1 * c
    return out


def qkv_projection(x: np.ndarray, w_qkv: np.ndarray, H: int, H_kv: int, d: int, use_rope: bool = False):
    """x [B, T, C], w_qkv [(H + 2 H_kv) d, C] -> q [B, H, T, d], k, v [B, H_kv, T, d]:
    Y = X W_qkv^T (nt), split into Q, K, V and into heads; RoPE on q and k if asked."""
    B, T, C = x.shape
    y = gemm(x.reshape(B * T, C), w_qkv, "nt")
    q = split_heads(y[:, : H * d], B, T, H, d)
    k = split_heads(y[:, H * d: (H + H_kv) * d], B, T, H_kv, d)
    v = split_heads(y[:, (H + H_kv) * d:], B, T, H_kv, d)
    if use_rope:
        q, k = rope(q), rope(k)
    return q, k, v


def out_projection(o: np.ndarray, w_o: np.ndarray) -> np.ndarray:
    """o [B, H, T, d], w_o [C, H d] -> y [B, T, C] = merge(O) W_o^T (nt)."""
    B, H, T, d = o.shape
    return gemm(merge_heads(o), w_o, "nt").reshape(B, T, -1)


def out_projection_backward(dy: np.ndarray, o: np.ndarray, w_o: np.ndarray):
    """Gradients of y = out_projection(o, w_o) given dy [B, T, C]:
    dO = split(dY W_o) (nn) and dW_o = dY^T merge(O) (tn)."""
    B, H, T, d = o.shape
    dy2 = dy.reshape(B * T, -1)
    do = split_heads(gemm(dy2, w_o, "nn"), B, T, H, d)
    dw_o = gemm(dy2, merge_heads(o), "tn")
    return do, dw_o


def qkv_projection_backward(dq: np.ndarray, dk: np.ndarray, dv: np.ndarray, x: np.ndarray, w_qkv: np.ndarray,
                            use_rope: bool = False):
    """Gradients of qkv_projection given dq [B, H, T, d], dk, dv [B, H_kv, T, d]:
    with RoPE, dQ and dK are first rotated back; then dY = [merge(dQ) | merge(dK) |
    merge(dV)], dX = dY W_qkv (nn) and dW_qkv = dY^T X (tn)."""
    B, T, C = x.shape
    if use_rope:
        dq, dk = rope(dq, inverse=True), rope(dk, inverse=True)
    dy = np.concatenate([merge_heads(dq), merge_heads(dk), merge_heads(dv)], axis=1)
    dx = gemm(dy, w_qkv, "nn").reshape(B, T, C)
    dw = gemm(dy, x.reshape(B * T, C), "tn")
    return dx, dw


def gemm_flops(M: int, N: int, K: int) -> float:
    """2 M N K: one multiply and one add per term."""
    return 2.0 * M * N * K
