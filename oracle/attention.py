"""CPU oracle for causal multi-head attention, forward and backward.

TEST INFRASTRUCTURE ONLY. Nothing in the library imports this module; only the test
suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` use it.
It shares no code with the CUDA path.

Plain, slow and obviously correct: for each (batch, head) it builds the full T x T
score matrix in fp64 (or fp32 for the "fp32 instantiation"), with a library matmul as
the only borrowed step. There is no tiling, no online softmax and no fusion: the
formulas are written out exactly as the pages state them.

Definitions followed (page, section):

* Forward: S = Q K^T * scale; causal mask; softmax; O = P V; the per-row
  logsumexp L = m + log(l) is saved for the backward. Forge RESEARCH.md, section 6
  "Fused attention design (flash-style)" (the algorithm block and its last line
  L = m + log(l)). The online rescaling loop there is an implementation of the same
  softmax; here the softmax is computed directly from full rows.
* Causal convention: a key column later than the query row is masked (the mask
  test "column > row" of the cooperative-tensors guide, section 5.3 / the assembled
  kernel's causal mask), i.e. key j is visible to query i iff j <= i.
* Backward: D = rowsum(dO * O) (Forge RESEARCH.md section 6, the bullet on the D term;
  Forge paper, section "Ecosystem survey"); P recomputed from L as P = exp(S - L)
  (RESEARCH.md section 6, "Backward (training)"); dV = P^T dO, dP = dO V^T,
  dS = P * (dP - D), dQ = dS K * scale, dK = dS^T Q * scale.

Readings where the pages leave a step open:
* The logsumexp is in natural-log units and includes the scale: L_i = log sum_j
  exp(scale * q_i . k_j) over visible j.
* The O that feeds D is the oracle's own fp64 O.
* Masked entries are excluded (exp of -inf = 0); with causal masking every row sees
  at least its own key, so no row is fully masked.
* Grouped key/value heads (GQA / MQA): K and V may have H_kv heads with H_kv dividing
  H; query head h attends with key/value head h // (H / H_kv), the index mapping of
  Forge RESEARCH.md section 6 (integer division of the query head by the group size, no
  repeated copies). A key/value head's dK and dV are the sums of the contributions of the
  query heads that use it (each contribution is the single-head backward above).
"""
from __future__ import annotations

import numpy as np


def causal_mask(T: int) -> np.ndarray:
    """Boolean [T, T]: True where key j is visible to query i (j <= i)."""
    i = np.arange(T)[:, None]
    j = np.arange(T)[None, :]
    return j <= i


def head_forward(q, k, v, scale, causal=True, dtype=np.float64):
    """One (b, h) head. q, k, v: [T, d]. Returns (O [T, d], L [T], P [T, T])."""
    q = np.asarray(q, dtype=dtype)
    k = np.asarray(k, dtype=dtype)
    v = np.asarray(v, dtype=dtype)
    T = q.shape[0]
    s = (q @ k.T) * dtype(scale)                       # S = Q K^T * scale
    if causal:
        s = np.where(causal_mask(T), s, dtype(-np.inf))  # key j > query i is masked
    m = s.max(axis=1)                                   # row max
    l = np.exp(s - m[:, None]).sum(axis=1)              # row sum of exp
    lse = m + np.log(l)                                 # L = m + log(l)
    p = np.exp(s - lse[:, None])                        # softmax, masked -> 0
    o = p @ v                                           # O = P V
    return o, lse, p


def head_backward(q, k, v, do, scale, causal=True, dtype=np.float64, o=None, lse=None):
    """One (b, h) head. Returns (dQ, dK, dV, D), each for that head.

    If ``o``/``lse`` are not given they are the oracle's own forward outputs.
    """
    q = np.asarray(q, dtype=dtype)
    k = np.asarray(k, dtype=dtype)
    v = np.asarray(v, dtype=dtype)
    do = np.asarray(do, dtype=dtype)
    T = q.shape[0]
    if o is None or lse is None:
        o, lse, _ = head_forward(q, k, v, scale, causal, dtype)
    s = (q @ k.T) * dtype(scale)                        # recompute S
    if causal:
        s = np.where(causal_mask(T), s, dtype(-np.inf))
    p = np.exp(s - np.asarray(lse, dtype=dtype)[:, None])  # P = exp(S - L)
    D = (do * np.asarray(o, dtype=dtype)).sum(axis=1)   # D = rowsum(dO * O)
    dv = p.T @ do                                       # dV = P^T dO
    dp = do @ v.T                                       # dP = dO V^T
    ds = p * (dp - D[:, None])                          # dS = P * (dP - D)
    dq = (ds @ k) * dtype(scale)                        # dQ = dS K * scale
    dk = (ds.T @ q) * dtype(scale)                      # dK = dS^T Q * scale
    return dq, dk, dv, D


def _heads(B, H, heads):
    if heads is None:
        return [(b, h) for b in range(B) for h in range(H)]
    return list(heads)


def kv_head(h, H, H_kv):
    """The key/value head that query head h uses (RESEARCH.md's GQA mapping)."""
    if H % H_kv:
        raise ValueError("the number of key/value heads must divide the number of query heads")
    return h // (H // H_kv)


def forward(q, k, v, scale, causal=True, dtype=np.float64, heads=None):
    """q: [B, H, T, d]; k, v: [B, H_kv, T, d] (H_kv = H, or a divisor of H for grouped
    key/value heads). Returns O [B, H, T, d] and L [B, H, T].

    With ``heads`` (a list of (b, h)) only those query heads are computed; the other
    entries of the outputs are NaN.
    """
    B, H, T, d = q.shape
    H_kv = k.shape[1]
    o = np.full((B, H, T, d), np.nan, dtype=dtype)
    lse = np.full((B, H, T), np.nan, dtype=dtype)
    for b, h in _heads(B, H, heads):
        g = kv_head(h, H, H_kv)
        o[b, h], lse[b, h], _ = head_forward(q[b, h], k[b, g], v[b, g], scale, causal, dtype)
    return o, lse


def backward(q, k, v, do, scale, causal=True, dtype=np.float64, heads=None):
    """Returns dQ [B, H, T, d], dK, dV [B, H_kv, T, d] and D [B, H, T].

    dK and dV of a key/value head sum the contributions of its query heads. With
    ``heads`` (query heads), dQ and D are NaN outside them, and dK / dV are NaN for every
    key/value head whose query heads are not all included.
    """
    B, H, T, d = q.shape
    H_kv = k.shape[1]
    dq = np.full((B, H, T, d), np.nan, dtype=dtype)
    D = np.full((B, H, T), np.nan, dtype=dtype)
    dk = np.zeros((B, H_kv, T, d), dtype=dtype)
    dv = np.zeros_like(dk)
    seen = np.zeros((B, H_kv), dtype=np.int64)
    for b, h in _heads(B, H, heads):
        g = kv_head(h, H, H_kv)
        dq[b, h], dk_h, dv_h, D[b, h] = head_backward(q[b, h], k[b, g], v[b, g], do[b, h], scale, causal, dtype)
        dk[b, g] += dk_h
        dv[b, g] += dv_h
        seen[b, g] += 1
    incomplete = seen != H // H_kv
    dk[incomplete] = np.nan
    dv[incomplete] = np.nan
    return dq, dk, dv, D


def preprocess_D(o, do, dtype=np.float64):
    """D = rowsum(dO * O) for given O and dO, [B, H, T, d] -> [B, H, T]."""
    return (np.asarray(do, dtype=dtype) * np.asarray(o, dtype=dtype)).sum(axis=-1)


def credited_flops(B, H, T, d):
    """Credited causal FLOPs: forward 2*B*H*T^2*d, backward 2.5 times that.

    The convention that reproduces the Forge RESEARCH.md section 6 table (gpt-10m
    forward, 2.3 ms at 5.7 TF).
    """
    fwd = 2.0 * B * H * T * T * d
    return fwd, 2.5 * fwd
