"""Python binding of libattn.so: fused causal attention forward/backward on GB300.

Argument marshalling only. Every step of the computation runs in the library's CUDA
kernels; PyTorch supplies device memory and streams. If the library has not been
built (``python causal_attention_gb300/build.py``) importing this package raises.

The functions named like the C ABI (``attn_fwd``, ``attn_bwd``, ...) take torch
tensors and pass their device pointers; ``forward``/``backward`` allocate outputs;
``CausalAttention`` wraps both as a ``torch.autograd.Function``.
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

from ._lib import load_library, ATTN_OK, AttnError, STATUS_NAMES, LIB_PATH, DEBUG_LIB_PATH  # noqa: F401

# ATTN_BOUNDS_CHECK=1 in the environment loads the bounds-checked build of the library
# (libattn_debug.so: every TMA coordinate, bulk-copy range and global store index checked
# on the device; a failed check skips the access and is reported by check_device_error).
_dll = load_library(DEBUG_LIB_PATH if os.environ.get("ATTN_BOUNDS_CHECK") == "1" else LIB_PATH)


def _stream_handle(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _check(status, what):
    if status != ATTN_OK:
        raise AttnError(status, what, _dll.attn_last_cuda_error().decode())


def _shape(q):
    if q.dim() != 4:
        raise ValueError("expected a [B, H, T, d] tensor")
    return tuple(int(x) for x in q.shape)


def _need(t, name, dtype):
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    if not t.is_cuda:
        raise ValueError(f"{name}: must be a CUDA tensor")


def abi_version() -> int:
    return _dll.attn_abi_version()


def attn_bwd_workspace_size(B, H, T, d) -> int:
    return int(_dll.attn_bwd_workspace_size(B, H, T, d))


def _kv_heads(q, *kv):
    """H_kv of k / v tensors [B, H_kv, T, d] that go with q [B, H, T, d]."""
    B, H, T, d = _shape(q)
    H_kv = _shape(kv[0])[1]
    for t in kv:
        if _shape(t) != (B, H_kv, T, d):
            raise ValueError(f"key/value tensors must be [B, H_kv, T, d] = {(B, H_kv, T, d)}, got {tuple(t.shape)}")
    return H_kv


def attn_fwd(q, k, v, o, lse, scale, causal=True, stream=None):
    """O = softmax(Q K^T * scale [causal]) V and the natural-log LSE, in place. k and v
    may have fewer heads than q (grouped key/value heads: query head h reads key/value
    head h // (H / H_kv))."""
    B, H, T, d = _shape(q)
    H_kv = _kv_heads(q, k, v)
    for n, t in (("q", q), ("k", k), ("v", v), ("o", o)):
        _need(t, n, torch.bfloat16)
    _need(lse, "lse", torch.float32)
    _check(_dll.attn_fwd_gqa(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, H_kv, T, d,
                             ctypes.c_float(scale), int(causal), _stream_handle(stream)), "attn_fwd_gqa")


def attn_bwd(q, k, v, o, do, lse, dq, dk, dv, workspace, scale, causal=True, stream=None):
    """dQ, dK, dV in place. k, v, dk, dv may have fewer heads than q (grouped key/value
    heads; dK / dV then sum over each key/value head's query heads)."""
    B, H, T, d = _shape(q)
    H_kv = _kv_heads(q, k, v, dk, dv)
    for n, t in (("q", q), ("k", k), ("v", v), ("o", o), ("do", do), ("dq", dq), ("dk", dk), ("dv", dv)):
        _need(t, n, torch.bfloat16)
    _need(lse, "lse", torch.float32)
    _check(_dll.attn_bwd_gqa(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse), _ptr(dq), _ptr(dk),
                             _ptr(dv), _ptr(workspace), workspace.numel() * workspace.element_size(),
                             B, H, H_kv, T, d, ctypes.c_float(scale), int(causal), _stream_handle(stream)),
           "attn_bwd_gqa")


def attn_bwd_preprocess(o, do, lse, workspace, stream=None):
    B, H, T, d = _shape(o)
    _check(_dll.attn_bwd_preprocess(_ptr(o), _ptr(do), _ptr(lse), _ptr(workspace),
                                    workspace.numel() * workspace.element_size(), B, H, T, d,
                                    _stream_handle(stream)), "attn_bwd_preprocess")


def attn_bwd_dkdv(q, k, v, do, dk, dv, workspace, scale, causal=True, stream=None):
    B, H, T, d = _shape(q)
    _check(_dll.attn_bwd_dkdv(_ptr(q), _ptr(k), _ptr(v), _ptr(do), _ptr(dk), _ptr(dv), _ptr(workspace),
                              workspace.numel() * workspace.element_size(), B, H, T, d,
                              ctypes.c_float(scale), int(causal), _stream_handle(stream)), "attn_bwd_dkdv")


def attn_bwd_dq(q, k, v, o, do, lse, dq, workspace, scale, causal=True, stream=None):
    """dQ; at d <= 64 it also writes D and -LSE*log2(e) into the workspace (no
    attn_bwd_preprocess needed before it, and attn_bwd_dkdv may follow it)."""
    B, H, T, d = _shape(q)
    _check(_dll.attn_bwd_dq(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse), _ptr(dq), _ptr(workspace),
                            workspace.numel() * workspace.element_size(), B, H, T, d,
                            ctypes.c_float(scale), int(causal), _stream_handle(stream)), "attn_bwd_dq")


def attn_bwd_dkdv_dq(q, k, v, do, dk, dv, workspace, scale, causal=True, stream=None):
    """dK, dV and (into the workspace) the fp32 dQ sums in one kernel; d <= 64 and a
    workspace of attn_bwd_fused_workspace_size bytes, prepared by attn_bwd_preprocess."""
    B, H, T, d = _shape(q)
    _check(_dll.attn_bwd_dkdv_dq(_ptr(q), _ptr(k), _ptr(v), _ptr(do), _ptr(dk), _ptr(dv), _ptr(workspace),
                                 workspace.numel() * workspace.element_size(), B, H, T, d,
                                 ctypes.c_float(scale), int(causal), _stream_handle(stream)), "attn_bwd_dkdv_dq")


def attn_bwd_dq_finish(dq, workspace, scale, stream=None):
    """dQ (bf16) = scale times the fp32 sums attn_bwd_dkdv_dq left in the workspace."""
    B, H, T, d = _shape(dq)
    _check(_dll.attn_bwd_dq_finish(_ptr(dq), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                   B, H, T, d, ctypes.c_float(scale), _stream_handle(stream)),
           "attn_bwd_dq_finish")


def attn_bwd_noalloc(q, k, v, o, do, lse, dq, dk, dv, scale, causal=True, stream=None):
    """attn_bwd without a workspace: the library's fixed 8 MiB device scratch is used
    instead (B*H*T_pad <= 1,048,576). For callers that cannot allocate device memory;
    calls that overlap on the GPU share that scratch and must be serialised."""
    B, H, T, d = _shape(q)
    for n, t in (("q", q), ("k", k), ("v", v), ("o", o), ("do", do), ("dq", dq), ("dk", dk), ("dv", dv)):
        _need(t, n, torch.bfloat16)
    _need(lse, "lse", torch.float32)
    _check(_dll.attn_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse), _ptr(dq),
                                 _ptr(dk), _ptr(dv), B, H, T, d, ctypes.c_float(scale), int(causal),
                                 _stream_handle(stream)), "attn_bwd_noalloc")


def selftest_wait_timeout(stream=None):
    """Launches the bounded-wait self-test (see attn.h); the next check_device_error on the
    stream raises AttnError with ATTN_ERR_DEVICE_TIMEOUT."""
    _check(_dll.attn_selftest_wait_timeout(_stream_handle(stream)), "attn_selftest_wait_timeout")


def check_device_error(stream=None):
    """Synchronises the stream and raises AttnError if a kernel's bounded wait expired."""
    _check(_dll.attn_check_device_error(_stream_handle(stream)), "attn_check_device_error")


def attn_bwd_fused_workspace_size(B, H, T, d) -> int:
    return int(_dll.attn_bwd_fused_workspace_size(B, H, T, d))


def attn_bwd_gqa_workspace_size(B, H, H_kv, T, d) -> int:
    return int(_dll.attn_bwd_gqa_workspace_size(B, H, H_kv, T, d))


def new_workspace(B, H, T, d, device=None, fused_dq=False, kv_heads=None):
    """Device workspace for attn_bwd (with fused_dq, for the fused-dQ stages; with kv_heads
    fewer than H, for attn_bwd_gqa's split dK/dV)."""
    if kv_heads is not None and kv_heads != H:
        n = attn_bwd_gqa_workspace_size(B, H, kv_heads, T, d)
    else:
        n = (attn_bwd_fused_workspace_size if fused_dq else attn_bwd_workspace_size)(B, H, T, d)
    if n == 0:
        raise ValueError("invalid sizes" + (" (the fused dQ needs d <= 64)" if fused_dq else ""))
    return torch.empty(n // 4, dtype=torch.float32, device=device or "cuda")


def forward(q, k, v, scale=None, causal=True, stream=None):
    """Allocates and returns (O, LSE)."""
    B, H, T, d = _shape(q)
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    o = torch.empty_like(q)
    lse = torch.empty((B, H, T), dtype=torch.float32, device=q.device)
    attn_fwd(q, k, v, o, lse, scale, causal, stream)
    return o, lse


def backward(q, k, v, o, do, lse, scale=None, causal=True, stream=None, workspace=None):
    """Allocates and returns (dQ, dK, dV)."""
    B, H, T, d = _shape(q)
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    if workspace is None:
        workspace = new_workspace(B, H, T, d, q.device, kv_heads=int(k.shape[1]))
    attn_bwd(q, k, v, o, do, lse, dq, dk, dv, workspace, scale, causal, stream)
    return dq, dk, dv


class CausalAttention(torch.autograd.Function):
    """softmax(Q K^T * scale [causal]) V with the library's fused backward."""

    @staticmethod
    def forward(ctx, q, k, v, scale=None, causal=True):
        q, k, v = (t.contiguous() for t in (q, k, v))
        o, lse = forward(q, k, v, scale, causal)
        ctx.save_for_backward(q, k, v, o, lse)
        ctx.scale, ctx.causal = scale, causal
        return o

    @staticmethod
    def backward(ctx, do):
        q, k, v, o, lse = ctx.saved_tensors
        dq, dk, dv = backward(q, k, v, o, do.contiguous().to(torch.bfloat16), lse, ctx.scale, ctx.causal)
        return dq, dk, dv, None, None


def attention(q, k, v, scale=None, causal=True):
    return CausalAttention.apply(q, k, v, scale, causal)


# ---------------------------------------------------------------------------
# Projections around the attention (the attention block's training GEMMs)
# ---------------------------------------------------------------------------
GEMM_LAYOUTS = {"nt": 0, "nn": 1, "tn": 2}


def _nbytes(t):
    return t.numel() * t.element_size() if t is not None else 0


def attn_gemm_workspace_size(M, N, K, layout) -> int:
    return int(_dll.attn_gemm_workspace_size(M, N, K, GEMM_LAYOUTS[layout]))


def attn_gemm(a, b, c, layout, workspace=None, stream=None):
    """c = op(a) op(b) in place: "nt" a [M, K], b [N, K]; "nn" a [M, K], b [K, N]; "tn"
    a [K, M], b [K, N] (c fp32 [M, N]; bf16 [M, N] otherwise)."""
    lay = GEMM_LAYOUTS[layout]
    if lay == 2:
        (K, M), N = a.shape, b.shape[1]
    else:
        (M, K), N = a.shape, (b.shape[0] if lay == 0 else b.shape[1])
    for n, t in (("a", a), ("b", b)):
        _need(t, n, torch.bfloat16)
    _need(c, "c", torch.float32 if lay == 2 else torch.bfloat16)
    if tuple(c.shape) != (M, N):
        raise ValueError(f"c must be [{M}, {N}]")
    _check(_dll.attn_gemm(_ptr(a), _ptr(b), _ptr(c), M, N, K, lay, _ptr(workspace), _nbytes(workspace),
                          _stream_handle(stream)), "attn_gemm")


def gemm(a, b, layout, stream=None):
    """Allocates and returns op(a) op(b) (bf16, or fp32 for "tn")."""
    lay = GEMM_LAYOUTS[layout]
    M = a.shape[1] if lay == 2 else a.shape[0]
    N = b.shape[0] if lay == 0 else b.shape[1]
    K = a.shape[0] if lay == 2 else a.shape[1]
    c = torch.empty((M, N), dtype=torch.float32 if lay == 2 else torch.bfloat16, device=a.device)
    n = attn_gemm_workspace_size(M, N, K, layout)
    ws = torch.empty(n // 4, dtype=torch.float32, device=a.device) if n else None
    attn_gemm(a, b, c, layout, ws, stream)
    return c


def rope_table(T, d, device=None, stream=None):
    """fp32 [T, d/2, 2]: (cos, sin) of t * 10000^(-2k/d)."""
    tab = torch.empty((T, d // 2, 2), dtype=torch.float32, device=device or "cuda")
    _check(_dll.attn_rope_table(_ptr(tab), T, d, _stream_handle(stream)), "attn_rope_table")
    return tab


def attn_rope(x, y, tab, inverse=False, stream=None):
    """y = RoPE(x) (inverse: the backward rotation) for [B, H, T, d] bf16 tensors."""
    B, H, T, d = _shape(x)
    _need(x, "x", torch.bfloat16)
    _need(y, "y", torch.bfloat16)
    _check(_dll.attn_rope(_ptr(x), _ptr(y), _ptr(tab), B, H, T, d, int(inverse), _stream_handle(stream)),
           "attn_rope")


def _proj_dims(x, w_qkv, H, H_kv, d):
    B, T, C = (int(s) for s in x.shape)
    if tuple(w_qkv.shape) != ((H + 2 * H_kv) * d, C):
        raise ValueError(f"w_qkv must be [{(H + 2 * H_kv) * d}, {C}]")
    return B, T, C


def attn_qkv_proj(x, w_qkv, q, k, v, rope_tab=None, stream=None):
    """q, k, v = split(x W_qkv^T) in place (q, k rotated when rope_tab is given)."""
    B, H, T, d = _shape(q)
    H_kv = _shape(k)[1]
    _proj_dims(x, w_qkv, H, H_kv, d)
    for n, t in (("x", x), ("w_qkv", w_qkv), ("q", q), ("k", k), ("v", v)):
        _need(t, n, torch.bfloat16)
    C = int(x.shape[2])
    _check(_dll.attn_qkv_proj(_ptr(x), _ptr(w_qkv), _ptr(q), _ptr(k), _ptr(v), _ptr(rope_tab), B, T, C, H, H_kv, d,
                              _stream_handle(stream)), "attn_qkv_proj")


def attn_out_proj(o, w_o, y, stream=None):
    """y [B, T, C] = merge(o) W_o^T in place."""
    B, H, T, d = _shape(o)
    C = int(w_o.shape[0])
    for n, t in (("o", o), ("w_o", w_o), ("y", y)):
        _need(t, n, torch.bfloat16)
    _check(_dll.attn_out_proj(_ptr(o), _ptr(w_o), _ptr(y), B, T, H, d, C, _stream_handle(stream)), "attn_out_proj")


def attn_proj_bwd_workspace_size(B, T, C, H, H_kv, d) -> int:
    return int(_dll.attn_proj_bwd_workspace_size(B, T, C, H, H_kv, d))


def new_proj_workspace(B, T, C, H, H_kv, d, device=None):
    n = attn_proj_bwd_workspace_size(B, T, C, H, H_kv, d)
    return torch.empty(max(n, 16) // 4, dtype=torch.float32, device=device or "cuda")


def attn_out_proj_bwd(dy, o, w_o, d_o, dw_o, workspace, stream=None):
    B, H, T, d = _shape(o)
    C = int(w_o.shape[0])
    for n, t in (("dy", dy), ("o", o), ("w_o", w_o), ("d_o", d_o)):
        _need(t, n, torch.bfloat16)
    _need(dw_o, "dw_o", torch.float32)
    _check(_dll.attn_out_proj_bwd(_ptr(dy), _ptr(o), _ptr(w_o), _ptr(d_o), _ptr(dw_o), _ptr(workspace),
                                  _nbytes(workspace), B, T, H, d, C, _stream_handle(stream)), "attn_out_proj_bwd")


def attn_qkv_proj_bwd(dq, dk, dv, x, w_qkv, dx, dw_qkv, workspace, rope_tab=None, stream=None):
    B, H, T, d = _shape(dq)
    H_kv = _shape(dk)[1]
    _, _, C = _proj_dims(x, w_qkv, H, H_kv, d)
    for n, t in (("dq", dq), ("dk", dk), ("dv", dv), ("x", x), ("w_qkv", w_qkv), ("dx", dx)):
        _need(t, n, torch.bfloat16)
    _need(dw_qkv, "dw_qkv", torch.float32)
    _check(_dll.attn_qkv_proj_bwd(_ptr(dq), _ptr(dk), _ptr(dv), _ptr(x), _ptr(w_qkv), _ptr(rope_tab), _ptr(dx),
                                  _ptr(dw_qkv), _ptr(workspace), _nbytes(workspace), B, T, C, H, H_kv, d,
                                  _stream_handle(stream)), "attn_qkv_proj_bwd")


def qkv_projection(x, w_qkv, H, H_kv, d, rope_tab=None):
    """Allocates and returns (q, k, v)."""
    B, T, C = _proj_dims(x, w_qkv, H, H_kv, d)
    q = torch.empty((B, H, T, d), dtype=torch.bfloat16, device=x.device)
    k = torch.empty((B, H_kv, T, d), dtype=torch.bfloat16, device=x.device)
    v = torch.empty_like(k)
    attn_qkv_proj(x, w_qkv, q, k, v, rope_tab)
    return q, k, v


def out_projection(o, w_o):
    B, H, T, d = _shape(o)
    y = torch.empty((B, T, int(w_o.shape[0])), dtype=torch.bfloat16, device=o.device)
    attn_out_proj(o, w_o, y)
    return y


def out_projection_backward(dy, o, w_o, workspace=None):
    """Allocates and returns (dO, dW_o)."""
    B, H, T, d = _shape(o)
    C = int(w_o.shape[0])
    d_o = torch.empty_like(o)
    dw_o = torch.empty((C, H * d), dtype=torch.float32, device=o.device)
    if workspace is None:
        workspace = new_proj_workspace(B, T, C, H, H, d, o.device)
    attn_out_proj_bwd(dy, o, w_o, d_o, dw_o, workspace)
    return d_o, dw_o


def qkv_projection_backward(dq, dk, dv, x, w_qkv, rope_tab=None, workspace=None):
    """Allocates and returns (dX, dW_qkv)."""
    B, H, T, d = _shape(dq)
    H_kv = _shape(dk)[1]
    C = int(x.shape[2])
    dx = torch.empty_like(x)
    dw = torch.empty(tuple(w_qkv.shape), dtype=torch.float32, device=x.device)
    if workspace is None:
        workspace = new_proj_workspace(B, T, C, H, H_kv, d, x.device)
    attn_qkv_proj_bwd(dq, dk, dv, x, w_qkv, dx, dw, workspace, rope_tab)
    return dx, dw
