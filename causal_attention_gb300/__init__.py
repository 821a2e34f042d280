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

import torch

from ._lib import load_library, ATTN_OK, AttnError, STATUS_NAMES  # noqa: F401

_dll = load_library()


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
