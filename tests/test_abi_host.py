"""The C-ABI library on the host: it loads without a GPU, exports every function
that include/attn.h declares, and rejects invalid calls before touching CUDA."""
import ctypes
import os
import re

import pytest

from causal_attention_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn.h")


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(_lib.LIB_PATH):
        import causal_attention_gb300.build as b
        b.build()
    return _lib.load_library()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?\w+\*?\s+\*?(attn_\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_expected_entry_points():
    names = declared_functions()
    for n in ("attn_fwd", "attn_bwd", "attn_bwd_workspace_size", "attn_bwd_preprocess", "attn_bwd_dkdv",
              "attn_bwd_dq", "attn_check_device_error", "attn_status_string", "attn_abi_version",
              "attn_gemm", "attn_qkv_proj", "attn_out_proj", "attn_out_proj_bwd", "attn_qkv_proj_bwd"):
        assert n in names
    assert set(names) == set(_lib.SIGNATURES), "binding signatures out of sync with attn.h"


def test_every_declared_symbol_is_exported(lib):
    for n in declared_functions():
        assert hasattr(lib, n), n


def test_bounds_checked_build_loads_and_exports_the_same_symbols(lib):
    """libattn_debug.so (device-side bounds checks) is the same C ABI."""
    if not os.path.exists(_lib.DEBUG_LIB_PATH):
        import causal_attention_gb300.build as b
        b.build()
    dbg = _lib.load_library(_lib.DEBUG_LIB_PATH)
    for n in declared_functions():
        assert hasattr(dbg, n), n
    assert dbg.attn_abi_version() == lib.attn_abi_version()
    assert b"bounds" in dbg.attn_status_string(8)


def test_abi_version(lib):
    assert lib.attn_abi_version() == 3


def test_status_strings(lib):
    for code in range(9):
        assert lib.attn_status_string(code)
    assert b"unknown" in lib.attn_status_string(99)


def base_ws(B, H, T):
    return 2 * 4 * B * H * ((T + 127) // 128 * 128)


def test_workspace_size(lib):
    assert lib.attn_bwd_workspace_size(2, 3, 200, 64) == base_ws(2, 3, 200) == 2 * 4 * 2 * 3 * 256
    assert lib.attn_bwd_workspace_size(1, 1, 128, 128) == 2 * 4 * 128
    assert lib.attn_bwd_workspace_size(0, 1, 128, 64) == 0
    assert lib.attn_bwd_workspace_size(1, 1, 128, 48) == 0
    assert lib.attn_bwd_workspace_size(1, 1, 128, 80) == 2 * 4 * 128  # d = 80 is served


def test_fused_workspace_size(lib):
    # base (two fp32 [B*H, T_pad] arrays) + fp32 dQ tiles + int32 counters per 128-row
    # query tile rounded up to 256 bytes; no fused path at d = 128
    f = lib.attn_bwd_fused_workspace_size
    assert f(2, 3, 200, 64) == base_ws(2, 3, 200) + 6 * 256 * 64 * 4 + 256
    assert f(1, 2, 1, 32) == base_ws(1, 2, 1) + 2 * 128 * 32 * 4 + 256
    assert f(4, 64, 1024, 64) == base_ws(4, 64, 1024) + 256 * 1024 * 64 * 4 + 8192
    assert f(1, 1, 128, 128) == 0 and f(1, 1, 128, 80) == 0
    assert f(0, 1, 128, 64) == 0


P = 0x10000  # a fake, 16-byte aligned address: never dereferenced when a check fails first


def fwd(lib, B=1, H=1, T=64, d=64, scale=0.125, causal=1, ptrs=(P, P, P, P, P)):
    return lib.attn_fwd(*[ctypes.c_void_p(p) for p in ptrs], B, H, T, d, ctypes.c_float(scale), causal,
                        ctypes.c_void_p(0))


@pytest.mark.parametrize("kw,code", [
    (dict(B=0), 1), (dict(H=-1), 1), (dict(T=0), 1), (dict(T=1 << 25), 1),
    (dict(d=48), 2), (dict(d=256), 2), (dict(d=96), 2),
    (dict(scale=0.0), 1), (dict(scale=float("inf")), 1), (dict(scale=float("nan")), 1), (dict(scale=-1.0), 1),
    (dict(causal=2), 1),
    (dict(ptrs=(0, P, P, P, P)), 1), (dict(ptrs=(P, P, P, P, 0)), 1),
    (dict(ptrs=(P + 8, P, P, P, P)), 3), (dict(ptrs=(P, P, P, P + 4, P)), 3),
])
def test_fwd_rejects_invalid_calls(lib, kw, code):
    assert fwd(lib, **kw) == code


def test_bwd_rejects_invalid_calls(lib):
    v = [ctypes.c_void_p(P)] * 9
    ws = lib.attn_bwd_workspace_size(1, 1, 64, 64)
    args = lambda wsp, wsb, d=64: (*v, ctypes.c_void_p(wsp), wsb, 1, 1, 64, d, ctypes.c_float(0.125), 1,
                                   ctypes.c_void_p(0))
    assert lib.attn_bwd(*args(0, ws)) == 4            # no workspace
    assert lib.attn_bwd(*args(P, ws - 16)) == 4       # too small
    assert lib.attn_bwd(*args(P + 4, ws)) == 3        # misaligned workspace
    assert lib.attn_bwd(*args(P, ws, d=40)) == 2
    assert lib.attn_bwd_preprocess(ctypes.c_void_p(P), ctypes.c_void_p(P), ctypes.c_void_p(P),
                                   ctypes.c_void_p(P), base_ws(1, 1, 64) - 1, 1, 1, 64, 64, ctypes.c_void_p(0)) == 4


def test_fused_dq_stages_reject_invalid_calls(lib):
    """The fused dK/dV/dQ stage needs d <= 64 and the full workspace."""
    v = [ctypes.c_void_p(P)] * 6
    ws = lib.attn_bwd_fused_workspace_size(1, 1, 64, 64)
    call = lambda wsb, d=64: lib.attn_bwd_dkdv_dq(*v, ctypes.c_void_p(P), wsb, 1, 1, 64, d, ctypes.c_float(0.125),
                                                   1, ctypes.c_void_p(0))
    assert call(ws - 16) == 4                 # base-sized workspace: not enough for the fused path
    assert call(base_ws(1, 1, 64) - 16) == 4
    assert call(10 ** 9, d=128) == 2          # no fused path at d = 128
    assert call(ws, d=48) == 2
    fin = lambda wsb, d=64: lib.attn_bwd_dq_finish(ctypes.c_void_p(P), ctypes.c_void_p(P), wsb, 1, 1, 64, d,
                                                    ctypes.c_float(0.125), ctypes.c_void_p(0))
    assert fin(ws - 16) == 4
    assert fin(10 ** 9, d=128) == 2
    assert lib.attn_bwd_dq_finish(ctypes.c_void_p(P + 8), ctypes.c_void_p(P), ws, 1, 1, 64, 64,
                                  ctypes.c_float(0.125), ctypes.c_void_p(0)) == 3


def test_valid_call_without_gpu_fails_cleanly(lib):
    """With no CUDA device the checks pass and the first CUDA call reports an error."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert fwd(lib) == 7
    assert lib.attn_last_cuda_error()


@pytest.mark.parametrize("H,H_kv,code", [(6, 4, 1), (6, 0, 1), (6, 7, 1), (6, -2, 1)])
def test_gqa_rejects_invalid_head_counts(lib, H, H_kv, code):
    args = [ctypes.c_void_p(P)] * 5
    assert lib.attn_fwd_gqa(*args, 1, H, H_kv, 64, 64, ctypes.c_float(0.125), 1, ctypes.c_void_p(0)) == code
    ws = lib.attn_bwd_workspace_size(1, H, 64, 64)
    bargs = [ctypes.c_void_p(P)] * 10
    assert lib.attn_bwd_gqa(*bargs, ws, 1, H, H_kv, 64, 64, ctypes.c_float(0.125), 1, ctypes.c_void_p(0)) == code


def test_gqa_workspace_size(lib):
    f = lib.attn_bwd_gqa_workspace_size
    # at least one dK/dV work item per SM (B * H_kv * n_q >= 152): the attn_bwd workspace
    assert f(4, 16, 16, 2048, 64) == base_ws(4, 16, 2048)
    assert f(4, 64, 16, 2048, 64) == base_ws(4, 64, 2048)  # 4*16*16 = 1024 items
    assert f(4, 16, 4, 2048, 64) == base_ws(4, 16, 2048)  # 256 items
    assert f(1, 16, 4, 4864, 64) == base_ws(1, 16, 4864)  # exactly 152 items
    # 151 items: split up to 304 items, ceil(304 / 151) = 3 splits
    assert f(1, 16, 1, 151 * 128, 64) == base_ws(1, 16, 151 * 128) + 2 * 3 * 1 * 151 * 128 * 64 * 4
    # MQA at B4 T2048: 64 items -> S = min(16, ceil(304 / 64)) = 5 splits of fp32 dK, dV
    assert f(4, 16, 1, 2048, 64) == base_ws(4, 16, 2048) + 2 * 5 * 4 * 1 * 2048 * 64 * 4
    # the split count is bounded by the group size
    assert f(1, 2, 1, 128, 32) == base_ws(1, 2, 128) + 2 * 2 * 1 * 1 * 128 * 32 * 4
    assert f(1, 6, 4, 128, 64) == 0 and f(1, 6, 0, 128, 64) == 0


# ---------------------------------------------------------------------------
# projections
# ---------------------------------------------------------------------------
def _cp(x):
    return ctypes.c_void_p(x)


def gemm_call(lib, M=128, N=256, K=64, layout=0, ptrs=(P, P, P)):
    return lib.attn_gemm(*[_cp(p) for p in ptrs], M, N, K, layout, _cp(0), 0, _cp(0))


@pytest.mark.parametrize("kw,code", [
    (dict(M=0), 1), (dict(N=-8), 1), (dict(K=0), 1), (dict(M=100), 1), (dict(K=12), 1), (dict(layout=3), 1),
    (dict(layout=-1), 1), (dict(M=1 << 25), 1),
    (dict(ptrs=(0, P, P)), 1), (dict(ptrs=(P, P, 0)), 1), (dict(ptrs=(P + 8, P, P)), 3), (dict(ptrs=(P, P + 4, P)), 3),
])
def test_gemm_rejects_invalid_calls(lib, kw, code):
    assert gemm_call(lib, **kw) == code


def test_gemm_workspace_size(lib):
    f = lib.attn_gemm_workspace_size
    assert f(1024, 1024, 8192, 0) == 0 and f(1024, 1024, 8192, 1) == 0  # nt / nn never split
    # tn: 8 x 4 = 32 output tiles of 128 x 256 -> floor(152 / 32) = 4 splits of 32 K-steps of 64
    assert f(1024, 1024, 8192, 2) == 4 * 1024 * 1024 * 4
    # 24 x 4 = 96 tiles -> one split, no workspace
    assert f(3072, 1024, 8192, 2) == 0
    # at least 8 K-steps per split: K = 256 is 4 K-steps -> no split
    assert f(128, 256, 256, 2) == 0
    # at most 16 splits: one tile, K = 64 * 1024 -> 16 splits of 64 K-steps
    assert f(128, 256, 65536, 2) == 16 * 128 * 256 * 4
    # 152 / 1 = 152 -> capped at 16; K = 64 * 20 -> min(16, 20 // 8 = 2) = 2 splits of 10 K-steps
    assert f(64, 64, 1280, 2) == 2 * 64 * 64 * 4
    assert f(0, 64, 64, 2) == 0 and f(64, 64, 64, 3) == 0


def test_proj_bwd_workspace_size(lib):
    f = lib.attn_proj_bwd_workspace_size
    # B4 T2048 C1024 H16 d64: dW_o is 1024 x 1024 over K = 8192 -> 4 splits (16 MiB); dW_qkv
    # 3072 x 1024 -> no split; the rotated dQ, dK take 2 * 4 * 16 * 2048 * 64 * 2 bytes
    rot = 2 * 4 * 16 * 2048 * 64 * 2
    assert f(4, 2048, 1024, 16, 16, 64) == max(4 * 1024 * 1024 * 4, rot)
    assert f(4, 2048, 1024, 16, 16, 32) == 0  # d must be 64 or 128
    assert f(4, 2048, 1000, 16, 16, 64) > 0 and f(4, 2048, 1004, 16, 16, 64) == 0  # C % 8
    assert f(1, 64, 64, 6, 4, 64) == 0  # H_kv must divide H


def test_projections_reject_invalid_calls(lib):
    ten = [_cp(P)] * 10
    ok_sizes = (2, 64, 128, 2, 2, 64)  # B, T, C, H, H_kv, d
    # qkv: (x, w, q, k, v, rope_tab, B, T, C, H, H_kv, d, stream)
    assert lib.attn_qkv_proj(*ten[:5], _cp(0), 2, 64, 128, 2, 2, 32, _cp(0)) == 2  # d = 32
    assert lib.attn_qkv_proj(*ten[:5], _cp(0), 2, 64, 100, 2, 2, 64, _cp(0)) == 1  # C % 8
    assert lib.attn_qkv_proj(*ten[:5], _cp(0), 2, 64, 128, 4, 3, 64, _cp(0)) == 1  # H_kv
    assert lib.attn_qkv_proj(_cp(0), *ten[:4], _cp(0), *ok_sizes, _cp(0)) == 1
    assert lib.attn_qkv_proj(*ten[:5], _cp(P + 4), *ok_sizes, _cp(0)) == 3  # misaligned table
    # out: (o, w_o, y, B, T, H, d, C, stream)
    assert lib.attn_out_proj(*ten[:3], 2, 64, 2, 80, 128, _cp(0)) == 2
    assert lib.attn_out_proj(*ten[:2], _cp(P + 2), 2, 64, 2, 64, 128, _cp(0)) == 3
    # out bwd: (dy, o, w_o, d_o, dw_o, ws, ws_bytes, B, T, H, d, C, stream)
    assert lib.attn_out_proj_bwd(*ten[:4], _cp(0), _cp(0), 0, 2, 64, 2, 64, 128, _cp(0)) == 1
    # qkv bwd with RoPE needs the workspace for the rotated dQ, dK
    assert lib.attn_qkv_proj_bwd(*ten[:5], _cp(P), _cp(P), _cp(P), _cp(0), 0, *ok_sizes, _cp(0)) == 4
    # rope: (x, y, tab, B, H, T, d, inverse, stream)
    assert lib.attn_rope(*ten[:3], 1, 1, 8, 12, 0, _cp(0)) == 1
    assert lib.attn_rope(*ten[:3], 1, 1, 8, 64, 2, _cp(0)) == 1
    assert lib.attn_rope_table(_cp(P), 8, 6, _cp(0)) == 1
