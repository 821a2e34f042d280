"""ctypes declarations of the C ABI in include/attn.h."""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "lib", "libattn.so")
# the same library built with device-side bounds checks (see build.py)
DEBUG_LIB_PATH = os.path.join(_HERE, "lib", "libattn_debug.so")

ATTN_OK = 0
STATUS_NAMES = {
    0: "ATTN_OK",
    1: "ATTN_ERR_INVALID_ARG",
    2: "ATTN_ERR_UNSUPPORTED",
    3: "ATTN_ERR_MISALIGNED",
    4: "ATTN_ERR_WORKSPACE",
    5: "ATTN_ERR_LAUNCH",
    6: "ATTN_ERR_DEVICE_TIMEOUT",
    7: "ATTN_ERR_CUDA",
    8: "ATTN_ERR_DEVICE_BOUNDS",
}


class AttnError(RuntimeError):
    def __init__(self, status, what, detail=""):
        self.status = status
        super().__init__(f"{what}: {STATUS_NAMES.get(status, status)}" + (f" ({detail})" if detail else ""))


_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float
_S = ctypes.c_size_t

SIGNATURES = {
    "attn_abi_version": (_I, []),
    "attn_fwd": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _F, _I, _P]),
    "attn_fwd_gqa": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _P]),
    "attn_bwd_workspace_size": (_S, [_I, _I, _I, _I]),
    "attn_bwd_fused_workspace_size": (_S, [_I, _I, _I, _I]),
    "attn_bwd_gqa_workspace_size": (_S, [_I, _I, _I, _I, _I]),
    "attn_bwd": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _S, _I, _I, _I, _I, _F, _I, _P]),
    "attn_bwd_gqa": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _S, _I, _I, _I, _I, _I, _F, _I, _P]),
    "attn_bwd_preprocess": (_I, [_P, _P, _P, _P, _S, _I, _I, _I, _I, _P]),
    "attn_bwd_dkdv": (_I, [_P, _P, _P, _P, _P, _P, _P, _S, _I, _I, _I, _I, _F, _I, _P]),
    "attn_bwd_dq": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _S, _I, _I, _I, _I, _F, _I, _P]),
    "attn_bwd_dkdv_dq": (_I, [_P, _P, _P, _P, _P, _P, _P, _S, _I, _I, _I, _I, _F, _I, _P]),
    "attn_bwd_dq_finish": (_I, [_P, _P, _S, _I, _I, _I, _I, _F, _P]),
    "attn_bwd_noalloc": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _F, _I, _P]),
    "attn_check_device_error": (_I, [_P]),
    "attn_selftest_wait_timeout": (_I, [_P]),
    "attn_gemm_workspace_size": (_S, [_I, _I, _I, _I]),
    "attn_gemm": (_I, [_P, _P, _P, _I, _I, _I, _I, _P, _S, _P]),
    "attn_rope_table": (_I, [_P, _I, _I, _P]),
    "attn_rope": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _P]),
    "attn_qkv_proj": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P]),
    "attn_out_proj": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _P]),
    "attn_proj_bwd_workspace_size": (_S, [_I, _I, _I, _I, _I, _I]),
    "attn_out_proj_bwd": (_I, [_P, _P, _P, _P, _P, _P, _S, _I, _I, _I, _I, _I, _P]),
    "attn_qkv_proj_bwd": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _S, _I, _I, _I, _I, _I, _I, _P]),
    "attn_status_string": (ctypes.c_char_p, [_I]),
    "attn_last_cuda_error": (ctypes.c_char_p, []),
}


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Loads libattn.so; raises if it is missing (there is no fallback path)."""
    if not os.path.exists(path):
        raise ImportError(
            f"libattn.so not found at {path}; build it with `python causal_attention_gb300/build.py`")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib
