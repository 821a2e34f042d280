"""attn_bwd_noalloc: the backward for callers that cannot allocate device memory (a
plug-in whose host framework owns every device allocation, or a latency-critical step
that must not call cudaMalloc/cudaFree, which can synchronise the device). It keeps its
scratch in the library's fixed device array instead of a caller workspace.

Checked through the C ABI against attn_bwd (with a workspace) on the same inputs, on two
calls in a row: the second call finds the first call's contents in the shared scratch
and must still match. Collected last, so that a run stopping at the first failure has
run every other test; it also passes on its own in a fresh process."""
import pytest
import torch

import seeded_inputs as si
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


def test_noalloc_matches_workspace_backward_twice():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import causal_attention_gb300 as ca
    for w in (si.WORKLOADS["gpt12m"], si.Workload("noalloc-ragged", 2, 3, 300, 128, seed=31)):
        x = si.make_inputs(w)
        q, k, v, do = (gu.to_device(x[n]) for n in ("q", "k", "v", "do"))
        o, lse = ca.forward(q, k, v, w.scale, True)
        ref = dict(zip(("dq", "dk", "dv"), ca.backward(q, k, v, o, do, lse, w.scale, True)))
        ca.check_device_error()
        for call in range(2):
            got = {n: torch.full_like(q, float("nan")) for n in ("dq", "dk", "dv")}
            ca.attn_bwd_noalloc(q, k, v, o, do, lse, got["dq"], got["dk"], got["dv"], w.scale, True)
            ca.check_device_error()
            for n in ("dq", "dk", "dv"):
                a, b = gu.to_f64(got[n]), gu.to_f64(ref[n])
                assert gu.rel_rms(a, b) <= gu.TOL_GRAD_REL_RMS, f"{w.name} call {call} {n}"
                assert gu.max_abs(a, b) <= 1e-2, f"{w.name} call {call} {n}"


def test_noalloc_rejects_shapes_beyond_its_scratch():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import causal_attention_gb300 as ca
    from causal_attention_gb300 import AttnError
    t = torch.empty(8, dtype=torch.bfloat16, device="cuda")  # never touched: rejected first
    B, H, T, d = 8, 16, 8192 + 1, 64                          # B*H*T_pad = 1,064,960 > 1,048,576
    big = t.as_strided((B, H, T, d), (0, 0, 0, 0))
    lse = torch.empty(1, device="cuda").as_strided((B, H, T), (0, 0, 0))
    with pytest.raises(AttnError, match="WORKSPACE"):
        ca._dll and ca._check(ca._dll.attn_bwd_noalloc(*(ca._ptr(x) for x in (big,) * 5), ca._ptr(lse),
                                                       *(ca._ptr(x) for x in (big,) * 3), B, H, T, d,
                                                       ca.ctypes.c_float(0.125), 1, ca._stream_handle(None)),
                              "attn_bwd_noalloc")
