"""attn_bwd_noalloc: the backward for callers that cannot allocate device memory (a
plug-in whose host framework owns every device allocation, or a latency-critical step
that must not call cudaMalloc/cudaFree, which can synchronise the device). It keeps its
scratch in the library's fixed device array instead of a caller workspace.

Checked through the C ABI against attn_bwd (with a workspace) on the same inputs. Both
run the same kernels in the same order on the same values, and the backward is bitwise
deterministic, so the results must be identical, not merely close: any difference would
come from the shared scratch (stale contents of an earlier call, or two calls racing on
it). Two cases: two calls in a row with a synchronisation after each (the second finds the
first call's contents in the scratch), and two calls with different inputs queued back to
back on one stream with a single synchronisation at the end (the second call's first
kernel must not overwrite the scratch while the first call's last kernel still reads it).
Collected last, so that a run stopping at the first failure has run every other test; it
also passes on its own in a fresh process."""
import pytest
import torch

import seeded_inputs as si
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

OUTS = ("dq", "dk", "dv")


def _inputs(w):
    import causal_attention_gb300 as ca
    x = si.make_inputs(w)
    q, k, v, do = (gu.to_device(x[n]) for n in ("q", "k", "v", "do"))
    o, lse = ca.forward(q, k, v, w.scale, True)
    ref = dict(zip(OUTS, ca.backward(q, k, v, o, do, lse, w.scale, True)))
    ca.check_device_error()
    return (q, k, v, o, do, lse), ref


def _noalloc(args, w, stream=None):
    import causal_attention_gb300 as ca
    q = args[0]
    got = {n: torch.full_like(q, float("nan")) for n in OUTS}
    ca.attn_bwd_noalloc(*args, got["dq"], got["dk"], got["dv"], w.scale, True, stream)
    return got


WORKLOADS = (si.WORKLOADS["gpt12m"], si.Workload("noalloc-ragged", 2, 3, 300, 128, seed=31))


def test_noalloc_matches_workspace_backward_twice():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import causal_attention_gb300 as ca
    for w in WORKLOADS:
        args, ref = _inputs(w)
        for call in range(2):
            got = _noalloc(args, w)
            ca.check_device_error()
            for n in OUTS:
                assert torch.equal(got[n], ref[n]), f"{w.name} call {call} {n}"


@pytest.mark.parametrize("w", WORKLOADS, ids=lambda w: w.name)
def test_noalloc_back_to_back_on_one_stream(w):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import causal_attention_gb300 as ca
    args_a, ref_a = _inputs(w)
    args_b, ref_b = _inputs(w.with_(seed=w.seed + 17))
    st = torch.cuda.Stream()
    torch.cuda.synchronize()  # inputs and references are ready before the stream starts
    got_a = _noalloc(args_a, w, st)
    got_b = _noalloc(args_b, w, st)
    ca.check_device_error(st)
    for n in OUTS:
        assert torch.equal(got_a[n], ref_a[n]), f"first call {n}"
        assert torch.equal(got_b[n], ref_b[n]), f"second call {n}"


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
