"""The oracle over every head of a workload, the heads spread over a pool of `spawn`ed
processes (a forked child of a process that has used CUDA can hang). This module imports
neither torch nor the library, so that each worker starts quickly: a worker imports
numpy, the oracle and the seeded-input conversions only."""
from __future__ import annotations

import multiprocessing as mp
import os

import numpy as np

import oracle
import seeded_inputs as si


def _head(args):
    """One head of the oracle (forward and backward) from its bf16 bit patterns."""
    qb, kb, vb, dob, scale, causal = args
    q, k, v, do = (si.bf16_bits_to_f64(b) for b in (qb, kb, vb, dob))
    o, lse, _ = oracle.head_forward(q, k, v, scale, causal)
    dq, dk, dv, _ = oracle.head_backward(q, k, v, do, scale, causal, o=o, lse=lse)
    return o, lse, dq, dk, dv


def all_heads(scale, causal, x, workers=8):
    """Forward and backward of every head (one key/value head per query head) of the
    seeded bit patterns x (q, k, v, do: [B, H, T, d]). Each worker runs one head at a time
    with two BLAS threads. Returns {o, lse, dq, dk, dv} as fp64 arrays."""
    B, H = x["q"].shape[:2]
    jobs = [(x["q"][b, h], x["k"][b, h], x["v"][b, h], x["do"][b, h], scale, causal)
            for b in range(B) for h in range(H)]
    saved = {n: os.environ.get(n) for n in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS")}
    os.environ.update(OPENBLAS_NUM_THREADS="2", OMP_NUM_THREADS="2")
    try:
        n = max(1, min(workers, len(jobs), (os.cpu_count() or 2) // 2))
        with mp.get_context("spawn").Pool(n) as pool:
            res = pool.map(_head, jobs, chunksize=1)
    finally:
        for k, val in saved.items():
            if val is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = val
    out = {}
    for j, name in enumerate(("o", "lse", "dq", "dk", "dv")):
        out[name] = np.stack([r[j] for r in res]).reshape((B, H) + res[0][j].shape)
    return out
