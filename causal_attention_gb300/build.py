"""Builds libattn.so (the C-ABI attention library) in-tree for sm_103a.

Each CUDA translation unit is compiled by its own nvcc process (in parallel), then
linked into ``causal_attention_gb300/lib/libattn.so``. The CUDA runtime is the shared
``libcudart.so.13``: when PyTorch has loaded its copy first, the library uses that same
runtime (one current device per thread for both); otherwise the toolkit's copy is found
through the RPATH. Nothing links libcuda, so the library loads without a GPU driver
(the driver is looked up on first use). Run ``python causal_attention_gb300/build.py`` (by path: importing
the package loads the library it builds).
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
LIBDIR = os.path.join(PKG, "lib")
LIB = os.path.join(LIBDIR, "libattn.so")
# the same library with device-side bounds checks (-DATTN_DEBUG_BOUNDS=1): every TMA
# coordinate, bulk-copy range and global store index is checked before the access
DEBUG_LIB = os.path.join(LIBDIR, "libattn_debug.so")
SOURCES = ["attn_api.cu", "attn_fwd.cu", "attn_bwd.cu", "gemm.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libattn.so")


def _flags(extra=()):
    return [*ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
            "-I" + os.path.join(ROOT, "include"), *extra]


def build(verbose: bool = False, ptxas_verbose: bool = False, debug: bool = True) -> str:
    """Builds libattn.so and (debug=True) libattn_debug.so, every translation unit of both
    compiled in parallel. Returns the path of libattn.so."""
    os.makedirs(LIBDIR, exist_ok=True)
    cc = nvcc()
    extra = ["-Xptxas", "-v"] if ptxas_verbose else []
    variants = [(LIB, os.path.join(LIBDIR, "obj"), [])]
    if debug:
        variants.append((DEBUG_LIB, os.path.join(LIBDIR, "obj_debug"), ["-DATTN_DEBUG_BOUNDS=1"]))
    jobs = []
    for lib, objdir, defs in variants:
        os.makedirs(objdir, exist_ok=True)
        jobs += [(src, objdir, defs) for src in SOURCES]

    def compile_one(job):
        src, objdir, defs = job
        obj = os.path.join(objdir, src.replace(".cu", ".o"))
        cmd = [cc, *_flags(extra + defs), "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src} {' '.join(defs)}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stdout + r.stderr

    with cf.ThreadPoolExecutor(max_workers=len(jobs)) as ex:
        results = list(ex.map(compile_one, jobs))
    logs = "".join(log for _, log in results[:len(SOURCES)])
    if verbose or ptxas_verbose:
        sys.stdout.write(logs)
    cuda_lib = os.path.join(os.path.dirname(os.path.dirname(cc)), "lib64")
    for i, (lib, _, _) in enumerate(variants):
        objs = [o for o, _ in results[i * len(SOURCES):(i + 1) * len(SOURCES)]]
        tmp = lib + ".tmp"
        cmd = [cc, *ARCH, "-shared", "-cudart", "shared", "-Xlinker", f"-rpath,{cuda_lib}", "-o", tmp, *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib)
    return LIB


if __name__ == "__main__":
    print(build(verbose=True, ptxas_verbose="-v" in sys.argv))
