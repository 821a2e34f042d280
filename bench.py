"""Throughput of the fused causal attention forward + backward on GB300.

One step = attn_fwd followed by attn_bwd over one batch of the workload, through the
C ABI (at d <= 64 the backward is the dQ kernel, which also forms D, then dK/dV; at
d = 80 and 128 D, dK/dV, dQ; with --fused-dq, at d <= 64: D, dK/dV with dQ fused, dQ
conversion). Prints ONE JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

* value: credited causal TFLOP/s of the whole job (forward 2*B*H*T^2*d, backward
  2.5x that), inputs resident in HBM; inputs rotate over several buffer sets whose
  total size exceeds L2 three times, so no step reads another's operands from L2. The
  K timed steps are launched as one CUDA graph (captured after the warm-up, replayed once
  before the measurement; --eager launches them one by one). The per-kernel durations
  (the roofline's) come from a second pass over the same K steps right after, launched
  one by one with a CUDA event before and after every kernel.
* e2e: the same metric through the public API with pinned host buffers: every step
  copies Q, K, V, dO host->device and O, LSE, dQ, dK, dV device->host; steps are
  pipelined over two device buffer sets and three streams, as a caller would run them.
* roofline: the kernel with the largest share of step time, its algorithmic FLOPs
  per launch over its mean CUDA-event duration, against the measured bf16 peak.
* cpu_baseline: the CPU oracle timed on this host on a bounded sample (whole heads of
  the same workload until about 10 s of work), as it stands.
* parity_receipt: before anything is timed, one step of the same shape on the GPU is
  compared with that oracle run on the sampled heads (the tests' bars); a failed receipt
  ends the run without a line. Warm-up, timed steps and the end-to-end measurement run
  under an exclusive file lock per GPU, so that two runs never time one device at once.
* --impl reference: the CPU oracle as the reference arm (the pages publish no code
  that runs here), each step a bounded sample of the workload.

Multi-GPU: one process per GPU under torchrun; every rank runs its own replica of the
workload (independent problems, no collective on the data path), "scaling": "weak".
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

L2_BYTES = 129 * 1024 * 1024


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="long8k",
                    help="seeded workload (default long8k, B1 H16 T8192 d128: the largest configuration)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    # The end-to-end steps run as a pipeline (copies in, compute, copies out on three
    # streams): the first step's copy in and the last step's copy out are not overlapped, so
    # the measurement runs enough steps that they weigh little (1.5 % of 100 long8k steps).
    ap.add_argument("--e2e-steps", type=int, default=100)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--kv-heads", type=int, default=0,
                    help="grouped key/value heads: H_kv (dividing H); the step is attn_fwd + attn_bwd timed whole")
    ap.add_argument("--non-causal", action="store_true",
                    help="the workload's shapes without the causal mask (credited FLOPs doubled)")
    ap.add_argument("--head-dim", type=int, default=0,
                    help="the workload's shapes at another head dimension (32, 64, 80 or 128)")
    ap.add_argument("--block", action="store_true",
                    help="the attention block's training step: QKV projection (RoPE) -> attention -> output "
                         "projection, and the backward of all three (model width C = H d)")
    ap.add_argument("--eager", action="store_true",
                    help="launch the timed steps one by one instead of replaying them as one CUDA graph")
    ap.add_argument("--fused-dq", action="store_true",
                    help="time the fused-dQ backward stages (d <= 64) instead of attn_bwd's kernels")
    ap.add_argument("--order", default="fwd-bwd", choices=["fwd-bwd", "bwd-fwd"],
                    help="launch order within a step: the backward of a buffer set may run before its "
                         "forward (its O and LSE then come from that set's previous forward)")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d.get("bf16_tflops", 1900.0), d.get("hbm_gbs", 6800.0), "measured"
    return 1900.0, 6800.0, "fallback"


def sustained_peak():
    """The bf16 matmul rate held for seconds under the power cap (a second denominator,
    beside the burst peak the fractions use), or the fallback figure."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        v = json.load(open(p)).get("bf16_tflops_sustained")
        if v:
            return float(v), "measured"
    return 1700.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu_index = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu_index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


class NvmlClockSampler:
    """The SM clock and the clock-event reasons of the benchmark's GPU, read through NVML
    (the driver's library, by ctypes) about every millisecond from a thread while the timed
    region runs: nvidia-smi's 200 ms loop sees at most a sample or two of a region this
    short. The GPU is found by its UUID, so the right one is read whatever
    CUDA_VISIBLE_DEVICES maps. Reads only; changes no setting."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, device):
        import ctypes
        import threading
        self.ok = False
        self.samples, self.mask = [], 0
        self.stop_flag = threading.Event()
        self.thread = None
        try:
            import torch
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                return
            self.lib, self.h = lib, ctypes.c_void_p()
            uuid = str(getattr(torch.cuda.get_device_properties(device), "uuid", ""))
            uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
            if lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(self.h)) != 0:
                return
            self.reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons")
            mx = ctypes.c_uint()
            self.max_mhz = float(mx.value) if lib.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(mx)) == 0 else None
            self.ok = True
        except (OSError, AttributeError, ImportError):
            self.ok = False

    def _run(self):
        import ctypes
        mhz, mask = ctypes.c_uint(), ctypes.c_ulonglong()
        while not self.stop_flag.is_set():
            if self.lib.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(mhz)) == 0:  # 1: the SM clock
                self.samples.append(float(mhz.value))
            if self.reasons_fn(self.h, ctypes.byref(mask)) == 0:
                self.mask |= int(mask.value)
            time.sleep(0.001)

    def start(self):
        if self.ok:
            import threading
            self.thread = threading.Thread(target=self._run, daemon=True)
            self.thread.start()

    def stop(self):
        if not self.ok or self.thread is None:
            return None
        self.stop_flag.set()
        self.thread.join(timeout=5)
        if not self.samples:
            return None
        return {"sm_mhz": statistics.median(self.samples), "sm_max_mhz": self.max_mhz,
                "reasons": sorted(n for b, n in self.REASONS.items() if self.mask & b),
                "samples": len(self.samples), "source": "NVML, every ~1 ms during the timed region"}


def oracle_sample(w, n_heads, x=None, budget_s=None, H_kv=None):
    """Runs the CPU oracle fwd + bwd on up to n_heads query heads (stopping once budget_s
    seconds have passed, after at least one head); with H_kv key/value heads in x, query
    head h uses key/value head h // (H / H_kv). Returns (credited FLOPs, seconds, heads
    run, {(b, h): (O, LSE, dQ, dK, dV) of that head}), dK and dV being that query head's
    contribution to its key/value head."""
    import numpy as np  # noqa: F401
    import oracle
    import seeded_inputs as si
    x = x or si.make_inputs(w)
    G = w.H // (H_kv or w.H)
    heads = [(i // w.H % w.B, i % w.H) for i in range(n_heads)]
    q, k, v, do = (si.bf16_bits_to_f64(x[n]) for n in ("q", "k", "v", "do"))
    t0 = time.perf_counter()
    outs = {}
    for b, h in heads:
        g = h // G
        o, lse, _ = oracle.head_forward(q[b, h], k[b, g], v[b, g], w.scale, w.causal)
        dq, dk, dv, _ = oracle.head_backward(q[b, h], k[b, g], v[b, g], do[b, h], w.scale, w.causal)
        outs[(b, h)] = (o, lse, dq, dk, dv)
        if budget_s is not None and time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    fwd, bwd = credited_flops(1, 1, w.T, w.d)
    return (fwd + bwd) * (1.0 if w.causal else 2.0) * len(outs), dt, len(outs), outs


# The bars a timed line must pass first (the tests' tolerances): O max-abs and rel-RMS,
# LSE max-abs, and rel-RMS of each gradient, over the heads the oracle sampled.
RECEIPT_BARS = {"o_max_abs": 2e-2, "o_rel_rms": 5e-3, "lse_max_abs": 1e-3, "grad_rel_rms": 1e-2}


def parity_receipt(gpu, ref, G=1):
    """Compares GPU outputs with the oracle's on the sampled heads. gpu and ref map (b, h)
    to (O, LSE, dQ, dK, dV) (fp64 arrays; dK and dV of the GPU are those of the head's
    key/value head). A key/value head's dK and dV are compared only when all G query heads
    that use it were sampled (their contributions summed). Returns the receipt dict."""
    import numpy as np

    def rel(a, b):
        return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))

    keys = sorted(ref)
    cat = lambda src, i: np.concatenate([np.ravel(src[key][i]) for key in keys])
    o_g, o_r = cat(gpu, 0), cat(ref, 0)
    l_g, l_r = cat(gpu, 1), cat(ref, 1)
    r = {"heads": len(keys), "o_max_abs": float(np.max(np.abs(o_g - o_r))), "o_rel_rms": rel(o_g, o_r),
         "lse_max_abs": float(np.max(np.abs(l_g - l_r))), "dq_rel_rms": rel(cat(gpu, 2), cat(ref, 2))}
    groups = {}
    for b, h in keys:
        groups.setdefault((b, h // G), []).append((b, h))
    full = [kv for kv, hs in groups.items() if len(hs) == G]
    if full:
        for i, name in ((3, "dk_rel_rms"), (4, "dv_rel_rms")):
            g_ = np.concatenate([np.ravel(gpu[groups[kv][0]][i]) for kv in full])
            r_ = np.concatenate([np.ravel(sum(ref[hk][i] for hk in groups[kv])) for kv in full])
            r[name] = rel(g_, r_)
    bars = RECEIPT_BARS
    r["pass"] = bool(r["o_max_abs"] <= bars["o_max_abs"] and r["o_rel_rms"] <= bars["o_rel_rms"]
                     and r["lse_max_abs"] <= bars["lse_max_abs"]
                     and all(r[k] <= bars["grad_rel_rms"] for k in ("dq_rel_rms", "dk_rel_rms", "dv_rel_rms") if k in r))
    return r


class GpuLock:
    """An exclusive file lock per GPU around the timed work, so that two runs of this
    bench never time the same device at once (released when the process exits)."""

    def __init__(self, index):
        self.path = os.path.join(tempfile.gettempdir(), f"causal_attention_gb300.gpu{index}.lock")
        self.fd = None

    def __enter__(self):
        import fcntl
        self.fd = open(self.path, "w")
        fcntl.flock(self.fd, fcntl.LOCK_EX)
        return self

    def __exit__(self, *exc):
        import fcntl
        fcntl.flock(self.fd, fcntl.LOCK_UN)
        self.fd.close()
        return False


def blas_threads():
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        if os.environ.get(var):
            return int(os.environ[var])
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


def run_reference(args, rank, world):
    """The CPU oracle as the reference arm: each step a bounded sample (one head)."""
    import seeded_inputs as si
    w = si.WORKLOADS[args.workload]
    w = variant(w, args)
    if rank != 0:
        return
    x = si.make_inputs(w)
    H_kv = args.kv_heads or w.H  # the same key/value heads as our arm: the first H_kv slices
    if H_kv != w.H:
        x = dict(x, k=x["k"][:, :H_kv].copy(), v=x["v"][:, :H_kv].copy())
    heads_per_step = 1
    for _ in range(args.warmup if w.T <= 2048 else 0):
        oracle_sample(w, heads_per_step, x, H_kv=H_kv)
    flops = secs = 0.0
    for _ in range(args.steps):
        f, s, _, _ = oracle_sample(w, heads_per_step, x, H_kv=H_kv)
        flops += f
        secs += s
    value = flops / secs / 1e12
    line = {
        "impl": "reference", "metric": "causal attention fwd+bwd TFLOP/s (bf16) and % of GB300 dense BF16 peak",
        "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": secs / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "H_kv": H_kv, "T": w.T, "d": w.d, "causal": w.causal,
                   "parallelism": "replicas", "sample": f"{heads_per_step} head(s) per step"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": blas_threads(), "kind": "oracle",
                         "sample": f"{heads_per_step} head of {w.B * w.H} per step, fp64 numpy oracle"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "provenance": provenance(w.seed),
    }
    print(json.dumps(line), flush=True)


def variant(w, args):
    """The workload as the flags change it (no causal mask; another head dimension; fewer
    key/value heads), renamed so that its traffic records are its own."""
    if args.non_causal:  # renamed: its kernels and traffic differ from the causal workload's
        w = w.with_(name=f"{w.name}_noncausal", causal=False)
    if args.head_dim and args.head_dim != w.d:
        w = w.with_(name=f"{w.name}_d{args.head_dim}", d=args.head_dim)
    kv = getattr(args, "kv_heads", None)
    if kv and kv != w.H:
        w = w.with_(name=f"{w.name}_kv{kv}")
    return w


def kernels_for(d, fused_dq):
    """The launches of one step, in order: the forward, then attn_bwd's stages (d <= 64:
    dQ, which also forms D, then dK/dV; d = 80, 128: D, dK/dV, dQ), or with --fused-dq the
    fused-dQ stages (D, dK/dV with dQ formed inside, dQ conversion)."""
    if fused_dq and d <= 64:
        return ("fwd", "bwd_preprocess", "bwd_dkdv_dq", "bwd_dq_finish")
    if d <= 64:
        return ("fwd", "bwd_dq", "bwd_dkdv")
    return ("fwd", "bwd_preprocess", "bwd_dkdv", "bwd_dq")


def captured_traffic(workload, kernel):
    """DRAM bytes per launch from the committed ncu capture, if the kernel source is
    unchanged since the capture (else None)."""
    import hashlib
    prof = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(prof):
        return None
    rec = json.load(open(prof)).get(f"{workload}:{kernel}")
    if not rec:
        return None
    src = open(os.path.join(ROOT, rec["kernel_source"]), "rb").read()
    if hashlib.sha256(src).hexdigest()[:16] != rec["source_sha256_prefix"]:
        return None
    return rec["bytes_per_launch"]


def provenance(seed, device=None):
    """What produced a line: the sha256 of the library's sources, the GPU, the software
    versions, the seed of the inputs and the host cores."""
    import glob
    import hashlib
    h = hashlib.sha256()
    srcs = sorted(glob.glob(os.path.join(ROOT, "causal_attention_gb300", "csrc", "*"))) + [
        os.path.join(ROOT, "include", "attn.h")]
    for f in srcs:
        h.update(os.path.basename(f).encode())
        h.update(open(f, "rb").read())
    out = {"source_sha256": h.hexdigest()[:16], "seed": seed, "host_cores": os.cpu_count()}
    try:
        import torch
        out.update(torch=torch.__version__, cuda=torch.version.cuda)
        if device is not None and torch.cuda.is_available():
            out["gpu"] = torch.cuda.get_device_name(device)
    except ImportError:
        pass
    return out


def replica(w, rank):
    """The workload of one rank: its own replica (same shapes, seed offset by 1000 per rank),
    so that the ranks solve independent problems (no collective on the data path)."""
    return w.with_(seed=w.seed + 1000 * rank)


def max_over_ranks(value, device=None):
    """The largest value over all ranks (the job ends with its slowest rank); the value
    itself on a single process."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(flops_per_step, steps, world, seconds):
    """Throughput of the whole job: every rank ran `steps` steps of `flops_per_step` within
    `seconds` (the slowest rank's time)."""
    return flops_per_step * steps * world / seconds / 1e12


def spread(values_ms):
    """min / median / p95 of per-launch durations (ms)."""
    v = sorted(values_ms)
    return {"ms_min": round(v[0], 5), "ms_median": round(statistics.median(v), 5),
            "ms_p95": round(v[min(len(v) - 1, int(round(0.95 * (len(v) - 1))))], 5)}


def to_device(bits):
    """A device bf16 tensor from seeded bf16 bit patterns (numpy uint16 / int16)."""
    import numpy as np
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def credited_flops(B, H, T, d):
    """The metric's credited causal FLOPs: forward 2*B*H*T^2*d, backward 2.5 times that (the
    convention that reproduces the Forge RESEARCH.md section 6 table)."""
    fwd = 2.0 * B * H * T * T * d
    return fwd, 2.5 * fwd


def kernel_flops(w):
    """Algorithmic FLOPs per launch of each kernel (causal half of every T x T GEMM)."""
    g = w.B * w.H * w.T * w.T * w.d * (1.0 if w.causal else 2.0)  # one causal GEMM = B*H*T^2*d
    # "bwd": the whole attn_bwd (dQ kernel with its two recomputed GEMMs + dK/dV kernel)
    return {"fwd": 2 * g, "bwd_dkdv": 4 * g, "bwd_dq": 3 * g, "bwd_dkdv_dq": 5 * g, "bwd": 7 * g}


def kernel_bytes(w):
    n = w.B * w.H * w.T
    return {"bwd_preprocess": 2 * n * w.d * 2 + 4 * n + 8 * n, "bwd_dq_finish": n * w.d * (4 + 2)}


def timed_steps(args, step, sets, n_events, stream):
    """The K timed steps, measured twice back to back on `stream`:
    1. throughput: the K steps captured as one CUDA graph (after the warm-up; replayed once
       before the measurement) and replayed between two events, so the timed region holds
       no host launch overhead (--eager: launched one by one instead);
    2. per-kernel durations: the same K steps launched one by one with a timing event before
       and after every kernel (events inside a graph would cost more than the launches).
    Returns (elapsed ms of pass 1, the per-step event lists of pass 2, launch mode)."""
    import torch
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    graph, mode = None, "eager"
    if not args.eager:
        try:
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=stream):
                for i in range(args.steps):
                    step(sets[i % len(sets)], None, stream)
            with torch.cuda.stream(stream):
                graph.replay()
            torch.cuda.synchronize()
            mode = "cuda graph of the K timed steps (per-kernel durations: an eager pass with events)"
        except RuntimeError as e:
            torch.cuda.synchronize()
            graph, mode = None, f"eager (graph capture failed: {e})"
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(n_events)] for _ in range(args.steps)]
    t0.record(stream)
    if graph is not None:
        with torch.cuda.stream(stream):
            graph.replay()
    else:
        for i in range(args.steps):
            step(sets[i % len(sets)], evs[i], stream)
    t1.record(stream)
    if graph is not None:
        for i in range(args.steps):
            step(sets[i % len(sets)], evs[i], stream)
    torch.cuda.synchronize()
    return t0.elapsed_time(t1), evs, mode


def run_ours(args, rank, world, local):
    import torch
    import torch.distributed as dist
    import causal_attention_gb300 as ca
    import seeded_inputs as si

    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    w = variant(si.WORKLOADS[args.workload], args)
    # each rank: its own replica of the workload (different seed, same shape)
    wr = replica(w, rank)
    x = si.make_inputs(wr)
    B, H, T, d = wr.shape
    scale, causal = wr.scale, wr.causal
    dev = torch.device("cuda", local)

    H_kv = args.kv_heads or H
    if H % H_kv:
        raise SystemExit(f"--kv-heads {H_kv} does not divide H = {H}")
    gqa = H_kv != H
    KERNELS = ("fwd", "bwd") if gqa else kernels_for(d, args.fused_dq)
    fused = "bwd_dkdv_dq" in KERNELS
    if args.order == "bwd-fwd":  # the forward last: KERNELS starts with it
        KERNELS = KERNELS[1:] + KERNELS[:1]
    ws_bytes = (ca.attn_bwd_gqa_workspace_size(B, H, H_kv, T, d) if gqa else
                (ca.attn_bwd_fused_workspace_size if fused else ca.attn_bwd_workspace_size)(B, H, T, d))
    per_set = 8 * B * H * T * d * 2 + B * H * T * 4 + ws_bytes
    # attn_bwd_gqa: 2 (d <= 64) or 3 launches, plus the sum of the split dK/dV when its
    # workspace holds the partial sums
    split = gqa and ws_bytes > ca.attn_bwd_workspace_size(B, H, T, d)
    launches_per_step = 1 + (2 if d <= 64 else 3) + int(split) if gqa else len(KERNELS)
    n_sets = max(2, -(-3 * L2_BYTES // per_set))
    if gqa:  # key/value heads: the seeded bytes of the first H_kv heads
        import numpy as np
        x = dict(x, k=np.ascontiguousarray(x["k"][:, :H_kv]), v=np.ascontiguousarray(x["v"][:, :H_kv]))
    base = {n: to_device(x[n]) for n in ("q", "k", "v", "do")}
    sets = []
    for i in range(n_sets):
        s = {n: base[n].clone() for n in base}
        s["o"] = torch.empty_like(s["q"])
        s["lse"] = torch.empty((B, H, T), dtype=torch.float32, device=dev)
        s["dq"], s["dk"], s["dv"] = torch.empty_like(s["q"]), torch.empty_like(s["k"]), torch.empty_like(s["v"])
        s["ws"] = ca.new_workspace(B, H, T, d, dev, fused_dq=fused, kv_heads=H_kv)
        sets.append(s)
    stream = torch.cuda.Stream(device=dev)

    launch = {
        "fwd": lambda s: ca.attn_fwd(s["q"], s["k"], s["v"], s["o"], s["lse"], scale, causal, stream),
        "bwd_preprocess": lambda s: ca.attn_bwd_preprocess(s["o"], s["do"], s["lse"], s["ws"], stream),
        "bwd_dkdv": lambda s: ca.attn_bwd_dkdv(s["q"], s["k"], s["v"], s["do"], s["dk"], s["dv"], s["ws"], scale,
                                               causal, stream),
        "bwd_dq": lambda s: ca.attn_bwd_dq(s["q"], s["k"], s["v"], s["o"], s["do"], s["lse"], s["dq"], s["ws"],
                                           scale, causal, stream),
        "bwd_dkdv_dq": lambda s: ca.attn_bwd_dkdv_dq(s["q"], s["k"], s["v"], s["do"], s["dk"], s["dv"], s["ws"],
                                                     scale, causal, stream),
        "bwd_dq_finish": lambda s: ca.attn_bwd_dq_finish(s["dq"], s["ws"], scale, stream),
        "bwd": lambda s: ca.attn_bwd(s["q"], s["k"], s["v"], s["o"], s["do"], s["lse"], s["dq"], s["dk"], s["dv"],
                                     s["ws"], scale, causal, stream),
    }

    def step(s, ev=None, st=None):
        # the stages attn_bwd runs, called one by one so that each can be timed
        for j, k in enumerate(KERNELS):
            if ev is not None:
                ev[j].record(stream)
            launch[k](s)
        if ev is not None:
            ev[len(KERNELS)].record(stream)

    lock = GpuLock(local).__enter__()  # held until the end-to-end measurement is done
    cpu = receipt = None
    if world == 1 and not args.no_cpu_baseline:
        # A parity receipt at this exact shape before anything is timed: one step on the
        # first buffer set against the CPU oracle on the heads its bounded sample reaches
        # (whole heads until about 10 s of CPU work; that run is also the cpu_baseline).
        import numpy as np
        s0 = sets[0]
        if args.order == "bwd-fwd":
            launch["fwd"](s0)
        step(s0)
        torch.cuda.synchronize()
        ca.check_device_error(stream)
        f, sec, n_heads, ref = oracle_sample(wr, B * H, x, budget_s=10.0, H_kv=H_kv)
        G = H // H_kv
        host = lambda t: t.float().cpu().numpy().astype(np.float64)
        gpu = {(b, h): tuple(host(s0[n][b, h]) for n in ("o", "lse", "dq")) +
               tuple(host(s0[n][b, h // G]) for n in ("dk", "dv")) for b, h in ref}
        receipt = parity_receipt(gpu, ref, G)
        if not receipt["pass"]:
            print(json.dumps({"error": "parity receipt failed: nothing was timed", "parity_receipt": receipt}),
                  file=sys.stderr, flush=True)
            raise SystemExit(1)
        cpu = {"value": f / sec / 1e12, "unit": "TFLOP/s", "cores": blas_threads(), "kind": "oracle",
               "sample": f"{n_heads} of {B * H} heads, fwd+bwd, fp64 numpy oracle, {sec:.1f} s"}
    if args.order == "bwd-fwd":  # every set's O and LSE exist before its first backward
        for s in sets:
            launch["fwd"](s)
    for i in range(max(3, args.warmup)):
        step(sets[i % n_sets])
    ca.check_device_error(stream)

    nvml = NvmlClockSampler(dev) if rank == 0 else None
    sampler = ClockSampler(local) if rank == 0 and not (nvml and nvml.ok) else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    if nvml:
        nvml.start()
    elapsed_ms, evs, launch_mode = timed_steps(args, step, sets, len(KERNELS) + 1, stream)
    clocks = nvml.stop() if nvml else None
    if world > 1:
        dist.barrier()
    if sampler:
        clocks = sampler.stop()
    ca.check_device_error(stream)

    per_kernel = {k: [] for k in KERNELS}
    for ev in evs:
        for j, k in enumerate(KERNELS):
            per_kernel[k].append(ev[j].elapsed_time(ev[j + 1]))
    mean_ms = {k: statistics.fmean(v) for k, v in per_kernel.items()}

    elapsed_ms = max_over_ranks(elapsed_ms, dev)
    fwd_f, bwd_f = credited_flops(B, H, T, d)
    step_flops = (fwd_f + bwd_f) * (1.0 if causal else 2.0)
    value = whole_job_tflops(step_flops, args.steps, world, elapsed_ms * 1e-3)

    # ------------------------------------------------------------------ e2e
    # The public API with host buffers: every step copies its inputs in from pinned host
    # memory, runs attn_fwd + attn_bwd and copies every output back. Steps are pipelined
    # as a user of the API would run them: two device buffer sets, three streams (copies in,
    # compute, copies out), so one step's copies overlap its neighbours' compute.
    pinned = {n: torch.from_numpy(x[n].view("int16")).view(torch.bfloat16).pin_memory() for n in ("q", "k", "v", "do")}

    def host_outs():
        o = {n: torch.empty((B, H, T, d), dtype=torch.bfloat16).pin_memory() for n in ("o", "dq")}
        o.update({n: torch.empty((B, H_kv, T, d), dtype=torch.bfloat16).pin_memory() for n in ("dk", "dv")})
        o["lse"] = torch.empty((B, H, T), dtype=torch.float32).pin_memory()
        return o
    e2e_sets = [sets[0], sets[1 % n_sets]]
    outs_h = [host_outs(), host_outs()]
    h2d = sum(t.numel() * t.element_size() for t in pinned.values())
    d2h = sum(t.numel() * t.element_size() for t in outs_h[0].values())
    s_in, s_cmp, s_out = (torch.cuda.Stream(device=dev) for _ in range(3))
    ev_in, ev_cmp, ev_out = ([torch.cuda.Event() for _ in range(2)] for _ in range(3))
    used = [False, False]

    def e2e_step(i):
        b = i % 2
        sb, oh = e2e_sets[b], outs_h[b]
        if used[b]:
            s_in.wait_event(ev_cmp[b])  # the compute two steps back has read these inputs
        with torch.cuda.stream(s_in):
            for n in ("q", "k", "v", "do"):
                sb[n].copy_(pinned[n], non_blocking=True)
        ev_in[b].record(s_in)
        s_cmp.wait_event(ev_in[b])
        if used[b]:
            s_cmp.wait_event(ev_out[b])  # the outputs two steps back have been copied out
        if fused:
            ca.attn_fwd(sb["q"], sb["k"], sb["v"], sb["o"], sb["lse"], scale, causal, s_cmp)
            ca.attn_bwd_preprocess(sb["o"], sb["do"], sb["lse"], sb["ws"], s_cmp)
            ca.attn_bwd_dkdv_dq(sb["q"], sb["k"], sb["v"], sb["do"], sb["dk"], sb["dv"], sb["ws"], scale, causal, s_cmp)
            ca.attn_bwd_dq_finish(sb["dq"], sb["ws"], scale, s_cmp)
        else:
            ca.attn_fwd(sb["q"], sb["k"], sb["v"], sb["o"], sb["lse"], scale, causal, s_cmp)
            ca.attn_bwd(sb["q"], sb["k"], sb["v"], sb["o"], sb["do"], sb["lse"], sb["dq"], sb["dk"], sb["dv"],
                        sb["ws"], scale, causal, s_cmp)
        ev_cmp[b].record(s_cmp)
        s_out.wait_event(ev_cmp[b])
        with torch.cuda.stream(s_out):
            for n in ("o", "lse", "dq", "dk", "dv"):
                oh[n].copy_(sb[n], non_blocking=True)
        ev_out[b].record(s_out)
        used[b] = True

    for i in range(3):
        e2e_step(i)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    t0 = time.perf_counter()
    for i in range(args.e2e_steps):
        e2e_step(i)
    torch.cuda.synchronize()
    e2e_s = max_over_ranks(time.perf_counter() - t0, dev)
    ca.check_device_error(stream)
    e2e_value = whole_job_tflops(step_flops, args.e2e_steps, world, e2e_s)
    lock.__exit__(None, None, None)

    if rank != 0:
        dist.destroy_process_group()
        return

    # ------------------------------------------------------------------ roofline
    peak_tf, peak_gbs, peak_kind = load_peaks()
    kf = {k: f for k, f in kernel_flops(wr).items() if k in KERNELS}
    top = max(kf, key=lambda k: mean_ms[k])
    achieved = kf[top] / (mean_ms[top] * 1e-3) / 1e12
    traffic = captured_traffic(wr.name, top)
    roofline = {"bound": "tensor", "kernel": f"attn_{top}", "achieved": round(achieved, 2), "peak": peak_tf,
                "unit": "TFLOP/s", "frac": round(achieved / peak_tf, 4), "traffic": traffic,
                "peak_kind": f"bf16 dense burst, {peak_kind}"}
    kernels = {}
    for k in KERNELS:
        e = {"ms": round(mean_ms[k], 5), **spread(per_kernel[k]), "share": round(mean_ms[k] / sum(mean_ms.values()), 4)}
        if k in kf:
            tf = kf[k] / (mean_ms[k] * 1e-3) / 1e12
            e.update(tflops=round(tf, 2), frac=round(tf / peak_tf, 4))
        else:
            gbs = kernel_bytes(wr)[k] / (mean_ms[k] * 1e-3) / 1e9
            e.update(gbs=round(gbs, 1), frac=round(gbs / peak_gbs, 4))
        kernels[k] = e
    fwd_tf = fwd_f * (1.0 if causal else 2.0) / (mean_ms["fwd"] * 1e-3) / 1e12
    bwd_ms = sum(mean_ms[k] for k in KERNELS if k != "fwd")
    bwd_tf = bwd_f * (1.0 if causal else 2.0) / (bwd_ms * 1e-3) / 1e12

    sust_tf, sust_kind = sustained_peak()

    line = {
        "metric": "causal attention fwd+bwd TFLOP/s (bf16) and % of GB300 dense BF16 peak",
        "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(elapsed_ms / args.steps, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": wr.name, "B": B, "H": H, "H_kv": H_kv, "T": T, "d": d, "causal": causal,
                   "parallelism": f"replicas x{world}", "l2": f"inputs rotate over {n_sets} sets ({n_sets * per_set / 2**20:.0f} MiB > L2)",
                   "launch": launch_mode, "order": args.order},
        "frac_of_peak": round(value / peak_tf, 4),
        "fwd_tflops": round(fwd_tf, 2), "bwd_tflops": round(bwd_tf, 2),
        "fwd_frac": round(fwd_tf / peak_tf, 4), "bwd_frac": round(bwd_tf / peak_tf, 4),
        "vs_sustained_peak": {"peak": sust_tf, "peak_kind": f"bf16 dense sustained, {sust_kind}",
                              "frac": round(value / sust_tf, 4), "fwd_frac": round(fwd_tf / sust_tf, 4),
                              "bwd_frac": round(bwd_tf / sust_tf, 4)},
        "kernels": kernels,
        "roofline": roofline,
        "cpu_baseline": cpu,
        "parity_receipt": receipt,
        "e2e": {"value": round(e2e_value, 3), "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "steps": args.e2e_steps},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
        "provenance": provenance(wr.seed, dev),
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main():
    args = parse()
    rank, world, local = dist_env()
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if args.block:
        if args.order != "fwd-bwd":
            raise SystemExit("--order applies to the attention line, not to --block")
        run_block(args, rank, world, local)
        return
    run_ours(args, rank, world, local)


BLOCK_STAGES = ("qkv_proj", "attn_fwd", "out_proj", "out_proj_bwd", "attn_bwd", "qkv_proj_bwd")


def block_flops(B, H, H_kv, T, d, C, causal):
    """Credited FLOPs per stage: the attention's (forward 2 B H T^2 d, backward 2.5x, causal
    halves counted as in the attention line) and 2 M N K per GEMM."""
    fwd, bwd = credited_flops(B, H, T, d)
    mul = 1.0 if causal else 2.0
    n_qkv, tok = (H + 2 * H_kv) * d, B * T
    return {"qkv_proj": 2.0 * tok * n_qkv * C, "attn_fwd": fwd * mul, "out_proj": 2.0 * tok * C * H * d,
            "out_proj_bwd": 2 * 2.0 * tok * C * H * d, "attn_bwd": bwd * mul, "qkv_proj_bwd": 2 * 2.0 * tok * n_qkv * C}


def run_block(args, rank, world, local):
    """One training step of the attention block on the workload's shapes, every stage through
    the C ABI: q, k, v = split(x W_qkv^T) with RoPE on q, k; o = attention(q, k, v); y =
    merge(o) W_o^T; then dO, dW_o from dy; dQ, dK, dV from dO; dX, dW_qkv from those."""
    import torch
    import torch.distributed as dist
    import causal_attention_gb300 as ca
    import seeded_inputs as si

    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    w = variant(si.WORKLOADS[args.workload], args)
    wr = replica(w, rank)
    B, H, T, d = wr.shape
    H_kv = args.kv_heads or H
    C = H * d
    scale, causal = wr.scale, wr.causal
    dev = torch.device("cuda", local)
    n_qkv = (H + 2 * H_kv) * d
    # seeded inputs: activations N(0, 1), weights N(0, 0.02^2) (the pages' initialisation),
    # upstream gradient N(0, sigma_do^2)
    x_bits = si.normal_bf16_bits(wr.seed, 10, (B, T, C))
    dy_bits = si.normal_bf16_bits(wr.seed, 11, (B, T, C), wr.sigma_do)
    w_qkv = to_device(si.normal_bf16_bits(wr.seed, 12, (n_qkv, C), 0.02))
    w_o = to_device(si.normal_bf16_bits(wr.seed, 13, (C, H * d), 0.02))
    tab = ca.rope_table(T, d, dev)
    n_sets = 2  # one step's tensors alone exceed L2; two sets alternate all the same

    def new_set():
        s = {"x": to_device(x_bits), "dy": to_device(dy_bits)}
        s["q"] = torch.empty((B, H, T, d), dtype=torch.bfloat16, device=dev)
        for n in ("k", "v", "dk", "dv"):
            s[n] = torch.empty((B, H_kv, T, d), dtype=torch.bfloat16, device=dev)
        for n in ("o", "do", "dq"):
            s[n] = torch.empty_like(s["q"])
        s["lse"] = torch.empty((B, H, T), dtype=torch.float32, device=dev)
        s["y"], s["dx"] = torch.empty_like(s["x"]), torch.empty_like(s["x"])
        s["dw_o"] = torch.empty((C, H * d), dtype=torch.float32, device=dev)
        s["dw_qkv"] = torch.empty((n_qkv, C), dtype=torch.float32, device=dev)
        s["ws"] = ca.new_workspace(B, H, T, d, dev, kv_heads=H_kv)
        s["wsp"] = ca.new_proj_workspace(B, T, C, H, H_kv, d, dev)
        return s
    sets = [new_set() for _ in range(n_sets)]
    stream = torch.cuda.Stream(device=dev)
    launch = {
        "qkv_proj": lambda s, st: ca.attn_qkv_proj(s["x"], w_qkv, s["q"], s["k"], s["v"], tab, st),
        "attn_fwd": lambda s, st: ca.attn_fwd(s["q"], s["k"], s["v"], s["o"], s["lse"], scale, causal, st),
        "out_proj": lambda s, st: ca.attn_out_proj(s["o"], w_o, s["y"], st),
        "out_proj_bwd": lambda s, st: ca.attn_out_proj_bwd(s["dy"], s["o"], w_o, s["do"], s["dw_o"], s["wsp"], st),
        "attn_bwd": lambda s, st: ca.attn_bwd(s["q"], s["k"], s["v"], s["o"], s["do"], s["lse"], s["dq"], s["dk"],
                                              s["dv"], s["ws"], scale, causal, st),
        "qkv_proj_bwd": lambda s, st: ca.attn_qkv_proj_bwd(s["dq"], s["dk"], s["dv"], s["x"], w_qkv, s["dx"],
                                                           s["dw_qkv"], s["wsp"], tab, st),
    }

    def step(s, ev=None, st=stream):
        for j, k in enumerate(BLOCK_STAGES):
            if ev is not None:
                ev[j].record(st)
            launch[k](s, st)
        if ev is not None:
            ev[len(BLOCK_STAGES)].record(st)

    for i in range(max(3, args.warmup)):
        step(sets[i % n_sets])
    ca.check_device_error(stream)
    nvml = NvmlClockSampler(dev) if rank == 0 else None
    sampler = ClockSampler(local) if rank == 0 and not (nvml and nvml.ok) else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    if nvml:
        nvml.start()
    elapsed_ms, evs, launch_mode = timed_steps(args, step, sets, len(BLOCK_STAGES) + 1, stream)
    clocks = nvml.stop() if nvml else None
    if world > 1:
        dist.barrier()
    if sampler:
        clocks = sampler.stop()
    ca.check_device_error(stream)
    elapsed_ms = max_over_ranks(elapsed_ms, dev)
    per_stage = {k: [ev[j].elapsed_time(ev[j + 1]) for ev in evs] for j, k in enumerate(BLOCK_STAGES)}
    mean_ms = {k: statistics.fmean(v) for k, v in per_stage.items()}
    flops = block_flops(B, H, H_kv, T, d, C, causal)
    step_flops = sum(flops.values())
    value = whole_job_tflops(step_flops, args.steps, world, elapsed_ms * 1e-3)

    # e2e: host buffers through the public API, every step copying x and dy in from pinned
    # memory and y, dx, dW_qkv, dW_o out; pipelined as a caller would run it: the two
    # device buffer sets alternate over three streams (copies in, compute, copies out), so
    # one step's copies overlap its neighbours' compute
    x_h = torch.from_numpy(x_bits.view("int16")).view(torch.bfloat16).pin_memory()
    dy_h = torch.from_numpy(dy_bits.view("int16")).view(torch.bfloat16).pin_memory()
    outs_h = [{n: torch.empty(sets[0][n].shape, dtype=sets[0][n].dtype).pin_memory()
               for n in ("y", "dx", "dw_qkv", "dw_o")} for _ in range(n_sets)]
    h2d = 2 * x_h.numel() * 2
    d2h = sum(t.numel() * t.element_size() for t in outs_h[0].values())
    s_in, s_cmp, s_out = (torch.cuda.Stream(device=dev) for _ in range(3))
    ev_in, ev_cmp, ev_out = ([torch.cuda.Event() for _ in range(n_sets)] for _ in range(3))
    used = [False] * n_sets

    def e2e_step(i):
        b = i % n_sets
        s, oh = sets[b], outs_h[b]
        if used[b]:
            s_in.wait_event(ev_cmp[b])  # the compute two steps back has read these inputs
        with torch.cuda.stream(s_in):
            s["x"].copy_(x_h, non_blocking=True)
            s["dy"].copy_(dy_h, non_blocking=True)
        ev_in[b].record(s_in)
        s_cmp.wait_event(ev_in[b])
        if used[b]:
            s_cmp.wait_event(ev_out[b])  # the outputs two steps back have been copied out
        step(s, None, s_cmp)
        ev_cmp[b].record(s_cmp)
        s_out.wait_event(ev_cmp[b])
        with torch.cuda.stream(s_out):
            for n, t in oh.items():
                t.copy_(s[n], non_blocking=True)
        ev_out[b].record(s_out)
        used[b] = True
    for i in range(3):
        e2e_step(i)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    t0 = time.perf_counter()
    for i in range(args.e2e_steps):
        e2e_step(i)
    torch.cuda.synchronize()
    e2e_s = max_over_ranks(time.perf_counter() - t0, dev)
    ca.check_device_error(stream)
    if rank != 0:
        dist.destroy_process_group()
        return

    peak_tf, _, peak_kind = load_peaks()
    stages = {k: {"ms": round(mean_ms[k], 5), **spread(per_stage[k]), "share": round(mean_ms[k] / sum(mean_ms.values()), 4),
                  "tflops": round(flops[k] / (mean_ms[k] * 1e-3) / 1e12, 2)} for k in BLOCK_STAGES}
    top = max(mean_ms, key=mean_ms.get)
    achieved = flops[top] / (mean_ms[top] * 1e-3) / 1e12
    # kernel launches per step: qkv 1; attention fwd 1; out 1; out bwd 2 (+1 split-K sum);
    # attention bwd 2 (d <= 64) or 3 (+1 split dK/dV sum); qkv bwd 1 rotation (dQ and dK) + 2 (+1)
    # (the projections' tn products take B * ceil(T / 64) K-steps of 64 tokens)
    k_tok = B * ((T + 63) // 64) * 64
    n_red_o = int(ca.attn_gemm_workspace_size(C, H * d, k_tok, "tn") > 0)
    n_red_q = int(ca.attn_gemm_workspace_size(n_qkv, C, k_tok, "tn") > 0)
    split_kv = H_kv != H and ca.attn_bwd_gqa_workspace_size(B, H, H_kv, T, d) > ca.attn_bwd_workspace_size(B, H, T, d)
    launches = 1 + 1 + 1 + 2 + n_red_o + (2 if d <= 64 else 3) + int(split_kv) + 1 + 2 + n_red_q
    line = {
        "metric": "attention block training step TFLOP/s (bf16): QKV projection + RoPE, causal attention, "
                  "output projection, forward and backward",
        "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(elapsed_ms / args.steps, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{wr.name}_block", "B": B, "H": H, "H_kv": H_kv, "T": T, "d": d, "C": C,
                   "causal": causal, "rope": True, "parallelism": f"replicas x{world}",
                   "l2": f"one step's tensors exceed L2; {n_sets} sets alternate", "launch": launch_mode},
        "frac_of_peak": round(value / peak_tf, 4),
        "stages": stages,
        "roofline": {"bound": "tensor", "kernel": top, "achieved": round(achieved, 2), "peak": peak_tf,
                     "unit": "TFLOP/s", "frac": round(achieved / peak_tf, 4), "traffic": None,
                     "peak_kind": f"bf16 dense burst, {peak_kind}"},
        "cpu_baseline": None,
        "e2e": {"value": round(whole_job_tflops(step_flops, args.e2e_steps, world, e2e_s), 3), "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": args.e2e_steps},
        "gpu_launches": launches * args.steps,
        "clocks": clocks,
        "provenance": provenance(wr.seed, dev),
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
