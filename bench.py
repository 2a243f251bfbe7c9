#!/usr/bin/env python
"""Attention TFLOP/s of the fused causal GQA forward + backward on GB300.

One step = the whole hot path over one batch of synthetic input:
fa_fwd, then the three backward stages (fa_bwd_preprocess, fa_bwd_dkdv,
fa_bwd_dq), all through the C ABI on one stream, with CUDA events between
the kernels so every kernel's duration is measured live.

Counted FLOPs: 4*B*H*D*pairs for the forward and 10*B*H*D*pairs for
forward+backward, pairs = T^2/2 under causal masking, T*W - W(W-1)/2 with a
window.  The headline value is forward+backward TFLOP/s of the whole job.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload ID] [--shape B,H,HKV,T]

Under torchrun (N > 1) every rank runs its own batch of the workload (weak
scaling, no data-path collective); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from flash_attention_attn_gb300.inputs import WORKLOADS, Workload, make_inputs, torch_dtype  # noqa: E402

METRIC = "attention TFLOP/s fwd and fwd+bwd (causal GQA bf16) and % of BF16 tensor peak"
DEFAULT_WORKLOAD = 5
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# NVIDIA's published dense (no 2:4 sparsity) bf16 tensor rate of one GB300:
# a third denominator, for context beside the two measured ones
NOMINAL_BF16_TFLOPS = 2250.0
L2_BYTES = 129 * 2**20
KERNELS = ("fwd", "bwd_preprocess", "bwd_dkdv", "bwd_dq", "bwd_dkdv_dq")


# ------------------------------------------------------------------ counting

def visible_pairs(w: Workload) -> float:
    """Visible (query, key) pairs per head as the metric counts them: T^2/2
    under causal masking (the metric's "halved"), T*W - W(W-1)/2 with a
    causal window W < T, and the exact count without causal masking (a
    window there only drops keys more than W-1 before the query)."""
    T, W = w.T, w.window
    if not w.causal:
        return float(T) * T - ((T - W) * (T - W + 1) / 2.0 if W and W < T else 0.0)
    if W and W < T:
        return float(T) * W - W * (W - 1) / 2.0
    return T * T / 2.0


def counted_flops(w: Workload) -> dict:
    base = w.B * w.H * w.D * visible_pairs(w)
    return {"fwd": 4.0 * base, "fwd_bwd": 10.0 * base}


def kernel_work(w: Workload, elem_bytes: int) -> dict:
    """Algorithmic work of one launch of each kernel (flops, or bytes for the
    HBM-bound preprocess): forward 2 matmuls per pair, dK/dV 4, dQ 3, the
    fused dK/dV + dQ 5 (dQ from the same dS tiles, without recomputing S and
    dP)."""
    base = w.B * w.H * w.D * visible_pairs(w)
    rows = w.B * w.H * w.T
    return {
        "fwd": ("tensor", 4.0 * base),
        "bwd_preprocess": ("hbm", 2.0 * rows * w.D * elem_bytes + 4.0 * rows),
        "bwd_dkdv": ("tensor", 8.0 * base),
        "bwd_dq": ("tensor", 6.0 * base),
        "bwd_dkdv_dq": ("tensor", 10.0 * base),
    }


def fused_backward(w: Workload) -> bool:
    """fa_bwd_dkdv_dq (dK, dV and dQ in one kernel, dQ without the recompute)
    takes 16-bit elements, head dims up to 64 and causal masking."""
    return w.dtype in ("bf16", "fp16") and w.D <= 64 and w.causal


def backward_stages(w: Workload) -> list:
    """The launches of fa_bwd, as its stage entry points."""
    return ["bwd_preprocess", "bwd_dkdv", "bwd_dq"]


def load_peaks() -> tuple[dict, str]:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            with open(path) as f:
                d = json.load(f)
            out = dict(FALLBACK_PEAKS)
            for k in out:
                if isinstance(d.get(k), (int, float)):
                    out[k] = float(d[k])
            return out, "measured"
        except Exception:
            pass
    return dict(FALLBACK_PEAKS), "fallback"


def source_sha(name: str) -> str:
    h = hashlib.sha256()
    for f in (name, "sm103_ptx.cuh", "fa_internal.h"):
        with open(os.path.join(ROOT, "flash_attention_attn_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


KERNEL_SOURCES = {"fwd": "fa_fwd_bf16.cu", "bwd_preprocess": "fa_delta.cu",
                  "bwd_dkdv": "fa_bwd_bf16.cu", "bwd_dq": "fa_bwd_bf16.cu", "bwd_dkdv_dq": "fa_bwd_fused.cu"}


def ncu_traffic(kernel: str, workload_name: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    this workload with the kernel source unchanged since; else None."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    if not os.path.exists(path):
        return None
    sha = source_sha(KERNEL_SOURCES[kernel])
    with open(path) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            parts = dict(kv.split("=", 1) for kv in line.strip().split(";") if "=" in kv)
            if parts.get("kernel") == kernel and parts.get("workload") == workload_name and parts.get("sha") == sha:
                try:
                    return float(parts["bytes_per_launch"])
                except (KeyError, ValueError):
                    return None
    return None


# -------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    _count = 0

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        ClockSampler._count += 1  # a file of its own: several samplers run in one process
        self.path = os.path.join("/tmp", f"fa_clocks_{os.getpid()}_{ClockSampler._count}.csv")

    def __enter__(self):
        self.skip = 0
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
            # nvidia-smi takes a while to start: wait for its first sample so
            # that the region is covered from its start, and drop the samples
            # taken before it
            t0 = time.time()
            while time.time() - t0 < 20.0 and self.proc.poll() is None:
                with open(self.path) as f:
                    n = sum(1 for _ in f)
                if n:
                    self.skip = n
                    break
                time.sleep(0.02)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    def summary(self) -> dict:
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        try:
            with open(self.path) as f:
                for k, line in enumerate(f):
                    if k < self.skip:
                        continue
                    cols = [c.strip() for c in line.split(",")]
                    if len(cols) < 8:
                        continue
                    try:
                        sm.append(float(cols[0]))
                        mx.append(float(cols[1]))
                    except ValueError:
                        continue
                    for n, v in zip(names, cols[4:8]):
                        if v.lower() == "active":
                            reasons.add(n)
            os.unlink(self.path)
        except OSError:
            pass
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# -------------------------------------------------------------- CPU baseline

def cpu_sample_workload(w: Workload, T: int, heads: int = 0) -> Workload:
    """One KV head and `heads` of its query heads (default: its whole group)
    of the workload over its first T positions: same recipe and value
    distributions, bounded size."""
    rep = w.H // w.HKV
    hq = heads if heads > 0 else rep
    return w.replace(B=1, H=hq, HKV=1, T=T, window=min(w.window, T) if w.window else 0)


def cpu_sample_run(wid: int, T: int, steps: int, heads: int = 0) -> dict:
    """Time the fp64 oracle (fwd + bwd) on the bounded sample; one run per step."""
    import oracle
    from flash_attention_attn_gb300.inputs import as_f64

    w = cpu_sample_workload(WORKLOADS[wid], T, heads)
    inp = make_inputs(w)
    Q, K, V, dO = (as_f64(inp[n]) for n in ("q", "k", "v", "do"))
    oracle.build()
    times = []
    for _ in range(steps):
        t0 = time.perf_counter()
        oracle.fwd(Q, K, V, w.scale, w.causal, w.window)
        oracle.bwd(Q, K, V, dO, w.scale, w.causal, w.window)
        times.append(time.perf_counter() - t0)
    return {"seconds": times, "flops": counted_flops(w)["fwd_bwd"], "T": T, "heads": w.H}


def cpu_baseline(wid: int, T: int, steps: int = 1, heads: int = 0) -> dict:
    """Run cpu_sample_run in a fresh process with OpenMP over every core we may use."""
    cores = len(os.sched_getaffinity(0))
    env = dict(os.environ, OMP_NUM_THREADS=str(cores), OMP_PROC_BIND="false")
    code = ("import json,sys; sys.path.insert(0, %r); import bench; "
            "print(json.dumps(bench.cpu_sample_run(%d, %d, %d, %d)))" % (ROOT, wid, T, steps, heads))
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=3600)
    if r.returncode != 0:
        raise RuntimeError(f"cpu baseline failed: {r.stderr[-2000:]}")
    d = json.loads(r.stdout.strip().splitlines()[-1])
    d["cores"] = cores
    return d


# ------------------------------------------------------------------ GPU arm

def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"  # gloo in the host tests
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def measure_prologue(w: Workload, dev, reps: int = 10):
    """Device time of the pre-attention prologue (QK RMS-norm + rotary,
    forward and backward) on this workload's shape: tokens = B*T, hq = H,
    hk = HKV query/key heads of the packed projection, RoPE factors of base
    10000.  HBM-bound: bytes = what each kernel must read and write."""
    import torch
    import flash_attention_attn_gb300 as fa
    if w.dtype not in ("bf16", "fp16") or w.D not in (64, 128):
        return None
    dt = torch_dtype(w.dtype)
    tokens = w.B * w.T
    gen = torch.Generator(device=dev).manual_seed(1000 + w.wid)
    qk = torch.randn((tokens, w.H + w.HKV, w.D), generator=gen, device=dev).to(dt)
    pos = torch.arange(w.T, device=dev).repeat(w.B).float()
    inv = 10000.0 ** (-torch.arange(0, w.D, 2, device=dev).float() / w.D)
    theta = pos[:, None] * inv[None, :]
    f1 = torch.repeat_interleave(torch.cos(theta), 2, dim=1).contiguous()
    f2 = torch.stack([-torch.sin(theta), torch.sin(theta)], dim=2).reshape(tokens, w.D).contiguous()
    q, k = fa.qk_norm_rope_fwd(qk, f1, f2, w.H)
    dq = torch.randn(q.shape, generator=gen, device=dev).to(dt)
    dk = torch.randn(k.shape, generator=gen, device=dev).to(dt)
    dqk = fa.qk_norm_rope_bwd(dq, dk, qk, f1, f2)
    out = {}
    elem = qk.element_size()
    fbytes = 2 * f1.numel() * 4
    # the two options need as many query as key heads: HKV of each, same
    # tokens; paired heads take factor rows twice as wide, the key offset a
    # half-width rotary part (its re-read of the previous token's key row is
    # not counted: it is the same data)
    h2 = max(2, w.HKV - (w.HKV % 2))
    qk2 = torch.randn((tokens, 2 * h2, w.D), generator=gen, device=dev).to(dt)
    f1p, f2p = torch.cat([f1, f1], dim=1).contiguous(), torch.cat([f2, f2], dim=1).contiguous()
    opt_bytes = (2 * qk2.numel()) * elem  # read qk2, write q and k
    g2 = torch.randn((tokens, h2, w.D), generator=gen, device=dev).to(dt)  # gradients of q and k
    g2p = g2.reshape(2 * tokens, h2 // 2, w.D)
    for name, fn, nbytes in (
            ("fwd", lambda: fa.qk_norm_rope_fwd(qk, f1, f2, w.H, q=q, k=k), (qk.numel() + q.numel() + k.numel()) * elem + fbytes),
            ("bwd", lambda: fa.qk_norm_rope_bwd(dq, dk, qk, f1, f2, dqk=dqk),
             (dq.numel() + dk.numel() + qk.numel() + dqk.numel()) * elem + fbytes),
            ("paired_fwd", lambda: fa.qk_norm_rope_fwd_opt(qk2, f1p, f2p, h2, 0, True, False), opt_bytes + 2 * fbytes),
            ("key_offset_fwd", lambda: fa.qk_norm_rope_fwd_opt(qk2, f1, f2, h2, w.D // 2, False, True),
             opt_bytes + fbytes),
            ("paired_bwd", lambda: fa.qk_norm_rope_bwd_opt(g2p, g2p, qk2, f1p, f2p, h2, 0, True, False),
             opt_bytes + qk2.numel() * elem + 2 * fbytes),
            ("key_offset_bwd", lambda: fa.qk_norm_rope_bwd_opt(g2, g2, qk2, f1, f2, h2, w.D // 2, False, True),
             opt_bytes + qk2.numel() * elem + fbytes)):
        for _ in range(3):
            fn()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            fn()
        e1.record()
        torch.cuda.synchronize(dev)
        ms = e0.elapsed_time(e1) / reps
        out[name] = {"ms": ms, "bytes": nbytes, "achieved_gbs": nbytes / (ms / 1e3) / 1e9}
    return out


class _Sets:
    """Device buffers of one workload, `n` independent sets of inputs and
    outputs: consecutive timed iterations use different sets, so that with
    enough sets the loop's working set exceeds L2 and every iteration reads
    its inputs from HBM."""

    def __init__(self, w: Workload, dev, n: int, lib, fb):
        import torch
        self.w, self.lib, self.fb = w, lib, fb
        self.dt = {"bf16": fb.FA_DTYPE_BF16, "fp16": fb.FA_DTYPE_FP16, "fp32": fb.FA_DTYPE_FP32}[w.dtype]
        inp = make_inputs(w, seed=w.wid, with_dO=w.bwd)
        op = fb.FA_OP_BWD_FUSED if fused_backward(w) else fb.FA_OP_BWD
        self.ws_bytes = fb.fa_workspace_size(op, w.B, w.T, w.H, w.HKV, w.D, self.dt)
        self.sets = []
        for _ in range(n):
            q, k, v = (inp[x].to(dev) for x in ("q", "k", "v"))
            do = inp["do"].to(dev) if w.bwd else q
            o = torch.empty_like(q)
            lse = torch.empty((w.B, w.H, w.T), dtype=torch.float32, device=dev)
            dq, dk, dv = (torch.empty_like(t) for t in (q, k, v)) if w.bwd else (q, k, v)
            ws = torch.zeros(self.ws_bytes, dtype=torch.uint8, device=dev)
            self.sets.append((q, k, v, o, lse, do, dq, dk, dv, ws))
        self.stream = torch.cuda.current_stream(dev).cuda_stream

    def stage(self, name: str, i: int):
        w, lib, fb = self.w, self.lib, self.fb
        q, k, v, o, lse, do, dq, dk, dv, ws = (t.data_ptr() for t in self.sets[i % len(self.sets)])
        a = (w.B, w.T, w.H, w.HKV, w.D)
        sc, c, win, dt, n, s = float(w.scale), int(w.causal), int(w.window), self.dt, self.ws_bytes, self.stream
        if name == "fwd":
            st = lib.fa_fwd(q, k, v, o, lse, *a, sc, c, win, dt, ws, n, s)
        elif name == "bwd_preprocess":
            st = lib.fa_bwd_preprocess(o, do, *a, dt, ws, n, s)
        elif name == "bwd_dkdv":
            st = lib.fa_bwd_dkdv(q, k, v, lse, do, dk, dv, *a, sc, c, win, dt, ws, n, s)
        elif name == "bwd_dkdv_dq":
            st = lib.fa_bwd_dkdv_dq(q, k, v, lse, do, dq, dk, dv, *a, sc, c, win, dt, ws, n, s)
        elif name == "bwd":  # the public call: Delta, dK/dV, then dQ overlapping the dK/dV tail
            st = lib.fa_bwd(q, k, v, o, lse, do, dq, dk, dv, *a, sc, c, win, dt, ws, n, s)
        else:
            st = lib.fa_bwd_dq(q, k, v, lse, do, dq, *a, sc, c, win, dt, ws, n, s)
        if st != 0:
            raise fb.FaError(st, name)

    def check(self):
        for t in self.sets:
            st, word = self.fb.fa_check_status(t[-1].data_ptr(), self.stream)
            if st != 0:
                raise RuntimeError(f"device error word {word:#x}")


def _loop_ms(fn, steps: int, stream) -> float:
    """Device time of `steps` back-to-back calls of fn(i), two CUDA events
    on the launching stream around the whole loop, per call."""
    import torch
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for i in range(steps):
        fn(i)
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps


def measure_workload(w: Workload, dev, peaks: dict, min_loop_ms: float = 200.0, repeats: int = 5,
                     kernel_loop_ms: float = 100.0) -> dict:
    """Throughput of one workload at its full size, timed the way short
    kernels need: each timed loop runs at least min_loop_ms of back-to-back
    steps (the step count comes from a calibration pass) and the step time is
    the median over `repeats` such loops; each kernel is also timed alone in
    loops of at least kernel_loop_ms (median of 3).  The loop cycles through
    enough input sets that its working set is more than twice L2; the clock
    sampler runs over the whole measurement."""
    import torch
    import flash_attention_attn_gb300 as fa
    from flash_attention_attn_gb300 import _binding as fb

    lib = fa.load()
    elem = {"bf16": 2, "fp16": 2, "fp32": 4}[w.dtype]
    set_bytes = w.B * w.T * (w.H * (2 if w.bwd else 1) + 2 * w.HKV) * w.D * elem
    n_sets = max(1, min(2048, math.ceil(2 * L2_BYTES / set_bytes)))
    sets = _Sets(w, dev, n_sets, lib, fb)
    stages = ["fwd"] + (backward_stages(w) if w.bwd else [])
    # the alternative second stage, timed alone beside the step (not part of it)
    extra = ["bwd_dkdv_dq"] if w.bwd and fused_backward(w) else []
    stream = torch.cuda.current_stream(dev)

    calls = ["fwd", "bwd"] if w.bwd else ["fwd"]  # a step is what a user runs: fa_fwd, then fa_bwd

    def step(i):
        for name in calls:
            sets.stage(name, i)

    for i in range(max(3, n_sets)):  # warm-up: every set gets a valid O, LSE and Delta
        step(i)
    torch.cuda.synchronize(dev)
    sets.check()
    est = _loop_ms(step, max(3, min(n_sets, 50)), stream)
    steps = max(n_sets, int(math.ceil(min_loop_ms / max(est, 1e-3))))
    with ClockSampler(dev.index or 0) as clocks:
        loops = [_loop_ms(step, steps, stream) for _ in range(repeats)]
        kern = {}
        for name in stages + extra:
            f = (lambda nm: (lambda i: sets.stage(nm, i)))(name)
            one = _loop_ms(f, max(3, min(n_sets, 50)), stream)
            ksteps = max(n_sets, int(math.ceil(kernel_loop_ms / max(one, 1e-3))))
            kern[name] = statistics.median(_loop_ms(f, ksteps, stream) for _ in range(3))
    sets.check()
    step_ms = statistics.median(loops)
    flops = counted_flops(w)
    work = kernel_work(w, elem)
    burst, sust = peaks["bf16_tflops"], peaks["bf16_tflops_sustained"]
    tensor = w.dtype in ("bf16", "fp16")
    out = {"workload": w.name, "dtype": w.dtype, "B": w.B, "H": w.H, "HKV": w.HKV, "T": w.T, "head_dim": w.D,
           "window": w.window, "causal": w.causal, "steps_per_loop": steps, "loops": repeats,
           "loop_ms": [ms * steps for ms in loops], "step_ms": step_ms, "step": " + ".join(f"fa_{c}" for c in calls),
           "l2": (f"{n_sets} rotating input sets, {n_sets * set_bytes / 2**20:.0f} MiB of inputs per pass "
                  f"(more than twice L2), no flush"),
           "clocks": clocks.summary()}
    fwd_ms = kern["fwd"]  # the forward alone, in loops of its own
    out["fwd_ms"] = fwd_ms
    out["fwd_tflops"] = flops["fwd"] / (fwd_ms / 1e3) / 1e12
    if w.bwd:
        out["fwd_bwd_ms"] = step_ms
        out["fwd_bwd_tflops"] = flops["fwd_bwd"] / (step_ms / 1e3) / 1e12
    if tensor:
        out["fwd_pct_of_burst"] = 100.0 * out["fwd_tflops"] / burst
        out["fwd_pct_of_sustained"] = 100.0 * out["fwd_tflops"] / sust
        if w.bwd:
            out["fwd_bwd_pct_of_burst"] = 100.0 * out["fwd_bwd_tflops"] / burst
            out["fwd_bwd_pct_of_sustained"] = 100.0 * out["fwd_bwd_tflops"] / sust
            out["fwd_bwd_pct_of_nominal"] = 100.0 * out["fwd_bwd_tflops"] / NOMINAL_BF16_TFLOPS
        out["fwd_pct_of_nominal"] = 100.0 * out["fwd_tflops"] / NOMINAL_BF16_TFLOPS
    else:
        out["note"] = "fp32 CUDA-core kernels (correctness workload); no tensor-peak target"
    out["kernels"] = {}
    for name in stages + extra:
        bound, amount = work[name]
        ms = kern[name]
        if bound == "tensor":
            ach = amount / (ms / 1e3) / 1e12
            k = {"ms": ms, "achieved": ach, "unit": "TFLOP/s"}
            if tensor:
                k.update(frac_of_burst=ach / burst, frac_of_sustained=ach / sust)
        else:
            ach = amount / (ms / 1e3) / 1e9
            k = {"ms": ms, "achieved": ach, "unit": "GB/s", "frac": ach / peaks["hbm_gbs"]}
        out["kernels"][name] = k
    if extra:
        out["kernels"]["bwd_dkdv_dq"]["note"] = (
            "fa_bwd_dkdv_dq: dK, dV and dQ in one kernel, dQ without recomputing S and dP; not part of the step "
            "(fa_bwd runs bwd_dkdv + bwd_dq, which are faster here)")
    del sets
    torch.cuda.empty_cache()
    return out


def run_ours(args, w: Workload, world: int, rank: int, local: int) -> dict:
    import torch
    import flash_attention_attn_gb300 as fa
    from flash_attention_attn_gb300 import _binding as fb

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    fa.load()
    inp = make_inputs(w, seed=w.wid + 1000 * rank)
    q, k, v, do = (inp[n].to(dev) for n in ("q", "k", "v", "do"))
    dt = fb.FA_DTYPE_BF16 if w.dtype == "bf16" else fb.FA_DTYPE_FP32
    B, T, H, HKV, D = w.B, w.T, w.H, w.HKV, w.D
    o = torch.empty_like(q)
    lse = torch.empty((B, H, T), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    fused = bool(args.fused_bwd) and fused_backward(w)
    if args.fused_bwd and not fused:
        raise SystemExit("--fused-bwd needs a causal 16-bit workload with a head dim of at most 64")
    ws_bytes = fb.fa_workspace_size(fb.FA_OP_BWD_FUSED if fused else fb.FA_OP_BWD, B, T, H, HKV, D, dt)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    s = stream.cuda_stream
    lib = fb.load()
    sc, causal, win = float(w.scale), int(w.causal), int(w.window)
    P = [t.data_ptr() for t in (q, k, v, o, lse, do, dq, dk, dv)]
    wsp = ws.data_ptr()

    def check(st, what):
        if st != 0:
            raise fb.FaError(st, what)

    def k_fwd():
        check(lib.fa_fwd(P[0], P[1], P[2], P[3], P[4], B, T, H, HKV, D, sc, causal, win, dt, wsp, ws_bytes, s), "fa_fwd")

    def k_pre():
        check(lib.fa_bwd_preprocess(P[3], P[5], B, T, H, HKV, D, dt, wsp, ws_bytes, s), "fa_bwd_preprocess")

    def k_dkdv():
        check(lib.fa_bwd_dkdv(P[0], P[1], P[2], P[4], P[5], P[7], P[8], B, T, H, HKV, D, sc, causal, win, dt,
                              wsp, ws_bytes, s), "fa_bwd_dkdv")

    def k_dq():
        check(lib.fa_bwd_dq(P[0], P[1], P[2], P[4], P[5], P[6], B, T, H, HKV, D, sc, causal, win, dt,
                            wsp, ws_bytes, s), "fa_bwd_dq")

    def k_fused():
        check(lib.fa_bwd_dkdv_dq(P[0], P[1], P[2], P[4], P[5], P[6], P[7], P[8], B, T, H, HKV, D, sc, causal, win,
                                 dt, wsp, ws_bytes, s), "fa_bwd_dkdv_dq")

    # the step: fa_fwd and fa_bwd's three stages, or with --fused-bwd the
    # opt-in second stage that forms dQ without recomputing S and dP
    kernels = ["fwd"] + (["bwd_preprocess", "bwd_dkdv_dq"] if fused else backward_stages(w))
    by_name = {"fwd": k_fwd, "bwd_preprocess": k_pre, "bwd_dkdv": k_dkdv, "bwd_dq": k_dq, "bwd_dkdv_dq": k_fused}
    stages = tuple(by_name[n] for n in kernels)
    in_bytes = sum(t.numel() * t.element_size() for t in (q, k, v, do))
    flush = None if in_bytes > L2_BYTES else torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev)

    for _ in range(args.warmup):
        for f in stages:
            f()
    torch.cuda.synchronize(dev)
    st, word = fb.fa_check_status(wsp, s)
    if st != 0:
        raise RuntimeError(f"warm-up reported device error word {word:#x}")

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(stages) + 1)] for _ in range(K)]
    barrier(world)
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clocks:
        for i in range(K):
            if flush is not None:
                flush.zero_()  # evict the inputs from L2 between steps (outside the events)
            ev[i][0].record(stream)
            for j, f in enumerate(stages):
                f()
                ev[i][j + 1].record(stream)
        torch.cuda.synchronize(dev)
        barrier(world)
    clock_summary = clocks.summary()
    st, word = fb.fa_check_status(wsp, s)
    if st != 0:
        raise RuntimeError(f"timed region reported device error word {word:#x}")

    per_kernel = {name: [ev[i][j].elapsed_time(ev[i][j + 1]) for i in range(K)] for j, name in enumerate(kernels)}
    step_ms = [ev[i][0].elapsed_time(ev[i][len(stages)]) for i in range(K)]
    total_s = max_over_ranks(sum(step_ms) / 1e3, world)

    # e2e: host buffers in pinned memory, every step's copies inside the timed
    # region.  Two device buffer sets and a copy stream: the inputs of step
    # i + 1 go up and the results of step i - 1 come down while step i
    # computes, the way a training or serving loop feeds the GPU.  The serial
    # form (copy in, compute, copy out, one after the other) is reported too.
    e2e = None
    if not args.no_e2e:
        h_in = [t.cpu().pin_memory() for t in (inp["q"], inp["k"], inp["v"], inp["do"])]
        outs0 = (o, lse, dq, dk, dv)
        h_out = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outs0]
        h2d = sum(t.numel() * t.element_size() for t in h_in)
        d2h = sum(t.numel() * t.element_size() for t in h_out)
        sets = [(q, k, v, do) + outs0,
                tuple(torch.empty_like(t) for t in (q, k, v, do)) + tuple(torch.empty_like(t) for t in outs0)]

        def run_set(bs):  # the public calls: fa_fwd, then fa_bwd
            qq, kk, vv, dd, oo, ll, gq, gk, gv = (t.data_ptr() for t in bs)
            check(lib.fa_fwd(qq, kk, vv, oo, ll, B, T, H, HKV, D, sc, causal, win, dt, wsp, ws_bytes, s), "fa_fwd")
            if fused:
                check(lib.fa_bwd_preprocess(oo, dd, B, T, H, HKV, D, dt, wsp, ws_bytes, s), "fa_bwd_preprocess")
                check(lib.fa_bwd_dkdv_dq(qq, kk, vv, ll, dd, gq, gk, gv, B, T, H, HKV, D, sc, causal, win, dt, wsp,
                                         ws_bytes, s), "fa_bwd_dkdv_dq")
                return
            check(lib.fa_bwd(qq, kk, vv, oo, ll, dd, gq, gk, gv, B, T, H, HKV, D, sc, causal, win, dt, wsp,
                             ws_bytes, s), "fa_bwd")

        def timed(pipelined, steps):
            # Uploads and downloads run on streams of their own, so that the two
            # directions of the host link work at the same time.  Set i % 2
            # serves step i; its inputs may be overwritten once the compute of
            # step i - 2 is done, its outputs once their download is done.
            cs, ds = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
            done = [None, None]     # compute of the set's last step finished
            fetched = [None, None]  # outputs of the set's last step copied out
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            barrier(world)
            torch.cuda.synchronize(dev)
            e0.record(stream)

            def mark(st):
                ev = torch.cuda.Event()
                ev.record(st)
                return ev

            def upload(i, after):  # inputs of step i into set i % 2, on the upload stream
                cs.wait_event(after)
                if done[i % 2] is not None:
                    cs.wait_event(done[i % 2])
                with torch.cuda.stream(cs):
                    for hsrc, ddst in zip(h_in, sets[i % 2][:4]):
                        ddst.copy_(hsrc, non_blocking=True)
                return mark(cs)

            def compute(i, ready):
                stream.wait_event(ready)
                if fetched[i % 2] is not None:
                    stream.wait_event(fetched[i % 2])
                run_set(sets[i % 2])
                done[i % 2] = mark(stream)

            def download(i):  # results of step i, once its compute is done
                ds.wait_event(done[i % 2])
                with torch.cuda.stream(ds):
                    for dsrc, hdst in zip(sets[i % 2][4:], h_out):
                        hdst.copy_(dsrc, non_blocking=True)
                fetched[i % 2] = mark(ds)

            if pipelined:
                # step i + 1's inputs go up and step i - 1's results come down
                # while step i computes
                ready = upload(0, e0)
                for i in range(steps):
                    nxt = upload(i + 1, e0) if i + 1 < steps else None
                    compute(i, ready)
                    download(i)
                    ready = nxt
            else:
                # copy in, compute, copy out, one after the other
                after = e0
                for i in range(steps):
                    compute(i, upload(i, after))
                    download(i)
                    after = fetched[i % 2]
            stream.wait_event(fetched[(steps - 1) % 2])
            e1.record(stream)
            torch.cuda.synchronize(dev)
            barrier(world)
            return max_over_ranks(e0.elapsed_time(e1) / 1e3, world)

        e2e_steps = max(3, min(K, 10))  # the pipeline fills and drains once per measurement
        timed(True, 2)  # warm the copy path and the second buffer set
        e2e_s = timed(True, e2e_steps)
        serial_s = timed(False, e2e_steps)
        st, word = fb.fa_check_status(wsp, s)
        if st != 0:
            raise RuntimeError(f"e2e region reported device error word {word:#x}")
        flops = world * e2e_steps * counted_flops(w)["fwd_bwd"]
        e2e = {"value": flops / e2e_s / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps,
               "ms_per_step": 1e3 * e2e_s / e2e_steps, "pipelined": True,
               "serial": {"value": flops / serial_s / 1e12, "ms_per_step": 1e3 * serial_s / e2e_steps}}

    prologue = None if args.no_prologue else measure_prologue(w, dev)
    side = None
    if not args.no_workloads and world == 1:
        peaks, _ = load_peaks()
        side = {str(i): measure_workload(WORKLOADS[i], dev, peaks) for i in sorted(WORKLOADS) if i != w.wid}
    return {"workloads": side, "kernels": kernels, "per_kernel_ms": per_kernel, "step_ms": step_ms, "total_s": total_s, "clocks": clock_summary,
            "e2e": e2e, "elem_bytes": q.element_size(), "prologue": prologue}


def workload_from_args(args) -> Workload:
    w = WORKLOADS[args.workload]
    if args.shape:
        B, H, HKV, T = (int(x) for x in args.shape.split(","))
        w = w.replace(B=B, H=H, HKV=HKV, T=T, name=f"{w.name} [reduced to B{B} H{H}/{HKV} T{T}]")
    return w


def config_of(w: Workload, l2_note: str) -> dict:
    return {"workload": w.name, "B": w.B, "H": w.H, "HKV": w.HKV, "T": w.T, "head_dim": w.D,
            "window": w.window, "causal": w.causal, "scale": w.scale, "input_recipe": w.recipe,
            "flops_per_step_fwd_bwd": counted_flops(w)["fwd_bwd"],
            "flop_count": "fwd 4*B*H*D*pairs, fwd+bwd 10*B*H*D*pairs; pairs = T^2/2 causal, T*W - W(W-1)/2 windowed",
            "l2": l2_note}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", type=int, default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--shape", default=None, help="B,H,HKV,T: reduced size of the same workload (profiling)")
    ap.add_argument("--cpu-T", type=int, default=16384, help="sequence prefix of the CPU-baseline sample")
    ap.add_argument("--ref-T", type=int, default=4096, help="sequence prefix per reference-arm step")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-prologue", action="store_true", help="skip the QK-norm + rotary prologue measurement")
    ap.add_argument("--no-workloads", action="store_true", help="skip the other configurations' loops")
    ap.add_argument("--fused-bwd", action="store_true",
                    help="step with the opt-in fused backward stage (causal 16-bit, head dim <= 64)")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours" and not args.shape:
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)

    w = workload_from_args(args)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))

    if args.impl == "reference":
        # the reference arm is the fp64 oracle on the host cores, rank 0 only
        if rank != 0:
            return
        s = cpu_baseline(w.wid, args.ref_T, steps=args.warmup + args.steps, heads=1)
        times = s["seconds"][args.warmup:]
        tot = sum(times)
        val = len(times) * s["flops"] / tot / 1e12
        sample = (f"fp64 oracle fwd+bwd of one query head of '{w.name}' over its first "
                  f"{args.ref_T} positions per step ({s['flops'] / 1e9:.1f} GFLOP counted)")
        line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "TFLOP/s", "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot / len(times),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "config": config_of(w, "host run; no GPU"),
                "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": s["cores"], "kind": "oracle",
                                 "sample": sample},
                "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return

    # CPU baseline first (a fresh process, before this one touches the GPU)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w.wid, args.cpu_T, steps=1)

    world, rank, local = dist_setup(args)
    r = run_ours(args, w, world, rank, local)
    if rank != 0:
        return
    import torch

    peaks, peak_src = load_peaks()
    flops = counted_flops(w)
    work = kernel_work(w, r["elem_bytes"])
    value = world * args.steps * flops["fwd_bwd"] / r["total_s"] / 1e12
    kern = {}
    for name in r["kernels"]:
        ms = statistics.mean(r["per_kernel_ms"][name])
        bound, amount = work[name]
        if bound == "tensor":
            peak = peaks["bf16_tflops"]
            achieved = amount / (ms / 1e3) / 1e12
            unit = "TFLOP/s"
        else:
            peak = peaks["hbm_gbs"]
            achieved = amount / (ms / 1e3) / 1e9
            unit = "GB/s"
        kern[name] = {"ms": ms, "bound": bound, "achieved": achieved, "unit": unit, "peak": peak,
                      "frac": achieved / peak, "work_per_launch": amount}
        if bound == "tensor":
            kern[name]["frac_of_sustained"] = achieved / peaks["bf16_tflops_sustained"]
    dom = max(r["kernels"], key=lambda n: kern[n]["ms"])
    traffic = ncu_traffic(dom, w.name)
    roof = {"bound": kern[dom]["bound"], "achieved": kern[dom]["achieved"], "peak": kern[dom]["peak"],
            "unit": kern[dom]["unit"], "frac": kern[dom]["frac"], "traffic": traffic, "kernel": dom,
            "work_per_launch": kern[dom]["work_per_launch"],
            "peak_source": f"{peak_src} ({'burst cuBLAS bf16' if kern[dom]['bound'] == 'tensor' else 'HBM copy'})"}
    if kern[dom]["bound"] == "tensor":
        roof["frac_of_sustained"] = kern[dom]["frac_of_sustained"]
    fwd_ms = statistics.mean(r["per_kernel_ms"]["fwd"])
    in_bytes = w.B * w.T * (2 * w.H + 2 * w.HKV) * w.D * r["elem_bytes"]
    l2_note = ("inputs larger than L2 (no flush)" if in_bytes > L2_BYTES
               else "L2 flushed between steps (256 MiB write, outside the events)")
    line = {
        "metric": METRIC,
        "value": value,
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": statistics.mean(r["step_ms"]),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": w.dtype,
        "data": "synthetic",
        "config": config_of(w, l2_note),
        "fwd_tflops": flops["fwd"] / (fwd_ms / 1e3) / 1e12,
        "fwd_pct_of_peak": 100.0 * flops["fwd"] / (fwd_ms / 1e3) / 1e12 / peaks["bf16_tflops"],
        "fwd_bwd_pct_of_peak": 100.0 * value / world / peaks["bf16_tflops"],
        "fwd_pct_of_sustained": 100.0 * flops["fwd"] / (fwd_ms / 1e3) / 1e12 / peaks["bf16_tflops_sustained"],
        "fwd_bwd_pct_of_sustained": 100.0 * value / world / peaks["bf16_tflops_sustained"],
        "fwd_pct_of_nominal": 100.0 * flops["fwd"] / (fwd_ms / 1e3) / 1e12 / NOMINAL_BF16_TFLOPS,
        "fwd_bwd_pct_of_nominal": 100.0 * value / world / NOMINAL_BF16_TFLOPS,
        "fwd_bwd_tflops_x14": 14.0 / 10.0 * value,
        # the other reading of "10*B*H*T^2*D": FlashAttention's count for the
        # backward alone, over the three backward kernels' time
        "bwd_only_tflops_x10": flops["fwd_bwd"] / (sum(statistics.mean(r["per_kernel_ms"][n])
                                                     for n in r["kernels"] if n != "fwd") / 1e3) / 1e12,
        "peak_bf16_tflops": peaks["bf16_tflops"],
        "peak_bf16_tflops_sustained": peaks["bf16_tflops_sustained"],
        "peak_nominal_bf16_tflops": NOMINAL_BF16_TFLOPS,
        "peak_source": f"{peak_src}: pct_of_peak against the burst cuBLAS bf16 rate, _of_sustained against the "
                       "seconds-long loop under the power cap, _of_nominal against NVIDIA's published dense rate",
        "roofline": roof,
        "kernels": kern,
        "backward": ("fa_bwd_preprocess + fa_bwd_dkdv_dq (opt-in fused stage)" if "bwd_dkdv_dq" in r["kernels"]
                     else "fa_bwd: fa_bwd_preprocess + fa_bwd_dkdv + fa_bwd_dq"),
        "gpu_launches": len(r["kernels"]) * args.steps,
        "clocks": r["clocks"],
        "e2e": r["e2e"],
        "device": torch.cuda.get_device_name(0),
    }
    if r["prologue"] is not None:
        # outside the timed step: the QK-norm + rotary prologue on the same shape (HBM-bound)
        line["prologue"] = {n: dict(v, peak_gbs=peaks["hbm_gbs"], frac=v["achieved_gbs"] / peaks["hbm_gbs"])
                            for n, v in r["prologue"].items()}
    if r["workloads"]:
        # the other configurations, each in its own >= 200 ms loops (median of 5)
        line["workloads"] = r["workloads"]
        line["gpu_launches_workloads"] = "outside the timed steps; not counted in gpu_launches"
    if cpu is not None:
        t = cpu["seconds"][0]
        line["cpu_baseline"] = {
            "value": cpu["flops"] / t / 1e12, "unit": "TFLOP/s", "cores": cpu["cores"], "kind": "oracle",
            "seconds": t,
            "sample": (f"fp64 oracle fwd+bwd of one KV head and its {cpu['heads']} query heads of '{w.name}' "
                       f"over the first {cpu['T']} positions ({cpu['flops'] / 1e9:.1f} GFLOP counted)")}
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
