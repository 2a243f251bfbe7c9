"""Seeded synthetic inputs for the attention workloads.

This module only draws random numbers: it holds none of the attention
arithmetic.  Both sides of every parity check (the CUDA path and the fp64
oracle) receive tensors made here, so they see bit-identical inputs.

Recipe (one CPU ``torch.Generator`` per workload, seed = the workload id):
draw fp32 N(0, 1) in the order Q, K, V, dO, then shape them per workload and
round to the compute dtype (bf16 or fp16 round-to-nearest-even, or keep fp32).

* ``rms_qk``: every Q and K head vector is RMS-normalised,
  x / sqrt(mean(x^2) + eps) with eps = 1.1920928955078125e-7, the QK-norm
  epsilon of the modded-nanogpt page (qkv_rope.py, `_qk_norm_rope_forward_kernel`).
* ``sharpen2``: Q and K are multiplied by 2 (score std about 4), which makes
  the softmax rows nearly one-hot.
* ``normal``: plain N(0, 1).
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch

RMS_EPS = 1.1920928955078125e-7


@dataclass(frozen=True)
class Workload:
    """Sizes and recipe of one attention workload."""

    wid: int
    name: str
    dtype: str  # "bf16", "fp16" or "fp32"
    B: int
    H: int
    HKV: int
    T: int
    D: int
    window: int
    causal: bool
    bwd: bool
    recipe: str  # "normal" | "rms_qk" | "sharpen2"

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    def replace(self, **kw) -> "Workload":
        d = dict(self.__dict__)
        d.update(kw)
        return Workload(**d)


WORKLOADS: dict[int, Workload] = {
    1: Workload(1, "causal MHA fp32 B1 H2 T128 D64", "fp32", 1, 2, 2, 128, 64, 0, True, True, "normal"),
    2: Workload(2, "causal GQA bf16 B4 H8/2 T1024 D64 (fwd only)", "bf16", 4, 8, 2, 1024, 64, 0, True, False, "normal"),
    3: Workload(3, "causal MHA bf16 B64 H8 T1024 D64", "bf16", 64, 8, 8, 1024, 64, 0, True, True, "normal"),
    4: Workload(4, "causal sliding-window GQA bf16 B2 H16/4 T8192 D128 W1024", "bf16", 2, 16, 4, 8192, 128, 1024, True, True, "rms_qk"),
    5: Workload(5, "causal long-context GQA bf16 B1 H32/8 T32768 D128", "bf16", 1, 32, 8, 32768, 128, 0, True, True, "sharpen2"),
}


def torch_dtype(name: str) -> torch.dtype:
    return {"bf16": torch.bfloat16, "fp16": torch.float16, "fp32": torch.float32}[name]


def make_inputs(w: Workload, seed: int | None = None, with_dO: bool = True) -> dict[str, torch.Tensor]:
    """CPU tensors q, k, v[, do] in the workload's dtype, [B,T,H|HKV,D] contiguous."""
    g = torch.Generator(device="cpu")
    g.manual_seed(w.wid if seed is None else seed)
    q = torch.randn((w.B, w.T, w.H, w.D), generator=g, dtype=torch.float32)
    k = torch.randn((w.B, w.T, w.HKV, w.D), generator=g, dtype=torch.float32)
    v = torch.randn((w.B, w.T, w.HKV, w.D), generator=g, dtype=torch.float32)
    do = torch.randn((w.B, w.T, w.H, w.D), generator=g, dtype=torch.float32) if with_dO else None
    if w.recipe == "rms_qk":
        q = q / torch.sqrt(q.pow(2).mean(dim=-1, keepdim=True) + RMS_EPS)
        k = k / torch.sqrt(k.pow(2).mean(dim=-1, keepdim=True) + RMS_EPS)
    elif w.recipe == "sharpen2":
        q = q * 2.0
        k = k * 2.0
    elif w.recipe != "normal":
        raise ValueError(f"unknown recipe {w.recipe}")
    dt = torch_dtype(w.dtype)
    out = {"q": q.to(dt).contiguous(), "k": k.to(dt).contiguous(), "v": v.to(dt).contiguous()}
    if with_dO:
        out["do"] = do.to(dt).contiguous()
    return out


def make_cross_inputs(dtype: str, B: int, H: int, HKV: int, Tq: int, Tk: int, D: int,
                      seed: int) -> dict[str, torch.Tensor]:
    """Cross-attention inputs: q, do [B,Tq,H,D] and k, v [B,Tk,HKV,D], iid
    N(0, 1) drawn in the order q, k, v, do, then cast to `dtype`."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    shapes = {"q": (B, Tq, H, D), "k": (B, Tk, HKV, D), "v": (B, Tk, HKV, D), "do": (B, Tq, H, D)}
    dt = torch_dtype(dtype)
    return {n: torch.randn(sh, generator=g, dtype=torch.float32).to(dt).contiguous() for n, sh in shapes.items()}


def as_f64(t: torch.Tensor):
    """Exact widening of a CPU tensor to a float64 numpy array."""
    return t.detach().to("cpu").to(torch.float64).numpy()
