"""Bounded waits: a kernel whose pipeline wait runs out of budget reports it
through the device error word and leaves the context usable.

The test hook makes the next launch of one kernel (the 16-bit forward, dK/dV
or dQ) withhold its first tile loads (a barrier that nothing completes), with
a 0.2 s wait budget.  No fault, trap or unbounded spin is involved: the
kernel's own timer ends every wait.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import flash_attention_attn_gb300 as fa
from flash_attention_attn_gb300.inputs import Workload, as_f64, make_inputs

pytestmark = pytest.mark.gpu


def test_stalled_forward_times_out_and_recovers():
    from flash_attention_attn_gb300.build import build
    build()
    w = Workload(200, "timeout", "bf16", 1, 2, 2, 256, 64, 0, True, False, "normal")
    inp = make_inputs(w, seed=3, with_dO=False)
    dev = torch.device("cuda", 0)
    q, k, v = (inp[n].to(dev) for n in ("q", "k", "v"))
    fa.check_status()  # clear anything earlier tests left
    try:
        fa.fa_debug_config(200_000_000, 1)
        fa.attention_fwd(q, k, v, causal=True)
        st, word = fa.check_status()
    finally:
        fa.fa_debug_config(0, 0)
    assert st == fa.FA_ERR_TIMEOUT
    assert word & 1  # FA_DEVERR_FWD_TIMEOUT
    # the context still works and the next call is correct
    o, lse = fa.attention_fwd(q, k, v, causal=True)
    st, word = fa.check_status()
    assert st == fa.FA_OK, hex(word)
    O, L = oracle.fwd(as_f64(inp["q"]), as_f64(inp["k"]), as_f64(inp["v"]), w.scale, True, 0)
    assert np.max(np.abs(o.float().cpu().numpy() - O)) <= 2e-2
    assert np.max(np.abs(lse.cpu().numpy() - L)) <= 1e-3


@pytest.mark.parametrize("kind,bit,D", [(2, 2, 128), (3, 4, 128), (2, 2, 64)], ids=["dkdv", "dq", "fused"])
def test_stalled_backward_kernel_times_out_and_recovers(kind, bit, D):
    """The dK/dV kernel and the dQ kernel (head dim 128), and the fused
    dK/dV + dQ kernel (head dim 64, which takes the dK/dV hook): the stalled
    kernel gives up, reports only its own bit, and the next backward -- the
    fused one with its turn counters reset -- is correct."""
    from flash_attention_attn_gb300.build import build
    build()
    w = Workload(201, "timeout-bwd", "bf16", 1, 4, 2, 300, D, 0, True, True, "normal")
    inp = make_inputs(w, seed=4)
    dev = torch.device("cuda", 0)
    q, k, v, do = (inp[n].to(dev) for n in ("q", "k", "v", "do"))
    o, lse = fa.attention_fwd(q, k, v, causal=True)
    fa.check_status()
    try:
        fa.fa_debug_config(200_000_000, kind)
        fa.attention_bwd(q, k, v, o, lse, do, causal=True)
        st, word = fa.check_status()
    finally:
        fa.fa_debug_config(0, 0)
    assert st == fa.FA_ERR_TIMEOUT
    assert word & bit and not word & ~bit & 7, hex(word)  # only the stalled kernel reports
    # the context still works and the next backward is correct
    dq, dk, dv = fa.attention_bwd(q, k, v, o, lse, do, causal=True)
    st, word = fa.check_status()
    assert st == fa.FA_OK, hex(word)
    Q, K, V, dO = (as_f64(inp[n]) for n in ("q", "k", "v", "do"))
    dQ, dK, dV, _ = oracle.bwd(Q, K, V, dO, w.scale, True, 0)
    for got, ref in ((dq, dQ), (dk, dK), (dv, dV)):
        g = got.float().cpu().numpy().astype(np.float64)
        assert np.linalg.norm(g - ref) / np.linalg.norm(ref) <= 2e-2


def test_stall_hook_rejects_unknown_kinds():
    assert fa.fa_debug_config(0, 4) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_debug_config(0, -1) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_debug_config(0, 0) == fa.FA_OK
