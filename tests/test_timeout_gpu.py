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


@pytest.mark.parametrize("ctas", [0, 1], ids=["all-sms", "1-cta"])
def test_stalled_forward_times_out_and_recovers(ctas):
    from flash_attention_attn_gb300.build import build
    build()
    w = Workload(200, "timeout", "bf16", 1, 2, 2, 256, 64, 0, True, False, "normal")
    inp = make_inputs(w, seed=3, with_dO=False)
    dev = torch.device("cuda", 0)
    q, k, v = (inp[n].to(dev) for n in ("q", "k", "v"))
    fa.check_status()  # clear anything earlier tests left
    try:
        fa.fa_debug_config(200_000_000, 1)
        assert fa.fa_debug_max_ctas(ctas) == fa.FA_OK
        fa.attention_fwd(q, k, v, causal=True)
        st, word = fa.check_status()
    finally:
        fa.fa_debug_config(0, 0)
        fa.fa_debug_max_ctas(0)
    assert st == fa.FA_ERR_TIMEOUT
    assert word & 1  # FA_DEVERR_FWD_TIMEOUT
    # the context still works and the next call is correct
    o, lse = fa.attention_fwd(q, k, v, causal=True)
    st, word = fa.check_status()
    assert st == fa.FA_OK, hex(word)
    O, L = oracle.fwd(as_f64(inp["q"]), as_f64(inp["k"]), as_f64(inp["v"]), w.scale, True, 0)
    assert np.max(np.abs(o.float().cpu().numpy() - O)) <= 2e-2
    assert np.max(np.abs(lse.cpu().numpy() - L)) <= 1e-3


@pytest.mark.parametrize("ctas", [0, 3], ids=["all-sms", "3-ctas"])
@pytest.mark.parametrize("kind,bit", [(2, 2), (3, 4)], ids=["dkdv", "dq"])
def test_stalled_backward_kernel_times_out_and_recovers(kind, bit, ctas):
    """With every SM or with three CTAs (each aborting CTA still counts
    itself out of the persistent scheduler, so the work counters are zero
    again for the next call, which the oracle check below would notice)."""
    from flash_attention_attn_gb300.build import build
    build()
    w = Workload(201, "timeout-bwd", "bf16", 1, 4, 2, 300, 64, 0, True, True, "normal")
    inp = make_inputs(w, seed=4)
    dev = torch.device("cuda", 0)
    q, k, v, do = (inp[n].to(dev) for n in ("q", "k", "v", "do"))
    o, lse = fa.attention_fwd(q, k, v, causal=True)
    fa.check_status()
    try:
        fa.fa_debug_config(200_000_000, kind)
        assert fa.fa_debug_max_ctas(ctas) == fa.FA_OK
        fa.attention_bwd(q, k, v, o, lse, do, causal=True)
        st, word = fa.check_status()
    finally:
        fa.fa_debug_config(0, 0)
        fa.fa_debug_max_ctas(0)
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


def test_stalled_fused_backward_times_out_and_recovers():
    """The fused dK/dV + dQ kernel (fa_bwd_dkdv_dq) takes the dK/dV hook: its
    waits give up (the turn waits among them), only the dK/dV bit is set, and
    the next call -- its turn counters cleared again -- is correct."""
    from flash_attention_attn_gb300.build import build
    build()
    w = Workload(202, "timeout-fused", "bf16", 1, 4, 2, 300, 64, 0, True, True, "normal")
    inp = make_inputs(w, seed=5)
    dev = torch.device("cuda", 0)
    q, k, v, do = (inp[n].to(dev) for n in ("q", "k", "v", "do"))
    o, lse = fa.attention_fwd(q, k, v, causal=True)
    fa.check_status()
    n = fa.fa_workspace_size(fa.FA_OP_BWD_FUSED, w.B, w.T, w.H, w.HKV, w.D, fa.FA_DTYPE_BF16)
    ws = torch.zeros(n, dtype=torch.uint8, device=dev)
    s = torch.cuda.current_stream(dev).cuda_stream
    P = [t.data_ptr() for t in (q, k, v, o, lse, do)]
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    args = (w.B, w.T, w.H, w.HKV, w.D, w.scale, 1, 0, fa.FA_DTYPE_BF16, ws.data_ptr(), n, s)

    def run():
        assert fa.fa_bwd_preprocess(P[3], P[5], w.B, w.T, w.H, w.HKV, w.D, fa.FA_DTYPE_BF16, ws.data_ptr(), n,
                                    s) == fa.FA_OK
        assert fa.fa_bwd_dkdv_dq(P[0], P[1], P[2], P[4], P[5], dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                                 *args) == fa.FA_OK
        return fa.fa_check_status(ws.data_ptr(), s)

    try:
        fa.fa_debug_config(200_000_000, 2)
        st, word = run()
    finally:
        fa.fa_debug_config(0, 0)
    assert st == fa.FA_ERR_TIMEOUT
    assert word == 2, hex(word)
    st, word = run()
    assert st == fa.FA_OK, hex(word)
    Q, K, V, dO = (as_f64(inp[x]) for x in ("q", "k", "v", "do"))
    dQ, dK, dV, _ = oracle.bwd(Q, K, V, dO, w.scale, True, 0)
    for got, ref in ((dq, dQ), (dk, dK), (dv, dV)):
        g = got.float().cpu().numpy().astype(np.float64)
        assert np.linalg.norm(g - ref) / np.linalg.norm(ref) <= 2e-2
