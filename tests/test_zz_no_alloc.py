"""fa_bwd_static_scratch: the backward for callers that cannot allocate.

Some callers may not call cudaMalloc where they run the backward (inside
another allocator's callback, in a plugin whose host owns all device memory,
while a graph is being built), so they cannot provide fa_bwd's workspace.
This entry point keeps that scratch in a static device array inside the
library.  The tests call it through the C ABI several times in a row, each
call reusing the array as the previous one left it:

* with a different dO each time and then a smaller shape, so that Delta or
  an error word left over from an earlier call would show;
* each result bitwise equal to fa_bwd's on the same inputs (the backward
  is deterministic: same kernels, fixed order, no atomics), and the first
  also against the fp64 oracle at the bf16 tolerance of the other tests
  (relative Frobenius 2e-2);
* one call with a dK/dV wait made to run out of budget (the library's test
  hook withholds that kernel's first loads; its own 0.2 s timer ends the
  wait): the caller's error word gets only the dK/dV bit, and the next call
  reports 0 and is exact again;
* shapes past the array's capacity are refused before anything runs.
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

import oracle
import flash_attention_attn_gb300 as fa
from flash_attention_attn_gb300.inputs import Workload, as_f64, make_inputs

pytestmark = pytest.mark.gpu

MAX_ROWS = 4 * 1024 * 1024  # FA_STATIC_SCRATCH_MAX_ROWS in include/fa.h
DKDV_BIT = 2                # FA_DEVERR_DKDV_TIMEOUT


def _entry():
    from flash_attention_attn_gb300.build import build
    build()
    f = fa.load().fa_bwd_static_scratch
    vp, i = ctypes.c_void_p, ctypes.c_int
    f.argtypes = [vp] * 9 + [i] * 5 + [ctypes.c_float, i, i, i, vp, vp]
    f.restype = i
    return f


def _rel_fro(got, ref):
    g = got.float().cpu().numpy().astype(np.float64)
    return float(np.linalg.norm(g - ref) / np.linalg.norm(ref))


class _Case:
    """Inputs of one shape on the GPU, with the forward already run."""

    def __init__(self, w: Workload, seed: int):
        self.w = w
        self.inp = make_inputs(w, seed=seed)
        dev = torch.device("cuda", 0)
        self.q, self.k, self.v, self.do = (self.inp[n].to(dev) for n in ("q", "k", "v", "do"))
        self.o, self.lse = fa.attention_fwd(self.q, self.k, self.v, scale=w.scale, causal=w.causal,
                                            window=w.window)

    def with_do(self, seed: int):
        """The same Q, K, V, O, LSE with another upstream gradient dO."""
        g = torch.Generator().manual_seed(seed)
        self.do = torch.randn(self.do.shape, generator=g).to(self.do.dtype).to(self.do.device)
        return self

    def reference(self):
        w = self.w
        return fa.attention_bwd(self.q, self.k, self.v, self.o, self.lse, self.do, scale=w.scale,
                                causal=w.causal, window=w.window)

    def static(self, f, err):
        w = self.w
        dq, dk, dv = torch.empty_like(self.q), torch.empty_like(self.k), torch.empty_like(self.v)
        stream = torch.cuda.current_stream(self.q.device).cuda_stream
        st = f(self.q.data_ptr(), self.k.data_ptr(), self.v.data_ptr(), self.o.data_ptr(), self.lse.data_ptr(),
               self.do.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), w.B, w.T, w.H, w.HKV, w.D,
               w.scale, int(w.causal), w.window, fa.FA_DTYPE_BF16, err.data_ptr(), stream)
        assert st == fa.FA_OK, fa.fa_status_string(st)
        torch.cuda.synchronize(self.q.device)
        return dq, dk, dv


def _assert_same(got, want):
    for name, a, b in zip(("dQ", "dK", "dV"), got, want):
        assert torch.equal(a, b), f"{name} differs from fa_bwd's"


def test_static_scratch_backward_equals_fa_bwd_on_consecutive_calls():
    f = _entry()
    dev = torch.device("cuda", 0)
    err = torch.full((1,), 7, dtype=torch.int32, device=dev)  # the call must overwrite it
    big = _Case(Workload(300, "no-alloc", "bf16", 2, 4, 2, 333, 128, 0, True, True, "normal"), seed=300)

    # 1: against fa_bwd (bitwise) and against the oracle
    got = big.static(f, err)
    assert int(err.item()) == 0
    _assert_same(got, big.reference())
    Q, K, V, dO = (as_f64(big.inp[n]) for n in ("q", "k", "v", "do"))
    dQ, dK, dV, _ = oracle.bwd(Q, K, V, dO, big.w.scale, True, 0)
    for name, g, r in zip(("dQ", "dK", "dV"), got, (dQ, dK, dV)):
        assert _rel_fro(g, r) <= 2e-2, name

    # 2: another dO, so a stale Delta from call 1 would change the result
    big.with_do(301)
    err.fill_(7)
    got = big.static(f, err)
    assert int(err.item()) == 0
    _assert_same(got, big.reference())

    # 3: a smaller shape with a window (fewer Delta rows than the array holds
    # from call 2)
    small = _Case(Workload(302, "no-alloc-small", "bf16", 1, 2, 1, 200, 64, 50, True, True, "normal"), seed=302)
    err.fill_(7)
    got = small.static(f, err)
    assert int(err.item()) == 0
    _assert_same(got, small.reference())


def test_static_scratch_reports_a_timeout_then_recovers():
    f = _entry()
    dev = torch.device("cuda", 0)
    case = _Case(Workload(303, "no-alloc-timeout", "bf16", 1, 4, 2, 300, 64, 0, True, True, "normal"), seed=303)
    fa.check_status()  # clear anything earlier tests left in the default workspace
    err = torch.zeros((1,), dtype=torch.int32, device=dev)
    try:
        fa.fa_debug_config(200_000_000, 2)  # the next dK/dV launch withholds its first loads
        case.static(f, err)
    finally:
        fa.fa_debug_config(0, 0)
    assert int(err.item()) == DKDV_BIT, hex(int(err.item()))
    # the error word inside the array is cleared by the next call
    err.fill_(7)
    got = case.static(f, err)
    assert int(err.item()) == 0
    _assert_same(got, case.reference())


def test_static_scratch_rejects_shapes_beyond_its_capacity():
    f = _entry()
    fake = 0x10000  # never dereferenced: the size check comes first
    T = MAX_ROWS // 8 + 1
    st = f(*([fake] * 9), 1, T, 8, 8, 128, 0.088, 1, 0, fa.FA_DTYPE_BF16, None, None)
    assert st == fa.FA_ERR_WORKSPACE


def test_static_scratch_rejects_bad_pointers_before_launching():
    f = _entry()
    dev = torch.device("cuda", 0)
    q = torch.zeros((1, 64, 2, 64), dtype=torch.bfloat16, device=dev)
    lse = torch.zeros((1, 2, 64), dtype=torch.float32, device=dev)
    ptrs = [q.data_ptr()] * 9
    ptrs[4] = lse.data_ptr()
    ptrs[6] = q.data_ptr() + 2  # misaligned dQ
    st = f(*ptrs, 1, 64, 2, 2, 64, 0.125, 1, 0, fa.FA_DTYPE_BF16, None, None)
    assert st == fa.FA_ERR_INVALID_ARG
