"""fa_bwd_static_scratch: the backward for callers that cannot allocate.

Some callers may not call cudaMalloc where they run the backward (inside
another allocator's callback, in a plugin whose host owns all device memory,
while a graph is being built), so they cannot provide fa_bwd's workspace.
This entry point keeps that scratch in a static device array inside the
library.  The test calls it through the C ABI twice in a row (the second call
reuses the array as the first left it) and checks each result against
fa_bwd's within the parity tolerance of the other tests (relative Frobenius
2e-2 for bf16), plus the size limit.
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

import flash_attention_attn_gb300 as fa
from flash_attention_attn_gb300.inputs import Workload, make_inputs

pytestmark = pytest.mark.gpu

MAX_ROWS = 4 * 1024 * 1024  # FA_STATIC_SCRATCH_MAX_ROWS in include/fa.h


def _entry():
    from flash_attention_attn_gb300.build import build
    build()
    f = fa.load().fa_bwd_static_scratch
    vp, i = ctypes.c_void_p, ctypes.c_int
    f.argtypes = [vp] * 9 + [i] * 5 + [ctypes.c_float, i, i, i, vp, vp]
    f.restype = i
    return f


def _rel_fro(a, b):
    a = a.float().cpu().numpy().astype(np.float64)
    b = b.float().cpu().numpy().astype(np.float64)
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


def test_static_scratch_backward_matches_fa_bwd_twice():
    f = _entry()
    w = Workload(300, "no-alloc", "bf16", 2, 4, 2, 333, 128, 0, True, True, "normal")
    inp = make_inputs(w, seed=300)
    dev = torch.device("cuda", 0)
    q, k, v, do = (inp[n].to(dev) for n in ("q", "k", "v", "do"))
    o, lse = fa.attention_fwd(q, k, v, scale=w.scale, causal=True)
    ref = fa.attention_bwd(q, k, v, o, lse, do, scale=w.scale, causal=True)
    err = torch.full((1,), 7, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev).cuda_stream
    for _ in range(2):
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        st = f(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), do.data_ptr(),
               dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), w.B, w.T, w.H, w.HKV, w.D, w.scale, 1, 0,
               fa.FA_DTYPE_BF16, err.data_ptr(), stream)
        assert st == fa.FA_OK, fa.fa_status_string(st)
        torch.cuda.synchronize(dev)
        assert int(err.item()) == 0
        for name, got, want in (("dQ", dq, ref[0]), ("dK", dk, ref[1]), ("dV", dv, ref[2])):
            assert _rel_fro(got, want) <= 2e-2, name


def test_static_scratch_rejects_shapes_beyond_its_capacity():
    f = _entry()
    fake = 0x10000  # never dereferenced: the size check comes first
    T = MAX_ROWS // 8 + 1
    st = f(*([fake] * 9), 1, T, 8, 8, 128, 0.088, 1, 0, fa.FA_DTYPE_BF16, None, None)
    assert st == fa.FA_ERR_WORKSPACE
