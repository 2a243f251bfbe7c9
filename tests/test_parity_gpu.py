"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Small shapes are compared element by element: several 128-row tiles, ragged
tails, GQA ratios 1..8, causal and non-causal, windows from 1 past T.  The
five named workloads run at full size in the same calls the benchmark times
and are checked on sampled rows the oracle computes one by one, plus
identities that hold at any size.

Tolerances (fixed for this method):
  fp32  : max |err| <= 1e-4 on O, dQ, dK, dV
  bf16, fp16 : max |err| <= 2e-2 on O; relative Frobenius <= 2e-2 on dQ, dK, dV
  LSE   : max |err| <= 1e-3
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import flash_attention_attn_gb300 as fa
from flash_attention_attn_gb300.inputs import WORKLOADS, Workload, as_f64, make_cross_inputs, make_inputs

pytestmark = pytest.mark.gpu

TOL = {"fp32": dict(o=1e-4, grad_abs=1e-4), "bf16": dict(o=2e-2, grad_rel=2e-2), "fp16": dict(o=2e-2, grad_rel=2e-2)}
LSE_TOL = 1e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from flash_attention_attn_gb300.build import build
    build()
    fa.load()
    fa.fa_debug_config(0, 0)


def run_gpu(w: Workload, inp, bwd=True):
    dev = torch.device("cuda", 0)
    q, k, v = (inp[n].to(dev) for n in ("q", "k", "v"))
    o, lse = fa.attention_fwd(q, k, v, scale=w.scale, causal=w.causal, window=w.window)
    out = {"o": o, "lse": lse}
    if bwd:
        do = inp["do"].to(dev)
        dq, dk, dv = fa.attention_bwd(q, k, v, o, lse, do, scale=w.scale, causal=w.causal, window=w.window)
        out.update(dq=dq, dk=dk, dv=dv)
    st, word = fa.check_status()
    assert st == fa.FA_OK, f"device error word {word:#x}"
    return {n: t.float().cpu().numpy().astype(np.float64) for n, t in out.items()}


def rel_fro(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def check_fwd(w, got_o, ref_o, got_lse, ref_lse):
    assert np.all(np.isfinite(got_o)) and np.all(np.isfinite(got_lse))
    err_o = np.max(np.abs(got_o - ref_o))
    err_l = np.max(np.abs(got_lse - ref_lse))
    assert err_o <= TOL[w.dtype]["o"], f"O max-abs {err_o:.3e}"
    assert err_l <= LSE_TOL, f"LSE max-abs {err_l:.3e}"


def check_grad(w, name, got, ref):
    assert np.all(np.isfinite(got)), name
    if w.dtype == "fp32":
        err = np.max(np.abs(got - ref))
        assert err <= TOL["fp32"]["grad_abs"], f"{name} max-abs {err:.3e}"
    elif np.linalg.norm(ref) <= 1e-9 * np.sqrt(ref.size):
        # The exact gradient is zero (every row sees a single key: T = 1 or
        # window = 1, where the softmax has no gradient w.r.t. the scores), so
        # a relative error is undefined; bound the absolute residue instead.
        err = np.max(np.abs(got))
        assert err <= 1e-4, f"{name} (exactly zero) max-abs {err:.3e}"
    else:
        err = rel_fro(got, ref)
        assert err <= TOL[w.dtype]["grad_rel"], f"{name} rel-Frobenius {err:.3e}"


# ------------------------------------------------------ small, element-wise

SMALL = [
    # dtype, B, H, HKV, T, D, window, causal
    ("fp32", 1, 2, 2, 128, 64, 0, True),      # the fp32 workload itself
    ("fp32", 2, 4, 2, 77, 128, 0, True),
    ("fp32", 1, 2, 1, 50, 64, 7, True),
    ("fp32", 1, 2, 2, 40, 64, 0, False),
    ("bf16", 2, 4, 2, 300, 64, 0, True),      # 3 tiles, ragged tail
    ("bf16", 1, 8, 1, 256, 128, 0, True),     # GQA 8:1, exact tiles
    ("bf16", 1, 4, 2, 513, 128, 200, True),   # window not a multiple of the tile
    ("bf16", 1, 2, 2, 384, 64, 256, True),    # window a multiple of the tile
    ("bf16", 1, 2, 1, 200, 64, 0, False),     # non-causal, ragged
    ("bf16", 1, 2, 2, 130, 128, 100, False),  # non-causal window
    ("bf16", 3, 2, 2, 1, 64, 0, True),        # T = 1
    ("bf16", 1, 2, 2, 127, 64, 0, True),
    ("bf16", 1, 2, 2, 129, 128, 0, True),
    ("bf16", 1, 4, 4, 260, 64, 1, True),      # window 1: O = V
    ("bf16", 1, 2, 1, 200, 128, 4096, True),  # window past T
    # head dims other than 64 and 128 (the kernels run at 64 or 128 and read
    # zeros past D)
    ("bf16", 1, 4, 2, 300, 16, 0, True),
    ("bf16", 2, 2, 1, 200, 32, 0, True),
    ("bf16", 1, 4, 2, 260, 48, 100, True),
    ("bf16", 1, 4, 4, 300, 80, 0, True),
    ("bf16", 1, 8, 2, 513, 96, 0, True),
    ("bf16", 1, 2, 1, 130, 96, 0, False),
    ("fp16", 1, 4, 2, 300, 96, 0, True),
    # fp16 elements through the same tensor-core kernels
    ("fp16", 2, 4, 2, 300, 64, 0, True),
    ("fp16", 1, 8, 2, 513, 128, 0, True),
    ("fp16", 1, 4, 2, 513, 128, 200, True),
    ("fp16", 1, 2, 1, 130, 128, 0, False),
    ("fp16", 1, 2, 2, 1, 64, 0, True),
]


@pytest.mark.parametrize("case", SMALL, ids=lambda c: "-".join(map(str, c)))
def test_small_elementwise(case):
    dtype, B, H, HKV, T, D, window, causal = case
    w = Workload(100, "small", dtype, B, H, HKV, T, D, window, causal, True, "normal")
    inp = make_inputs(w, seed=1000 + T + D + H)
    got = run_gpu(w, inp)
    Q, K, V, dO = (as_f64(inp[n]) for n in ("q", "k", "v", "do"))
    O, LSE = oracle.fwd(Q, K, V, w.scale, causal, window)
    dQ, dK, dV, _ = oracle.bwd(Q, K, V, dO, w.scale, causal, window)
    check_fwd(w, got["o"], O, got["lse"], LSE)
    check_grad(w, "dQ", got["dq"], dQ)
    check_grad(w, "dK", got["dk"], dK)
    check_grad(w, "dV", got["dv"], dV)


FWD_TILE_CASES = [
    # dtype, B, H, HKV, T, D, window, causal
    ("bf16", 2, 4, 2, 300, 64, 0, True),      # 3 query tiles: the last pair has no tile B
    ("bf16", 1, 2, 2, 129, 128, 0, True),     # tile B holds one row
    ("bf16", 1, 4, 2, 513, 128, 200, True),   # window: tile A and B ranges differ at both ends
    ("bf16", 1, 2, 2, 384, 64, 128, True),    # window of one tile
    ("bf16", 1, 2, 1, 520, 128, 0, False),    # non-causal, ragged
    ("bf16", 1, 2, 2, 260, 128, 100, False),  # non-causal window
    ("bf16", 1, 4, 4, 260, 64, 1, True),      # window 1
    ("bf16", 1, 8, 1, 1024, 128, 0, True),    # GQA 8:1, four pairs
    ("fp16", 1, 4, 2, 513, 128, 200, True),
    ("fp16", 2, 4, 2, 300, 64, 0, True),
    ("bf16", 1, 4, 2, 513, 96, 0, True),
    ("bf16", 1, 2, 2, 300, 48, 64, True),
    # one query tile: head pairs let GQA shapes use the two-tile kernel
    ("bf16", 2, 8, 2, 100, 128, 0, True),
    ("fp16", 1, 4, 2, 128, 64, 0, False),
    ("bf16", 1, 6, 3, 77, 128, 16, True),
]


@pytest.mark.parametrize("tiles", [1, 2, 3])
@pytest.mark.parametrize("case", FWD_TILE_CASES, ids=lambda c: "-".join(map(str, c)))
def test_forward_tiles_per_cta(case, tiles):
    """Every forward kernel mode (one 128-row query tile per CTA; two tiles
    that are adjacent query blocks of one head; two tiles that are one query
    block of two heads sharing a KV head) against the oracle, element by
    element."""
    dtype, B, H, HKV, T, D, window, causal = case
    w = Workload(103, "tiles", dtype, B, H, HKV, T, D, window, causal, False, "normal")
    inp = make_inputs(w, seed=2000 + T + D + H + window, with_dO=False)
    assert fa.fa_debug_fwd_tiles(tiles) == fa.FA_OK
    try:
        got = run_gpu(w, inp, bwd=False)
    finally:
        fa.fa_debug_fwd_tiles(0)
    O, LSE = oracle.fwd(as_f64(inp["q"]), as_f64(inp["k"]), as_f64(inp["v"]), w.scale, causal, window)
    check_fwd(w, got["o"], O, got["lse"], LSE)


PERSISTENT_CASES = [
    # dtype, B, H, HKV, T, D, window, causal
    ("bf16", 2, 4, 2, 300, 64, 0, True),      # head pairs, ragged tail
    ("bf16", 1, 8, 2, 513, 128, 200, True),   # window, units of different lengths
    ("fp16", 1, 6, 3, 700, 128, 0, True),     # odd H/HKV: block pairs in the forward
    ("bf16", 2, 2, 2, 260, 96, 0, False),     # non-causal
    ("bf16", 1, 4, 4, 129, 64, 1, True),      # units of one block
]


@pytest.mark.parametrize("ctas", [1, 3, 7])
@pytest.mark.parametrize("case", PERSISTENT_CASES, ids=lambda c: "-".join(map(str, c)))
def test_persistent_kernels_with_few_ctas(case, ctas):
    """The persistent forward and backward kernels with their CTA count
    capped, so that every CTA walks several work units (phases of every
    barrier, the TMEM accumulators and the resident tiles carried from one
    unit to the next): against the oracle element by element, and bitwise
    equal to the run with one CTA per SM (a unit's arithmetic does not depend
    on the CTA that runs it)."""
    dtype, B, H, HKV, T, D, window, causal = case
    w = Workload(106, "persistent", dtype, B, H, HKV, T, D, window, causal, True, "normal")
    inp = make_inputs(w, seed=5000 + T + D + H + ctas)
    dev = torch.device("cuda", 0)
    q, k, v, do = (inp[n].to(dev) for n in ("q", "k", "v", "do"))

    def run():
        o, lse = fa.attention_fwd(q, k, v, scale=w.scale, causal=causal, window=window)
        grads = fa.attention_bwd(q, k, v, o, lse, do, scale=w.scale, causal=causal, window=window)
        st, word = fa.check_status()
        assert st == fa.FA_OK, f"device error word {word:#x}"
        return (o, lse) + tuple(grads)

    assert fa.fa_debug_max_ctas(ctas) == fa.FA_OK
    try:
        capped = run()
    finally:
        fa.fa_debug_max_ctas(0)
    full = run()
    for a, b in zip(capped, full):
        assert torch.equal(a, b)
    got = {n: t.float().cpu().numpy().astype(np.float64) for n, t in zip(("o", "lse", "dq", "dk", "dv"), capped)}
    Q, K, V, dO = (as_f64(inp[n]) for n in ("q", "k", "v", "do"))
    O, LSE = oracle.fwd(Q, K, V, w.scale, causal, window)
    dQ, dK, dV, _ = oracle.bwd(Q, K, V, dO, w.scale, causal, window)
    check_fwd(w, got["o"], O, got["lse"], LSE)
    check_grad(w, "dQ", got["dq"], dQ)
    check_grad(w, "dK", got["dk"], dK)
    check_grad(w, "dV", got["dv"], dV)


def _random_cases(n=32, seed=2026):
    """Seeded random shapes across the supported space: dtype, batch, GQA
    ratio, ragged lengths, head dims 16..128, causal or not, windows."""
    rng = np.random.default_rng(seed)
    cases = []
    for _ in range(n):
        hkv = int(rng.choice([1, 2, 4]))
        h = hkv * int(rng.choice([1, 2, 4]))
        T = int(rng.integers(1, 700))
        D = int(rng.choice([16, 32, 48, 64, 72, 96, 128]))
        causal = bool(rng.random() < 0.75)
        window = int(rng.choice([0, 0, 1, 17, 128, 300]))
        dtype = str(rng.choice(["bf16", "fp16"]))
        cases.append((dtype, int(rng.integers(1, 3)), h, hkv, T, D, window, causal))
    return cases


@pytest.mark.parametrize("case", _random_cases(), ids=lambda c: "-".join(map(str, c)))
def test_random_shapes_elementwise(case):
    dtype, B, H, HKV, T, D, window, causal = case
    w = Workload(104, "random", dtype, B, H, HKV, T, D, window, causal, True, "normal")
    inp = make_inputs(w, seed=3000 + T + D + H)
    got = run_gpu(w, inp)
    Q, K, V, dO = (as_f64(inp[n]) for n in ("q", "k", "v", "do"))
    O, LSE = oracle.fwd(Q, K, V, w.scale, causal, window)
    dQ, dK, dV, _ = oracle.bwd(Q, K, V, dO, w.scale, causal, window)
    check_fwd(w, got["o"], O, got["lse"], LSE)
    check_grad(w, "dQ", got["dq"], dQ)
    check_grad(w, "dK", got["dk"], dK)
    check_grad(w, "dV", got["dv"], dV)


# ------------------------------------------------ cross-attention (Tq != Tk)

CROSS_CASES = [
    # dtype, B, H, HKV, Tq, Tk, D
    ("bf16", 2, 4, 2, 300, 77, 64),      # fewer keys than one block, ragged queries
    ("bf16", 1, 8, 2, 129, 513, 128),    # two-tile forward, five key blocks with a tail
    ("bf16", 1, 4, 1, 700, 128, 128),    # many query tiles over one exact key block
    ("fp16", 1, 4, 4, 1, 1000, 96),      # a single query row (decode-like)
    ("fp16", 2, 2, 1, 255, 256, 64),
    ("bf16", 1, 2, 2, 128, 1, 64),       # a single key: O = V_0, dQ = dK = 0
    ("fp32", 1, 2, 2, 50, 200, 64),
    ("fp32", 2, 4, 2, 130, 33, 128),
]


@pytest.mark.parametrize("case", CROSS_CASES, ids=lambda c: "-".join(map(str, c)))
def test_cross_attention_elementwise(case):
    dtype, B, H, HKV, Tq, Tk, D = case
    inp = make_cross_inputs(dtype, B, H, HKV, Tq, Tk, D, seed=4000 + Tq + Tk)
    w = Workload(105, "cross", dtype, B, H, HKV, Tq, D, 0, False, True, "normal")
    dev = torch.device("cuda", 0)
    q, k, v, do = (inp[n].to(dev) for n in ("q", "k", "v", "do"))
    o, lse = fa.attention_fwd(q, k, v, scale=w.scale, causal=False)
    dq, dk, dv = fa.attention_bwd(q, k, v, o, lse, do, scale=w.scale, causal=False)
    st, word = fa.check_status()
    assert st == fa.FA_OK, f"device error word {word:#x}"
    assert dk.shape == k.shape and lse.shape == (B, H, Tq)
    Q, K, V, dO = (as_f64(inp[n]) for n in ("q", "k", "v", "do"))
    O, LSE = oracle.fwd(Q, K, V, w.scale, False, 0)
    dQ, dK, dV, _ = oracle.bwd(Q, K, V, dO, w.scale, False, 0)
    got = {n: t.float().cpu().numpy().astype(np.float64) for n, t in dict(o=o, lse=lse, dq=dq, dk=dk, dv=dv).items()}
    check_fwd(w, got["o"], O, got["lse"], LSE)
    check_grad(w, "dQ", got["dq"], dQ)
    check_grad(w, "dK", got["dk"], dK)
    check_grad(w, "dV", got["dv"], dV)


def _random_cross_cases(n=20, seed=2027):
    """Seeded random cross-attention shapes: dtype, batch, GQA ratio, query
    and key lengths from 1 to 900 (ragged on both sides), head dims 16-128."""
    rng = np.random.default_rng(seed)
    cases = []
    for _ in range(n):
        hkv = int(rng.choice([1, 2, 4]))
        h = hkv * int(rng.choice([1, 2, 3, 4]))
        Tq, Tk = (int(x) for x in rng.integers(1, 900, size=2))
        D = int(rng.choice([16, 32, 64, 80, 96, 128]))
        dtype = str(rng.choice(["bf16", "fp16"]))
        cases.append((dtype, int(rng.integers(1, 3)), h, hkv, Tq, Tk, D))
    return cases


@pytest.mark.parametrize("case", _random_cross_cases(), ids=lambda c: "-".join(map(str, c)))
def test_random_cross_shapes_elementwise(case):
    test_cross_attention_elementwise(case)


def test_cross_attention_rejects_masks():
    inp = make_cross_inputs("bf16", 1, 2, 2, 64, 96, 64, seed=1)
    dev = torch.device("cuda", 0)
    q, k, v = (inp[n].to(dev) for n in ("q", "k", "v"))
    for kw in (dict(causal=True), dict(causal=False, window=16)):
        with pytest.raises(fa.FaError) as e:
            fa.attention_fwd(q, k, v, **kw)
        assert e.value.status == fa.FA_ERR_UNSUPPORTED


@pytest.mark.parametrize("D,window", [(128, 0), (64, 0), (64, 200), (32, 0)], ids=["d128", "d64", "d64-window", "d32"])
def test_backward_is_bitwise_reproducible(D, window):
    """Repeated backwards give identical bits, with the default CTA count and
    with fewer CTAs (a unit's arithmetic does not depend on the CTA, and dQ
    sums its KV blocks in a fixed order)."""
    w = Workload(101, "repro", "bf16", 1, 8, 2, 640, D, window, True, True, "normal")
    inp = make_inputs(w, seed=7)
    dev = torch.device("cuda", 0)
    q, k, v, do = (inp[n].to(dev) for n in ("q", "k", "v", "do"))
    o, lse = fa.attention_fwd(q, k, v, causal=True, window=window)
    g1 = fa.attention_bwd(q, k, v, o, lse, do, causal=True, window=window)
    g2 = fa.attention_bwd(q, k, v, o, lse, do, causal=True, window=window)
    assert fa.fa_debug_max_ctas(5) == fa.FA_OK
    try:
        g3 = fa.attention_bwd(q, k, v, o, lse, do, causal=True, window=window)
    finally:
        fa.fa_debug_max_ctas(0)
    st, word = fa.check_status()
    assert st == fa.FA_OK, hex(word)
    for a, b, c in zip(g1, g2, g3):
        assert torch.equal(a, b) and torch.equal(a, c)


OVERLAP_CASES = [
    # dtype, B, H, HKV, T, D, window, CTA cap (0 = one per SM)
    ("bf16", 1, 8, 2, 640, 64, 0, 0),      # 10 dK/dV units: most SMs start on dQ at once
    ("bf16", 2, 8, 4, 4096, 128, 0, 0),    # 256 dK/dV units: dQ fills the dK/dV tail
    ("fp16", 1, 4, 4, 1000, 128, 300, 3),  # three CTAs each: dQ runs beside all of dK/dV
    ("bf16", 2, 4, 1, 777, 32, 0, 5),      # ragged tail, head dim 32
]


@pytest.mark.parametrize("case", OVERLAP_CASES, ids=lambda c: "-".join(map(str, c)))
def test_backward_call_equals_its_stages(case):
    """fa_bwd launches dQ as a programmatic dependent of dK/dV, so that dQ
    CTAs start on the SMs dK/dV leaves idle; the stage entry points launch
    them one after the other.  Both give the same bits, and work queued after
    fa_bwd sees its dK and dV (read here right after the call)."""
    dtype, B, H, HKV, T, D, window, cap = case
    w = Workload(108, "overlap", dtype, B, H, HKV, T, D, window, True, True, "normal")
    inp = make_inputs(w, seed=7000 + T + D)
    dev = torch.device("cuda", 0)
    q, k, v, do = (inp[n].to(dev) for n in ("q", "k", "v", "do"))
    o, lse = fa.attention_fwd(q, k, v, scale=w.scale, causal=True, window=window)
    dt = fa.FA_DTYPE_BF16 if dtype == "bf16" else fa.FA_DTYPE_FP16
    n = fa.fa_workspace_size(fa.FA_OP_BWD, B, T, H, HKV, D, dt)
    ws = torch.zeros(n, dtype=torch.uint8, device=dev)
    s = torch.cuda.current_stream(dev).cuda_stream
    P = [t.data_ptr() for t in (q, k, v, o, lse, do)]
    args = (B, T, H, HKV, D, w.scale, 1, window, dt, ws.data_ptr(), n, s)
    outs = {}
    assert fa.fa_debug_max_ctas(cap) == fa.FA_OK
    try:
        for path in ("stages", "fa_bwd", "fa_bwd-again"):
            dq, dk, dv = (torch.full_like(t, float("nan")) for t in (q, k, v))
            if path == "stages":
                assert fa.fa_bwd_preprocess(P[3], P[5], B, T, H, HKV, D, dt, ws.data_ptr(), n, s) == fa.FA_OK
                assert fa.fa_bwd_dkdv(P[0], P[1], P[2], P[4], P[5], dk.data_ptr(), dv.data_ptr(), *args) == fa.FA_OK
                assert fa.fa_bwd_dq(P[0], P[1], P[2], P[4], P[5], dq.data_ptr(), *args) == fa.FA_OK
            else:
                assert fa.fa_bwd(*P, dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), *args) == fa.FA_OK
            # consumers on the same stream, queued before any host synchronisation
            outs[path] = tuple(t.clone() for t in (dq, dk, dv))
            st, word = fa.fa_check_status(ws.data_ptr(), s)
            assert st == fa.FA_OK, hex(word)
    finally:
        fa.fa_debug_max_ctas(0)
    for path in ("fa_bwd", "fa_bwd-again"):
        for name, a, b in zip(("dQ", "dK", "dV"), outs["stages"], outs[path]):
            assert torch.equal(a, b), (path, name)
    if T > 1024:
        return  # the stage path is checked against the oracle at these sizes elsewhere
    Q, K, V, dO = (as_f64(inp[x]) for x in ("q", "k", "v", "do"))
    dQ, dK, dV, _ = oracle.bwd(Q, K, V, dO, w.scale, True, window)
    for name, got, ref in zip(("dQ", "dK", "dV"), outs["fa_bwd"], (dQ, dK, dV)):
        check_grad(w, name, got.float().cpu().numpy().astype(np.float64), ref)


FUSED_CASES = [
    # dtype, B, H, HKV, T, D, window
    ("bf16", 2, 4, 2, 300, 64, 0),     # ragged tail, GQA
    ("bf16", 1, 8, 1, 1024, 64, 0),    # GQA 8:1, eight query blocks, up to eight partials per block
    ("fp16", 1, 4, 4, 513, 64, 200),   # window: partials from at most three KV blocks
    ("bf16", 1, 2, 2, 129, 32, 0),     # a one-row last block, head dim 32
    ("bf16", 3, 2, 1, 1, 64, 0),       # T = 1
    ("bf16", 1, 4, 2, 700, 48, 1),     # window 1: dQ = 0
]


@pytest.mark.parametrize("case", FUSED_CASES, ids=lambda c: "-".join(map(str, c)))
def test_fused_backward_against_separate_kernels_and_oracle(case):
    """The fused backward (fa_bwd_dkdv_dq: dQ from the dK/dV kernel's dS
    tiles, partials added in a fixed order) and the separate dK/dV and dQ
    kernels, through the stage entry points on the same Delta: dK and dV are
    the same kernels' arithmetic and must agree bit for bit; dQ, summed in a
    different order, agrees with the oracle at the parity tolerance."""
    dtype, B, H, HKV, T, D, window = case
    w = Workload(107, "fused", dtype, B, H, HKV, T, D, window, True, True, "normal")
    inp = make_inputs(w, seed=6000 + T + D + H)
    dev = torch.device("cuda", 0)
    q, k, v, do = (inp[n].to(dev) for n in ("q", "k", "v", "do"))
    o, lse = fa.attention_fwd(q, k, v, scale=w.scale, causal=True, window=window)
    dt = fa.FA_DTYPE_BF16 if dtype == "bf16" else fa.FA_DTYPE_FP16
    n = fa.fa_workspace_size(fa.FA_OP_BWD_FUSED, B, T, H, HKV, D, dt)
    ws = torch.zeros(n, dtype=torch.uint8, device=dev)
    s = torch.cuda.current_stream(dev).cuda_stream
    P = [t.data_ptr() for t in (q, k, v, o, lse, do)]
    outs = {}
    for path in ("separate", "fused", "fused-again", "fused-5-ctas"):
        if path == "fused-5-ctas":
            assert fa.fa_debug_max_ctas(5) == fa.FA_OK
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        assert fa.fa_bwd_preprocess(P[3], P[5], B, T, H, HKV, D, dt, ws.data_ptr(), n, s) == fa.FA_OK
        args = (B, T, H, HKV, D, w.scale, 1, window, dt, ws.data_ptr(), n, s)
        if path == "separate":
            assert fa.fa_bwd_dkdv(P[0], P[1], P[2], P[4], P[5], dk.data_ptr(), dv.data_ptr(), *args) == fa.FA_OK
            assert fa.fa_bwd_dq(P[0], P[1], P[2], P[4], P[5], dq.data_ptr(), *args) == fa.FA_OK
        else:
            try:
                assert fa.fa_bwd_dkdv_dq(P[0], P[1], P[2], P[4], P[5], dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                                         *args) == fa.FA_OK
            finally:
                fa.fa_debug_max_ctas(0)
        st, word = fa.fa_check_status(ws.data_ptr(), s)
        assert st == fa.FA_OK, hex(word)
        outs[path] = (dq, dk, dv)
    assert torch.equal(outs["separate"][1], outs["fused"][1]), "dK"
    assert torch.equal(outs["separate"][2], outs["fused"][2]), "dV"
    # the fused dQ sums its partials in a fixed order: the same bits every time
    for again in ("fused-again", "fused-5-ctas"):
        for a, b in zip(outs["fused"], outs[again]):
            assert torch.equal(a, b), again
    Q, K, V, dO = (as_f64(inp[n]) for n in ("q", "k", "v", "do"))
    dQ, _, _, _ = oracle.bwd(Q, K, V, dO, w.scale, True, window)
    for path in ("separate", "fused"):
        check_grad(w, f"dQ ({path})", outs[path][0].float().cpu().numpy().astype(np.float64), dQ)


def test_attention_bwd_without_dq_recompute():
    """attention_bwd(recompute_dq=False) is the fused stage: dK and dV the
    same bits as the default path, dQ within the parity tolerance of the
    oracle and the same bits on a second call; shapes it does not cover are
    refused before any launch."""
    w = Workload(110, "fused-api", "bf16", 2, 4, 2, 520, 64, 200, True, True, "normal")
    inp = make_inputs(w, seed=12)
    dev = torch.device("cuda", 0)
    q, k, v, do = (inp[n].to(dev) for n in ("q", "k", "v", "do"))
    o, lse = fa.attention_fwd(q, k, v, causal=True, window=w.window)
    ref = fa.attention_bwd(q, k, v, o, lse, do, causal=True, window=w.window)
    g1 = fa.attention_bwd(q, k, v, o, lse, do, causal=True, window=w.window, recompute_dq=False)
    g2 = fa.attention_bwd(q, k, v, o, lse, do, causal=True, window=w.window, recompute_dq=False)
    st, word = fa.check_status()
    assert st == fa.FA_OK, hex(word)
    assert torch.equal(g1[1], ref[1]) and torch.equal(g1[2], ref[2])
    for a, b in zip(g1, g2):
        assert torch.equal(a, b)
    Q, K, V, dO = (as_f64(inp[x]) for x in ("q", "k", "v", "do"))
    dQ, _, _, _ = oracle.bwd(Q, K, V, dO, w.scale, True, w.window)
    check_grad(w, "dQ", g1[0].float().cpu().numpy().astype(np.float64), dQ)
    q128 = torch.zeros(1, 128, 2, 128, dtype=torch.bfloat16, device=dev)
    o128, lse128 = fa.attention_fwd(q128, q128, q128, causal=True)
    with pytest.raises(fa.FaError):
        fa.attention_bwd(q128, q128, q128, o128, lse128, q128, causal=True, recompute_dq=False)
    with pytest.raises(fa.FaError):
        fa.attention_bwd(q, k, v, o, lse, do, causal=False, recompute_dq=False)


def test_every_output_element_is_written():
    w = Workload(102, "poison", "bf16", 2, 4, 2, 333, 64, 0, True, True, "normal")
    inp = make_inputs(w, seed=9)
    dev = torch.device("cuda", 0)
    q, k, v, do = (inp[n].to(dev) for n in ("q", "k", "v", "do"))
    nan = float("nan")
    o = torch.full_like(q, nan)
    lse = torch.full((w.B, w.H, w.T), nan, device=dev)
    fa.attention_fwd(q, k, v, causal=True, out=o, lse=lse)
    dq, dk, dv = (torch.full_like(t, nan) for t in (q, k, v))
    fa.attention_bwd(q, k, v, o, lse, do, causal=True, dq=dq, dk=dk, dv=dv)
    torch.cuda.synchronize()
    for t in (o, lse, dq, dk, dv):
        assert torch.isfinite(t).all()


@pytest.mark.parametrize("D", [128, 64])
def test_outputs_at_16_byte_offsets(D):
    """Outputs whose rows start 16 but not 32 bytes into a sector take the
    16-byte store path (32-byte aligned outputs leave in whole sectors): the
    same kernels' arithmetic, so the same bits, and nothing written outside
    the views."""
    w = Workload(109, "offset", "bf16", 2, 4, 2, 300, D, 0, True, True, "normal")
    inp = make_inputs(w, seed=11)
    dev = torch.device("cuda", 0)
    q, k, v, do = (inp[n].to(dev) for n in ("q", "k", "v", "do"))

    def shifted(t):  # a view 8 elements (16 bytes) into a larger NaN-filled buffer
        buf = torch.full((t.numel() + 16,), float("nan"), dtype=t.dtype, device=dev)
        view = buf[8:8 + t.numel()].view(t.shape)
        assert view.data_ptr() % 32 == 16
        return buf, view

    o_ref, lse_ref = fa.attention_fwd(q, k, v, causal=True)
    g_ref = fa.attention_bwd(q, k, v, o_ref, lse_ref, do, causal=True)
    ob, o = shifted(q)
    lse = torch.empty_like(lse_ref)
    fa.attention_fwd(q, k, v, causal=True, out=o, lse=lse)
    bufs = [shifted(t) for t in (q, k, v)]
    fa.attention_bwd(q, k, v, o, lse, do, causal=True, dq=bufs[0][1], dk=bufs[1][1], dv=bufs[2][1])
    st, word = fa.check_status()
    assert st == fa.FA_OK, hex(word)
    assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)
    for (buf, view), ref in zip(bufs, g_ref):
        assert torch.equal(view, ref)
    for buf in (ob, *(b for b, _ in bufs)):  # the 8 elements either side stay NaN
        assert torch.isnan(buf[:8]).all() and torch.isnan(buf[-8:]).all()


# ----------------------------------------- named workloads, full size, sampled

def _sample_rows(T, rng, n_random):
    fixed = {0, 1, min(T - 1, 127), min(T - 1, 128), T // 2, T - 2, T - 1}
    rnd = set(rng.integers(0, T, size=n_random).tolist())
    return sorted(r for r in fixed | rnd if 0 <= r < T)


def _dkdv_sample(w: Workload, rng):
    if w.window > 0 or w.T <= 2048:
        return _sample_rows(w.T, rng, 12)
    # Plain causal masking over a long sequence: key j is seen by query rows
    # j..T-1 of every head of its group (forge flash_attn_bwd_dk / _dv, query
    # range starting at j), so the early keys carry the longest accumulations
    # and key 0 sums over every query row.  Take those keys, the ones either
    # side of the first block edge and of the middle, the last keys, and
    # random keys over the whole range.  With key 0 in the set the oracle
    # evaluates every query row of the group once (about 1.1e12 fp64 flops
    # per KV head at T = 32768).
    T = w.T
    fixed = {0, 1, 127, 128, 129, T // 2, T // 2 + 1, T - 256, T - 129, T - 2, T - 1}
    rnd = rng.integers(0, T, size=8).tolist() + rng.integers(T - 256, T, size=4).tolist()
    return sorted(fixed | set(rnd))


@pytest.mark.parametrize("wid", [1, 2, 3, 4, 5])
def test_named_workload_full_size(wid):
    w = WORKLOADS[wid]
    inp = make_inputs(w, with_dO=w.bwd)
    got = run_gpu(w, inp, bwd=w.bwd)
    Q, K, V = (as_f64(inp[n]) for n in ("q", "k", "v"))
    dO = as_f64(inp["do"]) if w.bwd else None
    rng = np.random.default_rng(wid)
    heads = sorted({0, w.H - 1, int(rng.integers(0, w.H))})
    bs = sorted({0, w.B - 1})
    rows = _sample_rows(w.T, rng, 24)
    for b in bs:
        for h in heads:
            O_r, L_r = oracle.fwd_rows(Q, K, V, w.scale, w.causal, w.window, b, h, rows)
            check_fwd(w, got["o"][b, rows, h], O_r, got["lse"][b, h, rows], L_r)
            if w.bwd:
                dq_r, _ = oracle.dq_rows(Q, K, V, dO, w.scale, w.causal, w.window, b, h, rows)
                check_grad(w, f"dQ[b={b},h={h}]", got["dq"][b, rows, h], dq_r)
    if not w.bwd:
        return
    cols = _dkdv_sample(w, rng)
    for b in bs:
        for g in sorted({0, w.HKV - 1}):
            dk_r, dv_r = oracle.dkdv_rows(Q, K, V, dO, w.scale, w.causal, w.window, b, g, cols)
            check_grad(w, f"dK[b={b},g={g}]", got["dk"][b, cols, g], dk_r)
            check_grad(w, f"dV[b={b},g={g}]", got["dv"][b, cols, g], dv_r)
    # identities over every key row: sum_j dK_j = 0 and sum_j dV_j = sum of dO
    # over the group (each row of P sums to 1, of dS to 0)
    rep = w.H // w.HKV
    dk_sum = got["dk"].sum(axis=1)
    dk_scale = np.abs(got["dk"]).sum(axis=1)
    assert np.all(np.abs(dk_sum) <= 2e-2 * dk_scale + 1e-6)
    dv_sum = got["dv"].sum(axis=1)
    want = dO.reshape(w.B, w.T, w.HKV, rep, w.D).sum(axis=(1, 3))
    assert rel_fro(dv_sum, want) <= 2e-2
    # causal row 0 sees only key 0: O row 0 = V row 0 (up to bf16 output rounding)
    if w.causal:
        g_of_h = np.arange(w.H) // rep
        np.testing.assert_allclose(got["o"][:, 0], V[:, 0][:, g_of_h], rtol=0, atol=TOL[w.dtype]["o"])
