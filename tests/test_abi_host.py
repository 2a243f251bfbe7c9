"""Host-side tests of the C ABI: no kernel runs here.

* the library loads and exports every function include/fa.h declares;
* argument validation returns the documented status codes before touching
  the GPU;
* the tile planner (the kernels' block-range and block-mask logic, exported
  as fa_plan_*) agrees with brute-force visibility, and with the block-offset
  (triu) scheme of the Graphcore page through the oracle's walk.
"""
from __future__ import annotations

import ctypes
import os
import re

import numpy as np
import pytest

import oracle
from flash_attention_attn_gb300 import _binding as fb
from flash_attention_attn_gb300.build import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build()
    return fb.load()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "fa.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z0-9_]+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert {"fa_fwd", "fa_bwd", "fa_workspace_size", "fa_check_status", "fa_status_string"} <= set(names)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in fa.h but not exported"


def test_workspace_sizes(lib):
    assert fb.fa_workspace_size(fb.FA_OP_FWD, 1, 128, 2, 2, 64, fb.FA_DTYPE_BF16) == 256
    bwd = fb.fa_workspace_size(fb.FA_OP_BWD, 2, 1000, 8, 2, 128, fb.FA_DTYPE_BF16)
    assert bwd >= 256 + 4 * 2 * 8 * 1000 and bwd % 256 == 0
    assert fb.fa_workspace_size(fb.FA_OP_BWD, 1, 128, 3, 2, 64, fb.FA_DTYPE_BF16) == 0  # H % HKV
    assert fb.fa_workspace_size(7, 1, 128, 2, 2, 64, fb.FA_DTYPE_BF16) == 0
    # fp16 runs the same kernels with the same workspace
    assert fb.fa_workspace_size(fb.FA_OP_BWD, 2, 1000, 8, 2, 128, fb.FA_DTYPE_FP16) == bwd
    assert fb.fa_workspace_size(fb.FA_OP_BWD, 2, 1000, 8, 2, 128, 3) == 0


def _r256(x):
    return (x + 255) // 256 * 256


@pytest.mark.parametrize("D", [16, 48, 64])
def test_workspace_sizes_of_the_fused_backward(lib, D):
    """FA_OP_BWD_FUSED (16-bit elements, head dims up to 64): the backward's
    workspace plus the fused path's fp32 dQ accumulator [B,T,H,D] and one turn
    counter per (b, h, 128-row query block), each rounded up to 256 bytes."""
    B, T, H, HKV = 2, 1000, 8, 2
    base = 256 + _r256(4 * B * H * T)
    want = base + _r256(4 * B * T * H * D) + _r256(4 * B * H * ((T + 127) // 128))
    for dt in (fb.FA_DTYPE_BF16, fb.FA_DTYPE_FP16):
        assert fb.fa_workspace_size(fb.FA_OP_BWD_FUSED, B, T, H, HKV, D, dt) == want
        assert fb.fa_workspace_size(fb.FA_OP_BWD, B, T, H, HKV, D, dt) == base
    # the fused path takes neither fp32 nor wider heads
    assert fb.fa_workspace_size(fb.FA_OP_BWD_FUSED, B, T, H, HKV, 64, fb.FA_DTYPE_FP32) == 0
    assert fb.fa_workspace_size(fb.FA_OP_BWD_FUSED, B, T, H, HKV, 72, fb.FA_DTYPE_BF16) == 0


def test_fused_backward_validation(lib):
    """fa_bwd_dkdv_dq refuses shapes it does not take and a workspace without
    the accumulator, before touching the device."""
    p = [FAKE] * 8
    full = fb.fa_workspace_size(fb.FA_OP_BWD_FUSED, 1, 300, 4, 2, 64, fb.FA_DTYPE_BF16)
    args = (1, 300, 4, 2)
    call = lambda D, causal, dt, ws_bytes: fb.fa_bwd_dkdv_dq(*p, *args, D, 0.125, causal, 0, dt, FAKE, ws_bytes, None)
    assert call(64, 0, fb.FA_DTYPE_BF16, full) == fb.FA_ERR_UNSUPPORTED   # not causal
    assert call(128, 1, fb.FA_DTYPE_BF16, 1 << 30) == fb.FA_ERR_UNSUPPORTED  # head dim above 64
    assert call(64, 1, fb.FA_DTYPE_FP32, 1 << 30) == fb.FA_ERR_UNSUPPORTED  # fp32
    assert call(64, 1, fb.FA_DTYPE_BF16, full - 256) == fb.FA_ERR_WORKSPACE  # no room for the accumulator


FAKE = 0x10000  # aligned, never dereferenced: validation fails first


def call_fwd(B=1, T=128, H=2, HKV=2, D=64, scale=0.125, causal=1, window=0, dtype=fb.FA_DTYPE_BF16,
             ptrs=None, ws=FAKE, ws_bytes=1 << 20):
    p = ptrs or [FAKE] * 5
    return fb.fa_fwd(*p, B, T, H, HKV, D, scale, causal, window, dtype, ws, ws_bytes, None)


@pytest.mark.parametrize("kw,code", [
    (dict(B=0), fb.FA_ERR_INVALID_ARG),
    (dict(T=0), fb.FA_ERR_INVALID_ARG),
    (dict(H=3, HKV=2), fb.FA_ERR_INVALID_ARG),
    (dict(window=-1), fb.FA_ERR_INVALID_ARG),
    (dict(scale=0.0), fb.FA_ERR_INVALID_ARG),
    (dict(scale=-1.0), fb.FA_ERR_INVALID_ARG),
    (dict(scale=float("nan")), fb.FA_ERR_INVALID_ARG),
    (dict(scale=float("inf")), fb.FA_ERR_INVALID_ARG),
    (dict(causal=2), fb.FA_ERR_INVALID_ARG),
    (dict(D=100), fb.FA_ERR_UNSUPPORTED),   # head dim not a multiple of 8
    (dict(D=136), fb.FA_ERR_UNSUPPORTED),   # above 128
    (dict(D=8), fb.FA_ERR_UNSUPPORTED),     # below 16
    (dict(D=96, dtype=fb.FA_DTYPE_FP32), fb.FA_ERR_UNSUPPORTED),  # fp32 kernels: 64 or 128 only
    (dict(dtype=5), fb.FA_ERR_UNSUPPORTED),
    (dict(dtype=3), fb.FA_ERR_UNSUPPORTED),
    (dict(dtype=fb.FA_DTYPE_FP16, D=100), fb.FA_ERR_UNSUPPORTED),
    (dict(ptrs=[FAKE, 0, FAKE, FAKE, FAKE]), fb.FA_ERR_INVALID_ARG),
    (dict(ptrs=[FAKE, FAKE + 8, FAKE, FAKE, FAKE]), fb.FA_ERR_INVALID_ARG),
    (dict(ws=0), fb.FA_ERR_WORKSPACE),
    (dict(ws=FAKE + 16), fb.FA_ERR_WORKSPACE),
    (dict(ws_bytes=16), fb.FA_ERR_WORKSPACE),
])
def test_fwd_validation(lib, kw, code):
    assert call_fwd(**kw) == code


def test_bwd_validation(lib):
    p = [FAKE] * 9
    args = (1, 128, 2, 2, 64, 0.125, 1, 0, fb.FA_DTYPE_BF16)
    assert fb.fa_bwd(*p, *args, FAKE, 256, None) == fb.FA_ERR_WORKSPACE  # needs room for Delta
    p[5] = 0
    assert fb.fa_bwd(*p, *args, FAKE, 1 << 20, None) == fb.FA_ERR_INVALID_ARG


def call_fwd_cross(B=1, Tq=100, Tk=300, H=2, HKV=1, D=64, scale=0.125, dtype=fb.FA_DTYPE_BF16, ptrs=None,
                   ws=FAKE, ws_bytes=1 << 20):
    p = ptrs or [FAKE] * 5
    return fb.fa_fwd_cross(*p, B, Tq, Tk, H, HKV, D, scale, dtype, ws, ws_bytes, None)


@pytest.mark.parametrize("kw,code", [
    (dict(Tq=0), fb.FA_ERR_INVALID_ARG),
    (dict(Tk=0), fb.FA_ERR_INVALID_ARG),
    (dict(H=3, HKV=2), fb.FA_ERR_INVALID_ARG),
    (dict(scale=0.0), fb.FA_ERR_INVALID_ARG),
    (dict(D=100), fb.FA_ERR_UNSUPPORTED),
    (dict(D=96, dtype=fb.FA_DTYPE_FP32), fb.FA_ERR_UNSUPPORTED),
    (dict(dtype=7), fb.FA_ERR_UNSUPPORTED),
    (dict(ptrs=[FAKE, FAKE, 0, FAKE, FAKE]), fb.FA_ERR_INVALID_ARG),
    (dict(ptrs=[FAKE, FAKE + 8, FAKE, FAKE, FAKE]), fb.FA_ERR_INVALID_ARG),
    (dict(ws=0), fb.FA_ERR_WORKSPACE),
    (dict(ws_bytes=16), fb.FA_ERR_WORKSPACE),
])
def test_fwd_cross_validation(lib, kw, code):
    assert call_fwd_cross(**kw) == code


def test_bwd_cross_validation(lib):
    p = [FAKE] * 9
    args = (1, 100, 300, 2, 1, 64, 0.125, fb.FA_DTYPE_BF16)
    assert fb.fa_bwd_cross(*p, *args, FAKE, 256, None) == fb.FA_ERR_WORKSPACE  # needs room for Delta (Tq rows)
    assert fb.fa_bwd_cross(*p, 1, 100, 0, 2, 1, 64, 0.125, fb.FA_DTYPE_BF16, FAKE, 1 << 20, None) == \
        fb.FA_ERR_INVALID_ARG
    p[7] = 0
    assert fb.fa_bwd_cross(*p, *args, FAKE, 1 << 20, None) == fb.FA_ERR_INVALID_ARG


def test_no_gpu_means_error_not_fallback(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    st = call_fwd()
    assert st in (fb.FA_ERR_CUDA, fb.FA_ERR_UNSUPPORTED)
    assert call_fwd_cross() in (fb.FA_ERR_CUDA, fb.FA_ERR_UNSUPPORTED)


def test_forward_tiles_hook_validates(lib):
    assert fb.fa_debug_fwd_tiles(4) == fb.FA_ERR_INVALID_ARG
    assert fb.fa_debug_fwd_tiles(-1) == fb.FA_ERR_INVALID_ARG
    for t in (1, 2, 3, 0):
        assert fb.fa_debug_fwd_tiles(t) == fb.FA_OK


def test_persistent_ctas_hook_validates(lib):
    assert fb.fa_debug_max_ctas(-1) == fb.FA_ERR_INVALID_ARG
    for n in (1, 3, 0):
        assert fb.fa_debug_max_ctas(n) == fb.FA_OK


def test_status_strings(lib):
    for code in range(6):
        assert fb.fa_status_string(code) not in ("", "unknown status")
    assert fb.fa_status_string(99) == "unknown status"


# ------------------------------------------------------------ tile planner

def visible(T, causal, window):
    i = np.arange(T)[:, None]
    j = np.arange(T)[None, :]
    v = np.ones((T, T), bool)
    if causal:
        v &= j <= i
    if window:
        v &= (i - j) < window
    return v


PLAN_CASES = [(T, BM, BN, c, W)
              for T in (1, 5, 127, 128, 129, 300, 513)
              for (BM, BN) in ((128, 128), (64, 128), (128, 64), (2, 3), (2, 4))
              for c in (0, 1)
              for W in (0, 1, 3, 64, 128, 200, 1024)]


@pytest.mark.parametrize("T,BM,BN,causal,W", PLAN_CASES)
def test_plan_matches_brute_force(lib, T, BM, BN, causal, W):
    vis = visible(T, causal, W)
    nq, nk = -(-T // BM), -(-T // BN)
    for qb in range(nq):
        lo, hi = fb.fa_plan_kv_range(T, BM, BN, causal, W, qb)
        rows = vis[qb * BM:(qb + 1) * BM]
        for kb in range(nk):
            blk = rows[:, kb * BN:(kb + 1) * BN]
            if blk.any():
                assert lo <= kb <= hi, (qb, kb, lo, hi)
            # a block in range with no visible element is allowed only at the
            # range ends (whole-row granularity); skipping must never lose work
        full_rows = np.zeros((BM, nk * BN), bool)
        full_rows[:rows.shape[0], :T] = rows
        for kb in range(lo, hi + 1):
            blk = full_rows[:, kb * BN:(kb + 1) * BN]
            needs = fb.fa_plan_block_mask(T, BM, BN, causal, W, qb, kb)
            assert needs == int(not blk.all()), (qb, kb)
    for kb in range(nk):
        lo, hi = fb.fa_plan_q_range(T, BM, BN, causal, W, kb)
        cols = vis[:, kb * BN:(kb + 1) * BN]
        for qb in range(nq):
            if cols[qb * BM:(qb + 1) * BM].any():
                assert lo <= qb <= hi


@pytest.mark.parametrize("Tq,Tk", [(1, 1), (7, 7), (130, 130), (9, 20), (20, 9)])
@pytest.mark.parametrize("causal,W", [(0, 0), (1, 0), (1, 3), (0, 4), (1, 1), (1, 200)])
def test_row_key_ranges_match_brute_force(lib, Tq, Tk, causal, W):
    """The per-element rule inside masked blocks, as ranges, against the
    visibility rule evaluated element by element (rows and keys past the end
    included)."""
    i = np.arange(Tq + 3)[:, None]
    j = np.arange(Tk + 3)[None, :]
    vis = (i < Tq) & (j < Tk)
    if causal:
        vis &= j <= i
    if W:
        vis &= (i - j) < W
    for r in range(Tq + 3):
        lo, hi = fb.fa_plan_row_keys(Tq, Tk, causal, W, r)
        want = np.flatnonzero(vis[r])
        got = np.arange(lo, hi + 1) if lo <= hi else np.array([], int)
        assert np.array_equal(got, want), (r, lo, hi)
    for c in range(Tk + 3):
        lo, hi = fb.fa_plan_key_rows(Tq, Tk, causal, W, c)
        want = np.flatnonzero(vis[:, c])
        got = np.arange(lo, hi + 1) if lo <= hi else np.array([], int)
        assert np.array_equal(got, want), (c, lo, hi)


@pytest.mark.parametrize("BM,BN", [(2, 2), (2, 3), (2, 4), (3, 5), (128, 128), (64, 128)])
def test_masked_causal_blocks_follow_triu_offsets(lib, BM, BN):
    """Masked blocks of a causal schedule are the page's diagonal-crossing
    blocks, met in the order of the walk, with offset k = qb*BM - kb*BN + 1."""
    n = int(np.lcm(BM, BN)) * 4
    walk = oracle.triu_offsets(BM, BN)
    seen = []
    for qb in range(n // BM):
        lo, hi = fb.fa_plan_kv_range(n, BM, BN, 1, 0, qb)
        for kb in range(lo, hi + 1):
            if fb.fa_plan_block_mask(n, BM, BN, 1, 0, qb, kb):
                k = qb * BM - kb * BN + 1
                # inside the block, element (r, c) is in the future iff c - r >= k
                r = np.arange(BM)[:, None]
                c = np.arange(BN)[None, :]
                fut = (kb * BN + c) > (qb * BM + r)
                assert np.array_equal(fut, (c - r) >= k)
                seen.append(k)
    assert seen == [walk[i % len(walk)] for i in range(len(seen))]


def test_tile_sizes(lib):
    assert fb.fa_tile_m() == 128 and fb.fa_tile_n() == 128


# ------------------------------------------------ randomised planner checks

def test_planner_properties_on_random_shapes(lib):
    """Random (Tq = Tk = T, tile sizes, causal, window): every visible element
    lies in a visited block, every block outside the visited range is wholly
    masked, and a block flagged mask-free has no masked element (the
    properties the kernels rely on; hypothesis when installed, else a seeded
    sample)."""
    def check(T, BM, BN, causal, W):
        vis = visible(T, causal, W)
        nq, nk = -(-T // BM), -(-T // BN)
        for qb in range(nq):
            lo, hi = fb.fa_plan_kv_range(T, BM, BN, causal, W, qb)
            rows = vis[qb * BM:(qb + 1) * BM]
            for kb in range(nk):
                blk = rows[:, kb * BN:(kb + 1) * BN]
                if not (lo <= kb <= hi):
                    assert not blk.any(), (T, BM, BN, causal, W, qb, kb)
                elif fb.fa_plan_block_mask(T, BM, BN, causal, W, qb, kb) == 0:
                    assert blk.shape == (BM, BN) and blk.all(), (T, BM, BN, causal, W, qb, kb)
        for kb in range(nk):
            lo, hi = fb.fa_plan_q_range(T, BM, BN, causal, W, kb)
            for qb in range(nq):
                if not (lo <= qb <= hi):
                    assert not vis[qb * BM:(qb + 1) * BM, kb * BN:(kb + 1) * BN].any()

    try:
        from hypothesis import given, settings, strategies as st
    except ImportError:
        rng = np.random.default_rng(7)
        for _ in range(200):
            check(int(rng.integers(1, 400)), int(rng.integers(1, 130)), int(rng.integers(1, 130)),
                  int(rng.integers(0, 2)), int(rng.choice([0, 0, 1, int(rng.integers(1, 500))])))
        return

    @settings(max_examples=300, deadline=None)
    @given(st.integers(1, 400), st.integers(1, 130), st.integers(1, 130), st.integers(0, 1),
           st.one_of(st.just(0), st.integers(1, 500)))
    def run(T, BM, BN, causal, W):
        check(T, BM, BN, causal, W)

    run()
