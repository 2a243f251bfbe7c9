"""Pins for the fp64 oracle, independent of the oracle's own code.

Each test checks the oracle against something the pages or the mathematics
fix: printed worked examples (tests/golden), closed forms, a library routine
(torch's float64 scaled_dot_product_attention and autograd), brute-force
finite differences and exact special cases.  Together they are chosen so that
a dropped term, a wrong sign, a wrong index or head map, or a transposed
operand anywhere in the oracle fails at least one of them.
"""
from __future__ import annotations

import itertools
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rand_qkv(rng, B, T, H, HKV, D, scale_qk=1.0):
    Q = rng.standard_normal((B, T, H, D)) * scale_qk
    K = rng.standard_normal((B, T, HKV, D)) * scale_qk
    V = rng.standard_normal((B, T, HKV, D))
    dO = rng.standard_normal((B, T, H, D))
    return Q, K, V, dO


def visible_np(T, causal, window):
    i = np.arange(T)[:, None]
    j = np.arange(T)[None, :]
    vis = np.ones((T, T), bool)
    if causal:
        vis &= j <= i
    if window > 0:
        vis &= (i - j) < window
    return vis


CASES = [
    # B, T, H, HKV, D, causal, window
    (1, 1, 1, 1, 4, True, 0),
    (1, 7, 2, 1, 3, True, 0),
    (2, 9, 4, 2, 5, True, 3),
    (1, 11, 3, 3, 4, False, 0),
    (1, 10, 4, 1, 6, False, 4),
    (2, 13, 6, 2, 8, True, 1),
    (1, 8, 2, 2, 4, True, 8),
]


# ------------------------------------------------------------ softmax pins

@pytest.mark.parametrize("case", CASES)
def test_prob_rows_sum_to_one_and_mask_exact(case):
    B, T, H, HKV, D, causal, window = case
    rng = np.random.default_rng(11)
    Q, K, V, _ = rand_qkv(rng, B, T, H, HKV, D)
    vis = visible_np(T, causal, window)
    for b, h in itertools.product(range(B), range(H)):
        P, _ = oracle.probs(Q, K, 0.37, causal, window, b, h)
        assert np.all(P[~vis] == 0.0)
        assert np.all(P[vis] > 0.0)
        assert np.max(np.abs(P.sum(axis=1) - 1.0)) <= 1e-12


@pytest.mark.parametrize("case", [c for c in CASES if c[5]])
def test_causal_row0_is_v0(case):
    B, T, H, HKV, D, causal, window = case
    rng = np.random.default_rng(3)
    Q, K, V, _ = rand_qkv(rng, B, T, H, HKV, D, scale_qk=3.0)
    O, LSE = oracle.fwd(Q, K, V, 0.5, True, window)
    rep = H // HKV
    for h in range(H):
        # Only key 0 is visible to query 0: P = [1], O = V[0] exactly.
        assert np.array_equal(O[:, 0, h, :], V[:, 0, h // rep, :])
        # and LSE_0 is the single score itself
        s00 = 0.5 * np.sum(Q[:, 0, h, :] * K[:, 0, h // rep, :], axis=-1)
        np.testing.assert_allclose(LSE[:, h, 0], s00, rtol=0, atol=1e-14)


@pytest.mark.parametrize("causal,window", [(True, 0), (True, 3), (False, 0), (False, 2)])
def test_identical_keys_give_mean_of_visible_v(causal, window):
    B, T, H, HKV, D = 2, 9, 4, 2, 5
    rng = np.random.default_rng(5)
    Q, K, V, _ = rand_qkv(rng, B, T, H, HKV, D)
    K[:] = K[:, :1]  # every key row of a head equal to row 0
    O, _ = oracle.fwd(Q, K, V, 0.8, causal, window)
    vis = visible_np(T, causal, window)
    rep = H // HKV
    for b, h, i in itertools.product(range(B), range(H), range(T)):
        want = V[b, vis[i], h // rep, :].mean(axis=0)
        np.testing.assert_allclose(O[b, i, h], want, rtol=0, atol=1e-13)


@pytest.mark.parametrize("case", CASES)
def test_lse_is_log_sum_exp_of_masked_scores(case):
    B, T, H, HKV, D, causal, window = case
    rng = np.random.default_rng(17)
    Q, K, V, _ = rand_qkv(rng, B, T, H, HKV, D, scale_qk=0.3)
    scale = 0.9
    _, LSE = oracle.fwd(Q, K, V, scale, causal, window)
    vis = visible_np(T, causal, window)
    rep = H // HKV
    from scipy.special import logsumexp
    for b, h in itertools.product(range(B), range(H)):
        S = scale * np.einsum("id,jd->ij", Q[b, :, h], K[b, :, h // rep]).astype(np.longdouble)
        for i in range(T):
            # direct sum, no max shift, in extended precision (inputs are small)
            direct = np.log(np.sum(np.exp(S[i, vis[i]])))
            assert abs(float(direct) - LSE[b, h, i]) <= 1e-13
            lib = logsumexp(np.asarray(S[i, vis[i]], dtype=np.float64))
            assert abs(lib - LSE[b, h, i]) <= 1e-13


# ----------------------------------------------------- library routine pin

def _sdpa_reference(Q, K, V, dO, scale, causal, window):
    """torch float64 SDPA (math path) + autograd, GQA via enable_gqa."""
    q = torch.tensor(Q).permute(0, 2, 1, 3).requires_grad_(True)
    k = torch.tensor(K).permute(0, 2, 1, 3).requires_grad_(True)
    v = torch.tensor(V).permute(0, 2, 1, 3).requires_grad_(True)
    T = Q.shape[1]
    mask = torch.tensor(visible_np(T, causal, window))
    o = torch.nn.functional.scaled_dot_product_attention(
        q, k, v, attn_mask=mask, scale=scale, enable_gqa=True)
    o.backward(torch.tensor(dO).permute(0, 2, 1, 3))
    out = o.detach().permute(0, 2, 1, 3).numpy()
    grads = [t.grad.permute(0, 2, 1, 3).numpy() for t in (q, k, v)]
    return out, grads


@pytest.mark.parametrize("case", CASES)
def test_matches_torch_sdpa_and_autograd(case):
    B, T, H, HKV, D, causal, window = case
    rng = np.random.default_rng(23)
    Q, K, V, dO = rand_qkv(rng, B, T, H, HKV, D)
    scale = 1.0 / np.sqrt(D)
    O, _ = oracle.fwd(Q, K, V, scale, causal, window)
    dQ, dK, dV, _ = oracle.bwd(Q, K, V, dO, scale, causal, window)
    O_ref, (dQ_ref, dK_ref, dV_ref) = _sdpa_reference(Q, K, V, dO, scale, causal, window)
    for a, r in ((O, O_ref), (dQ, dQ_ref), (dK, dK_ref), (dV, dV_ref)):
        np.testing.assert_allclose(a, r, rtol=0, atol=1e-12)


# ------------------------------------------------------- finite differences

@pytest.mark.parametrize("T,HKV,D,causal,window", [
    (1, 1, 2, True, 0), (3, 2, 3, True, 0), (5, 1, 2, True, 2), (5, 2, 3, False, 0),
    (3, 1, 3, False, 1), (5, 2, 2, True, 1), (4, 1, 3, False, 2),
])
def test_gradients_match_central_differences(T, HKV, D, causal, window):
    B, H = 1, 2
    rng = np.random.default_rng(31 + T + D)
    Q, K, V, dO = rand_qkv(rng, B, T, H, HKV, D)
    scale = 0.7

    def loss(Qx, Kx, Vx):
        O, _ = oracle.fwd(Qx, Kx, Vx, scale, causal, window)
        return float(np.sum(O * dO))

    dQ, dK, dV, _ = oracle.bwd(Q, K, V, dO, scale, causal, window)
    h = 1e-6
    for name, X, G in (("Q", Q, dQ), ("K", K, dK), ("V", V, dV)):
        fd = np.zeros_like(X)
        for idx in np.ndindex(X.shape):
            Xp = X.copy()
            Xm = X.copy()
            Xp[idx] += h
            Xm[idx] -= h
            args_p = {"Q": Q, "K": K, "V": V}
            args_m = dict(args_p)
            args_p[name] = Xp
            args_m[name] = Xm
            fd[idx] = (loss(args_p["Q"], args_p["K"], args_p["V"])
                       - loss(args_m["Q"], args_m["K"], args_m["V"])) / (2 * h)
        err = np.abs(fd - G)
        tol = 1e-7 * np.maximum(1.0, np.abs(G))
        assert np.all(err <= tol), f"d{name}: max err {err.max():.3e}"


# ------------------------------------------------------------ closed forms

def test_window_one_is_identity():
    B, T, H, HKV, D = 2, 9, 4, 2, 5
    rng = np.random.default_rng(41)
    Q, K, V, _ = rand_qkv(rng, B, T, H, HKV, D)
    O, LSE = oracle.fwd(Q, K, V, 0.6, True, 1)
    rep = H // HKV
    for h in range(H):
        assert np.array_equal(O[:, :, h], V[:, :, h // rep])
        sii = 0.6 * np.sum(Q[:, :, h] * K[:, :, h // rep], axis=-1)
        np.testing.assert_allclose(LSE[:, h, :], sii, rtol=0, atol=1e-14)


@pytest.mark.parametrize("causal", [True, False])
def test_window_at_least_T_equals_no_window(causal):
    B, T, H, HKV, D = 1, 8, 2, 1, 4
    rng = np.random.default_rng(43)
    Q, K, V, dO = rand_qkv(rng, B, T, H, HKV, D)
    # without causal masking the window only bounds keys from below: W = 2T
    # covers every i - j, which is < T.
    W = T if causal else 2 * T
    a = oracle.fwd(Q, K, V, 0.5, causal, 0)
    b = oracle.fwd(Q, K, V, 0.5, causal, W)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)
    ga = oracle.bwd(Q, K, V, dO, 0.5, causal, 0)
    gb = oracle.bwd(Q, K, V, dO, 0.5, causal, W)
    for x, y in zip(ga, gb):
        assert np.array_equal(x, y)


@pytest.mark.parametrize("causal,window", [(True, 0), (True, 3), (False, 0)])
def test_gqa_equals_mha_with_repeat_interleaved_kv(causal, window):
    B, T, H, HKV, D = 2, 7, 6, 2, 4
    rep = H // HKV
    rng = np.random.default_rng(47)
    Q, K, V, dO = rand_qkv(rng, B, T, H, HKV, D)
    Kr = np.repeat(K, rep, axis=2)  # head h uses kv head h // rep
    Vr = np.repeat(V, rep, axis=2)
    O_g, L_g = oracle.fwd(Q, K, V, 0.5, causal, window)
    O_m, L_m = oracle.fwd(Q, Kr, Vr, 0.5, causal, window)
    assert np.array_equal(O_g, O_m) and np.array_equal(L_g, L_m)
    dQg, dKg, dVg, _ = oracle.bwd(Q, K, V, dO, 0.5, causal, window)
    dQm, dKm, dVm, _ = oracle.bwd(Q, Kr, Vr, dO, 0.5, causal, window)
    np.testing.assert_allclose(dQg, dQm, rtol=0, atol=1e-13)
    # the GQA key gradient is the sum over the group's heads of the MHA one
    np.testing.assert_allclose(dKg, dKm.reshape(B, T, HKV, rep, D).sum(axis=3), rtol=0, atol=1e-12)
    np.testing.assert_allclose(dVg, dVm.reshape(B, T, HKV, rep, D).sum(axis=3), rtol=0, atol=1e-12)


@pytest.mark.parametrize("case", CASES)
def test_delta_definition_equals_rowsum_dO_O(case):
    B, T, H, HKV, D, causal, window = case
    rng = np.random.default_rng(53)
    Q, K, V, dO = rand_qkv(rng, B, T, H, HKV, D)
    O, _ = oracle.fwd(Q, K, V, 0.4, causal, window)
    _, _, _, Delta = oracle.bwd(Q, K, V, dO, 0.4, causal, window)
    ident = np.einsum("bthd,bthd->bht", dO, O)
    np.testing.assert_allclose(Delta, ident, rtol=0, atol=1e-12)


def test_key_gradient_sums_to_zero_and_value_gradient_sums_dO():
    B, T, H, HKV, D = 2, 12, 4, 2, 6
    rng = np.random.default_rng(59)
    Q, K, V, dO = rand_qkv(rng, B, T, H, HKV, D)
    dQ, dK, dV, _ = oracle.bwd(Q, K, V, dO, 0.45, True, 5)
    # sum_j dS_ij = 0 per row  =>  sum_j dK_j = 0 per (b, g)
    np.testing.assert_allclose(dK.sum(axis=1), 0.0, rtol=0, atol=1e-12)
    # sum_j P_ij = 1 per row   =>  sum_j dV_j = sum over the group's heads and rows of dO
    want = dO.reshape(B, T, HKV, H // HKV, D).sum(axis=(1, 3))
    np.testing.assert_allclose(dV.sum(axis=1), want, rtol=0, atol=1e-12)


# ------------------------------------------------------- sampled-row forms

@pytest.mark.parametrize("case", CASES)
def test_row_functions_agree_with_full_functions(case):
    B, T, H, HKV, D, causal, window = case
    rng = np.random.default_rng(61)
    Q, K, V, dO = rand_qkv(rng, B, T, H, HKV, D)
    O, LSE = oracle.fwd(Q, K, V, 0.5, causal, window)
    dQ, dK, dV, Delta = oracle.bwd(Q, K, V, dO, 0.5, causal, window)
    rows = sorted(set([0, T - 1, T // 2]))
    b = B - 1
    for h in range(H):
        o_r, l_r = oracle.fwd_rows(Q, K, V, 0.5, causal, window, b, h, rows)
        np.testing.assert_allclose(o_r, O[b, rows, h], rtol=0, atol=1e-13)
        np.testing.assert_allclose(l_r, LSE[b, h, rows], rtol=0, atol=1e-13)
        dq_r, de_r = oracle.dq_rows(Q, K, V, dO, 0.5, causal, window, b, h, rows)
        np.testing.assert_allclose(dq_r, dQ[b, rows, h], rtol=0, atol=1e-13)
        np.testing.assert_allclose(de_r, Delta[b, h, rows], rtol=0, atol=1e-13)
    for g in range(HKV):
        dk_r, dv_r = oracle.dkdv_rows(Q, K, V, dO, 0.5, causal, window, b, g, rows)
        np.testing.assert_allclose(dk_r, dK[b, rows, g], rtol=0, atol=1e-12)
        np.testing.assert_allclose(dv_r, dV[b, rows, g], rtol=0, atol=1e-12)


# ------------------------------------------------ block-offset (triu) scheme

def _read_golden(name):
    meta = {}
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line.startswith("# rows="):
                meta = dict(kv.split("=") for kv in line[2:].split())
                continue
            if not line or line.startswith("#") or set(line) <= {"-"}:
                continue
            rows.append([int(x) for x in line.replace("|", " ").split()])
    return {k: int(v) for k, v in meta.items()}, np.array(rows, dtype=np.int64)


def _blocks_needing_mask(n, bq, bkv):
    """(i, j, k) in q-outer order for blocks that have a visible and a masked element.

    Written from the block conditions of the page's forward loop: a block runs
    when its last query row reaches its first key, and is masked when its
    first query row is below its last key; its offset is k = i*bq - j*bkv + 1.
    """
    out = []
    for i in range(n // bq):
        for j in range(n // bkv):
            runs = (i + 1) * bq > j * bkv
            masked = i * bq < (j + 1) * bkv - 1
            if runs and masked:
                out.append((i, j, i * bq - j * bkv + 1))
    return out


GOLDEN_FILES = ["triu_4x4_blocks2x2.txt", "triu_6x6_blocks2x3.txt", "triu_8x8_blocks2x4.txt"]


def test_triu_walk_sequences_hand_derived():
    assert oracle.triu_offsets(2, 2) == [1]
    assert oracle.triu_offsets(2, 3) == [1, 0, 2]
    assert oracle.triu_offsets(2, 4) == [1, 3]


def test_triu_walk_rejects_single_column_blocks():
    # The walk starts at offset 1, outside its range (numCols - 1 = 0) when a
    # block is one key wide, so it never returns to its start; the oracle
    # reports that instead of looping.
    with pytest.raises(RuntimeError):
        oracle.triu_offsets(2, 1)


@pytest.mark.parametrize("bq,bkv", [(a, b) for a in range(1, 9) for b in range(2, 9)])
def test_triu_walk_matches_closed_form_cycled(bq, bkv):
    n = np.lcm(bq, bkv) * 3
    walk = oracle.triu_offsets(bq, bkv)
    closed = [k for (_, _, k) in _blocks_needing_mask(n, bq, bkv)]
    assert len(set(walk)) == len(walk)
    cycled = [walk[c % len(walk)] for c in range(len(closed))]
    assert cycled == closed


@pytest.mark.parametrize("name", GOLDEN_FILES)
def test_triu_blocks_reproduce_printed_diagrams(name):
    meta, diagram = _read_golden(name)
    n, bq, bkv = meta["rows"], meta["block_rows"], meta["block_cols"]
    assert diagram.shape == (n, n)
    walk = oracle.triu_offsets(bq, bkv)
    crossing = _blocks_needing_mask(n, bq, bkv)
    # Rebuild the picture block by block.  Blocks that need a mask take their
    # offset k from the walk, in visit order; every other block is either
    # wholly masked, wholly visible, or (in the picture only) touches the
    # diagonal with nothing strictly above it, and takes k = i*bq - j*bkv + 1.
    picture = np.zeros((n, n), np.int64)
    mask = np.zeros((n, n), np.int64)
    ks = {(i, j): walk[c % len(walk)] for c, (i, j, _) in enumerate(crossing)}
    for i in range(n // bq):
        for j in range(n // bkv):
            blk = (slice(i * bq, (i + 1) * bq), slice(j * bkv, (j + 1) * bkv))
            k = ks.get((i, j), i * bq - j * bkv + 1)
            picture[blk] = np.triu(np.ones((bq, bkv), np.int64), k - 1)
            mask[blk] = np.triu(np.ones((bq, bkv), np.int64), k)
    assert np.array_equal(picture, diagram)
    # the masks the code adds cover exactly the strictly-upper (future) part
    assert np.array_equal(mask, np.triu(np.ones((n, n), np.int64), 1))


# ------------------------------------------------ cross-attention (Tq != Tk)
#
# The teeny-kernels page (flash_attn2.rs, `flash_attention2_forward`) takes
# separate query and key lengths and visits every key of every query row:
# unmasked attention of Tq query rows over Tk key rows.

CROSS = [
    # B, Tq, Tk, H, HKV, D
    (1, 3, 8, 2, 1, 4),
    (2, 9, 4, 4, 2, 5),
    (1, 1, 13, 3, 3, 3),
    (1, 12, 1, 2, 2, 4),
    (2, 6, 11, 6, 2, 6),
]


def rand_cross(rng, B, Tq, Tk, H, HKV, D):
    Q = rng.standard_normal((B, Tq, H, D))
    K = rng.standard_normal((B, Tk, HKV, D))
    V = rng.standard_normal((B, Tk, HKV, D))
    dO = rng.standard_normal((B, Tq, H, D))
    return Q, K, V, dO


@pytest.mark.parametrize("case", CROSS)
def test_cross_attention_matches_torch_sdpa_and_autograd(case):
    B, Tq, Tk, H, HKV, D = case
    rng = np.random.default_rng(71 + Tq + Tk)
    Q, K, V, dO = rand_cross(rng, B, Tq, Tk, H, HKV, D)
    scale = 0.6
    O, LSE = oracle.fwd(Q, K, V, scale, False, 0)
    dQ, dK, dV, Delta = oracle.bwd(Q, K, V, dO, scale, False, 0)
    assert O.shape == Q.shape and LSE.shape == (B, H, Tq) and dK.shape == K.shape and Delta.shape == (B, H, Tq)
    q = torch.tensor(Q).permute(0, 2, 1, 3).requires_grad_(True)
    k = torch.tensor(K).permute(0, 2, 1, 3).requires_grad_(True)
    v = torch.tensor(V).permute(0, 2, 1, 3).requires_grad_(True)
    o = torch.nn.functional.scaled_dot_product_attention(q, k, v, scale=scale, enable_gqa=True)
    o.backward(torch.tensor(dO).permute(0, 2, 1, 3))
    np.testing.assert_allclose(O, o.detach().permute(0, 2, 1, 3).numpy(), rtol=0, atol=1e-12)
    for a, t in ((dQ, q), (dK, k), (dV, v)):
        np.testing.assert_allclose(a, t.grad.permute(0, 2, 1, 3).numpy(), rtol=0, atol=1e-12)
    rep = H // HKV
    kk = torch.tensor(K).repeat_interleave(rep, dim=2)
    S = scale * torch.einsum("bihd,bjhd->bhij", torch.tensor(Q), kk)
    np.testing.assert_allclose(LSE, torch.logsumexp(S, dim=-1).numpy(), rtol=0, atol=1e-12)


@pytest.mark.parametrize("case", CROSS[:3] + CROSS[4:])
def test_cross_attention_key_split_merges_by_lse(case):
    """Attention over keys [K1; K2] is the LSE-weighted merge of attention
    over K1 and over K2: O = (e^L1 O1 + e^L2 O2) / (e^L1 + e^L2),
    L = log(e^L1 + e^L2)."""
    B, Tq, Tk, H, HKV, D = case
    rng = np.random.default_rng(83 + Tk)
    Q, K, V, _ = rand_cross(rng, B, Tq, Tk, H, HKV, D)
    cut = Tk // 2
    O, L = oracle.fwd(Q, K, V, 0.5, False, 0)
    O1, L1 = oracle.fwd(Q, K[:, :cut], V[:, :cut], 0.5, False, 0)
    O2, L2 = oracle.fwd(Q, K[:, cut:], V[:, cut:], 0.5, False, 0)
    Lm = np.logaddexp(L1, L2)
    w1 = np.exp(L1 - Lm).transpose(0, 2, 1)[..., None]
    w2 = np.exp(L2 - Lm).transpose(0, 2, 1)[..., None]
    np.testing.assert_allclose(L, Lm, rtol=0, atol=1e-12)
    np.testing.assert_allclose(O, w1 * O1 + w2 * O2, rtol=0, atol=1e-12)


@pytest.mark.parametrize("case", CROSS)
def test_cross_attention_is_invariant_to_key_order(case):
    """Permuting the key rows (K and V together) leaves O, LSE and dQ
    unchanged and permutes dK and dV the same way."""
    B, Tq, Tk, H, HKV, D = case
    rng = np.random.default_rng(89 + Tq)
    Q, K, V, dO = rand_cross(rng, B, Tq, Tk, H, HKV, D)
    perm = rng.permutation(Tk)
    O, L = oracle.fwd(Q, K, V, 0.7, False, 0)
    Op, Lp = oracle.fwd(Q, K[:, perm], V[:, perm], 0.7, False, 0)
    np.testing.assert_allclose(Op, O, rtol=0, atol=1e-12)
    np.testing.assert_allclose(Lp, L, rtol=0, atol=1e-12)
    dQ, dK, dV, _ = oracle.bwd(Q, K, V, dO, 0.7, False, 0)
    dQp, dKp, dVp, _ = oracle.bwd(Q, K[:, perm], V[:, perm], dO, 0.7, False, 0)
    np.testing.assert_allclose(dQp, dQ, rtol=0, atol=1e-12)
    np.testing.assert_allclose(dKp, dK[:, perm], rtol=0, atol=1e-12)
    np.testing.assert_allclose(dVp, dV[:, perm], rtol=0, atol=1e-12)


@pytest.mark.parametrize("Tq,Tk,HKV", [(2, 5, 1), (4, 3, 2), (1, 4, 1)])
def test_cross_attention_gradients_match_central_differences(Tq, Tk, HKV):
    B, H, D = 1, 2, 2
    rng = np.random.default_rng(97 + Tq * Tk)
    Q, K, V, dO = rand_cross(rng, B, Tq, Tk, H, HKV, D)
    dQ, dK, dV, _ = oracle.bwd(Q, K, V, dO, 0.9, False, 0)

    def loss(q, k, v):
        return float(np.sum(oracle.fwd(q, k, v, 0.9, False, 0)[0] * dO))

    h = 1e-6
    for X, G, which in ((Q, dQ, 0), (K, dK, 1), (V, dV, 2)):
        for idx in np.ndindex(X.shape):
            plus = [Q.copy(), K.copy(), V.copy()]
            minus = [Q.copy(), K.copy(), V.copy()]
            plus[which][idx] += h
            minus[which][idx] -= h
            fd = (loss(*plus) - loss(*minus)) / (2 * h)
            assert abs(fd - G[idx]) <= 1e-7 * max(1.0, abs(G[idx])), (which, idx, fd, G[idx])


@pytest.mark.parametrize("case", CROSS)
def test_cross_attention_row_functions_agree_with_full_functions(case):
    B, Tq, Tk, H, HKV, D = case
    rng = np.random.default_rng(101)
    Q, K, V, dO = rand_cross(rng, B, Tq, Tk, H, HKV, D)
    O, LSE = oracle.fwd(Q, K, V, 0.5, False, 0)
    dQ, dK, dV, Delta = oracle.bwd(Q, K, V, dO, 0.5, False, 0)
    rows = sorted({0, Tq - 1, Tq // 2})
    cols = sorted({0, Tk - 1, Tk // 2})
    b = B - 1
    for h in range(H):
        o_r, l_r = oracle.fwd_rows(Q, K, V, 0.5, False, 0, b, h, rows)
        np.testing.assert_allclose(o_r, O[b, rows, h], rtol=0, atol=1e-13)
        np.testing.assert_allclose(l_r, LSE[b, h, rows], rtol=0, atol=1e-13)
        dq_r, de_r = oracle.dq_rows(Q, K, V, dO, 0.5, False, 0, b, h, rows)
        np.testing.assert_allclose(dq_r, dQ[b, rows, h], rtol=0, atol=1e-13)
        np.testing.assert_allclose(de_r, Delta[b, h, rows], rtol=0, atol=1e-13)
    for g in range(HKV):
        dk_r, dv_r = oracle.dkdv_rows(Q, K, V, dO, 0.5, False, 0, b, g, cols)
        np.testing.assert_allclose(dk_r, dK[b, cols, g], rtol=0, atol=1e-12)
        np.testing.assert_allclose(dv_r, dV[b, cols, g], rtol=0, atol=1e-12)
