"""The oracle's pins catch plausible mistakes.

Each case plants one mistake in a copy of the oracle's C source (a dropped
term, a wrong sign, index or head map, a transposed operand, an off-by-one
mask), builds that copy into its own library on the CPU, and runs a battery
of the independent pins (torch float64 SDPA + autograd, finite differences,
closed forms, the printed triu walk) against it.  Every mutant must fail at
least one pin; the unmodified oracle must pass them all.
"""
from __future__ import annotations

import os

import numpy as np
import pytest
import torch

import oracle


def _visible(T, causal, window):
    i = np.arange(T)[:, None]
    j = np.arange(T)[None, :]
    v = np.ones((T, T), bool)
    if causal:
        v &= j <= i
    if window:
        v &= (i - j) < window
    return v


def _sdpa(Q, K, V, dO, scale, causal, window):
    q, k, v = (torch.tensor(x).permute(0, 2, 1, 3).requires_grad_(True) for x in (Q, K, V))
    mask = torch.tensor(_visible(Q.shape[1], causal, window))
    o = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=mask, scale=scale, enable_gqa=True)
    o.backward(torch.tensor(dO).permute(0, 2, 1, 3))
    return o.detach().permute(0, 2, 1, 3).numpy(), [t.grad.permute(0, 2, 1, 3).numpy() for t in (q, k, v)]


def _pin_sdpa():
    rng = np.random.default_rng(5)
    for (B, T, H, HKV, D, causal, W) in ((1, 9, 4, 2, 5, True, 3), (2, 7, 2, 1, 4, False, 0), (1, 11, 6, 3, 4, True, 0)):
        Q, K, V, dO = (rng.standard_normal(s) for s in ((B, T, H, D), (B, T, HKV, D), (B, T, HKV, D), (B, T, H, D)))
        sc = 0.6
        O, LSE = oracle.fwd(Q, K, V, sc, causal, W)
        dQ, dK, dV, _ = oracle.bwd(Q, K, V, dO, sc, causal, W)
        Or, (dQr, dKr, dVr) = _sdpa(Q, K, V, dO, sc, causal, W)
        for a, r in ((O, Or), (dQ, dQr), (dK, dKr), (dV, dVr)):
            if not np.allclose(a, r, rtol=0, atol=1e-10):
                return False
        # LSE against the log-sum-exp of the masked scores
        rep = H // HKV
        vis = _visible(T, causal, W)
        for h in range(H):
            S = sc * np.einsum("id,jd->ij", Q[0, :, h], K[0, :, h // rep])
            want = np.array([np.log(np.sum(np.exp(S[i, vis[i]]))) for i in range(T)])
            if not np.allclose(LSE[0, h], want, rtol=0, atol=1e-10):
                return False
    return True


def _pin_rows_match_full():
    rng = np.random.default_rng(6)
    B, T, H, HKV, D = 1, 10, 4, 2, 3
    Q, K, V, dO = (rng.standard_normal(s) for s in ((B, T, H, D), (B, T, HKV, D), (B, T, HKV, D), (B, T, H, D)))
    O, LSE = oracle.fwd(Q, K, V, 0.5, True, 4)
    dQ, dK, dV, _ = oracle.bwd(Q, K, V, dO, 0.5, True, 4)
    rows = [0, 3, 9]
    for h in range(H):
        o, l = oracle.fwd_rows(Q, K, V, 0.5, True, 4, 0, h, rows)
        dq, _ = oracle.dq_rows(Q, K, V, dO, 0.5, True, 4, 0, h, rows)
        if not (np.allclose(o, O[0, rows, h], atol=1e-12) and np.allclose(l, LSE[0, h, rows], atol=1e-12)
                and np.allclose(dq, dQ[0, rows, h], atol=1e-12)):
            return False
    for g in range(HKV):
        dk, dv = oracle.dkdv_rows(Q, K, V, dO, 0.5, True, 4, 0, g, rows)
        if not (np.allclose(dk, dK[0, rows, g], atol=1e-12) and np.allclose(dv, dV[0, rows, g], atol=1e-12)):
            return False
    return True


def _pin_triu():
    """The walk's offsets: the hand-derived sequences of the printed examples,
    and the closed form k = i*bq - j*bkv + 1 over the blocks that need a mask,
    in visit order, for every block shape up to 8 x 8."""
    try:
        if not (oracle.triu_offsets(2, 2) == [1] and oracle.triu_offsets(2, 3) == [1, 0, 2]
                and oracle.triu_offsets(2, 4) == [1, 3]):
            return False
        for bq in range(1, 9):
            for bkv in range(2, 9):
                n = int(np.lcm(bq, bkv)) * 3
                closed = [i * bq - j * bkv + 1 for i in range(n // bq) for j in range(n // bkv)
                          if (i + 1) * bq > j * bkv and i * bq < (j + 1) * bkv - 1]
                walk = oracle.triu_offsets(bq, bkv)
                if [walk[c % len(walk)] for c in range(len(closed))] != closed:
                    return False
        return True
    except RuntimeError:
        return False


def _pin_finite_differences():
    rng = np.random.default_rng(7)
    Q, K, V, dO = (rng.standard_normal(s) for s in ((1, 4, 2, 2), (1, 4, 1, 2), (1, 4, 1, 2), (1, 4, 2, 2)))
    sc, causal, W = 0.8, True, 3
    dQ, dK, dV, _ = oracle.bwd(Q, K, V, dO, sc, causal, W)

    def loss(q, k, v):
        return float(np.sum(oracle.fwd(q, k, v, sc, causal, W)[0] * dO))

    h = 1e-6
    for X, G, which in ((Q, dQ, 0), (K, dK, 1), (V, dV, 2)):
        for idx in np.ndindex(X.shape):
            args_p = [Q.copy(), K.copy(), V.copy()]
            args_m = [Q.copy(), K.copy(), V.copy()]
            args_p[which][idx] += h
            args_m[which][idx] -= h
            fd = (loss(*args_p) - loss(*args_m)) / (2 * h)
            if abs(fd - G[idx]) > 1e-6 * max(1.0, abs(G[idx])):
                return False
    return True


def _pin_prologue():
    """QK-norm + rotary: rotation as complex multiplication, unit RMS under
    identity factors, and the backward against finite differences."""
    rng = np.random.default_rng(8)
    tokens, hq, hk, D = 3, 2, 1, 4
    qk = rng.standard_normal((tokens, hq + hk, D))
    ones, zeros = np.ones((tokens, D)), np.zeros((tokens, D))
    n = np.concatenate(oracle.qk_norm_rope_fwd(qk, ones, zeros, hq), axis=1)
    ms = np.mean(qk ** 2, axis=-1)
    if not np.allclose(np.mean(n ** 2, axis=-1), ms / (ms + 1.1920928955078125e-7), rtol=1e-12):
        return False
    theta = rng.uniform(-3, 3, size=(tokens, D // 2))
    f1 = np.repeat(np.cos(theta), 2, axis=1)
    f2 = np.stack([-np.sin(theta), np.sin(theta)], axis=2).reshape(tokens, D)
    y = np.concatenate(oracle.qk_norm_rope_fwd(qk, f1, f2, hq), axis=1)
    z = (n[..., 0::2] + 1j * n[..., 1::2]) * np.exp(1j * theta)[:, None, :]
    if not (np.allclose(y[..., 0::2], z.real, atol=1e-12) and np.allclose(y[..., 1::2], z.imag, atol=1e-12)):
        return False
    f1, f2 = rng.standard_normal((tokens, D)), rng.standard_normal((tokens, D))
    gq, gk = rng.standard_normal((tokens, hq, D)), rng.standard_normal((tokens, hk, D))
    dqk = oracle.qk_norm_rope_bwd(gq, gk, qk, f1, f2)
    h = 1e-6
    for idx in np.ndindex(qk.shape):
        xp, xm = qk.copy(), qk.copy()
        xp[idx] += h
        xm[idx] -= h
        lp = sum(float(np.sum(a * g)) for a, g in zip(oracle.qk_norm_rope_fwd(xp, f1, f2, hq), (gq, gk)))
        lm = sum(float(np.sum(a * g)) for a, g in zip(oracle.qk_norm_rope_fwd(xm, f1, f2, hq), (gq, gk)))
        if abs((lp - lm) / (2 * h) - dqk[idx]) > 1e-6 * max(1.0, abs(dqk[idx])):
            return False
    return True


def _pin_cross():
    """Tq != Tk (fewer queries than keys, so that a planted length mix-up
    stays inside the buffers): torch float64 SDPA + autograd, and the
    sampled-row functions against the full ones."""
    rng = np.random.default_rng(9)
    for (B, Tq, Tk, H, HKV, D) in ((2, 3, 8, 4, 2, 3), (1, 5, 7, 2, 1, 4)):
        Q, K, V, dO = (rng.standard_normal(s) for s in ((B, Tq, H, D), (B, Tk, HKV, D), (B, Tk, HKV, D), (B, Tq, H, D)))
        O, LSE = oracle.fwd(Q, K, V, 0.6, False, 0)
        dQ, dK, dV, _ = oracle.bwd(Q, K, V, dO, 0.6, False, 0)
        q, k, v = (torch.tensor(x).permute(0, 2, 1, 3).requires_grad_(True) for x in (Q, K, V))
        o = torch.nn.functional.scaled_dot_product_attention(q, k, v, scale=0.6, enable_gqa=True)
        o.backward(torch.tensor(dO).permute(0, 2, 1, 3))
        refs = [o.detach()] + [t.grad for t in (q, k, v)]
        for a, r in zip((O, dQ, dK, dV), refs):
            if not np.allclose(a, r.permute(0, 2, 1, 3).numpy(), rtol=0, atol=1e-10):
                return False
        cols = [0, Tk - 1]
        for h in range(H):
            o_r, l_r = oracle.fwd_rows(Q, K, V, 0.6, False, 0, 0, h, [Tq - 1])
            dq_r, _ = oracle.dq_rows(Q, K, V, dO, 0.6, False, 0, 0, h, [Tq - 1])
            if not (np.allclose(o_r, O[0, [Tq - 1], h], atol=1e-12) and np.allclose(l_r, LSE[0, h, [Tq - 1]], atol=1e-12)
                    and np.allclose(dq_r, dQ[0, [Tq - 1], h], atol=1e-12)):
                return False
        for g in range(HKV):
            dk_r, dv_r = oracle.dkdv_rows(Q, K, V, dO, 0.6, False, 0, 0, g, cols)
            if not (np.allclose(dk_r, dK[0, cols, g], atol=1e-12) and np.allclose(dv_r, dV[0, cols, g], atol=1e-12)):
                return False
    return True


def _pin_prologue_options():
    """Paired heads relocate base outputs; key offset shifts the stationary
    key dims by one token; both backward modes match finite differences."""
    rng = np.random.default_rng(10)
    tokens, heads, D, rot = 3, 4, 4, 2
    qk = rng.standard_normal((tokens, 2 * heads, D))
    f1, f2 = rng.standard_normal((tokens, 2 * D)), rng.standard_normal((tokens, 2 * D))
    q, k = oracle.qk_norm_rope_fwd_opt(qk, f1, f2, heads, D, True, False)
    for half in (0, 1):
        bq, bk = oracle.qk_norm_rope_fwd(qk, f1[:, half * D:(half + 1) * D], f2[:, half * D:(half + 1) * D], heads)
        for t in range(tokens):
            for h in range(half, heads, 2):
                pos = (2 * t + h // (heads // 2), h % (heads // 2))
                if not (np.allclose(q[pos], bq[t, h], atol=1e-13) and np.allclose(k[pos], bk[t, h], atol=1e-13)):
                    return False
    g1, g2 = f1[:, :D], f2[:, :D]
    q, k = oracle.qk_norm_rope_fwd_opt(qk, g1, g2, heads, rot, False, True)
    bq, bk = oracle.qk_norm_rope_fwd(qk, g1, g2, heads)
    _, nk = oracle.qk_norm_rope_fwd(qk, np.ones((tokens, D)), np.zeros((tokens, D)), heads)
    if not (np.allclose(q, bq, atol=1e-13) and np.allclose(k[0], bk[0], atol=1e-13)
            and np.allclose(k[1:, :, :rot], bk[1:, :, :rot], atol=1e-13)
            and np.allclose(k[1:, :, rot:], nk[:-1, :, rot:], atol=1e-13)):
        return False
    for paired, key_offset, a, b in ((True, False, f1, f2), (False, True, g1, g2)):
        shape = (2 * tokens, heads // 2, D) if paired else (tokens, heads, D)
        gq, gk = rng.standard_normal(shape), rng.standard_normal(shape)
        dqk = oracle.qk_norm_rope_bwd_opt(gq, gk, qk, a, b, heads, rot, paired, key_offset)
        h = 1e-6
        for idx in np.ndindex(qk.shape):
            xp, xm = qk.copy(), qk.copy()
            xp[idx] += h
            xm[idx] -= h
            lp = sum(float(np.sum(o * g)) for o, g in zip(oracle.qk_norm_rope_fwd_opt(xp, a, b, heads, rot, paired,
                                                                                       key_offset), (gq, gk)))
            lm = sum(float(np.sum(o * g)) for o, g in zip(oracle.qk_norm_rope_fwd_opt(xm, a, b, heads, rot, paired,
                                                                                       key_offset), (gq, gk)))
            if abs((lp - lm) / (2 * h) - dqk[idx]) > 1e-6 * max(1.0, abs(dqk[idx])):
                return False
    return True


PINS = {"sdpa+lse": _pin_sdpa, "rows": _pin_rows_match_full, "triu": _pin_triu, "fd": _pin_finite_differences,
        "prologue": _pin_prologue, "cross": _pin_cross, "prologue options": _pin_prologue_options}


def _failing_pins():
    failed = []
    for name, pin in PINS.items():
        try:
            ok = pin()
        except Exception:
            ok = False
        if not ok:
            failed.append(name)
    return failed


# (name, text in attn_oracle.c, replacement, which occurrence to replace)
MUTANTS = [
    ("score scale dropped", "S_row[j] = s->scale * dot(", "S_row[j] = dot(", 0),
    ("GQA map h % HKV", "const long g = h / (s->H / s->HKV);\n  const double* qi", "const long g = h % s->HKV;\n  const double* qi", 0),
    ("window off by one", "i - j >= s->window) return 0;", "i - j > s->window) return 0;", 0),
    ("causal drops diagonal", "if (s->causal && j > i) return 0;", "if (s->causal && j >= i) return 0;", 0),
    ("softmax not normalised", "S_row[j] = exp(S_row[j] - m) / l;", "S_row[j] = exp(S_row[j] - m);", 0),
    ("LSE without log", "return m + log(l);", "return m + l;", 0),
    ("Delta term dropped", "dSi[j] = Pi[j] * (dSi[j] - delta);", "dSi[j] = Pi[j] * dSi[j];", 0),
    ("dS sign flipped", "dSi[j] = Pi[j] * (dSi[j] - delta);", "dSi[j] = Pi[j] * (delta - dSi[j]);", 0),
    ("dQ without scale", "for (int d = 0; d < D; ++d) dqi[d] *= scale;", "", 0),
    ("dQ uses V", "const double* kj = K + kv_index(&s, b, j, g);\n            for (int d = 0; d < D; ++d) dqi[d]",
     "const double* kj = V + kv_index(&s, b, j, g);\n            for (int d = 0; d < D; ++d) dqi[d]", 0),
    ("dK without scale", "dkj[d] += scale * ds * qi[d];", "dkj[d] += ds * qi[d];", 0),
    ("dV from dS", "for (int d = 0; d < D; ++d) dvj[d] += p * doi[d];", "for (int d = 0; d < D; ++d) dvj[d] += ds * doi[d];", 0),
    ("P transposed in dK/dV", "const double p = P[(size_t)i * Tk + j];", "const double p = P[(size_t)j * Tk + i];", 0),
    ("dP reads the wrong V row", "dot(doi, V + kv_index(s, b, j, g), s->D)", "dot(doi, V + kv_index(s, b, i, g), s->D)", 0),
    ("triu wrap too small", "if (k > numCols - 1) k -= numRows + numCols;", "if (k > numCols - 1) k -= numCols;", 0),
    ("prologue partner d+1", "(x[d ^ 1] * rstd)", "(x[(d + 1) % D] * rstd)", 0),
    ("prologue eps dropped", "return 1.0 / sqrt(ms + kQkEps);", "return 1.0 / sqrt(ms);", 0),
    ("prologue norm correction dropped", "dx[e] = rstd * (gn[e] - (x[e] * rstd) * corr);", "dx[e] = rstd * gn[e];", 0),
    ("prologue grad partner factor", "f2[(size_t)t * D + (e ^ 1)] * g[e ^ 1]", "f2[(size_t)t * D + e] * g[e ^ 1]", 0),
    ("K row stride uses the query length", "return (((size_t)b * s->Tk + t) * s->HKV + g) * s->D;",
     "return (((size_t)b * s->T + t) * s->HKV + g) * s->D;", 0),
    ("scores over the query length", "for (long j = 0; j < s->Tk; ++j) {\n    if (visible(s, i, j))",
     "for (long j = 0; j < s->T; ++j) {\n    if (visible(s, i, j))", 0),
    ("probability rows strided by the query length", "double* row = P + (size_t)i * Tk;",
     "double* row = P + (size_t)i * T;", 0),
    ("dK/dV rows: Delta over the query length", "for (long j = 0; j < Tk; ++j) delta += P[j] * dP[j];",
     "for (long j = 0; j < T; ++j) delta += P[j] * dP[j];", 1),
    ("paired factor half ignored", "const double* a = f1 + (size_t)t * F + (paired ? (h % 2) * D : 0);\n"
     "      const double* b = f2 + (size_t)t * F + (paired ? (h % 2) * D : 0);\n      double* y",
     "const double* a = f1 + (size_t)t * F;\n      const double* b = f2 + (size_t)t * F;\n      double* y", 0),
    ("paired output token by head parity", "return ((size_t)(2 * t + h / half) * half + (h % half)) * D;",
     "return ((size_t)(2 * t + h % 2) * half + (h % half)) * D;", 0),
    ("key offset reads its own token", "const double* xp = qk + ((size_t)(t - 1) * 2 * heads + c) * D;",
     "const double* xp = qk + ((size_t)t * 2 * heads + c) * D;", 0),
    ("stationary gradient misses the next token", "gn[e] += dk[qk_out_index((int)t + 1, h, heads, D, paired) + e];",
     "gn[e] += 0.0;", 0),
    ("rotation gradient kept on shifted dims", "const int own = !shifted || t == 0 || e < rot;",
     "const int own = 1;", 0),
    ("row LSE missing in dq rows", "softmax_row(P, Tk);\n        dp_row(&s, V, dO, b, h, i, dP);\n        double delta",
     "dp_row(&s, V, dO, b, h, i, dP);\n        double delta", 0),
]


def _replace_nth(text, old, new, n):
    pos = -1
    for _ in range(n + 1):
        pos = text.find(old, pos + 1)
        if pos < 0:
            raise AssertionError(f"mutation anchor not found: {old!r}")
    return text[:pos] + new + text[pos + len(old):]


def test_unmodified_oracle_passes_the_battery():
    assert _failing_pins() == []


@pytest.mark.parametrize("name,old,new,nth", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(tmp_path, name, old, new, nth):
    src = _replace_nth(oracle.source(), old, new, nth)
    lib = os.path.join(tmp_path, "libmutant.so")
    oracle.compile_variant(src, lib)
    with oracle.use_library(lib):
        failed = _failing_pins()
    assert failed, f"mutant '{name}' passed every pin"
