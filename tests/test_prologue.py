"""Pre-attention prologue (QK RMS-norm + rotary, forward and backward).

CPU: the fp64 oracle functions are pinned by properties that do not restate
their formula:
  * rotary factors (cos, -sin / cos, +sin) over each lane pair turn the
    normalised pair into complex multiplication by e^(i theta);
  * identity factors leave a vector whose mean square is ms / (ms + eps);
  * swap factors (f1 = 0, f2 = 1) exchange the two lanes of every pair;
  * the output does not depend on the input's scale (up to eps);
  * the backward equals central finite differences of sum(q*Gq) + sum(k*Gk).
GPU: the CUDA kernels against the oracle, element by element (q, k: the
exact value rounded once to the 16-bit output, |err| <= half an ulp of it
plus 1e-4 for fp32 arithmetic; dqk: relative Frobenius <= 2e-2), and the C
ABI's argument checks.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle

EPS = 1.1920928955078125e-7


def _inputs(tokens, hq, hk, D, seed, scale=1.0):
    rng = np.random.default_rng(seed)
    qk = rng.standard_normal((tokens, hq + hk, D)) * scale
    f1 = rng.standard_normal((tokens, D))
    f2 = rng.standard_normal((tokens, D))
    return qk, f1, f2


def test_rotary_factors_are_complex_rotation():
    tokens, hq, hk, D = 5, 2, 1, 8
    qk, _, _ = _inputs(tokens, hq, hk, D, 1)
    theta = np.random.default_rng(2).uniform(-np.pi, np.pi, size=(tokens, D // 2))
    f1 = np.repeat(np.cos(theta), 2, axis=1)
    f2 = np.stack([-np.sin(theta), np.sin(theta)], axis=2).reshape(tokens, D)
    q, k = oracle.qk_norm_rope_fwd(qk, f1, f2, hq)
    y = np.concatenate([q, k], axis=1)
    # identity factors give the normalised vector itself
    n = np.concatenate(oracle.qk_norm_rope_fwd(qk, np.ones((tokens, D)), np.zeros((tokens, D)), hq), axis=1)
    z = (n[..., 0::2] + 1j * n[..., 1::2]) * np.exp(1j * theta)[:, None, :]
    np.testing.assert_allclose(y[..., 0::2], z.real, rtol=0, atol=1e-12)
    np.testing.assert_allclose(y[..., 1::2], z.imag, rtol=0, atol=1e-12)
    np.testing.assert_allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(n, axis=-1), rtol=1e-12)


def test_identity_factors_give_unit_rms():
    tokens, hq, hk, D = 4, 3, 2, 16
    for scale in (1.0, 1e-3):
        qk, _, _ = _inputs(tokens, hq, hk, D, 3, scale)
        n = np.concatenate(oracle.qk_norm_rope_fwd(qk, np.ones((tokens, D)), np.zeros((tokens, D)), hq), axis=1)
        ms = np.mean(qk ** 2, axis=-1)
        np.testing.assert_allclose(np.mean(n ** 2, axis=-1), ms / (ms + EPS), rtol=1e-12)
        # direction kept: n is a positive multiple of x
        cos = np.sum(n * qk, -1) / (np.linalg.norm(n, axis=-1) * np.linalg.norm(qk, axis=-1))
        np.testing.assert_allclose(cos, 1.0, rtol=0, atol=1e-12)


def test_swap_factors_exchange_pair_lanes():
    tokens, hq, hk, D = 3, 2, 2, 8
    qk, _, _ = _inputs(tokens, hq, hk, D, 4)
    n = np.concatenate(oracle.qk_norm_rope_fwd(qk, np.ones((tokens, D)), np.zeros((tokens, D)), hq), axis=1)
    y = np.concatenate(oracle.qk_norm_rope_fwd(qk, np.zeros((tokens, D)), np.ones((tokens, D)), hq), axis=1)
    np.testing.assert_array_equal(y[..., 0::2], n[..., 1::2])
    np.testing.assert_array_equal(y[..., 1::2], n[..., 0::2])


def test_scale_invariance():
    qk, f1, f2 = _inputs(6, 2, 2, 8, 5)
    a = np.concatenate(oracle.qk_norm_rope_fwd(qk, f1, f2, 2), axis=1)
    b = np.concatenate(oracle.qk_norm_rope_fwd(qk * 7.5, f1, f2, 2), axis=1)
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-6)


def test_backward_matches_finite_differences():
    tokens, hq, hk, D = 2, 2, 1, 6
    qk, f1, f2 = _inputs(tokens, hq, hk, D, 6)
    rng = np.random.default_rng(7)
    gq = rng.standard_normal((tokens, hq, D))
    gk = rng.standard_normal((tokens, hk, D))
    dqk = oracle.qk_norm_rope_bwd(gq, gk, qk, f1, f2)

    def loss(x):
        q, k = oracle.qk_norm_rope_fwd(x, f1, f2, hq)
        return float(np.sum(q * gq) + np.sum(k * gk))

    h = 1e-6
    for idx in np.ndindex(qk.shape):
        xp, xm = qk.copy(), qk.copy()
        xp[idx] += h
        xm[idx] -= h
        fd = (loss(xp) - loss(xm)) / (2 * h)
        assert abs(fd - dqk[idx]) <= 1e-6 * max(1.0, abs(dqk[idx])), (idx, fd, dqk[idx])


# ------------------------------------------ options: paired heads, key offset
#
# Pinned against the base mode (itself pinned above) and finite differences:
#   * paired: output (t, h) is the base output of (t, h) computed with factor
#     half h mod 2, stored at token 2t + h div (heads/2), head h mod (heads/2);
#   * key offset: queries and token 0 equal the base output; a later key
#     row's rotating dims equal the base output and its stationary dims the
#     previous token's normalised values (the base output under identity
#     factors);
#   * both backward modes equal central differences of the forward.


def _opt_inputs(tokens, heads, D, seed, paired):
    rng = np.random.default_rng(seed)
    qk = rng.standard_normal((tokens, 2 * heads, D))
    F = 2 * D if paired else D
    return qk, rng.standard_normal((tokens, F)), rng.standard_normal((tokens, F))


def test_paired_heads_relocate_base_outputs():
    tokens, heads, D = 3, 4, 6
    qk, f1, f2 = _opt_inputs(tokens, heads, D, 21, True)
    q, k = oracle.qk_norm_rope_fwd_opt(qk, f1, f2, heads, D, True, False)
    assert q.shape == (2 * tokens, heads // 2, D)
    for half in (0, 1):
        bq, bk = oracle.qk_norm_rope_fwd(qk, f1[:, half * D:(half + 1) * D], f2[:, half * D:(half + 1) * D], heads)
        for t in range(tokens):
            for h in range(half, heads, 2):
                pos = (2 * t + h // (heads // 2), h % (heads // 2))
                np.testing.assert_array_equal(q[pos], bq[t, h])
                np.testing.assert_array_equal(k[pos], bk[t, h])


@pytest.mark.parametrize("rot", [0, 2, 4, 8])
def test_key_offset_shifts_stationary_key_dims(rot):
    tokens, heads, D = 4, 2, 8
    qk, f1, f2 = _opt_inputs(tokens, heads, D, 22 + rot, False)
    q, k = oracle.qk_norm_rope_fwd_opt(qk, f1, f2, heads, rot, False, True)
    bq, bk = oracle.qk_norm_rope_fwd(qk, f1, f2, heads)
    _, nk = oracle.qk_norm_rope_fwd(qk, np.ones((tokens, D)), np.zeros((tokens, D)), heads)
    np.testing.assert_array_equal(q, bq)
    np.testing.assert_array_equal(k[0], bk[0])
    np.testing.assert_array_equal(k[1:, :, :rot], bk[1:, :, :rot])
    np.testing.assert_allclose(k[1:, :, rot:], nk[:-1, :, rot:], rtol=0, atol=1e-15)


@pytest.mark.parametrize("paired,key_offset,rot", [(False, False, 4), (True, False, 4), (False, True, 2),
                                                    (False, True, 0), (False, True, 4)])
def test_option_backward_matches_finite_differences(paired, key_offset, rot):
    tokens, heads, D = 3, 2, 4
    qk, f1, f2 = _opt_inputs(tokens, heads, D, 23 + rot, paired)
    rng = np.random.default_rng(24)
    shape = (2 * tokens, heads // 2, D) if paired else (tokens, heads, D)
    gq, gk = rng.standard_normal(shape), rng.standard_normal(shape)
    dqk = oracle.qk_norm_rope_bwd_opt(gq, gk, qk, f1, f2, heads, rot, paired, key_offset)

    def loss(x):
        q, k = oracle.qk_norm_rope_fwd_opt(x, f1, f2, heads, rot, paired, key_offset)
        return float(np.sum(q * gq) + np.sum(k * gk))

    h = 1e-6
    for idx in np.ndindex(qk.shape):
        xp, xm = qk.copy(), qk.copy()
        xp[idx] += h
        xm[idx] -= h
        fd = (loss(xp) - loss(xm)) / (2 * h)
        assert abs(fd - dqk[idx]) <= 1e-6 * max(1.0, abs(dqk[idx])), (idx, fd, dqk[idx])


def test_options_reject_invalid_combinations():
    qk, f1, f2 = _opt_inputs(2, 2, 4, 25, False)
    with pytest.raises(RuntimeError):
        oracle.qk_norm_rope_fwd_opt(qk, f1, f2, 2, 2, True, True)  # both options
    with pytest.raises(RuntimeError):
        oracle.qk_norm_rope_fwd_opt(qk, f1, f2, 2, 3, False, True)  # odd rotary dim


# ------------------------------------------------------------------ GPU

def _dev():
    from flash_attention_attn_gb300.build import build
    build()
    return torch.device("cuda", 0)


CASES = [(37, 4, 2, 64, torch.bfloat16), (64, 2, 2, 128, torch.bfloat16), (19, 8, 1, 128, torch.float16),
         (5, 1, 1, 64, torch.float16)]


@pytest.mark.gpu
@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0]}-{c[1]}-{c[2]}-{c[3]}-{str(c[4])[6:]}")
def test_gpu_matches_oracle(case):
    import flash_attention_attn_gb300 as fa
    tokens, hq, hk, D, dt = case
    dev = _dev()
    qk, f1, f2 = _inputs(tokens, hq, hk, D, 100 + tokens)
    rng = np.random.default_rng(200 + tokens)
    gq = rng.standard_normal((tokens, hq, D))
    gk = rng.standard_normal((tokens, hk, D))
    # the GPU gets the rounded 16-bit values; the oracle gets the same values exactly
    qk_t = torch.tensor(qk, dtype=torch.float32).to(dt)
    gq_t = torch.tensor(gq, dtype=torch.float32).to(dt)
    gk_t = torch.tensor(gk, dtype=torch.float32).to(dt)
    f1_t = torch.tensor(f1, dtype=torch.float32)
    f2_t = torch.tensor(f2, dtype=torch.float32)
    q, k = fa.qk_norm_rope_fwd(qk_t.to(dev), f1_t.to(dev), f2_t.to(dev), hq)
    dqk = fa.qk_norm_rope_bwd(gq_t.to(dev), gk_t.to(dev), qk_t.to(dev), f1_t.to(dev), f2_t.to(dev))
    torch.cuda.synchronize()
    x64 = qk_t.double().numpy()
    Q, K = oracle.qk_norm_rope_fwd(x64, f1, f2, hq)
    dX = oracle.qk_norm_rope_bwd(gq_t.double().numpy(), gk_t.double().numpy(), x64, f1, f2)
    # the 16-bit outputs are the exact values rounded once: relative error of
    # at most half an ulp (2^-8 for bf16, 2^-11 for fp16) plus fp32 arithmetic
    half_ulp = 2.0 ** -8 if dt == torch.bfloat16 else 2.0 ** -11
    for got, ref in ((q, Q), (k, K)):
        err = np.abs(got.double().cpu().numpy() - ref)
        assert np.all(err <= half_ulp * np.abs(ref) + 1e-4), float(np.max(err - half_ulp * np.abs(ref)))
    got = dqk.double().cpu().numpy()
    assert np.linalg.norm(got - dX) / np.linalg.norm(dX) <= 2e-2


OPT_CASES = [  # tokens, heads, D, rot, paired, key_offset, dtype
    (37, 4, 64, 0, True, False, torch.bfloat16),
    (19, 2, 128, 0, True, False, torch.float16),
    (33, 2, 64, 32, False, True, torch.bfloat16),
    (9, 3, 128, 96, False, True, torch.float16),
    (5, 2, 64, 0, False, True, torch.bfloat16),     # every dim stationary
    (12, 2, 128, 128, False, True, torch.bfloat16),  # no stationary dim: the plain prologue
    (21, 3, 64, 0, False, False, torch.bfloat16),    # neither option
]


@pytest.mark.gpu
@pytest.mark.parametrize("case", OPT_CASES, ids=lambda c: "-".join(str(x) for x in c[:6]) + "-" + str(c[6])[6:])
def test_gpu_options_match_oracle(case):
    import flash_attention_attn_gb300 as fa
    tokens, heads, D, rot, paired, key_offset, dt = case
    dev = _dev()
    qk, f1, f2 = _opt_inputs(tokens, heads, D, 300 + tokens, paired)
    shape = (2 * tokens, heads // 2, D) if paired else (tokens, heads, D)
    rng = np.random.default_rng(400 + tokens)
    gq, gk = rng.standard_normal(shape), rng.standard_normal(shape)
    qk_t = torch.tensor(qk, dtype=torch.float32).to(dt)
    gq_t = torch.tensor(gq, dtype=torch.float32).to(dt)
    gk_t = torch.tensor(gk, dtype=torch.float32).to(dt)
    f1_t, f2_t = (torch.tensor(f, dtype=torch.float32) for f in (f1, f2))
    q, k = fa.qk_norm_rope_fwd_opt(qk_t.to(dev), f1_t.to(dev), f2_t.to(dev), heads, rot, paired, key_offset)
    dqk = fa.qk_norm_rope_bwd_opt(gq_t.to(dev), gk_t.to(dev), qk_t.to(dev), f1_t.to(dev), f2_t.to(dev), heads, rot,
                                  paired, key_offset)
    torch.cuda.synchronize()
    x64 = qk_t.double().numpy()
    Q, K = oracle.qk_norm_rope_fwd_opt(x64, f1, f2, heads, rot, paired, key_offset)
    dX = oracle.qk_norm_rope_bwd_opt(gq_t.double().numpy(), gk_t.double().numpy(), x64, f1, f2, heads, rot, paired,
                                     key_offset)
    half_ulp = 2.0 ** -8 if dt == torch.bfloat16 else 2.0 ** -11
    for got, ref in ((q, Q), (k, K)):
        err = np.abs(got.double().cpu().numpy() - ref)
        assert np.all(err <= half_ulp * np.abs(ref) + 1e-4), float(np.max(err - half_ulp * np.abs(ref)))
    got = dqk.double().cpu().numpy()
    assert np.linalg.norm(got - dX) / np.linalg.norm(dX) <= 2e-2


def test_abi_argument_checks():
    from flash_attention_attn_gb300 import _binding as fb
    from flash_attention_attn_gb300.build import build
    build()
    fake = 0x10000
    ok_args = dict(tokens=4, hq=2, hk=2, head_dim=64, dtype=fb.FA_DTYPE_BF16)

    def fwd(ptrs=None, **kw):
        a = dict(ok_args, **kw)
        p = ptrs or [fake] * 5
        return fb.fa_qk_norm_rope_fwd(*p, a["tokens"], a["hq"], a["hk"], a["head_dim"], a["dtype"], None)

    assert fwd(tokens=0) == fb.FA_ERR_INVALID_ARG
    assert fwd(hk=0) == fb.FA_ERR_INVALID_ARG
    assert fwd(head_dim=96) == fb.FA_ERR_UNSUPPORTED
    assert fwd(dtype=fb.FA_DTYPE_FP32) == fb.FA_ERR_UNSUPPORTED
    assert fwd(ptrs=[fake, 0, fake, fake, fake]) == fb.FA_ERR_INVALID_ARG
    assert fwd(ptrs=[fake, fake, fake + 4, fake, fake]) == fb.FA_ERR_INVALID_ARG
    p = [fake] * 6
    assert fb.fa_qk_norm_rope_bwd(*p, 4, 2, 2, 100, fb.FA_DTYPE_BF16, None) == fb.FA_ERR_UNSUPPORTED
    if not torch.cuda.is_available():
        assert fwd() in (fb.FA_ERR_CUDA, fb.FA_ERR_UNSUPPORTED)  # no device: an error, never a fallback


def test_abi_option_argument_checks():
    from flash_attention_attn_gb300 import _binding as fb
    from flash_attention_attn_gb300.build import build
    build()
    fake = 0x10000

    def fwd(tokens=4, heads=2, D=64, rot=32, paired=0, key_offset=1, dtype=fb.FA_DTYPE_BF16, ptrs=None):
        p = ptrs or [fake] * 5
        return fb.fa_qk_norm_rope_fwd_opt(*p, tokens, heads, D, rot, paired, key_offset, dtype, None)

    assert fwd(tokens=0) == fb.FA_ERR_INVALID_ARG
    assert fwd(paired=1, key_offset=1) == fb.FA_ERR_INVALID_ARG  # the options are exclusive
    assert fwd(paired=1, key_offset=0, heads=3) == fb.FA_ERR_INVALID_ARG
    assert fwd(rot=33) == fb.FA_ERR_INVALID_ARG
    assert fwd(rot=66) == fb.FA_ERR_INVALID_ARG
    assert fwd(rot=-2) == fb.FA_ERR_INVALID_ARG
    assert fwd(D=96) == fb.FA_ERR_UNSUPPORTED
    assert fwd(dtype=fb.FA_DTYPE_FP32) == fb.FA_ERR_UNSUPPORTED
    assert fwd(ptrs=[fake, fake, fake + 4, fake, fake]) == fb.FA_ERR_INVALID_ARG
    p = [fake] * 6
    assert fb.fa_qk_norm_rope_bwd_opt(*p, 4, 2, 64, 0, 1, 1, fb.FA_DTYPE_BF16, None) == fb.FA_ERR_INVALID_ARG
    assert fb.fa_qk_norm_rope_bwd_opt(*p, 4, 2, 64, 3, 0, 1, fb.FA_DTYPE_BF16, None) == fb.FA_ERR_INVALID_ARG
    if not torch.cuda.is_available():
        assert fwd() in (fb.FA_ERR_CUDA, fb.FA_ERR_UNSUPPORTED)
