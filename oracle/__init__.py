"""fp64 CPU oracle for causal / sliding-window GQA attention.

TEST INFRASTRUCTURE ONLY: the test-suite, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` use it.  The product package never imports it,
and it imports nothing from the product package.

The arithmetic lives in ``attn_oracle.c`` (plain C, IEEE double); this module
compiles it with gcc into ``oracle/_build/`` and wraps it with ctypes + numpy.
Every function takes and returns float64 numpy arrays in the layouts

    Q, O, dO, dQ : [B, Tq, H,   D]
    K, V, dK, dV : [B, Tk, HKV, D]      (Tk = Tq for self-attention)
    LSE, Delta   : [B, H, Tq]

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(closed forms, library routines, finite differences, the printed triu
diagrams); none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libattn_oracle.so")

_lib = None
_lock = threading.Lock()

_D = ctypes.POINTER(ctypes.c_double)
_I = ctypes.POINTER(ctypes.c_int)


def build(force: bool = False) -> str:
    """Compile attn_oracle.c into a shared library (gcc, -O2, OpenMP)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
            "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True, text=True)
    except subprocess.CalledProcessError:
        # OpenMP only spreads rows over cores; the arithmetic is identical.
        subprocess.run(base, check=True, capture_output=True, text=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _bind(lib):
    common = [ctypes.c_int] * 6 + [ctypes.c_double, ctypes.c_int, ctypes.c_int]  # B, Tq, Tk, H, HKV, D, ...
    lib.oracle_attn_probs.argtypes = [_D, _D] + common + [ctypes.c_int, ctypes.c_int, _D, _D]
    lib.oracle_attn_fwd.argtypes = [_D, _D, _D] + common + [_D, _D]
    lib.oracle_attn_bwd.argtypes = [_D, _D, _D, _D] + common + [_D, _D, _D, _D]
    lib.oracle_attn_fwd_rows.argtypes = [_D, _D, _D] + common + [
        ctypes.c_int, ctypes.c_int, _I, ctypes.c_int, _D, _D]
    lib.oracle_attn_dq_rows.argtypes = [_D, _D, _D, _D] + common + [
        ctypes.c_int, ctypes.c_int, _I, ctypes.c_int, _D, _D]
    lib.oracle_attn_dkdv_rows.argtypes = [_D, _D, _D, _D] + common + [
        ctypes.c_int, ctypes.c_int, _I, ctypes.c_int, _D, _D]
    lib.oracle_triu_offsets.argtypes = [ctypes.c_int, ctypes.c_int, _I, ctypes.c_int]
    lib.oracle_qk_norm_rope_fwd.argtypes = [_D, _D, _D, _D, _D] + [ctypes.c_int] * 4
    lib.oracle_qk_norm_rope_bwd.argtypes = [_D, _D, _D, _D, _D, _D] + [ctypes.c_int] * 4
    lib.oracle_qk_norm_rope_fwd_opt.argtypes = [_D, _D, _D, _D, _D] + [ctypes.c_int] * 6
    lib.oracle_qk_norm_rope_bwd_opt.argtypes = [_D, _D, _D, _D, _D, _D] + [ctypes.c_int] * 6
    for name in ("oracle_attn_probs", "oracle_attn_fwd", "oracle_attn_bwd",
                 "oracle_attn_fwd_rows", "oracle_attn_dq_rows",
                 "oracle_attn_dkdv_rows", "oracle_triu_offsets",
                 "oracle_qk_norm_rope_fwd", "oracle_qk_norm_rope_bwd",
                 "oracle_qk_norm_rope_fwd_opt", "oracle_qk_norm_rope_bwd_opt"):
        getattr(lib, name).restype = ctypes.c_int
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
    return _lib


def compile_variant(src: str, out_path: str) -> None:
    """Compile C source text (the oracle with a planted mistake, in the
    mutation tests) into a shared library at out_path."""
    src_path = out_path + ".c"
    with open(src_path, "w") as f:
        f.write(src)
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                    src_path, "-o", out_path, "-lm"], check=True, capture_output=True, text=True)


class use_library:
    """Context manager: route every function of this module to another build
    of the oracle (used only by the mutation tests)."""

    def __init__(self, path: str):
        self.path = path

    def __enter__(self):
        global _lib
        self._saved = _load()
        _lib = _bind(ctypes.CDLL(self.path))
        return self

    def __exit__(self, *exc):
        global _lib
        _lib = self._saved


def source() -> str:
    with open(_SRC) as f:
        return f.read()


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _p(a: np.ndarray):
    return a.ctypes.data_as(_D)


def _shape(Q, K):
    """(B, Tq, Tk, H, HKV, D); queries and keys may differ in length."""
    B, T, H, D = Q.shape
    Bk, Tk, HKV, Dk = K.shape
    if (Bk, Dk) != (B, D):
        raise ValueError(f"Q {Q.shape} and K {K.shape} disagree")
    return B, T, Tk, H, HKV, D


def _check(rc: int, what: str):
    if rc != 0:
        raise RuntimeError(f"{what} failed with status {rc}")


def probs(Q, K, scale, causal, window, b, h):
    """Full Tq x Tk probability matrix P of one (b, h), and its LSE row."""
    Q, K = _f64(Q), _f64(K)
    B, T, Tk, H, HKV, D = _shape(Q, K)
    P = np.empty((T, Tk), np.float64)
    lse = np.empty((T,), np.float64)
    _check(_load().oracle_attn_probs(_p(Q), _p(K), B, T, Tk, H, HKV, D, float(scale),
                                     int(causal), int(window), int(b), int(h),
                                     _p(P), _p(lse)), "oracle_attn_probs")
    return P, lse


def fwd(Q, K, V, scale, causal, window):
    """(O [B,Tq,H,D], LSE [B,H,Tq]) by the plain definition."""
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    B, T, Tk, H, HKV, D = _shape(Q, K)
    if V.shape != K.shape:
        raise ValueError(f"K {K.shape} and V {V.shape} disagree")
    O = np.empty_like(Q)
    LSE = np.empty((B, H, T), np.float64)
    _check(_load().oracle_attn_fwd(_p(Q), _p(K), _p(V), B, T, Tk, H, HKV, D, float(scale),
                                   int(causal), int(window), _p(O), _p(LSE)),
           "oracle_attn_fwd")
    return O, LSE


def bwd(Q, K, V, dO, scale, causal, window):
    """(dQ, dK, dV, Delta) by the analytic gradient of the definition."""
    Q, K, V, dO = _f64(Q), _f64(K), _f64(V), _f64(dO)
    B, T, Tk, H, HKV, D = _shape(Q, K)
    if V.shape != K.shape or dO.shape != Q.shape:
        raise ValueError("V must match K and dO must match Q")
    dQ = np.empty_like(Q)
    dK = np.empty_like(K)
    dV = np.empty_like(V)
    Delta = np.empty((B, H, T), np.float64)
    _check(_load().oracle_attn_bwd(_p(Q), _p(K), _p(V), _p(dO), B, T, Tk, H, HKV, D,
                                   float(scale), int(causal), int(window),
                                   _p(dQ), _p(dK), _p(dV), _p(Delta)),
           "oracle_attn_bwd")
    return dQ, dK, dV, Delta


def _rows(rows, T):
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int32))
    if r.ndim != 1 or (r.size and (r.min() < 0 or r.max() >= T)):
        raise ValueError("row indices out of range")
    return r


def fwd_rows(Q, K, V, scale, causal, window, b, h, rows):
    """O rows [n, D] and LSE [n] of query rows `rows` of one (b, h)."""
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    B, T, Tk, H, HKV, D = _shape(Q, K)
    r = _rows(rows, T)
    O = np.empty((r.size, D), np.float64)
    L = np.empty((r.size,), np.float64)
    _check(_load().oracle_attn_fwd_rows(_p(Q), _p(K), _p(V), B, T, Tk, H, HKV, D, float(scale),
                                        int(causal), int(window), int(b), int(h),
                                        r.ctypes.data_as(_I), r.size, _p(O), _p(L)),
           "oracle_attn_fwd_rows")
    return O, L


def dq_rows(Q, K, V, dO, scale, causal, window, b, h, rows):
    """dQ rows [n, D] and Delta [n] of query rows `rows` of one (b, h)."""
    Q, K, V, dO = _f64(Q), _f64(K), _f64(V), _f64(dO)
    B, T, Tk, H, HKV, D = _shape(Q, K)
    r = _rows(rows, T)
    dq = np.empty((r.size, D), np.float64)
    de = np.empty((r.size,), np.float64)
    _check(_load().oracle_attn_dq_rows(_p(Q), _p(K), _p(V), _p(dO), B, T, Tk, H, HKV, D,
                                       float(scale), int(causal), int(window), int(b), int(h),
                                       r.ctypes.data_as(_I), r.size, _p(dq), _p(de)),
           "oracle_attn_dq_rows")
    return dq, de


def dkdv_rows(Q, K, V, dO, scale, causal, window, b, g, cols):
    """dK rows and dV rows [n, D] of key rows `cols` of one (b, kv head g)."""
    Q, K, V, dO = _f64(Q), _f64(K), _f64(V), _f64(dO)
    B, T, Tk, H, HKV, D = _shape(Q, K)
    c = _rows(cols, Tk)
    dk = np.empty((c.size, D), np.float64)
    dv = np.empty((c.size, D), np.float64)
    _check(_load().oracle_attn_dkdv_rows(_p(Q), _p(K), _p(V), _p(dO), B, T, Tk, H, HKV, D,
                                         float(scale), int(causal), int(window), int(b), int(g),
                                         c.ctypes.data_as(_I), c.size, _p(dk), _p(dv)),
           "oracle_attn_dkdv_rows")
    return dk, dv


def triu_offsets(num_rows: int, num_cols: int) -> list[int]:
    """Diagonal-crossing block offsets, in the order the block walk meets them."""
    cap = 4 * (num_rows + num_cols) + 8
    out = (ctypes.c_int * cap)()
    n = _load().oracle_triu_offsets(int(num_rows), int(num_cols), out, cap)
    if n < 0 or n > cap:
        raise RuntimeError(f"oracle_triu_offsets({num_rows}, {num_cols}) returned {n}")
    return [out[i] for i in range(n)]


def qk_norm_rope_fwd(qk, f1, f2, hq: int):
    """Pre-attention prologue: (q [tokens, hq, D], k [tokens, hk, D]) from the
    packed projection qk [tokens, hq + hk, D] and the rotary factors
    f1, f2 [tokens, D]: RMS-norm of every head vector, then
    y_d = f1_d n_d + f2_d n_(d xor 1)."""
    qk, f1, f2 = _f64(qk), _f64(f1), _f64(f2)
    tokens, heads, D = qk.shape
    hk = heads - int(hq)
    q = np.empty((tokens, hq, D), np.float64)
    k = np.empty((tokens, hk, D), np.float64)
    _check(_load().oracle_qk_norm_rope_fwd(_p(qk), _p(f1), _p(f2), _p(q), _p(k), tokens, int(hq), hk, D),
           "oracle_qk_norm_rope_fwd")
    return q, k


def qk_norm_rope_bwd(dq, dk, qk, f1, f2):
    """Gradient of the packed projection qk given the gradients of q and k."""
    dq, dk, qk, f1, f2 = _f64(dq), _f64(dk), _f64(qk), _f64(f1), _f64(f2)
    tokens, heads, D = qk.shape
    hq, hk = dq.shape[1], dk.shape[1]
    if hq + hk != heads:
        raise ValueError("dq and dk heads do not add up to qk's")
    dqk = np.empty_like(qk)
    _check(_load().oracle_qk_norm_rope_bwd(_p(dq), _p(dk), _p(qk), _p(f1), _p(f2), _p(dqk), tokens, hq, hk, D),
           "oracle_qk_norm_rope_bwd")
    return dqk


def qk_norm_rope_fwd_opt(qk, f1, f2, heads: int, rot: int, paired: bool, key_offset: bool):
    """(q, k) of the prologue with equally many query and key heads and the
    paired-heads or key-offset option: each [tokens, heads, D], or
    [2*tokens, heads/2, D] when paired (factor rows then 2*D wide)."""
    qk, f1, f2 = _f64(qk), _f64(f1), _f64(f2)
    tokens, heads2, D = qk.shape
    if heads2 != 2 * heads:
        raise ValueError("qk must hold 2*heads heads")
    shape = (2 * tokens, heads // 2, D) if paired else (tokens, heads, D)
    q = np.empty(shape, np.float64)
    k = np.empty(shape, np.float64)
    _check(_load().oracle_qk_norm_rope_fwd_opt(_p(qk), _p(f1), _p(f2), _p(q), _p(k), tokens, int(heads), D,
                                               int(rot), int(bool(paired)), int(bool(key_offset))),
           "oracle_qk_norm_rope_fwd_opt")
    return q, k


def qk_norm_rope_bwd_opt(dq, dk, qk, f1, f2, heads: int, rot: int, paired: bool, key_offset: bool):
    """Gradient of qk for qk_norm_rope_fwd_opt given the gradients of q and k."""
    dq, dk, qk, f1, f2 = _f64(dq), _f64(dk), _f64(qk), _f64(f1), _f64(f2)
    tokens, heads2, D = qk.shape
    if heads2 != 2 * heads:
        raise ValueError("qk must hold 2*heads heads")
    dqk = np.empty_like(qk)
    _check(_load().oracle_qk_norm_rope_bwd_opt(_p(dq), _p(dk), _p(qk), _p(f1), _p(f2), _p(dqk), tokens,
                                               int(heads), D, int(rot), int(bool(paired)),
                                               int(bool(key_offset))),
           "oracle_qk_norm_rope_bwd_opt")
    return dqk
