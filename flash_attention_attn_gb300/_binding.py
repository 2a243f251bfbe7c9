"""ctypes binding of libfa_gb300.so (the C ABI in include/fa.h).

Argument marshalling only: every attention step runs in the library's CUDA
kernels.  The library is loaded on first use and a missing or unbuildable
library raises immediately; there is no fallback implementation.

Two layers:
* ``fa_*`` functions with the C names and arguments (integers for pointers
  and the stream), returning the C status code;
* ``attention_fwd`` / ``attention_bwd`` for torch CUDA tensors, which
  allocate outputs and the workspace with torch and raise ``FaError`` on a
  nonzero status.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "libfa_gb300.so")

FA_OK = 0
FA_ERR_INVALID_ARG = 1
FA_ERR_UNSUPPORTED = 2
FA_ERR_CUDA = 3
FA_ERR_TIMEOUT = 4
FA_ERR_WORKSPACE = 5
FA_DTYPE_BF16 = 0
FA_DTYPE_FP32 = 1
FA_DTYPE_FP16 = 2
FA_OP_FWD = 0
FA_OP_BWD = 1
FA_OP_BWD_FUSED = 2

_lib = None
_lock = threading.Lock()

_vp = ctypes.c_void_p
_i = ctypes.c_int
_f = ctypes.c_float
_sz = ctypes.c_size_t


class FaError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {fa_status_string(status)} (status {status})")


def load(build_if_missing: bool = False) -> ctypes.CDLL:
    """Load the library (optionally building it first); raise if it is absent."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            if not build_if_missing:
                raise RuntimeError(
                    f"{LIB_PATH} is not built; run `python -c \"import __graft_entry__ as g; g.build()\"` "
                    "(there is no CPU fallback)")
            from .build import build
            build()
        lib = ctypes.CDLL(LIB_PATH)
        lib.fa_workspace_size.argtypes = [_i] * 7
        lib.fa_workspace_size.restype = _sz
        lib.fa_fwd.argtypes = [_vp] * 5 + [_i] * 5 + [_f, _i, _i, _i, _vp, _sz, _vp]
        lib.fa_fwd.restype = _i
        lib.fa_bwd.argtypes = [_vp] * 9 + [_i] * 5 + [_f, _i, _i, _i, _vp, _sz, _vp]
        lib.fa_bwd.restype = _i
        lib.fa_fwd_cross.argtypes = [_vp] * 5 + [_i] * 6 + [_f, _i, _vp, _sz, _vp]
        lib.fa_fwd_cross.restype = _i
        lib.fa_bwd_cross.argtypes = [_vp] * 9 + [_i] * 6 + [_f, _i, _vp, _sz, _vp]
        lib.fa_bwd_cross.restype = _i
        lib.fa_bwd_preprocess.argtypes = [_vp, _vp] + [_i] * 6 + [_vp, _sz, _vp]
        lib.fa_bwd_preprocess.restype = _i
        lib.fa_bwd_dkdv.argtypes = [_vp] * 7 + [_i] * 5 + [_f, _i, _i, _i, _vp, _sz, _vp]
        lib.fa_bwd_dkdv.restype = _i
        lib.fa_bwd_dq.argtypes = [_vp] * 6 + [_i] * 5 + [_f, _i, _i, _i, _vp, _sz, _vp]
        lib.fa_bwd_dq.restype = _i
        lib.fa_bwd_dkdv_dq.argtypes = [_vp] * 8 + [_i] * 5 + [_f, _i, _i, _i, _vp, _sz, _vp]
        lib.fa_bwd_dkdv_dq.restype = _i
        lib.fa_check_status.argtypes = [_vp, _vp, ctypes.POINTER(ctypes.c_uint)]
        lib.fa_check_status.restype = _i
        lib.fa_status_string.argtypes = [_i]
        lib.fa_status_string.restype = ctypes.c_char_p
        for name in ("fa_plan_kv_range", "fa_plan_q_range"):
            getattr(lib, name).argtypes = [_i] * 6 + [ctypes.POINTER(_i), ctypes.POINTER(_i)]
            getattr(lib, name).restype = _i
        lib.fa_plan_block_mask.argtypes = [_i] * 7
        for name in ("fa_plan_row_keys", "fa_plan_key_rows"):
            getattr(lib, name).argtypes = [_i] * 5 + [ctypes.POINTER(_i), ctypes.POINTER(_i)]
            getattr(lib, name).restype = _i
        lib.fa_plan_block_mask.restype = _i
        lib.fa_tile_m.argtypes = []
        lib.fa_tile_m.restype = _i
        lib.fa_tile_n.argtypes = []
        lib.fa_tile_n.restype = _i
        lib.fa_debug_config.argtypes = [ctypes.c_ulonglong, _i]
        lib.fa_debug_config.restype = _i
        lib.fa_debug_fwd_tiles.argtypes = [_i]
        lib.fa_debug_fwd_tiles.restype = _i
        lib.fa_debug_max_ctas.argtypes = [_i]
        lib.fa_debug_max_ctas.restype = _i
        lib.fa_qk_norm_rope_fwd.argtypes = [_vp] * 5 + [_i] * 5 + [_vp]
        lib.fa_qk_norm_rope_fwd.restype = _i
        lib.fa_qk_norm_rope_bwd.argtypes = [_vp] * 6 + [_i] * 5 + [_vp]
        lib.fa_qk_norm_rope_bwd.restype = _i
        lib.fa_qk_norm_rope_fwd_opt.argtypes = [_vp] * 5 + [_i] * 7 + [_vp]
        lib.fa_qk_norm_rope_fwd_opt.restype = _i
        lib.fa_qk_norm_rope_bwd_opt.argtypes = [_vp] * 6 + [_i] * 7 + [_vp]
        lib.fa_qk_norm_rope_bwd_opt.restype = _i
        _lib = lib
        return lib


# ------------------------------------------------------------- C-named layer

def fa_workspace_size(op, B, T, H, HKV, head_dim, dtype) -> int:
    return load().fa_workspace_size(op, B, T, H, HKV, head_dim, dtype)


def fa_fwd(Q, K, V, O, LSE, B, T, H, HKV, head_dim, scale, causal, window, dtype,
           workspace, workspace_bytes, stream) -> int:
    return load().fa_fwd(Q, K, V, O, LSE, B, T, H, HKV, head_dim, scale, causal, window, dtype,
                         workspace, workspace_bytes, stream)


def fa_bwd(Q, K, V, O, LSE, dO, dQ, dK, dV, B, T, H, HKV, head_dim, scale, causal, window, dtype,
           workspace, workspace_bytes, stream) -> int:
    return load().fa_bwd(Q, K, V, O, LSE, dO, dQ, dK, dV, B, T, H, HKV, head_dim, scale, causal,
                         window, dtype, workspace, workspace_bytes, stream)


def fa_fwd_cross(Q, K, V, O, LSE, B, Tq, Tk, H, HKV, head_dim, scale, dtype, workspace, workspace_bytes,
                 stream) -> int:
    return load().fa_fwd_cross(Q, K, V, O, LSE, B, Tq, Tk, H, HKV, head_dim, scale, dtype, workspace,
                               workspace_bytes, stream)


def fa_bwd_cross(Q, K, V, O, LSE, dO, dQ, dK, dV, B, Tq, Tk, H, HKV, head_dim, scale, dtype, workspace,
                 workspace_bytes, stream) -> int:
    return load().fa_bwd_cross(Q, K, V, O, LSE, dO, dQ, dK, dV, B, Tq, Tk, H, HKV, head_dim, scale, dtype,
                               workspace, workspace_bytes, stream)


def fa_bwd_preprocess(O, dO, B, T, H, HKV, head_dim, dtype, workspace, workspace_bytes, stream) -> int:
    return load().fa_bwd_preprocess(O, dO, B, T, H, HKV, head_dim, dtype, workspace, workspace_bytes, stream)


def fa_bwd_dkdv(Q, K, V, LSE, dO, dK, dV, B, T, H, HKV, head_dim, scale, causal, window, dtype,
                workspace, workspace_bytes, stream) -> int:
    return load().fa_bwd_dkdv(Q, K, V, LSE, dO, dK, dV, B, T, H, HKV, head_dim, scale, causal, window,
                              dtype, workspace, workspace_bytes, stream)


def fa_bwd_dq(Q, K, V, LSE, dO, dQ, B, T, H, HKV, head_dim, scale, causal, window, dtype,
              workspace, workspace_bytes, stream) -> int:
    return load().fa_bwd_dq(Q, K, V, LSE, dO, dQ, B, T, H, HKV, head_dim, scale, causal, window, dtype,
                            workspace, workspace_bytes, stream)


def fa_bwd_dkdv_dq(Q, K, V, LSE, dO, dQ, dK, dV, B, T, H, HKV, head_dim, scale, causal, window, dtype,
                   workspace, workspace_bytes, stream) -> int:
    return load().fa_bwd_dkdv_dq(Q, K, V, LSE, dO, dQ, dK, dV, B, T, H, HKV, head_dim, scale, causal, window,
                                 dtype, workspace, workspace_bytes, stream)


def fa_check_status(workspace, stream) -> tuple[int, int]:
    word = ctypes.c_uint(0)
    st = load().fa_check_status(workspace, stream, ctypes.byref(word))
    return st, word.value


def fa_status_string(status: int) -> str:
    try:
        return load().fa_status_string(int(status)).decode()
    except Exception:  # library missing: still format the message
        return f"status {status}"


def fa_plan_kv_range(T, BM, BN, causal, window, qb):
    lo, hi = _i(0), _i(0)
    st = load().fa_plan_kv_range(T, BM, BN, causal, window, qb, ctypes.byref(lo), ctypes.byref(hi))
    if st:
        raise FaError(st, "fa_plan_kv_range")
    return lo.value, hi.value


def fa_plan_row_keys(Tq, Tk, causal, window, i):
    lo, hi = _i(0), _i(0)
    st = load().fa_plan_row_keys(Tq, Tk, causal, window, i, ctypes.byref(lo), ctypes.byref(hi))
    if st:
        raise FaError(st, "fa_plan_row_keys")
    return lo.value, hi.value


def fa_plan_key_rows(Tq, Tk, causal, window, j):
    lo, hi = _i(0), _i(0)
    st = load().fa_plan_key_rows(Tq, Tk, causal, window, j, ctypes.byref(lo), ctypes.byref(hi))
    if st:
        raise FaError(st, "fa_plan_key_rows")
    return lo.value, hi.value


def fa_plan_q_range(T, BM, BN, causal, window, kb):
    lo, hi = _i(0), _i(0)
    st = load().fa_plan_q_range(T, BM, BN, causal, window, kb, ctypes.byref(lo), ctypes.byref(hi))
    if st:
        raise FaError(st, "fa_plan_q_range")
    return lo.value, hi.value


def fa_plan_block_mask(T, BM, BN, causal, window, qb, kb) -> int:
    return load().fa_plan_block_mask(T, BM, BN, causal, window, qb, kb)


def fa_tile_m() -> int:
    return load().fa_tile_m()


def fa_tile_n() -> int:
    return load().fa_tile_n()


def fa_debug_config(wait_timeout_ns: int = 0, inject_stall: int = 0) -> int:
    return load().fa_debug_config(int(wait_timeout_ns), int(inject_stall))


def fa_debug_fwd_tiles(tiles: int = 0) -> int:
    return load().fa_debug_fwd_tiles(int(tiles))


def fa_debug_max_ctas(ctas: int = 0) -> int:
    return load().fa_debug_max_ctas(int(ctas))


def fa_qk_norm_rope_fwd(qk, f1, f2, q, k, tokens, hq, hk, head_dim, dtype, stream) -> int:
    return load().fa_qk_norm_rope_fwd(qk, f1, f2, q, k, tokens, hq, hk, head_dim, dtype, stream)


def fa_qk_norm_rope_bwd(dq, dk, qk, f1, f2, dqk, tokens, hq, hk, head_dim, dtype, stream) -> int:
    return load().fa_qk_norm_rope_bwd(dq, dk, qk, f1, f2, dqk, tokens, hq, hk, head_dim, dtype, stream)


def fa_qk_norm_rope_fwd_opt(qk, f1, f2, q, k, tokens, heads, head_dim, rotary_dim, paired, key_offset, dtype,
                            stream) -> int:
    return load().fa_qk_norm_rope_fwd_opt(qk, f1, f2, q, k, tokens, heads, head_dim, rotary_dim, paired,
                                          key_offset, dtype, stream)


def fa_qk_norm_rope_bwd_opt(dq, dk, qk, f1, f2, dqk, tokens, heads, head_dim, rotary_dim, paired, key_offset,
                            dtype, stream) -> int:
    return load().fa_qk_norm_rope_bwd_opt(dq, dk, qk, f1, f2, dqk, tokens, heads, head_dim, rotary_dim, paired,
                                          key_offset, dtype, stream)


# ------------------------------------------------------------ torch layer

_ws_cache: dict = {}


def _torch():
    import torch
    return torch


def _dtype_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.bfloat16:
        return FA_DTYPE_BF16
    if t.dtype == torch.float32:
        return FA_DTYPE_FP32
    if t.dtype == torch.float16:
        return FA_DTYPE_FP16
    raise TypeError(f"unsupported dtype {t.dtype}")


def _check_tensor(name, t, shape, dtype, device):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if t.dtype != dtype:
        raise TypeError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def workspace(op: int, B, T, H, HKV, D, dtype_code, device, stream):
    """Zero-filled workspace tensor cached per (device, stream, op, size)."""
    torch = _torch()
    n = fa_workspace_size(op, B, T, H, HKV, D, dtype_code)
    if n == 0:
        raise FaError(FA_ERR_INVALID_ARG, "fa_workspace_size")
    key = (device.index, int(stream), op)
    ws = _ws_cache.get(key)
    if ws is None or ws.numel() < n:
        ws = torch.zeros(n, dtype=torch.uint8, device=device)
        _ws_cache[key] = ws
    return ws, n


def _stream(device, stream):
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return stream.cuda_stream


def attention_fwd(q, k, v, scale=None, causal=True, window=0, out=None, lse=None, stream=None):
    """O [B,T,H,D] and LSE [B,H,T] (fp32) for q [B,T,H,D], k/v [B,Tk,HKV,D].

    Tk != T (cross-attention) runs fa_fwd_cross: unmasked attention only, so
    causal and window must then be off."""
    torch = _torch()
    B, T, H, D = q.shape
    Tk, HKV = k.shape[1], k.shape[2]
    dev = q.device
    dt = _dtype_code(q)
    for name, t, shp in (("q", q, (B, T, H, D)), ("k", k, (B, Tk, HKV, D)), ("v", v, (B, Tk, HKV, D))):
        _check_tensor(name, t, shp, q.dtype, dev)
    if Tk != T and (causal or window):
        raise FaError(FA_ERR_UNSUPPORTED, "attention_fwd: causal or window masking needs len(k) == len(q)")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    o = torch.empty_like(q) if out is None else out
    l = torch.empty((B, H, T), dtype=torch.float32, device=dev) if lse is None else lse
    _check_tensor("out", o, (B, T, H, D), q.dtype, dev)
    _check_tensor("lse", l, (B, H, T), torch.float32, dev)
    s = _stream(dev, stream)
    ws, n = workspace(FA_OP_FWD, B, T, H, HKV, D, dt, dev, s)
    if Tk != T:
        st = fa_fwd_cross(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), l.data_ptr(), B, T, Tk, H, HKV,
                          D, float(scale), dt, ws.data_ptr(), n, s)
        if st != FA_OK:
            raise FaError(st, "fa_fwd_cross")
        return o, l
    st = fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), l.data_ptr(), B, T, H, HKV, D,
                float(scale), int(bool(causal)), int(window), dt, ws.data_ptr(), n, s)
    if st != FA_OK:
        raise FaError(st, "fa_fwd")
    return o, l


def attention_bwd(q, k, v, o, lse, do, scale=None, causal=True, window=0, dq=None, dk=None, dv=None,
                  stream=None, recompute_dq=True):
    """dQ, dK, dV given the forward's O and LSE and the output gradient dO
    (cross-attention when k and v are longer or shorter than q).

    recompute_dq=False runs fa_bwd_preprocess + fa_bwd_dkdv_dq: dQ from the
    dK/dV pass's dS tiles, summed in a fixed order, without recomputing S
    and dP (16-bit types, head dims up to 64, causal masking; slower than the
    default on GB300, see include/fa.h)."""
    torch = _torch()
    B, T, H, D = q.shape
    Tk, HKV = k.shape[1], k.shape[2]
    dev = q.device
    dt = _dtype_code(q)
    for name, t, shp in (("q", q, (B, T, H, D)), ("k", k, (B, Tk, HKV, D)), ("v", v, (B, Tk, HKV, D)),
                         ("o", o, (B, T, H, D)), ("do", do, (B, T, H, D))):
        _check_tensor(name, t, shp, q.dtype, dev)
    _check_tensor("lse", lse, (B, H, T), torch.float32, dev)
    if Tk != T and (causal or window):
        raise FaError(FA_ERR_UNSUPPORTED, "attention_bwd: causal or window masking needs len(k) == len(q)")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    s = _stream(dev, stream)
    if not recompute_dq:
        if Tk != T or not causal or fa_workspace_size(FA_OP_BWD_FUSED, B, T, H, HKV, D, dt) == 0:
            raise FaError(FA_ERR_UNSUPPORTED, "attention_bwd: recompute_dq=False needs causal self-attention "
                                              "with 16-bit elements and a head dim of at most 64")
        ws, n = workspace(FA_OP_BWD_FUSED, B, T, H, HKV, D, dt, dev, s)
        st = fa_bwd_preprocess(o.data_ptr(), do.data_ptr(), B, T, H, HKV, D, dt, ws.data_ptr(), n, s)
        if st != FA_OK:
            raise FaError(st, "fa_bwd_preprocess")
        st = fa_bwd_dkdv_dq(q.data_ptr(), k.data_ptr(), v.data_ptr(), lse.data_ptr(), do.data_ptr(), dq.data_ptr(),
                            dk.data_ptr(), dv.data_ptr(), B, T, H, HKV, D, float(scale), 1, int(window), dt,
                            ws.data_ptr(), n, s)
        if st != FA_OK:
            raise FaError(st, "fa_bwd_dkdv_dq")
        return dq, dk, dv
    ws, n = workspace(FA_OP_BWD, B, T, H, HKV, D, dt, dev, s)
    if Tk != T:
        st = fa_bwd_cross(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), do.data_ptr(),
                          dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, T, Tk, H, HKV, D, float(scale), dt,
                          ws.data_ptr(), n, s)
        if st != FA_OK:
            raise FaError(st, "fa_bwd_cross")
        return dq, dk, dv
    st = fa_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), do.data_ptr(),
                dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, T, H, HKV, D, float(scale),
                int(bool(causal)), int(window), dt, ws.data_ptr(), n, s)
    if st != FA_OK:
        raise FaError(st, "fa_bwd")
    return dq, dk, dv


def check_status(device=None, stream=None, op: int = FA_OP_BWD) -> tuple[int, int]:
    """Synchronise and read (and clear) the device error words of cached workspaces."""
    torch = _torch()
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    s = _stream(dev, stream)
    worst = (FA_OK, 0)
    for (di, si, _op), ws in list(_ws_cache.items()):
        if di == dev.index and si == s:
            st, word = fa_check_status(ws.data_ptr(), s)
            if st != FA_OK:
                worst = (st, word)
    return worst


def qk_norm_rope_fwd(qk, f1, f2, hq, q=None, k=None, stream=None):
    """Pre-attention prologue: q [tokens, hq, D] and k [tokens, hk, D] from the
    packed projection qk [tokens, hq + hk, D] (bf16 or fp16) and the fp32
    rotary factors f1, f2 [tokens, D]: RMS-norm of every head vector, then
    y_d = f1_d n_d + f2_d n_(d xor 1)."""
    torch = _torch()
    tokens, heads, D = qk.shape
    hk = heads - int(hq)
    dev = qk.device
    dt = _dtype_code(qk)
    for name, t in (("f1", f1), ("f2", f2)):
        _check_tensor(name, t, (tokens, D), torch.float32, dev)
    q = torch.empty((tokens, hq, D), dtype=qk.dtype, device=dev) if q is None else q
    k = torch.empty((tokens, hk, D), dtype=qk.dtype, device=dev) if k is None else k
    _check_tensor("qk", qk, (tokens, heads, D), qk.dtype, dev)
    _check_tensor("q", q, (tokens, hq, D), qk.dtype, dev)
    _check_tensor("k", k, (tokens, hk, D), qk.dtype, dev)
    st = fa_qk_norm_rope_fwd(qk.data_ptr(), f1.data_ptr(), f2.data_ptr(), q.data_ptr(), k.data_ptr(), tokens,
                             int(hq), hk, D, dt, _stream(dev, stream))
    if st != FA_OK:
        raise FaError(st, "fa_qk_norm_rope_fwd")
    return q, k


def qk_norm_rope_bwd(dq, dk, qk, f1, f2, dqk=None, stream=None):
    """Gradient of the packed projection qk given the gradients of q and k."""
    torch = _torch()
    tokens, heads, D = qk.shape
    hq, hk = dq.shape[1], dk.shape[1]
    dev = qk.device
    dt = _dtype_code(qk)
    _check_tensor("dq", dq, (tokens, hq, D), qk.dtype, dev)
    _check_tensor("dk", dk, (tokens, hk, D), qk.dtype, dev)
    for name, t in (("f1", f1), ("f2", f2)):
        _check_tensor(name, t, (tokens, D), torch.float32, dev)
    dqk = torch.empty_like(qk) if dqk is None else dqk
    _check_tensor("dqk", dqk, (tokens, heads, D), qk.dtype, dev)
    st = fa_qk_norm_rope_bwd(dq.data_ptr(), dk.data_ptr(), qk.data_ptr(), f1.data_ptr(), f2.data_ptr(),
                             dqk.data_ptr(), tokens, hq, hk, D, dt, _stream(dev, stream))
    if st != FA_OK:
        raise FaError(st, "fa_qk_norm_rope_bwd")
    return dqk


def qk_norm_rope_fwd_opt(qk, f1, f2, heads, rotary_dim=0, paired=False, key_offset=False, stream=None):
    """Prologue with the paired-heads or key-offset option: qk [tokens,
    2*heads, D] -> (q, k), each [tokens, heads, D] or, paired,
    [2*tokens, heads/2, D] (f1, f2 then [tokens, 2*D])."""
    torch = _torch()
    tokens, heads2, D = qk.shape
    dev = qk.device
    dt = _dtype_code(qk)
    _check_tensor("qk", qk, (tokens, 2 * int(heads), D), qk.dtype, dev)
    F = 2 * D if paired else D
    for name, t in (("f1", f1), ("f2", f2)):
        _check_tensor(name, t, (tokens, F), torch.float32, dev)
    shape = (2 * tokens, int(heads) // 2, D) if paired else (tokens, int(heads), D)
    q = torch.empty(shape, dtype=qk.dtype, device=dev)
    k = torch.empty(shape, dtype=qk.dtype, device=dev)
    st = fa_qk_norm_rope_fwd_opt(qk.data_ptr(), f1.data_ptr(), f2.data_ptr(), q.data_ptr(), k.data_ptr(), tokens,
                                 int(heads), D, int(rotary_dim), int(bool(paired)), int(bool(key_offset)), dt,
                                 _stream(dev, stream))
    if st != FA_OK:
        raise FaError(st, "fa_qk_norm_rope_fwd_opt")
    return q, k


def qk_norm_rope_bwd_opt(dq, dk, qk, f1, f2, heads, rotary_dim=0, paired=False, key_offset=False, stream=None):
    """Gradient of qk for qk_norm_rope_fwd_opt given the gradients of q and k."""
    torch = _torch()
    tokens, heads2, D = qk.shape
    dev = qk.device
    dt = _dtype_code(qk)
    _check_tensor("qk", qk, (tokens, 2 * int(heads), D), qk.dtype, dev)
    shape = (2 * tokens, int(heads) // 2, D) if paired else (tokens, int(heads), D)
    _check_tensor("dq", dq, shape, qk.dtype, dev)
    _check_tensor("dk", dk, shape, qk.dtype, dev)
    F = 2 * D if paired else D
    for name, t in (("f1", f1), ("f2", f2)):
        _check_tensor(name, t, (tokens, F), torch.float32, dev)
    dqk = torch.empty_like(qk)
    st = fa_qk_norm_rope_bwd_opt(dq.data_ptr(), dk.data_ptr(), qk.data_ptr(), f1.data_ptr(), f2.data_ptr(),
                                 dqk.data_ptr(), tokens, int(heads), D, int(rotary_dim), int(bool(paired)),
                                 int(bool(key_offset)), dt, _stream(dev, stream))
    if st != FA_OK:
        raise FaError(st, "fa_qk_norm_rope_bwd_opt")
    return dqk
