"""ORACLE — test infrastructure only.

A plain fp64 CPU implementation of the Flux-style attention call (RMSNorm on
q and k, multi-axis interleaved-pair RoPE, scaled-dot-product attention with
bool/additive/broadcast masks or causal masking, forward and backward). The
arithmetic lives in ``oracle.c``; this module compiles it with gcc and
marshals numpy arrays into it. It shares no code with the CUDA library.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(closed forms, invariants, brute-force finite differences, and a library
special case built from torch's fp64 CPU ops).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_SO = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into a shared object with gcc + OpenMP."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_SO)
            and os.path.getmtime(_SO) >= os.path.getmtime(_SRC)):
        return _SO
    tmp = _SO + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            dp = ctypes.POINTER(ctypes.c_double)
            ip = ctypes.POINTER(ctypes.c_int)
            i64p = ctypes.POINTER(ctypes.c_int64)
            vp = ctypes.c_void_p
            c_int, c_dbl, c_i64 = ctypes.c_int, ctypes.c_double, ctypes.c_int64
            lib.oracle_num_threads.restype = c_int
            lib.oracle_rope_angles.argtypes = [dp, c_i64, c_int, ip, c_dbl, dp]
            lib.oracle_rope_angles.restype = None
            lib.oracle_qk_transform.argtypes = [dp, c_i64, c_int, dp, c_dbl, dp, dp]
            lib.oracle_qk_transform.restype = None
            common = [c_int, c_int, c_int, c_int, c_int, c_int, dp, dp, dp, dp, dp, c_dbl, dp, c_int, dp, c_int,
                      c_int, vp, i64p, c_int, c_dbl]
            lib.oracle_fwd.argtypes = common + [ip, c_int, dp, dp]
            lib.oracle_fwd.restype = c_int
            lib.oracle_bwd.argtypes = common + [dp, ip, c_int, dp, dp, dp, dp, dp]
            lib.oracle_bwd.restype = c_int
            lib.oracle_qk_transform_tab.argtypes = [dp, c_i64, c_int, dp, c_dbl, dp, dp, dp]
            lib.oracle_qk_transform_tab.restype = None
            common_tab = [c_int, c_int, c_int, c_int, c_int, c_int, dp, dp, dp, dp, dp, c_dbl, dp, dp, c_int, dp, dp,
                          c_int, c_int, vp, i64p, c_int, c_dbl]
            lib.oracle_fwd_tab.argtypes = common_tab + [ip, c_int, dp, dp]
            lib.oracle_fwd_tab.restype = c_int
            lib.oracle_bwd_tab.argtypes = common_tab + [dp, ip, c_int, dp, dp, dp, dp, dp]
            lib.oracle_bwd_tab.restype = c_int
            _lib = lib
    return _lib


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _dp(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def rope_angles(ids, axes_dim, theta: float) -> np.ndarray:
    """Angles [..., S, D/2] for ids [..., S, n_axes] (see oracle_rope_angles)."""
    ids = _f64(ids)
    n_axes = ids.shape[-1]
    assert n_axes == len(axes_dim)
    D = int(sum(axes_dim))
    n_tok = int(np.prod(ids.shape[:-1]))
    phi = np.zeros(ids.shape[:-1] + (D // 2,), dtype=np.float64)
    axes = (ctypes.c_int * n_axes)(*[int(a) for a in axes_dim])
    _load().oracle_rope_angles(_dp(ids), n_tok, n_axes, axes, float(theta), _dp(phi))
    return phi


def qk_transform(x, w, eps: float, phi) -> np.ndarray:
    """RoPE(RMSNorm(x)) row by row: x [..., D], phi [..., D/2] (same leading shape)."""
    x = _f64(x)
    D = x.shape[-1]
    phi = _f64(np.broadcast_to(phi, x.shape[:-1] + (D // 2,)))
    w = _f64(w)
    out = np.zeros_like(x)
    n = int(np.prod(x.shape[:-1]))
    _load().oracle_qk_transform(_dp(x), n, D, _dp(w), float(eps), _dp(phi), _dp(out))
    return out


def _mask_args(mask, B, H, Sq, Skv):
    """(kind, array, strides) for a mask of shape [B|1, H|1, Sq|1, Skv] or None."""
    if mask is None:
        return 0, None, (ctypes.c_int64 * 4)(0, 0, 0, 0)
    m = np.asarray(mask)
    assert m.ndim == 4 and m.shape[3] == Skv
    for ax, full in zip(m.shape[:3], (B, H, Sq)):
        assert ax in (1, full)
    if m.dtype == np.bool_:
        arr = np.ascontiguousarray(m.astype(np.uint8))
        kind = 1
    else:
        arr = _f64(m)
        kind = 2
    st = [0, 0, 0, 0]
    acc = 1
    for ax in (3, 2, 1, 0):
        st[ax] = 0 if arr.shape[ax] == 1 else acc
        acc *= arr.shape[ax]
    return kind, arr, (ctypes.c_int64 * 4)(*st)


def _prep(q, k, v, wq, wk, ids_q, ids_k, axes_dim, theta):
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, Sq, H, D = q.shape
    Skv, Hkv = k.shape[1], k.shape[2]
    assert k.shape == (B, Skv, Hkv, D) and v.shape == k.shape and H % Hkv == 0
    assert sum(axes_dim) == D
    phi_q = rope_angles(ids_q, axes_dim, theta)
    phi_k = rope_angles(ids_q if ids_k is None else ids_k, axes_dim, theta)
    assert phi_q.shape[-2] == Sq and phi_k.shape[-2] == Skv
    phi_q = phi_q.reshape(-1, Sq, D // 2)
    phi_k = phi_k.reshape(-1, Skv, D // 2)
    return q, k, v, _f64(wq), _f64(wk), phi_q, phi_k, B, Sq, Skv, H, Hkv, D


def _heads_arg(heads, B, H):
    if heads is None:
        return None, 0
    flat = [int(b) * H + int(h) for (b, h) in heads]
    return (ctypes.c_int * len(flat))(*flat), len(flat)


def fwd(q, k, v, wq, wk, eps, ids_q, axes_dim, theta, mask=None, causal=False, scale=None, ids_k=None,
        heads=None):
    """O [B,Sq,H,D] and LSE [B,H,Sq] (natural log), fp64. k, v may have fewer heads
    (H_kv dividing H): query head h then uses K/V head h // (H // H_kv).

    heads: optional list of (b, h) to compute; other entries are left as NaN.
    """
    q, k, v, wq, wk, phi_q, phi_k, B, Sq, Skv, H, Hkv, D = _prep(q, k, v, wq, wk, ids_q, ids_k, axes_dim, theta)
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    kind, marr, mst = _mask_args(mask, B, H, Sq, Skv)
    o = np.full((B, Sq, H, D), np.nan)
    lse = np.full((B, H, Sq), np.nan)
    hp, nh = _heads_arg(heads, B, H)
    rc = _load().oracle_fwd(B, Sq, Skv, H, Hkv, D, _dp(q), _dp(k), _dp(v), _dp(wq), _dp(wk), float(eps), _dp(phi_q),
                            phi_q.shape[0], _dp(phi_k), phi_k.shape[0], kind,
                            None if marr is None else marr.ctypes.data, mst, int(bool(causal)), float(scale), hp, nh,
                            _dp(o), _dp(lse))
    if rc != 0:
        raise MemoryError("oracle_fwd could not allocate its work buffers")
    return o, lse


def bwd(q, k, v, wq, wk, eps, ids_q, axes_dim, theta, dout, mask=None, causal=False, scale=None, ids_k=None,
        heads=None):
    """dq [.., H, D], dk, dv [.., H_kv, D] and dwq, dwk [D], fp64 (dw summed over
    `heads`; dk, dv of a K/V head summed over the listed query heads of its group)."""
    q, k, v, wq, wk, phi_q, phi_k, B, Sq, Skv, H, Hkv, D = _prep(q, k, v, wq, wk, ids_q, ids_k, axes_dim, theta)
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    dout = _f64(dout)
    assert dout.shape == q.shape
    kind, marr, mst = _mask_args(mask, B, H, Sq, Skv)
    dq = np.full(q.shape, np.nan)
    dk = np.full(k.shape, np.nan)
    dv = np.full(v.shape, np.nan)
    dwq = np.zeros(D)
    dwk = np.zeros(D)
    hp, nh = _heads_arg(heads, B, H)
    rc = _load().oracle_bwd(B, Sq, Skv, H, Hkv, D, _dp(q), _dp(k), _dp(v), _dp(wq), _dp(wk), float(eps), _dp(phi_q),
                            phi_q.shape[0], _dp(phi_k), phi_k.shape[0], kind,
                            None if marr is None else marr.ctypes.data, mst, int(bool(causal)), float(scale),
                            _dp(dout), hp, nh, _dp(dq), _dp(dk), _dp(dv), _dp(dwq), _dp(dwk))
    if rc != 0:
        raise MemoryError("oracle_bwd could not allocate its work buffers")
    return dq, dk, dv, dwq, dwk


# ---------------------------------------------------------------- table form
# The pages' entry point takes the rotation as cos/sin tables ("Metal Flash
# Attention", section "Fused RoPE + SDPA": pair-duplicated, shape [S, D],
# [1, S, D] or per-sample [B, S, D]). The oracle applies them elementwise,
# y = x * cos + rot(x) * sin with rot(x) = (-x1, x0) per interleaved pair.


def _tables(cos_t, sin_t, S, D):
    """[Bp, S, D] fp64 copies of a table pair of shape [S, D] or [Bp, S, D]."""
    c, s = _f64(cos_t), _f64(sin_t)
    assert c.shape == s.shape and c.shape[-2:] == (S, D), (c.shape, s.shape, S, D)
    if c.ndim == 2:
        c, s = c[None], s[None]
    assert c.ndim == 3
    return np.ascontiguousarray(c), np.ascontiguousarray(s)


def qk_transform_tab(x, w, eps: float, cos_t, sin_t) -> np.ndarray:
    """RoPE(RMSNorm(x)) row by row with table rows: x, cos_t, sin_t [..., D]."""
    x = _f64(x)
    c = _f64(np.broadcast_to(cos_t, x.shape))
    s = _f64(np.broadcast_to(sin_t, x.shape))
    w = _f64(w)
    out = np.zeros_like(x)
    n = int(np.prod(x.shape[:-1]))
    _load().oracle_qk_transform_tab(_dp(x), n, x.shape[-1], _dp(w), float(eps), _dp(c), _dp(s), _dp(out))
    return out


def _prep_tab(q, k, v, wq, wk, cos_q, sin_q, cos_k, sin_k):
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, Sq, H, D = q.shape
    Skv, Hkv = k.shape[1], k.shape[2]
    assert k.shape == (B, Skv, Hkv, D) and v.shape == k.shape and H % Hkv == 0
    if cos_k is None:
        assert Sq == Skv, "cos_k/sin_k are required when S_q != S_kv"
        cos_k, sin_k = cos_q, sin_q
    cq, sq = _tables(cos_q, sin_q, Sq, D)
    ck, sk = _tables(cos_k, sin_k, Skv, D)
    assert cq.shape[0] in (1, B) and ck.shape[0] in (1, B)
    return q, k, v, _f64(wq), _f64(wk), cq, sq, ck, sk, B, Sq, Skv, H, Hkv, D


def fwd_tab(q, k, v, wq, wk, eps, cos_q, sin_q, mask=None, causal=False, scale=None, cos_k=None, sin_k=None,
            heads=None):
    """As fwd, with the rotation given by cos/sin tables instead of ids."""
    q, k, v, wq, wk, cq, sq, ck, sk, B, Sq, Skv, H, Hkv, D = _prep_tab(q, k, v, wq, wk, cos_q, sin_q, cos_k, sin_k)
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    kind, marr, mst = _mask_args(mask, B, H, Sq, Skv)
    o = np.full((B, Sq, H, D), np.nan)
    lse = np.full((B, H, Sq), np.nan)
    hp, nh = _heads_arg(heads, B, H)
    rc = _load().oracle_fwd_tab(B, Sq, Skv, H, Hkv, D, _dp(q), _dp(k), _dp(v), _dp(wq), _dp(wk), float(eps), _dp(cq),
                                _dp(sq), cq.shape[0], _dp(ck), _dp(sk), ck.shape[0], kind,
                                None if marr is None else marr.ctypes.data, mst, int(bool(causal)), float(scale), hp,
                                nh, _dp(o), _dp(lse))
    if rc != 0:
        raise MemoryError("oracle_fwd_tab could not allocate its work buffers")
    return o, lse


def bwd_tab(q, k, v, wq, wk, eps, cos_q, sin_q, dout, mask=None, causal=False, scale=None, cos_k=None, sin_k=None,
            heads=None):
    """As bwd, with the rotation given by cos/sin tables instead of ids."""
    q, k, v, wq, wk, cq, sq, ck, sk, B, Sq, Skv, H, Hkv, D = _prep_tab(q, k, v, wq, wk, cos_q, sin_q, cos_k, sin_k)
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    dout = _f64(dout)
    assert dout.shape == q.shape
    kind, marr, mst = _mask_args(mask, B, H, Sq, Skv)
    dq = np.full(q.shape, np.nan)
    dk = np.full(k.shape, np.nan)
    dv = np.full(v.shape, np.nan)
    dwq = np.zeros(D)
    dwk = np.zeros(D)
    hp, nh = _heads_arg(heads, B, H)
    rc = _load().oracle_bwd_tab(B, Sq, Skv, H, Hkv, D, _dp(q), _dp(k), _dp(v), _dp(wq), _dp(wk), float(eps), _dp(cq),
                                _dp(sq), cq.shape[0], _dp(ck), _dp(sk), ck.shape[0], kind,
                                None if marr is None else marr.ctypes.data, mst, int(bool(causal)), float(scale),
                                _dp(dout), hp, nh, _dp(dq), _dp(dk), _dp(dv), _dp(dwq), _dp(dwk))
    if rc != 0:
        raise MemoryError("oracle_bwd_tab could not allocate its work buffers")
    return dq, dk, dv, dwq, dwk
