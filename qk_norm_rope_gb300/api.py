"""Python binding of the st_rope_attn C-ABI (ctypes).

Argument marshalling only: every step of the computation runs in the CUDA
library. PyTorch supplies device memory (outputs, workspace) and the current
stream. There is no fallback: if the library cannot be built or loaded, or a
tensor is not on a CUDA device, the call raises.

Names follow the C-ABI: ``st_rope_attn_fwd``, ``st_rope_attn_bwd``,
``st_rope_attn_workspace_size``, ``st_get_stats``, ``st_reset_stats``,
``st_check_status``, ``st_last_error``. ``rope_attention`` wraps the pair in a
``torch.autograd.Function``.

The rotation is given either by position ids (``ids``, ``axes_dim``,
``theta``) or, in the form of the "Fused RoPE + SDPA" entry point, by
pair-duplicated cos/sin tables: pass ``RopeTables(cos, sin)`` in place of
``ids`` (``axes_dim`` and ``theta`` are then ignored).
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

from . import build as _build

ST_OK, ST_ERR_INVALID_ARG, ST_ERR_DTYPE, ST_ERR_SHAPE, ST_ERR_ALIGN, ST_ERR_WORKSPACE, ST_ERR_CUDA, \
    ST_ERR_TIMEOUT, ST_ERR_UNSUPPORTED = range(9)
ST_BF16, ST_F16, ST_F32, ST_BOOL, ST_I32 = range(5)
_DTYPES = {torch.bfloat16: ST_BF16, torch.float16: ST_F16, torch.float32: ST_F32, torch.bool: ST_BOOL,
           torch.int32: ST_I32}
STATUS_NAMES = ["ST_OK", "ST_ERR_INVALID_ARG", "ST_ERR_DTYPE", "ST_ERR_SHAPE", "ST_ERR_ALIGN", "ST_ERR_WORKSPACE",
                "ST_ERR_CUDA", "ST_ERR_TIMEOUT", "ST_ERR_UNSUPPORTED"]


class st_tensor(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("ndim", ctypes.c_int32),
                ("shape", ctypes.c_int64 * 4), ("stride", ctypes.c_int64 * 4)]


class st_rope(ctypes.Structure):
    _fields_ = [("ids", ctypes.POINTER(st_tensor)), ("ids_k", ctypes.POINTER(st_tensor)),
                ("n_axes", ctypes.c_int32), ("axes_dim", ctypes.c_int32 * 8), ("theta", ctypes.c_double),
                ("cos", ctypes.POINTER(st_tensor)), ("sin", ctypes.POINTER(st_tensor)),
                ("cos_k", ctypes.POINTER(st_tensor)), ("sin_k", ctypes.POINTER(st_tensor)),
                ("reuse_tables", ctypes.c_int32)]


class RopeTables:
    """Pair-duplicated cos/sin tables ([S, D], [1, S, D] or [B, S, D]; fp32,
    bf16 or fp16) for q, and optionally separate ones for k (required when
    S_q != S_kv). Stands in for ``ids`` in every call of this module."""

    def __init__(self, cos, sin, cos_k=None, sin_k=None):
        if (cos is None) != (sin is None) or (cos_k is None) != (sin_k is None):
            raise StError(ST_ERR_INVALID_ARG, "cos and sin come in pairs")
        self.cos, self.sin, self.cos_k, self.sin_k = cos, sin, cos_k, sin_k

    def tensors(self):
        return [t for t in (self.cos, self.sin, self.cos_k, self.sin_k) if t is not None]


class st_stats(ctypes.Structure):
    _fields_ = [(n, ctypes.c_uint64) for n in ("fwd_calls", "bwd_calls", "mask_all_true_skipped",
                                                "mixed_dtype_calls", "tiles_skipped", "tiles_total", "timeouts",
                                                "kernel_launches")]


KERNEL_KINDS = ["table", "classify", "fwd", "bwd_pre", "bwd", "dq_post", "dw_reduce", "qprime", "probe"]


class st_kernel_times(ctypes.Structure):
    _fields_ = [("launches", ctypes.c_uint64 * len(KERNEL_KINDS)), ("ms", ctypes.c_double * len(KERNEL_KINDS))]


class StError(RuntimeError):
    def __init__(self, status: int, message: str):
        self.status = status
        name = STATUS_NAMES[status] if 0 <= status < len(STATUS_NAMES) else str(status)
        super().__init__(f"{name}: {message}")


_lock = threading.Lock()
_lib = None
LIB_PATH = _build.LIB


def lib():
    """The loaded CUDA library (built in-tree on first use if missing)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.build()
            L = ctypes.CDLL(path)
            T = ctypes.POINTER(st_tensor)
            R = ctypes.POINTER(st_rope)
            vp, sz, fl, i = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_float, ctypes.c_int
            L.st_rope_attn_workspace_size.argtypes = [T, T, T, T, i, R, i]
            L.st_rope_attn_workspace_size.restype = sz
            L.st_rope_attn_fwd.argtypes = [T, T, T, T, T, fl, R, T, i, fl, T, T, vp, sz, vp]
            L.st_rope_attn_fwd.restype = i
            L.st_rope_attn_bwd.argtypes = [T, T, T, T, T, fl, R, T, i, fl, T, T, T, T, T, T, T, T, vp, sz, vp]
            L.st_rope_attn_bwd.restype = i
            L.st_last_error.restype = ctypes.c_char_p
            L.st_get_stats.argtypes = [ctypes.POINTER(st_stats)]
            L.st_get_stats.restype = i
            L.st_reset_stats.restype = None
            L.st_check_status.argtypes = [vp]
            L.st_check_status.restype = i
            L.st_rope_attn_fwd_noalloc.argtypes = [T, T, T, T, T, fl, R, T, i, fl, T, T, vp]
            L.st_rope_attn_fwd_noalloc.restype = i
            L.st_selftest_wait_timeout.argtypes = [ctypes.c_longlong, vp]
            L.st_selftest_wait_timeout.restype = i
            L.st_timing_enable.argtypes = [i]
            L.st_timing_enable.restype = i
            L.st_timing_read.argtypes = [ctypes.POINTER(st_kernel_times)]
            L.st_timing_read.restype = i
            _lib = L
    return _lib


def _t(x: torch.Tensor | None):
    if x is None:
        return None
    if x.dtype not in _DTYPES:
        raise StError(ST_ERR_DTYPE, f"unsupported tensor dtype {x.dtype}")
    if x.dim() > 4:
        raise StError(ST_ERR_SHAPE, "tensors have at most 4 dims")
    s = st_tensor()
    s.data = x.data_ptr() if x.numel() > 0 else None
    s.dtype = _DTYPES[x.dtype]
    s.ndim = x.dim()
    for a in range(x.dim()):
        s.shape[a] = x.shape[a]
        s.stride[a] = x.stride(a)
    return s


def _p(s):
    return None if s is None else ctypes.pointer(s)


def _check(status: int):
    if status != ST_OK:
        raise StError(status, lib().st_last_error().decode())


def _rope(ids, axes_dim, theta, ids_k, reuse_tables=False):
    r = st_rope()
    r.reuse_tables = int(bool(reuse_tables))
    if isinstance(ids, RopeTables):
        if ids_k is not None:
            raise StError(ST_ERR_INVALID_ARG, "ids_k cannot be combined with RopeTables (use cos_k/sin_k)")
        r._keep = [_t(x) for x in (ids.cos, ids.sin, ids.cos_k, ids.sin_k)]  # alive with the rope object
        r.cos, r.sin, r.cos_k, r.sin_k = (_p(x) for x in r._keep)
        return r
    r._ids = _t(ids)            # keep the structs alive with the rope object
    r._ids_k = _t(ids_k)
    r.ids = _p(r._ids)
    r.ids_k = _p(r._ids_k)
    r.n_axes = len(axes_dim)
    for a, d in enumerate(axes_dim):
        r.axes_dim[a] = int(d)
    r.theta = float(theta)
    return r


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _require_cuda(*ts):
    for t in ts:
        for x in (t.tensors() if isinstance(t, RopeTables) else [t]):
            if x is not None and not x.is_cuda:
                raise StError(ST_ERR_INVALID_ARG, "all tensors must live on a CUDA device")


def st_rope_attn_workspace_size(q, k, v, ids, axes_dim, theta, mask=None, causal=False, ids_k=None,
                                for_backward=False) -> int:
    r = _rope(ids, axes_dim, theta, ids_k)
    n = lib().st_rope_attn_workspace_size(_p(_t(q)), _p(_t(k)), _p(_t(v)), _p(_t(mask)), int(bool(causal)),
                                          ctypes.byref(r), int(bool(for_backward)))
    if n == 0 and lib().st_last_error():
        raise StError(ST_ERR_INVALID_ARG, lib().st_last_error().decode())
    return int(n)


def _workspace(q, k, v, ids, axes_dim, theta, mask, causal, ids_k, for_backward, workspace):
    n = st_rope_attn_workspace_size(q, k, v, ids, axes_dim, theta, mask, causal, ids_k, for_backward)
    if workspace is None or workspace.numel() < n:
        workspace = torch.empty(max(n, 256), dtype=torch.uint8, device=q.device)
    return workspace


def st_rope_attn_fwd(q, k, v, q_norm_w, k_norm_w, eps, ids, axes_dim, theta, mask=None, causal=False, scale=None,
                     ids_k=None, o=None, lse=None, workspace=None):
    """Returns (o [B,S_q,H,D] in v's dtype, lse [B,H,S_q] fp32)."""
    _require_cuda(q, k, v, q_norm_w, k_norm_w, ids, mask, ids_k)
    B, Sq, H, D = q.shape
    if o is None:
        o = torch.empty((B, Sq, H, D), dtype=v.dtype, device=q.device)
    if lse is None:
        lse = torch.empty((B, H, Sq), dtype=torch.float32, device=q.device)
    ws = _workspace(q, k, v, ids, axes_dim, theta, mask, causal, ids_k, False, workspace)
    r = _rope(ids, axes_dim, theta, ids_k)
    st = lib().st_rope_attn_fwd(_p(_t(q)), _p(_t(k)), _p(_t(v)), _p(_t(q_norm_w)), _p(_t(k_norm_w)), float(eps),
                                ctypes.byref(r), _p(_t(mask)), int(bool(causal)),
                                float(scale) if scale else 0.0, _p(_t(o)), _p(_t(lse)),
                                ctypes.c_void_p(ws.data_ptr()), ws.numel(), _stream())
    _check(st)
    return o, lse


def st_rope_attn_bwd(q, k, v, q_norm_w, k_norm_w, eps, ids, axes_dim, theta, o, lse, d_o, mask=None, causal=False,
                     scale=None, ids_k=None, workspace=None, dq=None, dk=None, dv=None, dwq=None, dwk=None,
                     reuse_tables=False):
    """Returns (dq, dk, dv, d_q_norm_w, d_k_norm_w). reuse_tables: the given
    workspace was passed to the forward of this call (same rotation and mask),
    so its tables and mask tile classes are reused instead of rebuilt."""
    if reuse_tables and workspace is None:
        raise StError(ST_ERR_INVALID_ARG, "reuse_tables needs the forward's workspace")
    _require_cuda(q, k, v, q_norm_w, k_norm_w, ids, mask, ids_k, o, lse, d_o)
    dq = torch.empty_like(q, memory_format=torch.contiguous_format) if dq is None else dq
    dk = torch.empty_like(k, memory_format=torch.contiguous_format) if dk is None else dk
    dv = torch.empty_like(v, memory_format=torch.contiguous_format) if dv is None else dv
    dwq = torch.empty_like(q_norm_w) if dwq is None else dwq
    dwk = torch.empty_like(k_norm_w) if dwk is None else dwk
    ws = _workspace(q, k, v, ids, axes_dim, theta, mask, causal, ids_k, True, workspace)
    if reuse_tables and ws is not workspace:
        raise StError(ST_ERR_WORKSPACE, "reuse_tables: the workspace is smaller than the backward needs")
    r = _rope(ids, axes_dim, theta, ids_k, reuse_tables)
    st = lib().st_rope_attn_bwd(_p(_t(q)), _p(_t(k)), _p(_t(v)), _p(_t(q_norm_w)), _p(_t(k_norm_w)), float(eps),
                                ctypes.byref(r), _p(_t(mask)), int(bool(causal)),
                                float(scale) if scale else 0.0, _p(_t(o)), _p(_t(lse)), _p(_t(d_o)),
                                _p(_t(dq)), _p(_t(dk)), _p(_t(dv)), _p(_t(dwq)), _p(_t(dwk)),
                                ctypes.c_void_p(ws.data_ptr()), ws.numel(), _stream())
    _check(st)
    return dq, dk, dv, dwq, dwk


def st_rope_attn_fwd_noalloc(q, k, v, q_norm_w, k_norm_w, eps, ids, axes_dim, theta, mask=None, causal=False,
                             scale=None, ids_k=None, o=None, lse=None):
    """Forward on the library's built-in scratch (no workspace, no device
    allocation inside the call; outputs are allocated here unless given)."""
    _require_cuda(q, k, v, q_norm_w, k_norm_w, ids, mask, ids_k)
    B, Sq, H, D = q.shape
    if o is None:
        o = torch.empty((B, Sq, H, D), dtype=v.dtype, device=q.device)
    if lse is None:
        lse = torch.empty((B, H, Sq), dtype=torch.float32, device=q.device)
    r = _rope(ids, axes_dim, theta, ids_k)
    st = lib().st_rope_attn_fwd_noalloc(_p(_t(q)), _p(_t(k)), _p(_t(v)), _p(_t(q_norm_w)), _p(_t(k_norm_w)),
                                        float(eps), ctypes.byref(r), _p(_t(mask)), int(bool(causal)),
                                        float(scale) if scale else 0.0, _p(_t(o)), _p(_t(lse)), _stream())
    _check(st)
    return o, lse


def st_last_error() -> str:
    return lib().st_last_error().decode()


def st_get_stats() -> dict:
    s = st_stats()
    _check(lib().st_get_stats(ctypes.byref(s)))
    return {n: int(getattr(s, n)) for n, _ in st_stats._fields_}


def st_reset_stats() -> None:
    lib().st_reset_stats()


def st_check_status(stream=None) -> None:
    h = ctypes.c_void_p(stream.cuda_stream if stream is not None else torch.cuda.current_stream().cuda_stream)
    _check(lib().st_check_status(h))


def st_selftest_wait_timeout(budget_cycles: int) -> None:
    """Enqueues the bounded-wait self-test (see the C header)."""
    _check(lib().st_selftest_wait_timeout(int(budget_cycles), _stream()))


def st_timing_enable(on: bool) -> None:
    _check(lib().st_timing_enable(int(bool(on))))


def st_timing_read() -> dict:
    """{kernel kind: (launches, total ms)} since the previous read (synchronises)."""
    t = st_kernel_times()
    _check(lib().st_timing_read(ctypes.byref(t)))
    return {n: (int(t.launches[i]), float(t.ms[i])) for i, n in enumerate(KERNEL_KINDS)}


class RopeAttention(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, q_norm_w, k_norm_w, eps, ids, axes_dim, theta, mask, causal, scale, ids_k):
        # one backward-sized workspace for both calls: the backward reuses the
        # rotary tables and mask tile classes the forward built in it
        ws = _workspace(q, k, v, ids, axes_dim, theta, mask, causal, ids_k, True, None)
        o, lse = st_rope_attn_fwd(q, k, v, q_norm_w, k_norm_w, eps, ids, axes_dim, theta, mask, causal, scale,
                                  ids_k, workspace=ws)
        tables = ids if isinstance(ids, RopeTables) else None  # no gradient flows to the tables
        ctx.save_for_backward(q, k, v, q_norm_w, k_norm_w, None if tables else ids, mask, ids_k, o, lse)
        ctx.cfg = (eps, tuple(axes_dim), theta, causal, scale, tables)
        ctx.ws = ws
        return o

    @staticmethod
    def backward(ctx, d_o):
        q, k, v, q_norm_w, k_norm_w, ids, mask, ids_k, o, lse = ctx.saved_tensors
        eps, axes_dim, theta, causal, scale, tables = ctx.cfg
        if tables is not None:
            ids = tables
        dq, dk, dv, dwq, dwk = st_rope_attn_bwd(q, k, v, q_norm_w, k_norm_w, eps, ids, axes_dim, theta, o, lse,
                                                d_o.contiguous(), mask, causal, scale, ids_k, workspace=ctx.ws,
                                                reuse_tables=True)
        ctx.ws = None
        return dq, dk, dv, dwq, dwk, None, None, None, None, None, None, None, None


def rope_attention(q, k, v, q_norm_w, k_norm_w, ids, axes_dim=(), theta=1e4, eps=1e-6, mask=None, causal=False,
                   scale=None, ids_k=None):
    """O = SDPA(RoPE(RMSNorm_q(q)), RoPE(RMSNorm_k(k)), v, mask | causal, scale), differentiable.
    ``ids`` may be a RopeTables (then ``axes_dim`` and ``theta`` are ignored)."""
    return RopeAttention.apply(q, k, v, q_norm_w, k_norm_w, eps, ids, tuple(axes_dim), theta, mask, causal, scale,
                               ids_k)


def rope_attention_bhsd(query, key, value, rope_cos, rope_sin, q_norm_w, k_norm_w, attn_mask=None,
                        is_causal=False, scale=None, eps=1e-6):
    """The "Fused RoPE + SDPA" calling convention: BHSD tensors (strided views
    such as transpose(1, 2) of a BSHD projection are consumed without copies)
    and pair-duplicated cos/sin tables; here q and k are RMS-normalised first.
    Returns O as a BHSD view."""
    q, k, v = (t.transpose(1, 2) for t in (query, key, value))
    o = rope_attention(q, k, v, q_norm_w, k_norm_w, RopeTables(rope_cos, rope_sin), eps=eps, mask=attn_mask,
                       causal=is_causal, scale=scale)
    return o.transpose(1, 2)


def default_scale(D: int = 128) -> float:
    return 1.0 / math.sqrt(D)
