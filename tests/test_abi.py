"""CPU checks of the C-ABI library: it builds, loads and exports every symbol
that include/*.h declares, and its host-side validation rejects bad arguments
with the documented status before touching the GPU."""
import ctypes
import glob
import os
import re

import pytest
import torch

from qk_norm_rope_gb300 import api

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
FAKE = 0x7f0000000000  # 256-byte aligned stand-in for a device address (never dereferenced)


def declared_symbols():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        names |= set(re.findall(r"ST_API\s+[\w\s\*]+?\b(st_\w+)\s*\(", src))
    return names


def test_library_exports_every_declared_symbol():
    L = api.lib()
    names = declared_symbols()
    assert {"st_rope_attn_fwd", "st_rope_attn_bwd", "st_rope_attn_workspace_size"} <= names
    for n in names:
        assert hasattr(L, n), n


def T(shape, dtype=api.ST_BF16, data=FAKE, strides=None):
    t = api.st_tensor()
    t.data = data
    t.dtype = dtype
    t.ndim = len(shape)
    if strides is None:
        strides, acc = [], 1
        for s in reversed(shape):
            strides.insert(0, acc)
            acc *= s
    for a, (s, st) in enumerate(zip(shape, strides)):
        t.shape[a] = s
        t.stride[a] = st
    return t


class Call:
    """A valid forward call on fake device pointers; tests perturb one field."""

    def __init__(self, B=1, S=256, Skv=None, H=2, D=128):
        Skv = S if Skv is None else Skv
        self.q = T([B, S, H, D])
        self.k = T([B, Skv, H, D])
        self.v = T([B, Skv, H, D])
        self.wq = T([D], api.ST_F32)
        self.wk = T([D], api.ST_F32)
        self.o = T([B, S, H, D])
        self.lse = T([B, H, S], api.ST_F32)
        self.ids = T([1, S, 3], api.ST_I32)
        self.ids_k = None
        self.axes = [16, 56, 56]
        self.theta = 1e4
        self.mask = None
        self.causal = 0
        self.ws_bytes = 1 << 30
        self.ws = FAKE
        self.tabs = None  # (cos, sin, cos_k, sin_k) for the table form

    def rope(self):
        r = api.st_rope()
        if self.tabs is not None:
            r.cos, r.sin, r.cos_k, r.sin_k = (None if t is None else ctypes.pointer(t) for t in self.tabs)
        r.ids = ctypes.pointer(self.ids) if self.ids is not None else None
        r.ids_k = ctypes.pointer(self.ids_k) if self.ids_k is not None else None
        r.n_axes = len(self.axes)
        for a, d in enumerate(self.axes):
            r.axes_dim[a] = d
        r.theta = self.theta
        return r

    def fwd(self):
        p = lambda t: None if t is None else ctypes.pointer(t)
        L = api.lib()
        return L.st_rope_attn_fwd(p(self.q), p(self.k), p(self.v), p(self.wq), p(self.wk), 1e-6,
                                  ctypes.byref(self.rope()), p(self.mask), self.causal, 0.0, p(self.o), p(self.lse),
                                  ctypes.c_void_p(self.ws), self.ws_bytes, None)

    def ws_size(self, bwd=0):
        p = lambda t: None if t is None else ctypes.pointer(t)
        return api.lib().st_rope_attn_workspace_size(p(self.q), p(self.k), p(self.v), p(self.mask), self.causal,
                                                     ctypes.byref(self.rope()), bwd)


def expect(c, status, pattern=None):
    st = c.fwd()
    msg = api.lib().st_last_error().decode()
    assert st == status, (api.STATUS_NAMES[st], msg)
    if pattern:
        assert re.search(pattern, msg), msg


def test_workspace_size_valid_and_grows_for_backward():
    c = Call()
    f, b = c.ws_size(0), c.ws_size(1)
    assert 0 < f < b
    c.mask = T([1, 1, 1, 256], api.ST_BOOL)
    assert c.ws_size(0) > f


def test_valid_call_without_gpu_reports_cuda_error():
    if torch.cuda.is_available():
        pytest.skip("only meaningful without a GPU")
    expect(Call(), api.ST_ERR_CUDA)


def test_null_and_shape_errors():
    c = Call(); c.q = None; expect(c, api.ST_ERR_INVALID_ARG)
    c = Call(D=64); c.wq = T([64], api.ST_F32); c.wk = T([64], api.ST_F32); expect(c, api.ST_ERR_UNSUPPORTED)
    c = Call(); c.k = T([1, 256, 3, 128]); expect(c, api.ST_ERR_SHAPE, "must divide")
    c = Call(); c.o = T([1, 255, 2, 128]); expect(c, api.ST_ERR_SHAPE, "o has shape")
    c = Call(); c.lse = T([1, 2, 255], api.ST_F32); expect(c, api.ST_ERR_SHAPE, "lse")
    c = Call(); c.wq = T([64], api.ST_F32); expect(c, api.ST_ERR_SHAPE, "q_norm_w")


def test_dtype_errors():
    c = Call(); c.q.dtype = api.ST_F16; expect(c, api.ST_ERR_DTYPE, "q and k must have the same dtype")
    c = Call(); c.q.dtype = c.k.dtype = api.ST_F16; expect(c, api.ST_ERR_DTYPE, "v's dtype")
    c = Call(); c.q.dtype = c.k.dtype = api.ST_I32; expect(c, api.ST_ERR_DTYPE, "q")
    c = Call(); c.v.dtype = api.ST_F32; expect(c, api.ST_ERR_DTYPE, "v's dtype")
    c = Call(); c.v.dtype = api.ST_I32; expect(c, api.ST_ERR_DTYPE, "v")
    c = Call(); c.o.dtype = api.ST_F32; expect(c, api.ST_ERR_DTYPE, "o")
    c = Call(); c.wk.dtype = api.ST_BF16; expect(c, api.ST_ERR_DTYPE, "k_norm_w")
    c = Call(); c.ids.dtype = api.ST_BF16; expect(c, api.ST_ERR_DTYPE, "ids")
    c = Call(); c.mask = T([1, 1, 1, 256], api.ST_I32); expect(c, api.ST_ERR_DTYPE, "mask")


def test_operand_types_accepted():
    """bf16 throughout, fp16 throughout, fp32 q/k with either 16-bit v, and
    fp32 throughout (the exact-fp32 kernels)."""
    for qk, v in ((api.ST_BF16, api.ST_BF16), (api.ST_F16, api.ST_F16), (api.ST_F32, api.ST_BF16),
                  (api.ST_F32, api.ST_F16), (api.ST_F32, api.ST_F32)):
        c = Call()
        c.q.dtype = c.k.dtype = qk
        c.v.dtype = c.o.dtype = v
        assert c.ws_size(0) > 0 and c.ws_size(1) > 0, (qk, v, api.lib().st_last_error())


def test_alignment_errors():
    c = Call(); c.q.data = FAKE + 8; expect(c, api.ST_ERR_ALIGN, "aligned")
    c = Call(); c.k.stride[3] = 2; expect(c, api.ST_ERR_ALIGN, "unit stride")
    c = Call(); c.v.stride[1] = 2 * 128 + 4; expect(c, api.ST_ERR_ALIGN, "multiple of 16")
    c = Call(); c.lse.stride[2] = 2; expect(c, api.ST_ERR_ALIGN, "contiguous")
    c = Call(); c.ws = FAKE + 16; expect(c, api.ST_ERR_ALIGN, "256-byte")


def test_rope_and_mask_errors():
    c = Call(); c.axes = [16, 56, 54]; c.ids = T([1, 256, 3], api.ST_I32); expect(c, api.ST_ERR_INVALID_ARG, "axes")
    c = Call(); c.axes = [16, 57, 55]; expect(c, api.ST_ERR_INVALID_ARG, "even")
    c = Call(); c.theta = -1.0; expect(c, api.ST_ERR_INVALID_ARG, "theta")
    c = Call(); c.ids = T([2, 256, 3], api.ST_I32); expect(c, api.ST_ERR_SHAPE, "ids")
    c = Call(); c.ids = T([1, 256, 2], api.ST_I32); expect(c, api.ST_ERR_SHAPE, "ids")
    c = Call(S=256, Skv=200); expect(c, api.ST_ERR_INVALID_ARG, "ids_k")
    c = Call(); c.mask = T([1, 1, 1, 256], api.ST_BOOL); c.causal = 1; expect(c, api.ST_ERR_INVALID_ARG, "causal")
    c = Call(); c.mask = T([1, 1, 1, 255], api.ST_BOOL); expect(c, api.ST_ERR_SHAPE, "mask")
    c = Call(); c.mask = T([1, 3, 1, 256], api.ST_BOOL); expect(c, api.ST_ERR_SHAPE, "mask")
    c = Call(); c.mask = T([1, 1, 256, 256], api.ST_F32, strides=[1, 1, 1, 256]); expect(c, api.ST_ERR_ALIGN)


def test_workspace_errors():
    c = Call()
    need = c.ws_size(0)
    c.ws_bytes = need - 1
    expect(c, api.ST_ERR_WORKSPACE, "smaller")
    c = Call(); c.ws = 0; expect(c, api.ST_ERR_WORKSPACE, "NULL")


def tables(c, S=256, B=None, dtype=api.ST_BF16, k=None):
    """The table form on a Call: [S, D] tables (or [B, S, D]), optional key tables."""
    shape = [S, 128] if B is None else [B, S, 128]
    kt = (None, None) if k is None else (T(k, dtype), T(k, dtype))
    c.ids = None
    c.tabs = (T(shape, dtype), T(shape, dtype)) + kt
    return c


def test_table_form_validation():
    """The pages' cos/sin table form: accepted shapes and dtypes, and every
    rejected combination with its status (no launch)."""
    for shape_b in (None, 1):
        for dt in (api.ST_F32, api.ST_BF16, api.ST_F16):
            c = tables(Call(), B=shape_b, dtype=dt)
            assert c.ws_size(0) > 0, api.lib().st_last_error().decode()
    assert tables(Call(B=2), B=2).ws_size(0) > tables(Call(B=2)).ws_size(0)  # per-sample tables take more room
    c = tables(Call()); c.ids = T([1, 256, 3], api.ST_I32); expect(c, api.ST_ERR_INVALID_ARG, "not both")
    c = tables(Call()); c.tabs = (c.tabs[0], None, None, None); expect(c, api.ST_ERR_INVALID_ARG, "both be given")
    c = tables(Call(), S=255); expect(c, api.ST_ERR_SHAPE, "rope.cos/sin")
    c = tables(Call()); c.tabs = (T([256, 64], api.ST_BF16), T([256, 64], api.ST_BF16), None, None)
    expect(c, api.ST_ERR_SHAPE, "rope.cos/sin")
    c = tables(Call(B=2), B=3); expect(c, api.ST_ERR_SHAPE, "batch dim")
    c = tables(Call()); c.tabs = (T([256, 128], api.ST_BF16), T([1, 256, 128], api.ST_BF16), None, None)
    expect(c, api.ST_ERR_SHAPE)
    c = tables(Call(), dtype=api.ST_I32); expect(c, api.ST_ERR_DTYPE, "fp32, bf16 or fp16")
    c = tables(Call()); c.tabs = (T([256, 128], api.ST_F32), T([256, 128], api.ST_BF16), None, None)
    expect(c, api.ST_ERR_DTYPE, "same dtype")
    c = tables(Call(S=256, Skv=200)); expect(c, api.ST_ERR_INVALID_ARG, "cos_k/sin_k are required")
    c = tables(Call(S=256, Skv=200), k=[200, 128])
    assert c.ws_size(0) > tables(Call()).ws_size(0) - 1  # separate key tables are planned
    c = tables(Call(S=256, Skv=200), k=[256, 128]); expect(c, api.ST_ERR_SHAPE, "rope.cos_k/sin_k")
    c = Call(); c.tabs = (None, None, T([256, 128]), T([256, 128])); expect(c, api.ST_ERR_INVALID_ARG, "need rope.cos")
    c = tables(Call()); c.tabs = (T([256, 128], data=0), T([256, 128]), None, None)
    expect(c, api.ST_ERR_INVALID_ARG, "NULL")


def test_python_rope_tables_marshalling():
    """RopeTables fills the table fields of the struct and nothing else."""
    cpu = torch.zeros(4, 128, dtype=torch.bfloat16)
    r = api._rope(api.RopeTables(cpu, cpu), (), 1e4, None)
    assert bool(r.cos) and bool(r.sin) and not r.cos_k and not r.ids and r.n_axes == 0
    assert r.cos.contents.shape[0] == 4 and r.cos.contents.dtype == api.ST_BF16
    with pytest.raises(api.StError):
        api._rope(api.RopeTables(cpu, cpu), (), 1e4, cpu)
    with pytest.raises(api.StError):
        api.RopeTables(cpu, None)
    with pytest.raises(api.StError):
        api._require_cuda(api.RopeTables(cpu, cpu))


def test_grouped_kv_heads_validation():
    """k and v may carry fewer heads than q when their count divides H (grouped
    K/V heads); dk and dv then have the K/V head count."""
    c = Call(H=4); c.k = T([1, 256, 2, 128]); c.v = T([1, 256, 2, 128])
    # the forward's shared K' tiles are held per K/V head (bf16 rows of 256 B)
    assert c.ws_size(1) > 0 and c.ws_size(0) == Call(H=4).ws_size(0) - 2 * 256 * 256
    c = Call(H=4); c.k = T([1, 256, 1, 128]); c.v = T([1, 256, 1, 128])
    assert c.ws_size(1) > 0
    c = Call(H=4); c.k = T([1, 256, 3, 128]); c.v = T([1, 256, 3, 128]); expect(c, api.ST_ERR_SHAPE, "must divide")
    c = Call(H=4); c.k = T([1, 256, 2, 128]); c.v = T([1, 256, 4, 128]); expect(c, api.ST_ERR_SHAPE, "v has shape")
