"""GPU parity of the table form of the rotation ("Metal Flash Attention",
section "Fused RoPE + SDPA": pair-duplicated cos/sin tables of shape [S, D],
[1, S, D] or per-sample [B, S, D], any float dtype) against the fp64 oracle's
table form, and against the ids form of the same call."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from _parity import compare, compare_all, f64, gpu_fwd_bwd, to_dev

pytestmark = pytest.mark.gpu


def dup_tables(ids, axes, theta, dtype):
    """Pair-duplicated (cos, sin) of the ids' angles, [..., S, D] in `dtype`."""
    phi = oracle.rope_angles(ids.numpy(), axes, theta)
    c = np.repeat(np.cos(phi), 2, axis=-1)
    s = np.repeat(np.sin(phi), 2, axis=-1)
    return torch.from_numpy(c).to(dtype), torch.from_numpy(s).to(dtype)


def gpu_tab(api, inp, tabs, d=None):
    d = d or to_dev(inp)
    rt = api.RopeTables(*[None if t is None else t.cuda() for t in tabs])
    o, lse = api.st_rope_attn_fwd(d["q"], d["k"], d["v"], d["wq"], d["wk"], inp.eps, rt, (), 0.0, mask=d["mask"],
                                  causal=inp.causal)
    dq, dk, dv, dwq, dwk = api.st_rope_attn_bwd(d["q"], d["k"], d["v"], d["wq"], d["wk"], inp.eps, rt, (), 0.0, o, lse,
                                                d["do"], mask=d["mask"], causal=inp.causal)
    api.st_check_status()
    torch.cuda.synchronize()
    return dict(o=o, lse=lse, dq=dq, dk=dk, dv=dv, dwq=dwq, dwk=dwk)


def oracle_tab(inp, tabs):
    cq, sq, ck, sk = (None if t is None else f64(t) for t in tabs)
    m = inp.mask
    m = None if m is None else (m.numpy() if m.dtype == torch.bool else m.double().numpy())
    args = (f64(inp.q), f64(inp.k), f64(inp.v), f64(inp.wq), f64(inp.wk), inp.eps, cq, sq)
    kw = dict(mask=m, causal=inp.causal, cos_k=ck, sin_k=sk)
    o, lse = oracle.fwd_tab(*args, **kw)
    dq, dk, dv, dwq, dwk = oracle.bwd_tab(*args, f64(inp.do), **kw)
    return dict(o=o, lse=lse, dq=dq, dk=dk, dv=dv, dwq=dwq, dwk=dwk)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32, torch.float16])
def test_shared_tables_match_oracle(cuda_lib, dtype):
    ids = wl.flux_ids(44, 16, 3)                       # S = 300: tiles 128, 128, 44
    inp = wl.make_custom(2, 2, 128, ids.shape[1], axes=(16, 56, 56), seed=61, ids=ids)
    c, s = dup_tables(ids, inp.axes, inp.theta, dtype)
    tabs = (c[0], s[0], None, None)                    # the [S, D] form
    compare_all(gpu_tab(cuda_lib, inp, tabs), oracle_tab(inp, tabs))


def test_per_sample_cross_length_tables_with_mask(cuda_lib):
    g = torch.Generator().manual_seed(62)
    ids = torch.randint(0, 64, (2, 200, 3), generator=g, dtype=torch.int32)
    ids_k = torch.randint(0, 64, (2, 333, 3), generator=g, dtype=torch.int32)
    inp = wl.make_custom(2, 2, 128, 200, 333, axes=(16, 56, 56), seed=63, ids=ids, ids_k=ids_k)
    m = torch.ones(2, 1, 1, 333, dtype=torch.bool)
    m[1, 0, 0, 250:] = False
    inp.mask = m
    cq, sq = dup_tables(ids, inp.axes, inp.theta, torch.float32)       # [B, S_q, D]
    ck, sk = dup_tables(ids_k, inp.axes, inp.theta, torch.float16)     # [B, S_kv, D]
    tabs = (cq, sq, ck, sk)
    compare_all(gpu_tab(cuda_lib, inp, tabs), oracle_tab(inp, tabs))


def test_tables_of_the_ids_reproduce_the_ids_form(cuda_lib):
    """fp32 tables holding the ids' cos/sin give the ids form's results (the
    device builds the same fp32 values from the ids, up to rounding)."""
    ids = wl.flux_ids(16, 12, 3)
    inp = wl.make_custom(1, 3, 128, ids.shape[1], axes=(16, 56, 56), seed=64, ids=ids, causal=True)
    c, s = dup_tables(ids, inp.axes, inp.theta, torch.float32)
    got = gpu_tab(cuda_lib, inp, (c, s, None, None))   # the [1, S, D] form
    ref = gpu_fwd_bwd(cuda_lib, inp)
    for key in ("o", "lse", "dq", "dk", "dv", "dwq", "dwk"):
        compare(key, got[key], f64(ref[key]), atol=1e-2, rel_fro=2e-3)


def test_strided_tables_and_bhsd_wrapper(cuda_lib):
    """Non-contiguous table views and the BHSD calling convention give the same
    results as contiguous tables on BSHD tensors."""
    ids = wl.flux_ids(40, 10, 3)
    inp = wl.make_custom(2, 2, 128, ids.shape[1], axes=(16, 56, 56), seed=65, ids=ids)
    c, s = dup_tables(ids, inp.axes, inp.theta, torch.bfloat16)
    c, s = c[0].cuda(), s[0].cuda()
    c_t = c.t().contiguous().t()                      # a strided [S, D] view
    s_t = s.t().contiguous().t()
    assert not c_t.is_contiguous()
    d = to_dev(inp)
    ref = gpu_tab(cuda_lib, inp, (c, s, None, None), d=d)
    got = gpu_tab(cuda_lib, inp, (c_t, s_t, None, None), d=d)
    for key in ("o", "lse", "dk", "dv", "dwq", "dwk"):
        assert torch.equal(got[key], ref[key]), key
    compare("dq", got["dq"], f64(ref["dq"]), atol=1e-2, rel_fro=1e-3)   # accumulation order may differ

    q = d["q"].transpose(1, 2).contiguous().requires_grad_()          # BHSD tensors
    k = d["k"].transpose(1, 2).contiguous().requires_grad_()
    v = d["v"].transpose(1, 2).contiguous().requires_grad_()
    o = cuda_lib.rope_attention_bhsd(q, k, v, c, s, d["wq"], d["wk"], eps=inp.eps)
    assert o.shape == q.shape
    assert torch.equal(o.transpose(1, 2), ref["o"])
    o.backward(d["do"].transpose(1, 2))
    compare("dv", v.grad.transpose(1, 2), f64(ref["dv"]), atol=1e-2, rel_fro=1e-3)
    compare("dk", k.grad.transpose(1, 2), f64(ref["dk"]), atol=1e-2, rel_fro=1e-3)
    compare("dq", q.grad.transpose(1, 2), f64(ref["dq"]), atol=1e-2, rel_fro=1e-3)
