"""Helpers for the GPU-vs-oracle parity tests.

Tolerances (fixed by the specification of this op): bf16 runs must match the
fp64 oracle with max |err| <= 2e-2 and relative Frobenius error <= 1e-2 on O,
dQ, dK and dV. The log-sum-exp and the norm-weight gradients, which the
specification does not list, use LSE max |err| <= 2e-2 and dW relative
Frobenius <= 1e-2.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle

ATOL = 2e-2
REL_FRO = 1e-2


def f64(t):
    return None if t is None else t.detach().double().cpu().numpy()


def compare(name, got, ref, atol=ATOL, rel_fro=REL_FRO, check_max=True):
    g = f64(got) if isinstance(got, torch.Tensor) else np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert g.shape == ref.shape, (name, g.shape, ref.shape)
    inf_g, inf_r = np.isinf(g), np.isinf(ref)
    assert np.array_equal(inf_g, inf_r), f"{name}: infinities differ ({inf_g.sum()} vs {inf_r.sum()})"
    if inf_r.any():
        assert np.array_equal(g[inf_r], ref[inf_r]), f"{name}: signs of infinities differ"
    fin = ~inf_r
    assert np.all(np.isfinite(g[fin])), f"{name}: non-finite values"
    err = np.abs(g[fin] - ref[fin])
    max_abs = float(err.max()) if err.size else 0.0
    nref = float(np.linalg.norm(ref[fin]))
    rel = float(np.linalg.norm(g[fin] - ref[fin]) / nref) if nref > 0 else float(np.linalg.norm(g[fin]))
    if check_max:
        assert max_abs <= atol, f"{name}: max_abs={max_abs:.3e} > {atol}  (rel_fro={rel:.3e})"
    assert rel <= rel_fro, f"{name}: rel_fro={rel:.3e} > {rel_fro}  (max_abs={max_abs:.3e})"
    return max_abs, rel


def to_dev(inp, dev="cuda"):
    g = lambda t: None if t is None else t.to(dev)
    return dict(q=g(inp.q), k=g(inp.k), v=g(inp.v), do=g(inp.do), wq=g(inp.wq), wk=g(inp.wk), ids=g(inp.ids),
                ids_k=g(inp.ids_k), mask=g(inp.mask))


def gpu_fwd_bwd(api, inp, d=None, scale=None, backward=True):
    d = d or to_dev(inp)
    o, lse = api.st_rope_attn_fwd(d["q"], d["k"], d["v"], d["wq"], d["wk"], inp.eps, d["ids"], inp.axes, inp.theta,
                                  mask=d["mask"], causal=inp.causal, scale=scale, ids_k=d["ids_k"])
    out = {"o": o, "lse": lse}
    if backward:
        dq, dk, dv, dwq, dwk = api.st_rope_attn_bwd(d["q"], d["k"], d["v"], d["wq"], d["wk"], inp.eps, d["ids"],
                                                    inp.axes, inp.theta, o, lse, d["do"], mask=d["mask"],
                                                    causal=inp.causal, scale=scale, ids_k=d["ids_k"])
        out.update(dq=dq, dk=dk, dv=dv, dwq=dwq, dwk=dwk)
    api.st_check_status()
    torch.cuda.synchronize()
    return out


def oracle_fwd_bwd(inp, scale=None, heads=None, backward=True, mask=None):
    m = inp.mask if mask is None else mask
    m = None if m is None else (m.numpy() if m.dtype == torch.bool else m.double().numpy())
    args = (f64(inp.q), f64(inp.k), f64(inp.v), f64(inp.wq), f64(inp.wk), inp.eps, inp.ids.numpy(), inp.axes,
            inp.theta)
    kw = dict(mask=m, causal=inp.causal, scale=scale, ids_k=None if inp.ids_k is None else inp.ids_k.numpy(),
              heads=heads)
    o, lse = oracle.fwd(*args, **kw)
    out = {"o": o, "lse": lse}
    if backward:
        dq, dk, dv, dwq, dwk = oracle.bwd(*args, f64(inp.do), **kw)
        out.update(dq=dq, dk=dk, dv=dv, dwq=dwq, dwk=dwk)
    return out


def compare_all(got, ref, keys=("o", "lse", "dq", "dk", "dv", "dwq", "dwk"), heads=None):
    """Compares GPU outputs with oracle outputs; with `heads`, only those (b, h)."""
    res = {}
    for k in keys:
        if k not in ref:
            continue
        g, r = got[k], ref[k]
        if heads is not None and k in ("o", "dq", "dk", "dv"):
            g = torch.stack([g[b, :, h] for b, h in heads])
            r = np.stack([r[b, :, h] for b, h in heads])
        elif heads is not None and k == "lse":
            g = torch.stack([g[b, h] for b, h in heads])
            r = np.stack([r[b, h] for b, h in heads])
        elif heads is not None:
            continue
        # dW sums B*S*H row terms, so its scale grows with the problem: it is
        # held to the relative Frobenius bound only.
        res[k] = compare(k, g, r, check_max=k not in ("dwq", "dwk"))
        print(f"  {k:4s} max_abs={res[k][0]:.3e} rel_fro={res[k][1]:.3e}")
    return res
