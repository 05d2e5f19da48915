"""Full-size parity: each workload at its real size, run through the same C-ABI
calls, with the same shared workspace and table reuse, that the benchmark
times, checked against the oracle on sampled heads (the oracle recomputes those
(b, h) heads one by one; heads are independent). The norm-weight gradients sum
over every head: the Flux1 1024px case checks them against the oracle's sums
over all 24 heads."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from _parity import compare, f64

pytestmark = pytest.mark.gpu


def head_oracle(inp, b, h, mask_head=None):
    """Oracle fwd+bwd of head (b, h) alone (inputs sliced to B=1, H=1)."""
    sl = lambda t: f64(t[b:b + 1, :, h:h + 1])
    m = None
    if mask_head is not None:
        m = mask_head.double().numpy()[None, None]
    elif inp.mask is not None:
        mm = inp.mask[min(b, inp.mask.shape[0] - 1):][:1][:, min(h, inp.mask.shape[1] - 1):][:, :1]
        m = mm.numpy() if mm.dtype == torch.bool else mm.double().numpy()
    ids = inp.ids[min(b, inp.ids.shape[0] - 1):][:1].numpy()
    args = (sl(inp.q), sl(inp.k), sl(inp.v), f64(inp.wq), f64(inp.wk), inp.eps, ids, inp.axes, inp.theta)
    kw = dict(mask=m, causal=inp.causal)
    o, lse = oracle.fwd(*args, **kw)
    dq, dk, dv, _, _ = oracle.bwd(*args, sl(inp.do), **kw)
    return dict(o=o[0, :, 0], lse=lse[0, 0], dq=dq[0, :, 0], dk=dk[0, :, 0], dv=dv[0, :, 0])


def run_full(api, inp, heads, mask_dev=None, mask_heads=None):
    dev = "cuda"
    q, k, v, do = (t.to(dev) for t in (inp.q, inp.k, inp.v, inp.do))
    wq, wk, ids = inp.wq.to(dev), inp.wk.to(dev), inp.ids.to(dev)
    mask = mask_dev if mask_dev is not None else (None if inp.mask is None else inp.mask.to(dev))
    ws = torch.empty(api.st_rope_attn_workspace_size(q, k, v, ids, inp.axes, inp.theta, mask, inp.causal,
                                                     for_backward=True), dtype=torch.uint8, device=dev)
    o, lse = api.st_rope_attn_fwd(q, k, v, wq, wk, inp.eps, ids, inp.axes, inp.theta, mask=mask, causal=inp.causal,
                                  workspace=ws)
    dq, dk, dv, dwq, dwk = api.st_rope_attn_bwd(q, k, v, wq, wk, inp.eps, ids, inp.axes, inp.theta, o, lse, do,
                                                mask=mask, causal=inp.causal, workspace=ws, reuse_tables=True)
    api.st_check_status()
    torch.cuda.synchronize()
    assert torch.isfinite(dwq).all() and torch.isfinite(dwk).all()
    got = dict(o=o, lse=lse, dq=dq, dk=dk, dv=dv, dwq=dwq, dwk=dwk)
    for (b, h) in heads:
        ref = head_oracle(inp, b, h, None if mask_heads is None else mask_heads[(b, h)])
        print(f"head ({b},{h})")
        for key in ("o", "lse", "dq", "dk", "dv"):
            g = got[key][b, h] if key == "lse" else got[key][b, :, h]
            ma, rf = compare(key, g, ref[key])
            print(f"  {key:4s} max_abs={ma:.3e} rel_fro={rf:.3e}")
    return got


def test_flux1_1024_all_true_mask(cuda_lib):
    inp = wl.make("flux1_1024")
    cuda_lib.st_reset_stats()
    got = run_full(cuda_lib, inp, heads=[(0, 0), (0, 23)])
    # the forward detects the all-True mask; the backward reuses its tile classes
    assert cuda_lib.st_get_stats()["mask_all_true_skipped"] == 1
    # the norm-weight gradients sum over all 24 heads: the oracle's full sums
    # (an all-True mask is the same as none, which the oracle's pins establish)
    args = (f64(inp.q), f64(inp.k), f64(inp.v), f64(inp.wq), f64(inp.wk), inp.eps, inp.ids.numpy(), inp.axes,
            inp.theta)
    _, _, _, dwq, dwk = oracle.bwd(*args, f64(inp.do))
    for key, ref in (("dwq", dwq), ("dwk", dwk)):
        ma, rf = compare(key, got[key], ref, check_max=False)
        print(f"  {key:4s} max_abs={ma:.3e} rel_fro={rf:.3e}")


def test_flux1_padded_batch_mixed_dtype(cuda_lib):
    inp = wl.make("flux1_padded")
    assert inp.q.dtype == torch.float32 and inp.v.dtype == torch.bfloat16
    cuda_lib.st_reset_stats()
    run_full(cuda_lib, inp, heads=[(0, 5), (3, 17)])
    st = cuda_lib.st_get_stats()
    assert st["mixed_dtype_calls"] == 2
    # key tiles lying wholly inside a sample's padded text range [L_b, 512) are
    # skipped by every query tile, once in the forward and once in the backward
    B, S, H, _ = inp.q.shape
    n_qt = (S + 127) // 128
    dead = sum(sum(1 for t in range(4) if t * 128 >= L) for L in inp.meta["valid_text"])
    assert st["tiles_skipped"] == 2 * H * n_qt * dead


def test_causal_8k(cuda_lib):
    inp = wl.make("causal_8k")
    run_full(cuda_lib, inp, heads=[(1, 9)])


def test_causal_8k_additive_mask(cuda_lib):
    inp = wl.make("causal_8k_additive")
    B, H, S = inp.q.shape[0], inp.q.shape[2], inp.q.shape[1]
    mask = torch.empty(B, H, S, S, dtype=torch.float32, device="cuda")
    heads = [(0, 3)]
    mask_heads = {}
    for b in range(B):
        for h in range(H):
            m = wl.additive_mask_head("causal_8k_additive", b, h)
            mask[b, h].copy_(m)
            if (b, h) in heads:
                mask_heads[(b, h)] = m
    run_full(cuda_lib, inp, heads=heads, mask_dev=mask, mask_heads=mask_heads)


def test_flux2_long(cuda_lib):
    inp = wl.make("flux2_long")
    run_full(cuda_lib, inp, heads=[(0, 31)])


@pytest.mark.parametrize("name,head", [("flux1_probe_6144", (0, 7)), ("flux1_probe_24576", (0, 11))])
def test_flux1_probe_shapes(cuda_lib, name, head):
    # the pages' probe shapes (1024px and 2048px images, no text tokens): the
    # whole problem runs on the GPU, one head is recomputed by the oracle
    # (at S = 24576 that is about a minute of host time)
    inp = wl.make(name)
    run_full(cuda_lib, inp, heads=[head])
