"""CPU checks of bench.py's eager arm (torch rms_norm + table rotation + SDPA):
its rotary tables equal the oracle's angles, and the composition, run in fp32
on the CPU, matches the fp64 oracle forward and backward."""
import numpy as np
import torch

import bench
import oracle
import workloads as wl


def test_eager_tables_match_oracle_angles():
    ids = wl.flux_ids(3, 4, 3, grid_w=5)
    c, s = bench.rope_tables_torch(ids, (16, 56, 56), 1e4)
    phi = oracle.rope_angles(ids.numpy(), (16, 56, 56), 1e4)
    np.testing.assert_allclose(c.numpy(), np.repeat(np.cos(phi), 2, -1), rtol=0, atol=1e-6)
    np.testing.assert_allclose(s.numpy(), np.repeat(np.sin(phi), 2, -1), rtol=0, atol=1e-6)


def test_eager_composition_matches_oracle():
    ids = wl.flux_ids(4, 3, 3)
    inp = wl.make_custom(2, 2, 128, ids.shape[1], axes=(16, 56, 56), qk_dtype="fp32", v_dtype="fp32", seed=71,
                         ids=ids)
    m = torch.ones(2, 1, 1, ids.shape[1], dtype=torch.bool)
    m[1, 0, 0, :3] = False
    c, s = bench.rope_tables_torch(ids, inp.axes, inp.theta)
    leaves = [t.clone().requires_grad_() for t in (inp.q, inp.k, inp.v, inp.wq, inp.wk)]
    o = bench.eager_attention(*leaves, inp.eps, c, s, mask=m)
    grads = torch.autograd.grad(o, leaves, inp.do)
    f64 = lambda t: t.double().numpy()
    args = (f64(inp.q), f64(inp.k), f64(inp.v), f64(inp.wq), f64(inp.wk), inp.eps, ids.numpy(), inp.axes, inp.theta)
    ro, _ = oracle.fwd(*args, mask=m.numpy())
    rg = oracle.bwd(*args, f64(inp.do), mask=m.numpy())
    np.testing.assert_allclose(o.detach().numpy(), ro, rtol=1e-4, atol=1e-5)
    for got, ref in zip(grads, rg):
        np.testing.assert_allclose(got.numpy(), ref, rtol=1e-4, atol=2e-5)


def test_probe_workload_shapes():
    """The pages' probe shapes: B=1 H=24 D=128 at S=6144 and S=24576, and the
    Z-Image DiT shape (1, 30, 4128, 128) in bf16."""
    want = {"flux1_probe_6144": (1, 24, 6144), "flux1_probe_24576": (1, 24, 24576), "zimage_dit": (1, 30, 4128)}
    for name, (B, H, S) in want.items():
        c = wl.WORKLOADS[name]
        ids = wl.flux_ids(c["n_text"], c["grid"], len(c["axes"]), c.get("grid_w"))
        assert (c["B"], c["H"], ids.shape[1], c["D"]) == (B, H, S, 128), name
        assert ids.shape[2] == len(c["axes"]) and sum(c["axes"]) == 128
        assert c["qk_dtype"] == c["v_dtype"] == "bf16" and c["mask"] == "none" and not c["causal"]
        # distinct image positions, text tokens at the origin
        img = ids[0, c["n_text"]:]
        assert len({tuple(r) for r in img.tolist()}) == img.shape[0]
        assert int(ids[0, :c["n_text"]].abs().sum()) == 0
    inp = wl.make("zimage_dit")
    assert tuple(inp.q.shape) == (1, 4128, 30, 128) and inp.q.dtype == torch.bfloat16 and inp.mask is None
    flops_f, flops_b = bench.nominal_flops(inp)
    assert flops_f == 4.0 * 30 * 4128 * 4128 * 128 and flops_b == 2.5 * flops_f
