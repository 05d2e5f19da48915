"""GPU parity of all-fp32 inputs against the fp64 oracle at the fp32 bound:
max |err| <= 1e-4 and relative Frobenius <= 1e-4 on O, dQ, dK and dV, LSE
max |err| <= 1e-4, norm-weight gradients relative Frobenius <= 1e-4. fp32 q,
k and v select the exact-fp32 kernels (every product and sum in fp32);
"Metal Flash Attention", section "Requirements", runs FP32 natively and its
section "Synthetic Memory Probe" reports FP32 parity against SDPA."""
import pytest
import torch

import workloads as wl
from _parity import compare, gpu_fwd_bwd, oracle_fwd_bwd, to_dev

pytestmark = pytest.mark.gpu

TOL32 = 1e-4


def run(api, inp, keys=("o", "lse", "dq", "dk", "dv", "dwq", "dwk")):
    got = gpu_fwd_bwd(api, inp)
    ref = oracle_fwd_bwd(inp)
    for k in keys:
        if k in ("dwq", "dwk"):
            ma, rf = compare(k, got[k], ref[k], check_max=False, rel_fro=TOL32)
        else:
            assert got[k].dtype == torch.float32, k
            ma, rf = compare(k, got[k], ref[k], atol=TOL32, rel_fro=TOL32)
        print(f"  {k:4s} max_abs={ma:.3e} rel_fro={rf:.3e}")
    return got


def f32_inputs(B, H, S, seed, Skv=None, **kw):
    return wl.make_custom(B, H, 128, S, Skv, seed=seed, qk_dtype="fp32", v_dtype="fp32", **kw)


def test_fp32_ragged_flux_ids(cuda_lib):
    ids = wl.flux_ids(44, 16, 3)  # S = 300
    run(cuda_lib, f32_inputs(2, 2, ids.shape[1], 130, axes=(16, 56, 56), ids=ids))


def test_fp32_causal(cuda_lib):
    run(cuda_lib, f32_inputs(1, 2, 200, 131, axes=(128,), causal=True))


def test_fp32_bool_and_additive_masks(cuda_lib):
    run(cuda_lib, f32_inputs(2, 2, 150, 132, axes=(128,), mask="bool_random", mask_shape=(2, 1, 1, 150)))
    run(cuda_lib, f32_inputs(1, 2, 130, 133, axes=(128,), mask="additive", mask_shape=(1, 2, 130, 130)))


def test_fp32_cross_lengths_and_grouped_heads(cuda_lib):
    g = torch.Generator().manual_seed(134)
    ids = torch.randint(0, 50, (1, 90, 3), generator=g, dtype=torch.int32)
    ids_k = torch.randint(0, 50, (1, 170, 3), generator=g, dtype=torch.int32)
    inp = f32_inputs(1, 4, 90, 135, Skv=170, axes=(16, 56, 56), ids=ids, ids_k=ids_k)
    inp.k = torch.randn(1, 170, 2, 128, generator=g)
    inp.v = torch.randn(1, 170, 2, 128, generator=g)
    run(cuda_lib, inp)


def test_fp32_deterministic(cuda_lib):
    inp = f32_inputs(1, 2, 140, 136, axes=(128,))
    d = to_dev(inp)
    a = gpu_fwd_bwd(cuda_lib, inp, d=d)
    b = gpu_fwd_bwd(cuda_lib, inp, d=d)
    for k in ("o", "lse", "dq", "dk", "dv", "dwq", "dwk"):
        assert torch.equal(a[k], b[k]), k
