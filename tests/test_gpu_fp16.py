"""GPU parity of fp16 inputs ("Metal Flash Attention", section "Requirements":
FP16 and BF16 inputs run on low-precision kernels, FP32 accumulation) against
the fp64 oracle. With fp16 v the tensor-core operands (Q', K', P, V, dO, dS)
are fp16 instead of bf16; the softmax, the accumulators and the norm/rotation
arithmetic stay fp32. fp16 keeps 10 mantissa bits to bf16's 7, so these cases
are held to a quarter of the bf16 bound (max |err| <= 5e-3, relative Frobenius
<= 2.5e-3) on O, dQ, dK and dV; LSE and the norm-weight gradients keep the
bf16 bounds."""
import pytest
import torch

import workloads as wl
from _parity import compare, gpu_fwd_bwd, oracle_fwd_bwd

pytestmark = pytest.mark.gpu

ATOL16, REL16 = 5e-3, 2.5e-3


def run(api, inp, keys=("o", "lse", "dq", "dk", "dv", "dwq", "dwk")):
    got = gpu_fwd_bwd(api, inp)
    ref = oracle_fwd_bwd(inp)
    for k in keys:
        if k in ("o", "dq", "dk", "dv"):
            assert got[k].dtype == (inp.v.dtype if k in ("o", "dv") else inp.q.dtype), k
            ma, rf = compare(k, got[k], ref[k], atol=ATOL16, rel_fro=REL16)
        else:
            ma, rf = compare(k, got[k], ref[k], check_max=k == "lse")
        print(f"  {k:4s} max_abs={ma:.3e} rel_fro={rf:.3e}")
    return got


def test_fp16_ragged_tiles(cuda_lib):
    ids = wl.flux_ids(44, 16, 3)  # S = 300: three 128-row tiles, the last one ragged
    run(cuda_lib, wl.make_custom(2, 3, 128, ids.shape[1], axes=(16, 56, 56), seed=120, ids=ids, qk_dtype="fp16",
                                 v_dtype="fp16"))


def test_fp16_bool_padding_mask(cuda_lib):
    inp = wl.make_custom(2, 2, 128, 260, axes=(128,), seed=121, qk_dtype="fp16", v_dtype="fp16", mask="bool_random",
                         mask_shape=(2, 1, 1, 260))
    run(cuda_lib, inp)


def test_fp16_additive_mask_per_query(cuda_lib):
    inp = wl.make_custom(1, 2, 128, 200, axes=(128,), seed=122, qk_dtype="fp16", v_dtype="fp16", mask="additive",
                         mask_shape=(1, 2, 200, 200))
    run(cuda_lib, inp)


def test_fp16_causal(cuda_lib):
    inp = wl.make_custom(1, 2, 128, 300, axes=(128,), seed=123, qk_dtype="fp16", v_dtype="fp16", causal=True)
    inp.do = (inp.do.float() * 0.5).to(inp.do.dtype)  # see test_gpu_gqa.half_do
    run(cuda_lib, inp)


def test_fp32_qk_with_fp16_v(cuda_lib):
    # the fp16 autocast mix: fp32 q/k (after the model's norm) with fp16 v,
    # cast to fp16 on load
    ids = wl.flux_ids(16, 12, 3)
    inp = wl.make_custom(1, 2, 128, ids.shape[1], axes=(16, 56, 56), seed=124, ids=ids, qk_dtype="fp32",
                         v_dtype="fp16")
    run(cuda_lib, inp)


def test_fp16_grouped_kv_heads(cuda_lib):
    inp = wl.make_custom(1, 4, 128, 256, axes=(128,), seed=125, qk_dtype="fp16", v_dtype="fp16")
    g = torch.Generator().manual_seed(126)
    inp.k = torch.randn(1, 256, 2, 128, generator=g).to(torch.float16)
    inp.v = torch.randn(1, 256, 2, 128, generator=g).to(torch.float16)
    run(cuda_lib, inp)


def test_mixed_16bit_types_are_rejected(cuda_lib):
    inp = wl.make_custom(1, 1, 128, 64, axes=(128,), seed=127, qk_dtype="bf16", v_dtype="fp16")
    with pytest.raises(cuda_lib.StError, match="v's dtype"):
        gpu_fwd_bwd(cuda_lib, inp, backward=False)
