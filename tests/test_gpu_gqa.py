"""GPU parity of grouped K/V heads ("Metal Flash Attention", section "Fused
RoPE + SDPA": GQA inputs are rotated at the K/V head count and expanded
afterwards) against the fp64 oracle: query head h attends with K/V head
h / (H / H_kv); dk and dv sum the gradients of each group's query heads."""
import pytest
import torch

import workloads as wl
from _parity import compare_all, gpu_fwd_bwd, oracle_fwd_bwd, to_dev

pytestmark = pytest.mark.gpu


def grouped(inp, Hkv, seed):
    """The same inputs with k, v drawn at H_kv heads (in their dtypes)."""
    B, Skv, _, D = inp.k.shape
    g = torch.Generator().manual_seed(seed)
    inp.k = torch.randn(B, Skv, Hkv, D, generator=g).to(inp.k.dtype)
    inp.v = torch.randn(B, Skv, Hkv, D, generator=g).to(inp.v.dtype)
    return inp


def run(api, inp):
    got = gpu_fwd_bwd(api, inp)
    assert got["dk"].shape == inp.k.shape and got["dv"].shape == inp.v.shape
    compare_all(got, oracle_fwd_bwd(inp))
    return got


def test_gqa_group2_ragged_tiles_bool_mask(cuda_lib):
    ids = wl.flux_ids(44, 16, 3)                                    # S = 300
    inp = grouped(wl.make_custom(2, 4, 128, ids.shape[1], axes=(16, 56, 56), seed=91, ids=ids), 2, 92)
    m = torch.ones(2, 1, 1, ids.shape[1], dtype=torch.bool)
    m[0, 0, 0, 10:40] = False
    m[1, 0, 0, 130:290] = False                                    # a whole key tile of sample 1 is False
    inp.mask = m
    run(cuda_lib, inp)


def test_gqa_group6_per_head_additive_mask(cuda_lib):
    # H = 12 query heads over 2 K/V heads; the mask differs per query head
    inp = grouped(wl.make_custom(1, 12, 128, 200, axes=(16, 56, 56), seed=98, mask="additive",
                                 mask_shape=(1, 12, 200, 200), ids=torch.randint(0, 30, (1, 200, 3), dtype=torch.int32)),
                  2, 99)
    run(cuda_lib, inp)


def test_gqa_group6_bool_mask_per_head_broadcast(cuda_lib):
    # a [B, H, 1, S_kv] bool mask: one key term per (query head, key)
    inp = grouped(wl.make_custom(1, 6, 128, 260, axes=(128,), seed=100, mask="bool_random",
                                 mask_shape=(1, 6, 1, 260)), 1, 101)
    run(cuda_lib, inp)


def half_do(inp):
    """dO at half scale: the first rows of a causal call see one to three keys,
    and with unit-scale dO their gradients reach 4 to 6, where bf16's own
    resolution (an ulp of 2^-6 .. 2^-5) leaves no room under the 2e-2
    absolute bound; halving dO halves every gradient and keeps the case in the
    bound's intended range (errors relative to the values are unchanged)."""
    inp.do = (inp.do.float() * 0.5).to(inp.do.dtype)
    return inp


def test_mqa_causal(cuda_lib):
    inp = grouped(wl.make_custom(1, 6, 128, 200, axes=(128,), causal=True, seed=93), 1, 94)
    run(cuda_lib, half_do(inp))


def test_gqa_group2_causal_multi_tile(cuda_lib):
    inp = grouped(wl.make_custom(2, 4, 128, 520, axes=(128,), causal=True, seed=102), 2, 103)
    run(cuda_lib, half_do(inp))


def test_gqa_fp32_qk_cross_lengths(cuda_lib):
    g = torch.Generator().manual_seed(95)
    ids = torch.randint(0, 64, (1, 130, 3), generator=g, dtype=torch.int32)
    ids_k = torch.randint(0, 64, (1, 257, 3), generator=g, dtype=torch.int32)
    inp = wl.make_custom(2, 4, 128, 130, 257, axes=(16, 56, 56), qk_dtype="fp32", seed=96, ids=ids, ids_k=ids_k)
    run(cuda_lib, grouped(inp, 1, 97))


def test_gqa_deterministic_dk_dv_and_tile_counts(cuda_lib):
    inp = grouped(wl.make_custom(1, 6, 128, 384, axes=(128,), causal=True, seed=104), 2, 105)
    d = to_dev(inp)
    cuda_lib.st_reset_stats()
    a = gpu_fwd_bwd(cuda_lib, inp, d=d)
    st = cuda_lib.st_get_stats()
    n = 3  # 128-row tiles
    # forward: per query head n x n (query tile, key tile) pairs; backward: per
    # K/V head and key tile, the query tiles of each of the group's 3 heads
    assert st["tiles_total"] == 2 * 6 * n * n
    assert st["tiles_skipped"] == 2 * 6 * n * (n - 1) // 2
    b = gpu_fwd_bwd(cuda_lib, inp, d=d)
    for k in ("o", "lse", "dk", "dv", "dwk"):
        assert torch.equal(a[k], b[k]), k
