"""The forward entry point that allocates nothing (st_rope_attn_fwd_noalloc).

It exists for callers that cannot allocate device memory (graph capture into a
fixed memory plan, plugins of inference runtimes that only hand out input and
output buffers, serving processes that forbid allocation after start-up). Its
scratch is a static device array inside the library. These checks call it
through the C-ABI, twice in a row on the same inputs, and compare each result
with the regular entry point's (which takes a caller workspace), within the
parity tolerances used everywhere else; they also check that a call needing
more than the built-in scratch is refused before anything is launched.

This file is collected last on purpose, so that a run stopping at the first
failure has already run every other test.
"""
import ctypes

import pytest
import torch

import workloads as wl
from _parity import compare

pytestmark = pytest.mark.gpu


def _inputs():
    ids = wl.flux_ids(44, 16, 3)          # S = 300: two full key tiles and a ragged one
    inp = wl.make_custom(2, 3, 128, ids.shape[1], axes=(16, 56, 56), seed=77, ids=ids)
    m = torch.ones(2, 1, 1, ids.shape[1], dtype=torch.bool)
    m[0, 0, 0, 10:44] = False             # text padding in sample 0 (mixed tile)
    m[1, 0, 0, 0:128] = False             # a whole key tile masked in sample 1 (skipped tile)
    inp.mask = m
    return inp


def test_noalloc_forward_matches_workspace_forward_twice(cuda_lib):
    inp = _inputs()
    dev = "cuda"
    q, k, v, wq, wk, ids, mask = (t.to(dev) for t in (inp.q, inp.k, inp.v, inp.wq, inp.wk, inp.ids, inp.mask))
    o_ref, lse_ref = cuda_lib.st_rope_attn_fwd(q, k, v, wq, wk, inp.eps, ids, inp.axes, inp.theta, mask=mask)
    torch.cuda.synchronize()
    o_ref, lse_ref = o_ref.double().cpu().numpy(), lse_ref.double().cpu().numpy()
    for _ in range(2):
        o = torch.full_like(q, float("nan"), dtype=v.dtype)
        lse = torch.full((q.shape[0], q.shape[2], q.shape[1]), float("nan"), dtype=torch.float32, device=dev)
        cuda_lib.st_rope_attn_fwd_noalloc(q, k, v, wq, wk, inp.eps, ids, inp.axes, inp.theta, mask=mask, o=o,
                                          lse=lse)
        cuda_lib.st_check_status()
        torch.cuda.synchronize()
        compare("o", o, o_ref)
        compare("lse", lse, lse_ref)


def test_noalloc_rejects_scratch_beyond_its_capacity(cuda_lib):
    # per-sample ids for 4 samples of 9000 tokens: 4 * 9000 * 512 B of tables > 16 MiB
    B, S, H = 4, 9000, 1
    q = torch.zeros(B, S, H, 128, dtype=torch.bfloat16, device="cuda")
    w = torch.ones(128, dtype=torch.float32, device="cuda")
    ids = torch.zeros(B, S, 1, dtype=torch.int32, device="cuda")
    launches = cuda_lib.st_get_stats()["kernel_launches"]
    with pytest.raises(cuda_lib.StError) as ei:
        cuda_lib.st_rope_attn_fwd_noalloc(q, q, q, w, w, 1e-6, ids, (128,), 1e4)
    assert ei.value.status == cuda_lib.ST_ERR_WORKSPACE
    assert "built-in scratch" in str(ei.value)
    assert cuda_lib.st_get_stats()["kernel_launches"] == launches
    assert ctypes.sizeof(ctypes.c_int) == 4
