"""GPU parity: the CUDA path (through the C-ABI) against the fp64 oracle on the
same seeded inputs, at sizes that span several 128-row tiles with ragged
tails, plus the edge cases of the method (masks of every broadcast pattern,
all-false tiles, fully masked rows, causal, mixed dtypes, strided views,
cross-attention lengths, empty inputs)."""
import numpy as np
import pytest
import torch

import workloads as wl
from _parity import compare, compare_all, gpu_fwd_bwd, oracle_fwd_bwd, to_dev

pytestmark = pytest.mark.gpu


def flux_inputs(B, H, n_text, grid, seed, qk="bf16", mask="none", axes=(16, 56, 56), theta=1e4, **kw):
    ids = wl.flux_ids(n_text, grid, len(axes))
    S = ids.shape[1]
    return wl.make_custom(B, H, 128, S, axes=axes, theta=theta, qk_dtype=qk, seed=seed, ids=ids, mask=mask, **kw)


def run_case(api, inp, scale=None, keys=("o", "lse", "dq", "dk", "dv", "dwq", "dwk")):
    got = gpu_fwd_bwd(api, inp, scale=scale)
    ref = oracle_fwd_bwd(inp, scale=scale)
    return compare_all(got, ref, keys), got, ref


def test_tiny_flux_config(cuda_lib):
    run_case(cuda_lib, wl.make("tiny_flux"))


def test_ragged_multi_tile(cuda_lib):
    inp = flux_inputs(2, 3, 44, 16, seed=21)   # S = 300: tiles 128, 128, 44
    run_case(cuda_lib, inp)


def test_single_head_batch(cuda_lib):
    inp = flux_inputs(3, 1, 16, 8, seed=22)
    run_case(cuda_lib, inp)


def test_cross_lengths(cuda_lib):
    g = torch.Generator().manual_seed(5)
    ids = torch.randint(0, 64, (1, 200, 3), generator=g, dtype=torch.int32)
    ids_k = torch.randint(0, 64, (1, 333, 3), generator=g, dtype=torch.int32)
    inp = wl.make_custom(2, 2, 128, 200, 333, axes=(16, 56, 56), seed=23, ids=ids, ids_k=ids_k)
    run_case(cuda_lib, inp)


def test_one_axis_long_positions(cuda_lib):
    inp = wl.make_custom(1, 2, 128, 384, axes=(128,), seed=24, ids=wl.linear_ids(384) + 7800)
    run_case(cuda_lib, inp)


def test_four_axes_theta_2e3(cuda_lib):
    inp = flux_inputs(1, 2, 32, 16, seed=25, axes=(32, 32, 32, 32), theta=2e3)
    run_case(cuda_lib, inp)


def test_float_ids_per_sample(cuda_lib):
    g = torch.Generator().manual_seed(6)
    ids = (torch.rand(2, 260, 3, generator=g) * 100).float()
    inp = wl.make_custom(2, 2, 128, 260, axes=(16, 56, 56), seed=26, ids=ids)
    inp.ids = ids  # fp32 ids, one set per batch element
    run_case(cuda_lib, inp)


def test_custom_scale(cuda_lib):
    inp = flux_inputs(1, 2, 20, 12, seed=27)
    run_case(cuda_lib, inp, scale=0.05)


def test_bool_padding_mask_broadcast(cuda_lib):
    inp = flux_inputs(3, 2, 150, 12, seed=28)   # S = 294
    m = torch.ones(3, 1, 1, inp.k.shape[1], dtype=torch.bool)
    m[0, 0, 0, 40:150] = False
    m[1, 0, 0, 0:130] = False                 # a whole key tile (0..127) all False for b=1
    m[2, 0, 0, 149:150] = False
    inp.mask = m
    run_case(cuda_lib, inp)


def test_bool_full_mask_mixed_tiles(cuda_lib):
    B, H, S = 2, 2, 300
    g = torch.Generator().manual_seed(7)
    m = torch.rand(B, H, S, S, generator=g) < 0.6
    m[:, :, :, :128] &= torch.rand(B, H, S, 1, generator=g) < 0.95
    m[0, 1, 128:256, 128:256] = False         # an all-False tile
    m[1, 0, 0:128, 256:] = True               # an all-True tile
    m[0, 0, 5, :] = False                     # a fully masked row
    inp = flux_inputs(B, H, 44, 16, seed=29)
    inp.mask = m
    res, got, _ = run_case(cuda_lib, inp)
    assert torch.all(got["o"][0, 5, 0] == 0) and torch.isneginf(got["lse"][0, 0, 5])
    assert torch.all(got["dq"][0, 5, 0] == 0)


def test_bool_mask_query_dependent_broadcast(cuda_lib):
    S = 260
    g = torch.Generator().manual_seed(8)
    m = torch.rand(1, 1, S, S, generator=g) < 0.5
    m[..., 0] = True
    inp = wl.make_custom(2, 2, 128, S, axes=(128,), seed=30)
    inp.mask = m
    run_case(cuda_lib, inp)


@pytest.mark.parametrize("shape", ["full", "bcast_key", "bcast_head"])
def test_additive_f32_mask(cuda_lib, shape):
    B, H, S = 2, 2, 270
    ms = {"full": (B, H, S, S), "bcast_key": (B, 1, 1, S), "bcast_head": (1, H, S, S)}[shape]
    inp = wl.make_custom(B, H, 128, S, axes=(128,), seed=31, mask="additive", mask_shape=ms)
    run_case(cuda_lib, inp)


def test_additive_bf16_mask(cuda_lib):
    inp = wl.make_custom(2, 2, 128, 200, axes=(128,), seed=32, mask="additive_bf16", mask_shape=(2, 2, 200, 200))
    run_case(cuda_lib, inp)


@pytest.mark.parametrize("S", [256, 300, 77])
def test_causal(cuda_lib, S):
    inp = wl.make_custom(2, 2, 128, S, axes=(128,), seed=33 + S, causal=True)
    # the first rows see one to three keys and their gradients reach 4-6, where
    # a bf16 ulp leaves no room under the absolute bound: dO at half scale, as
    # in the other causal cases (test_gpu_gqa.half_do)
    inp.do = (inp.do.float() * 0.5).to(inp.do.dtype)
    run_case(cuda_lib, inp)


def test_mixed_dtype_fp32_qk_bf16_v(cuda_lib):
    inp = flux_inputs(2, 2, 100, 12, seed=34, qk="fp32")
    m = torch.ones(2, 1, 1, inp.k.shape[1], dtype=torch.bool)
    m[0, 0, 0, 70:100] = False
    inp.mask = m
    res, got, _ = run_case(cuda_lib, inp)
    assert got["dq"].dtype == torch.float32 and got["dk"].dtype == torch.float32
    assert got["o"].dtype == torch.bfloat16


def test_strided_views_bhsd_and_fused_qkv(cuda_lib):
    base = flux_inputs(2, 3, 44, 16, seed=35)
    B, S, H, D = base.q.shape
    d = to_dev(base)
    # q as transpose(1, 2) of a BHSD tensor; k, v as views into a fused QKV buffer
    q_bhsd = d["q"].transpose(1, 2).contiguous()
    q_view = q_bhsd.transpose(1, 2)
    qkv = torch.stack([d["q"], d["k"], d["v"]], dim=2).contiguous()  # [B,S,3,H,D]
    k_view, v_view = qkv[:, :, 1], qkv[:, :, 2]
    assert not q_view.is_contiguous() and not k_view.is_contiguous()
    d2 = dict(d, q=q_view, k=k_view, v=v_view)
    got = gpu_fwd_bwd(cuda_lib, base, d=d2)
    ref = gpu_fwd_bwd(cuda_lib, base, d=d)
    for k in ("o", "lse", "dk", "dv", "dwk"):
        assert torch.equal(got[k], ref[k]), k
    # dq is bf16 and its fp32 accumulation order (atomic adds across key tiles)
    # differs between runs, so single elements may differ by one bf16 ulp
    compare("dq", got["dq"], ref["dq"].double().cpu().numpy(), atol=1e-2, rel_fro=1e-3)


def test_all_true_mask_is_identical_to_no_mask(cuda_lib):
    inp = flux_inputs(1, 2, 40, 12, seed=36)
    d = to_dev(inp)
    ref = gpu_fwd_bwd(cuda_lib, inp, d=d)
    cuda_lib.st_reset_stats()
    d2 = dict(d, mask=torch.ones(1, 1, 1, inp.k.shape[1], dtype=torch.bool, device="cuda"))
    got = gpu_fwd_bwd(cuda_lib, inp, d=d2)
    for k in ("o", "lse", "dk", "dv", "dwk"):
        assert torch.equal(got[k], ref[k]), k
    st = cuda_lib.st_get_stats()
    assert st["mask_all_true_skipped"] == 2  # forward and backward each detect it


def test_causal_tile_skip_counter(cuda_lib):
    S = 512
    inp = wl.make_custom(1, 1, 128, S, axes=(128,), seed=37, causal=True)
    cuda_lib.st_reset_stats()
    gpu_fwd_bwd(cuda_lib, inp, backward=False)
    st = cuda_lib.st_get_stats()
    n = S // 128
    assert st["tiles_total"] == n * n
    assert st["tiles_skipped"] == n * (n - 1) // 2


def test_deterministic_dk_dv_dw(cuda_lib):
    inp = flux_inputs(1, 3, 44, 16, seed=38)
    d = to_dev(inp)
    a = gpu_fwd_bwd(cuda_lib, inp, d=d)
    b = gpu_fwd_bwd(cuda_lib, inp, d=d)
    for k in ("o", "lse", "dk", "dv", "dwk"):
        assert torch.equal(a[k], b[k]), k


@pytest.mark.parametrize("mask", ["none", "bool", "additive"])
def test_backward_reusing_forward_tables(cuda_lib, mask):
    """A backward that reuses the forward's tables and mask tile classes from a
    shared workspace gives the same results as one that rebuilds them."""
    kw = dict(mask_shape=(2, 1, 1, 300)) if mask == "bool" else dict(mask_shape=(2, 3, 300, 300))
    inp = wl.make_custom(2, 3, 128, 300, axes=(16, 56, 56), seed=43, mask={"none": "none", "bool": "bool_random",
                                                                           "additive": "additive"}[mask],
                         ids=torch.randint(0, 40, (2, 300, 3), dtype=torch.int32), **kw)
    d = to_dev(inp)
    ref = gpu_fwd_bwd(cuda_lib, inp, d=d)
    ws = torch.empty(cuda_lib.st_rope_attn_workspace_size(d["q"], d["k"], d["v"], d["ids"], inp.axes, inp.theta,
                                                          d["mask"], False, for_backward=True),
                     dtype=torch.uint8, device="cuda")
    ws.fill_(0xAB)
    o, lse = cuda_lib.st_rope_attn_fwd(d["q"], d["k"], d["v"], d["wq"], d["wk"], inp.eps, d["ids"], inp.axes,
                                       inp.theta, mask=d["mask"], workspace=ws)
    got = dict(o=o, lse=lse)
    got["dq"], got["dk"], got["dv"], got["dwq"], got["dwk"] = cuda_lib.st_rope_attn_bwd(
        d["q"], d["k"], d["v"], d["wq"], d["wk"], inp.eps, d["ids"], inp.axes, inp.theta, o, lse, d["do"],
        mask=d["mask"], workspace=ws, reuse_tables=True)
    cuda_lib.st_check_status()
    for k in ("o", "lse", "dk", "dv", "dwk"):
        assert torch.equal(got[k], ref[k]), k
    compare("dq", got["dq"], ref["dq"].double().cpu().numpy(), atol=1e-2, rel_fro=1e-3)
    compare("dwq", got["dwq"], ref["dwq"].double().cpu().numpy(), check_max=False, rel_fro=1e-5)


def test_empty_inputs(cuda_lib):
    inp = wl.make_custom(1, 2, 128, 0, 0, axes=(128,), seed=39)
    d = to_dev(inp)
    o, lse = cuda_lib.st_rope_attn_fwd(d["q"], d["k"], d["v"], d["wq"], d["wk"], 1e-6, d["ids"], (128,), 1e4)
    assert o.numel() == 0 and lse.numel() == 0
    # keys but no queries: dk/dv/dw are zero
    inp = wl.make_custom(1, 2, 128, 0, 130, axes=(128,), seed=40, ids=torch.zeros(1, 0, 1, dtype=torch.int32),
                         ids_k=wl.linear_ids(130))
    d = to_dev(inp)
    o, lse = cuda_lib.st_rope_attn_fwd(d["q"], d["k"], d["v"], d["wq"], d["wk"], 1e-6, d["ids"], (128,), 1e4,
                                       ids_k=d["ids_k"])
    dq, dk, dv, dwq, dwk = cuda_lib.st_rope_attn_bwd(d["q"], d["k"], d["v"], d["wq"], d["wk"], 1e-6, d["ids"],
                                                     (128,), 1e4, o, lse, d["do"], ids_k=d["ids_k"])
    torch.cuda.synchronize()
    assert torch.all(dk == 0) and torch.all(dv == 0) and torch.all(dwq == 0) and torch.all(dwk == 0)
    # queries but no keys: O = 0, LSE = -inf
    inp = wl.make_custom(1, 2, 128, 50, 0, axes=(128,), seed=41, ids_k=torch.zeros(1, 0, 1, dtype=torch.int32))
    d = to_dev(inp)
    o, lse = cuda_lib.st_rope_attn_fwd(d["q"], d["k"], d["v"], d["wq"], d["wk"], 1e-6, d["ids"], (128,), 1e4,
                                       ids_k=d["ids_k"])
    torch.cuda.synchronize()
    assert torch.all(o == 0) and torch.all(torch.isneginf(lse))


def test_autograd_function(cuda_lib):
    inp = flux_inputs(1, 2, 20, 10, seed=42)
    d = to_dev(inp)
    q, k, v = (d[n].clone().requires_grad_() for n in ("q", "k", "v"))
    wq, wk = d["wq"].clone().requires_grad_(), d["wk"].clone().requires_grad_()
    o = cuda_lib.rope_attention(q, k, v, wq, wk, d["ids"], inp.axes, inp.theta, inp.eps)
    (o.float() * d["do"].float()).sum().backward()
    ref = oracle_fwd_bwd(inp)
    compare("o", o, ref["o"])
    for name, t in (("dq", q), ("dk", k), ("dv", v), ("dwq", wq), ("dwk", wk)):
        compare(name, t.grad, ref[name], check_max=name not in ("dwq", "dwk"))


def test_bounded_wait_reports_timeout_and_context_survives(cuda_lib):
    before = cuda_lib.st_get_stats()["timeouts"]
    cuda_lib.st_selftest_wait_timeout(2_000_000)  # ~1 ms of clock64 cycles
    with pytest.raises(cuda_lib.StError) as ei:
        cuda_lib.st_check_status()
    assert ei.value.status == cuda_lib.ST_ERR_TIMEOUT
    assert cuda_lib.st_get_stats()["timeouts"] == before + 1
    cuda_lib.st_check_status()  # the record is cleared
    run_case(cuda_lib, wl.make("tiny_flux"))  # and the context still computes correctly


# The forward takes P = exp2(s - bound) with a fixed reference when the mask
# adds no values, the operands are bf16 and the score bound
# scale*log2(e)*D*max|w_q|*max|w_k|*1.02 is at most 56 (the normalised operands
# cannot exceed it), else an online row maximum. With |w| clamped to
# [0.7, 1.3], scale = 0.2 puts the bound past the limit (63.7) while the scores
# stay moderate; one pair of q weights at 2.5 puts it just under (52.2), where P
# spans about 2^-54 .. 2^-40.

def _weights(inp, big=None):
    inp.wq = inp.wq.clamp(0.7, 1.3)
    inp.wk = inp.wk.clamp(0.7, 1.3)
    if big is not None:
        inp.wq[0:2] = big
    return inp


@pytest.mark.parametrize("mask,causal", [("none", False), ("bool", False), ("none", True)])
def test_online_maximum_past_the_bound(cuda_lib, mask, causal):
    kw = dict(mask="bool_random", mask_shape=(1, 1, 1, 260)) if mask == "bool" else {}
    inp = _weights(wl.make_custom(1, 2, 128, 260, axes=(128,), seed=150, causal=causal, **kw))
    if causal:
        inp.do = (inp.do.float() * 0.5).to(inp.do.dtype)  # see test_gpu_gqa.half_do
    got, ref = gpu_fwd_bwd(cuda_lib, inp, scale=0.2), oracle_fwd_bwd(inp, scale=0.2)
    compare_all(got, ref, keys=("o", "lse", "dv", "dwq", "dwk"))
    # dq and dk are proportional to the softmax scale: the absolute bound, set
    # for scale = 1/sqrt(D), grows with it (0.2 * sqrt(128) = 2.26)
    for k in ("dq", "dk"):
        compare(k, got[k], ref[k], atol=2e-2 * 0.2 * 128 ** 0.5)


@pytest.mark.parametrize("mask,causal", [("bool", False), ("none", True)])
def test_fixed_reference_near_its_limit(cuda_lib, mask, causal):
    kw = dict(mask="bool_random", mask_shape=(2, 1, 1, 300)) if mask == "bool" else {}
    inp = _weights(wl.make_custom(2, 2, 128, 300, axes=(128,), seed=152, causal=causal, **kw), 2.5)
    bound = 128 ** -0.5 * np.log2(np.e) * 128 * float(inp.wq.abs().max()) * float(inp.wk.abs().max()) * 1.02
    assert 50.0 < bound <= 56.0
    if causal:
        inp.do = (inp.do.float() * 0.5).to(inp.do.dtype)
    compare_all(gpu_fwd_bwd(cuda_lib, inp), oracle_fwd_bwd(inp))
