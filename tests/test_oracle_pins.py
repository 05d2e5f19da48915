"""Pins for the fp64 oracle: closed forms, invariants, finite differences and
a library special case, chosen so that a dropped term, a wrong sign or index,
or a transposed operand anywhere in the oracle fails at least one of them.

Sources: "Metal Flash Attention" (SimpleTuner docs) sections "Fused RoPE +
SDPA" and "Enable In SimpleTuner"; "Flux-family attention: flash-attn and
other backends fail in an autocast context" (diffusers issue 14104), "Root
cause" list (norm -> RoPE -> attention).
"""
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _np(t):
    return t.double().numpy() if isinstance(t, torch.Tensor) else np.asarray(t, dtype=np.float64)


def _fwd(inp, **kw):
    args = dict(mask=None if inp.mask is None else inp.mask.numpy(), causal=inp.causal,
                ids_k=None if inp.ids_k is None else inp.ids_k.numpy())
    args.update(kw)
    return oracle.fwd(_np(inp.q), _np(inp.k), _np(inp.v), _np(inp.wq), _np(inp.wk), inp.eps, inp.ids.numpy(),
                      inp.axes, inp.theta, **args)


def _tiny(B=1, H=2, Sq=8, Skv=None, D=8, axes=(2, 2, 4), seed=0, **kw):
    Skv = Sq if Skv is None else Skv
    g = torch.Generator().manual_seed(seed + 100)
    ids = torch.randint(0, 9, (1, Sq, len(axes)), generator=g, dtype=torch.int32)
    ids_k = torch.randint(0, 9, (1, Skv, len(axes)), generator=g, dtype=torch.int32) if Skv != Sq else None
    inp = wl.make_custom(B, H, D, Sq, Skv, axes=axes, qk_dtype="fp32", v_dtype="fp32", seed=seed, ids=ids,
                         ids_k=ids_k, **kw)
    return inp


# --------------------------------------------------------------------- RoPE
def test_rope_angles_closed_forms():
    rows = []
    with open(os.path.join(GOLDEN, "rope_angle_closed_forms.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            th, axes, a, j, idv, exp = line.split()
            rows.append((float(th), tuple(int(x) for x in axes.split(",")), int(a), int(j), float(idv), float(exp)))
    assert len(rows) >= 10
    for th, axes, a, j, idv, exp in rows:
        ids = np.zeros((1, len(axes)))
        ids[0, a] = idv
        phi = oracle.rope_angles(ids, axes, th)[0]
        pair = sum(axes[:a]) // 2 + j
        assert phi[pair] == pytest.approx(exp, rel=1e-13, abs=1e-15), (th, axes, a, j)
        # every pair owned by another axis sees id 0 -> angle 0
        others = [p for p in range(sum(axes) // 2) if not (sum(axes[:a]) // 2 <= p < sum(axes[:a + 1]) // 2)]
        assert np.all(phi[others] == 0.0)


def test_rotation_sign_closed_form():
    # x = (1, 0): RMSNorm (w=1, eps=0) gives (sqrt2, 0); rotating by phi gives
    # sqrt2 (cos phi, sin phi) under the counter-clockwise convention.
    for phi in (0.0, 1.0, -0.7, math.pi / 2):
        y = oracle.qk_transform(np.array([[1.0, 0.0]]), np.ones(2), 0.0, np.array([[phi]]))[0]
        assert y == pytest.approx([math.sqrt(2) * math.cos(phi), math.sqrt(2) * math.sin(phi)], abs=1e-15)
    # x = (0, 1) rotates to sqrt2 (-sin phi, cos phi)
    y = oracle.qk_transform(np.array([[0.0, 1.0]]), np.ones(2), 0.0, np.array([[0.3]]))[0]
    assert y == pytest.approx([-math.sqrt(2) * math.sin(0.3), math.sqrt(2) * math.cos(0.3)], abs=1e-15)


def test_identity_at_position_zero_matches_torch_rmsnorm():
    g = torch.Generator().manual_seed(1)
    x = torch.randn(37, 128, generator=g, dtype=torch.float64)
    w = 1 + 0.1 * torch.randn(128, generator=g, dtype=torch.float64)
    ref = F.rms_norm(x, (128,), w, 1e-6).numpy()
    out = oracle.qk_transform(x.numpy(), w.numpy(), 1e-6, np.zeros((37, 64)))
    np.testing.assert_allclose(out, ref, rtol=1e-13, atol=1e-13)


def test_rope_preserves_pair_norms_and_relative_angles():
    rng = np.random.default_rng(2)
    D = 128
    x = rng.standard_normal((20, D))
    y = rng.standard_normal((20, D))
    w = 1 + 0.1 * rng.standard_normal(D)
    phi = rng.uniform(-50, 50, (20, D // 2))
    psi = rng.uniform(-50, 50, (20, D // 2))
    x0 = oracle.qk_transform(x, w, 1e-6, np.zeros_like(phi))
    xr = oracle.qk_transform(x, w, 1e-6, phi)
    n0 = np.hypot(x0[:, 0::2], x0[:, 1::2])
    nr = np.hypot(xr[:, 0::2], xr[:, 1::2])
    np.testing.assert_allclose(nr, n0, rtol=1e-12)
    # q'.k' depends only on the angle difference: shift both by the same c
    c = rng.uniform(-30, 30, (1, D // 2))
    yr = oracle.qk_transform(y, w, 1e-6, psi)
    xs = oracle.qk_transform(x, w, 1e-6, phi + c)
    ys = oracle.qk_transform(y, w, 1e-6, psi + c)
    np.testing.assert_allclose(np.sum(xs * ys, 1), np.sum(xr * yr, 1), rtol=1e-10, atol=1e-10)
    # and it does change when only one side is shifted (guards a vacuous pass)
    assert np.max(np.abs(np.sum(xs * yr, 1) - np.sum(xr * yr, 1))) > 1e-3


def test_rmsnorm_invariants():
    rng = np.random.default_rng(3)
    D = 128
    x = rng.standard_normal((10, D)) * rng.uniform(0.1, 10, (10, 1))
    ones = np.ones(D)
    y = oracle.qk_transform(x, ones, 0.0, np.zeros((10, D // 2)))
    np.testing.assert_allclose(np.sqrt(np.mean(y * y, 1)), 1.0, rtol=1e-13)
    y2 = oracle.qk_transform(3.7 * x, ones, 0.0, np.zeros((10, D // 2)))
    np.testing.assert_allclose(y2, y, rtol=1e-12, atol=1e-13)
    # constant row a with eps: a / sqrt(a^2 + eps); weight scales per dimension
    a, eps = 0.25, 0.01
    w = np.linspace(0.5, 1.5, D)
    y3 = oracle.qk_transform(np.full((1, D), a), w, eps, np.zeros((1, D // 2)))[0]
    np.testing.assert_allclose(y3, w * a / math.sqrt(a * a + eps), rtol=1e-14)


# ---------------------------------------------------------------- attention
def test_all_true_mask_equals_no_mask():
    inp = _tiny(B=2, Sq=9)
    o0, l0 = _fwd(inp, mask=None)
    o1, l1 = _fwd(inp, mask=np.ones((1, 1, 1, 9), dtype=bool))
    np.testing.assert_array_equal(o1, o0)
    np.testing.assert_array_equal(l1, l0)


def test_row_constant_additive_mask_is_shift_invariant():
    inp = _tiny(B=2, Sq=9)
    o0, l0 = _fwd(inp, mask=None)
    c = np.random.default_rng(4).uniform(-5, 5, (2, 2, 9, 1))
    o1, l1 = _fwd(inp, mask=np.broadcast_to(c, (2, 2, 9, 9)).copy())
    np.testing.assert_allclose(o1, o0, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(l1, l0 + c[..., 0], rtol=1e-12, atol=1e-12)


def test_bool_false_equals_additive_minus_inf():
    inp = _tiny(B=2, Sq=10)
    rng = np.random.default_rng(5)
    mb = rng.uniform(size=(2, 2, 10, 10)) < 0.6
    mb[..., 0] = True  # keep every row alive
    ma = np.where(mb, 0.0, -np.inf)
    o1, l1 = _fwd(inp, mask=mb)
    o2, l2 = _fwd(inp, mask=ma)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)
    o0, _ = _fwd(inp, mask=None)
    assert np.max(np.abs(o1 - o0)) > 1e-3


def test_padded_keys_equal_deleted_keys():
    # broadcast [B,1,1,S_kv] padding mask == calling with those keys removed
    inp = _tiny(B=3, Sq=12)
    valid = [5, 12, 8]
    m = np.zeros((3, 1, 1, 12), dtype=bool)
    for b, n in enumerate(valid):
        m[b, 0, 0, :n] = True
    o, lse = _fwd(inp, mask=m)
    for b, n in enumerate(valid):
        sl = slice(b, b + 1)
        ob, lb = oracle.fwd(_np(inp.q[sl]), _np(inp.k[sl, :n]), _np(inp.v[sl, :n]), _np(inp.wq), _np(inp.wk),
                            inp.eps, inp.ids.numpy(), inp.axes, inp.theta, ids_k=inp.ids[:, :n].numpy())
        np.testing.assert_allclose(o[b], ob[0], rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(lse[b], lb[0], rtol=1e-12, atol=1e-13)


def test_causal_rows():
    inp = _tiny(B=2, Sq=11)
    oc, lc = _fwd(inp, causal=True)
    o0, l0 = _fwd(inp, causal=False)
    v = _np(inp.v)
    np.testing.assert_array_equal(oc[:, 0], v[:, 0])           # row 0 sees only key 0
    np.testing.assert_allclose(oc[:, -1], o0[:, -1], rtol=1e-12, atol=1e-13)  # last row sees everything
    np.testing.assert_allclose(lc[:, :, -1], l0[:, :, -1], rtol=1e-12)
    assert np.max(np.abs(oc[:, 3] - o0[:, 3])) > 1e-3


def test_identical_keys_return_mean_of_v():
    inp = _tiny(B=1, H=2, Sq=7)
    k = inp.k.clone()
    k[:] = k[:, :1]
    ids = inp.ids.clone()
    ids[:] = ids[:, :1]
    q = _np(inp.q)
    o, lse = oracle.fwd(q, _np(k), _np(inp.v), _np(inp.wq), _np(inp.wk), inp.eps, ids.numpy(), inp.axes,
                        inp.theta)
    np.testing.assert_allclose(o, np.broadcast_to(_np(inp.v).mean(1, keepdims=True), o.shape), rtol=1e-12,
                               atol=1e-13)
    # lse = s + ln(S_kv) with s the (common) score of each row
    phi = oracle.rope_angles(ids.numpy()[0], inp.axes, inp.theta)
    D = q.shape[-1]
    for h in range(2):
        qp = oracle.qk_transform(q[0, :, h], _np(inp.wq), inp.eps, phi)
        kp = oracle.qk_transform(_np(k)[0, :1, h], _np(inp.wk), inp.eps, phi[:1])
        s = qp @ kp[0] / math.sqrt(D)
        np.testing.assert_allclose(lse[0, h], s + math.log(7), rtol=1e-12)


def test_single_key_and_two_key_closed_forms():
    inp = _tiny(B=1, H=2, Sq=5, Skv=2)
    q, k, v = _np(inp.q), _np(inp.k), _np(inp.v)
    D = q.shape[-1]
    phq = oracle.rope_angles(inp.ids.numpy()[0], inp.axes, inp.theta)
    phk = oracle.rope_angles(inp.ids_k.numpy()[0], inp.axes, inp.theta)
    # S_kv = 1: O = v_0, lse = s_i0
    o1, l1 = oracle.fwd(q, k[:, :1], v[:, :1], _np(inp.wq), _np(inp.wk), inp.eps, inp.ids.numpy(), inp.axes,
                        inp.theta, ids_k=inp.ids_k[:, :1].numpy())
    np.testing.assert_allclose(o1, np.broadcast_to(v[:, :1], o1.shape), rtol=1e-13, atol=1e-14)
    o2, l2 = oracle.fwd(q, k, v, _np(inp.wq), _np(inp.wk), inp.eps, inp.ids.numpy(), inp.axes, inp.theta,
                        ids_k=inp.ids_k.numpy())
    for h in range(2):
        qp = oracle.qk_transform(q[0, :, h], _np(inp.wq), inp.eps, phq)
        kp = oracle.qk_transform(k[0, :, h], _np(inp.wk), inp.eps, phk)
        s = qp @ kp.T / math.sqrt(D)
        np.testing.assert_allclose(l1[0, h], s[:, 0], rtol=1e-12)
        # two keys: O = sigmoid(s0 - s1) v0 + sigmoid(s1 - s0) v1, lse = s1 + log1p(exp(s0 - s1))
        a = 1.0 / (1.0 + np.exp(-(s[:, 0] - s[:, 1])))
        ref = a[:, None] * v[0, 0, h] + (1 - a)[:, None] * v[0, 1, h]
        np.testing.assert_allclose(o2[0, :, h], ref, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(l2[0, h], s[:, 1] + np.log1p(np.exp(s[:, 0] - s[:, 1])), rtol=1e-12)


def test_fully_masked_row_reading():
    inp = _tiny(B=1, Sq=6)
    m = np.ones((1, 1, 6, 6), dtype=bool)
    m[0, 0, 2, :] = False
    o, lse = _fwd(inp, mask=m)
    assert np.all(o[0, 2] == 0.0) and np.all(np.isneginf(lse[0, :, 2]))
    assert np.all(np.isfinite(lse[0, :, [0, 1, 3, 4, 5]]))
    dq, dk, dv, dwq, dwk = oracle.bwd(_np(inp.q), _np(inp.k), _np(inp.v), _np(inp.wq), _np(inp.wk), inp.eps,
                                      inp.ids.numpy(), inp.axes, inp.theta, _np(inp.do), mask=m)
    assert np.all(dq[0, 2] == 0.0)
    assert np.all(np.isfinite(dk)) and np.all(np.isfinite(dv))


# ------------------------------------------------------- finite differences
def _loss(inp, q, k, v, wq, wk, dout, mask, causal):
    o, _ = oracle.fwd(q, k, v, wq, wk, inp.eps, inp.ids.numpy(), inp.axes, inp.theta, mask=mask, causal=causal,
                      ids_k=None if inp.ids_k is None else inp.ids_k.numpy())
    return float(np.sum(o * dout))


@pytest.mark.parametrize("case", ["plain", "bool", "additive", "causal", "cross"])
def test_gradients_match_central_differences(case):
    Skv = 6 if case == "cross" else None
    inp = _tiny(B=1, H=2, Sq=5 if case == "cross" else 6, Skv=Skv, D=8, axes=(2, 2, 4), seed=7)
    Sq, Skv = inp.q.shape[1], inp.k.shape[1]
    q, k, v, wq, wk, dout = (_np(t).copy() for t in (inp.q, inp.k, inp.v, inp.wq, inp.wk, inp.do))
    rng = np.random.default_rng(8)
    mask = None
    if case == "bool":
        mask = rng.uniform(size=(1, 2, Sq, Skv)) < 0.6
        mask[..., 0] = True
    elif case == "additive":
        mask = rng.uniform(-4, 0, (1, 1, Sq, Skv))
    causal = case == "causal"
    dq, dk, dv, dwq, dwk = oracle.bwd(q, k, v, wq, wk, inp.eps, inp.ids.numpy(), inp.axes, inp.theta, dout,
                                      mask=mask, causal=causal,
                                      ids_k=None if inp.ids_k is None else inp.ids_k.numpy())
    h = 1e-6
    for arr, grad in ((q, dq), (k, dk), (v, dv), (wq, dwq), (wk, dwk)):
        fd = np.zeros_like(arr)
        flat, fdf = arr.reshape(-1), fd.reshape(-1)
        for i in range(flat.size):
            x0 = flat[i]
            flat[i] = x0 + h
            lp = _loss(inp, q, k, v, wq, wk, dout, mask, causal)
            flat[i] = x0 - h
            lm = _loss(inp, q, k, v, wq, wk, dout, mask, causal)
            flat[i] = x0
            fdf[i] = (lp - lm) / (2 * h)
        np.testing.assert_allclose(grad, fd, rtol=1e-6, atol=1e-7)


# ------------------------------------------------- library special case
def _torch_reference(inp, mask, causal):
    """torch fp64 CPU: F.rms_norm, complex-multiply RoPE, SDPA, autograd."""
    q = inp.q.double().requires_grad_()
    k = inp.k.double().requires_grad_()
    v = inp.v.double().requires_grad_()
    wq = inp.wq.double().requires_grad_()
    wk = inp.wk.double().requires_grad_()
    D = q.shape[-1]
    phi_q = torch.from_numpy(oracle.rope_angles(inp.ids.numpy(), inp.axes, inp.theta))    # [1,Sq,D/2]
    ids_k = inp.ids if inp.ids_k is None else inp.ids_k
    phi_k = torch.from_numpy(oracle.rope_angles(ids_k.numpy(), inp.axes, inp.theta))

    def rot(x, phi):  # x [B,S,H,D]; Z-Image style complex multiply
        xc = torch.view_as_complex(x.reshape(*x.shape[:-1], D // 2, 2))
        r = torch.polar(torch.ones_like(phi), phi)[:, :, None, :]
        return torch.view_as_real(xc * r).reshape(x.shape)

    qp = rot(F.rms_norm(q, (D,), wq, inp.eps), phi_q).transpose(1, 2)
    kp = rot(F.rms_norm(k, (D,), wk, inp.eps), phi_k).transpose(1, 2)
    vt = v.transpose(1, 2)
    am = None if mask is None else torch.from_numpy(np.asarray(mask))
    o = F.scaled_dot_product_attention(qp, kp, vt, attn_mask=am, is_causal=causal).transpose(1, 2)
    s = qp @ kp.transpose(-1, -2) / math.sqrt(D)
    if am is not None:
        s = s.masked_fill(~am, -math.inf) if am.dtype == torch.bool else s + am
    if causal:
        Sq, Sk = s.shape[-2:]
        s = s.masked_fill(torch.ones(Sq, Sk, dtype=torch.bool).triu(1), -math.inf)
    lse = torch.logsumexp(s, -1)
    (o * inp.do.double()).sum().backward()
    return o.detach().numpy(), lse.detach().numpy(), [t.grad.numpy() for t in (q, k, v, wq, wk)]


@pytest.mark.parametrize("case", ["plain", "bool_bcast", "bool_full", "additive", "causal", "cross"])
def test_matches_torch_fp64_composition(case):
    B, H, Sq = 2, 3, 40
    Skv = 29 if case == "cross" else Sq
    g = torch.Generator().manual_seed(11)
    axes = (16, 56, 56)
    ids = torch.randint(0, 64, (1, Sq, 3), generator=g, dtype=torch.int32)
    ids_k = torch.randint(0, 64, (1, Skv, 3), generator=g, dtype=torch.int32) if case == "cross" else None
    inp = wl.make_custom(B, H, 128, Sq, Skv, axes=axes, qk_dtype="fp32", v_dtype="fp32", seed=12, ids=ids,
                         ids_k=ids_k)
    rng = np.random.default_rng(13)
    mask = None
    if case == "bool_bcast":
        mask = np.ones((B, 1, 1, Skv), dtype=bool)
        mask[0, 0, 0, 5:17] = False
        mask[1, 0, 0, 30:] = False
    elif case == "bool_full":
        mask = rng.uniform(size=(B, H, Sq, Skv)) < 0.5
        mask[..., 3] = True
    elif case == "additive":
        mask = rng.uniform(-4, 0, (B, H, Sq, Skv))
    causal = case == "causal"
    o, lse = _fwd(inp, mask=mask, causal=causal)
    grads = oracle.bwd(_np(inp.q), _np(inp.k), _np(inp.v), _np(inp.wq), _np(inp.wk), inp.eps, inp.ids.numpy(),
                       inp.axes, inp.theta, _np(inp.do), mask=mask, causal=causal,
                       ids_k=None if ids_k is None else ids_k.numpy())
    ro, rl, rg = _torch_reference(inp, mask, causal)
    np.testing.assert_allclose(o, ro, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(lse, rl, rtol=1e-10, atol=1e-12)
    for got, ref in zip(grads, rg):
        np.testing.assert_allclose(got, ref, rtol=1e-9, atol=1e-11)


def test_heads_subset_matches_full():
    inp = _tiny(B=2, H=3, Sq=9)
    o, lse = _fwd(inp)
    os_, ls = _fwd(inp, heads=[(1, 2), (0, 1)])
    for b, h in [(1, 2), (0, 1)]:
        np.testing.assert_array_equal(os_[b, :, h], o[b, :, h])
        np.testing.assert_array_equal(ls[b, h], lse[b, h])
    assert np.all(np.isnan(os_[0, :, 0]))


# ------------------------------------------------- table form of the rotation
# "Metal Flash Attention", section "Fused RoPE + SDPA": the entry point takes
# pair-duplicated cos/sin tables of shape [S, D], [1, S, D] or [B, S, D].
def _dup_tables(phi):
    """Pair-duplicated (cos, sin) [..., S, D] of angles [..., S, D/2]."""
    return np.repeat(np.cos(phi), 2, axis=-1), np.repeat(np.sin(phi), 2, axis=-1)


@pytest.mark.parametrize("per_sample", [False, True])
def test_table_form_equals_angle_form(per_sample):
    """Tables holding cos/sin of the ids' angles give the ids' results."""
    B, H, Sq, Skv = 2, 2, 7, 5
    g = torch.Generator().manual_seed(21)
    Bi = B if per_sample else 1
    ids = torch.randint(0, 9, (Bi, Sq, 3), generator=g, dtype=torch.int32)
    ids_k = torch.randint(0, 9, (Bi, Skv, 3), generator=g, dtype=torch.int32)
    inp = wl.make_custom(B, H, 8, Sq, Skv, axes=(2, 2, 4), qk_dtype="fp32", v_dtype="fp32", seed=22, ids=ids,
                         ids_k=ids_k)
    cq, sq = _dup_tables(oracle.rope_angles(ids.numpy(), inp.axes, inp.theta))
    ck, sk = _dup_tables(oracle.rope_angles(ids_k.numpy(), inp.axes, inp.theta))
    if not per_sample:
        cq, sq, ck, sk = cq[0], sq[0], ck[0], sk[0]  # the [S, D] form
    args = (_np(inp.q), _np(inp.k), _np(inp.v), _np(inp.wq), _np(inp.wk), inp.eps)
    o, lse = oracle.fwd(*args, ids.numpy(), inp.axes, inp.theta, ids_k=ids_k.numpy())
    ot, lset = oracle.fwd_tab(*args, cq, sq, cos_k=ck, sin_k=sk)
    np.testing.assert_allclose(ot, o, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(lset, lse, rtol=1e-13, atol=1e-14)
    ga = oracle.bwd(*args, ids.numpy(), inp.axes, inp.theta, _np(inp.do), ids_k=ids_k.numpy())
    gt = oracle.bwd_tab(*args, cq, sq, _np(inp.do), cos_k=ck, sin_k=sk)
    for a, t in zip(ga, gt):
        np.testing.assert_allclose(t, a, rtol=1e-12, atol=1e-13)


def _rand_tables(rng, shape):
    """Tables that are neither pair-duplicated nor unit rotations, so that every
    index of the elementwise form and of its transpose is exercised."""
    return rng.uniform(-1.2, 1.2, shape), rng.uniform(-1.2, 1.2, shape)


def test_table_form_matches_torch_elementwise_composition():
    """Library special case: torch fp64 rms_norm, x * cos + rot(x) * sin with
    rot(x) = (-x1, x0) per pair, SDPA and autograd."""
    B, H, Sq, D = 2, 3, 11, 16
    inp = wl.make_custom(B, H, D, Sq, Sq, axes=(8, 8), qk_dtype="fp32", v_dtype="fp32", seed=23)
    rng = np.random.default_rng(24)
    cq, sq = _rand_tables(rng, (B, Sq, D))
    mask = rng.uniform(size=(B, 1, Sq, Sq)) < 0.7
    mask[..., 0] = True
    args = (_np(inp.q), _np(inp.k), _np(inp.v), _np(inp.wq), _np(inp.wk), inp.eps)
    o, lse = oracle.fwd_tab(*args, cq, sq, mask=mask)
    grads = oracle.bwd_tab(*args, cq, sq, _np(inp.do), mask=mask)

    q, k, v, wq, wk = (t.double().requires_grad_() for t in (inp.q, inp.k, inp.v, inp.wq, inp.wk))
    c = torch.from_numpy(cq)[:, :, None, :]
    s = torch.from_numpy(sq)[:, :, None, :]

    def rot(x):
        xp = x.reshape(*x.shape[:-1], D // 2, 2)
        return torch.stack((-xp[..., 1], xp[..., 0]), dim=-1).reshape(x.shape)

    def tr(x, w):
        n = F.rms_norm(x, (D,), w, inp.eps)
        return (n * c + rot(n) * s).transpose(1, 2)

    am = torch.from_numpy(mask)
    ro = F.scaled_dot_product_attention(tr(q, wq), tr(k, wk), v.transpose(1, 2), attn_mask=am).transpose(1, 2)
    sc = tr(q, wq) @ tr(k, wk).transpose(-1, -2) / math.sqrt(D)
    rl = torch.logsumexp(sc.masked_fill(~am, -math.inf), -1)
    (ro * inp.do.double()).sum().backward()
    np.testing.assert_allclose(o, ro.detach().numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(lse, rl.detach().numpy(), rtol=1e-10, atol=1e-12)
    for got, t in zip(grads, (q, k, v, wq, wk)):
        np.testing.assert_allclose(got, t.grad.numpy(), rtol=1e-9, atol=1e-11)


def test_table_form_gradients_match_central_differences():
    B, H, Sq, Skv, D = 1, 2, 5, 6, 8
    inp = wl.make_custom(B, H, D, Sq, Skv, axes=(4, 4), qk_dtype="fp32", v_dtype="fp32", seed=25)
    rng = np.random.default_rng(26)
    cq, sq = _rand_tables(rng, (Sq, D))
    ck, sk = _rand_tables(rng, (Skv, D))
    q, k, v, wq, wk, dout = (_np(t).copy() for t in (inp.q, inp.k, inp.v, inp.wq, inp.wk, inp.do))

    def loss():
        o, _ = oracle.fwd_tab(q, k, v, wq, wk, inp.eps, cq, sq, cos_k=ck, sin_k=sk, causal=False)
        return float(np.sum(o * dout))

    grads = oracle.bwd_tab(q, k, v, wq, wk, inp.eps, cq, sq, dout, cos_k=ck, sin_k=sk)
    h = 1e-6
    for arr, grad in zip((q, k, v, wq, wk), grads):
        fd = np.zeros_like(arr)
        flat, fdf = arr.reshape(-1), fd.reshape(-1)
        for i in range(flat.size):
            x0 = flat[i]
            flat[i] = x0 + h
            lp = loss()
            flat[i] = x0 - h
            lm = loss()
            flat[i] = x0
            fdf[i] = (lp - lm) / (2 * h)
        np.testing.assert_allclose(grad, fd, rtol=1e-6, atol=1e-7)


def test_table_form_transform_rows():
    """qk_transform_tab on duplicated tables equals qk_transform on the angles,
    and unit tables (cos 1, sin 0) leave the normalised rows unrotated."""
    rng = np.random.default_rng(27)
    x = rng.normal(size=(6, 8))
    w = 1 + 0.1 * rng.normal(size=8)
    phi = rng.uniform(-3, 3, (6, 4))
    c, s = _dup_tables(phi)
    np.testing.assert_allclose(oracle.qk_transform_tab(x, w, 1e-6, c, s), oracle.qk_transform(x, w, 1e-6, phi),
                               rtol=1e-14, atol=1e-15)
    r = 1 / np.sqrt(np.mean(x * x, -1, keepdims=True) + 1e-6)
    np.testing.assert_allclose(oracle.qk_transform_tab(x, w, 1e-6, np.ones_like(x), np.zeros_like(x)), x * r * w,
                               rtol=1e-14, atol=1e-15)


# ------------------------------------------------------ grouped K/V heads (GQA)
# "Metal Flash Attention", section "Fused RoPE + SDPA": GQA inputs (fewer K/V
# heads) are rotated at the K/V head count and expanded afterwards.
def _gqa(B=2, H=4, Hkv=2, Sq=7, Skv=6, D=8, axes=(2, 2, 4), seed=81):
    inp = _tiny(B=B, H=H, Sq=Sq, Skv=Skv, D=D, axes=axes, seed=seed)
    g = torch.Generator().manual_seed(seed + 1)
    inp.k = torch.randn(B, Skv, Hkv, D, generator=g)
    inp.v = torch.randn(B, Skv, Hkv, D, generator=g)
    return inp


def _ids_k(inp):
    return None if inp.ids_k is None else inp.ids_k.numpy()


def test_gqa_equals_expanded_heads():
    """Grouped heads = the same call on K/V expanded head by head
    (repeat_interleave), with dk, dv summed over each group."""
    inp = _gqa()
    H, Hkv = inp.q.shape[2], inp.k.shape[2]
    grp = H // Hkv
    rng = np.random.default_rng(82)
    mask = rng.uniform(size=(2, H, inp.q.shape[1], inp.k.shape[1])) < 0.7
    mask[..., 0] = True
    kx, vx = (np.repeat(_np(t), grp, axis=2) for t in (inp.k, inp.v))
    a = (_np(inp.q), _np(inp.k), _np(inp.v), _np(inp.wq), _np(inp.wk), inp.eps, inp.ids.numpy(), inp.axes, inp.theta)
    ax = (_np(inp.q), kx, vx, _np(inp.wq), _np(inp.wk), inp.eps, inp.ids.numpy(), inp.axes, inp.theta)
    o, lse = oracle.fwd(*a, mask=mask, ids_k=_ids_k(inp))
    ox, lsex = oracle.fwd(*ax, mask=mask, ids_k=_ids_k(inp))
    np.testing.assert_allclose(o, ox, rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(lse, lsex, rtol=1e-14, atol=1e-15)
    dq, dk, dv, dwq, dwk = oracle.bwd(*a, _np(inp.do), mask=mask, ids_k=_ids_k(inp))
    dqx, dkx, dvx, dwqx, dwkx = oracle.bwd(*ax, _np(inp.do), mask=mask, ids_k=_ids_k(inp))
    B, Skv, _, D = dk.shape
    np.testing.assert_allclose(dq, dqx, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(dk, dkx.reshape(B, Skv, Hkv, grp, D).sum(3), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(dv, dvx.reshape(B, Skv, Hkv, grp, D).sum(3), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(dwq, dwqx, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(dwk, dwkx, rtol=1e-12, atol=1e-13)


def test_gqa_matches_torch_enable_gqa():
    """Library special case: torch fp64 rms_norm, complex-multiply RoPE at the
    K/V head count, SDPA with enable_gqa, autograd."""
    B, H, Hkv, S, D = 2, 6, 2, 9, 16
    inp = wl.make_custom(B, H, D, S, S, axes=(8, 8), qk_dtype="fp32", v_dtype="fp32", seed=83)
    g = torch.Generator().manual_seed(84)
    inp.k = torch.randn(B, S, Hkv, D, generator=g)
    inp.v = torch.randn(B, S, Hkv, D, generator=g)
    q, k, v, wq, wk = (t.double().requires_grad_() for t in (inp.q, inp.k, inp.v, inp.wq, inp.wk))
    phi = torch.from_numpy(oracle.rope_angles(inp.ids.numpy(), inp.axes, inp.theta))

    def rot(x):
        xc = torch.view_as_complex(x.reshape(*x.shape[:-1], D // 2, 2))
        return torch.view_as_real(xc * torch.polar(torch.ones_like(phi), phi)[:, :, None, :]).reshape(x.shape)

    qp = rot(F.rms_norm(q, (D,), wq, inp.eps)).transpose(1, 2)
    kp = rot(F.rms_norm(k, (D,), wk, inp.eps)).transpose(1, 2)
    ro = F.scaled_dot_product_attention(qp, kp, v.transpose(1, 2), is_causal=True, enable_gqa=True).transpose(1, 2)
    (ro * inp.do.double()).sum().backward()
    a = (_np(inp.q), _np(inp.k), _np(inp.v), _np(inp.wq), _np(inp.wk), inp.eps, inp.ids.numpy(), inp.axes, inp.theta)
    o, _ = oracle.fwd(*a, causal=True)
    grads = oracle.bwd(*a, _np(inp.do), causal=True)
    np.testing.assert_allclose(o, ro.detach().numpy(), rtol=1e-10, atol=1e-12)
    for got, t in zip(grads, (q, k, v, wq, wk)):
        np.testing.assert_allclose(got, t.grad.numpy(), rtol=1e-9, atol=1e-11)


def test_gqa_gradients_match_central_differences():
    inp = _gqa(B=1, H=4, Hkv=2, Sq=5, Skv=6, seed=85)
    q, k, v, wq, wk, dout = (_np(t).copy() for t in (inp.q, inp.k, inp.v, inp.wq, inp.wk, inp.do))

    def loss():
        o, _ = oracle.fwd(q, k, v, wq, wk, inp.eps, inp.ids.numpy(), inp.axes, inp.theta, ids_k=_ids_k(inp))
        return float(np.sum(o * dout))

    grads = oracle.bwd(q, k, v, wq, wk, inp.eps, inp.ids.numpy(), inp.axes, inp.theta, dout, ids_k=_ids_k(inp))
    h = 1e-6
    for arr, grad in zip((q, k, v, wq, wk), grads):
        fd = np.zeros_like(arr)
        flat, fdf = arr.reshape(-1), fd.reshape(-1)
        for i in range(flat.size):
            x0 = flat[i]
            flat[i] = x0 + h
            lp = loss()
            flat[i] = x0 - h
            lm = loss()
            flat[i] = x0
            fdf[i] = (lp - lm) / (2 * h)
        np.testing.assert_allclose(grad, fd, rtol=1e-6, atol=1e-7)


def test_gqa_heads_subset_sums_its_listed_group():
    """With every query head of one group listed, that K/V head's dk, dv equal
    the full call's; the other K/V head stays untouched (NaN)."""
    inp = _gqa(B=1, H=4, Hkv=2, seed=86)
    a = (_np(inp.q), _np(inp.k), _np(inp.v), _np(inp.wq), _np(inp.wk), inp.eps, inp.ids.numpy(), inp.axes, inp.theta,
         _np(inp.do))
    full = oracle.bwd(*a, ids_k=_ids_k(inp))
    part = oracle.bwd(*a, ids_k=_ids_k(inp), heads=[(0, 2), (0, 3)])   # the group of K/V head 1
    np.testing.assert_allclose(part[1][:, :, 1], full[1][:, :, 1], rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(part[2][:, :, 1], full[2][:, :, 1], rtol=1e-13, atol=1e-14)
    assert np.all(np.isnan(part[1][:, :, 0])) and np.all(np.isnan(part[2][:, :, 0]))
    np.testing.assert_allclose(part[0][:, :, 2:], full[0][:, :, 2:], rtol=1e-13, atol=1e-14)
