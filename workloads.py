"""Seeded synthetic inputs for the fused QK-RMSNorm + RoPE + attention call.

This module only draws random numbers and lays out position ids; it holds
none of the method's arithmetic. Both the CUDA path and the fp64 oracle are fed
from it, so they see bit-identical inputs.

Recipe (all draws from one CPU ``torch.Generator`` per workload, in this
order): q, k, v, dO ~ N(0, 1) in fp32 then cast to the stored dtype;
w_q, w_k ~ 1 + N(0, 0.1) fp32; then the mask. Position ids are integers:
Flux text tokens (0, 0, 0) followed by the image grid (0, row, col) in
row-major order; the 4-axis long sequence uses (0, 0, 0, 0) / (0, 0, row, col);
the causal workload uses a single axis with ids 0..S-1.

The pages' own probe shapes ("Metal Flash Attention", sections "FLUX Sequence
Lengths" and "Synthetic Memory Probe": B=1 H=24 D=128 with S=6144 at 1024px
and S=24576 at 2048px; section "Fused RoPE + SDPA": the Z-Image DiT shape
(1, 30, 4128, 128) in bf16) are included as well. The pages do not give their
token composition; ids are inputs and do not change the cost, so the probe
shapes take a rectangular image grid without text (64 x 96 and 128 x 192) and
the DiT shape 32 text tokens plus a 64 x 64 grid, all with the Flux axes.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

# name -> (B, H, D, n_text, grid, S_1axis, axes, theta, q/k dtype, v dtype, mask kind, causal, seed)
WORKLOADS = {
    # B=1 H=2 D=128, 16 text + 8x8 image (S=80), bf16, no mask
    "tiny_flux": dict(B=1, H=2, D=128, n_text=16, grid=8, axes=(16, 56, 56), theta=1e4,
                      qk_dtype="bf16", v_dtype="bf16", mask="none", causal=False, seed=0),
    # Flux1 1024px: B=1 H=24, 512 text + 64x64 image = 4608, all-true bool mask [1,1,1,S]
    "flux1_1024": dict(B=1, H=24, D=128, n_text=512, grid=64, axes=(16, 56, 56), theta=1e4,
                       qk_dtype="bf16", v_dtype="bf16", mask="all_true", causal=False, seed=1),
    # Flux1 padded batch: B=4, q/k fp32 (autocast mix), v bf16, text padding mask [B,1,1,S]
    "flux1_padded": dict(B=4, H=24, D=128, n_text=512, grid=64, axes=(16, 56, 56), theta=1e4,
                         qk_dtype="fp32", v_dtype="bf16", mask="text_pad", causal=False, seed=2),
    # causal training: B=2 H=16 S=8192, 1-axis RoPE over 0..S-1
    "causal_8k": dict(B=2, H=16, D=128, S=8192, axes=(128,), theta=1e4,
                      qk_dtype="bf16", v_dtype="bf16", mask="none", causal=True, seed=3),
    # the same with an additive fp32 mask [B,H,S,S] ~ U(-4, 0), not causal
    "causal_8k_additive": dict(B=2, H=16, D=128, S=8192, axes=(128,), theta=1e4,
                               qk_dtype="bf16", v_dtype="bf16", mask="additive", causal=False, seed=3),
    # Flux2-style long sequence: B=1 H=48, 512 text + 128x128 image = 16896, 4 axes
    "flux2_long": dict(B=1, H=48, D=128, n_text=512, grid=128, axes=(32, 32, 32, 32), theta=2e3,
                       qk_dtype="bf16", v_dtype="bf16", mask="none", causal=False, seed=4),
    # the pages' probe shapes: B=1 H=24 S=6144 (1024px) and S=24576 (2048px), no mask
    "flux1_probe_6144": dict(B=1, H=24, D=128, n_text=0, grid=64, grid_w=96, axes=(16, 56, 56), theta=1e4,
                             qk_dtype="bf16", v_dtype="bf16", mask="none", causal=False, seed=5),
    "flux1_probe_24576": dict(B=1, H=24, D=128, n_text=0, grid=128, grid_w=192, axes=(16, 56, 56), theta=1e4,
                              qk_dtype="bf16", v_dtype="bf16", mask="none", causal=False, seed=6),
    # the Z-Image DiT shape (1, 30, 4128, 128) bf16: 32 text + 64x64 image
    "zimage_dit": dict(B=1, H=30, D=128, n_text=32, grid=64, axes=(16, 56, 56), theta=1e4,
                       qk_dtype="bf16", v_dtype="bf16", mask="none", causal=False, seed=7),
}

_DT = {"bf16": torch.bfloat16, "fp32": torch.float32, "fp16": torch.float16}


@dataclass
class Inputs:
    name: str
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    do: torch.Tensor
    wq: torch.Tensor
    wk: torch.Tensor
    ids: torch.Tensor            # [1|B, S, A] int32
    axes: tuple
    theta: float
    mask: torch.Tensor | None    # [B|1, H|1, Sq|1, Skv], bool or float, or None
    causal: bool
    eps: float = 1e-6
    ids_k: torch.Tensor | None = None
    meta: dict = field(default_factory=dict)

    @property
    def shape(self):
        return tuple(self.q.shape)


def flux_ids(n_text: int, grid: int, n_axes: int, grid_w: int | None = None) -> torch.Tensor:
    """[1, n_text + grid*grid_w, n_axes] int32: text (0,..,0), then an image of
    `grid` rows by `grid_w` (default `grid`) columns, (0,..,row,col) row-major."""
    grid_w = grid if grid_w is None else grid_w
    S = n_text + grid * grid_w
    ids = torch.zeros(1, S, n_axes, dtype=torch.int32)
    rows = torch.arange(grid, dtype=torch.int32).repeat_interleave(grid_w)
    cols = torch.arange(grid_w, dtype=torch.int32).repeat(grid)
    ids[0, n_text:, n_axes - 2] = rows
    ids[0, n_text:, n_axes - 1] = cols
    return ids


def linear_ids(S: int) -> torch.Tensor:
    return torch.arange(S, dtype=torch.int32).reshape(1, S, 1)


def randn(shape, gen, dtype):
    return torch.randn(shape, generator=gen, dtype=torch.float32).to(dtype)


def make_custom(B, H, D, Sq, Skv=None, axes=None, theta=1e4, qk_dtype="bf16", v_dtype="bf16", mask="none",
                causal=False, seed=0, ids=None, ids_k=None, mask_shape=None, name="custom") -> Inputs:
    """General generator used by the parity tests (any shape, ragged S)."""
    Skv = Sq if Skv is None else Skv
    axes = (D,) if axes is None else tuple(axes)
    g = torch.Generator().manual_seed(seed)
    q = randn((B, Sq, H, D), g, _DT[qk_dtype])
    k = randn((B, Skv, H, D), g, _DT[qk_dtype])
    v = randn((B, Skv, H, D), g, _DT[v_dtype])
    do = randn((B, Sq, H, D), g, _DT[v_dtype])
    wq = 1.0 + 0.1 * torch.randn(D, generator=g, dtype=torch.float32)
    wk = 1.0 + 0.1 * torch.randn(D, generator=g, dtype=torch.float32)
    if ids is None:
        ids = linear_ids(Sq).expand(1, Sq, 1).repeat(1, 1, len(axes)) if len(axes) > 1 else linear_ids(Sq)
    if ids_k is None and Skv != Sq:
        ids_k = linear_ids(Skv).repeat(1, 1, len(axes))
    m = None
    ms = mask_shape or (B, 1, 1, Skv)
    if mask == "all_true":
        m = torch.ones(ms, dtype=torch.bool)
    elif mask == "bool_random":
        m = torch.rand(ms, generator=g) < 0.7
    elif mask == "additive":
        m = -4.0 * torch.rand(ms, generator=g, dtype=torch.float32)
    elif mask == "additive_bf16":
        m = (-4.0 * torch.rand(ms, generator=g, dtype=torch.float32)).to(torch.bfloat16)
    elif mask != "none":
        raise ValueError(mask)
    return Inputs(name, q, k, v, do, wq, wk, ids.contiguous().to(torch.int32), axes, float(theta), m, causal,
                  ids_k=None if ids_k is None else ids_k.contiguous().to(torch.int32))


def make(name: str, with_mask: bool = True) -> Inputs:
    """The named workload, on the CPU. For the additive [B,H,S,S] variant the
    mask is produced per head by ``additive_mask_head`` (8.6 GB in total), so
    ``mask`` is None here and ``meta['mask_per_head']`` is set."""
    c = WORKLOADS[name]
    B, H, D = c["B"], c["H"], c["D"]
    if "grid" in c:
        ids = flux_ids(c["n_text"], c["grid"], len(c["axes"]), c.get("grid_w"))
    else:
        ids = linear_ids(c["S"])
    S = ids.shape[1]
    g = torch.Generator().manual_seed(c["seed"])
    q = randn((B, S, H, D), g, _DT[c["qk_dtype"]])
    k = randn((B, S, H, D), g, _DT[c["qk_dtype"]])
    v = randn((B, S, H, D), g, _DT[c["v_dtype"]])
    do = randn((B, S, H, D), g, _DT[c["v_dtype"]])
    wq = 1.0 + 0.1 * torch.randn(D, generator=g, dtype=torch.float32)
    wk = 1.0 + 0.1 * torch.randn(D, generator=g, dtype=torch.float32)
    meta = {"seed": c["seed"]}
    mask = None
    if c["mask"] == "all_true":
        mask = torch.ones(1, 1, 1, S, dtype=torch.bool)
    elif c["mask"] == "text_pad":
        n_text = c["n_text"]
        valid = torch.randint(64, n_text + 1, (B,), generator=g)
        mask = torch.ones(B, 1, 1, S, dtype=torch.bool)
        for b in range(B):
            mask[b, 0, 0, int(valid[b]):n_text] = False
        meta["valid_text"] = [int(x) for x in valid]
    elif c["mask"] == "additive":
        meta["mask_per_head"] = True
        meta["mask_seed"] = c["seed"]
    return Inputs(name, q, k, v, do, wq, wk, ids, tuple(c["axes"]), float(c["theta"]), mask, c["causal"],
                  meta=meta)


def additive_mask_head(name: str, b: int, h: int) -> torch.Tensor:
    """[S, S] fp32 ~ U(-4, 0) for head (b, h) of an additive-mask workload,
    from its own generator seeded by (workload seed, b, h)."""
    c = WORKLOADS[name]
    S = c["S"]
    g = torch.Generator().manual_seed(1_000_003 * (c["seed"] + 1) + 1009 * b + h)
    return -4.0 * torch.rand(S, S, generator=g, dtype=torch.float32)

