"""Benchmark of the fused QK-RMSNorm + multi-axis RoPE + attention call.

One step = the whole hot path over one batch: st_rope_attn_fwd (rotary table,
mask tile classes, forward attention) followed by st_rope_attn_bwd (Delta,
backward attention with the dk epilogue, dq post-pass, norm-weight gradient
reduction; the tables and mask tile classes of the forward are reused from the
shared workspace, as the autograd Function does). Default workload: Flux1 1024px, B=1 H=24 S=4608 D=128 bf16, 3-axis
RoPE (16,56,56) theta 1e4, all-True bool mask [1,1,1,4608], forward+backward.

Metric: TFLOP/s with nominal FLOPs 4*B*H*S_q*S_kv*D forward (halved when
causal) and 2.5x that backward. L2 (129 MB) is flushed by writing a 256 MB
buffer before every timed step, outside the timed events.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the fp64 oracle on the host cores
  python bench.py --impl eager ...       # eager torch: rms_norm + rotation + SDPA

The eager arm is the comparison "Metal Flash Attention" (section "Fused RoPE +
SDPA") reports for its fused entry point: the same step with the norm and the
rotation as separate torch operations feeding torch's scaled_dot_product_attention
(whichever backend torch picks), forward and backward through autograd.

Under torchrun (N > 1) every rank runs its own replica of the workload (the
path shards over independent (b, h) heads; there is no exchange step), the
timed region is bracketed by barriers and the slowest rank's time is used.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as wl  # noqa: E402

METRIC = "fused norm+RoPE+attention fwd/bwd TFLOP/s and % of GB300 dense BF16 peak"
DENSE_BF16_PEAK_TFLOPS = 2250.0
FLUSH_BYTES = 256 << 20


def nominal_flops(inp):
    B, Sq, H, D = inp.q.shape
    Skv = inp.k.shape[1]
    f = 4.0 * B * H * Sq * Skv * D
    if inp.causal:
        f *= 0.5
    return f, 2.5 * f


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            d = json.load(fh)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def describe(name, inp):
    B, Sq, H, D = inp.q.shape
    m = "none" if inp.mask is None else f"{inp.mask.dtype} mask {list(inp.mask.shape)}"
    if inp.meta.get("mask_per_head"):
        m = f"fp32 additive mask [{B},{H},{Sq},{inp.k.shape[1]}]"
    return (f"{name} fwd+bwd: B={B} H={H} S_q={Sq} S_kv={inp.k.shape[1]} D={D} q/k {str(inp.q.dtype)[6:]} "
            f"v {str(inp.v.dtype)[6:]}, RoPE axes {list(inp.axes)} theta {inp.theta:g}, {m}, causal={inp.causal}")


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled while the timed region runs."""

    FIELDS = ["index", "clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", "--query-gpu=" + ",".join(self.FIELDS),
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for _, ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) != len(self.FIELDS):
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def reduce_max(value: float, world: int, device) -> float:
    """The maximum of `value` over all ranks (the slowest rank's time)."""
    if world <= 1:
        return float(value)
    t = torch.tensor([value], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_tflops(world: int, flops_per_step: float, steps: int, ms: float) -> float:
    """Whole-job throughput: every rank ran `steps` steps of `flops_per_step`
    (weak scaling), and the job took `ms` (the maximum over ranks)."""
    return world * flops_per_step * steps / (ms * 1e-3) / 1e12


def load_traffic(kernel: str):
    """Per-launch DRAM bytes of `kernel` from the committed ncu summary, if it
    was captured from the current kernel source (matching hash)."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    src = os.path.join(ROOT, "qk_norm_rope_gb300", "csrc", f"st_{kernel}.cu")
    try:
        h = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
        for ln in open(path):
            f = ln.split()
            if len(f) >= 4 and f[0] == kernel and f[1] == h:
                return float(f[2]), f[3]
    except OSError:
        pass
    return None, None


def device_mask(inp, name, dev):
    """The workload's mask on the device; a per-head additive mask is built one
    (b, h) slice at a time from the seeded generator the parity tests use."""
    if not inp.meta.get("mask_per_head"):
        return None if inp.mask is None else inp.mask.to(dev)
    B, Sq, H, _ = inp.q.shape
    mask = torch.empty(B, H, Sq, inp.k.shape[1], dtype=torch.float32, device=dev)
    for b in range(B):
        for h in range(H):
            mask[b, h].copy_(wl.additive_mask_head(name, b, h))
    return mask


def run_ours(args, rank, world, dev):
    from qk_norm_rope_gb300 import api

    inp = wl.make(args.workload)
    B, Sq, H, D = inp.q.shape
    f_fwd, f_bwd = nominal_flops(inp)
    step_flops = f_fwd + f_bwd
    g = lambda t: None if t is None else t.to(dev)
    q, k, v, do, wq, wk, ids = (g(t) for t in (inp.q, inp.k, inp.v, inp.do, inp.wq, inp.wk, inp.ids))
    mask = device_mask(inp, args.workload, dev)
    o = torch.empty(B, Sq, H, D, dtype=v.dtype, device=dev)
    lse = torch.empty(B, H, Sq, dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    dwq, dwk = torch.empty_like(wq), torch.empty_like(wk)
    # one backward-sized workspace serves both calls, as in the autograd
    # Function: the backward reuses the forward's rotary tables and mask tiles
    ws = torch.empty(api.st_rope_attn_workspace_size(q, k, v, ids, inp.axes, inp.theta, mask, inp.causal,
                                                     for_backward=True), dtype=torch.uint8, device=dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def fwd_call(q=q, k=k, v=v, wq=wq, wk=wk, ids=ids, mask=mask):
        api.st_rope_attn_fwd(q, k, v, wq, wk, inp.eps, ids, inp.axes, inp.theta, mask=mask, causal=inp.causal,
                             o=o, lse=lse, workspace=ws)

    def bwd_call(q=q, k=k, v=v, do=do, wq=wq, wk=wk, ids=ids, mask=mask):
        api.st_rope_attn_bwd(q, k, v, wq, wk, inp.eps, ids, inp.axes, inp.theta, o, lse, do, mask=mask,
                             causal=inp.causal, workspace=ws, dq=dq, dk=dk, dv=dv, dwq=dwq, dwk=dwk,
                             reuse_tables=True)

    def step(q=q, k=k, v=v, do=do, wq=wq, wk=wk, ids=ids, mask=mask):
        fwd_call(q, k, v, wq, wk, ids, mask)
        bwd_call(q, k, v, do, wq, wk, ids, mask)

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    def timed(n, fn):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        for a, b in evs:
            flush.zero_()
            a.record()
            fn()
            b.record()
        torch.cuda.synchronize()
        return sum(a.elapsed_time(b) for a, b in evs)

    for _ in range(args.warmup):
        step()
    api.st_check_status()

    # ---- timed region (device time, L2 flushed before every step)
    vis = [x for x in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if x.strip()]
    clocks = ClockSampler(vis[torch.cuda.current_device()] if vis else torch.cuda.current_device())
    clocks.start()
    time.sleep(0.2)
    barrier()
    launches0 = api.st_get_stats()["kernel_launches"]
    ms = timed(args.steps, step)
    launches = api.st_get_stats()["kernel_launches"] - launches0
    barrier()
    clk = clocks.stop()
    api.st_check_status()
    ms_max = reduce_max(ms, world, dev)
    ms_per_step = ms_max / args.steps
    value = job_tflops(world, step_flops, args.steps, ms_max)

    # ---- per-kernel device time (events on the launching stream, inside the library)
    api.st_timing_enable(True)
    api.st_timing_read()
    timed(args.steps, step)
    kt = api.st_timing_read()
    api.st_timing_enable(False)
    per_kernel = {n: {"launches": c, "avg_us": (m / c * 1e3 if c else None), "share": None} for n, (c, m) in kt.items()}
    tot = sum(m for _, m in kt.values()) or 1.0
    for n, (c, m) in kt.items():
        per_kernel[n]["share"] = round(m / tot, 4)
    dominant = max(kt, key=lambda n: kt[n][1])
    peaks = measured_peaks()
    kflops = {"fwd": f_fwd, "bwd": f_bwd}
    roof = None
    if dominant in kflops and kt[dominant][0]:
        avg_s = kt[dominant][1] / kt[dominant][0] * 1e-3
        achieved = kflops[dominant] / avg_s / 1e12
        traffic, _ = load_traffic(dominant)
        roof = {"kernel": f"st_{dominant}", "bound": "tensor", "achieved": round(achieved, 2),
                "peak": peaks["bf16_tflops"], "unit": "TFLOP/s", "frac": round(achieved / peaks["bf16_tflops"], 4),
                "peak_source": f"{peaks['source']} bf16 burst (cuBLAS 8192^3)", "traffic": traffic,
                "frac_of_dense_2250": round(achieved / DENSE_BF16_PEAK_TFLOPS, 4)}
    fwd_us = per_kernel["fwd"]["avg_us"]
    bwd_us = per_kernel["bwd"]["avg_us"]

    # ---- end to end through the public API with host buffers
    e2e = e2e_p = None
    if not args.no_e2e:
        pin = lambda t: None if t is None else t.cpu().pin_memory()
        hq, hk, hv, hdo, hwq, hwk, hids = (pin(t) for t in (q, k, v, do, wq, wk, ids))
        hmask = pin(mask) if (mask is not None and mask.numel() * mask.element_size() < (1 << 30)) else None
        dmask = mask if hmask is None else torch.empty_like(mask)
        dbuf = [torch.empty_like(t) for t in (q, k, v, do, wq, wk, ids)]
        outs = [o, lse, dq, dk, dv, dwq, dwk]
        houts = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outs]
        h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv, hdo, hwq, hwk, hids))
        if hmask is not None:
            h2d += hmask.numel() * hmask.element_size()
        d2h = sum(t.numel() * t.element_size() for t in outs)

        # The forward's inputs are copied first; dO (an input of the backward
        # only) follows on a copy stream while the forward runs, and O and LSE
        # go back to the host while the backward runs. Every copy of the step
        # completes before the step's end event (the compute stream joins the
        # copy stream).
        copy_stream = torch.cuda.Stream(device=dev)
        ev_in, ev_do, ev_fwd = torch.cuda.Event(), torch.cuda.Event(), torch.cuda.Event()
        bq, bk, bv, bdo, bwq, bwk, bids = dbuf

        def e2e_step():
            cur = torch.cuda.current_stream()
            copy_stream.wait_stream(cur)  # the previous step is done with the buffers
            for dst, src in ((bq, hq), (bk, hk), (bv, hv), (bwq, hwq), (bwk, hwk), (bids, hids)):
                dst.copy_(src, non_blocking=True)
            if hmask is not None:
                dmask.copy_(hmask, non_blocking=True)
            ev_in.record(cur)
            with torch.cuda.stream(copy_stream):
                copy_stream.wait_event(ev_in)  # behind the forward's inputs on the copy engine
                bdo.copy_(hdo, non_blocking=True)
                ev_do.record(copy_stream)
            fwd_call(bq, bk, bv, bwq, bwk, bids, dmask)
            ev_fwd.record(cur)
            with torch.cuda.stream(copy_stream):
                copy_stream.wait_event(ev_fwd)
                houts[0].copy_(o, non_blocking=True)
                houts[1].copy_(lse, non_blocking=True)
            cur.wait_event(ev_do)
            bwd_call(bq, bk, bv, bdo, bwq, bwk, bids, dmask)
            for dst, src in zip(houts[2:], outs[2:]):
                dst.copy_(src, non_blocking=True)
            cur.wait_stream(copy_stream)

        for _ in range(2):
            e2e_step()
        barrier()
        n_e2e = max(3, min(args.steps, 20))
        ms_e = timed(n_e2e, e2e_step)
        me = reduce_max(ms_e, world, dev)
        e2e = {"value": round(job_tflops(world, step_flops, n_e2e, me), 2), "unit": "TFLOP/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "steps": n_e2e,
               "ms_per_step": round(me / n_e2e, 4)}
        if hmask is None and mask is not None:
            e2e["note"] = "mask stays resident on the device (over 1 GB)"

        # Pipelined: the inputs of step i+1 go up on one copy stream while
        # step i computes, and the results of step i come down on another
        # while step i+1 computes (device inputs and outputs double-buffered;
        # the L2 flush stays on the compute stream before every step). The
        # timed region runs from before the first step's uploads to after the
        # last step's downloads, so every copy of every timed step is inside it.
        up, down = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
        dmask2 = dmask if hmask is None else torch.empty_like(dmask)  # a resident (or absent) mask is shared
        ins = [dbuf + [dmask], [torch.empty_like(t) for t in (q, k, v, do, wq, wk, ids)] + [dmask2]]
        outsets = [outs, [torch.empty_like(t) for t in outs]]
        ev_in = [torch.cuda.Event(), torch.cuda.Event()]
        ev_fwd = [torch.cuda.Event(), torch.cuda.Event()]
        ev_used = [torch.cuda.Event(), torch.cuda.Event()]
        ev_down = [torch.cuda.Event(), torch.cuda.Event()]
        hins = (hq, hk, hv, hdo, hwq, hwk, hids)
        pstate = {"i": 0}

        def pipelined_step():
            s = pstate["i"] % 2
            pstate["i"] += 1
            cur = torch.cuda.current_stream()
            pq, pk, pv, pdo, pwq, pwk, pids, pmask = ins[s]
            po, plse, pdq, pdk, pdv, pdwq, pdwk = outsets[s]
            with torch.cuda.stream(up):
                up.wait_event(ev_used[s])  # two steps back, the backward is done with these inputs
                for dst, src in zip((pq, pk, pv, pdo, pwq, pwk, pids), hins):
                    dst.copy_(src, non_blocking=True)
                if hmask is not None:
                    pmask.copy_(hmask, non_blocking=True)
                ev_in[s].record(up)
            flush.zero_()
            cur.wait_event(ev_in[s])
            cur.wait_event(ev_down[s])  # two steps back, these outputs have reached the host
            api.st_rope_attn_fwd(pq, pk, pv, pwq, pwk, inp.eps, pids, inp.axes, inp.theta, mask=pmask,
                                 causal=inp.causal, o=po, lse=plse, workspace=ws)
            ev_fwd[s].record(cur)
            api.st_rope_attn_bwd(pq, pk, pv, pwq, pwk, inp.eps, pids, inp.axes, inp.theta, po, plse, pdo, mask=pmask,
                                 causal=inp.causal, workspace=ws, dq=pdq, dk=pdk, dv=pdv, dwq=pdwq, dwk=pdwk,
                                 reuse_tables=True)
            ev_used[s].record(cur)
            with torch.cuda.stream(down):
                down.wait_event(ev_fwd[s])
                houts[0].copy_(po, non_blocking=True)
                houts[1].copy_(plse, non_blocking=True)
                down.wait_event(ev_used[s])
                for dst, src in zip(houts[2:], (pdq, pdk, pdv, pdwq, pdwk)):
                    dst.copy_(src, non_blocking=True)
                ev_down[s].record(down)

        def pipelined_run(n):
            cur = torch.cuda.current_stream()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(cur)
            up.wait_stream(cur)
            down.wait_stream(cur)
            for _ in range(n):
                pipelined_step()
            cur.wait_stream(up)
            cur.wait_stream(down)
            b.record(cur)
            torch.cuda.synchronize()
            return a.elapsed_time(b)

        pipelined_run(2)
        barrier()
        mp = reduce_max(pipelined_run(n_e2e), world, dev)
        e2e_p = {"value": round(job_tflops(world, step_flops, n_e2e, mp), 2), "unit": "TFLOP/s",
                 "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "steps": n_e2e,
                 "ms_per_step": round(mp / n_e2e, 4),
                 "note": "uploads of step i+1 and downloads of step i overlap the compute of steps i and i+1; "
                         "one L2 flush per step included"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(inp, args.workload, budget_s=args.cpu_seconds)

    sweep = None
    if world == 1 and not args.no_sweep and args.workload == "flux1_1024":
        del q, k, v, do, dq, dk, dv, ws, o, lse, mask
        torch.cuda.empty_cache()
        sweep = workload_sweep(dev, flush)

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1) inputs, norm weights 1+N(0,0.1))",
        "config": {"workload": describe(args.workload, inp), "global_batch": B * world, "seq_len": Sq,
                   "heads": H, "head_dim": D, "parallelism": "replicas" if world > 1 else "single",
                   "l2": "flushed (256 MB write) before every timed step",
                   "flops_per_step": step_flops, "fwd_flops": f_fwd, "bwd_flops": f_bwd},
        "pct_of_dense_bf16_peak": round(100 * value / world / DENSE_BF16_PEAK_TFLOPS, 2),
        "pct_of_measured_bf16": round(100 * value / world / peaks["bf16_tflops"], 2),
        "fwd_tflops": round(f_fwd / (fwd_us * 1e-6) / 1e12, 2) if fwd_us else None,
        "bwd_tflops": round(f_bwd / (bwd_us * 1e-6) / 1e12, 2) if bwd_us else None,
        "roofline": roof, "kernels": per_kernel, "gpu_launches": int(launches), "clocks": clk, "e2e": e2e, "e2e_pipelined": e2e_p,
        "cpu_baseline": cpu,
    }
    if sweep is not None:
        line["workloads"] = sweep
    return line


# The other configurations and the pages' probe shapes, measured briefly after
# the headline workload under the same rules (warm-up, L2 flush before every
# timed step, CUDA events); the Z-Image DiT shape also runs the eager torch
# composition the pages compare their fused entry point with.
SWEEP = ["tiny_flux", "flux1_padded", "causal_8k", "causal_8k_additive", "flux2_long", "flux1_probe_6144",
         "flux1_probe_24576", "zimage_dit"]


def workload_sweep(dev, flush, steps=3, warmup=2):
    from qk_norm_rope_gb300 import api
    out = {}
    for name in SWEEP:
        inp = wl.make(name)
        B, Sq, H, D = inp.q.shape
        Skv = inp.k.shape[1]
        f_fwd, f_bwd = nominal_flops(inp)
        g = lambda t: None if t is None else t.to(dev)
        q, k, v, do, wq, wk, ids = (g(t) for t in (inp.q, inp.k, inp.v, inp.do, inp.wq, inp.wk, inp.ids))
        mask = device_mask(inp, name, dev)
        ws = torch.empty(api.st_rope_attn_workspace_size(q, k, v, ids, inp.axes, inp.theta, mask, inp.causal,
                                                         for_backward=True), dtype=torch.uint8, device=dev)
        o = torch.empty(B, Sq, H, D, dtype=v.dtype, device=dev)
        lse = torch.empty(B, H, Sq, dtype=torch.float32, device=dev)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        dwq, dwk = torch.empty_like(wq), torch.empty_like(wk)

        def step():
            api.st_rope_attn_fwd(q, k, v, wq, wk, inp.eps, ids, inp.axes, inp.theta, mask=mask, causal=inp.causal,
                                 o=o, lse=lse, workspace=ws)
            api.st_rope_attn_bwd(q, k, v, wq, wk, inp.eps, ids, inp.axes, inp.theta, o, lse, do, mask=mask,
                                 causal=inp.causal, workspace=ws, dq=dq, dk=dk, dv=dv, dwq=dwq, dwk=dwk,
                                 reuse_tables=True)

        def timed(fn, n):
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
            for a, b in evs:
                flush.zero_()
                a.record()
                fn()
                b.record()
            torch.cuda.synchronize()
            return sum(a.elapsed_time(b) for a, b in evs) / n

        for _ in range(warmup):
            step()
        api.st_check_status()
        ms = timed(step, steps)
        api.st_timing_enable(True)
        api.st_timing_read()
        timed(step, steps)
        kt = api.st_timing_read()
        api.st_timing_enable(False)
        api.st_check_status()
        fwd_us = kt["fwd"][1] / max(kt["fwd"][0], 1) * 1e3
        bwd_us = kt["bwd"][1] / max(kt["bwd"][0], 1) * 1e3
        rec = {"shape": [B, Sq, H, D], "causal": inp.causal, "ms_per_step": round(ms, 4),
               "tflops": round((f_fwd + f_bwd) / (ms * 1e-3) / 1e12, 2),
               "fwd_kernel_us": round(fwd_us, 1), "bwd_kernel_us": round(bwd_us, 1),
               "fwd_tflops": round(f_fwd / (fwd_us * 1e-6) / 1e12, 2) if fwd_us else None,
               "bwd_tflops": round(f_bwd / (bwd_us * 1e-6) / 1e12, 2) if bwd_us else None,
               "pct_of_dense_bf16_peak": round(100 * (f_fwd + f_bwd) / (ms * 1e-3) / 1e12 / DENSE_BF16_PEAK_TFLOPS, 2),
               "q_dtype": str(inp.q.dtype)[6:], "mask": None if inp.mask is None and not inp.meta.get("mask_per_head")
               else list(mask.shape)}
        if name == "zimage_dit":
            cos, sin = rope_tables_torch(ids, inp.axes, inp.theta)
            leaves = [t.detach().requires_grad_() for t in (q, k, v, wq, wk)]

            def eager_step():
                oo = eager_attention(*leaves, inp.eps, cos, sin, mask=mask, causal=inp.causal)
                torch.autograd.grad(oo, leaves, do)

            def fused_fwd():
                api.st_rope_attn_fwd(q, k, v, wq, wk, inp.eps, ids, inp.axes, inp.theta, o=o, lse=lse, workspace=ws)

            def eager_fwd():
                with torch.no_grad():
                    eager_attention(q, k, v, wq, wk, inp.eps, cos, sin)

            for _ in range(warmup):
                eager_step()
                eager_fwd()
            rec["eager_ms_per_step"] = round(timed(eager_step, steps), 4)
            rec["fused_fwd_ms"] = round(timed(fused_fwd, steps), 4)
            rec["eager_fwd_ms"] = round(timed(eager_fwd, steps), 4)
            rec["eager"] = "torch rms_norm + table rotation (fp32) + scaled_dot_product_attention, autograd"
        out[name] = rec
        del q, k, v, do, mask, ws, o, lse, dq, dk, dv
        torch.cuda.empty_cache()
    return out


def rope_tables_torch(ids, axes, theta):
    """Pair-duplicated (cos, sin) [Bt, S, D] fp32 of the ids' angles, built with
    torch operations as a model's rotary module would (the eager arm's own
    tables; angle of pair j of axis a: id_a * theta^(-2j/d_a))."""
    parts = []
    for a, d_a in enumerate(axes):
        j = torch.arange(d_a // 2, dtype=torch.float64, device=ids.device)
        parts.append(ids[..., a:a + 1].double() * theta ** (-2.0 * j / d_a))
    phi = torch.cat(parts, -1)
    return (torch.cos(phi).float().repeat_interleave(2, -1), torch.sin(phi).float().repeat_interleave(2, -1))


def eager_attention(q, k, v, wq, wk, eps, cos, sin, mask=None, causal=False):
    """The eager composition on [B, S, H, D] tensors: rms_norm in fp32, the
    rotation x * cos + rot(x) * sin (rot(x) = (-x1, x0) per interleaved pair),
    a cast to v's dtype, then torch SDPA. cos, sin: [Bt, S, D] fp32."""
    import torch.nn.functional as F
    D = q.shape[-1]

    def tr(x, w):
        n = F.rms_norm(x.float(), (D,), w, eps)
        p = n.unflatten(-1, (D // 2, 2))
        r = torch.stack((-p[..., 1], p[..., 0]), -1).flatten(-2)
        return (n * cos[:, :, None, :] + r * sin[:, :, None, :]).to(v.dtype).transpose(1, 2)

    o = F.scaled_dot_product_attention(tr(q, wq), tr(k, wk), v.transpose(1, 2), attn_mask=mask, is_causal=causal)
    return o.transpose(1, 2)


def run_eager(args, rank, world, dev):
    """The eager arm: the same step and timing rules as run_ours."""
    inp = wl.make(args.workload)
    B, Sq, H, D = inp.q.shape
    f_fwd, f_bwd = nominal_flops(inp)
    g = lambda t: None if t is None else t.to(dev)
    q, k, v, do, wq, wk, ids = (g(t) for t in (inp.q, inp.k, inp.v, inp.do, inp.wq, inp.wk, inp.ids))
    mask = device_mask(inp, args.workload, dev)
    cos, sin = rope_tables_torch(ids, inp.axes, inp.theta)   # built once, as a model caches them
    leaves = [t.detach().requires_grad_() for t in (q, k, v, wq, wk)]
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def step():
        o = eager_attention(*leaves, inp.eps, cos, sin, mask=mask, causal=inp.causal)
        torch.autograd.grad(o, leaves, do)

    def timed(n):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        for a, b in evs:
            flush.zero_()
            a.record()
            step()
            b.record()
        torch.cuda.synchronize()
        return sum(a.elapsed_time(b) for a, b in evs)

    for _ in range(args.warmup):
        step()
    vis = [x for x in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if x.strip()]
    clocks = ClockSampler(vis[torch.cuda.current_device()] if vis else torch.cuda.current_device())
    clocks.start()
    time.sleep(0.2)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    ms = timed(args.steps)
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop()
    ms_max = reduce_max(ms, world, dev)
    value = job_tflops(world, f_fwd + f_bwd, args.steps, ms_max)
    return {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_max / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) inputs, norm weights 1+N(0,0.1))",
        "config": {"workload": describe(args.workload, inp), "global_batch": B * world, "seq_len": Sq, "heads": H,
                   "head_dim": D, "parallelism": "replicas" if world > 1 else "single",
                   "l2": "flushed (256 MB write) before every timed step"},
        "impl": "eager", "eager": "torch rms_norm + table rotation (fp32) + scaled_dot_product_attention, autograd",
        "clocks": clk,
    }


def oracle_step_flops(Sq_rows, Skv, D, causal=False):
    f = 4.0 * Sq_rows * Skv * D
    if causal:
        f *= 0.5
    return 3.5 * f


def oracle_sample(inp, b, h, r0, rows, mask_head=None):
    """The oracle's fwd+bwd on head (b, h), query rows [r0, r0+rows), all keys."""
    import oracle
    f64 = lambda t: t.double().numpy()
    sl_q = lambda t: f64(t[b:b + 1, r0:r0 + rows, h:h + 1])
    sl_k = lambda t: f64(t[b:b + 1, :, h:h + 1])
    ids = inp.ids[min(b, inp.ids.shape[0] - 1):][:1]
    m = None
    if mask_head is not None:
        m = mask_head[r0:r0 + rows].double().numpy()[None, None]
    elif inp.mask is not None:
        mm = inp.mask[min(b, inp.mask.shape[0] - 1):][:1][:, min(h, inp.mask.shape[1] - 1):][:, :1]
        if mm.shape[2] > 1:
            mm = mm[:, :, r0:r0 + rows]
        m = mm.numpy() if mm.dtype == torch.bool else mm.double().numpy()
    args = (sl_q(inp.q), sl_k(inp.k), sl_k(inp.v), f64(inp.wq), f64(inp.wk), inp.eps,
            ids[:, r0:r0 + rows].numpy(), inp.axes, inp.theta)
    kw = dict(mask=m, causal=False, ids_k=ids.numpy())
    oracle.fwd(*args, **kw)
    oracle.bwd(*args, sl_q(inp.do), **kw)


def cpu_baseline(inp, name, budget_s=15.0):
    """The fp64 oracle, as it stands, on the host cores: whole heads of the
    workload (all query rows, all keys), forward + backward, until the time
    budget is used (at least one head)."""
    import oracle
    oracle.build()
    B, Sq, H, D = inp.q.shape
    Skv = inp.k.shape[1]
    if inp.causal:
        return {"value": None, "unit": "TFLOP/s", "cores": oracle.num_threads(), "kind": "oracle",
                "sample": "skipped: causal sample needs whole heads; see --impl reference"}
    t0 = time.time()
    heads = 0
    while True:
        b, h = divmod(heads, H)
        mh = wl.additive_mask_head(name, b, h) if inp.meta.get("mask_per_head") else None
        oracle_sample(inp, b % B, h, 0, Sq, mh)
        heads += 1
        if time.time() - t0 >= budget_s or heads >= B * H:
            break
    dt = time.time() - t0
    fl = heads * oracle_step_flops(Sq, Skv, D)
    return {"value": round(fl / dt / 1e12, 6), "unit": "TFLOP/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{heads} whole head(s) of {name} (fwd+bwd, S_q={Sq}, S_kv={Skv}) in {dt:.1f} s",
            "seconds": round(dt, 2)}


def run_reference(args):
    """The oracle (plain fp64 C + OpenMP) timed on the host cores on this
    workload: every step is a bounded sample of it, the fwd+bwd of one head
    restricted to a block of query rows against all keys, sized so that the
    whole run stays within a few minutes."""
    import oracle
    oracle.build()
    inp = wl.make(args.workload)
    B, Sq, H, D = inp.q.shape
    Skv = inp.k.shape[1]
    causal = inp.causal
    target = max(0.3, min(3.0, 150.0 / (args.steps + args.warmup)))
    # calibrate the query-row block on one small sample
    rows = min(Sq, 128)
    t0 = time.time()
    oracle_sample(inp, 0, 0, 0, rows)
    per_row = (time.time() - t0) / rows
    if not causal:
        rows = int(max(64, min(Sq, target / max(per_row, 1e-9))) // 64 * 64) or min(Sq, 64)
    else:
        rows = Sq
    mask_cache = {}

    def one(i):
        b, h = divmod(i % (B * H), H)
        r0 = 0 if causal else ((i * rows) % max(1, Sq - rows + 1))
        mh = None
        if inp.meta.get("mask_per_head"):
            if (b, h) not in mask_cache:
                mask_cache.clear()
                mask_cache[(b, h)] = wl.additive_mask_head(args.workload, b, h)
            mh = mask_cache[(b, h)]
        if causal:
            import oracle as orc
            f64 = lambda t: t.double().numpy()
            sl = lambda t: f64(t[b:b + 1, :, h:h + 1])
            a = (sl(inp.q), sl(inp.k), sl(inp.v), f64(inp.wq), f64(inp.wk), inp.eps, inp.ids.numpy(), inp.axes,
                 inp.theta)
            orc.fwd(*a, causal=True)
            orc.bwd(*a, sl(inp.do), causal=True)
        else:
            oracle_sample(inp, b, h, r0, rows, mh)

    for i in range(args.warmup):
        one(i)
    t0 = time.time()
    for i in range(args.steps):
        one(args.warmup + i)
    dt = time.time() - t0
    fl = oracle_step_flops(rows, Skv, D, causal) * args.steps
    value = fl / dt / 1e12
    sample = (f"each step: oracle fwd+bwd of one (b,h) head of {args.workload}, "
              + ("all rows (causal)" if causal else f"{rows} query rows x {Skv} keys"))
    return {
        "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": describe(args.workload, inp), "global_batch": B, "seq_len": Sq, "heads": H,
                   "head_dim": D, "parallelism": "host cores (OpenMP)"},
        "impl": "reference",
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": oracle.num_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference", "eager"], default="ours")
    ap.add_argument("--workload", default="flux1_1024", choices=sorted(wl.WORKLOADS))
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-sweep", action="store_true",
                    help="skip the other workloads measured after the headline one")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (there is no CPU path)")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=dev)
    line = run_eager(args, rank, world, dev) if args.impl == "eager" else run_ours(args, rank, world, dev)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
