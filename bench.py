"""VSA layer benchmark on GB300: one JSON line on rank 0.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

A step is one forward + backward pass of the whole VSA hot path (stage, pool,
coarse attention + selection, block-sparse fine attention + gated combine,
and all gradients) over the 720p-shaped layer: latent 20x44x80 (70,400
tokens, 1,100 cubes), batch 1, 40 heads, head_dim 128, top-32 cubes.  Inputs
are seeded synthetic video-shaped tensors (trainable_block_sparse_gb300.synth)
and are resident in HBM when the timed region starts; each bf16 tensor is
721 MB, larger than the 129 MB L2, so no flush is needed between steps.

value: executed TFLOPS of the step (fine stage over selected 64x64 tiles only,
plus the dense coarse stage), whole job.  e2e: the same metric through the
C ABI with host buffers (host->device inputs and device->host outputs inside
the timed region).  roofline: the step's dominant kernel against the measured
dense tensor peak.  cpu_baseline: the fp64 oracle on the host cores, timed on
a bounded sample of the same layer (executed FLOPs of the sample / its
measured time).

Under torchrun each rank runs its own replica of the layer ("replicas only":
the method has no exchange step between (batch, head) slices).
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from trainable_block_sparse_gb300 import build, flops, synth  # noqa: E402

METRIC = "VSA fwd/fwd+bwd ms/layer & executed TFLOPS (% of BF16 peak), 16K–70K tokens"
WORKLOAD = "p720"
# kernels per call of vsa_forward / vsa_backward
LAUNCHES_FWD = 10  # stage x3, tf32 splits x2, coarse logits GEMM + select + O_c GEMM, pair
                   # lists, fine forward
LAUNCHES_BWD = 17  # gradient-scale max, combine bwd, coarse bwd (tf32 splits x2, row dot,
                   # dual GEMM, 3 GEMMs), pair lists, transposed lists (mask, count, scan,
                   # fill, pairs), fine bwd x2
SIDE_WORKLOADS = ("wan13b", "pretrain", "dynamic")  # timed per stage beside the headline layer
SIDE_REPS = 20
# Gradients leave the layer in the inputs' dtype, bf16 (what autograd hands back
# for bf16 tensors): the kernels accumulate in fp32 and round once at the store.
# The fp32-gradient step is timed beside it (fwdbwd_ms_fp32_grads).
GRAD_DTYPE = "bf16"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            threading.Thread(target=self._read, daemon=True).start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        rows = []
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) != 7:
                continue
            try:
                rows.append((float(parts[0]), float(parts[1]), parts[3:]))
            except ValueError:
                continue
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for _, _, flags in rows for n, v in zip(names, flags)
                          if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows),
                "sm_max_mhz": max(r[1] for r in rows), "reasons": reasons,
                "samples": len(rows)}


def executed_flops(wl, pairs: int) -> dict:
    """Executed FLOPs of one layer: selected tiles only, plus the dense coarse stage."""
    coarse_f = flops.coarse_fwd(wl)
    return {"fine_fwd": flops.fine_fwd_pairs(pairs, wl.head_dim),
            "fine_bwd": flops.fine_bwd_pairs(pairs, wl.head_dim),
            "coarse_fwd": coarse_f,
            "coarse_bwd": 2.5 * coarse_f}  # logits, dA, dQc, dKc, dVc: 5 products of 2*Nc^2*D


def timed(fn, steps, warmup, stream):
    """Device time (ms) per call of fn over `steps` calls after `warmup` untimed calls."""
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for _ in range(steps):
        fn()
    end.record(stream)
    torch.cuda.synchronize()
    return start.elapsed_time(end) / steps


class L2Flush:
    """Writes a buffer of twice the L2 before each timed call (outside the
    timed events), so every call starts with a cold L2."""

    def __init__(self, dev, l2_bytes=129 * 2 ** 20):
        self.buf = torch.empty(2 * l2_bytes // 4, dtype=torch.float32, device=dev)

    def __call__(self):
        self.buf.zero_()


def timed_median(fn, reps, warmup, stream, flush=None):
    """Median device time (ms) of single calls, each bracketed by its own CUDA
    events on `stream`; with `flush`, the L2 is flushed before every call."""
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(reps)]
    for a, b in ev:
        if flush is not None:
            flush()
        a.record(stream)
        fn()
        b.record(stream)
    torch.cuda.synchronize()
    return statistics.median(a.elapsed_time(b) for a, b in ev)


def workload(args):
    wl = synth.WORKLOADS[getattr(args, "workload", None) or WORKLOAD]
    return wl.replace(heads=args.heads) if getattr(args, "heads", 0) else wl


def max_over_ranks(ms: float, world: int, dev) -> float:
    """The slowest rank's time: every rank processes its own replica of the
    layer (no data exchange), so the job's time is the maximum."""
    if world <= 1:
        return ms
    t = torch.tensor([ms], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_throughput(step_flops: float, world: int, ms_max: float) -> float:
    """Whole-job TFLOPS: the work of all replicas over the slowest rank's time."""
    return world * step_flops / (ms_max * 1e-3) / 1e12


def gpu_arm(args, rank, world):
    from trainable_block_sparse_gb300 import vsa
    build.build()
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    wl = workload(args)
    inp = synth.Inputs(wl, with_grad=True)
    cfg = vsa.config_for(wl, grad_dtype=GRAD_DTYPE)
    t = {n: getattr(inp, n).to(dev) for n in ("q", "k", "v", "gc", "gf", "do")}
    bufs = vsa.Buffers(cfg, dev, with_backward=True)
    B, H, N, D = wl.batch, wl.heads, wl.tokens, wl.head_dim
    o = torch.empty_like(t["q"])
    grads = tuple(torch.empty(B, H, N, D, dtype=vsa.grad_torch_dtype(cfg), device=dev)
                  for _ in range(5))
    stream = torch.cuda.current_stream()

    def fwd():
        vsa.forward(cfg, t["q"], t["k"], t["v"], t["gc"], t["gf"], bufs, True, out=o)

    def step():
        fwd()
        vsa.backward(cfg, t["gc"], t["gf"], t["do"], bufs, grads)

    cfg32 = vsa.config_for(wl, grad_dtype="fp32")
    grads32 = tuple(torch.empty(B, H, N, D, dtype=torch.float32, device=dev) for _ in range(5))

    def step_fp32_grads():
        fwd()
        vsa.backward(cfg32, t["gc"], t["gf"], t["do"], bufs, grads32)

    bufs_inf = vsa.Buffers(cfg, dev, with_backward=False, inference_only=True)
    o_inf = torch.empty_like(t["q"])

    def fwd_inference():
        vsa.forward(cfg, t["q"], t["k"], t["v"], t["gc"], t["gf"], bufs_inf, False, out=o_inf)

    fwd()
    torch.cuda.synchronize()
    pairs = int(bufs.view("cnt", torch.int32, (B, H, wl.cubes)).sum().item())
    balance = balance_report(vsa, bufs, wl, dev)
    work = executed_flops(wl, pairs)
    step_flops = sum(work.values())

    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    # clocks sampled through every timed section (the step timing alone is
    # shorter than the sampling interval)
    with ClockSampler(dev.index) as clk:
        ms_step = timed(step, args.steps, args.warmup, stream)
        ms_fwd = timed(fwd, max(3, args.steps // 2), 1, stream)
        ms_fwd_inf = timed(fwd_inference, max(3, args.steps // 2), 1, stream)
        ms_step32 = timed(step_fp32_grads, max(3, args.steps // 2), 1, stream)
        status = bufs.device_status() or bufs_inf.device_status()
        if status != vsa.OK:
            raise RuntimeError(f"device status {status} after the timed steps")
        flush = L2Flush(dev)
        stages = stage_breakdown(vsa, cfg, wl, t, bufs, stream, dev, flush=flush)
        stages_warm = stage_breakdown(vsa, cfg, wl, t, bufs, stream, dev)
        fp8 = fp8_forward(vsa, cfg, wl, t, dev, pairs, flush)
    ms_max = max_over_ranks(ms_step, world, dev)
    e2e = end_to_end(vsa, cfg, wl, inp, bufs, stream, dev, step_flops, args)
    e2e["fp32_gradients"] = end_to_end(vsa, cfg32, wl, inp, None, stream, dev, step_flops, args,
                                       link=False)
    side = {}
    if rank == 0 and not args.no_side:
        del bufs, grads, grads32, o, t
        torch.cuda.empty_cache()
        side = {name: side_workload(vsa, name, dev) for name in SIDE_WORKLOADS}
    return {"wl": wl, "work": work, "pairs": pairs, "ms_step": ms_max, "ms_fwd": ms_fwd,
            "ms_fwd_inf": ms_fwd_inf, "ms_step_fp32_grads": ms_step32,
            "clocks": clk.summary(), "stages": stages, "stages_warm": stages_warm,
            "e2e": e2e, "inp": inp,
            "balance": balance, "side": side, "fp8": fp8}


# nominal dense rates (PFLOP/s): e4m3 against bf16
FP8_OVER_BF16 = 4.5 / 2.25


def fp8_forward(vsa, cfg, wl, t, dev, pairs, flush):
    """The e4m3 variant (head_dim 128, inference): the whole forward through
    vsa_forward_fp8 and its fine stage alone through vsa_fine_fwd_fp8, median
    of SIDE_REPS calls with the L2 flushed before each."""
    import ctypes
    if wl.head_dim != 128:
        return None
    L, P = vsa.lib(), vsa._ptr
    B, H, N, D, nc, cap = wl.batch, wl.heads, wl.tokens, wl.head_dim, wl.cubes, wl.list_capacity
    stream = torch.cuda.current_stream()
    bufs = vsa.Buffers(cfg, dev, with_backward=False)
    o = torch.empty_like(t["q"])

    def fwd():
        vsa.forward_fp8(cfg, t["q"], t["k"], t["v"], t["gc"], t["gf"], bufs, out=o)

    ms_fwd = timed_median(fwd, SIDE_REPS, 3, stream, flush)
    q8 = bufs.view("q16", torch.uint8, (B, H, N, D))
    k8 = bufs.view("k16", torch.uint8, (B, H, N, D))
    v8t = bufs.view("v16", torch.uint8, (B, H, nc, D, 64))
    scales = bufs.view("o_f", torch.float32, (B, H, 3))
    idx = bufs.view("idx", torch.int32, (B, H, nc, cap))
    cnt = bufs.view("cnt", torch.int32, (B, H, nc))
    oc = bufs.view("oc", torch.float32, (B, H, nc, D))
    lse = bufs.view("lse_f", torch.float32, (B, H, N))
    c, s = ctypes.byref(cfg), vsa._stream()

    def fine():
        st = L.vsa_fine_fwd_fp8(c, P(q8), P(k8), P(v8t), P(scales), P(idx), P(cnt), P(t["gc"]),
                                P(t["gf"]), P(oc), P(o), P(lse), P(bufs.ws), s)
        if st != vsa.OK:
            raise RuntimeError(f"vsa_fine_fwd_fp8 returned {st}")

    def stage():
        st = L.vsa_stage_fp8(c, P(t["q"]), P(t["k"]), P(t["v"]), P(q8), P(k8), P(v8t),
                             P(scales), P(bufs.view("qc", torch.float32, (B, H, nc, D))),
                             P(bufs.view("kc", torch.float32, (B, H, nc, D))),
                             P(bufs.view("vc", torch.float32, (B, H, nc, D))), P(bufs.ws), s)
        if st != vsa.OK:
            raise RuntimeError(f"vsa_stage_fp8 returned {st}")

    ms_fine = timed_median(fine, SIDE_REPS, 2, stream, flush)
    ms_stage = timed_median(stage, SIDE_REPS, 2, stream, flush)
    if bufs.device_status() != vsa.OK:
        raise RuntimeError(f"e4m3 forward: device status {bufs.device_status()}")
    peaks, _ = load_peaks()
    fine_tflops = flops.fine_fwd_pairs(pairs, D) / (ms_fine * 1e-3) / 1e12
    return {"fwd_ms_per_layer": ms_fwd, "fine_fwd_ms": ms_fine, "stage_fp8_ms": ms_stage,
            "fine_fwd_tflops": fine_tflops,
            "fine_fwd_frac_of_fp8_peak": fine_tflops / (peaks["bf16_tflops"] * FP8_OVER_BF16),
            "fine_fwd_frac_of_bf16_peak": fine_tflops / peaks["bf16_tflops"],
            "peak_note": "e4m3 peak = measured bf16 peak x the nominal e4m3/bf16 ratio (2)",
            "what": "vsa_forward_fp8: e4m3 staging + fp32 coarse stage + e4m3 fine stage "
                    "(Q, K, V, P in e4m3, fp32 accumulation), inference; median of "
                    f"{SIDE_REPS} calls, L2 flushed before each"}


def balance_report(vsa, bufs, wl, dev):
    """Per-CTA work of the persistent fine kernels under their static item
    assignment (max/mean of the step counts) and the list-length histogram."""
    from trainable_block_sparse_gb300 import schedule
    B, H, nc, cap = wl.batch, wl.heads, wl.cubes, wl.list_capacity
    idx = bufs.view("idx", torch.int32, (B * H, nc, cap)).cpu().numpy()
    cnt = bufs.view("cnt", torch.int32, (B * H, nc)).cpu().numpy()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    ordered = schedule.uses_cost_order(B * H, wl.tokens, wl.head_dim)
    return schedule.load_balance(idx, cnt, sms, ordered=ordered, head_dim=wl.head_dim)


def side_workload(vsa, name, dev):
    """Per-stage times of another configuration of the same layer (inputs
    resident, 3 repetitions per stage), its fwd and fwd+bwd time per layer,
    and the fine kernels' work distribution."""
    wl = synth.WORKLOADS[name]
    inp = synth.Inputs(wl, with_grad=True)
    cfg = vsa.config_for(wl, grad_dtype=GRAD_DTYPE)
    t = {n: getattr(inp, n).to(dev) for n in ("q", "k", "v", "gc", "gf", "do")}
    bufs = vsa.Buffers(cfg, dev, with_backward=True)
    B, H, N, D = wl.batch, wl.heads, wl.tokens, wl.head_dim
    o = torch.empty_like(t["q"])
    grads = tuple(torch.empty(B, H, N, D, dtype=vsa.grad_torch_dtype(cfg), device=dev)
                  for _ in range(5))
    stream = torch.cuda.current_stream()

    def fwd():
        vsa.forward(cfg, t["q"], t["k"], t["v"], t["gc"], t["gf"], bufs, True, out=o)

    def step():
        fwd()
        vsa.backward(cfg, t["gc"], t["gf"], t["do"], bufs, grads)

    flush = L2Flush(dev)
    bufs_inf = vsa.Buffers(cfg, dev, with_backward=False, inference_only=True)

    def fwd_inference():
        vsa.forward(cfg, t["q"], t["k"], t["v"], t["gc"], t["gf"], bufs_inf, False, out=o)

    ms_fwd = timed_median(fwd, SIDE_REPS, 3, stream, flush)
    ms_fwd_inf = timed_median(fwd_inference, SIDE_REPS, 3, stream, flush)
    ms_step = timed_median(step, SIDE_REPS, 3, stream, flush)
    warm_fwd = timed_median(fwd, SIDE_REPS, 1, stream)
    warm_step = timed_median(step, SIDE_REPS, 1, stream)
    if bufs.device_status() != vsa.OK:
        raise RuntimeError(f"{name}: device status {bufs.device_status()}")
    pairs = int(bufs.view("cnt", torch.int32, (B, H, wl.cubes)).sum().item())
    work = executed_flops(wl, pairs)
    balance = balance_report(vsa, bufs, wl, dev)
    stages = stage_breakdown(vsa, cfg, wl, t, bufs, stream, dev, flush=flush)
    stages_warm = stage_breakdown(vsa, cfg, wl, t, bufs, stream, dev)
    fp8 = fp8_forward(vsa, cfg, wl, t, dev, pairs, flush)
    peaks, _ = load_peaks()
    return {"workload": wl.name, "selected_pairs": pairs, "fwd_ms_per_layer": ms_fwd,
            "fwd_inference_ms_per_layer": ms_fwd_inf,
            "fwdbwd_ms_per_layer": ms_step, "stages_ms": stages,
            "timing": f"median of {SIDE_REPS} single calls, L2 flushed before each "
                      f"(a {2 * 129} MB write); *_warm: the same without the flush",
            "fwd_ms_per_layer_warm": warm_fwd, "fwdbwd_ms_per_layer_warm": warm_step,
            "stages_ms_warm": stages_warm,
            "fine_fwd_frac_of_peak_warm": work["fine_fwd"] / (stages_warm["fine_fwd"] * 1e-3)
            / 1e12 / peaks["bf16_tflops"],
            "fine_fwd_tflops": work["fine_fwd"] / (stages["fine_fwd"] * 1e-3) / 1e12,
            "fine_fwd_frac_of_peak": work["fine_fwd"] / (stages["fine_fwd"] * 1e-3) / 1e12
            / peaks["bf16_tflops"],
            "fine_bwd_tflops": work["fine_bwd"] / (stages["fine_bwd"] * 1e-3) / 1e12,
            "load_balance": balance, **({"fp8_forward": fp8} if fp8 else {})}


def stage_breakdown(vsa, cfg, wl, t, bufs, stream, dev, reps=SIDE_REPS, flush=None):
    """Each stage alone through its own C-ABI entry point: median ms per call
    (L2 flushed before each call when `flush` is given)."""
    import ctypes
    L, P = vsa.lib(), vsa._ptr
    B, H, N, D, nc, cap = wl.batch, wl.heads, wl.tokens, wl.head_dim, wl.cubes, wl.list_capacity
    v = {n: bufs.view(n, torch.float16, (B, H, N, D)) for n in ("q16", "k16", "v16")}
    for n in ("qc", "kc", "vc", "oc"):
        v[n] = bufs.view(n, torch.float32, (B, H, nc, D))
    v["lse_c"] = bufs.view("lse_c", torch.float32, (B, H, nc))
    v["idx"] = bufs.view("idx", torch.int32, (B, H, nc, cap))
    v["cnt"] = bufs.view("cnt", torch.int32, (B, H, nc))
    v["o_f"] = bufs.view("o_f", torch.float16, (B, H, N, D))
    v["lse_f"] = bufs.view("lse_f", torch.float32, (B, H, N))
    f32 = dict(dtype=torch.float32, device=dev)
    o = torch.empty_like(t["q"])
    dgc, dgf, dq, dk, dv = (torch.empty(B, H, N, D, dtype=vsa.grad_torch_dtype(cfg), device=dev)
                            for _ in range(5))
    dof = torch.empty(B, H, N, D, dtype=torch.float16, device=dev)
    doc, dqc, dkc, dvc = (torch.empty(B, H, nc, D, **f32) for _ in range(4))
    delta = torch.empty(B, H, N, **f32)
    gscale = torch.empty(B, H, **f32)
    ws, c, s = bufs.ws, ctypes.byref(cfg), vsa._stream()

    def ck(st, name):
        if st != vsa.OK:
            raise RuntimeError(f"{name} returned {st}")

    calls = {
        "stage_pool": lambda: [ck(L.vsa_stage(c, P(t[n]), P(v[n + "16"]), P(v[n + "c"]), P(ws), s),
                                  "vsa_stage") for n in ("q", "k", "v")],
        # from the cube means the forward already holds (the pooling is stage_pool's)
        "coarse_select": lambda: ck(L.vsa_coarse_select(
            c, None, None, None, P(v["qc"]), P(v["kc"]), P(v["vc"]), P(v["oc"]),
            P(v["lse_c"]), P(v["idx"]), P(v["cnt"]), P(ws), s), "vsa_coarse_select"),
        "fine_fwd": lambda: ck(L.vsa_fine_fwd(
            c, P(v["q16"]), P(v["k16"]), P(v["v16"]), P(v["idx"]), P(v["cnt"]), P(t["gc"]),
            P(t["gf"]), P(v["oc"]), P(o), P(v["o_f"]), P(v["lse_f"]), P(ws), s), "vsa_fine_fwd"),
        "fine_fwd_bf16": lambda: ck(L.vsa_fine_fwd_bf16(
            c, P(t["q"]), P(t["k"]), P(t["v"]), P(v["idx"]), P(v["cnt"]), P(t["gc"]),
            P(t["gf"]), P(v["oc"]), P(o), P(v["lse_f"]), P(ws), s), "vsa_fine_fwd_bf16"),
        "combine_bwd": lambda: ck(L.vsa_combine_bwd(
            c, P(t["do"]), P(t["gc"]), P(t["gf"]), P(v["o_f"]), P(v["oc"]), P(dgc), P(dgf),
            P(dof), P(doc), P(delta), P(gscale), P(ws), s), "vsa_combine_bwd"),
        "coarse_bwd": lambda: ck(L.vsa_coarse_bwd(
            c, P(v["qc"]), P(v["kc"]), P(v["vc"]), P(v["oc"]), P(v["lse_c"]), P(doc), P(dqc),
            P(dkc), P(dvc), P(ws), s), "vsa_coarse_bwd"),
        "fine_bwd": lambda: ck(L.vsa_fine_bwd(
            c, P(v["q16"]), P(v["k16"]), P(v["v16"]), P(v["idx"]), P(v["cnt"]), P(v["lse_f"]),
            P(dof), P(delta), P(gscale), P(dqc), P(dkc), P(dvc), P(dq), P(dk), P(dv), P(ws), s),
            "vsa_fine_bwd"),
    }
    return {name: timed_median(fn, reps, 2, stream, flush) for name, fn in calls.items()}


def end_to_end(vsa, cfg, wl, inp, bufs, stream, dev, step_flops, args, link=True):
    """Host inputs in, host outputs out, every step, through the library's
    host-buffer pipeline (HostPipeline: units of 5 heads, copies in and out
    overlapped with the kernels of the neighbouring units)."""
    from trainable_block_sparse_gb300.host_pipeline import HostPipeline, IN_NAMES, OUT_NAMES
    del bufs  # the pipeline owns per-unit buffers
    host_in = {n: getattr(inp, n).pin_memory() for n in IN_NAMES}
    B, H, N, D = wl.batch, wl.heads, wl.tokens, wl.head_dim
    host_out = {n: torch.empty(B, H, N, D, pin_memory=True,
                               dtype=torch.bfloat16 if n == "o" else vsa.grad_torch_dtype(cfg))
                for n in OUT_NAMES}
    pipe = HostPipeline(cfg, dev, heads_per_unit=5)
    reps = max(2, args.steps // 3)
    for _ in range(2):  # warm-up: allocates the per-unit buffers
        pipe.step(host_in, host_out)
    if pipe.check_status() != vsa.OK:
        raise RuntimeError("device status after the host-pipeline warm-up")
    t0 = time.perf_counter()
    for _ in range(reps):
        pipe.step(host_in, host_out)
    torch.cuda.synchronize(dev)
    ms = (time.perf_counter() - t0) * 1e3 / reps
    if pipe.check_status() != vsa.OK:
        raise RuntimeError("device status after the host-pipeline steps")
    h2d = sum(x.numel() * x.element_size() for x in host_in.values())
    d2h = sum(x.numel() * x.element_size() for x in host_out.values())
    out = {"ms": ms, "value": step_flops / (ms * 1e-3) / 1e12, "h2d": h2d, "d2h": d2h,
           "units": sum(1 for _ in pipe.units())}
    del pipe, host_in, host_out
    if link:
        out["link"] = host_link(dev)
    return out


def host_link(dev, nbytes=1 << 30, reps=3):
    """Pinned host <-> device copy rates of this machine (GB/s): each direction
    alone, and both at once on two streams (the bound under the end-to-end
    number)."""
    h = torch.empty(2, nbytes, dtype=torch.uint8, pin_memory=True)
    d = torch.empty(2, nbytes, dtype=torch.uint8, device=dev)
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def rate(fn, moved):
        fn()
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        for _ in range(reps):
            fn()
        torch.cuda.synchronize(dev)
        return moved * reps / (time.perf_counter() - t0) / 1e9

    def h2d():
        with torch.cuda.stream(s_in):
            d[0].copy_(h[0], non_blocking=True)

    def d2h():
        with torch.cuda.stream(s_out):
            h[1].copy_(d[1], non_blocking=True)

    def both():
        h2d()
        d2h()

    out = {"h2d_gbs": rate(h2d, nbytes), "d2h_gbs": rate(d2h, nbytes),
           "both_gbs": rate(both, 2 * nbytes), "copy_bytes": nbytes}
    del h, d
    return out


def oracle_sample(inp, b, h, cubes, budget_s=None):
    """Runs the fp64 oracle, as it stands, on part of one layer: the whole
    coarse stage of slice (b, h) (tiling, pooling, coarse attention, selection,
    coarse backward) and the fine forward and backward of query cubes (their
    rows, their query-side gradients and their terms of the key-side
    gradients): the given cubes, or, with budget_s, cubes in a fixed spread-out
    order until that many seconds have passed.  Returns (seconds, executed
    FLOPs of that work counted like the GPU's: 4*Nc^2*D + 10*Nc^2*D for the
    coarse stage, (4 + 10)*64^2*D per selected pair of the cubes, cubes done)."""
    from oracle import vsa_oracle as O
    wl = inp.wl
    t0 = time.perf_counter()
    hd = O.head_of(inp, b, h)
    order = list(cubes) if budget_s is None else [(i * 97) % wl.cubes for i in range(wl.cubes)]
    done = []
    for c in order:
        hd.rows(c)
        hd.grad_query_cube(c)
        hd.fine_key_partials([c])
        hd.forget(c)
        done.append(c)
        if budget_s is not None and time.perf_counter() - t0 >= budget_s:
            break
    secs = time.perf_counter() - t0
    pairs = int(sum(int(hd.cnt[c]) for c in done))
    work = (4 + 10) * wl.cubes ** 2 * wl.head_dim + pairs * (4 + 10) * 64 * 64 * wl.head_dim
    return secs, work, len(done)


def cpu_cores():
    return int(os.environ.get("OPENBLAS_NUM_THREADS") or os.environ.get("OMP_NUM_THREADS")
               or os.cpu_count() or 1)


def cpu_baseline(inp, step_flops):
    wl = inp.wl
    secs, work, n = oracle_sample(inp, 0, 0, None, budget_s=12.0)
    value = work / secs / 1e12
    return {"value": value, "unit": "TFLOPS", "cores": cpu_cores(), "kind": "oracle",
            "sample_s": secs, "sample_tflop": work / 1e12,
            "layer_s_estimated": step_flops / 1e12 / value,
            "sample": f"fp64 numpy oracle on slice (b=0,h=0) of {wl.name}: its whole coarse "
                      f"stage plus the fine forward and backward of {n} of {wl.cubes} query "
                      f"cubes (as many as ~12 s allow); value = executed FLOPs of that work / "
                      f"its measured time (layer_s_estimated extrapolates it to the layer)"}


# nominal dense tensor rates (PFLOP/s): tf32 against bf16/fp16
TF32_OVER_BF16 = 1.1 / 2.25


def stage_roofline(name, ms, work, wl, peaks, src, grad_bytes):
    """Algorithmic work of one stage call against its bound.

    HBM stages count the bytes the method must move once (the combine
    backward: dO, G_c, G_f in bf16 and O_f in fp16 read; dG_c, dG_f
    (grad_bytes per element), dO_f in fp16 and delta written; its slice-maximum pre-pass re-reads dO
    and G_f, which is not counted).  Tensor stages count executed FLOPs: the
    fine stages on fp16 UMMAs (the bf16 rate), the coarse stages as fp32
    contractions run on tf32 UMMAs (the tf32 rate: the measured bf16 peak
    times the nominal tf32/bf16 ratio)."""
    S = flops.tensor_bytes(wl)  # one bf16 [B, heads, N, D] tensor
    small = wl.bh * wl.cubes * wl.head_dim * 4
    rows = wl.bh * wl.tokens * 4
    table = {
        "stage_pool": ("hbm", 3 * (S + S) + 3 * small),          # read bf16, write fp16 + means
        "combine_bwd": ("hbm", 3 * S + S + grad_bytes * S + S + rows + small),
        "fine_fwd": ("tensor", work["fine_fwd"]),
        "fine_fwd_bf16": ("tensor", work["fine_fwd"]),
        "fine_bwd": ("tensor", work["fine_bwd"]),
        "coarse_select": ("tensor_tf32", work["coarse_fwd"]),
        "coarse_bwd": ("tensor_tf32", work["coarse_bwd"]),
    }
    bound, amount = table[name]
    if bound == "hbm":
        achieved, peak, unit = amount / (ms * 1e-3) / 1e9, peaks["hbm_gbs"], "GB/s"
    elif bound == "tensor":
        # fp16 and bf16 dense UMMA share one nominal rate: the measured bf16 peak applies
        achieved, peak, unit = amount / (ms * 1e-3) / 1e12, peaks["bf16_tflops"], "TFLOP/s"
    else:
        achieved = amount / (ms * 1e-3) / 1e12
        peak, unit, bound = peaks["bf16_tflops"] * TF32_OVER_BF16, "TFLOP/s", "tensor"
    return {"kernel": name, "bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
            "frac": achieved / peak, "peak_source": src, "ms": ms, "algorithmic": amount}


def traffic_for(stage):
    """DRAM bytes per launch from the committed ncu summary, if the kernel is unchanged."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        rec = json.load(open(path)).get(stage)
    except (OSError, ValueError):
        return None
    if not rec:
        return None
    h = hashlib.sha256()
    for f in rec["sources"]:
        h.update(open(os.path.join(ROOT, f), "rb").read())
    return rec["bytes_per_launch"] if h.hexdigest() == rec["sha256"] else None


def config_json(wl):
    return {"workload": wl.name, "T": wl.T, "H": wl.H, "W": wl.W, "tokens": wl.tokens,
            "cubes": wl.cubes, "batch": wl.batch, "heads": wl.heads, "head_dim": wl.head_dim,
            "topk": wl.topk, "step": "forward+backward of one layer",
            "io": f"bf16 in/out, {GRAD_DTYPE} gradients (fp32 accumulation, one rounding "
                  f"at the store)", "mma": "fp16 x fp16 -> fp32 (tcgen05)",
            "l2": (f"inputs larger than L2 ({flops.tensor_bytes(wl) / 1e6:.0f} MB per bf16 "
                   f"tensor vs 129 MB): no flush" if flops.tensor_bytes(wl) > 129 * 2 ** 20
                   else "inputs fit in L2: back-to-back steps are warm-L2 (profiling runs)"),
            "parallelism": "replicas"}


def reference_arm(args):
    """The fp64 oracle on the host cores, each step a bounded sample of the
    layer (one slice's coarse stage and the fine forward and backward of two
    query cubes).  value = the executed FLOPs of the samples / their measured
    time; ms_per_step is the measured time of one sample, ms_per_step_estimated
    the whole layer at that rate."""
    wl = workload(args)
    inp = synth.Inputs(wl, with_grad=True)
    pairs = wl.bh * wl.cubes * wl.topk
    step_flops = sum(executed_flops(wl, pairs).values())
    secs, work = [], []
    for i in range(args.warmup + args.steps):
        h = i % wl.heads
        c = (i * 97) % wl.cubes
        t, w, _ = oracle_sample(inp, 0, h, [c, (c + wl.cubes // 2) % wl.cubes])
        if i >= args.warmup:
            secs.append(t)
            work.append(w)
    value = sum(work) / sum(secs) / 1e12
    sample = (f"per step: fp64 numpy oracle on one (batch, head) slice of {wl.name}: its "
              f"coarse stage plus the fine forward and backward of 2 of {wl.cubes} query "
              f"cubes; value = executed FLOPs of the samples / their measured time")
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOPS",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": statistics.mean(secs) * 1e3,
            "ms_per_step_estimated": step_flops / 1e12 / value * 1e3,
            "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_json(wl),
            "cpu_baseline": {"value": value, "unit": "TFLOPS", "cores": cpu_cores(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "TFLOPS", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def oracle_table(args):
    """Wall time of the fp64 oracle, as it stands, per configuration on this
    host's cores (a reported baseline, not a target).

    tiny and pretrain: the whole layer measured, forward and forward+backward,
    on every core (a spawn-started pool of single-threaded processes sharing
    the slices' query cubes) and in one single-threaded process (tiny: the
    whole layer; pretrain: one whole slice).  wan13b, p720, dynamic: one whole
    slice measured on every core, the layer estimated at that rate."""
    from oracle.pool import OraclePool
    every = OraclePool()
    single = OraclePool(processes=1)
    rows = []
    # start-up of the worker processes (interpreter, numpy and torch imports) is
    # not the oracle's time: one tiny call on each pool first
    warm = synth.Inputs(synth.WORKLOADS["tiny"], with_grad=True)
    for pool in (every, single):
        pool.layer(warm, [(0, 0)], "warmup", backward=True)

    def run(pool, inp, slices, backward):
        t0 = time.perf_counter()
        pool.layer(inp, slices, "timing", backward=backward)
        return time.perf_counter() - t0

    try:
        for name in ("tiny", "pretrain", "wan13b", "p720", "dynamic"):
            wl = synth.WORKLOADS[name]
            inp = synth.Inputs(wl, with_grad=True)
            everything = [(b, h) for b in range(wl.batch) for h in range(wl.heads)]
            whole = name in ("tiny", "pretrain")
            slices = everything if whole else [(0, 0)]
            row = {"workload": wl.name, "slices_timed": len(slices), "slices": wl.bh,
                   "cores": every.processes}
            modes = (False, True) if wl.backward else (False,)
            for bwd in modes:
                key = "fwdbwd" if bwd else "fwd"
                t = run(every, inp, slices, bwd)
                if whole:
                    row[f"{key}_s"] = t
                else:
                    row[f"{key}_s_one_slice"] = t
                    row[f"{key}_s_estimated"] = t * wl.bh
                if name in ("tiny", "pretrain"):
                    one = everything if name == "tiny" else [(0, 0)]
                    t1 = run(single, inp, one, bwd)
                    row[f"{key}_s_1thread" + ("" if name == "tiny" else "_one_slice")] = t1
            rows.append(row)
    finally:
        every.close()
        single.close()
    return {"oracle_wall_time": rows, "host_cpus": os.cpu_count(),
            "how": "oracle.pool.OraclePool: query cubes of each slice spread over single-"
                   "threaded spawn-started processes; the literal masked-dense fine stage "
                   "of the oracle; *_estimated = one slice x slices"}


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-side", action="store_true",
                    help="skip the per-stage timing of the other configurations")
    ap.add_argument("--workload", choices=sorted(synth.WORKLOADS), default=WORKLOAD,
                    help="layer to time (default: the 720p layer; the others are the "
                         "parity-test configurations, for profiling)")
    ap.add_argument("--oracle-table", action="store_true",
                    help="print the fp64 oracle's wall time per configuration (host only)")
    ap.add_argument("--heads", type=int, default=0,
                    help="run the layer with this many heads instead of 40 (smaller "
                         "profiling case of the same kernels)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.oracle_table:
        if rank == 0:
            print(json.dumps(oracle_table(args)), flush=True)
        return
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(reference_arm(args)), flush=True)
        return
    if world > 1:
        torch.distributed.init_process_group("nccl")
    r = gpu_arm(args, rank, world)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
    if rank != 0:
        return
    wl, work = r["wl"], r["work"]
    step_flops = sum(work.values())
    peaks, src = load_peaks()
    stages = r["stages"]
    # the dominant kernel's roofline from its time as it runs inside the step:
    # back-to-back calls, L2 as the previous call left it (the step flushes
    # nothing); the L2-flushed medians are reported beside it
    warm = r["stages_warm"]
    top = max((k for k in warm if k != "fine_fwd_bf16"), key=warm.get)
    roof = stage_roofline(top, warm[top], work, wl, peaks, src,
                          grad_bytes=2 if GRAD_DTYPE == "bf16" else 4)
    roof["traffic"] = traffic_for(top)
    roof["timing"] = (f"median of {SIDE_REPS} calls of the stage's C-ABI entry point, "
                      f"back to back (as in the step); includes its list building")
    # shares of the training step's stages (the in-place inference fine stage is extra)
    train = {k: v for k, v in stages.items() if k != "fine_fwd_bf16"}
    total = sum(train.values())
    line = {
        "metric": METRIC,
        "value": job_throughput(step_flops, world, r["ms_step"]),
        "unit": "TFLOPS", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": r["ms_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16", "data": "synthetic", "config": config_json(wl),
        "fwd_ms_per_layer": r["ms_fwd"], "fwdbwd_ms_per_layer": r["ms_step"],
        "fwd_inference_ms_per_layer": r["ms_fwd_inf"],
        "fwdbwd_ms_fp32_grads": r["ms_step_fp32_grads"],
        "fwd_inference_note": "vsa_forward without the backward: cube means, coarse stage, "
                              "and the fine stage reading the bf16 inputs in place (5-D "
                              "cube copies, no staged fp16 copies)",
        "fwd_tflops": (work["fine_fwd"] + work["coarse_fwd"]) / (r["ms_fwd"] * 1e-3) / 1e12,
        "executed_gflop": {k: v / 1e9 for k, v in work.items()}, "selected_pairs": r["pairs"],
        "stages_ms": stages, "stages_ms_warm": warm,
        "stages_timing": f"median of {SIDE_REPS} single calls; stages_ms with the L2 "
                         f"flushed before each call, stages_ms_warm back to back",
        "stage_share": {k: v / total for k, v in train.items()},
        "fine_fwd_frac_of_peak": work["fine_fwd"] / (stages["fine_fwd"] * 1e-3) / 1e12
        / peaks["bf16_tflops"],
        "roofline": roof,
        "clocks": r["clocks"],
        "e2e": {"value": world * r["e2e"]["value"], "unit": "TFLOPS",
                "h2d_bytes_per_step": r["e2e"]["h2d"], "d2h_bytes_per_step": r["e2e"]["d2h"],
                "ms_per_step": r["e2e"]["ms"], "pipeline_units": r["e2e"]["units"],
                "timer": "host clock between device synchronisations (three streams)",
                "host_link": r["e2e"]["link"],
                "with_fp32_gradients": {
                    "ms_per_step": r["e2e"]["fp32_gradients"]["ms"],
                    "value": world * r["e2e"]["fp32_gradients"]["value"],
                    "d2h_bytes_per_step": r["e2e"]["fp32_gradients"]["d2h"]}},
        "gpu_launches": (LAUNCHES_FWD + LAUNCHES_BWD) * args.steps,
        "load_balance": r["balance"],
    }
    if r["fp8"]:
        line["fp8_forward"] = r["fp8"]
    if r["side"]:
        line["other_configs"] = r["side"]
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(r["inp"], step_flops)
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
