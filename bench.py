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
dense tensor peak.  cpu_baseline: the fp64 oracle on the host cores, on a
bounded sample of the same layer, extrapolated to the layer.

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
LAUNCHES_FWD = 9   # stage x3, tf32 split, coarse logits GEMM + select + O_c GEMM, pair lists,
                   # fine forward
LAUNCHES_BWD = 16  # combine bwd, coarse bwd (row dot, tf32 split, 5 GEMMs), pair lists,
                   # transposed lists (mask, count, scan, fill, pairs), fine bwd x2
SIDE_WORKLOADS = ("wan13b", "dynamic")  # timed per stage beside the headline layer
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


def workload(args):
    wl = synth.WORKLOADS[WORKLOAD]
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
    cfg = vsa.config_for(wl)
    t = {n: getattr(inp, n).to(dev) for n in ("q", "k", "v", "gc", "gf", "do")}
    bufs = vsa.Buffers(cfg, dev, with_backward=True)
    B, H, N, D = wl.batch, wl.heads, wl.tokens, wl.head_dim
    o = torch.empty_like(t["q"])
    grads = tuple(torch.empty(B, H, N, D, dtype=torch.float32, device=dev) for _ in range(5))
    stream = torch.cuda.current_stream()

    def fwd():
        vsa.forward(cfg, t["q"], t["k"], t["v"], t["gc"], t["gf"], bufs, True, out=o)

    def step():
        fwd()
        vsa.backward(cfg, t["gc"], t["gf"], t["do"], bufs, grads)

    fwd()
    torch.cuda.synchronize()
    pairs = int(bufs.view("cnt", torch.int32, (B, H, wl.cubes)).sum().item())
    balance = balance_report(vsa, bufs, wl, dev)
    work = executed_flops(wl, pairs)
    step_flops = sum(work.values())

    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(dev.index) as clk:
        ms_step = timed(step, args.steps, args.warmup, stream)
    ms_fwd = timed(fwd, max(3, args.steps // 2), 1, stream)
    status = bufs.device_status()
    if status != vsa.OK:
        raise RuntimeError(f"device status {status} after the timed steps")
    ms_max = max_over_ranks(ms_step, world, dev)

    stages = stage_breakdown(vsa, cfg, wl, t, bufs, stream, dev)
    e2e = end_to_end(vsa, cfg, wl, inp, bufs, stream, dev, step_flops, args)
    side = {}
    if rank == 0 and not args.no_side:
        del bufs, grads, o, t
        torch.cuda.empty_cache()
        side = {name: side_workload(vsa, name, dev) for name in SIDE_WORKLOADS}
    return {"wl": wl, "work": work, "pairs": pairs, "ms_step": ms_max, "ms_fwd": ms_fwd,
            "clocks": clk.summary(), "stages": stages, "e2e": e2e, "inp": inp,
            "balance": balance, "side": side}


def balance_report(vsa, bufs, wl, dev):
    """Per-CTA work of the persistent fine kernels under their static item
    assignment (max/mean of the step counts) and the list-length histogram."""
    from trainable_block_sparse_gb300 import schedule
    B, H, nc, cap = wl.batch, wl.heads, wl.cubes, wl.list_capacity
    idx = bufs.view("idx", torch.int32, (B * H, nc, cap)).cpu().numpy()
    cnt = bufs.view("cnt", torch.int32, (B * H, nc)).cpu().numpy()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    ordered = schedule.uses_cost_order(B * H, wl.tokens, wl.head_dim)
    return schedule.load_balance(idx, cnt, sms, ordered=ordered)


def side_workload(vsa, name, dev):
    """Per-stage times of another configuration of the same layer (inputs
    resident, 3 repetitions per stage), its fwd and fwd+bwd time per layer,
    and the fine kernels' work distribution."""
    wl = synth.WORKLOADS[name]
    inp = synth.Inputs(wl, with_grad=True)
    cfg = vsa.config_for(wl)
    t = {n: getattr(inp, n).to(dev) for n in ("q", "k", "v", "gc", "gf", "do")}
    bufs = vsa.Buffers(cfg, dev, with_backward=True)
    B, H, N, D = wl.batch, wl.heads, wl.tokens, wl.head_dim
    o = torch.empty_like(t["q"])
    grads = tuple(torch.empty(B, H, N, D, dtype=torch.float32, device=dev) for _ in range(5))
    stream = torch.cuda.current_stream()

    def fwd():
        vsa.forward(cfg, t["q"], t["k"], t["v"], t["gc"], t["gf"], bufs, True, out=o)

    def step():
        fwd()
        vsa.backward(cfg, t["gc"], t["gf"], t["do"], bufs, grads)

    ms_fwd = timed(fwd, 5, 3, stream)
    ms_step = timed(step, 5, 3, stream)
    if bufs.device_status() != vsa.OK:
        raise RuntimeError(f"{name}: device status {bufs.device_status()}")
    pairs = int(bufs.view("cnt", torch.int32, (B, H, wl.cubes)).sum().item())
    work = executed_flops(wl, pairs)
    balance = balance_report(vsa, bufs, wl, dev)
    stages = stage_breakdown(vsa, cfg, wl, t, bufs, stream, dev)
    peaks, _ = load_peaks()
    return {"workload": wl.name, "selected_pairs": pairs, "fwd_ms_per_layer": ms_fwd,
            "fwdbwd_ms_per_layer": ms_step, "stages_ms": stages,
            "fine_fwd_tflops": work["fine_fwd"] / (stages["fine_fwd"] * 1e-3) / 1e12,
            "fine_fwd_frac_of_peak": work["fine_fwd"] / (stages["fine_fwd"] * 1e-3) / 1e12
            / peaks["bf16_tflops"],
            "fine_bwd_tflops": work["fine_bwd"] / (stages["fine_bwd"] * 1e-3) / 1e12,
            "load_balance": balance}


def stage_breakdown(vsa, cfg, wl, t, bufs, stream, dev, reps=3):
    """Each stage alone through its own C-ABI entry point: ms per call."""
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
    dgc, dgf, dq, dk, dv = (torch.empty(B, H, N, D, **f32) for _ in range(5))
    dof = torch.empty(B, H, N, D, dtype=torch.float16, device=dev)
    doc, dqc, dkc, dvc = (torch.empty(B, H, nc, D, **f32) for _ in range(4))
    delta = torch.empty(B, H, N, **f32)
    ws, c, s = bufs.ws, ctypes.byref(cfg), vsa._stream()

    def ck(st, name):
        if st != vsa.OK:
            raise RuntimeError(f"{name} returned {st}")

    calls = {
        "stage_pool": lambda: [ck(L.vsa_stage(c, P(t[n]), P(v[n + "16"]), P(v[n + "c"]), P(ws), s),
                                  "vsa_stage") for n in ("q", "k", "v")],
        "coarse_select": lambda: ck(L.vsa_coarse_select(
            c, P(t["q"]), P(t["k"]), P(t["v"]), P(v["qc"]), P(v["kc"]), P(v["vc"]), P(v["oc"]),
            P(v["lse_c"]), P(v["idx"]), P(v["cnt"]), P(ws), s), "vsa_coarse_select"),
        "fine_fwd": lambda: ck(L.vsa_fine_fwd(
            c, P(v["q16"]), P(v["k16"]), P(v["v16"]), P(v["idx"]), P(v["cnt"]), P(t["gc"]),
            P(t["gf"]), P(v["oc"]), P(o), P(v["o_f"]), P(v["lse_f"]), P(ws), s), "vsa_fine_fwd"),
        "combine_bwd": lambda: ck(L.vsa_combine_bwd(
            c, P(t["do"]), P(t["gc"]), P(t["gf"]), P(v["o_f"]), P(v["oc"]), P(dgc), P(dgf),
            P(dof), P(doc), P(delta), P(ws), s), "vsa_combine_bwd"),
        "coarse_bwd": lambda: ck(L.vsa_coarse_bwd(
            c, P(v["qc"]), P(v["kc"]), P(v["vc"]), P(v["oc"]), P(v["lse_c"]), P(doc), P(dqc),
            P(dkc), P(dvc), P(ws), s), "vsa_coarse_bwd"),
        "fine_bwd": lambda: ck(L.vsa_fine_bwd(
            c, P(v["q16"]), P(v["k16"]), P(v["v16"]), P(v["idx"]), P(v["cnt"]), P(v["lse_f"]),
            P(dof), P(delta), P(dqc), P(dkc), P(dvc), P(dq), P(dk), P(dv), P(ws), s),
            "vsa_fine_bwd"),
    }
    return {name: timed(fn, reps, 1, stream) for name, fn in calls.items()}


def end_to_end(vsa, cfg, wl, inp, bufs, stream, dev, step_flops, args):
    """Host inputs in, host outputs out, every step, through the library's
    host-buffer pipeline (HostPipeline: units of 5 heads, copies in and out
    overlapped with the kernels of the neighbouring units)."""
    from trainable_block_sparse_gb300.host_pipeline import HostPipeline, IN_NAMES, OUT_NAMES
    del bufs  # the pipeline owns per-unit buffers
    host_in = {n: getattr(inp, n).pin_memory() for n in IN_NAMES}
    B, H, N, D = wl.batch, wl.heads, wl.tokens, wl.head_dim
    host_out = {n: torch.empty(B, H, N, D, dtype=torch.bfloat16 if n == "o" else torch.float32,
                               pin_memory=True) for n in OUT_NAMES}
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
    return {"ms": ms, "value": step_flops / (ms * 1e-3) / 1e12, "h2d": h2d, "d2h": d2h,
            "units": sum(1 for _ in pipe.units())}


def oracle_sample(inp, b, h, cubes):
    """Times the fp64 oracle on one (batch, head) slice and a few cubes.

    Returns (estimated seconds for the whole slice, seconds actually spent).
    The slice estimate is the oracle as it stands: the per-slice part (tiling,
    pooling, coarse attention, selection, coarse backward) once, plus per cube
    its fine forward rows, its query-side gradient and its key-side gradient.
    """
    from oracle import vsa_oracle as O
    wl = inp.wl
    t0 = time.perf_counter()
    hd = O.head_of(inp, b, h)
    t_head = time.perf_counter() - t0
    per_cube = []
    for c in cubes:
        t1 = time.perf_counter()
        hd.rows(c)
        hd.grad_query_cube(c)
        t_q = time.perf_counter() - t1
        for i in range(wl.cubes):  # the selectors' forward rows belong to their own cubes
            if c in hd.idx[i][: hd.cnt[i]]:
                hd.rows(i)
        t2 = time.perf_counter()
        hd.grad_key_cube(c)
        per_cube.append(t_q + time.perf_counter() - t2)
    spent = time.perf_counter() - t0
    return t_head + wl.cubes * statistics.mean(per_cube), spent


def cpu_cores():
    return int(os.environ.get("OPENBLAS_NUM_THREADS") or os.environ.get("OMP_NUM_THREADS")
               or os.cpu_count() or 1)


def cpu_baseline(inp, step_flops):
    wl = inp.wl
    cubes = [0, wl.cubes // 2]
    slice_s, spent = oracle_sample(inp, 0, 0, cubes)
    layer_s = slice_s * wl.bh
    return {"value": step_flops / layer_s / 1e12, "unit": "TFLOPS", "cores": cpu_cores(),
            "kind": "oracle", "layer_s_estimated": layer_s, "sample_s": spent,
            "sample": f"fp64 numpy oracle, forward+backward of slice (b=0,h=0) of {wl.name}: "
                      f"per-slice coarse work once plus {len(cubes)} of {wl.cubes} cubes "
                      f"(fine rows, query- and key-side gradients), extrapolated to "
                      f"{wl.cubes} cubes x {wl.bh} slices"}


def stage_roofline(name, ms, work, wl, peaks, src):
    S = flops.tensor_bytes(wl)  # one bf16 [B, heads, N, D] tensor
    small = wl.bh * wl.cubes * wl.head_dim * 4
    alu_peak = 152 * 128 * 2 * peaks.get("sm_max_mhz", 2070.0) * 1e6 / 1e12  # fp32 FMA lanes
    table = {
        "stage_pool": ("hbm", 3 * (S + S) + 3 * small),          # read bf16, write fp16 + means
        "combine_bwd": ("hbm", 3 * S + 2 * S + 4 * S + S + wl.bh * wl.tokens * 4 + small),
        "fine_fwd": ("tensor", work["fine_fwd"]),
        "fine_bwd": ("tensor", work["fine_bwd"]),
        "coarse_select": ("alu", work["coarse_fwd"]),
        "coarse_bwd": ("alu", work["coarse_bwd"]),
    }
    bound, amount = table[name]
    if bound == "hbm":
        achieved, peak, unit = amount / (ms * 1e-3) / 1e9, peaks["hbm_gbs"], "GB/s"
    elif bound == "tensor":
        # fp16 and bf16 dense UMMA share one nominal rate: the measured bf16 peak applies
        achieved, peak, unit = amount / (ms * 1e-3) / 1e12, peaks["bf16_tflops"], "TFLOP/s"
    else:
        achieved, peak, unit = amount / (ms * 1e-3) / 1e12, alu_peak, "TFLOP/s"
    return {"kernel": name, "bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
            "frac": achieved / peak, "peak_source": src, "ms": ms}


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
            "io": "bf16 in/out, fp32 gradients", "mma": "fp16 x fp16 -> fp32 (tcgen05)",
            "l2": "inputs larger than L2 (721 MB per bf16 tensor vs 129 MB): no flush",
            "parallelism": "replicas"}


def reference_arm(args):
    """The fp64 oracle on the host cores, each step a bounded sample of the layer."""
    wl = workload(args)
    inp = synth.Inputs(wl, with_grad=True)
    pairs = wl.bh * wl.cubes * wl.topk
    step_flops = sum(executed_flops(wl, pairs).values())
    layer_s = []
    for i in range(args.warmup + args.steps):
        h = i % wl.heads
        c = (i * 97) % wl.cubes
        slice_s, _ = oracle_sample(inp, 0, h, [c])
        if i >= args.warmup:
            layer_s.append(slice_s * wl.bh)
    sec = statistics.mean(layer_s)
    value = step_flops / sec / 1e12
    sample = (f"per step: fp64 numpy oracle on one (batch, head) slice of {wl.name} (per-slice "
              f"coarse work + 1 of {wl.cubes} cubes), extrapolated to the layer")
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOPS",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": sec * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_json(wl),
            "cpu_baseline": {"value": value, "unit": "TFLOPS", "cores": cpu_cores(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "TFLOPS", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-side", action="store_true",
                    help="skip the per-stage timing of the other configurations")
    ap.add_argument("--heads", type=int, default=0,
                    help="run the layer with this many heads instead of 40 (smaller "
                         "profiling case of the same kernels)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
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
    top = max(stages, key=stages.get)
    roof = stage_roofline(top, stages[top], work, wl, peaks, src)
    roof["traffic"] = traffic_for(top)
    total = sum(stages.values())
    line = {
        "metric": METRIC,
        "value": job_throughput(step_flops, world, r["ms_step"]),
        "unit": "TFLOPS", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": r["ms_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16", "data": "synthetic", "config": config_json(wl),
        "fwd_ms_per_layer": r["ms_fwd"], "fwdbwd_ms_per_layer": r["ms_step"],
        "fwd_tflops": (work["fine_fwd"] + work["coarse_fwd"]) / (r["ms_fwd"] * 1e-3) / 1e12,
        "executed_gflop": {k: v / 1e9 for k, v in work.items()}, "selected_pairs": r["pairs"],
        "stages_ms": stages, "stage_share": {k: v / total for k, v in stages.items()},
        "fine_fwd_frac_of_peak": work["fine_fwd"] / (stages["fine_fwd"] * 1e-3) / 1e12
        / peaks["bf16_tflops"],
        "roofline": roof,
        "clocks": r["clocks"],
        "e2e": {"value": world * r["e2e"]["value"], "unit": "TFLOPS",
                "h2d_bytes_per_step": r["e2e"]["h2d"], "d2h_bytes_per_step": r["e2e"]["d2h"],
                "ms_per_step": r["e2e"]["ms"], "pipeline_units": r["e2e"]["units"],
                "timer": "host clock between device synchronisations (three streams)"},
        "gpu_launches": (LAUNCHES_FWD + LAUNCHES_BWD) * args.steps,
        "load_balance": r["balance"],
    }
    if r["side"]:
        line["other_configs"] = r["side"]
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(r["inp"], step_flops)
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
