#!/usr/bin/env python
"""Throughput of one pre-LN tensor-parallel GPT layer, forward + backward, on GB300.

A step is one forward and one backward pass of the whole layer (every kernel of
the C ABI's mtl_layer_fwd and mtl_layer_bwd) over one batch of seeded synthetic
input.  Default workload: the 8.3B-model-shaped layer (h=3072, 32 heads, seq
1024, batch 16, ffn 12288, t=8 partitions laid out on one GPU).  Its inputs and
activations (several GB) are far larger than L2, so no flush is needed between
steps.

Prints one JSON line (rank 0).  `--impl reference` times the fp64 CPU oracle
on a bounded sample instead.  Under torchrun each rank runs an independent
replica (the layer is not sharded across GPUs).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synthetic  # noqa: E402

METRIC = "layer fwd+bwd TFLOP/s on 1 GB300 and % of BF16 dense peak; oracle-match"
KIND_NAMES = {1: "gemm_tc", 2: "gemm_simt", 3: "attn_fwd", 4: "attn_bwd", 5: "ln_fwd", 9: "gemv_tc",
              10: "attn_decode", 11: "kv_write",
              6: "ln_bwd", 7: "colsum", 8: "finalize"}


def layer_flops(s, batch=None):
    b = s.batch if batch is None else batch
    n = b * s.seq
    gemm_fwd = 2 * n * (3 * s.h * s.h + s.h * s.h + 2 * s.ffn * s.h)
    attn_fwd = 2 * b * s.seq * (s.seq + 1) * s.h
    return 3 * (gemm_fwd + attn_fwd)


def megatron_flops(s):
    n = s.batch * s.seq
    return 72 * n * s.h * s.h + 12 * s.batch * s.seq * s.seq * s.h


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return p, "measured"
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, mx, reasons = [], 0.0, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = max(mx, float(parts[1]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def traffic_record(kernel_file):
    """DRAM bytes per launch of the dominant kernel from the committed ncu summary,
    or None when absent or taken on a different revision of the kernel source."""
    path = os.path.join(ROOT, "profiles", "gemm_tc_traffic.txt")
    try:
        rec = {}
        for ln in open(path):
            if ":" in ln:
                k, v = ln.split(":", 1)
                rec[k.strip()] = v.strip()
        src = open(kernel_file, "rb").read()
        if rec.get("source_sha256") != hashlib.sha256(src).hexdigest():
            return None
        return rec
    except Exception:
        return None


def aggregate_over_ranks(ms, flops_per_step, steps, world, dist=None, device=None):
    """Whole-job throughput of `world` replicas: the slowest rank's time over
    the units all ranks processed.  Returns (max_ms, TFLOP/s)."""
    if world > 1 and dist is not None:
        import torch
        t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    return ms, flops_per_step * steps * world / (ms / 1e3) / 1e12


# ---------------------------------------------------------------- reference arm

def run_reference(args, shape, rank, world):
    if rank != 0:
        return
    import oracle
    cores = len(os.sched_getaffinity(0))
    sample_batch = 1
    flops = layer_flops(shape, sample_batch)
    x, p, dy = synthetic.make_layer(shape, seed=0, batch=sample_batch)
    for _ in range(max(0, min(args.warmup, 1))):
        pass  # the oracle has no warm state worth priming; keep the run bounded
    times = []
    steps = max(1, min(args.steps, 3))
    for _ in range(steps):
        t0 = time.perf_counter()
        y, cache = oracle.layer_fwd(p, x, shape.heads, dropout=args.drop)
        oracle.layer_bwd(p, cache, dy)
        times.append(time.perf_counter() - t0)
    sec = float(np.mean(times))
    value = flops / sec / 1e12
    sample = (f"{shape.name} at batch {sample_batch} (of {shape.batch}), "
              f"{steps} fwd+bwd passes of the fp64 numpy oracle")
    out = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
           "steps": steps, "warmup": 0, "ms_per_step": sec * 1e3, "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "impl": "reference",
           "config": {"workload": f"{args.config}: {shape.name}, t={args.t}",
                      "h": shape.h, "heads": shape.heads, "seq": shape.seq,
                      "batch": sample_batch, "ffn": shape.ffn, "t": args.t,
                      "dropout": args.drop},
           "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores,
                            "kind": "oracle", "sample": sample},
           "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def cpu_baseline(shape, drop=None):
    import oracle
    x, p, dy = synthetic.make_layer(shape, seed=0, batch=1)
    t0 = time.perf_counter()
    y, cache = oracle.layer_fwd(p, x, shape.heads, dropout=drop)
    oracle.layer_bwd(p, cache, dy)
    sec = time.perf_counter() - t0
    return {"value": layer_flops(shape, 1) / sec / 1e12, "unit": "TFLOP/s",
            "cores": len(os.sched_getaffinity(0)), "kind": "oracle",
            "sample": f"{shape.name} at batch 1 (of {shape.batch}): one fwd+bwd of the "
                      f"fp64 numpy oracle, {sec:.1f} s"}


# ---------------------------------------------------------------- our arm

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="D", choices=sorted(synthetic.CONFIGS))
    ap.add_argument("--t", type=int, default=None)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--p-drop", type=float, default=0.0,
                    help="dropout probability of the attention and hidden sites (default 0)")
    args = ap.parse_args()
    args.drop = None
    if args.p_drop > 0:
        pd = float(np.float32(args.p_drop))
        args.drop = {"p_attn": pd, "p_hidden": pd, "seed": 1234}
    shape = synthetic.CONFIGS[args.config]
    if args.t is None:
        args.t = shape.t[0]
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        run_reference(args, shape, rank, world)
        return

    import torch
    import torch.distributed as dist
    from tensor_model_transformer_gb300 import mtl

    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    dt = torch.bfloat16 if shape.dtype == "bf16" else torch.float32
    x, p, dy = synthetic.make_layer(shape, seed=rank)
    drop = args.drop or {}
    desc = mtl.layer_desc(shape.h, shape.heads, shape.seq, shape.batch, shape.ffn, args.t,
                          shape.dtype, p_attn=drop.get("p_attn", 0.0),
                          p_hidden=drop.get("p_hidden", 0.0), seed=drop.get("seed", 0))
    w = {k: torch.from_numpy(v).cuda().to(dt) for k, v in p.items()}
    x_h = torch.from_numpy(x).to(dt).pin_memory()
    dy_h = torch.from_numpy(dy).to(dt).pin_memory()
    del x, p, dy
    xd = x_h.cuda()
    dyd = dy_h.cuda()
    y = torch.empty_like(xd)
    dx = torch.empty_like(xd)
    saved, ws, grads = mtl.alloc_layer_buffers(desc)
    stream = torch.cuda.current_stream()

    def step():
        mtl.layer_fwd(desc, w, xd, y, saved, ws, stream)
        n1 = mtl.last_launch_count()
        mtl.layer_bwd(desc, w, xd, saved, dyd, dx, grads, ws, stream)
        return n1 + mtl.last_launch_count()

    def barrier():
        if world > 1:
            dist.barrier()

    for _ in range(args.warmup):
        launches_per_step = step()
    mtl.layer_check(ws)
    torch.cuda.synchronize()

    # ---- timed region: inputs resident in HBM
    clocks = ClockSampler(local)
    clocks.start()
    barrier()
    torch.cuda.synchronize()
    evs_step = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    evs_step[0].record(stream)
    launches = 0
    for i in range(args.steps):
        launches += step()
        evs_step[i + 1].record(stream)
    evs_step[-1].synchronize()
    torch.cuda.synchronize()
    barrier()
    ms = evs_step[0].elapsed_time(evs_step[-1])
    per_step = sorted(evs_step[i].elapsed_time(evs_step[i + 1]) for i in range(args.steps))
    clk = clocks.stop()
    mtl.layer_check(ws)
    flops = layer_flops(shape)
    ms, value = aggregate_over_ranks(ms, flops, args.steps, world, dist if world > 1 else None,
                                     "cuda")
    ms_step = ms / args.steps

    # ---- end to end: host buffers in, results out, every step.  Each step's x
    # and dy are copied from pinned host memory and its y and dx are copied
    # back; a copy stream overlaps step i's copies with step i-1's compute
    # through double-buffered device inputs and outputs.
    barrier()
    torch.cuda.synchronize()
    copy = torch.cuda.Stream()
    xs = [xd, torch.empty_like(xd)]
    dys = [dyd, torch.empty_like(dyd)]
    ys = [y, torch.empty_like(y)]
    dxs = [dx, torch.empty_like(dx)]
    y_h = [torch.empty_like(x_h).pin_memory() for _ in range(2)]
    dx_h = [torch.empty_like(x_h).pin_memory() for _ in range(2)]
    loaded = [torch.cuda.Event() for _ in range(2)]
    computed = [torch.cuda.Event() for _ in range(2)]
    drained = [torch.cuda.Event() for _ in range(2)]

    def e2e_step_io(i):
        b = i % 2
        with torch.cuda.stream(copy):
            if i >= 2:
                copy.wait_event(computed[b])        # step i-2 is done with buffer b
            xs[b].copy_(x_h, non_blocking=True)
            dys[b].copy_(dy_h, non_blocking=True)
            loaded[b].record(copy)

    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    copy.wait_event(e0)
    e2e_step_io(0)
    for i in range(args.steps):
        b = i % 2
        if i + 1 < args.steps:
            e2e_step_io(i + 1)
        stream.wait_event(loaded[b])
        if i >= 2:
            stream.wait_event(drained[b])           # outputs of step i-2 copied out
        mtl.layer_fwd(desc, w, xs[b], ys[b], saved, ws, stream)
        mtl.layer_bwd(desc, w, xs[b], saved, dys[b], dxs[b], grads, ws, stream)
        computed[b].record(stream)
        with torch.cuda.stream(copy):
            copy.wait_event(computed[b])
            y_h[b].copy_(ys[b], non_blocking=True)
            dx_h[b].copy_(dxs[b], non_blocking=True)
            drained[b].record(copy)
    e1.record(copy)
    e1.synchronize()
    torch.cuda.synchronize()
    ms_e2e = e0.elapsed_time(e1)
    ms_e2e, e2e_value = aggregate_over_ranks(ms_e2e, flops, args.steps, world,
                                             dist if world > 1 else None, "cuda")
    nbytes = x_h.numel() * x_h.element_size()

    # ---- per-kernel times: the same steps again with events around every kernel
    cap = launches_per_step * args.steps + 16
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(2 * cap)]
    for e in evs:
        e.record(stream)
    torch.cuda.synchronize()
    import ctypes
    handles = (ctypes.c_void_p * (2 * cap))(*[e.cuda_event for e in evs])
    kinds = (ctypes.c_int32 * cap)()
    work = (ctypes.c_double * cap)()
    mtl.lib().mtl_profile_set(handles, cap, kinds, work)
    for _ in range(args.steps):
        step()
    count = mtl.lib().mtl_profile_count()
    mtl.lib().mtl_profile_set(None, 0, None, None)
    torch.cuda.synchronize()
    per_kind = {}
    for i in range(count):
        dur = evs[2 * i].elapsed_time(evs[2 * i + 1])
        k = KIND_NAMES.get(kinds[i], str(kinds[i]))
        rec = per_kind.setdefault(k, {"launches": 0, "ms": 0.0, "work": 0.0})
        rec["launches"] += 1
        rec["ms"] += dur
        rec["work"] += work[i]
    total_ms = sum(r["ms"] for r in per_kind.values()) or 1.0
    breakdown = {k: {"launches_per_step": r["launches"] // args.steps,
                     "ms_per_step": r["ms"] / args.steps, "share": r["ms"] / total_ms}
                 for k, r in sorted(per_kind.items(), key=lambda kv: -kv[1]["ms"])}

    pk, pk_src = peaks()
    dom = max(per_kind.items(), key=lambda kv: kv[1]["ms"])[0] if per_kind else None
    roofline = None
    if dom is not None:
        r = per_kind[dom]
        if dom in ("gemm_tc", "gemm_simt", "attn_fwd", "attn_bwd"):
            achieved = r["work"] / (r["ms"] / 1e3) / 1e12
            peak = pk.get("bf16_tflops_sustained", pk["bf16_tflops"])
            unit, bound = "TFLOP/s", "tensor"
        else:
            achieved = r["work"] / (r["ms"] / 1e3) / 1e9
            peak = pk["hbm_gbs"]
            unit, bound = "GB/s", "hbm"
        tr = traffic_record(os.path.join(ROOT, "tensor_model_transformer_gb300", "csrc",
                                         "gemm_tc.cu")) if dom == "gemm_tc" else None
        traffic = None
        if tr and "dram_bytes_per_launch_full" in tr:
            traffic = float(tr["dram_bytes_per_launch_full"])
        roofline = {"bound": bound, "kernel": dom, "achieved": achieved, "peak": peak,
                    "unit": unit, "frac": achieved / peak, "traffic": traffic,
                    "peak_source": f"{pk_src} bf16 sustained" if bound == "tensor"
                    else f"{pk_src} hbm"}

    out = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "step_ms": {"median": per_step[len(per_step) // 2], "min": per_step[0],
                    "max": per_step[-1]},
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": shape.dtype, "data": "synthetic",
        "config": {"workload": f"{args.config}: {shape.name}, t={args.t}", "h": shape.h,
                   "heads": shape.heads, "seq": shape.seq, "batch": shape.batch,
                   "ffn": shape.ffn, "t": args.t, "parallelism": f"replicas x{world}",
                   "l2": "inputs larger than L2 (no flush)",
                   "flops_per_step": flops, "megatron_flops_per_step": megatron_flops(shape),
                   "dropout": args.drop},
        "pct_of_bf16_peak": 100.0 * value / world / pk["bf16_tflops"],
        "peak_source": pk_src,
        "gpu_launches": launches,
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": 2 * nbytes,
                "d2h_bytes_per_step": 2 * nbytes},
        "roofline": roofline,
        "kernels": breakdown,
    }
    if clk:
        out["clocks"] = clk
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(shape, args.drop)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
