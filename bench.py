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
import gc
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
              10: "attn_decode", 11: "kv_write", 12: "gemm_fp8", 13: "fp8_quant",
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


# Idle seconds before the end-to-end pass, so that it starts from the same
# rested clock state as the device-only pass.
REST_S = 1.5
E2E_PASSES = 3   # timed end-to-end passes; the median is reported
# Nominal dense (no 2:4 sparsity) tensor rates of a GB300, TFLOP/s.
NOMINAL_TFLOPS = {"bf16": 2250.0, "fp8": 4500.0}
# Below this timed-region length a kernel is timed as a burst, so the burst
# (not the seconds-long, power-capped) measured peak is its denominator.
BURST_REGION_S = 1.0


def tensor_peak(pk, pk_src, timed_s, fp8=False):
    """(peak TFLOP/s, source text) for a tensor-bound kernel in a timed region
    of timed_s seconds: the measured burst peak for a short region, the
    sustained one for a region of a second or more; FP8 at twice the bf16
    figure (the nominal 4.5 : 2.25 dense ratio)."""
    if timed_s < BURST_REGION_S or "bf16_tflops_sustained" not in pk:
        peak, kind = pk["bf16_tflops"], "burst"
    else:
        peak, kind = pk["bf16_tflops_sustained"], "sustained"
    src = f"{pk_src} bf16 {kind} (timed region {timed_s:.2f} s)"
    if fp8:
        peak *= 2.0
        src += " x 2 (nominal fp8:bf16)"
    return peak, src


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return p, "measured"
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled while the timed region runs.

    The nvidia-smi process is started before the warm-up and left running:
    starting it inside a timed region stalls the host's kernel launches for
    milliseconds while it initialises."""

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
            self.lines.append((time.monotonic(), line.strip()))

    def window(self, t0, t1):
        """Statistics of the samples taken in [t0, t1 + 0.15] (monotonic seconds;
        a sample is printed up to one period after it is taken), or of the
        first sample after t0 when none falls inside."""
        time.sleep(0.2)
        inside = [ln for t, ln in list(self.lines) if t0 <= t <= t1 + 0.15]
        if not inside:
            inside = [ln for t, ln in list(self.lines) if t >= t0][:1]
        return self._stats(inside)

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
        return self._stats([ln for _, ln in self.lines])

    def _stats(self, lines):
        if self.proc is None:
            return None
        sm, mx, reasons = [], 0.0, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in lines:
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


def gemm_source_sha():
    """sha256 of the tensor-core GEMM's sources (gemm_core.cuh, gemm_tc.cu, the
    tail-slice instantiations gemm_split.cu, then common.cuh, which holds the
    epilogue's helpers and GeLU)."""
    csrc = os.path.join(ROOT, "tensor_model_transformer_gb300", "csrc")
    data = b"".join(open(os.path.join(csrc, f), "rb").read()
                    for f in ("gemm_core.cuh", "gemm_tc.cu", "gemm_split.cu", "common.cuh"))
    return hashlib.sha256(data).hexdigest()


def traffic_record():
    """DRAM bytes per launch of the dominant kernel from the committed ncu summary,
    or None when absent or taken on a different revision of the kernel source."""
    path = os.path.join(ROOT, "profiles", "gemm_tc_traffic.txt")
    try:
        rec = {}
        for ln in open(path):
            if ":" in ln:
                k, v = ln.split(":", 1)
                rec[k.strip()] = v.strip()
        if rec.get("source_sha256") != gemm_source_sha():
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
    # each step is one fwd+bwd of the oracle on the batch-1 sample (~2.5 s on 16
    # cores); warm-ups and steps are as asked, bounded so a run stays within a
    # few minutes
    warm = max(0, min(args.warmup, 5))
    steps = max(1, min(args.steps, 40))
    for _ in range(warm):
        y, cache = oracle.layer_fwd(p, x, shape.heads, dropout=args.drop)
        oracle.layer_bwd(p, cache, dy)
    times = []
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
           "steps": steps, "warmup": warm, "ms_per_step": sec * 1e3, "higher_is_better": True,
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


# ---------------------------------------------------------------- decode workload

DECODE_METRIC = "decode tokens/s on 1 GB300 (one token per sequence per step, KV cache)"


def decode_bytes(s, lengths, esz=2):
    """Algorithmic HBM bytes of one decode step: every weight once, the K and V
    cache of each sequence up to and including its new position (written once,
    read once), the small vectors; token-sized activations left out."""
    weights = (3 * s.h * s.h + s.h * s.h + 2 * s.h * s.ffn) * esz
    vectors = (3 * s.h + s.h + s.ffn + s.h + 4 * s.h) * esz
    kv = sum(2 * (int(L) + 1) * s.h * esz for L in lengths)
    return weights + vectors + kv


def decode_flops(s, lengths):
    g = 2 * (3 * s.h * s.h + s.h * s.h + 2 * s.h * s.ffn) * len(lengths)
    a = sum(4 * (int(L) + 1) * s.h for L in lengths)
    return g + a


def run_decode_reference(args, shape, rank, world):
    if rank != 0:
        return
    out = decode_cpu_baseline(shape, args.steps)
    line = {"metric": DECODE_METRIC, "value": out["value"], "unit": "tokens/s", "n_gpus": world,
            "steps": out["steps"], "warmup": 0, "ms_per_step": out["ms_per_step"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference",
            "config": {"workload": f"decode {args.config}: {shape.name}, batch 1 (of "
                                   f"{shape.batch}), context {shape.seq}", "h": shape.h,
                       "heads": shape.heads, "ffn": shape.ffn, "batch": 1, "context": shape.seq},
            "cpu_baseline": {"value": out["value"], "unit": "tokens/s", "cores": out["cores"],
                             "kind": "oracle", "sample": out["sample"]},
            "e2e": {"value": out["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def decode_cpu_baseline(shape, steps):
    """The oracle's decode step at batch 1 with a random cache of the prompt length."""
    import oracle
    d = shape.h // shape.heads
    _, p, _ = synthetic.make_layer(shape.with_(batch=1, seq=1), seed=0)
    rng = np.random.default_rng(3)
    cache = oracle.decode.kv_cache(1, shape.heads, shape.seq + steps + 1, d)
    cache["k"][:, :, :shape.seq] = rng.standard_normal((1, shape.heads, shape.seq, d))
    cache["v"][:, :, :shape.seq] = rng.standard_normal((1, shape.heads, shape.seq, d))
    cache["len"][:] = shape.seq
    n = max(1, min(steps, 5))
    t0 = time.perf_counter()
    for _ in range(n):
        oracle.decode.decode_step(p, rng.standard_normal((1, shape.h)), shape.heads, cache)
    sec = (time.perf_counter() - t0) / n
    return {"value": 1.0 / sec, "unit": "tokens/s", "cores": len(os.sched_getaffinity(0)),
            "kind": "oracle", "steps": n, "ms_per_step": sec * 1e3,
            "sample": f"{shape.name} at batch 1, context {shape.seq}: {n} decode steps of the "
                      f"fp64 numpy oracle, {sec:.2f} s each"}


def run_decode(args, shape, rank, world, local):
    import ctypes
    import torch
    import torch.distributed as dist
    from tensor_model_transformer_gb300 import mtl

    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dt = torch.bfloat16 if shape.dtype == "bf16" else torch.float32
    prompt, batch = shape.seq, shape.batch
    max_seq = prompt + max(args.steps, args.warmup) + 8
    x, p, _ = synthetic.make_layer(shape, seed=rank)
    desc = mtl.layer_desc(shape.h, shape.heads, prompt, batch, shape.ffn, args.t, shape.dtype)
    kvb, pwb, dwb = mtl.infer_sizes(desc, max_seq)
    w = {k: torch.from_numpy(v).cuda().to(dt) for k, v in p.items()}
    xd = torch.from_numpy(x).to(dt).cuda()
    del x
    yd = torch.empty_like(xd)
    kv = torch.zeros(kvb, dtype=torch.uint8, device="cuda")
    pws = torch.empty(pwb, dtype=torch.uint8, device="cuda")
    dws = torch.empty(dwb, dtype=torch.uint8, device="cuda")
    lens = torch.zeros(batch, dtype=torch.int32, device="cuda")
    rng = np.random.default_rng(rank + 11)
    tok_h = torch.from_numpy(rng.standard_normal((batch, shape.h)).astype(np.float32)).to(dt)
    tok_h = tok_h.pin_memory()
    x_in = tok_h.cuda()
    y_out = torch.empty_like(x_in)
    stream = torch.cuda.current_stream()

    # prefill (timed once after one warm-up)
    for _ in range(2):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        mtl.layer_prefill(desc, w, xd, yd, kv, max_seq, lens, pws, stream)
        e1.record(stream)
    mtl.layer_check(pws, stream)
    prefill_ms = e0.elapsed_time(e1)
    del pws

    def reset():
        lens.fill_(prompt)

    # eager warm-up, then one decode step captured as a CUDA graph
    reset()
    for _ in range(args.warmup):
        mtl.layer_decode(desc, w, x_in, y_out, kv, max_seq, lens, dws, stream)
    launches_per_step = mtl.last_launch_count()
    mtl.layer_check(dws, stream)
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side, capture_error_mode="relaxed"):
            mtl.layer_decode(desc, w, x_in, y_out, kv, max_seq, lens, dws, side)
    torch.cuda.synchronize()

    # ---- timed region: graph replays, inputs resident in HBM
    reset()
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    evs[0].record(stream)
    for i in range(args.steps):
        graph.replay()
        evs[i + 1].record(stream)
    evs[-1].synchronize()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    ms = evs[0].elapsed_time(evs[-1])
    per_step = sorted(evs[i].elapsed_time(evs[i + 1]) for i in range(args.steps))
    clk = clocks.stop()
    mtl.layer_check(dws, stream)
    if world > 1:
        t = torch.tensor([ms], dtype=torch.float64, device="cuda")
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    lengths = [prompt + i for i in range(args.steps)]
    total_bytes = sum(decode_bytes(shape, [L] * batch) for L in lengths)
    total_flops = sum(decode_flops(shape, [L] * batch) for L in lengths)
    tokens = batch * args.steps * world
    value = tokens / (ms / 1e3)

    # ---- end to end: each step copies its tokens in from pinned host memory and
    # its outputs back out
    reset()
    y_h = torch.empty_like(tok_h).pin_memory()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(args.steps):
        x_in.copy_(tok_h, non_blocking=True)
        graph.replay()
        y_h.copy_(y_out, non_blocking=True)
    e1.record(stream)
    e1.synchronize()
    ms_e2e = e0.elapsed_time(e1)
    e2e_value = tokens / (ms_e2e / 1e3)
    nbytes = tok_h.numel() * tok_h.element_size()

    # ---- per-kernel times (eager calls with events around every kernel)
    reset()
    cap = launches_per_step * args.steps + 16
    kev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * cap)]
    for e in kev:
        e.record(stream)
    torch.cuda.synchronize()
    handles = (ctypes.c_void_p * (2 * cap))(*[e.cuda_event for e in kev])
    kinds = (ctypes.c_int32 * cap)()
    work = (ctypes.c_double * cap)()
    mtl.lib().mtl_profile_set(handles, cap, kinds, work)
    for _ in range(args.steps):
        mtl.layer_decode(desc, w, x_in, y_out, kv, max_seq, lens, dws, stream)
    count = mtl.lib().mtl_profile_count()
    mtl.lib().mtl_profile_set(None, 0, None, None)
    torch.cuda.synchronize()
    per_kind = {}
    for i in range(count):
        k = KIND_NAMES.get(kinds[i], str(kinds[i]))
        rec = per_kind.setdefault(k, {"launches": 0, "ms": 0.0, "work": 0.0})
        rec["launches"] += 1
        rec["ms"] += kev[2 * i].elapsed_time(kev[2 * i + 1])
        rec["work"] += work[i]
    # attention's bytes are known here, not in the library (lengths live on the device)
    if "attn_decode" in per_kind:
        per_kind["attn_decode"]["work"] = float(sum(2 * (L + 1) * shape.h * 2 * batch
                                                    for L in lengths))
    total_ms = sum(r["ms"] for r in per_kind.values()) or 1.0
    breakdown = {k: {"launches_per_step": r["launches"] // args.steps,
                     "ms_per_step": r["ms"] / args.steps, "share": r["ms"] / total_ms,
                     "gbs": (r["work"] / (r["ms"] / 1e3) / 1e9) if r["work"] else None}
                 for k, r in sorted(per_kind.items(), key=lambda kv: -kv[1]["ms"])}
    pk, pk_src = peaks()
    dom = max(per_kind.items(), key=lambda kv: kv[1]["ms"])[0]
    r = per_kind[dom]
    achieved = r["work"] / (r["ms"] / 1e3) / 1e9
    step_gbs = total_bytes / (ms / 1e3) / 1e9 / world
    out = {
        "metric": DECODE_METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms / args.steps,
        "step_ms": {"median": per_step[len(per_step) // 2], "min": per_step[0],
                    "max": per_step[-1]},
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": shape.dtype, "data": "synthetic",
        "config": {"workload": f"decode {args.config}: {shape.name}, t={args.t}, batch {batch}, "
                               f"context {prompt}..{prompt + args.steps - 1}",
                   "h": shape.h, "heads": shape.heads, "ffn": shape.ffn, "t": args.t,
                   "batch": batch, "prompt": prompt, "max_seq": max_seq,
                   "parallelism": f"replicas x{world}", "cuda_graph": True,
                   "l2": "weights and KV cache larger than L2 (no flush)",
                   "bytes_per_step": total_bytes / args.steps,
                   "flops_per_step": total_flops / args.steps},
        "gpu_launches": launches_per_step * args.steps,
        "step_hbm_gbs": step_gbs, "step_hbm_frac": step_gbs / pk["hbm_gbs"],
        "prefill": {"ms": prefill_ms, "tflops": layer_flops(shape) / 3 / (prefill_ms / 1e3) / 1e12,
                    "tokens": batch * prompt},
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": nbytes,
                "d2h_bytes_per_step": nbytes},
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": pk["hbm_gbs"],
                     "unit": "GB/s", "frac": achieved / pk["hbm_gbs"], "traffic": None,
                     "peak_source": f"{pk_src} hbm"},
        "kernels": breakdown,
    }
    if clk:
        out["clocks"] = clk
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cb = decode_cpu_baseline(shape, 3)
        out["cpu_baseline"] = {k: cb[k] for k in ("value", "unit", "cores", "kind", "sample")}
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        dist.destroy_process_group()


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
    ap.add_argument("--fp8", nargs="?", const="fwd", choices=["fwd", "hybrid"], default=None,
                    help="FP8 GEMMs: fwd = E4M3 forward, bf16 backward; hybrid = also the "
                         "backward in FP8 (E5M2 gradients x E4M3)")
    ap.add_argument("--post-ln", action="store_true", help="Post-LN (original BERT) layer")
    ap.add_argument("--recompute", action="store_true",
                    help="selective recomputation of the LayerNorm outputs and GeLU(z)")
    ap.add_argument("--workload", choices=["train", "decode"], default="train",
                    help="train: fwd+bwd step (default); decode: prefill, then one-token "
                         "decode steps over the KV cache")
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

    if args.workload == "decode":
        if args.impl == "reference":
            run_decode_reference(args, shape, rank, world)
        else:
            run_decode(args, shape, rank, world, local)
        return
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
                          p_hidden=drop.get("p_hidden", 0.0), seed=drop.get("seed", 0),
                          fp8={None: 0, "fwd": 1, "hybrid": 2}[args.fp8],
                          post_ln=1 if args.post_ln else 0,
                          recompute=1 if args.recompute else 0)
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

    clocks = ClockSampler(local)
    clocks.start()
    for _ in range(args.warmup):
        launches_per_step = step()
    mtl.layer_check(ws)
    torch.cuda.synchronize()

    # ---- timed region: inputs resident in HBM.  Python's garbage collector is
    # off inside the timed regions: a full collection pauses the launching
    # thread for milliseconds, which the GPU sees as an idle gap.
    barrier()
    torch.cuda.synchronize()
    gc.collect()
    gc.disable()
    t_dev = time.monotonic()
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
    gc.enable()
    clk = clocks.window(t_dev, time.monotonic())
    mtl.layer_check(ws)
    flops = layer_flops(shape)
    ms, value = aggregate_over_ranks(ms, flops, args.steps, world, dist if world > 1 else None,
                                     "cuda")
    ms_step = ms / args.steps

    # ---- end to end: host buffers in, results out, every step.  Each step's x
    # and dy are copied from pinned host memory and its y and dx are copied
    # back; one stream per copy direction overlaps step i's copies with the
    # neighbouring steps' compute through double-buffered device inputs and
    # outputs (the two directions run on their own copy engines at once).
    # Both timed passes start from a rested GPU: under seconds of sustained
    # load the power limit lowers the clock (a step measured at 7.0 ms after
    # rest took 7.8 ms half a second into a run), which would otherwise be
    # charged to whichever pass runs second.  After the rest a few untimed
    # steps of the same pipeline wake the host and the GPU up (the first
    # launches after an idle second were measured arriving milliseconds late).
    barrier()
    torch.cuda.synchronize()
    time.sleep(REST_S)
    copy = torch.cuda.Stream()
    copy_out = torch.cuda.Stream()
    xs = [xd, torch.empty_like(xd)]
    dys = [dyd, torch.empty_like(dyd)]
    ys = [y, torch.empty_like(y)]
    dxs = [dx, torch.empty_like(dx)]
    y_h = [torch.empty_like(x_h).pin_memory() for _ in range(2)]
    dx_h = [torch.empty_like(x_h).pin_memory() for _ in range(2)]
    loaded = [torch.cuda.Event() for _ in range(2)]
    computed = [torch.cuda.Event() for _ in range(2)]
    drained = [torch.cuda.Event() for _ in range(2)]

    def e2e_pass(nsteps):
        """nsteps pipelined steps; (ms from start to the last copy out, per-step
        event intervals on the compute, copy-in and copy-out streams)."""
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        tev = {k: [torch.cuda.Event(enable_timing=True) for _ in range(nsteps)]
               for k in ("c0", "c1", "i0", "i1", "o0", "o1")}
        torch.cuda.synchronize()
        e0.record(stream)
        copy.wait_event(e0)
        copy_out.wait_event(e0)

        def io_in(i):
            b = i % 2
            with torch.cuda.stream(copy):
                if i >= 2:
                    copy.wait_event(computed[b])    # step i-2 is done with buffer b
                tev["i0"][i].record(copy)
                xs[b].copy_(x_h, non_blocking=True)
                dys[b].copy_(dy_h, non_blocking=True)
                tev["i1"][i].record(copy)
                loaded[b].record(copy)

        io_in(0)
        host = []
        for i in range(nsteps):
            host.append(time.perf_counter())
            b = i % 2
            if i + 1 < nsteps:
                io_in(i + 1)
            stream.wait_event(loaded[b])
            if i >= 2:
                stream.wait_event(drained[b])       # outputs of step i-2 copied out
            tev["c0"][i].record(stream)
            mtl.layer_fwd(desc, w, xs[b], ys[b], saved, ws, stream)
            mtl.layer_bwd(desc, w, xs[b], saved, dys[b], dxs[b], grads, ws, stream)
            tev["c1"][i].record(stream)
            computed[b].record(stream)
            with torch.cuda.stream(copy_out):
                copy_out.wait_event(computed[b])
                tev["o0"][i].record(copy_out)
                y_h[b].copy_(ys[b], non_blocking=True)
                dx_h[b].copy_(dxs[b], non_blocking=True)
                tev["o1"][i].record(copy_out)
                drained[b].record(copy_out)
        host.append(time.perf_counter())
        e1.record(copy_out)
        e1.synchronize()
        torch.cuda.synchronize()
        # longest host time to enqueue one step
        host_ms = max(1e3 * (host[i + 1] - host[i]) for i in range(nsteps))
        return e0.elapsed_time(e1), tev, e0, host_ms

    e2e_pass(3)                                      # untimed: wake up after the rest
    # Three timed passes of K steps each; the median one is reported (a single
    # host stall -- a descheduled enqueue thread -- once delayed the first copy
    # of a pass by 13 ms), all three are listed in e2e.passes_ms.
    passes = []
    for _ in range(E2E_PASSES):
        barrier()
        gc.collect()
        gc.disable()
        t_e2e = time.monotonic()
        res = e2e_pass(args.steps)
        gc.enable()
        passes.append((res, t_e2e, time.monotonic()))
    order = sorted(range(len(passes)), key=lambda i: passes[i][0][0])
    (ms_e2e, tev, e0, host_ms), t_e2e, t_e2e_end = passes[order[len(order) // 2]]
    e2e_clk = clocks.window(t_e2e, t_e2e_end)
    med = lambda v: sorted(v)[len(v) // 2]  # noqa: E731
    span = lambda a, b: [tev[a][i].elapsed_time(tev[b][i]) for i in range(args.steps)]  # noqa: E731
    comp_ms = span("c0", "c1")
    gaps = [tev["c1"][i - 1].elapsed_time(tev["c0"][i]) for i in range(1, args.steps)]
    e2e_timeline = {
        "compute_ms_median": med(comp_ms), "h2d_ms_median": med(span("i0", "i1")),
        "d2h_ms_median": med(span("o0", "o1")),
        # time per step not covered by compute: copies or waits on the compute stream
        "exposed_ms_per_step": (ms_e2e - sum(comp_ms)) / args.steps,
        "first_compute_start_ms": e0.elapsed_time(tev["c0"][0]),
        "gap_ms_max": max(gaps) if gaps else 0.0,
        "gap_ms_mean": sum(gaps) / len(gaps) if gaps else 0.0,
        "device_only_step_ms_median": per_step[len(per_step) // 2],
        "host_enqueue_ms_max": host_ms,
        "passes_ms": [round(p[0][0], 4) for p in passes],
    }
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
    flop_kinds = ("gemm_tc", "gemm_simt", "attn_fwd", "attn_bwd", "gemm_fp8")
    breakdown = {k: {"launches_per_step": r["launches"] // args.steps,
                     "ms_per_step": r["ms"] / args.steps, "share": r["ms"] / total_ms,
                     "tflops" if k in flop_kinds else "gbs":
                         r["work"] / (r["ms"] / 1e3) / (1e12 if k in flop_kinds else 1e9)}
                 for k, r in sorted(per_kind.items(), key=lambda kv: -kv[1]["ms"])}

    pk, pk_src = peaks()
    timed_s = ms / 1e3
    dom = max(per_kind.items(), key=lambda kv: kv[1]["ms"])[0] if per_kind else None
    roofline = None
    if dom is not None:
        r = per_kind[dom]
        if dom in ("gemm_tc", "gemm_simt", "attn_fwd", "attn_bwd", "gemm_fp8"):
            achieved = r["work"] / (r["ms"] / 1e3) / 1e12
            peak, peak_src = tensor_peak(pk, pk_src, timed_s, fp8=(dom == "gemm_fp8"))
            nominal = NOMINAL_TFLOPS["fp8" if dom == "gemm_fp8" else "bf16"]
            unit, bound = "TFLOP/s", "tensor"
        else:
            achieved = r["work"] / (r["ms"] / 1e3) / 1e9
            peak, peak_src, nominal = pk["hbm_gbs"], f"{pk_src} hbm", None
            unit, bound = "GB/s", "hbm"
        tr = traffic_record() if dom == "gemm_tc" else None
        traffic = None
        if tr and "dram_bytes_per_launch_full" in tr:
            traffic = float(tr["dram_bytes_per_launch_full"])
        roofline = {"bound": bound, "kernel": dom, "achieved": achieved, "peak": peak,
                    "unit": unit, "frac": achieved / peak, "traffic": traffic,
                    "peak_source": peak_src,
                    "sm_mhz": (clk or {}).get("sm_mhz")}
        if nominal:
            roofline["peak_nominal"] = nominal
            roofline["frac_nominal"] = achieved / nominal
    step_peak, step_peak_src = tensor_peak(pk, pk_src, timed_s)

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
                   "dropout": args.drop,
                   "gemm_precision": {None: "bf16", "fwd": "fp8 e4m3 forward, bf16 backward",
                                      "hybrid": "fp8 hybrid: e4m3 forward, e5m2 x e4m3 "
                                                "backward"}[args.fp8],
                   "layer": "post-ln" if args.post_ln else "pre-ln",
                   "recompute": bool(args.recompute),
                   "saved_bytes": saved.numel()},
        "pct_of_bf16_peak": 100.0 * value / world / step_peak,
        "pct_of_bf16_nominal": 100.0 * value / world / NOMINAL_TFLOPS["bf16"],
        "peak_source": step_peak_src,
        "gpu_launches": launches,
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": 2 * nbytes,
                "d2h_bytes_per_step": 2 * nbytes, "clocks": e2e_clk, "timeline": e2e_timeline},
        "roofline": roofline,
        "kernels": breakdown,
    }
    clocks.stop()
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
