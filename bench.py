"""Benchmark: µs per MoE layer and expert-weight GB/s at M=1 decode, on the
gpt-oss-20B-shaped routed-expert layer (H = I = 2880, 32 experts, top-4,
MXFP4 weights, bf16 activations), through the libmoe C ABI.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step = one whole decode layer (router top-k + softmax, gate_up dequant
GEMV, SwiGLU, down dequant GEMV, weighted combine into the residual) on fresh
synthetic inputs (x, residual and router logits ~N(0,1)).  Step s uses layer
s mod 24 of 24 resident layers (10.2 GB of distinct weights), so the 53 MB a
step reads is never L2-resident from a previous step (L2 is 129 MB).

--impl reference times the fp64 CPU oracle on the host cores on the same
workload (a bounded sample: each step is one layer for one token).

Multi-GPU: the decode layer does not shard here (one GPU holds all experts);
N ranks run N independent replicas and the value is aggregated over them.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from bit_moe_decode_02_gb300 import synth  # noqa: E402

METRIC = "µs per MoE layer & expert-weight GB/s vs GB300 HBM peak at M=1 decode"
UNIT = "us/layer"
SHAPE = synth.GPTOSS_STACK          # 24 distinct gpt-oss-20B-shaped layers
WORKLOAD = ("gpt-oss-20B-shaped MXFP4 MoE layer decode, H=I=2880, E=32, top-4, M=1; "
            "step s runs layer s mod 24 of 24 resident layers")
KERNEL_SOURCES = ("bit_moe_decode_02_gb300/csrc/moe_decode.cu",)


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def kernel_hash() -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        h.update(open(os.path.join(ROOT, f), "rb").read())
    return h.hexdigest()[:16]


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def stored_traffic():
    """Per-forward DRAM bytes from the committed ncu summary, if it was taken
    on the current kernel source; else None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    if d.get("kernel_hash") != kernel_hash():
        return None
    return d.get("dram_bytes_per_forward")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None
        time.sleep(0.25)
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- CPU oracle

def oracle_layer_seconds(steps: int, warmup: int, nthreads: int, budget_s: float = 60.0):
    """Time the fp64 oracle on up to `steps` single-token layer forwards,
    stopping early once `budget_s` seconds of timed work are done."""
    import oracle
    shape = SHAPE
    times = []
    for s in range(warmup + steps):
        if sum(times) > budget_s:
            break
        layer = s % shape.layers
        x, r, logits = synth.step_inputs(shape, s, M=1, layers=1)
        idx, _ = oracle.route(logits[0], shape.top_k)
        t = synth.layer_tensors(shape, layer, idx.ravel())
        t0 = time.perf_counter()
        oracle.layer(shape.fmt, shape.hidden, shape.intermediate, shape.experts, shape.top_k, t,
                     x, logits[0], r, group=shape.group, nthreads=nthreads)
        dt = time.perf_counter() - t0
        if s >= warmup:
            times.append(dt)
    return times


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    n = oracle.max_threads()
    times = oracle_layer_seconds(max(1, args.steps), min(args.warmup, 3), n, budget_s=90.0)
    steps = len(times)
    us = 1e6 * sum(times) / len(times)
    line = {
        "impl": "reference", "metric": METRIC, "value": us, "unit": UNIT,
        "n_gpus": args.gpus, "steps": steps, "warmup": args.warmup,
        "ms_per_step": us / 1e3, "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "tokens_per_step": 1,
                   "l2": "not applicable (CPU)"},
        "cpu_baseline": {"value": us, "unit": UNIT, "cores": n, "kind": "oracle",
                         "sample": f"{steps} of the {args.steps} requested single-token layer "
                                   f"forwards (stops after 90 s of timed work), fp64, OpenMP "
                                   f"over output rows"},
        "e2e": {"value": us, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- GPU arm

def run_ours(args):
    import torch
    import torch.distributed as dist
    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    from bit_moe_decode_02_gb300 import build_ext
    if rank == 0 or not os.path.exists(build_ext.LIB):
        build_ext.build()
    if world > 1:
        dist.barrier()
    import bit_moe_decode_02_gb300 as moe

    shape = SHAPE
    L = shape.layers
    H, E, k = shape.hidden, shape.experts, shape.top_k
    h = moe.moe_create(H, shape.intermediate, E, L, 1, k, moe.MOE_FMT_MXFP4, 32, 1)
    for l in range(L):
        t = synth.layer_tensors(shape, l)
        moe.moe_load_experts(h, l, t.gu_codes, t.gu_scales, t.gu_bias, t.dn_codes, t.dn_scales,
                             t.dn_bias)
        del t
    n_in = args.warmup + args.steps
    xs, rs, ls = [], [], []
    for s in range(n_in):
        x, r, lg = synth.step_inputs(shape, 1000 + s, M=1, layers=1)
        xs.append(x)
        rs.append(r)
        ls.append(lg[0])
    xd = torch.from_numpy(np.stack(xs).view(np.int16)).cuda()
    rd0 = torch.from_numpy(np.stack(rs).view(np.int16)).cuda()
    ld = torch.from_numpy(np.stack(ls)).cuda()
    rd = rd0.clone()
    stream = torch.cuda.current_stream()

    def step(s):
        moe.moe_forward(h, s % L, xd[s], ld[s], 1, k, rd[s], stream)

    for s in range(args.warmup):
        step(s)
    torch.cuda.synchronize()
    # algorithmic bytes: distinct selected experts of each timed step
    bytes_per_step = []
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(torch.cuda.current_device()) as clk:
        ev0.record(stream)
        for s in range(args.warmup, n_in):
            step(s)
        ev1.record(stream)
        torch.cuda.synchronize()
    ms = ev0.elapsed_time(ev1)
    launches = 2 * args.steps
    for s in range(args.warmup, n_in):
        step(s)
        bytes_per_step.append(moe.moe_last_bytes(h, stream))
    if world > 1:
        t = torch.tensor([ms], device="cuda")
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())

    # end to end through the public API with host buffers (pinned)
    xh = torch.from_numpy(np.stack(xs).view(np.int16)).pin_memory()
    lh = torch.from_numpy(np.stack(ls)).pin_memory()
    oh = torch.from_numpy(np.stack(rs).view(np.int16)).pin_memory()
    for s in range(args.warmup):
        moe.moe_forward_host(h, s % L, xh[s], lh[s], 1, k, oh[s], stream)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for s in range(args.warmup, n_in):
        moe.moe_forward_host(h, s % L, xh[s], lh[s], 1, k, oh[s], stream)
    e2e_s = time.perf_counter() - t0
    if world > 1:
        t = torch.tensor([e2e_s], device="cuda")
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        e2e_s = float(t.item())

    us_per_layer = 1e3 * ms / (args.steps * world)
    avg_bytes = float(np.mean(bytes_per_step))
    peak, peak_kind = measured_peaks()
    fwd_s = ms / 1e3 / args.steps
    achieved = avg_bytes / fwd_s / 1e9
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        n = oracle.max_threads()
        times = oracle_layer_seconds(args.cpu_steps, 1, n)
        cpu = {"value": 1e6 * sum(times) / len(times), "unit": UNIT, "cores": n, "kind": "oracle",
               "sample": f"{len(times)} single-token layer forwards of this workload, fp64, "
                         f"OpenMP over output rows"}
    moe.moe_destroy(h)
    if rank != 0:
        return 0
    clocks = clk.summary()
    line = {
        "metric": METRIC, "value": us_per_layer, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms / args.steps,
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
        "dtype": "fp32 (MXFP4 weights, bf16 activations)", "data": "synthetic",
        "config": {"workload": WORKLOAD, "tokens_per_step": 1, "layers_resident": L,
                   "resident_bytes": L * E * shape.expert_bytes(),
                   "l2": "inputs larger than L2: 24 distinct layers (10.2 GB), one per step",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "gbs": achieved,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_kind": peak_kind,
                     "kernel": "moe_forward: gate_up_kernel + down_kernel (PDL-chained)",
                     "bytes_per_launch": avg_bytes, "traffic": stored_traffic()},
        "e2e": {"value": 1e6 * e2e_s / (args.steps * world), "unit": UNIT,
                "h2d_bytes_per_step": H * 2 * 2 + E * 4, "d2h_bytes_per_step": H * 2},
        "gpu_launches": launches,
        "clocks": clocks,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-steps", type=int, default=24)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
