"""Benchmark: µs per MoE layer and expert-weight GB/s at M=1 decode, on the
gpt-oss-20B-shaped routed-expert layer (H = I = 2880, 32 experts, top-4,
MXFP4 weights, bf16 activations), through the libmoe C ABI.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step = one whole decode layer (router top-k + softmax, gate_up dequant
GEMV, SwiGLU, down dequant GEMV, weighted combine into the residual) on fresh
synthetic inputs (x, residual and router logits ~N(0,1)).  Step s uses layer
s mod 24 of 24 resident layers (10.2 GB of distinct weights), so the 53 MB a
step reads is never L2-resident from a previous step (L2 is 129 MB).  The K
timed steps run as one moe_forward_steps call: one persistent launch in which
step s + 1 reads its routing and inputs only after step s's output is complete
(a grid barrier), as consecutive layers of a decode must.  The same K steps as
K separate launches (moe_forward, PDL-chained in one CUDA graph) are reported
next to it in extra.per_launch_graph.

The same JSON line carries an "extra" object with the other workloads, each
measured in the same run with its own clock record: the 24-layer MXFP4 stack
and the 48-layer int4 stack at M = 1 and 4 (tokens/s of the expert path, one
CUDA graph of the stack per step, fresh router logits every step), and the
batched M = 512 layer, uniform and skewed (µs, TFLOP/s, HBM fraction).
--no-extra leaves them out.

--impl reference times the fp64 CPU oracle on the host cores on the same
workload (a bounded sample: each step is one layer for one token).

Multi-GPU: the decode layer does not shard here (one GPU holds all experts);
N ranks run N independent replicas and the value is aggregated over them.
"""
from __future__ import annotations

import argparse
import hashlib
import re
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
KERNEL_SOURCES = ("bit_moe_decode_02_gb300/csrc/moe_decode_tc.cu", "bit_moe_decode_02_gb300/csrc/tc_ptx.cuh",
                  "bit_moe_decode_02_gb300/csrc/route.cuh")


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def _code_only(src: str) -> str:
    """The source without its comments and trailing blanks: the counters stay
    valid across comment edits, not across code changes."""
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    src = re.sub(r"//[^\n]*", "", src)
    return "\n".join(line.rstrip() for line in src.splitlines() if line.strip())


def kernel_hash() -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        h.update(_code_only(open(os.path.join(ROOT, f)).read()).encode())
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

def _setup(args):
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
    return rank, world


def _max_over_ranks(v, world):
    """The maximum of v over the ranks (the slowest rank's time)."""
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _load_all(moe, h, shape, L):
    for l in range(L):
        t = synth.layer_tensors(shape, l)
        moe.moe_load_experts(h, l, t.gu_codes, t.gu_scales, t.gu_bias, t.dn_codes, t.dn_scales,
                             t.dn_bias)
        del t


def run_ours(args):
    import torch
    rank, world = _setup(args)
    import bit_moe_decode_02_gb300 as moe

    shape = SHAPE
    L = args.layers or shape.layers
    H, E, k = shape.hidden, shape.experts, shape.top_k
    # max_tokens 16: the same resident layers also serve the stacks and the M
    # sweep of "extra" (M <= 4 on the decode kernel, 8 and 16 on the batched path)
    h = moe.moe_create(H, shape.intermediate, E, L, 16, k, moe.MOE_FMT_MXFP4, 32, 1)
    _load_all(moe, h, shape, L)
    W, K = args.warmup, args.steps
    n_in = W + K
    xs = np.empty((n_in, 1, H), np.uint16)
    rs = np.empty((n_in, 1, H), np.uint16)
    ls = np.empty((n_in, 1, E), np.float32)
    for s in range(n_in):
        x, r, lg = synth.step_inputs(shape, 1000 + s, M=1, layers=1)
        xs[s], rs[s], ls[s] = x, r, lg[0]
    xd = torch.from_numpy(xs.view(np.int16)).cuda()
    rd = torch.from_numpy(rs.view(np.int16)).cuda()
    ld = torch.from_numpy(ls).cuda()
    xp = [xd[s].data_ptr() for s in range(n_in)]
    lp = [ld[s].data_ptr() for s in range(n_in)]
    rp = [rd[s].data_ptr() for s in range(n_in)]

    stream = torch.cuda.current_stream()
    # warm-up steps, then the K timed steps: each a moe_forward_steps launch
    moe.moe_forward_steps(h, W, 0, xp[0], lp[0], 1, k, rp[0], stream)
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(torch.cuda.current_device()) as clk:
        ev0.record(stream)
        moe.moe_forward_steps(h, K, W % L, xp[W], lp[W], 1, k, rp[W], stream)
        ev1.record(stream)
        torch.cuda.synchronize()
    ms = _max_over_ranks(ev0.elapsed_time(ev1), world)
    launches = moe.moe_last_launches(h)
    assert moe.moe_get_status(h) == 0

    # the same steps as separate launches (one per layer call), captured into a
    # CUDA graph so that the timed region is the GPU's work, not the Python loop
    cap = torch.cuda.Stream()
    gw, gk = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    torch.cuda.synchronize()
    with torch.cuda.graph(gw, stream=cap):
        for s in range(W):
            moe.moe_forward(h, s % L, xp[s], lp[s], 1, k, rp[s], cap)
    with torch.cuda.graph(gk, stream=cap):
        for s in range(W, n_in):
            moe.moe_forward(h, s % L, xp[s], lp[s], 1, k, rp[s], cap)
    gw.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(torch.cuda.current_device()) as clk_g:
        e0.record(stream)
        gk.replay()
        e1.record(stream)
        torch.cuda.synchronize()
    ms_graph = _max_over_ranks(e0.elapsed_time(e1), world)
    assert moe.moe_get_status(h) == 0

    # the streaming floor of the same bytes: each resident layer's first
    # avg-bytes read with the decode kernels' copy engine and stage sizes and
    # nothing else, the layers one after another with a grid barrier between
    # them (moe_debug_stream_weights)
    fl_bytes = None

    bytes_per_step = []
    for s in range(W, min(n_in, W + 256)):
        moe.moe_forward(h, s % L, xp[s], lp[s], 1, k, rp[s], stream)
        bytes_per_step.append(moe.moe_last_bytes(h, stream))

    # end to end through the public API with host buffers: the same K steps with
    # their inputs and results in page-locked host memory, which the kernel reads
    # and writes over the host-device link step by step (every step's x, logits
    # and residual come in from the host, its result goes out to it); the host
    # clock runs from the call to the end of the stream synchronisation.
    xh = torch.from_numpy(xs.view(np.int16)).pin_memory()
    lh = torch.from_numpy(ls).pin_memory()
    oh = torch.from_numpy(rs.view(np.int16)).pin_memory()
    sp = stream.cuda_stream
    moe.moe_forward_steps(h, W, 0, xh[0].data_ptr(), lh[0].data_ptr(), 1, k, oh[0].data_ptr(), sp)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    moe.moe_forward_steps(h, K, W % L, xh[W].data_ptr(), lh[W].data_ptr(), 1, k, oh[W].data_ptr(), sp)
    stream.synchronize()
    e2e_s = _max_over_ranks(time.perf_counter() - t0, world)
    assert moe.moe_get_status(h) == 0
    # one moe_forward_host call per step instead (a host memcpy into the handle's
    # mapped staging, one launch and one synchronisation each)
    ohp = [oh[s].data_ptr() for s in range(n_in)]
    nh = min(K, 200)
    for s in range(W):
        moe.moe_forward_host(h, s % L, xh[s].data_ptr(), lh[s].data_ptr(), 1, k, ohp[s], sp)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for s in range(W, W + nh):
        moe.moe_forward_host(h, s % L, xh[s].data_ptr(), lh[s].data_ptr(), 1, k, ohp[s], sp)
    e2e_call_us = 1e6 * (time.perf_counter() - t0) / nh

    us_per_layer = 1e3 * ms / (K * world)
    avg_bytes = float(np.mean(bytes_per_step))
    fl_bytes = int(avg_bytes) // 16 * 16
    moe.moe_debug_stream_weights(h, 0, L, fl_bytes, stream)
    torch.cuda.synchronize()
    reps = 8
    ev0.record(stream)
    for _ in range(reps):
        moe.moe_debug_stream_weights(h, 0, L, fl_bytes, stream)
    ev1.record(stream)
    torch.cuda.synchronize()
    assert moe.moe_get_status(h) == 0
    floor_us = 1e3 * ev0.elapsed_time(ev1) / (reps * L)
    peak, peak_kind = measured_peaks()
    achieved = avg_bytes / (ms / 1e3 / K) / 1e9
    extra = None
    if not args.no_extra:
        extra = {"per_launch_graph": {
            "workload": WORKLOAD, "metric": METRIC, "value": 1e3 * ms_graph / (K * world), "unit": UNIT,
            "gbs": float(np.mean(bytes_per_step)) / (ms_graph / 1e3 / K) / 1e9,
            "launch": "the same K steps as K moe_forward launches (PDL-chained) in one CUDA graph",
            "gpu_launches": K, "clocks": clk_g.summary()},
            "stream_floor": {"us_per_layer": floor_us, "bytes_per_layer": fl_bytes,
                             "gbs": fl_bytes / floor_us / 1e3, "layer_over_floor": us_per_layer / floor_us,
                             "what": "the same bytes per layer read with the decode kernels' bulk copies "
                                     "(32 KB stages, 128 KB in flight per SM, one CTA per SM) and no compute, "
                                     f"{L} layers one after another with a grid barrier between them, "
                                     f"{reps} launches"},
            "e2e_per_call": {"value": e2e_call_us, "unit": UNIT, "calls": nh,
                             "api": "moe_forward_host per step (host memcpy into mapped staging, one launch, "
                                    "one stream synchronisation)"}}
        for M in (1, 4):
            extra[f"stack24_m{M}"] = measure_stack(moe, h, synth.GPTOSS_STACK, L, M, args.extra_steps, 8)
        for M in (1, 4):
            extra[f"stack24_steps_m{M}"] = measure_stack_steps(moe, h, synth.GPTOSS_STACK, L, M,
                                                               args.extra_steps, 4)
        for l in range(L):
            moe.moe_load_router(h, l, *synth.router_tensors(synth.GPTOSS_STACK, l))
        for M in (1, 4):
            extra[f"stack24_router_m{M}"] = measure_stack_steps(moe, h, synth.GPTOSS_STACK, L, M,
                                                                args.extra_steps, 4, router=True)
        extra["m_sweep"] = measure_m_sweep(moe, h, shape, L, max(args.extra_steps, 64))
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        n = oracle.max_threads()
        times = oracle_layer_seconds(args.cpu_steps, 1, n, budget_s=30.0)
        cpu = {"value": 1e6 * sum(times) / len(times), "unit": UNIT, "cores": n, "kind": "oracle",
               "sample": f"{len(times)} single-token layer forwards of this workload, fp64, "
                         f"OpenMP over output rows"}
    moe.moe_destroy(h)
    if extra is not None:
        extra.update(extra_workloads(moe, args))
    if rank != 0:
        return 0
    line = {
        "metric": METRIC, "value": us_per_layer, "unit": UNIT, "n_gpus": world,
        "steps": K, "warmup": W, "ms_per_step": ms / K,
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
        "dtype": "fp32 (MXFP4 weights, bf16 activations)", "data": "synthetic",
        "config": {"workload": WORKLOAD, "tokens_per_step": 1, "layers_resident": L,
                   "resident_bytes": L * E * shape.expert_bytes(),
                   "l2": f"inputs larger than L2: {L} distinct layers "
                         f"({L * E * shape.expert_bytes() / 1e9:.1f} GB), one per step",
                   "launch": "K steps in one persistent launch (moe_forward_steps); step s+1 reads its "
                             "routing and inputs after step s's output is complete",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "gbs": achieved,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_kind": peak_kind,
                     "kernel": "decode_tc_kernel (persistent, one CTA per SM, K layer calls per launch)",
                     "bytes_per_launch": avg_bytes, "traffic": stored_traffic()},
        "e2e": {"value": 1e6 * e2e_s / (K * world), "unit": UNIT,
                "h2d_bytes_per_step": H * 2 * 2 + E * 4, "d2h_bytes_per_step": H * 2,
                "api": "moe_forward_steps on page-locked host buffers (the kernel reads each step's "
                       "inputs and writes its result over the host-device link); host clock around the "
                       "call and the stream synchronisation"},
        "gpu_launches": launches,
        "clocks": clk.summary(),
        "cpu_baseline": cpu,
    }
    if extra is not None:
        line["extra"] = extra
    print(json.dumps(line), flush=True)
    return 0


def measure_stack_steps(moe, h, shape, L, M, steps, warmup, router=False):
    """Tokens/s of the expert stack with every step of the timed run in ONE
    launch (moe_forward_stack_steps: steps x L layer calls, each step on its own
    fresh residual and logits, each layer reading its logits only after the
    previous layer's output is complete).  With ``router`` the logits are not
    given: every layer computes them from its own input inside the launch."""
    import torch
    k = shape.top_k
    n = warmup + steps
    ins = [synth.step_inputs(shape, 6000 + s, M=M, layers=L) for s in range(n)]
    rd = torch.from_numpy(np.stack([r for _, r, _ in ins]).view(np.int16)).cuda()
    ld = torch.from_numpy(np.ascontiguousarray(np.stack([lg for _, _, lg in ins]))).cuda()
    stream = torch.cuda.current_stream()
    moe.moe_forward_stack_steps(h, warmup, rd[0], None if router else ld[0], M, k, stream)
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(torch.cuda.current_device()) as clk:
        ev0.record(stream)
        moe.moe_forward_stack_steps(h, steps, rd[warmup], None if router else ld[warmup], M, k, stream)
        ev1.record(stream)
        torch.cuda.synchronize()
    ms = ev0.elapsed_time(ev1)
    assert moe.moe_get_status(h) == 0
    launches = moe.moe_last_launches(h)
    nbytes = moe.moe_last_bytes(h, stream) / steps   # per step (the last step's layers)
    us = 1e3 * ms / steps
    peak, kind = measured_peaks()
    gbs = nbytes / (us / 1e6) / 1e9
    rt = ", router GEMV in the launch (logits from each layer's input)" if router else ""
    return {"workload": f"{shape.name}, M={M}, {steps} steps x {L} layers in one launch{rt}",
            "metric": "tokens/s of the expert stack", "value": M * 1e6 / us, "unit": "tok/s",
            "us_per_step": us, "us_per_layer": us / L, "steps": steps, "warmup": warmup,
            "bytes_per_step": nbytes, "gbs": gbs, "frac_of_peak": gbs / peak, "peak": peak, "peak_kind": kind,
            "clocks": clk.summary(), "gpu_launches": launches,
            "launch": "one persistent launch for all steps x layers (moe_forward_stack_steps)"}


def measure_m_sweep(moe, h, shape, L, steps):
    """Per-layer time and throughput of the gpt-oss layer against the number of
    tokens M: M <= 4 on the decode kernel (moe_forward_steps, one launch),
    M = 8 and 16 on the batched tensor-core path (moe_forward per step in a
    CUDA graph).  Step s runs resident layer s mod L (inputs larger than L2)."""
    import torch
    k, H, E = shape.top_k, shape.hidden, shape.experts
    stream = torch.cuda.current_stream()
    peak, kind = measured_peaks()
    out = {}
    for M in (1, 2, 3, 4, 8, 16):
        ins = [synth.step_inputs(shape, 8000 + 97 * M + s, M=M, layers=1) for s in range(steps)]
        xd = torch.from_numpy(np.stack([x for x, _, _ in ins]).view(np.int16)).cuda()
        rd = torch.from_numpy(np.stack([r for _, r, _ in ins]).view(np.int16)).cuda()
        ld = torch.from_numpy(np.ascontiguousarray(np.stack([lg[0] for _, _, lg in ins]))).cuda()
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if M <= 4:
            moe.moe_forward_steps(h, 8, 0, xd[0], ld[0], M, k, rd[0], stream)
            torch.cuda.synchronize()
            ev0.record(stream)
            moe.moe_forward_steps(h, steps, 0, xd[0], ld[0], M, k, rd[0], stream)
            ev1.record(stream)
            torch.cuda.synchronize()
            nbytes = moe.moe_last_bytes(h, stream) / steps
            path, launches = "decode kernel, one launch for all steps", 1
        else:
            cap = torch.cuda.Stream()
            g = torch.cuda.CUDAGraph()
            torch.cuda.synchronize()
            with torch.cuda.graph(g, stream=cap):
                for s in range(steps):
                    moe.moe_forward(h, s % L, xd[s], ld[s], M, k, rd[s], cap)
            launches = moe.moe_last_launches(h) * steps
            g.replay()
            torch.cuda.synchronize()
            ev0.record(stream)
            g.replay()
            ev1.record(stream)
            torch.cuda.synchronize()
            nb = []
            for s in range(min(steps, 16)):
                moe.moe_forward(h, s % L, xd[s], ld[s], M, k, rd[s], stream)
                nb.append(moe.moe_last_bytes(h, stream))
            nbytes = float(np.mean(nb))
            path = "batched tensor-core path, moe_forward per step in one CUDA graph"
        assert moe.moe_get_status(h) == 0
        us = 1e3 * ev0.elapsed_time(ev1) / steps
        gbs = nbytes / (us / 1e6) / 1e9
        out[f"m{M}"] = {"us_per_layer": us, "tok_per_s_per_layer": M * 1e6 / us, "bytes_per_layer": nbytes,
                        "gbs": gbs, "frac_of_peak": gbs / peak, "path": path, "steps": steps,
                        "gpu_launches": launches}
    out["peak"], out["peak_kind"] = peak, kind
    out["workload"] = f"{shape.name} layer, step s on resident layer s mod {L}"
    return out


def measure_stack(moe, h, shape, L, M, steps, warmup):
    """Tokens/s of the expert stack through moe_forward_stack on a loaded
    handle: every step copies fresh router logits [L][M][E] into the buffer the
    cached graph reads, then runs the L layers (each layer reads its logits only
    after the previous layer's output is complete)."""
    import torch
    k = shape.top_k
    logits = np.stack([synth.step_inputs(shape, 5000 + s, M=M, layers=L)[2] for s in range(warmup + steps)])
    _, r, _ = synth.step_inputs(shape, 4999, M=M, layers=L)
    ld = torch.from_numpy(logits).cuda()
    lbuf = torch.empty_like(ld[0])
    rd = torch.from_numpy(r.view(np.int16)).cuda()
    stream = torch.cuda.current_stream()

    def step(s):
        lbuf.copy_(ld[s], non_blocking=True)
        moe.moe_forward_stack(h, rd, lbuf, M, k, stream)

    for s in range(warmup):
        step(s)
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(torch.cuda.current_device()) as clk:
        ev0.record(stream)
        for s in range(warmup, warmup + steps):
            step(s)
        ev1.record(stream)
        torch.cuda.synchronize()
    ms = ev0.elapsed_time(ev1)
    assert moe.moe_get_status(h) == 0
    launches = moe.moe_last_launches(h)
    nbytes = []
    for s in range(warmup, warmup + min(steps, 16)):
        step(s)
        nbytes.append(moe.moe_last_bytes(h, stream))
    us_step = 1e3 * ms / steps
    peak, peak_kind = measured_peaks()
    gbs = float(np.mean(nbytes)) / (us_step / 1e6) / 1e9
    return {"workload": shape.name + f", M={M}, {L} layers", "metric": "tokens/s of the expert stack",
            "value": M * steps / (ms / 1e3), "unit": "tok/s", "us_per_step": us_step,
            "us_per_layer": us_step / L, "steps": steps, "warmup": warmup,
            "bytes_per_step": float(np.mean(nbytes)), "gbs": gbs, "frac_of_peak": gbs / peak, "peak": peak,
            "peak_kind": peak_kind, "clocks": clk.summary(), "gpu_launches_per_step": launches,
            "launch": f"one cached CUDA graph of {launches} PDL-chained layer kernels per step"}


def measure_batched(moe, shape, steps, warmup, bf16=False):
    """The batched MXFP4 layer (H = I = 2880, 128 experts, top-4, M = 512)
    through moe_forward's tensor-core path.  One layer is resident (1.7 GB of
    expert weights, 13x L2); P = 4 input sets are cycled, so a step's weights
    are never L2-resident from the previous step."""
    import torch
    H, I, E, k, M = shape.hidden, shape.intermediate, shape.experts, shape.top_k, shape.tokens
    h = moe.moe_create(H, I, E, 1, M, k, moe.MOE_FMT_MXFP4, 32, 1)
    if bf16:
        moe.moe_set_batched_numerics(h, moe.MOE_BATCHED_BF16)
    _load_all(moe, h, shape, 1)
    P = 4
    ins = [synth.step_inputs(shape, 7000 + i) for i in range(P)]
    xd = [torch.from_numpy(x.view(np.int16)).cuda() for x, _, _ in ins]
    rd = [torch.from_numpy(r.view(np.int16)).cuda() for _, r, _ in ins]
    ld = [torch.from_numpy(np.ascontiguousarray(lg[0])).cuda() for _, _, lg in ins]
    cap = torch.cuda.Stream()
    gw, gk = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    torch.cuda.synchronize()
    with torch.cuda.graph(gw, stream=cap):
        for s in range(warmup):
            moe.moe_forward(h, 0, xd[s % P], ld[s % P], M, k, rd[s % P], cap)
    with torch.cuda.graph(gk, stream=cap):
        for s in range(steps):
            moe.moe_forward(h, 0, xd[s % P], ld[s % P], M, k, rd[s % P], cap)
    launches = moe.moe_last_launches(h)
    stream = torch.cuda.current_stream()
    gw.replay()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(torch.cuda.current_device()) as clk:
        ev0.record(stream)
        gk.replay()
        ev1.record(stream)
        torch.cuda.synchronize()
    ms = ev0.elapsed_time(ev1)
    assert moe.moe_get_status(h) == 0
    nbytes = []
    for i in range(P):
        moe.moe_forward(h, 0, xd[i], ld[i], M, k, rd[i], stream)
        nbytes.append(moe.moe_last_bytes(h, stream))
    moe.moe_destroy(h)
    us = 1e3 * ms / steps
    flops = 2.0 * M * k * (2 * I * H + H * I)
    peak_hbm, kind = measured_peaks()
    # the tensor peak of the MMA kind the numerics issues: kind::f16 (bf16) or kind::mxf4
    tc_peak, tc_src = _bf16_peak() if bf16 else _fp4_peak()
    gbs = float(np.mean(nbytes)) / (us / 1e6) / 1e9
    tflops = flops / (us / 1e6) / 1e12
    numerics = ("bf16: tcgen05 kind::f16 on weights dequantised to bf16, x as given, h as bf16 hi + lo" if bf16
                else "MXFP4 activations: tcgen05 kind::mxf4")
    return {"workload": shape.name, "numerics": numerics,
            "metric": "us per batched MoE layer; TFLOP/s and expert-weight GB/s",
            "value": us, "unit": "us/layer", "steps": steps, "warmup": warmup, "tokens": M,
            "tflops": tflops, "tflops_peak": tc_peak, "tflops_peak_dtype": "bf16" if bf16 else "fp4",
            "tflops_peak_source": tc_src, "tflops_frac": tflops / tc_peak, "bytes_per_step": float(np.mean(nbytes)), "gbs": gbs,
            "hbm_frac": gbs / peak_hbm, "hbm_peak": peak_hbm, "peak_kind": kind,
            "gpu_launches_per_step": launches,
            "l2": "each step reads ~1.7 GB of expert weights (13x L2); 4 input sets cycled",
            "launch": f"K steps of {launches} kernels captured in one CUDA graph", "clocks": clk.summary()}


def extra_workloads(moe, args):
    """The int4 stack and the batched layer (the MXFP4 stack runs on the
    headline handle)."""
    out = {}
    shape = synth.INT4_STACK
    L = shape.layers
    h = moe.moe_create(shape.hidden, shape.intermediate, shape.experts, L, 4, shape.top_k, moe.MOE_FMT_INT4,
                       shape.group, 0)
    _load_all(moe, h, shape, L)
    for M in (1, 4):
        out[f"int4stack48_m{M}"] = measure_stack(moe, h, shape, L, M, args.extra_steps, 8)
    moe.moe_destroy(h)
    out["batched"] = measure_batched(moe, synth.BATCHED, max(args.extra_steps // 4, 8), 3)
    out["batched_skewed"] = measure_batched(moe, synth.BATCHED_SKEWED, max(args.extra_steps // 4, 8), 3)
    out["batched_bf16"] = measure_batched(moe, synth.BATCHED, max(args.extra_steps // 4, 8), 3, bf16=True)
    return out


def run_stack(args):
    """One stack workload alone (--workload stack24 / int4stack48)."""
    rank, world = _setup(args)
    import bit_moe_decode_02_gb300 as moe
    shape = synth.GPTOSS_STACK if args.workload == "stack24" else synth.INT4_STACK
    L = min(args.layers, shape.layers) if args.layers else shape.layers
    fmt = moe.MOE_FMT_MXFP4 if shape.fmt == synth.FMT_MXFP4 else moe.MOE_FMT_INT4
    h = moe.moe_create(shape.hidden, shape.intermediate, shape.experts, L, args.tokens, shape.top_k, fmt,
                       shape.group, 1 if shape.has_bias else 0)
    _load_all(moe, h, shape, L)
    line = measure_stack(moe, h, shape, L, args.tokens, args.steps, args.warmup)
    moe.moe_destroy(h)
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def run_batched(args):
    """One batched workload alone (--workload batched / batched_skewed)."""
    rank, world = _setup(args)
    import bit_moe_decode_02_gb300 as moe
    shape = synth.BATCHED_SKEWED if args.workload == "batched_skewed" else synth.BATCHED
    line = measure_batched(moe, shape, args.steps, args.warmup, bf16=args.workload == "batched_bf16")
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def _bf16_peak():
    """Dense bf16 tensor peak in TFLOP/s: the measured cuBLAS bf16 GEMM burst
    figure (MEASURED_PEAKS.json), else the 1.9 PFLOP/s fallback."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        return float(json.load(open(p))["bf16_tflops"]), "measured bf16 (MEASURED_PEAKS.json)"
    return 1900.0, "fallback bf16 1.9 PFLOP/s"


def _fp4_peak():
    """Dense FP4 tensor peak in TFLOP/s and where it comes from: the measured
    cuBLAS bf16 GEMM peak (MEASURED_PEAKS.json, burst) times the ratio of
    NVIDIA's nominal dense GB300 rates, 13.5 PFLOP/s FP4 to 2.25 PFLOP/s bf16
    (the figures without 2:4 sparsity); 1.9 PFLOP/s bf16 if no measurement."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        bf16, src = json.load(open(p))["bf16_tflops"], "measured bf16 (MEASURED_PEAKS.json) x 13.5/2.25"
    else:
        bf16, src = 1900.0, "fallback bf16 1.9 PFLOP/s x 13.5/2.25"
    return bf16 * 13.5 / 2.25, src


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=40000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--layers", type=int, default=None,
                    help="resident layers (default: 24 for the layer workload, all for the "
                         "stacks; smaller for profiling)")
    ap.add_argument("--workload", choices=["layer", "stack24", "int4stack48", "batched", "batched_skewed",
                                           "batched_bf16"],
                    default="layer")
    ap.add_argument("--tokens", type=int, default=1, help="M for the stack workloads")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-steps", type=int, default=24)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true", help="headline workload only")
    ap.add_argument("--extra-steps", type=int, default=128,
                    help="timed steps of the stack workloads in extra (batched: a quarter)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    if args.workload.startswith("batched"):
        return run_batched(args)
    if args.workload != "layer":
        return run_stack(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
