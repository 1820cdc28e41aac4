#!/usr/bin/env python
"""Benchmark of the fused int8 Conv2D forward pass on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl fconv|reference]

Prints ONE JSON line (rank 0).  A step is one fconv_run of the whole fused
path (one launch that packs the filter and widens the int8 input to fp16,
then the implicit-GEMM convolution with the fused epilogue) over one batch
of the workload: N=256 28x28x512
int8, 3x3 stride 1 SAME, side input, ReLU (implicit GEMM 200704 x 512 x
4608).  ``value`` is TOPS counted the usual way (2*M*N*K, padded taps
included) over all ranks; the roofline block reports the convolution
kernel alone against its own tensor-core peak.

Under torchrun every rank runs its own plan on its own GPU with no exchange
on the data path.  By default each rank convolves the whole batch (weak
scaling); ``--strong`` splits the batch's images over the ranks
(``shard_range``), each rank convolving its slice of x and side into its
slice of y.

``--impl reference`` times the CPU oracle (the reference this build is
checked against) on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import signal
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import fconv_inputs as FI  # noqa: E402

METRIC = "fused int8 Conv2D TOPS (1 GB300) and % of dense int8 tensor peak"
UNIT = "TOPS"
DEFAULT_WORKLOAD = "large_i8_28x28x512"
L2_BYTES = 129 * 1024 * 1024
# dense 16-bit (kind::f16) tensor-core flops per SM per cycle
TENSOR_FLOPS_PER_CYCLE_PER_SM = 8192
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "traffic.json")
KERNEL_SOURCES = [os.path.join(ROOT, "quantized_conv2d_gb300", "csrc", f)
                  for f in ("fconv_kernels.cu", "fconv_device.cuh", "fconv_internal.h")]


# ---------------------------------------------------------------- geometry
def axis(in_, filt, stride, padding):
    if padding == "VALID":
        out = (in_ - filt) // stride + 1
        return out, 0
    out = -(-in_ // stride)
    total = max(0, (out - 1) * stride + filt - in_)
    return out, total // 2


def ops_counts(wl):
    """(nominal ops 2*M*N*K with padded taps, ops over in-bounds taps only).
    Transposed convolutions: nominal = 2 * every input pixel x tap x channel
    pair of the scatter; in-bounds = those whose target is in the output."""
    if wl.transposed_pads is not None:
        pt, pb, pl, pr = wl.transposed_pads
        P = (wl.H - 1) * wl.stride + wl.R - pt - pb
        Q = (wl.W - 1) * wl.stride + wl.S - pl - pr
        nominal = 2 * wl.N * wl.H * wl.W * wl.C * wl.K * wl.R * wl.S
        rows = sum(1 for p in range(wl.H) for r in range(wl.R) if 0 <= p * wl.stride + r - pt < P)
        cols = sum(1 for q in range(wl.W) for s in range(wl.S) if 0 <= q * wl.stride + s - pl < Q)
        return nominal, 2 * wl.N * wl.C * wl.K * rows * cols, P, Q
    P, pt = axis(wl.H, wl.R, wl.stride, wl.padding)
    Q, pl = axis(wl.W, wl.S, wl.stride, wl.padding)
    nominal = 2 * wl.N * P * Q * wl.K * wl.R * wl.S * wl.C
    rows = sum(sum(1 for r in range(wl.R) if 0 <= p * wl.stride + r - pt < wl.H) for p in range(P))
    cols = sum(sum(1 for s in range(wl.S) if 0 <= q * wl.stride + s - pl < wl.W) for q in range(Q))
    inbounds = 2 * wl.N * wl.K * wl.C * rows * cols
    return nominal, inbounds, P, Q


def algorithmic_bytes(wl):
    """HBM bytes one step must move at least: x read once (for a 1x1 filter
    at a stride above 1, only the pixels the convolution reads), the filter,
    the side input, the output written once, and the bias."""
    elt = 1 if wl.dtype == "int8" else 2
    _, _, P, Q = ops_counts(wl)
    if wl.transposed_pads is None and wl.R == 1 and wl.S == 1 and wl.stride > 1:
        x = wl.N * P * Q * wl.C * elt
    else:
        x = wl.N * wl.H * wl.W * wl.C * elt
    w = wl.R * wl.S * wl.C * wl.K * elt
    y = wl.N * P * Q * wl.K * elt
    side = y if wl.has_side else 0
    return x + w + side + y + 4 * wl.K


def kernel_hash() -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            d = json.load(fh)
        return d.get("bf16_tflops"), d.get("bf16_tflops_sustained"), d.get("hbm_gbs"), "measured"
    except (OSError, ValueError):
        return 1900.0, 1700.0, 6800.0, "fallback"


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi sampled every 100 ms while the timed region runs."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.send_signal(signal.SIGTERM)
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.close()
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as fh:
            for line in fh:
                f = [v.strip() for v in line.split(",")]
                if len(f) < 9:
                    continue
                try:
                    sm.append(float(f[1]))
                    smax = float(f[2])
                except ValueError:
                    continue
                for name, v in zip(names, f[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(name)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": smax, "reasons": sorted(reasons), "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- ranks
def reduce_max(value: float, device=None) -> float:
    """Maximum of a per-rank number over all ranks (the value itself when no
    process group is running).  Works with any torch.distributed backend."""
    import torch
    import torch.distributed as tdist
    if not (tdist.is_available() and tdist.is_initialized()) or tdist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    tdist.all_reduce(t, op=tdist.ReduceOp.MAX)
    return float(t.item())


def barrier():
    import torch.distributed as tdist
    if tdist.is_available() and tdist.is_initialized() and tdist.get_world_size() > 1:
        tdist.barrier()


def weak_scaling_tops(world: int, steps: int, ops_per_step: float, max_ms: float) -> float:
    """Whole-job throughput: every rank runs `steps` steps of its own batch;
    the job takes as long as the slowest rank."""
    return world * steps * ops_per_step / (max_ms / 1e3) / 1e12


def job_tops(steps: int, job_ops_per_step: float, max_ms: float) -> float:
    """Whole-job throughput: the operations of `steps` steps of all ranks
    together, over the slowest rank's time."""
    return steps * job_ops_per_step / (max_ms / 1e3) / 1e12


def shard_range(n: int, world: int, rank: int) -> tuple[int, int]:
    """The images [lo, hi) of a batch of n that rank `rank` of `world`
    convolves when the batch is split over the ranks (images are
    independent, so the shards need no exchange): lo = floor(rank*n/world),
    hi = floor((rank+1)*n/world).  Consecutive ranks get consecutive,
    disjoint ranges covering the batch; sizes differ by at most one."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError(f"rank {rank} of {world}")
    if n < world:
        raise ValueError(f"a batch of {n} images cannot give {world} ranks one image each")
    return rank * n // world, (rank + 1) * n // world


# ---------------------------------------------------------------- CPU oracle timing
class OracleSample:
    """The CPU oracle on a bounded sample of a workload: whole images, all
    channels, full epilogue.  Inputs are drawn once per sample size (their
    generation is not timed)."""

    def __init__(self, wl, P, Q):
        import oracle
        oracle.build()
        self.oracle, self.wl, self.P, self.Q = oracle, wl, P, Q
        self.pad = oracle.SAME if wl.padding == "SAME" else oracle.VALID
        self.inputs = {}

    def run(self, n):
        """Seconds for one oracle pass over n images."""
        orc, wl = self.oracle, self.wl
        if n not in self.inputs:
            self.inputs = {n: FI.generate(wl, (self.P, self.Q), batch=n)}
        inp = self.inputs[n]
        t0 = time.perf_counter()
        if wl.transposed_pads is not None:
            acc = (orc.convT_acc_i8 if wl.dtype == "int8" else orc.convT_acc_bf16_f64)(
                inp["x"], inp["w"], wl.stride, wl.transposed_pads)
        elif wl.dtype == "int8":
            acc = orc.conv_acc_i8(inp["x"], inp["w"], wl.stride, self.pad)
        else:
            acc = orc.conv_acc_bf16_f64(inp["x"], inp["w"], wl.stride, self.pad)
        if wl.dtype == "int8":
            orc.epilogue_i8(acc, inp["bias"], inp["side"], wl.conv_scale, wl.side_scale, wl.relu)
        else:
            orc.epilogue_f64(acc, inp["bias"], inp["side"], wl.conv_scale, wl.side_scale, wl.relu)
        return time.perf_counter() - t0

    def images_for(self, target_s: float) -> int:
        """Whole images whose oracle pass takes about target_s (at least 1)."""
        t1 = self.run(1)
        return int(max(1, min(self.wl.N, target_s / max(t1, 1e-6))))

    def tops(self, n: int, seconds: float) -> float:
        return ops_counts(self.wl)[0] / self.wl.N * n / seconds / 1e12

    def threads(self) -> int:
        return self.oracle.num_threads()


def time_oracle(wl, P, Q, target_s: float, max_images: int):
    """Time the CPU oracle on a bounded sample (whole images of the workload,
    all channels, full epilogue).  Returns (TOPS nominal, images, seconds, threads)."""
    sample = OracleSample(wl, P, Q)
    n = min(max_images, sample.images_for(target_s))
    t = sample.run(n)
    return sample.tops(n, t), n, t, sample.threads()


# ---------------------------------------------------------------- arms
def run_reference(args, rank, world):
    if rank != 0:
        return
    wl = FI.workload(args.workload)
    _, _, P, Q = ops_counts(wl)
    # each step one oracle pass over the same bounded sample, sized so that
    # all steps together take about 150 s
    step_target = min(2.0, 150.0 / max(1, args.steps + args.warmup))
    sample = OracleSample(wl, P, Q)
    n_img = sample.images_for(step_target)
    threads = sample.threads()
    values, secs = [], []
    for i in range(args.warmup + args.steps):
        t = sample.run(n_img)
        if i >= args.warmup:
            values.append(sample.tops(n_img, t))
            secs.append(t)
    value = statistics.median(values)
    sample = f"{n_img} of {wl.N} images per step (all {wl.K} channels, full epilogue)"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * statistics.median(secs), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": wl.dtype, "data": "synthetic (seeded)", "config": config_of(wl),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def config_of(wl):
    cfg = {"workload": f"{wl.name}: {wl.note}", "N": wl.N, "H": wl.H, "W": wl.W, "C": wl.C,
           "K": wl.K, "R": wl.R, "S": wl.S, "stride": wl.stride, "padding": wl.padding,
           "dtype": wl.dtype, "side_input": wl.has_side, "relu": wl.relu}
    if wl.transposed_pads is not None:
        cfg["transposed"] = True
        cfg["padding"] = "explicit (top, bottom, left, right) = " + str(tuple(wl.transposed_pads))
    return cfg


# epilogue variants: (activation code or None for the workload's own, alpha, beta,
# per-channel conv scale)
VARIANTS = {
    "plain": (None, 0.0, 0.0, False),
    "channel_scale": (None, 0.0, 0.0, True),
    "leaky_relu": (2, 0.1, 0.0, False),
    "clipped_relu": (3, 6.0, 0.0, False),
    "clamp": (4, -20.0, 20.0, False),
}


def run_fconv(args, rank, world, local_rank):
    import torch
    import quantized_conv2d_gb300 as fc

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    wl = FI.workload(args.workload)
    if args.batch:
        # a smaller batch of the same layer (profiling captures of a size a
        # profiler replays quickly; not a benchmark configuration)
        import dataclasses
        wl = dataclasses.replace(wl, N=args.batch, note=wl.note + f" (batch {args.batch})")
    nominal, inbounds, P, Q = ops_counts(wl)
    # weak scaling: every rank convolves the whole batch; strong: the batch
    # is split over the ranks (shard_range) and each convolves its images
    lo, hi = shard_range(wl.N, world, rank) if args.strong else (0, wl.N)
    n_local = hi - lo
    inbounds_local = inbounds * n_local // wl.N
    abytes = algorithmic_bytes(wl) * n_local // wl.N   # this rank's share
    hbm_peak = measured_peaks()[2]
    job_ops_per_step = nominal if args.strong else world * nominal
    act, alpha, beta, per_channel = VARIANTS[args.variant]
    plan = fc.Conv2dPlan(n_local, wl.H, wl.W, wl.C, wl.K, wl.R, wl.S, wl.stride, wl.padding,
                         wl.dtype, wl.relu if act is None else act, device=dev, alpha=alpha,
                         beta=beta, transposed_pads=wl.transposed_pads)
    if args.gather:
        fc.fconv_plan_set_gather(plan.handle, {"auto": fc.FCONV_GATHER_AUTO,
                                               "im2col": fc.FCONV_GATHER_IM2COL,
                                               "halo": fc.FCONV_GATHER_HALO}[args.gather])
    if args.tile:
        plan.set_tile(args.tile)
    if args.tile_shape:
        px, ch = (int(v) for v in args.tile_shape.split(","))
        fc.fconv_plan_set_tile_shape(plan.handle, px, ch)
    if args.splits:
        fc.fconv_plan_set_splits(plan.handle, args.splits)
    if args.widen:
        fc.fconv_plan_set_input_widening(plan.handle, args.widen)
    assert plan.out_shape == (n_local, P, Q, wl.K)
    inp = FI.generate(wl, (P, Q))
    if n_local != wl.N:
        for key in ("x", "side"):
            if inp[key] is not None:
                inp[key] = np.ascontiguousarray(inp[key][lo:hi])

    def to_dev(a):
        if a is None:
            return None
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)
        return torch.from_numpy(a).to(dev)

    x, w, bias, side = to_dev(inp["x"]), to_dev(inp["w"]), to_dev(inp["bias"]), to_dev(inp["side"])
    y = plan.new_output()
    stream = torch.cuda.current_stream(dev)
    # a per-channel scale spreads the workload's scalar over [0.5, 1.5] x
    cs = wl.conv_scale
    if per_channel:
        cs = torch.linspace(0.5 * wl.conv_scale, 1.5 * wl.conv_scale, wl.K,
                            dtype=torch.float32, device=dev)

    def step(st=None):
        plan.run(x, w, bias, side, cs, wl.side_scale, y=y, stream=stream if st is None else st)

    for _ in range(args.warmup):
        step()
    plan.check()

    # stage events: [before pack, after pack, after widen, after conv] per step
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    for row in evs:
        for e in row:
            e.record(stream)
    torch.cuda.synchronize(dev)

    clocks = ClockSampler(local_rank)
    barrier()
    torch.cuda.synchronize(dev)
    clocks.start()
    time.sleep(0.25)   # let the sampler start before the timed region
    # inputs smaller than L2: flush it before every timed step (a 256 MB
    # write), outside the step's own events, and time the steps by those
    footprint = sum(t.numel() * t.element_size() for t in (x, w, side, y) if t is not None) \
        + plan.ws_bytes
    flush = None if footprint > L2_BYTES else torch.empty(2 * L2_BYTES, dtype=torch.uint8,
                                                          device=dev)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(args.steps):
        if flush is not None:
            flush.zero_()
        fc.fconv_plan_set_stage_events(plan.handle, [e.cuda_event for e in evs[i]])
        step()
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    clk = clocks.stop()
    fc.fconv_plan_set_stage_events(plan.handle, None)
    plan.check()
    total_ms = t_start.elapsed_time(t_end)
    if flush is not None:
        total_ms = sum(evs[i][0].elapsed_time(evs[i][3]) for i in range(args.steps))
    conv_ms = [evs[i][2].elapsed_time(evs[i][3]) for i in range(args.steps)]
    prep_ms = [evs[i][0].elapsed_time(evs[i][1]) for i in range(args.steps)]
    total_ms = reduce_max(total_ms, dev)
    ms_per_step = total_ms / args.steps
    value = job_tops(args.steps, job_ops_per_step, total_ms)

    # ------------------------------------------------ the same steps from a CUDA graph
    # (GPU time without the host's launch gaps, which small workloads feel;
    # L2 flushed by a memset node before each step when the tensors fit in it)
    graph = None
    if args.graph:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            if flush is not None:
                flush.zero_()
            step(torch.cuda.current_stream(dev))   # the capture stream
        g.replay()
        torch.cuda.synchronize(dev)
        flush_ms = 0.0
        if flush is not None:
            gf = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gf):
                flush.zero_()
            f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            f0.record(stream)
            for _ in range(args.steps):
                gf.replay()
            f1.record(stream)
            torch.cuda.synchronize(dev)
            flush_ms = f0.elapsed_time(f1)
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier()
        g0.record(stream)
        for _ in range(args.steps):
            g.replay()
        g1.record(stream)
        torch.cuda.synchronize(dev)
        plan.check()
        graph_ms = reduce_max(max(g0.elapsed_time(g1) - flush_ms, 1e-6), dev)
        graph = {"value": job_tops(args.steps, job_ops_per_step, graph_ms), "unit": UNIT,
                 "ms_per_step": graph_ms / args.steps,
                 "step_hbm_frac": abytes / (graph_ms / args.steps / 1e3) / 1e9 / hbm_peak,
                 "how": "one step captured in a CUDA graph, replayed steps times"
                        + (" after an L2-flush node, flush time subtracted" if flush is not None
                           else "")}
        if flush is not None:
            # the same steps without the flush, inputs left in L2 by the step
            # before; 20 steps a graph so that the host's replay calls do not
            # pace the GPU
            per = 20
            gw = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gw):
                for _ in range(per):
                    step(torch.cuda.current_stream(dev))
            gw.replay()
            torch.cuda.synchronize(dev)
            reps = max(1, args.steps // per)
            w0, w1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            barrier()
            w0.record(stream)
            for _ in range(reps):
                gw.replay()
            w1.record(stream)
            torch.cuda.synchronize(dev)
            plan.check()
            warm_ms = reduce_max(w0.elapsed_time(w1), dev)
            graph["warm_l2"] = {"value": job_tops(reps * per, job_ops_per_step, warm_ms),
                                "ms_per_step": warm_ms / (reps * per),
                                "step_hbm_frac": abytes / (warm_ms / (reps * per) / 1e3) / 1e9
                                                 / hbm_peak,
                                "how": f"{per} steps a graph, replayed {reps} times"}

    # ------------------------------------------------ end to end, host buffers
    e2e = None
    if not args.no_e2e and not per_channel:   # the host-buffer entry takes a scalar scale
        nbytes = fc.fconv_host_workspace_size(plan.handle, side is not None)
        dws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        def pinned(a):
            if a is None:
                return None
            return torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).pin_memory()

        hx, hw, hb, hs = pinned(inp["x"]), pinned(inp["w"]), pinned(inp["bias"]), pinned(inp["side"])
        hy = torch.empty(plan.out_shape, dtype=plan.torch_dtype).pin_memory()
        h2d = sum(t.numel() * t.element_size() for t in (hx, hw, hb, hs) if t is not None)
        d2h = hy.numel() * hy.element_size()

        def host_step():
            fc.fconv_run_host(plan.handle, hx.data_ptr(), hw.data_ptr(), hb.data_ptr(),
                              hs.data_ptr() if hs is not None else None, wl.conv_scale,
                              wl.side_scale, hy.data_ptr(), dws.data_ptr(), nbytes,
                              stream.cuda_stream)
            stream.synchronize()

        for _ in range(3):
            host_step()
        n_e2e = max(3, min(args.steps, 50))
        barrier()
        t0 = time.perf_counter()
        for _ in range(n_e2e):
            host_step()
        el = reduce_max(time.perf_counter() - t0, dev)
        plan.check()
        e2e = {"value": job_tops(n_e2e, job_ops_per_step, el * 1e3), "unit": UNIT,
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "steps": n_e2e}
        del dws

    # ------------------------------------------------ roofline of the conv kernel
    burst, sustained, hbm, src = measured_peaks()
    long_run = total_ms > 1000.0
    peak = sustained if long_run else burst
    conv_avg_s = statistics.mean(conv_ms) / 1e3
    achieved = inbounds_local / conv_avg_s / 1e12
    traffic = None
    try:
        with open(PROFILE_TRAFFIC) as fh:
            tr = json.load(fh)
        rec = tr.get(args.workload)
        if rec and rec.get("kernel_hash") == kernel_hash() and rec.get("block_n") == plan.config()[0]:
            traffic = rec["dram_bytes_per_launch"]
    except (OSError, ValueError):
        pass
    # the same launch in SM cycles at the clock sampled during the timed
    # steps, against the tensor pipe's dense 16-bit rate of 8192 flops per
    # cycle per SM: a fraction that does not move with the clock the power
    # cap allows
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    mhz = clk.get("sm_mhz") if clk else None
    cycles = conv_avg_s * mhz * 1e6 if mhz else None
    ideal_cycles = inbounds_local / (TENSOR_FLOPS_PER_CYCLE_PER_SM * sms)
    # HBM side: the path's algorithmic bytes over the conv kernel, and over
    # the whole step; the bound is whichever ideal time (flops at the
    # tensor peak, bytes at the copy bandwidth) is the longer
    hbm_achieved = abytes / conv_avg_s / 1e9
    hbm_bound = abytes / (hbm * 1e9) > inbounds_local / (peak * 1e12)
    kernel_form = fc.fconv_plan_kernel(plan.handle)
    kernel_fn = ("conv_fprop_cpasync_kernel" if kernel_form.startswith("cp-async")
                 else "conv_fprop_tma_kernel")
    roofline = {"bound": "hbm" if hbm_bound else "tensor",
                "achieved": hbm_achieved if hbm_bound else achieved,
                "peak": hbm if hbm_bound else peak,
                "unit": "GB/s" if hbm_bound else "TFLOP/s",
                "frac": hbm_achieved / hbm if hbm_bound else achieved / peak,
                "traffic": traffic,
                "tensor_tflops": achieved, "tensor_frac": achieved / peak,
                "frac_burst": achieved / burst, "frac_sustained": achieved / sustained,
                "hbm_gbs": hbm_achieved, "hbm_frac": hbm_achieved / hbm,
                "algorithmic_bytes_per_launch": abytes,
                "step_hbm_frac": abytes / (ms_per_step / 1e3) / 1e9 / hbm,
                "sm_mhz": mhz, "cycles_per_launch": cycles,
                "ideal_tensor_cycles": ideal_cycles,
                "tensor_cycle_frac": ideal_cycles / cycles if cycles else None,
                "kernel": (f"{kernel_fn}<{plan.config()[0]}, {wl.dtype}> "
                           f"({kernel_form}, tcgen05.mma kind::f16)"),
                "peak_source": (f"copy bandwidth of {src}" if hbm_bound else
                                f"{'sustained' if long_run else 'burst'} bf16 dense of {src} "
                                f"(fp16 rate = bf16 rate; no int8 tensor-core MMA on sm_103a)"),
                "ops_per_launch": inbounds_local, "ops_definition": "2*MAC over in-bounds taps"}

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "strong" if args.strong else "weak", "vs_baseline": None, "dtype": wl.dtype,
        "data": "synthetic (seeded)",
        "config": dict(config_of(wl), block_n=plan.config()[0],
                       input_widening=("in the kernel" if fc.fconv_plan_get_input_widening(plan.handle)
                                       else "fp16 copy" if wl.dtype == "int8" else "none (bf16)"),
                       images_per_rank=(f"[{lo}, {hi}) of {wl.N} (batch split over {world} ranks)"
                                        if args.strong else f"all {wl.N} (each rank its own batch)"),
                       splits=fc.fconv_plan_get_splits(plan.handle), variant=args.variant,
                       l2=(f"inputs larger than L2: x+w+side+y+workspace = {footprint / 1e6:.0f} MB"
                           f" > {L2_BYTES / 1e6:.0f} MB") if flush is None else
                          (f"L2 flushed before every step (x+w+side+y+workspace = "
                           f"{footprint / 1e6:.0f} MB); steps timed by their own events")),
        "stage_ms": {"prep (filter copy + int8->fp16 widening)": statistics.mean(prep_ms),
                     "conv": statistics.mean(conv_ms)},
        "roofline": roofline,
        "e2e": e2e,
        "graph": graph,
        "gpu_launches": args.steps * fc.fconv_plan_launch_count(plan.handle),
        "clocks": clk,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, n_img, t, threads = time_oracle(wl, P, Q, args.cpu_seconds, wl.N)
        line["cpu_baseline"] = {"value": v, "unit": UNIT, "cores": threads, "kind": "oracle",
                                "sample": f"{n_img} of {wl.N} images, all channels, full epilogue "
                                          f"({t:.1f} s)"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    plan.close()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["fconv", "reference"], default="fconv")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD,
                    choices=list(FI.WORKLOADS) + list(FI.VARIANT_WORKLOADS))
    ap.add_argument("--variant", default="plain", choices=list(VARIANTS),
                    help="epilogue variant: per-channel conv scale or another activation")
    ap.add_argument("--tile", type=int, default=0)
    ap.add_argument("--tile-shape", default="",
                    help="PIXELS,CHANNELS: force the output tile (128 or 256 pixels)")
    ap.add_argument("--batch", type=int, default=0,
                    help="run the workload's layer on this many images (profiling only)")
    ap.add_argument("--widen", type=int, default=0, choices=[0, 1, 2],
                    help="int8 input widening: 0 automatic, 1 in the kernel, 2 an fp16 copy")
    ap.add_argument("--gather", default="", choices=["", "auto", "im2col", "halo"],
                    help="input gather: the plan's own choice, never the halo gather, or the "
                         "halo gather (stride-1 layers with 64 input channels)")
    ap.add_argument("--splits", type=int, default=0,
                    help="force a split-K count (1: none; 0: the plan's own choice)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--graph", action="store_true",
                    help="also time the steps replayed from a CUDA graph (GPU time alone)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--strong", action="store_true",
                    help="split the workload's batch over the ranks (strong scaling) instead of "
                         "giving every rank the whole batch (weak scaling)")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        import torch
        import torch.distributed as tdist
        torch.cuda.set_device(local_rank)
        tdist.init_process_group("nccl")
    run_fconv(args, rank, world, local_rank)
    if world > 1:
        import torch.distributed as tdist
        tdist.destroy_process_group()


if __name__ == "__main__":
    main()
