#!/usr/bin/env python3
"""Throughput of the fused 3x3 conv + epilogue on GB300.

One step = one conv_epi_forward over the whole batch of the workload (conv +
fused chain), inputs resident in HBM.  Default workload (the largest of the
five, and the headline): x[64,64,256,256], Conv2d 64->128 (k3, s1, p0) with
bias, x 2.0, min over channels (``c4_scale_min``), in the tf32 tensor-core
mode.  L2 is flushed between timed steps (outside the step's events): a write
of a buffer larger than L2 evicts what the previous step left there, and a
read of a second one replaces the flush's own dirty lines with clean ones, so
that their write-back does not land inside the next timed step.

Prints ONE JSON line (rank 0).  Metric: TFLOP/s = 2*N*Cout*Ho*Wo*Cin*9 / time.
  value      - whole-job TFLOP/s over the K timed steps (sum of the steps'
               event times; max over ranks)
  e2e        - the same metric through conv_epi_forward_host, host buffers in
               and out (pinned), copies inside the timed region
  roofline   - the forward against the tf32 tensor peak derived from the
               measured bf16 peak (x 1.1/2.25, the nominal dense tf32:bf16
               ratio of the GB300's published rates), and against the
               measured HBM copy bandwidth; with --mode fp32 against the
               fp32 FMA rate instead (bound "alu")
  per_config - every other workload timed the same way in the same process:
               TFLOP/s, ms, both roofline fractions, the oracle on the host
               cores and the unfused comparator
  cpu_baseline - the fp64 oracle on the host cores over a bounded sample
  clocks     - nvidia-smi samples taken during the timed regions
  unfused    - context only, off the measured path: the unfused design the
               pages plan for (PyTorch conv2d on cuDNN writing the full conv
               output to HBM, then the chain as one fused post-pass kernel,
               conv_epi_postpass; also the chain as PyTorch ops), same inputs,
               same arithmetic mode, timed the same way

``--impl reference`` times the oracle instead (the only reference this
method has), on the same workload and metric, one bounded sample per step.

Multi-GPU (torchrun): every rank runs its own full replica of the workload
(weak scaling, no collective on the data path); value = all ranks' FLOPs /
the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synth  # noqa: E402

METRIC = "fused conv+epilogue TFLOP/s and % of GB300 TF32 dense peak (1 GPU)"
# nominal dense tensor rates of a GB300 (no 2:4 sparsity): tf32 1.1 PFLOP/s,
# bf16 2.25 PFLOP/s; the tf32 peak is the measured bf16 peak times their ratio
TF32_PER_BF16 = 1.1 / 2.25
FALLBACK_BF16_TFLOPS = 1900.0
FALLBACK_HBM_GBS = 6800.0
FALLBACK_SM_MAX_MHZ = 2070.0  # the GB300 maximum SM clock, where nvidia-smi gave no sample


def conv_flops(wl) -> int:
    """2 * N * Cout * Ho * Wo * Cin * 9 (multiply-adds counted twice)."""
    return 2 * wl.N * wl.Cout * (wl.H - 2) * (wl.W - 2) * wl.Cin * 9


def algorithmic_bytes(wl) -> int:
    """x read once + filter + bias + chain parameters + the chain's output."""
    n_out = {synth.KIND_MIN_TANH2: wl.N * (wl.H - 2) * (wl.W - 2),
             synth.KIND_SCALE_MIN: wl.N * (wl.H - 2) * (wl.W - 2),
             synth.KIND_MUL_LRELU_GELU: wl.N * wl.Cout * (wl.H - 2) * (wl.W - 2),
             synth.KIND_GN_SCALE_POOL_CLAMP: wl.N * wl.Cout * ((wl.H - 2 - wl.pool_k) // wl.pool_k + 1) *
             ((wl.W - 2 - wl.pool_k) // wl.pool_k + 1)}[wl.kind]
    params = {synth.KIND_MUL_LRELU_GELU: 1, synth.KIND_GN_SCALE_POOL_CLAMP: 3}.get(wl.kind, 0)
    return 4 * (wl.N * wl.Cin * wl.H * wl.W + wl.Cout * wl.Cin * 9 + wl.Cout * (1 + params) + n_out)


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d.get("bf16_tflops", FALLBACK_BF16_TFLOPS), d.get("hbm_gbs", FALLBACK_HBM_GBS), "measured"
    return FALLBACK_BF16_TFLOPS, FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.rows = []
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append([c.strip() for c in line.split(",")])

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.t.join(timeout=2)

    def summary(self):
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = [float(r[1]) for r in self.rows if len(r) > 2 and r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in self.rows if len(r) > 2 and r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in self.rows:
            for k, nm in enumerate(names):
                if len(r) > 5 + k and r[5 + k].lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(self.rows)}


def dist_setup():
    """Ranks from the torchrun environment; NCCL between GPUs, gloo where no
    GPU is visible (the CPU tests of this host logic)."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        dist.init_process_group(backend="nccl" if torch.cuda.is_available() else "gloo")
    return world, rank, local


def _on_gpu():
    import torch.distributed as dist
    return dist.get_backend() == "nccl"


def barrier(world):
    if world > 1:
        import torch
        import torch.distributed as dist
        if _on_gpu():
            dist.barrier(device_ids=[torch.cuda.current_device()])
        else:
            dist.barrier()


def max_over_ranks(v, world):
    """The largest of every rank's v (the slowest rank's time)."""
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device="cuda" if _on_gpu() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# the single-core oracle figure is taken on one image where that image's
# conv is at most this many FLOPs (about a second on one host core)
SINGLE_CORE_MAX_FLOPS = 2.0e9


def oracle_sample(wl, seconds: float, max_images: int, cores: int = 0):
    """Time the fp64 oracle on whole images of the workload until ~seconds,
    on `cores` threads (0: every host core)."""
    import oracle
    one = wl.with_batch(1)
    t = synth.make_inputs(one, seed=0)
    ch = oracle.chain_for(one, t)
    cores = cores or os.cpu_count() or 1
    done, t0 = 0, time.perf_counter()
    while True:
        oracle.forward(t.x, t.w, t.b, ch, nthreads=cores, want_index=False)
        done += 1
        el = time.perf_counter() - t0
        if el >= seconds or done >= max_images:
            break
    return conv_flops(one) * done / el / 1e12, el, done, cores


def unfused_chain(wl, dev, mode_tf32: bool):
    """The unfused pipeline as a PyTorch function of the resident inputs:
    conv2d (cuDNN; tf32 allowed only in the tf32 mode) writing the full conv
    output, then the chain in PyTorch ops."""
    import torch
    import torch.nn.functional as F
    torch.backends.cudnn.allow_tf32 = mode_tf32
    torch.backends.cuda.matmul.allow_tf32 = mode_tf32
    x, w, b = dev["x"], dev["w"], dev["b"]

    def run():
        y = F.conv2d(x, w, b)
        if wl.kind == synth.KIND_MIN_TANH2:
            return torch.tanh(torch.tanh(torch.min(y * wl.scalar, dim=1, keepdim=True)[0]))
        if wl.kind == synth.KIND_SCALE_MIN:
            return torch.min(y * wl.scalar, dim=1, keepdim=True)[0]
        if wl.kind == synth.KIND_MUL_LRELU_GELU:
            return F.gelu(F.leaky_relu(y * dev["mult"].view(1, -1, 1, 1), wl.lrelu_slope))
        z = F.group_norm(y, wl.groups, dev["gamma"], dev["beta"], wl.eps) * dev["scale"].view(1, -1, 1, 1)
        return torch.clamp(F.max_pool2d(z, wl.pool_k), wl.clamp_lo, wl.clamp_hi)
    return run


def traffic_for(kernel_src_hash: str, workload: str):
    """DRAM bytes per launch of the dominant kernel from the committed ncu
    summary, if it was taken on the current kernel source."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(workload)
    if not e or e.get("src_sha1") != kernel_src_hash:
        return None
    return e.get("dram_bytes_per_launch")


def kernel_hash():
    h = hashlib.sha1()
    for name in ("tc.cu", "internal.h"):
        with open(os.path.join(ROOT, "x3_conv2d_epilogue_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def run_reference(args, wl, world, rank):
    if rank != 0:
        return 0
    for _ in range(args.warmup):
        oracle_sample(wl, 0.0, 1)
    vals, t_all = [], 0.0
    cores = os.cpu_count() or 1
    for _ in range(args.steps):
        v, el, done, cores = oracle_sample(wl, args.ref_seconds, 1 << 30)
        vals.append(v)
        t_all += el
    value = float(np.mean(vals))
    line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * t_all / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded SplitMix64)",
            "config": {"workload": wl.name, "x": [wl.N, wl.Cin, wl.H, wl.W], "Cout": wl.Cout, "chain": wl.desc},
            "impl": "reference",
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                             "sample": f"whole images of {wl.name}, ~{args.ref_seconds:.0f} s per step"},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


class L2Flush:
    """Evicts L2 between timed steps, outside their events: a write of a
    buffer larger than L2 (what the previous step left there goes out), then
    a read of a second such buffer (the write's dirty lines are replaced by
    clean ones, so their write-back does not land in the next timed step)."""

    def __init__(self, torch, stream):
        l2 = int(getattr(torch.cuda.get_device_properties(torch.cuda.current_device()), "L2_cache_size", 0))
        self.bytes = max(2 * l2, 256 << 20)
        self.w = torch.empty(self.bytes // 4, dtype=torch.float32, device="cuda")
        self.r = torch.zeros(self.bytes // 4, dtype=torch.float32, device="cuda")
        self.sink = torch.empty(1, dtype=torch.float32, device="cuda")
        self.stream = stream
        self.torch = torch
        self.l2 = l2

    def __call__(self):
        with self.torch.cuda.stream(self.stream):
            self.w.fill_(1.0)
            self.torch.amax(self.r, dim=0, keepdim=True, out=self.sink)

    def describe(self):
        return (f"L2 ({self.l2 / 1e6:.0f} MB) flushed between timed steps, outside the steps' events: "
                f"write {self.bytes / 1e6:.0f} MB, then read {self.bytes / 1e6:.0f} MB")


class Case:
    """One workload on the device: resident inputs, its chain, a handle and
    the output, with the forward as a step."""

    def __init__(self, wl, mode_name, layout_name, stream):
        import torch
        import x3_conv2d_epilogue_gb300 as ce
        self.ce = ce
        self.wl, self.stream = wl, stream
        self.mode = ce.MODE_TF32 if mode_name == "tf32" else ce.MODE_FP32
        self.nhwc = layout_name == "nhwc"
        t = synth.make_inputs(wl, seed=0)
        if self.nhwc:  # the same values, channels last
            t.x = np.ascontiguousarray(t.x.transpose(0, 2, 3, 1))
        self.host = {k: getattr(t, k) for k in ("x", "w", "b", "mult", "gamma", "beta", "scale")}
        self.dev = {k: (None if v is None else torch.from_numpy(v).cuda()) for k, v in self.host.items()}
        self.epi = self.epilogue(self.dev)
        self.h = ce.conv_epi_create(wl.N, wl.Cin, wl.H, wl.W, wl.Cout, self.mode,
                                    ce.LAYOUT_NHWC if self.nhwc else ce.LAYOUT_NCHW)
        ce.conv_epi_reserve(self.h, self.epi)
        self.shape = ce.conv_epi_output_shape(wl.N, wl.Cin, wl.H, wl.W, wl.Cout, self.epi, self.mode)
        self.out = torch.empty(self.shape, device="cuda", dtype=torch.float32)

    def epilogue(self, t):
        wl = self.wl
        chan = t["mult"] if wl.kind == synth.KIND_MUL_LRELU_GELU else t["scale"]
        return self.ce.epilogue(wl.kind, scalar=wl.scalar, chan_scale=chan, lrelu_slope=wl.lrelu_slope,
                                groups=wl.groups, eps=wl.eps, gamma=t["gamma"], beta=t["beta"],
                                pool_k=wl.pool_k, clamp_lo=wl.clamp_lo, clamp_hi=wl.clamp_hi)

    def step(self):
        self.ce.conv_epi_forward(self.h, self.dev["x"], self.dev["w"], self.dev["b"], self.epi, self.out, self.stream)

    def sync(self):
        self.ce.conv_epi_sync(self.h, self.stream)

    def close(self):
        if self.h:
            self.ce.conv_epi_destroy(self.h)
            self.h = None


def time_steps(step, stream, steps, warmup, flush, world=1):
    """W untimed warm-up steps, then K steps, each bracketed by CUDA events on
    the launching stream, with the L2 flush between them (outside the events);
    a barrier and a device synchronize on both sides.  Returns the per-step
    times (ms)."""
    import torch
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            flush()
            step()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    barrier(world)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for a, b in evs:
            flush()
            a.record(stream)
            step()
            b.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    return [a.elapsed_time(b) for a, b in evs]


def fp32_roofline(tflops, sm_count, sm_max_mhz):
    """The strict mode runs on the CUDA cores: its roofline is the fp32 FMA
    rate (SMs x 128 FMA lanes x 2 flops x the maximum SM clock, the sampled
    one or the GB300's 2070 MHz), and the tensor kernel's DRAM capture does
    not describe it."""
    sm_max = sm_max_mhz or FALLBACK_SM_MAX_MHZ
    peak = sm_count * 128 * 2 * sm_max * 1e-6
    return {"bound": "alu", "peak": peak, "frac": tflops / peak, "traffic": None,
            "peak_source": f"{sm_count} SMs x 128 fp32 FMA/clk x 2 x {sm_max:.0f} MHz (derived)",
            "kernel": "conv_epi forward (fused fp32 CUDA-core kernel)"}


def roofline_of(wl, ms, tf32_peak, hbm):
    """Both roofline fractions of one forward; `bound` is the roofline with
    the longer ideal time at the measured peaks."""
    flops, nbytes = conv_flops(wl), algorithmic_bytes(wl)
    tflops = flops / (ms * 1e-3) / 1e12
    gbs = nbytes / (ms * 1e-3) / 1e9
    bound = "tensor" if flops / (tf32_peak * 1e12) >= nbytes / (hbm * 1e9) else "hbm"
    return {"tflops": tflops, "tensor_frac": tflops / tf32_peak, "hbm_gbs": gbs, "hbm_frac": gbs / hbm,
            "bound": bound, "flops": flops, "algorithmic_bytes": nbytes}


def measure_unfused(wl, case, mode_name, steps, warmup, flush, stream, kern_ms):
    """The unfused design the pages plan for, on the case's inputs (context
    only, off the measured path): PyTorch conv2d on cuDNN (tf32 allowed only in
    the tf32 mode) writing the full conv output, then the chain as ONE fused
    post-pass kernel of this library (conv_epi_postpass); and, as a second
    reference, the chain as a string of PyTorch ops."""
    import torch
    import torch.nn.functional as F
    import x3_conv2d_epilogue_gb300 as ce
    torch.backends.cudnn.allow_tf32 = mode_name == "tf32"
    torch.backends.cuda.matmul.allow_tf32 = mode_name == "tf32"
    x, w, b = case.dev["x"], case.dev["w"], case.dev["b"]
    h = ce.conv_epi_create(wl.N, wl.Cin, wl.H, wl.W, wl.Cout, ce.MODE_FP32)
    out = torch.empty(case.shape, device="cuda", dtype=torch.float32)

    def run_post():
        y = F.conv2d(x, w, b)
        ce.conv_epi_postpass(h, y, case.epi, out, stream)

    n = min(steps, 10)
    p_ms = float(np.mean(time_steps(run_post, stream, n, warmup, flush)))
    ce.conv_epi_sync(h, stream)
    ce.conv_epi_destroy(h)
    del out
    torch.cuda.empty_cache()
    t_ms = float(np.mean(time_steps(unfused_chain(wl, case.dev, mode_name == "tf32"), stream, n, warmup, flush)))
    torch.cuda.empty_cache()
    return {"value": conv_flops(wl) / (p_ms * 1e-3) / 1e12, "unit": "TFLOP/s", "ms_per_step": p_ms,
            "fused_speedup": p_ms / kern_ms,
            "kind": "PyTorch conv2d (cuDNN, full conv output to HBM) + the chain as one fused post-pass kernel "
                    "(conv_epi_postpass); context only, not on the measured path",
            "torch_ops": {"value": conv_flops(wl) / (t_ms * 1e-3) / 1e12, "ms_per_step": t_ms,
                          "fused_speedup": t_ms / kern_ms,
                          "kind": "PyTorch conv2d (cuDNN) + the chain as separate PyTorch ops"}}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="c4_scale_min", choices=sorted(synth.WORKLOADS))
    ap.add_argument("--mode", choices=["tf32", "fp32"], default="tf32")
    ap.add_argument("--layout", choices=["nchw", "nhwc"], default="nchw",
                    help="memory layout of x handed to the library (nhwc: channels last)")
    ap.add_argument("--e2e-steps", type=int, default=3)
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="oracle sample length for cpu_baseline")
    ap.add_argument("--cfg-cpu-seconds", type=float, default=4.0, help="oracle sample length per per_config entry")
    ap.add_argument("--ref-seconds", type=float, default=15.0, help="oracle sample length per reference step")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer leg (profiling runs)")
    ap.add_argument("--no-unfused", action="store_true", help="skip the unfused PyTorch/cuDNN comparison (context only)")
    ap.add_argument("--no-per-config", action="store_true", help="time the chosen workload only")
    ap.add_argument("--no-flush", action="store_true", help="no L2 flush between steps (profiling runs only)")
    ap.add_argument("--batch", type=int, default=0, help="override the workload's batch (profiling runs only)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    wl = synth.WORKLOADS[args.workload]
    if args.batch:
        wl = wl.with_batch(args.batch)
    world, rank, local = dist_setup()
    if args.impl == "reference":
        return run_reference(args, wl, world, rank)

    import torch
    import x3_conv2d_epilogue_gb300 as ce
    torch.cuda.set_device(local)
    ce._lib()  # the CUDA library must load: there is no fallback
    stream = torch.cuda.Stream()
    flush = (lambda: None) if args.no_flush else L2Flush(torch, stream)
    bf16, hbm, src = peaks()
    tf32_peak = bf16 * TF32_PER_BF16
    sm_count = torch.cuda.get_device_properties(local).multi_processor_count

    # ---- the headline workload: K timed steps, per-step CUDA events ----
    case = Case(wl, args.mode, args.layout, stream)
    with ClockSampler(local) as clk:
        time.sleep(0.3)  # let the sampler start
        per = time_steps(case.step, stream, args.steps, args.warmup, flush, world)
        launches_per_step = ce.conv_epi_last_launch_count(case.h)
        case.sync()
        total_ms = max_over_ranks(float(np.sum(per)), world)
        kern_ms = float(np.mean(per))

        # ---- every other workload, timed the same way in the same process ----
        per_config = {}
        if not args.no_per_config and not args.batch:
            for name in sorted(synth.WORKLOADS):
                if name == wl.name:
                    continue
                other = synth.WORKLOADS[name]
                oc = Case(other, args.mode, args.layout, stream)
                o_per = time_steps(oc.step, stream, args.steps, args.warmup, flush)
                oc.sync()
                o_ms = float(np.mean(o_per))
                entry = {"workload": name, "chain": other.desc, "ms": o_ms, "ms_min": float(np.min(o_per)),
                         **roofline_of(other, o_ms, tf32_peak, hbm)}
                entry["launches_per_step"] = ce.conv_epi_last_launch_count(oc.h)
                if not args.no_unfused and not oc.nhwc and rank == 0:
                    entry["unfused"] = measure_unfused(other, oc, args.mode, args.steps, 3, flush, stream, o_ms)
                oc.close()
                per_config[name] = entry
                del oc
                torch.cuda.empty_cache()
    flops = conv_flops(wl)
    value = flops * args.steps * world / (total_ms * 1e-3) / 1e12

    # ---- end to end through the host-buffer entry point ----
    e2e = None
    if not args.no_e2e:
        host = case.host
        pin = {k: (None if v is None else torch.from_numpy(v).pin_memory()) for k, v in host.items()}
        epi_h = case.epilogue(pin)
        out_h = torch.empty(case.shape, dtype=torch.float32).pin_memory()
        ce.conv_epi_forward_host(case.h, pin["x"], pin["w"], pin["b"], epi_h, out_h, stream)   # warm (allocates staging)
        barrier(world)
        t0 = time.perf_counter()
        for _ in range(args.e2e_steps):
            ce.conv_epi_forward_host(case.h, pin["x"], pin["w"], pin["b"], epi_h, out_h, stream)
        e2e_s = max_over_ranks(time.perf_counter() - t0, world)
        h2d = sum(v.nbytes for v in host.values() if v is not None)
        e2e = {"value": flops * args.e2e_steps * world / e2e_s / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": out_h.numel() * 4}

    # ---- context: the unfused pipeline on the same inputs (not the product) ----
    unfused = None
    if not args.no_unfused and not case.nhwc and rank == 0:
        del case.out
        torch.cuda.empty_cache()
        unfused = measure_unfused(wl, case, args.mode, args.steps, 3, flush, stream, kern_ms)
    case.close()

    if rank != 0:
        return 0

    rl = roofline_of(wl, kern_ms, tf32_peak, hbm)
    cpu = None
    if not args.no_cpu_baseline:
        v, el, done, cores = oracle_sample(wl, args.cpu_seconds, wl.N)
        cpu = {"value": v, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
               "sample": f"{done} of {wl.N} images of {wl.name} ({el:.1f} s, fp64 direct loops)"}
        if conv_flops(wl.with_batch(1)) <= SINGLE_CORE_MAX_FLOPS:  # one image on one core, where that is short
            v1, el1, _, _ = oracle_sample(wl, 0.0, 1, cores=1)
            cpu["single_core"] = {"value": v1, "unit": "TFLOP/s", "sample": f"1 image on 1 thread ({el1:.2f} s)"}
        for name, entry in per_config.items():
            other = synth.WORKLOADS[name]
            ov, oel, odone, ocores = oracle_sample(other, args.cfg_cpu_seconds, other.N)
            entry["oracle"] = {"value": ov, "unit": "TFLOP/s", "cores": ocores,
                               "sample": f"{odone} of {other.N} images ({oel:.1f} s)"}
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": args.mode, "data": "synthetic (seeded SplitMix64)",
        "config": {"workload": wl.name, "x": [wl.N, wl.Cin, wl.H, wl.W], "Cout": wl.Cout, "chain": wl.desc,
                   "mode": args.mode, "layout": args.layout,
                   "l2": "no flush (profiling run)" if args.no_flush else flush.describe(),
                   "per_gpu_batch": wl.N},
        "roofline": {"bound": rl["bound"], "achieved": rl["tflops"], "peak": tf32_peak, "unit": "TFLOP/s",
                     "frac": rl["tensor_frac"],
                     "traffic": traffic_for(kernel_hash(), wl.name + ("_nhwc" if args.layout == "nhwc" else "")),
                     "peak_source": f"{src} bf16 burst {bf16:.1f} x {TF32_PER_BF16:.4f} (of {src})",
                     "kernel": "conv_epi forward (filter pack + fused conv kernel)",
                     "hbm_gbs": rl["hbm_gbs"], "hbm_peak_gbs": hbm, "hbm_frac": rl["hbm_frac"]},
        "per_config": per_config,
        "cpu_baseline": cpu,
        "unfused": unfused,
        "e2e": e2e,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk.summary(),
        "kernel_ms": {"mean": kern_ms, "min": float(np.min(per)), "max": float(np.max(per))},
    }
    if args.mode == "fp32":
        line["roofline"].update(fp32_roofline(rl["tflops"], sm_count, line["clocks"].get("sm_max_mhz")))
    print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
