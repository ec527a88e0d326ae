"""Benchmark: ConvTranspose3d + fused epilogue, useful TFLOP/s and ms/forward on GB300.

One step = one pass of the whole hot path over one batch: weight pack/split,
input staging, the implicit-GEMM kernel with its fused epilogue, statistics
finalisation and (GroupNorm) the normalise pass -- every kernel of
convt3d_pack_weights + convt3d_forward.  Inputs are resident in HBM; L2 is
flushed (a 256 MiB write) before every timed step.  Each step is timed with
CUDA events on the launching stream.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                  [--precision 3xtf32|3xbf16|tf32|bf16|ffma] [--impl gpu|reference]

Under torchrun (N > 1) every rank runs an independent replica of the workload
on its own GPU (the path shards by batch with no collective on the data path);
`value` is the useful flop of all ranks over the slowest rank's time.
`--impl reference` times the CPU oracle on the host cores instead (rank 0 only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads  # noqa: E402

# The largest configuration (l2_p77's module: ConvTranspose3d k=5, x2, BatchNorm3d
# with batch statistics, AdaptiveAvgPool3d(1); 5.37e11 useful flop per step).
DEFAULT_WORKLOAD = workloads.BN.name
# The other configurations, timed GPU-only in the same process for the
# "configs" key of the line (the bench's own workload is left out).
OTHER_WORKLOADS = [workloads.TINY, workloads.GN, workloads.BN, workloads.SOFTMAX, workloads.IDENTITY,
                   workloads.BN_EVAL]
TF32_OVER_BF16 = 1.1 / 2.25   # nominal dense TF32 / BF16 tensor rates (GB300)
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
FP32_FMA_PER_CLK_PER_SM = 128
SMS = 152


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(workloads.BY_NAME))
    ap.add_argument("--precision", default="3xtf32", choices=["3xtf32", "3xbf16", "tf32", "bf16", "fp16", "ffma"])
    ap.add_argument("--impl", default="gpu", choices=["gpu", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="target wall time of the CPU baseline sample")
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--e2e-chunks", type=int, default=8, help="sample chunks the end-to-end pipeline overlaps")
    ap.add_argument("--io-bf16", action="store_true",
                    help="x, w and y as bf16 tensors (requires --precision bf16)")
    ap.add_argument("--io-fp16", action="store_true",
                    help="x, w and y as fp16 tensors (requires --precision fp16)")
    ap.add_argument("--e2e-copy-streams", type=int, default=1,
                    help="streams per copy direction in the end-to-end pipeline")
    ap.add_argument("--config-steps", type=int, default=10,
                    help="timed steps per other configuration in the \"configs\" key (0: leave it out)")
    ap.add_argument("--config-precisions", default="3xtf32,3xbf16",
                    help="precisions the other configurations are timed in")
    return ap.parse_args()


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "sm_max_mhz": float(p.get("sm_max_mhz", 2070.0)), "source": "measured"}
    except Exception:
        return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": FALLBACK_BF16_TFLOPS,
                "bf16_tflops_sustained": 1700.0, "sm_max_mhz": 2070.0, "source": "fallback"}


# ----------------------------------------------------------------- clocks ----

class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while running."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id):
        self.gpu = str(gpu_id)
        self.proc = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "100", "-i", self.gpu], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if not self.proc:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        rows = []
        for line in out.strip().splitlines():
            f = [v.strip() for v in line.split(",")]
            if len(f) < 9:
                continue
            try:
                rows.append({"sm": float(f[1]), "max": float(f[2]), "power": float(f[3]),
                             "hw": f[5], "hw_thermal": f[6], "sw_thermal": f[7], "sw_power": f[8]})
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        peak_power = max(r["power"] for r in rows)
        loaded = [r for r in rows if r["power"] >= 0.5 * peak_power] or rows
        reasons = set()
        for r in loaded:
            for key, name in (("hw", "hw_slowdown"), ("hw_thermal", "hw_thermal_slowdown"),
                              ("sw_thermal", "sw_thermal_slowdown"), ("sw_power", "sw_power_cap")):
                if r[key].lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in loaded), "sm_max_mhz": max(r["max"] for r in rows),
                "reasons": sorted(reasons), "samples": len(loaded), "power_w_max": peak_power}


# ------------------------------------------------------- traffic from ncu ----

# main kernel of a plan (convt3d_info_t.main_kernel) -> its name and source file
MAIN_KERNELS = {0: ("convt3d_tc_gemm", "tc.cu"), 1: ("ffma_conv_kernel", "ffma.cu"), 2: ("convt3d_direct_gemm", "direct.cu")}


def kernel_source_sha(main_kernel):
    """Fingerprint of the main kernel's sources: its .cu file plus the shared headers."""
    csrc = os.path.join(ROOT, "transposed_convolution_convt3d_gb300", "csrc")
    h = hashlib.sha256()
    for src in (MAIN_KERNELS[main_kernel][1], "epimath.cuh", "ptx.cuh", "convt3d_internal.h"):
        with open(os.path.join(csrc, src), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def committed_profile_value(precision, workload, field, main_kernel):
    """A number (`field = value`) from the committed ncu summary of the main
    kernel, if that summary was taken on the current kernel source (else None)."""
    d = os.path.join(ROOT, "profiles")
    if not os.path.isdir(d):
        return None
    want = kernel_source_sha(main_kernel)
    for name in sorted(os.listdir(d)):
        if not name.endswith((".md", ".txt")):
            continue
        text = open(os.path.join(d, name)).read()
        m_sha = re.search(r"kernel_source_sha\s*[:=]\s*([0-9a-f]{16})", text)
        m_w = re.search(r"workload\s*[:=]\s*(\S+)", text)
        m_t = re.search(field + r"\s*[:=]\s*([0-9.eE+]+)", text)
        m_p = re.search(r"precision\s*[:=]\s*(\S+)", text)
        if m_sha and m_t and m_w and m_sha.group(1) == want and m_w.group(1) == workload and \
                (not m_p or m_p.group(1) == precision):
            return float(m_t.group(1))
    return None


def committed_traffic(precision, workload, main_kernel):
    """DRAM bytes per launch of the main kernel (ncu dram__bytes_read.sum +
    dram__bytes_write.sum) from the committed summary, else None."""
    return committed_profile_value(precision, workload, "traffic_bytes_per_launch", main_kernel)


def committed_tensor_active(precision, workload, main_kernel):
    """ncu's sm__pipe_tensor_cycles_active (fraction of elapsed cycles) of the
    main kernel from the committed summary, else None."""
    v = committed_profile_value(precision, workload, "tensor_pipe_active", main_kernel)
    return None if v is None else (v / 100.0 if v > 1.0 else v)


# ------------------------------------------------------------ replicas ----

def max_over_ranks(value, device=None):
    """Max of a per-rank float over all ranks (identity without a process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(useful_flop_per_rank, world, slowest_ms_per_step):
    """Whole-job useful TFLOP/s: every rank processed its own batch in the slowest rank's time."""
    return useful_flop_per_rank * world / (slowest_ms_per_step * 1e-3) / 1e12


# ------------------------------------------------------------ CPU oracle ----

def oracle_running_stats(spec):
    """The running statistics the evaluation-mode epilogue reads (fresh copies), else nothing."""
    if spec.epilogue != workloads.EPI_SCALE_BATCHNORM_EVAL_AVGPOOL:
        return {}
    rm, rv = workloads.make_running_stats(spec)
    return {"running_mean": rm.numpy().copy(), "running_var": rv.numpy().copy()}


def cpu_oracle_sample(spec, inputs, target_s, max_samples=None):
    """Time the oracle on a bounded sample of the batch: whole samples of the
    per-sample epilogues (for BatchNorm the first n samples form a smaller
    batch).  Returns (useful TFLOP/s, seconds, samples, cores)."""
    import oracle
    f = lambda t: None if t is None else t.float().numpy()  # noqa: E731
    done, elapsed, n = 0, 0.0, 0
    limit = spec.N if max_samples is None else min(spec.N, max_samples)
    step = 1
    while n < limit:
        m = min(step, limit - n)
        sub = workloads.sample_slice(inputs, n, n + m)
        s = spec.replace(N=m)
        t0 = time.perf_counter()
        oracle.forward(f(sub["x"]), f(sub["w"]), f(sub["bias"]), stride=s.stride, pad=s.pad, out_pad=s.out_pad,
                       epilogue=s.epilogue, groups=s.groups, eps=s.eps, scale=s.scale, gamma=f(sub["gamma"]),
                       beta=f(sub["beta"]), **oracle_running_stats(spec))
        elapsed += time.perf_counter() - t0
        done += s.useful_flop()
        n += m
        if elapsed >= target_s:
            break
    return done / elapsed / 1e12, elapsed, n, oracle.num_threads()


def run_reference(args, spec):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    oracle.build()
    inputs = workloads.make_inputs(spec)
    f = lambda t: None if t is None else t.numpy()  # noqa: E731
    sub = workloads.sample_slice(inputs, 0, 1)
    s = spec.replace(N=1)

    def step():
        oracle.forward(f(sub["x"]), f(sub["w"]), f(sub["bias"]), stride=s.stride, pad=s.pad, out_pad=s.out_pad,
                       epilogue=s.epilogue, groups=s.groups, eps=s.eps, scale=s.scale, gamma=f(sub["gamma"]),
                       beta=f(sub["beta"]), **oracle_running_stats(spec))
    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / args.steps
    value = s.useful_flop() / dt / 1e12
    sample = f"1 of {spec.N} batch samples per step ({s.useful_flop():.3e} useful flop)"
    line = {
        "impl": "reference", "metric": "useful_tflops", "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": spec.name, "sample": sample, "oracle": "CPU scatter-form fp64 loop nest (OpenMP)"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": oracle.num_threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# -------------------------------------------------------------- roofline ----

def roofline(info, precision, useful, kernel_ms, ms_per_step, pk, eval_bn):
    """Roofline of the main kernel: algorithmic work of one launch over its
    CUDA-event time, against the measured peak of its bound."""
    if eval_bn:
        # two HBM-bound kernels (box sums over x, contraction with the packed weight)
        achieved = info["forward_min_bytes"] / (kernel_ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / pk["hbm_gbs"], "peak_source": f"{pk['source']} HBM copy bandwidth",
                "algorithmic_bytes": info["forward_min_bytes"]}
    elif precision != "ffma":
        bf = precision in ("bf16", "3xbf16", "fp16")  # kind::f16: the same tensor rate for bf16 and fp16
        peak = pk["bf16_tflops"] * (1.0 if bf else TF32_OVER_BF16)
        achieved = useful / (kernel_ms * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                "peak_source": (f"{pk['source']} bf16 burst" if bf else
                                f"{pk['source']} bf16 burst x nominal TF32/BF16 ratio {TF32_OVER_BF16:.4f}"),
                # issued tensor flop (three products per term in the split formats) over that peak;
                # the peak was measured at a lower clock than these kernels run at, so this can
                # read above 1: the tensor pipe's own utilisation is tensor_pipe_active (ncu)
                "issued_frac": info["issued_mma_flop"] / (kernel_ms * 1e-3) / 1e12 / peak}
        if precision in ("3xtf32", "3xbf16"):
            roof["frac_of_" + precision + "_peak"] = achieved / (peak / 3.0)
        # Where the kernel's arithmetic intensity (useful flop per algorithmic byte) times the
        # measured HBM bandwidth is below its useful-flop ceiling (a third of the tensor peak
        # for the split formats), HBM bounds it (the softmax workload): report that roofline.
        ceiling = peak / 3.0 if precision in ("3xtf32", "3xbf16") else peak
        ai = useful / info["gemm_min_bytes"]
        if ai * pk["hbm_gbs"] * 1e9 < ceiling * 1e12:
            gbs = info["gemm_min_bytes"] / (kernel_ms * 1e-3) / 1e9
            tensor = {k: roof[k] for k in ("achieved", "peak", "unit", "frac", "peak_source")}
            roof = {"bound": "hbm", "achieved": gbs, "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": gbs / pk["hbm_gbs"],
                    "peak_source": f"{pk['source']} HBM copy bandwidth", "algorithmic_bytes": info["gemm_min_bytes"],
                    "tensor": tensor, "issued_frac": roof["issued_frac"]}
    else:
        peak = SMS * FP32_FMA_PER_CLK_PER_SM * 2 * pk["sm_max_mhz"] * 1e6 / 1e12
        achieved = useful / (kernel_ms * 1e-3) / 1e12
        roof = {"bound": "alu", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                "peak_source": "152 SMs x 128 fp32 FMA/clk x 2 flop x max SM clock",
                "issued_frac": info["issued_mma_flop"] / (kernel_ms * 1e-3) / 1e12 / peak}
    roof["kernel"] = ("boxsum_kernel + bn_eval_out_kernel" if eval_bn else
                      MAIN_KERNELS[info["main_kernel"]][0])
    roof["kernel_ms"] = kernel_ms
    roof["kernel_share_of_step"] = kernel_ms / ms_per_step
    roof["min_bytes"] = info["gemm_min_bytes"]
    return roof


def gpu_hold(cycles=300_000):
    """Keep the GPU busy for ~0.15 ms before a step's start event, so that the
    host has queued the step's launches by the time the event is recorded: the
    timed region then holds the device work of the step, not the host's
    enqueue latency after the previous step's synchronisation."""
    import torch
    if hasattr(torch.cuda, "_sleep"):
        torch.cuda._sleep(cycles)


PRECISION_CODES = {"3xtf32": 0, "ffma": 1, "tf32": 2, "bf16": 3, "3xbf16": 4, "fp16": 5}


def time_config(spec, precision, steps, warmup, dev, stream, flush, pk):
    """GPU-only timing of one configuration: pack_weights + forward per step,
    L2 flushed before each, CUDA events on the launching stream (the main
    kernel's own events from the library's profiling hooks)."""
    import torch

    from transposed_convolution_convt3d_gb300 import Plan
    inputs = workloads.make_inputs(spec)
    d = {k: (v.to(dev) if v is not None else None) for k, v in inputs.items()}
    plan = Plan.from_spec(spec, precision=PRECISION_CODES[precision])
    info = plan.info
    ws = plan.new_workspace(dev)
    y = plan.new_output(dev)
    eval_bn = spec.epilogue == workloads.EPI_SCALE_BATCHNORM_EVAL_AVGPOOL
    if eval_bn:
        plan.set_running_stats(*(t.to(dev) for t in workloads.make_running_stats(spec)))
    step_ms, kern_ms = [], []
    for i in range(warmup + steps):
        flush.fill_(float(i))
        gpu_hold()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        plan.profile_enable(not eval_bn and i >= warmup)
        a.record(stream)
        plan.pack_weights(d["w"], ws, stream)
        f0.record(stream)
        plan.forward(d["x"], y, ws, d["bias"], d["gamma"], d["beta"], stream)
        f1.record(stream)
        b.record(stream)
        if i >= warmup:
            b.synchronize()
            step_ms.append(a.elapsed_time(b))
            kern_ms.append(f0.elapsed_time(f1) if eval_bn else plan.profile_read())
    plan.profile_enable(False)
    plan.check(ws, stream)
    ms = sum(step_ms) / len(step_ms)
    km = sum(kern_ms) / len(kern_ms)
    useful = spec.useful_flop()
    roof = roofline(info, precision, useful, km, ms, pk, eval_bn)
    out = {"workload": spec.name, "precision": precision, "ms_per_step": ms,
           "useful_tflops": useful / (ms * 1e-3) / 1e12, "kernel": roof["kernel"], "kernel_ms": km,
           "bound": roof["bound"], "frac": roof["frac"],
           "hbm_frac_whole_step": info["forward_min_bytes"] / (ms * 1e-3) / 1e9 / pk["hbm_gbs"]}
    for k in ("issued_frac", "frac_of_3xtf32_peak", "frac_of_3xbf16_peak"):
        if k in roof:
            out[k] = roof[k]
    out["tensor_pipe_active"] = None if eval_bn else committed_tensor_active(precision, spec.name, info["main_kernel"])
    del ws, y, d
    torch.cuda.synchronize()
    return out


# ------------------------------------------------------------------ GPU ----

def run_gpu(args, spec):
    import torch
    import torch.distributed as dist

    from transposed_convolution_convt3d_gb300 import HostPipeline, Plan

    world, rank, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    prec = PRECISION_CODES[args.precision]

    io16 = torch.bfloat16 if args.io_bf16 else (torch.float16 if args.io_fp16 else None)
    if io16 is not None:
        spec = spec.replace(io_bf16=args.io_bf16, io_fp16=args.io_fp16)
    inputs = workloads.make_inputs(spec)
    if io16 is not None:
        inputs["x"], inputs["w"] = inputs["x"].to(io16), inputs["w"].to(io16)
    d = {k: (v.to(dev) if v is not None else None) for k, v in inputs.items()}
    plan = Plan.from_spec(spec, precision=prec)
    info = plan.info
    ws = plan.new_workspace(dev)
    y = plan.new_output(dev)
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    # evaluation-mode BatchNorm runs no GEMM: its kernels are timed as the whole forward
    eval_bn = spec.epilogue == workloads.EPI_SCALE_BATCHNORM_EVAL_AVGPOOL
    running = None
    if eval_bn:
        running = tuple(t.to(dev) for t in workloads.make_running_stats(spec))
        plan.set_running_stats(*running)

    fwd_ev = []

    def step():
        plan.pack_weights(d["w"], ws, stream)
        if fwd_ev:
            fwd_ev[-1][0].record(stream)
        plan.forward(d["x"], y, ws, d["bias"], d["gamma"], d["beta"], stream)
        if fwd_ev:
            fwd_ev[-1][1].record(stream)

    for _ in range(max(args.warmup, 3)):
        step()
    plan.check(ws, stream)
    torch.cuda.synchronize()

    plan.profile_enable(not eval_bn)
    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        gpu_id = str(local)
    clocks = ClockSampler(gpu_id)
    clocks.start()
    time.sleep(0.3)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    step_ms, gemm_ms = [], []
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    for i in range(args.steps):
        flush.fill_(float(i))  # evict x, y and the packed weights from L2 between steps
        gpu_hold()
        ev[i][0].record(stream)
        if eval_bn:
            fwd_ev.append((torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)))
        step()
        ev[i][1].record(stream)
        if eval_bn:
            fwd_ev[-1][1].synchronize()
            gemm_ms.append(fwd_ev[-1][0].elapsed_time(fwd_ev[-1][1]))
        else:
            gemm_ms.append(plan.profile_read())  # synchronises on the GEMM's end event
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    wall = time.perf_counter() - wall0
    clk = clocks.stop()
    plan.profile_enable(False)
    plan.check(ws, stream)
    step_ms = [a.elapsed_time(b) for a, b in ev]
    total_ms = max_over_ranks(sum(step_ms), dev)
    ms_per_step = total_ms / args.steps
    useful = spec.useful_flop()
    value = replica_throughput(useful, world, ms_per_step)

    # end to end through the public API from pinned host buffers: HostPipeline
    # copies x, w, bias, gamma, beta in and y out, overlapped with the
    # computation over chunks of samples (per-sample epilogues)
    e2e = None
    if args.e2e_steps > 0:
        host = {k: (v.pin_memory() if v is not None else None) for k, v in inputs.items()}
        pipe = HostPipeline(spec.N, spec.Cin, spec.Cout, spec.D, spec.H, spec.W, spec.k, spec.stride, spec.pad,
                            spec.out_pad, spec.bias, spec.epilogue, spec.groups, spec.eps, spec.scale, prec,
                            chunks=args.e2e_chunks, device=dev, copy_streams=args.e2e_copy_streams,
                            io_bf16=args.io_bf16, io_fp16=args.io_fp16)
        if running is not None:
            pipe.set_running_stats(*running)
        y_host = torch.empty(pipe.full_shape, dtype=pipe.plan.io_dtype).pin_memory()
        h2d = sum(v.numel() * v.element_size() for v in host.values() if v is not None)
        d2h = y_host.numel() * y_host.element_size()
        e2e_ms = []
        for i in range(args.e2e_steps + 1):
            flush.fill_(float(i))
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            pipe(host["x"], host["w"], y_host, host["bias"], host["gamma"], host["beta"])
            b.record(stream)
            b.synchronize()
            if i > 0:
                e2e_ms.append(a.elapsed_time(b))
        e2e_chunks = pipe.chunks
        e2e_t = max_over_ranks(sum(e2e_ms) / len(e2e_ms), dev)
        link_t = host_link_ms(host, y, y_host, stream, dev)
        e2e = {"value": replica_throughput(useful, world, e2e_t), "unit": "TFLOP/s", "ms_per_step": e2e_t,
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "host_link_bound_ms": link_t, "host_link_frac": link_t / e2e_t,
               "path": f"HostPipeline, {e2e_chunks} chunk(s) of samples, {args.e2e_copy_streams} copy stream(s) "
                       "per direction, pinned host buffers"}

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    pk = peaks()
    gemm_avg = sum(gemm_ms) / len(gemm_ms)
    roof = roofline(info, args.precision, useful, gemm_avg, ms_per_step, pk, eval_bn)
    roof["traffic"] = committed_traffic(args.precision, spec.name, info["main_kernel"])
    hbm_frac = info["forward_min_bytes"] / (ms_per_step * 1e-3) / 1e9 / pk["hbm_gbs"]

    roof["tensor_pipe_active"] = None if eval_bn else committed_tensor_active(args.precision, spec.name, info["main_kernel"])

    # the other configurations, GPU-only, same process
    configs = None
    if args.config_steps > 0 and world == 1:
        configs = []
        for cs in OTHER_WORKLOADS:
            for pr in [p for p in args.config_precisions.split(",") if p]:
                if cs.name == spec.name and pr == args.precision:
                    continue
                if cs.epilogue == workloads.EPI_SCALE_BATCHNORM_EVAL_AVGPOOL and pr != "3xtf32":
                    continue
                configs.append(time_config(cs, pr, args.config_steps, 3, dev, stream, flush, pk))

    cpu = None
    if not args.no_cpu_baseline and world == 1:
        v, secs, nsamp, cores = cpu_oracle_sample(spec, inputs, args.cpu_seconds)
        cpu = {"value": v, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
               "sample": f"{nsamp} of {spec.N} batch samples ({secs:.1f} s)"}

    line = {
        "metric": "useful_tflops", "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": compute_dtype(args.precision), "data": "synthetic",
        "config": {"workload": spec.name, "precision": args.precision,
                   "io": "bf16" if args.io_bf16 else ("fp16" if args.io_fp16 else "f32"),
                   "x": [spec.N, spec.Cin, spec.D, spec.H, spec.W],
                   "w": [spec.Cin, spec.Cout, spec.k, spec.k, spec.k], "stride": spec.stride, "pad": spec.pad,
                   "out_pad": spec.out_pad, "out": list(plan.out_shape), "epilogue": spec.epilogue,
                   "step": "pack_weights + forward (all kernels)", "l2": "flushed (256 MiB write) before each step",
                   "useful_flop_per_step": useful, "parallelism": f"replicas x{world}"},
        "hbm_frac_whole_step": hbm_frac,
        "roofline": roof,
        "configs": configs,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": (info["launches_per_forward"] + info["launches_per_pack"]) * args.steps,
        "clocks": clk,
        "wall_s_timed": wall,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def compute_dtype(precision):
    """The arithmetic type of the products: the split formats (and the FFMA
    ablation) compute to fp32 accuracy; the single-product formats round their
    operands to TF32 or bf16."""
    return {"3xtf32": "f32", "3xbf16": "f32", "ffma": "f32", "tf32": "tf32", "bf16": "bf16", "fp16": "f16"}[precision]


def host_link_ms(host, y_dev, y_host, stream, dev, reps=3):
    """The host link's bound on one end-to-end step: the same bytes copied with
    nothing else running, the inputs host->device on a second stream while the
    output goes device->host (median of `reps` after one warm-up)."""
    import torch
    h2d = sum(t.numel() * t.element_size() for t in host.values() if t is not None)
    scratch = torch.empty(int(h2d), dtype=torch.uint8, device=dev)
    s_in = torch.cuda.Stream(device=dev)
    times = []
    for i in range(reps + 1):
        a, b, c = (torch.cuda.Event(enable_timing=True) for _ in range(3))
        a.record(stream)
        s_in.wait_event(a)
        with torch.cuda.stream(s_in):
            o = 0
            for t in host.values():
                if t is None:
                    continue
                n = t.numel() * t.element_size()
                scratch[o:o + n].copy_(t.reshape(-1).view(torch.uint8), non_blocking=True)
                o += n
            c.record(s_in)
        y_host.copy_(y_dev, non_blocking=True)
        stream.wait_event(c)
        b.record(stream)
        b.synchronize()
        if i > 0:
            times.append(a.elapsed_time(b))
    return sorted(times)[len(times) // 2]


def main():
    args = parse()
    spec = workloads.BY_NAME[args.workload]
    if args.impl == "reference":
        run_reference(args, spec)
    else:
        run_gpu(args, spec)


if __name__ == "__main__":
    main()
