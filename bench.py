#!/usr/bin/env python
"""Benchmark: dgrad useful TFLOP/s, % of the GB300 TF32 roofline, us per call.

One step = one pass of the whole hot path on one batch through the C ABI
(dgrad_run): the pack kernel (weights and, on the frame path, grad_out into
the channels-last frame) and the main implicit-GEMM kernel, chained with
programmatic dependent launch, inputs resident in HBM.  L2 is flushed
(256 MiB write) before every timed step, outside the timed events.  The main
kernel is also timed alone (dgrad_run_main after dgrad_prepack and
dgrad_pack_grad_out) for the roofline line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--precision tf32|tf32x3|fp32]
  python bench.py --impl reference ...   # the CPU oracle on the host cores
  python bench.py --all ...              # plus one info line per workload and precision, and per workload
                                         # the weight gradient (wgrad_run) of the same convolution
  python bench.py --profile [--op wgrad] [--path col2im]   # W + K steps only, for ncu

With N > 1 (torchrun, one rank per GPU) every rank runs an independent
replica of the workload (the batch shards with no collective on the data
path); ``value`` is the total useful FLOPs of all ranks / the slowest rank's
time.  Prints one JSON line on rank 0.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "dgrad useful TFLOP/s and % of GB300 TF32 roofline at 1 GPU; µs per call"
TF32_OVER_BF16 = 1.1 / 2.25          # nominal dense TF32 / BF16 ratio
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "sm_max_mhz": 2070.0}
FLUSH_BYTES = 256 << 20
MAIN_KERNEL_SOURCES = ["tc_kernel.cuh", "tc_kernel.cu", "tc_kernel_fused.cu", "tc_kernel_tmem.cu", "tc_kernel_staged.cu",
                       "tc_kernel_staged_fused.cu", "simt_kernel.cu", "gather.cuh", "ptx.cuh", "dgrad_internal.h"]
WORKLOAD_ORDER = ("tiny", "resnet_stage", "strided_downsample", "pointwise", "stem")


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return dict(FALLBACK), "fallback"


_LIVE_PEAKS = {}


def measure_peaks(torch, dg):
    """The two compute peaks the driver does not measure, measured here once
    per process on this GPU (timing only; no clock or power setting changes):
      * TF32 dense: torch.matmul of two fp32 8192 x 8192 matrices with TF32
        allowed (cuBLAS on the tensor cores), 2*8192^3 FLOP, best of 10 by
        CUDA events after warm-up -- the same method as the driver's bf16 peak;
      * FP32 FFMA: dgrad_probe_ffma (eight independent FMA chains per thread,
        8 blocks of 256 threads per SM over every SM of the device), best of 5.
    Returns {"tf32_tflops", "ffma_tflops", "sm_count", "ffma_nominal_tflops"}."""
    if _LIVE_PEAKS:
        return _LIVE_PEAKS
    import ctypes
    props = torch.cuda.get_device_properties(torch.cuda.current_device())
    sms = props.multi_processor_count
    stream = torch.cuda.current_stream()
    prev = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = True
    try:
        n = 8192
        g = torch.Generator(device="cuda").manual_seed(0)
        a = torch.randn((n, n), device="cuda", generator=g)
        b = torch.randn((n, n), device="cuda", generator=g)
        for _ in range(3):
            torch.matmul(a, b)
        best = float("inf")
        for _ in range(10):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            torch.matmul(a, b)
            e1.record(stream)
            torch.cuda.synchronize()
            best = min(best, e0.elapsed_time(e1) * 1e-3)
        tf32 = 2.0 * n ** 3 / best / 1e12
        del a, b
    finally:
        torch.backends.cuda.matmul.allow_tf32 = prev
    lib = dg.load_library()
    blocks, iters = sms * 8, 20000
    out = torch.empty(blocks * 256, device="cuda")
    h = ctypes.c_void_p(int(stream.cuda_stream))
    for _ in range(2):
        assert lib.dgrad_probe_ffma(blocks, iters, ctypes.c_void_p(out.data_ptr()), h) == 0
    best = float("inf")
    for _ in range(5):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        assert lib.dgrad_probe_ffma(blocks, iters, ctypes.c_void_p(out.data_ptr()), h) == 0
        e1.record(stream)
        torch.cuda.synchronize()
        best = min(best, e0.elapsed_time(e1) * 1e-3)
    ffma = 2.0 * blocks * 256 * 8 * iters / best / 1e12
    peaks, _ = load_peaks()
    _LIVE_PEAKS.update({"tf32_tflops": tf32, "ffma_tflops": ffma, "sm_count": sms,
                        "ffma_nominal_tflops": sms * 256 * peaks.get("sm_max_mhz", 2070.0) * 1e6 / 1e12})
    return _LIVE_PEAKS


def kernel_source_hash():
    h = hashlib.sha256()
    for name in MAIN_KERNEL_SOURCES:
        with open(os.path.join(ROOT, "conv2d_backward_implicit_dgrad_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic_entry(workload, precision):
    """The main kernel's ncu counters per launch from the committed summary
    (DRAM read + write bytes; bytes the SMs wrote into L2, which the DRAM
    counters miss while the writes stay in L2), only while the kernel sources
    are unchanged since the capture."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    e = rec.get(f"{workload}/{precision}")
    if not e or e.get("source_hash") != kernel_source_hash():
        return None
    return e


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while the GPU works."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
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
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=5)
        sms, maxs, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sms.append(float(parts[1]))
                maxs.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sms) if sms else None, "sm_max_mhz": max(maxs) if maxs else None,
                "power_w_max": max(power) if power else None, "reasons": sorted(reasons), "samples": len(sms)}


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_oracle_run(wl, images, seed=0, reps=1, threads=None):
    """Time the oracle (as it stands) on the first `images` images of the
    workload, on all host cores (or `threads` of them)."""
    import oracle
    from conv2d_backward_implicit_dgrad_gb300.workloads import make_tensors
    go, w = make_tensors((images, wl.Co, wl.oH, wl.oW), wl.w_shape, seed, wl.dist)
    go, w = go.numpy(), w.numpy()
    cores = cpu_cores() if threads is None else threads
    oracle.build()
    times = []
    for _ in range(reps):
        t0 = time.perf_counter()
        oracle.dgrad(go, w, wl.H, wl.W, wl.stride, wl.pad_h, wl.pad_w, nthreads=cores)
        times.append(time.perf_counter() - t0)
    flops = 2.0 * images * wl.Co * wl.oH * wl.oW * wl.Ci * wl.kH * wl.kW
    return flops, times, min(cores, images)


def wl_config(wl):
    return {"workload": wl.name, **{k: getattr(wl, k) for k in ("N", "Ci", "Co", "H", "W", "kH", "kW", "stride",
                                                                "pad_h", "pad_w")}}


def reference_arm(args, wl):
    if int(os.environ.get("RANK", "0")) != 0:
        return 0
    images = min(wl.N, 8)
    for _ in range(args.warmup):
        cpu_oracle_run(wl, images)
    step_times = []
    flops, cores = 0.0, 1
    for _ in range(args.steps):
        flops, times, cores = cpu_oracle_run(wl, images)
        step_times.append(times[0])
    t = statistics.mean(step_times)
    value = flops / t / 1e12
    sample = f"{images} of {wl.N} images of {wl.name} per step (fp64 scatter oracle, {cores} threads)"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": t * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": wl_config(wl),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


def graph_timings(torch, plan, go, w, gi, flush, calls=20, reps=10):
    """Per-call times from CUDA graphs of `calls` dgrad_run calls, best of
    `reps` replays: back to back (warm L2: inputs, frame and output stay in
    L2 between calls), and each call after the L2-flush fill (cold), less a
    graph of the fills alone.  None if the graphs cannot be captured."""
    def capture(body):
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            body()   # warm-up outside the capture
        torch.cuda.current_stream().wait_stream(side)
        with torch.cuda.graph(g):
            body()
        return g

    def replay_us(g):
        best = float("inf")
        s = torch.cuda.current_stream()
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s)
            g.replay()
            e1.record(s)
            torch.cuda.synchronize()
            best = min(best, e0.elapsed_time(e1) * 1e3)
        return best

    def calls_only():
        for _ in range(calls):
            plan.run(go, w, gi, torch.cuda.current_stream())

    def flushed_calls():
        for _ in range(calls):
            flush.zero_()
            plan.run(go, w, gi, torch.cuda.current_stream())

    def flushes():
        for _ in range(calls):
            flush.zero_()

    try:
        warm = replay_us(capture(calls_only)) / calls
        cold = (replay_us(capture(flushed_calls)) - replay_us(capture(flushes))) / calls
    except Exception as ex:   # capture not possible on this stack: report why, time nothing
        torch.cuda.synchronize()
        return {"error": str(ex).splitlines()[0][:200]}
    plan.check()
    return {"warm_us_per_call": warm, "cold_us_per_call": cold, "calls_per_graph": calls, "replays": reps}


def time_workload(dg, torch, wl, precision, steps, warmup, rank, barrier, device_index, clocks, e2e, **opts):
    from conv2d_backward_implicit_dgrad_gb300.workloads import make_inputs
    go_h, w_h = make_inputs(wl, seed=rank)
    go, w = go_h.cuda(), w_h.cuda()
    gi = torch.empty(wl.gi_shape, device="cuda")
    flush = torch.empty(FLUSH_BYTES // 4, device="cuda")
    plan = dg.Plan(*wl.plan_args(), precision=precision, **opts)
    stream = torch.cuda.current_stream()

    def step():
        plan.run(go, w, gi, stream)   # pack kernel (weights + frame) -> main kernel

    for _ in range(max(3, warmup)):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    plan.check()

    sampler = ClockSampler(device_index) if clocks else None
    if sampler:
        sampler.start()
        # keep the GPU under this load long enough for the sampler to see it
        t_end = time.perf_counter() + 1.0
        while time.perf_counter() < t_end:
            flush.zero_()
            step()
        torch.cuda.synchronize()

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
    torch.cuda.synchronize()
    barrier()
    for i in range(steps):
        flush.zero_()
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    barrier()
    clock_info = sampler.stop() if sampler else None
    plan.check()
    step_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)

    # The stages apart, same flushing: the pack kernels (weights, frame) and
    # then the main kernel alone, each bracketed by events on this stream.
    se = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    for i in range(steps):
        flush.zero_()
        se[i][0].record(stream)
        plan.prepack(w, stream)
        plan.pack_grad_out(go, stream)
        se[i][1].record(stream)
        plan.run_main(go, gi, stream)
        se[i][2].record(stream)
    torch.cuda.synchronize()
    plan.check()
    prepack_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in se)
    main_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in se)
    fused_ms = step_ms

    graph = graph_timings(torch, plan, go, w, gi, flush) if e2e else None

    e2e_s = None
    copy_floor = None
    if e2e:
        go_p, w_p = go_h.pin_memory(), w_h.pin_memory()
        gi_p = torch.empty(wl.gi_shape, pin_memory=True)
        for _ in range(3):
            plan.run_host(go_p, w_p, gi_p, stream)
        ts = []
        for _ in range(max(5, min(steps, 50))):
            flush.zero_()
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            plan.run_host(go_p, w_p, gi_p, stream)   # H2D copies, both kernels, D2H copy, stream sync
            ts.append(time.perf_counter() - t0)
        e2e_s = statistics.mean(ts)
        plan.check()
        # The host link's floor for the same bytes: plain copies of the same
        # pinned buffers (grad_out and W up, grad_input down), one after the
        # other on one stream, and with the download on a second stream.
        go_d, w_d, gi_d = torch.empty_like(go), torch.empty_like(w), torch.empty_like(gi)
        down = torch.cuda.Stream()

        def copies(overlap):
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            go_d.copy_(go_p, non_blocking=True)
            w_d.copy_(w_p, non_blocking=True)
            with torch.cuda.stream(down if overlap else stream):
                gi_p.copy_(gi_d, non_blocking=True)
            torch.cuda.synchronize()
            return time.perf_counter() - t0

        for ov in (False, True):
            copies(ov)
        copy_floor = {ov: statistics.mean(copies(ov) for _ in range(max(5, min(steps, 50)))) for ov in (False, True)}
    info = plan.info
    plan.close()
    return {"ms_per_step": step_ms, "main_ms": main_ms, "prepack_ms": prepack_ms, "fused_ms": fused_ms,
            "e2e_s": e2e_s, "copy_floor_s": copy_floor, "graph": graph, "clocks": clock_info, "plan": info, "flops": info["useful_flops"],
            "bytes": info["algorithmic_bytes"], "steps": steps}


def roofline(wl, precision, flops, nbytes, main_s, step_s, live, plan=None):
    """Roofline of the main kernel.  `live` = measure_peaks(): the TF32 and
    FFMA peaks measured in this run on this GPU; HBM bandwidth from
    MEASURED_PEAKS.json (driver-measured).  `achieved` / `peak` / `frac` are
    in the bound's own unit: GB/s of algorithmic bytes against the HBM peak
    when the workload is bound by HBM at its roofline, else TFLOP/s of useful
    FLOP against the compute peak; `compute` always gives the latter (and the
    nominal-ratio TF32 figure, measured bf16 burst x 1.1/2.25, beside it)."""
    peaks, src = load_peaks()
    hbm = peaks["hbm_gbs"]
    nominal_tf32 = peaks["bf16_tflops"] * TF32_OVER_BF16
    if precision == "tf32":
        peak_tf, alt = live["tf32_tflops"], nominal_tf32
        note = ("TF32 measured in this run: cuBLAS fp32 matmul 8192^3 with TF32, best of 10; "
                f"alt = {src} bf16 burst {peaks['bf16_tflops']} TFLOP/s x nominal 1.1/2.25")
    elif precision == "tf32x3":
        # three TF32 MMAs (hi*lo, lo*hi, hi*hi) per useful product
        peak_tf, alt = live["tf32_tflops"] / 3, nominal_tf32 / 3
        note = "TF32X3 = the TF32 peak measured in this run / 3 MMAs per useful product; alt = nominal-ratio TF32 / 3"
    else:
        peak_tf, alt = live["ffma_tflops"], live["ffma_nominal_tflops"]
        note = (f"FP32 FFMA measured in this run: dgrad_probe_ffma over all {live['sm_count']} SMs, best of 5; "
                f"alt = {live['sm_count']} SMs x 256 FLOP/clk x max SM clock")
    t_flop = flops / (peak_tf * 1e12)
    t_hbm = nbytes / (hbm * 1e9)
    if t_flop >= t_hbm:
        bound = "alu" if precision == "fp32" else "tensor"
    else:
        bound = "hbm"
    achieved_tf = flops / main_s / 1e12
    gbs = nbytes / main_s / 1e9
    if bound == "hbm":
        achieved, peak, unit = gbs, hbm, "GB/s"
    else:
        achieved, peak, unit = achieved_tf, peak_tf, "TFLOP/s"
    rec = recorded_traffic_entry(wl.name, precision)
    if precision != "fp32":
        kernel = "tc_dgrad_kernel"
    else:
        kernel = "simt_pipe_kernel" if plan and plan.get("a_source") == "frame" else "simt_dgrad_kernel"
    return {
        "bound": bound, "achieved": achieved, "peak": peak, "unit": unit, "frac": achieved / peak,
        "traffic": rec.get("dram_bytes_per_launch") if rec else None,
        "traffic_l2_write": rec.get("l2_write_bytes_per_launch") if rec else None,
        "kernel": kernel,
        "compute": {"achieved": achieved_tf, "peak": peak_tf, "unit": "TFLOP/s", "frac": achieved_tf / peak_tf,
                    "peak_alt": alt, "frac_alt": achieved_tf / alt},
        "peak_source": f"{note}; HBM {hbm} GB/s ({src})",
        "roofline_us": max(t_flop, t_hbm) * 1e6,
        "frac_of_roofline_step": max(t_flop, t_hbm) / step_s,
        "frac_of_roofline_kernel": max(t_flop, t_hbm) / main_s,
        "hbm_gbs_achieved_kernel": nbytes / main_s / 1e9,
    }


def slowest_rank(torch, dist, r, device):
    """Replace this rank's times in `r` by the maximum over all ranks (one
    all-reduce of three numbers, outside the timed region).  A rank without an
    end-to-end time contributes 0 to that maximum."""
    t = torch.tensor([r["ms_per_step"], r["main_ms"], r["e2e_s"] or 0.0], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    r["ms_per_step"], r["main_ms"], e2e_s = t.tolist()
    r["e2e_s"] = e2e_s or None
    return r


def build_line(args, wl, r, world):
    flops, nbytes = r["flops"], r["bytes"]
    step_s, main_s = r["ms_per_step"] * 1e-3, r["main_ms"] * 1e-3
    value = world * flops / step_s / 1e12
    go_b = 4 * wl.N * wl.Co * wl.oH * wl.oW
    w_b = 4 * wl.Co * wl.Ci * wl.kH * wl.kW
    gi_b = 4 * wl.N * wl.Ci * wl.H * wl.W
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": r["steps"],
        "warmup": args.warmup, "ms_per_step": r["ms_per_step"], "us_per_call": r["ms_per_step"] * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": args.precision, "data": "synthetic",
        "config": {**wl_config(wl), "precision": args.precision, "parallelism": f"replicas x{world}",
                   "l2": "flushed (256 MiB write) before every timed step",
                   "step": "pack kernel (weights + grad_out frame) + main kernel (C ABI dgrad_run)"},
        "roofline": roofline(wl, args.precision, flops, nbytes, main_s, step_s, r["peaks"], r["plan"]),
        "main_kernel_us": r["main_ms"] * 1e3, "pack_stages_us": r["prepack_ms"] * 1e3,
        "peaks_measured": {k: r["peaks"][k] for k in ("tf32_tflops", "ffma_tflops", "sm_count")},
        "gpu_launches": 2 * r["steps"],
        "plan": {k: r["plan"][k] for k in ("path", "tile_blocks", "slice_n", "chunk_k", "n_chunks", "grid",
                                           "n_work", "b_resident", "smem_bytes", "tmem_cols")},
        "clocks": r["clocks"],
    }
    if r["e2e_s"]:
        line["e2e"] = {"value": world * flops / r["e2e_s"] / 1e12, "unit": "TFLOP/s",
                       "h2d_bytes_per_step": go_b + w_b, "d2h_bytes_per_step": gi_b,
                       "us_per_call": r["e2e_s"] * 1e6, "api": "dgrad_run_host (pinned host buffers)"}
        if r.get("graph"):
            line["graph"] = dict(r["graph"], method="CUDA graphs of dgrad_run calls, best of the replays; warm: "
                                 "back to back; cold: each call after the 256 MiB L2-flush fill, less a graph of "
                                 "the fills alone")
        if r.get("copy_floor_s"):
            # plain pinned copies of the same bytes, no kernels: the host link's floor
            line["e2e"]["copy_floor_us"] = {"serial": r["copy_floor_s"][False] * 1e6,
                                            "up_and_down_overlapped": r["copy_floor_s"][True] * 1e6}
    return line


def time_wgrad(dg, torch, wl, steps, warmup, precision="tf32"):
    """The weight gradient of the same convolution (grad_out and the forward
    input, seeded), each step after the same L2 flush, CUDA events around
    wgrad_run (frame pack, tcgen05 split-K GEMM, reduction)."""
    from conv2d_backward_implicit_dgrad_gb300.workloads import make_inputs
    go_h, _ = make_inputs(wl, seed=0)
    x_h = torch.randn((wl.N, wl.Ci, wl.H, wl.W), generator=torch.Generator().manual_seed(1))
    go, x = go_h.cuda(), x_h.cuda()
    dw = torch.empty((wl.Co, wl.Ci, wl.kH, wl.kW), device="cuda")
    flush = torch.empty(FLUSH_BYTES // 4, device="cuda")
    stream = torch.cuda.current_stream()
    with dg.WgradPlan(*wl.plan_args(), precision=precision) as plan:
        for _ in range(max(3, warmup)):
            flush.zero_()
            plan.run(go, x, dw, stream)
        torch.cuda.synchronize()
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
        for i in range(steps):
            flush.zero_()
            ev[i][0].record(stream)
            plan.run(go, x, dw, stream)
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        plan.check()
        info = plan.info
    ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
    return {"ms_per_step": ms, "flops": info["useful_flops"], "bytes": info["algorithmic_bytes"], "plan": info}


def profile_steps(dg, torch, wl, args):
    """W warm-up steps then K steps (dgrad_run), each after an L2 flush; nothing else."""
    from conv2d_backward_implicit_dgrad_gb300.workloads import make_inputs
    go_h, w_h = make_inputs(wl, 0)
    go, w = go_h.cuda(), w_h.cuda()
    flush = torch.empty(FLUSH_BYTES // 4, device="cuda")
    if args.op == "wgrad":
        x = torch.randn((wl.N, wl.Ci, wl.H, wl.W), generator=torch.Generator().manual_seed(1)).cuda()
        dw = torch.empty((wl.Co, wl.Ci, wl.kH, wl.kW), device="cuda")
        with dg.WgradPlan(*wl.plan_args(), precision=args.precision) as plan:
            for _ in range(args.warmup + args.steps):
                flush.zero_()
                plan.run(go, x, dw)
            torch.cuda.synchronize()
            plan.check()
            print(json.dumps({"profile": wl.name, "op": "wgrad", "steps": args.steps, "warmup": args.warmup,
                              "plan": plan.info}), flush=True)
        return 0
    gi = torch.empty(wl.gi_shape, device="cuda")
    with dg.Plan(*wl.plan_args(), precision=args.precision, path=args.path) as plan:
        for _ in range(args.warmup + args.steps):
            flush.zero_()
            plan.run(go, w, gi)
        torch.cuda.synchronize()
        plan.check()
        print(json.dumps({"profile": wl.name, "precision": args.precision, "steps": args.steps,
                          "warmup": args.warmup, "plan": plan.info}), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="resnet_stage")
    ap.add_argument("--precision", default="tf32", choices=["tf32", "tf32x3", "fp32"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--all", action="store_true", help="also print one info line per workload and precision")
    ap.add_argument("--op", default="dgrad", choices=["dgrad", "wgrad"],
                    help="with --profile: which operation's kernels run")
    ap.add_argument("--path", default="auto", choices=["auto", "simt", "tcgen05", "col2im"],
                    help="with --profile: the dgrad kernel family (auto: the plan's own choice)")
    ap.add_argument("--profile", action="store_true",
                    help="only run W + K steps (for ncu captures: few launches, no extra timing loops)")
    args = ap.parse_args()

    from conv2d_backward_implicit_dgrad_gb300.workloads import WORKLOADS
    wl = WORKLOADS[args.workload]
    if args.impl == "reference":
        return reference_arm(args, wl)

    import torch
    import torch.distributed as dist
    import conv2d_backward_implicit_dgrad_gb300 as dg

    if args.profile:
        return profile_steps(dg, torch, wl, args)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    def barrier():
        if world > 1:
            dist.barrier()

    r = time_workload(dg, torch, wl, args.precision, args.steps, args.warmup, rank, barrier, local,
                      clocks=True, e2e=True)
    r["peaks"] = measure_peaks(torch, dg)   # after the timed region: it does not heat the GPU before it
    if world > 1:
        slowest_rank(torch, dist, r, "cuda")

    if rank == 0:
        line = build_line(args, wl, r, world)
        if world == 1 and wl.name == "resnet_stage" and args.precision == "tf32" and not args.all:
            # the other target workloads, TF32, same method (flushed steps, events); informational
            line["other_configs"] = []
            for name in ("strided_downsample", "pointwise", "stem"):
                x = time_workload(dg, torch, WORKLOADS[name], "tf32", 50, 5, rank, lambda: None, local,
                                  clocks=False, e2e=False)
                rf = roofline(WORKLOADS[name], "tf32", x["flops"], x["bytes"], x["main_ms"] * 1e-3,
                              x["ms_per_step"] * 1e-3, r["peaks"], x["plan"])
                line["other_configs"].append({
                    "workload": name, "precision": "tf32", "us_per_call": x["ms_per_step"] * 1e3,
                    "tflops": x["flops"] / (x["ms_per_step"] * 1e-3) / 1e12, "main_kernel_us": x["main_ms"] * 1e3,
                    "roofline": {k: rf[k] for k in ("bound", "achieved", "peak", "unit", "frac", "roofline_us")},
                    "compute_frac": rf["compute"]["frac"]})
        if world == 1 and not args.no_cpu_baseline:
            flops, times, cores = cpu_oracle_run(wl, wl.N, reps=2)
            line["cpu_baseline"] = {
                "value": flops / min(times) / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                "sample": f"the whole batch ({wl.N} images) of {wl.name}, fp64 scatter oracle, "
                          f"best of {len(times)}"}
            one = min(wl.N, 2)
            f1, t1, _ = cpu_oracle_run(wl, one, reps=2, threads=1)
            line["cpu_baseline"]["single_thread"] = {
                "value": f1 / min(t1) / 1e12, "unit": "TFLOP/s", "cores": 1,
                "sample": f"{one} images of {wl.name}, one thread, best of {len(t1)}"}
        print(json.dumps(line), flush=True)
        if args.all:
            for name in WORKLOAD_ORDER:
                for prec in ("tf32", "tf32x3", "fp32"):
                    x = time_workload(dg, torch, WORKLOADS[name], prec, 10 if prec == "fp32" else 50, 5, rank,
                                      lambda: None, local, clocks=False, e2e=False)
                    rf = roofline(WORKLOADS[name], prec, x["flops"], x["bytes"], x["main_ms"] * 1e-3,
                                  x["ms_per_step"] * 1e-3, r["peaks"], x["plan"])
                    print(json.dumps({"info": "workload", "workload": name, "precision": prec,
                                      **{k: x[k] for k in ("ms_per_step", "main_ms", "prepack_ms")},
                                      "tflops": x["flops"] / (x["ms_per_step"] * 1e-3) / 1e12,
                                      "main_tflops": rf["compute"]["achieved"], "frac_peak": rf["compute"]["frac"],
                                      "frac_of_roofline_kernel": rf["frac_of_roofline_kernel"],
                                      "plan": {k: x["plan"][k] for k in ("path", "tile_blocks", "slice_n",
                                                                         "chunk_k", "grid", "n_work",
                                                                         "b_resident", "smem_bytes")}}),
                          flush=True)
            # the opt-in GEMM + col2im path on the few-input-channel stem
            x = time_workload(dg, torch, WORKLOADS["stem"], "tf32", 50, 5, rank, lambda: None, local, clocks=False,
                              e2e=False, path="col2im")
            rf = roofline(WORKLOADS["stem"], "tf32", x["flops"], x["bytes"], x["main_ms"] * 1e-3,
                          x["ms_per_step"] * 1e-3, r["peaks"])
            print(json.dumps({"info": "workload", "workload": "stem", "precision": "tf32", "path": "col2im",
                              **{k: x[k] for k in ("ms_per_step", "main_ms", "prepack_ms")},
                              "tflops": x["flops"] / (x["ms_per_step"] * 1e-3) / 1e12,
                              "main_tflops": rf["compute"]["achieved"], "frac_peak": rf["compute"]["frac"],
                              "frac_of_roofline_kernel": rf["frac_of_roofline_kernel"]}), flush=True)
            tf32_peak = r["peaks"]["tf32_tflops"]
            for name, prec in [(n, p) for p in ("tf32", "tf32x3") for n in WORKLOAD_ORDER]:
                x = time_wgrad(dg, torch, WORKLOADS[name], 50, 5, prec)
                tf = x["flops"] / (x["ms_per_step"] * 1e-3) / 1e12
                print(json.dumps({"info": "wgrad", "workload": name, "precision": prec,
                                  "ms_per_step": x["ms_per_step"], "tflops": tf, "frac_peak": tf / tf32_peak,
                                  "plan": {k: x["plan"][k] for k in ("n_mt", "n_nt", "n_ks", "slice_n", "n_units",
                                                                     "grid", "stages", "n_copies")}}),
                      flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
