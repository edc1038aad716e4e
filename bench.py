"""Benchmark: SGEMM TFLOPS (2MNK / device time) on GB300, one JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload square8192|rowmajor4096|...] [--modes ffma,tf32,3xtf32]

A step is one pass of the hot path over one synthetic problem: one sgemm call
per arithmetic mode (FFMA, TF32, 3xTF32) on the same resident inputs.  The
default workload is the 8192^3 column-major product with alpha = 1, beta = 1
and A, B, Cin ~ U[-1, 1) drawn from seed 0 (the size at which the targets are
stated).  Inputs (768 MiB) exceed the 129 MB L2, so no flush is needed between
iterations.  With --gpus N > 1 (under torchrun) every rank runs the same
problem on its own GPU: replicas, no collective on the data path; value is the
total over ranks divided by the slowest rank's time.

--impl reference times the CPU oracle (plain C, double accumulation) on the same
workload, over a bounded sample of output entries per step.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from precision_gemm_gb300 import synth  # noqa: E402

WORKLOADS = {
    "square8192": ("sgemm column-major NN 8192^3, alpha=1 beta=1, A,B,Cin ~ U[-1,1) seed 0",
                   synth.Problem(8192, 8192, 8192, alpha=1.0, beta=1.0, dist="uniform", seed=0)),
    "square16384": ("sgemm column-major NN 16384^3, alpha=1 beta=1, A,B,Cin ~ U[-1,1) seed 0",
                    synth.Problem(16384, 16384, 16384, alpha=1.0, beta=1.0, dist="uniform", seed=0)),
    "square4096": ("sgemm column-major NN 4096^3, alpha=1 beta=1, A,B,Cin ~ U[-1,1) seed 0",
                   synth.Problem(4096, 4096, 4096, alpha=1.0, beta=1.0, dist="uniform", seed=0)),
    "rowmajor4096": ("sgemm row-major 4096^3, alpha=1 beta=0, A,B ~ U[-1,1) seed 0",
                     synth.Problem(4096, 4096, 4096, alpha=1.0, beta=0.0, dist="uniform", seed=0, layout="row")),
    "rowmajor2048": ("sgemm row-major 2048^3, alpha=1 beta=0, A,B ~ U[-1,1) seed 0",
                     synth.config_problems()["c2_rm2048"]),
    "rowmajor1024": ("sgemm row-major 1024^3, alpha=1 beta=0, A,B ~ U[-1,1) seed 0",
                     synth.config_problems()["c2_rm1024"]),
    "ragged": ("sgemm column-major 3000x1500x777, lda=3013 ldb=784 ldc=3005, alpha=1.5 beta=-0.5, N(0,1)",
               synth.config_problems()["c3_ragged"]),
    "skinny_k64": ("sgemm column-major 16384x16384x64, N(0,1)", synth.config_problems()["c5a_16384x16384x64"]),
    "splitk_262144": ("sgemm column-major 128x128x262144, N(0,1)", synth.config_problems()["c5b_128x128x262144"]),
    "tall_thin": ("sgemm column-major 8192x64x8192, N(0,1)", synth.config_problems()["c5c_8192x64x8192"]),
}

# Nominal ratio of dense TF32 to dense BF16 tensor throughput (1.1 / 2.25 PFLOP/s).
TF32_PER_BF16 = 1.1 / 2.25
# TF32 flops per clock per SM of tcgen05 (2048 FMA): the register/TMEM-only probe
# (probes/tf32_ceiling.cu, `bench.py --tf32-ceiling`) measured 4090 on GB300.
TF32_FLOPS_PER_CLK_SM = 4096
# The acceptance workloads timed after the headline step, one entry each (the
# 8192^3 product is the headline itself).
SWEEP = ("c1_256", "c2_rm1024", "c2_rm2048", "c2_rm4096", "c3_ragged", "c4_16384", "c5a_16384x16384x64",
         "c5b_128x128x262144", "c5c_8192x64x8192")
L2_FLUSH_BYTES = 512 << 20  # > 2x the 129 MB L2
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "sm_max_mhz": 2070.0}


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            d = json.load(fh)
        return d, "measured"
    except Exception:
        return dict(FALLBACK), "fallback"


def fp32_alu_peak_tflops(num_sms: int, mhz: float) -> float:
    """CUDA-core FP32 FMA peak: SMs x 128 FP32 lanes x 2 flops x clock."""
    return num_sms * 128 * 2 * mhz * 1e6 / 1e12


def tensor_pipe_tflops(num_sms: int, mhz: float) -> float:
    """TF32 tensor-pipe peak: SMs x 4096 flops/clk (measured by the probe) x clock."""
    return num_sms * TF32_FLOPS_PER_CLK_SM * mhz * 1e6 / 1e12


def alg_bytes(p) -> int:
    """A and B read once, C written, C read when beta != 0 (4 B each)."""
    return (p.m * p.k + p.k * p.n + p.m * p.n * (2 if p.beta != 0 else 1)) * 4


def make_config(wl_name: str, p, modes, world: int) -> dict:
    """The `config` object of both arms' JSON lines (identical keys and values)."""
    desc = WORKLOADS[wl_name][0]
    return {"workload": desc, "name": wl_name, "m": p.m, "n": p.n, "k": p.k, "modes": list(modes),
            "layout": p.layout, "parallelism": "replicas" if world > 1 else "single GPU",
            "l2": "inputs larger than L2 (no flush)" if alg_bytes(p) > 129e6 else "L2 not flushed; inputs fit"}


def mode_figures(mode: str, p, ms: float, peaks: dict) -> dict:
    """TFLOP/s of one call and its fractions: of the mode's compute peak, of the
    roofline min(compute peak, AI x HBM), and (tensor-core modes) of the TF32
    tensor pipe at the maximum SM clock, counting 3xTF32's three products."""
    flops = p.flops()
    tflops = flops / (ms * 1e-3) / 1e12
    compute = {"ffma": peaks["fp32"], "tf32": peaks["tf32"], "3xtf32": peaks["tf32"] / 3.0}[mode]
    hbm_roof = (flops / alg_bytes(p)) * peaks["hbm"] / 1e3  # AI [flop/B] x HBM [GB/s] -> TFLOP/s
    roof = min(compute, hbm_roof)
    out = {"ms_median": ms, "tflops": tflops, "compute_peak_tflops": compute,
           "frac_of_compute_peak": tflops / compute, "bound": "hbm" if hbm_roof < compute else "compute",
           "roofline_tflops": roof, "frac_of_roofline": tflops / roof}
    if mode != "ffma":
        out["frac_of_tensor_pipe"] = tflops * (3 if mode == "3xtf32" else 1) / peaks["pipe"]
    return out


# ----------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.3)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as fh:
            for line in fh:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        loaded = [x for x in sm if mx and x > 0.5 * max(mx)] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ----------------------------------------------------------------- our arm

def run_ours(args, wl_name):
    import precision_gemm_gb300 as pg

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    pg.load_library()
    desc, p = WORKLOADS[wl_name]
    modes = [m for m in args.modes.split(",") if m]
    A, B, C = synth.make(p)
    dA, dB, dC0 = A.cuda(), B.cuda(), C.cuda()
    dC = dC0.clone()
    stream = torch.cuda.current_stream()
    flops = p.flops()
    props = torch.cuda.get_device_properties(local)
    num_sms = props.multi_processor_count

    def call(mode, Cbuf):
        if p.layout == "col":
            pg.sgemm(p.transa, p.transb, p.m, p.n, p.k, p.alpha, dA, p.lda, dB, p.ldb, p.beta, Cbuf, p.ldc, mode,
                     stream)
        else:
            pg.sgemm_rm(p.m, p.n, p.k, p.alpha, dA, p.lda, dB, p.ldb, p.beta, Cbuf, p.ldc, mode, stream)

    def step(events=None):
        for mode in modes:
            if events is not None:
                events[mode][0].record(stream)
            call(mode, dC)
            if events is not None:
                events[mode][1].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if pg.device_status() != 0:
        raise RuntimeError("a kernel reported a failed bounded wait during warm-up")

    evs = [{m: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for m in modes}
           for _ in range(args.steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local) if rank == 0 else None
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    if clocks:
        clocks.start()
        time.sleep(0.4)
    launches0 = pg.launch_count()
    start.record(stream)
    for i in range(args.steps):
        step(evs[i])
    end.record(stream)
    torch.cuda.synchronize()
    launches = pg.launch_count() - launches0
    if dist:
        dist.barrier()
    clk = clocks.stop() if clocks else None
    total_ms = start.elapsed_time(end)
    per_mode_ms = {m: [evs[i][m][0].elapsed_time(evs[i][m][1]) for i in range(args.steps)] for m in modes}
    status = pg.device_status()

    t = torch.tensor([total_ms], dtype=torch.float64, device="cuda")
    if dist:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    total_ms = float(t.item())

    # End to end through the public host-buffer entry point: pinned host inputs,
    # every step copies A, B (and Cin when beta != 0) in and C out for each mode.
    # The modes' calls are queued with sgemm_host_async on one stream each, so one
    # call's copies overlap another's arithmetic; the step ends when all are done.
    e2e = None
    if not args.skip_e2e:
        hA, hB = A.pin_memory(), B.pin_memory()
        hCs = {mode: C.clone().pin_memory() for mode in modes}  # each call reads and writes its own C
        hstreams = {mode: torch.cuda.Stream() for mode in modes}
        h2d = (A.numel() + B.numel() + (C.numel() if p.beta != 0 else 0)) * 4 * len(modes)
        d2h = p.m * p.n * 4 * len(modes)

        def host_step():
            go = torch.cuda.Event()
            go.record(stream)
            for mode in modes:
                s = hstreams[mode]
                s.wait_event(go)
                if p.layout == "col":
                    pg.sgemm_host_async(p.transa, p.transb, p.m, p.n, p.k, p.alpha, hA, p.lda, hB, p.ldb, p.beta,
                                        hCs[mode], p.ldc, mode, s)
                else:
                    pg.sgemm_host_async("N", "N", p.n, p.m, p.k, p.alpha, hB, p.ldb, hA, p.lda, p.beta, hCs[mode],
                                        p.ldc, mode, s)
            for mode in modes:
                stream.wait_stream(hstreams[mode])
        for _ in range(max(1, min(args.warmup, 2))):
            host_step()
        # each step timed on its own (events on the launching stream); the median
        # step stands for the run, the slowest and fastest are reported beside it
        e_steps = max(1, min(args.steps, 5))
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        e_ms = []
        for _ in range(e_steps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            host_step()
            e1.record(stream)
            e1.synchronize()
            e_ms.append(e0.elapsed_time(e1))
        te = torch.tensor([statistics.median(e_ms)], dtype=torch.float64, device="cuda")
        if dist:
            dist.all_reduce(te, op=dist.ReduceOp.MAX)
        e2e = {"value": world * flops * len(modes) / (float(te.item()) * 1e-3) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e_steps,
               "ms_per_step": float(te.item()), "ms_min": min(e_ms), "ms_max": max(e_ms),
               "api": "sgemm_host_async, one stream per mode (pinned host buffers)"}

    # The hybrid CPU + GPU column split, end to end through the synchronous host
    # entry: per mode, calls with the automatic ratio (warm-up calls let it settle
    # on the measured speed ratio) against the same calls with the split off.
    hybrid = None
    if args.host_split and world == 1 and not args.skip_e2e:
        hA, hB = A.pin_memory(), B.pin_memory()
        hC = C.clone().pin_memory()

        def host_calls(reps):
            t0 = time.perf_counter()
            for _ in range(reps):
                if p.layout == "col":
                    pg.sgemm_host(p.transa, p.transb, p.m, p.n, p.k, p.alpha, hA, p.lda, hB, p.ldb, p.beta, hC,
                                  p.ldc, mode, stream)
                else:
                    pg.sgemm_host("N", "N", p.n, p.m, p.k, p.alpha, hB, p.ldb, hA, p.lda, p.beta, hC, p.ldc, mode,
                                  stream)
            return (time.perf_counter() - t0) / reps
        hybrid = {"api": "sgemm_host (synchronous, pinned host buffers), one call per mode; host time per call",
                  "modes": {}}
        for mode in modes:
            pg.set_host_split(0.0)
            host_calls(1)
            t_off = host_calls(3)
            pg.set_host_split(-1.0)
            host_calls(4)  # the automatic ratio settles on the measured speeds
            t_on = host_calls(3)
            q = pg.host_split_ratio(mode)
            pg.set_host_split(0.0)
            n_cpu = int(p.n // (q + 1.0)) if p.layout == "col" else int(p.m // (q + 1.0))
            hybrid["modes"][mode] = {"q": q, "cpu_columns": n_cpu, "ms_split_off": t_off * 1e3,
                                     "ms_split_auto": t_on * 1e3, "tflops_split_off": flops / t_off / 1e12,
                                     "tflops_split_auto": flops / t_on / 1e12}

    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return None

    peaks, peak_src = measured_peaks()
    sm_max = float(peaks.get("sm_max_mhz") or FALLBACK["sm_max_mhz"])
    fp32_peak = fp32_alu_peak_tflops(num_sms, sm_max)
    tf32_peak = float(peaks.get("bf16_tflops") or FALLBACK["bf16_tflops"]) * TF32_PER_BF16
    hbm = float(peaks.get("hbm_gbs") or FALLBACK["hbm_gbs"])
    pk = {"fp32": fp32_peak, "tf32": tf32_peak, "hbm": hbm, "pipe": tensor_pipe_tflops(num_sms, sm_max)}
    mode_info = {}
    for m in modes:
        ms = statistics.median(per_mode_ms[m])
        mode_info[m] = mode_figures(m, p, ms, pk)
        mode_info[m]["ms_min"] = min(per_mode_ms[m])
        tflops = mode_info[m]["tflops"]
        if clk and clk.get("sm_mhz") and m == "ffma":
            mode_info[m]["frac_of_peak_at_run_clock"] = tflops / fp32_alu_peak_tflops(num_sms, clk["sm_mhz"])
        if clk and clk.get("sm_mhz") and m != "ffma":
            mode_info[m]["frac_of_tensor_pipe_at_run_clock"] = (
                tflops * (3 if m == "3xtf32" else 1) / tensor_pipe_tflops(num_sms, clk["sm_mhz"]))

    # Dominant kernel: the mode whose launches take longest in the step.
    dom = max(modes, key=lambda m: mode_info[m]["ms_median"])
    dplan = pg.sgemm_plan(p.transa, p.transb, p.m, p.n, p.k, p.alpha, 256, p.lda, 256, p.ldb, p.beta, 256, p.ldc,
                          dom, num_sms)
    kname, tile = dplan["kernel_name"], "%dx%d" % (dplan["bm"], dplan["bn"])
    dom_kernel = "%s_gemm_kernel (%s%s tiles)" % (kname, "" if dom == "ffma" else dom + ", ", tile)
    traffic = read_traffic(dom, kname, tile, wl_name)
    if dom == "ffma":
        roofline = {"bound": "alu", "achieved": mode_info[dom]["tflops"], "peak": fp32_peak, "unit": "TFLOP/s",
                    "frac": mode_info[dom]["tflops"] / fp32_peak,
                    "peak_source": "derived: %d SMs x 128 FP32 lanes x 2 x %.0f MHz (%s max SM clock)"
                                   % (num_sms, sm_max, peak_src)}
    else:
        dom_peak = tf32_peak if dom == "tf32" else tf32_peak / 3.0
        roofline = {"bound": "tensor", "achieved": mode_info[dom]["tflops"], "peak": dom_peak, "unit": "TFLOP/s",
                    "frac": mode_info[dom]["tflops"] / dom_peak,
                    "peak_source": "%s bf16 burst x %.3f (nominal tf32/bf16)%s" % (
                        peak_src, TF32_PER_BF16, " / 3" if dom == "3xtf32" else "")}
    roofline["kernel"] = dom_kernel
    roofline["traffic"] = traffic

    sweep = None
    if not args.no_sweep and world == 1:  # per-workload timings: single-GPU runs only
        # the headline step's buffers are no longer needed
        del dA, dB, dC0, dC
        torch.cuda.empty_cache()
        sweep = run_sweep(args, modes, pk, stream)

    value = world * flops * len(modes) / (total_ms / args.steps * 1e-3) / 1e12
    line = {
        "metric": "SGEMM TFLOPS (2MNK/s) at 4096^3/8192^3 fp32; % of FP32 & TF32 peak",
        "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": total_ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic (seeded CPU draws: A, B and C_in in storage order, padding set to NaN)",
        "config": make_config(wl_name, p, modes, world),
        "modes": mode_info, "roofline": roofline, "e2e": e2e, "gpu_launches": launches,
        "device_status": status, "clocks": clk, "gpu": torch.cuda.get_device_name(local), "sms": num_sms,
        "tensor_pipe_peak": {"tflops": pk["pipe"], "source": "%d SMs x %d TF32 flops/clk/SM (probe-measured) x "
                                                             "%.0f MHz" % (num_sms, TF32_FLOPS_PER_CLK_SM, sm_max)},
    }
    if sweep is not None:
        line["workloads"] = sweep
    if hybrid is not None:
        line["e2e_host_split"] = hybrid
    if not args.skip_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(p, args.cpu_seconds, args.cpu_threads)
    if dist:
        dist.destroy_process_group()
    return line


def run_sweep(args, modes, pk, stream):
    """Every acceptance workload besides the headline: per mode, W warm-up calls
    and a few timed calls (CUDA events on the launching stream around each call).
    A workload whose algorithmic bytes exceed the L2 runs back to back (inputs
    larger than L2).  A smaller one gets an L2 flush before each timed call,
    outside the timed interval: a 512 MiB buffer is written, then a 256 MiB one
    read, so that the flush's dirty lines are written back before the call
    instead of during it.  Returns {name: entry}."""
    import precision_gemm_gb300 as pg
    cfg = synth.config_problems()
    reps = max(3, min(args.steps, args.sweep_reps))
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    evict = torch.empty(L2_FLUSH_BYTES // 8, dtype=torch.float32, device="cuda").zero_()
    out = {}
    for name in SWEEP:
        p = cfg[name]
        A, B, C = synth.make(p)
        dA, dB, dC = A.cuda(), B.cuda(), C.cuda()

        def call(mode):
            if p.layout == "col":
                pg.sgemm(p.transa, p.transb, p.m, p.n, p.k, p.alpha, dA, p.lda, dB, p.ldb, p.beta, dC, p.ldc, mode,
                         stream)
            else:
                pg.sgemm_rm(p.m, p.n, p.k, p.alpha, dA, p.lda, dB, p.ldb, p.beta, dC, p.ldc, mode, stream)
        big = alg_bytes(p) > 129e6
        entry = {"m": p.m, "n": p.n, "k": p.k, "layout": p.layout, "alpha": p.alpha, "beta": p.beta,
                 "lda": p.lda, "ldb": p.ldb, "ldc": p.ldc, "dist": p.dist, "reps": reps,
                 "l2": ("inputs larger than L2 (no flush)" if big else
                        "flushed before each timed call (512 MiB written, then 256 MiB read)"), "modes": {}}
        for mode in modes:
            for _ in range(args.warmup):
                call(mode)
            times = []
            for _ in range(reps):
                if not big:
                    flush.zero_()
                    evict.sum()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                call(mode)
                e1.record(stream)
                e1.synchronize()
                times.append(e0.elapsed_time(e1))
            entry["modes"][mode] = mode_figures(mode, p, statistics.median(times), pk)
            entry["modes"][mode]["ms_min"] = min(times)
        out[name] = entry
        del dA, dB, dC
    del flush, evict
    torch.cuda.empty_cache()
    if pg.device_status() != 0:
        raise RuntimeError("a kernel reported a failed bounded wait during the workload sweep")
    return out


def read_traffic(mode: str, kname: str, tile: str, wl_name: str):
    """DRAM bytes per launch of the dominant kernel from the committed ncu summary
    (profiles/<mode>_<workload>.md: 'traffic_bytes_per_launch: N' plus the tile shape
    and the hash of the kernel source it was taken on); None when absent, or taken
    on a different source or tile shape."""
    import hashlib
    src = "%s_kernel.cu" % kname
    path = os.path.join(ROOT, "profiles", "%s_%s.md" % (mode, wl_name))
    try:
        text = open(path).read()
    except OSError:
        return None
    digest = hashlib.sha256(open(os.path.join(ROOT, "precision_gemm_gb300", "csrc", src), "rb").read()).hexdigest()
    fields = dict(line.split(":", 1) for line in text.splitlines() if ":" in line and not line.startswith("#"))
    if fields.get("source_sha256", "").strip() != digest or fields.get("tile", "").strip() != tile:
        return None
    try:
        return int(fields["traffic_bytes_per_launch"].strip())
    except (KeyError, ValueError):
        return None


# ----------------------------------------------------------------- oracle timing

def cpu_baseline(p, seconds: float, threads: int):
    """The oracle as it stands, on a bounded sample of the same workload: entries
    drawn as in the sampled parity checks, count sized to ~`seconds` of CPU work."""
    import oracle
    O = oracle.Oracle()
    nthreads = threads or O.max_threads()
    A, B, C = synth.make(p)
    args, _ = (((p.transa, p.transb, p.m, p.n, p.k, p.alpha, A, p.lda, B, p.ldb, p.beta, C, p.ldc), False)
               if p.layout == "col" else
               (("N", "N", p.n, p.m, p.k, p.alpha, B, p.ldb, A, p.lda, p.beta, C, p.ldc), True))
    mm, nn = args[2], args[3]
    rng = np.random.default_rng(2024)
    count = max(nthreads, 64)
    while True:
        ii = rng.integers(0, mm, size=count)
        jj = rng.integers(0, nn, size=count)
        t0 = time.perf_counter()
        O.entries(*args, ii, jj, threads=nthreads)
        dt = time.perf_counter() - t0
        if dt >= 0.25 * seconds or count >= mm * nn:
            break
        count = int(min(mm * nn, count * max(2.0, 0.5 * seconds / max(dt, 1e-3))))
    flops = 2.0 * p.k * count
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": nthreads, "kind": "oracle",
            "sample": "%d output entries of the %dx%dx%d problem (%.1f s, %d threads)" % (count, p.m, p.n, p.k, dt,
                                                                                          nthreads)}


def run_reference(args, wl_name):
    """The reference arm: the CPU oracle, timed on host cores, on our config."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return None
    import oracle
    oracle.build()
    desc, p = WORKLOADS[wl_name]
    O = oracle.Oracle()
    nthreads = args.cpu_threads or O.max_threads()
    A, B, C = synth.make(p)
    args_o = ((p.transa, p.transb, p.m, p.n, p.k, p.alpha, A, p.lda, B, p.ldb, p.beta, C, p.ldc)
              if p.layout == "col" else ("N", "N", p.n, p.m, p.k, p.alpha, B, p.ldb, A, p.lda, p.beta, C, p.ldc))
    mm, nn = args_o[2], args_o[3]
    rng = np.random.default_rng(7)
    budget = (args.ref_step_seconds if args.ref_step_seconds else
              max(2.0, min(15.0, 150.0 / max(1, args.steps + args.warmup))))
    probe = max(nthreads, 64)
    t0 = time.perf_counter()
    O.entries(*args_o, rng.integers(0, mm, probe), rng.integers(0, nn, probe), threads=nthreads)
    per_entry = (time.perf_counter() - t0) / probe
    count = int(max(probe, min(mm * nn, budget / max(per_entry, 1e-9))))
    times = []
    for s in range(args.warmup + args.steps):
        ii, jj = rng.integers(0, mm, count), rng.integers(0, nn, count)
        t0 = time.perf_counter()
        O.entries(*args_o, ii, jj, threads=nthreads)
        if s >= args.warmup:
            times.append(time.perf_counter() - t0)
    step_s = sum(times) / len(times)
    value = 2.0 * p.k * count / step_s / 1e12
    sample = "%d output entries per step of the %dx%dx%d problem, %d threads" % (count, p.m, p.n, p.k, nthreads)
    return {"impl": "reference", "metric": "SGEMM TFLOPS (2MNK/s) at 4096^3/8192^3 fp32; % of FP32 & TF32 peak",
            "value": value, "unit": "TFLOP/s", "n_gpus": int(os.environ.get("WORLD_SIZE", "1")),
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_s * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded, same buffers as the GPU arm)",
            "config": make_config(wl_name, p, [m for m in args.modes.split(",") if m],
                                  int(os.environ.get("WORLD_SIZE", "1"))),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": nthreads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="square8192")
    ap.add_argument("--modes", default="ffma,tf32,3xtf32")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--cpu-threads", type=int, default=0)
    ap.add_argument("--skip-e2e", action="store_true")
    ap.add_argument("--skip-cpu-baseline", action="store_true")
    ap.add_argument("--host-split", type=int, default=1,
                    help="1: also time the hybrid CPU + GPU column split of sgemm_host end to end (0: skip)")
    ap.add_argument("--no-sweep", action="store_true",
                    help="skip the per-workload timings of the other acceptance configs")
    ap.add_argument("--sweep-reps", type=int, default=5, help="timed calls per mode and workload in the sweep")
    ap.add_argument("--ref-step-seconds", type=float, default=0.0,
                    help="reference arm: CPU seconds per step (default: the run bounded to ~150 s)")
    ap.add_argument("--fma-ceiling", action="store_true",
                    help="run only the register-only FP32 FMA throughput probe and print its JSON line")
    ap.add_argument("--tf32-ceiling", action="store_true",
                    help="run only the shared-memory-resident tcgen05 TF32 throughput probe and print its JSON line")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)  # timing rule: at least three untimed warm-up steps
    if args.fma_ceiling or args.tf32_ceiling:
        from precision_gemm_gb300 import build as pgbuild
        subprocess.run([pgbuild.build_probe("fma_ceiling" if args.fma_ceiling else "tf32_ceiling")], check=True)
        return
    if args.impl == "reference":
        line = run_reference(args, args.workload)
    else:
        line = run_ours(args, args.workload)
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
