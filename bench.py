#!/usr/bin/env python3
"""Benchmark of the fp16 GEMM C = A . B^T on GB300.

One step = one GEMM of the workload (default: the 8192^3, fp16-output
workload with uniform[-1, 1] operands from seed 2) through the C ABI, with the
operands resident in device memory.  Prints one JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME]
                  [--variant V] [--depth D] [--block-n BN] [--impl ours|reference]

Timing: W untimed warm-up steps, then exactly K steps bracketed by a barrier
and a device synchronise on both sides, timed with two CUDA events on the
launch stream around the K back-to-back launches; max over ranks.  The
operands (A + B = 256 MiB at 8192^3) and the output (128 MiB) are larger than
the 126 MiB L2, so no flush is inserted.

The environment variables GEMM_VARIANT and GEMM_PIPE_DEPTH, when set, give
the defaults of --variant and --depth (the library itself reads no
environment).

``--impl reference`` times the CPU oracle (the only other implementation of
this computation) on a bounded sample of the same workload on the host cores.
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
KERNEL_SOURCES = ["csrc/ptx.cuh", "csrc/gemm_common.h", "csrc/device_common.cuh",
                  "csrc/kernel_ws.cu", "csrc/kernel_ws2.cuh", "csrc/kernel_ws2.cu",
                  "csrc/kernel_ws2_dyn.cu", "csrc/kernels_ladder.cu", "csrc/api.cu",
                  "csrc/launch.h", "csrc/kernel_ws2_k2.cu", "csrc/kernel_ws2_dyn_k2.cu"]


def kernel_source_hash():
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "tma_pipelined_tensor_fp16_gb300", rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return FALLBACK_PEAKS, "fallback"


def load_traffic(workload, kernel_key):
    """DRAM bytes per launch from a committed ncu capture, if the kernel
    sources are unchanged since it was taken; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    e = d.get(workload, {}).get(kernel_key)
    if not e or e.get("kernel_source_hash") != kernel_source_hash():
        return None
    return e.get("dram_bytes_per_launch")


def find_config(name):
    from tma_pipelined_tensor_fp16_gb300 import inputs
    for c in inputs.CONFIGS:
        if c["name"] == name or name in c["name"]:
            return c
    raise SystemExit("unknown config %r; known: %s" % (name, [c["name"] for c in inputs.CONFIGS]))


def algorithmic(cfg):
    M, N, K = cfg["M"], cfg["N"], cfg["K"]
    out_bytes = 2 if cfg["out"] == "f16" else 4
    flops = 2.0 * M * N * K
    nbytes = 2.0 * M * K + 2.0 * N * K + out_bytes * M * N
    return flops, nbytes


# --------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi polling in the background; only samples whose timestamps fall
    inside the timed region (mark_start .. mark_end) are reported."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None
        self.t0 = self.t1 = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.5)

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()
        time.sleep(0.05)

    def stop(self):
        import datetime
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        rows = []
        try:
            with open(self.path) as f:
                for line in f:
                    parts = [p.strip() for p in line.split(",")]
                    if len(parts) < 10 or not parts[2].replace(".", "").isdigit():
                        continue
                    try:
                        ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                    except ValueError:
                        continue
                    rows.append((ts, parts[1:]))
        finally:
            try:
                os.unlink(self.path)
            except OSError:
                pass
        inside = [r for ts, r in rows if self.t0 is not None and self.t0 <= ts <= self.t1]
        window = "inside the timed region"
        if not inside and self.t0 is not None:
            # A timed region shorter than the sampling period: take the
            # samples closest to it (the warm-up just before, the tail just
            # after), within 100 ms, and say so.
            near = sorted(rows, key=lambda tr: max(self.t0 - tr[0], tr[0] - self.t1, 0.0))
            inside = [r for ts, r in near[:3] if max(self.t0 - ts, ts - self.t1) <= 0.1]
            window = "nearest samples within 100 ms of a timed region shorter than the sampling period"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "samples": 0,
                    "reasons": ["no nvidia-smi sample inside the timed region"]}
        sm = [float(r[1]) for r in inside]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in inside:
            for i, n in enumerate(names):
                if r[5 + i].lower().startswith("active"):
                    reasons.add(n)
        power = [float(r[3]) for r in inside if r[3].replace(".", "").isdigit()]
        return {"sm_mhz": statistics.median(sm), "sm_min_mhz": min(sm),
                "sm_max_mhz": float(inside[0][2]),
                "power_w_max": max(power) if power else None,
                "power_w_median": statistics.median(power) if power else None,
                "samples": len(inside), "window": window, "reasons": sorted(reasons)}


NOMINAL_F16_TFLOPS = 2250.0  # GB300 dense fp16/bf16 tensor rate, nominal
# Dense fp16 MMA rate of one SM per clock: 4096 multiply-adds.  At 152 SMs and
# about 1.8 GHz this is the nominal 2.25 PFLOP/s; an ncu capture of the 8192^3
# kernel (FLOP / duration / SMs / clock / tensor-pipe busy fraction) gives
# 7,940 FLOP per busy SM cycle at the capture's clock.
PIPE_FLOP_PER_SM_CYCLE = 8192


def clock_pass_record(clocks, launches, total_ms, flops, peaks, memory_bound, nbytes, sms):
    """The informational clock pass: the bench's plan launched back to back
    for about a second outside the timed region, with nvidia-smi sampling
    every 20 ms.  Its throughput against the sustained peak and against the
    tensor pipe's peak at the SM clock the samples saw, that clock, the power,
    and the launch time in SM cycles at that clock."""
    rec = {"launches": launches, "seconds": total_ms * 1e-3,
           "ms_per_launch": total_ms / launches,
           "sm_mhz_median": clocks.get("sm_mhz"), "sm_mhz_min": clocks.get("sm_min_mhz"),
           "sm_max_mhz": clocks.get("sm_max_mhz"), "power_w_median": clocks.get("power_w_median"),
           "power_w_max": clocks.get("power_w_max"), "samples": clocks.get("samples", 0),
           "reasons": clocks.get("reasons", [])}
    if memory_bound:
        rec["value"] = nbytes * launches / (total_ms * 1e-3) / 1e9
        rec["unit"] = "GB/s"
        rec["frac_of_hbm_gbs"] = rec["value"] / float(peaks["hbm_gbs"])
    else:
        rec["value"] = flops * launches / (total_ms * 1e-3) / 1e12
        rec["unit"] = "TFLOP/s"
        sus = float(peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"]))
        rec["frac_of_sustained_peak"] = rec["value"] / sus
        rec["frac_of_nominal"] = rec["value"] / NOMINAL_F16_TFLOPS
    mhz = clocks.get("sm_mhz")
    if mhz:
        rec["cycles_per_launch"] = rec["ms_per_launch"] * 1e-3 * mhz * 1e6
        if not memory_bound:
            pipe = sms * PIPE_FLOP_PER_SM_CYCLE * mhz * 1e6 / 1e12
            rec["pipe_peak_at_clock_tflops"] = pipe
            rec["frac_of_pipe_peak_at_clock"] = rec["value"] / pipe
    return rec


# --------------------------------------------------------------- oracle timing

def time_oracle(cfg, target_s, rows_cap=None):
    """Time the CPU oracle on whole rows of C for this workload; returns
    (flops_per_s, threads, rows, seconds)."""
    import oracle
    from tma_pipelined_tensor_fp16_gb300 import inputs
    M, N, K = cfg["M"], cfg["N"], cfg["K"]
    threads = oracle.default_threads()
    A, B = inputs.make_operands(M, N, K, cfg["dist"], cfg["seed"])
    # two probes separate the per-call decode of B from the per-row cost
    p1 = max(1, min(M, threads))
    p2 = max(p1 + 1, min(M, 4 * threads))
    t0 = time.perf_counter()
    oracle.gemm_rows(A, B, 0, p1, threads)
    t1 = time.perf_counter()
    oracle.gemm_rows(A, B, 0, p2, threads)
    t2 = time.perf_counter()
    per_row = max((t2 - t1) - (t1 - t0), 1e-9) / (p2 - p1)
    fixed = max((t1 - t0) - per_row * p1, 0.0)
    rows = int(max(p2, min(M, (target_s - fixed) / per_row)))
    if rows_cap:
        rows = min(rows, rows_cap)
    t0 = time.perf_counter()
    oracle.gemm_rows(A, B, 0, rows, threads)
    dt = time.perf_counter() - t0
    return 2.0 * rows * N * K / dt, threads, rows, dt, (A, B)


def run_reference(args, cfg, rank):
    if rank != 0:
        return
    import oracle
    from tma_pipelined_tensor_fp16_gb300 import inputs
    M, N, K = cfg["M"], cfg["N"], cfg["K"]
    A, B = inputs.make_operands(M, N, K, cfg["dist"], cfg["seed"])
    threads = oracle.default_threads()
    # size one step (a block of whole rows of C) to about 3 s of host work
    probe = max(1, min(M, threads))
    t0 = time.perf_counter()
    oracle.gemm_rows(A, B, 0, probe, threads)
    per_row = (time.perf_counter() - t0) / probe
    rows = int(max(1, min(M, 3.0 / max(per_row, 1e-9))))
    for _ in range(args.warmup):
        oracle.gemm_rows(A, B, 0, max(1, rows // 4), threads)
    t0 = time.perf_counter()
    for i in range(args.steps):
        r0 = (i * rows) % max(1, M - rows + 1)
        oracle.gemm_rows(A, B, r0, r0 + rows, threads)
    dt = time.perf_counter() - t0
    flops = 2.0 * rows * N * K * args.steps
    value = flops / dt / 1e12
    sample = "%d of %d rows of C (all %d columns, K=%d) per step, fp64 accumulate" % (rows, M, N, K)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": cfg["name"], "M": M, "N": N, "K": K, "out": cfg["out"],
                   "operands": "%s seed %d" % (cfg["dist"], cfg["seed"])},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


METRIC = "fp16 GEMM TFLOP/s at 8192^3 (1 GB300) and % of dense fp16 tensor peak"


# ------------------------------------------------------------- several ranks
#
# Under torchrun every rank runs the same GEMM on its own GPU (the GEMM needs
# no exchange: output tiles are independent, so N GPUs are N replicas --
# weak scaling).  The only collectives are a barrier around the timed region
# and the maximum of the ranks' times.

def max_over_ranks(value, dist, device):
    """The largest `value` over all ranks (the value itself without a process group)."""
    if dist is None:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(world, work_per_step, steps, max_ms, scale=1e12):
    """Aggregate rate of `world` replicas that each did `steps` steps of
    `work_per_step` units, timed by the slowest rank (`max_ms`)."""
    return world * work_per_step * steps / (max_ms * 1e-3) / scale


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="gemm_8192x8192x8192_f16out")
    ap.add_argument("--variant", default=os.environ.get("GEMM_VARIANT", "auto"))
    ap.add_argument("--depth", type=int, default=int(os.environ.get("GEMM_PIPE_DEPTH", "0")))
    ap.add_argument("--block-n", type=int, default=0)
    ap.add_argument("--block-k", type=int, default=0, choices=[0, 64, 128])
    ap.add_argument("--graph", action="store_true",
                    help="capture the K timed launches into one CUDA graph and time its replay "
                         "(launch overhead removed; per-launch times are the average)")
    ap.add_argument("--l2-flush", action="store_true",
                    help="cold L2: write a scratch buffer of twice the L2 size before every timed "
                         "launch; the rate is then taken from the launches' own events")
    ap.add_argument("--group-m", type=int, default=0)
    ap.add_argument("--stream-k", default="auto", choices=["auto", "off", "on"])
    ap.add_argument("--k-order", default="auto", choices=["auto", "up", "snake"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--clock-pass-seconds", type=float, default=1.5,
                    help="length of the informational clock pass after the timed region "
                         "(0 = none)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    cfg = find_config(args.config)

    if args.impl == "reference":
        run_reference(args, cfg, rank)
        return

    import numpy as np
    import torch

    import __graft_entry__
    import tma_pipelined_tensor_fp16_gb300 as pkg
    from tma_pipelined_tensor_fp16_gb300 import inputs

    torch.cuda.set_device(local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))

    def barrier():
        if dist is not None:
            dist.barrier()

    __graft_entry__.build()
    M, N, K = cfg["M"], cfg["N"], cfg["K"]
    A, B = inputs.make_operands(M, N, K, cfg["dist"], cfg["seed"])
    dA = torch.from_numpy(A.view(np.float16)).cuda()
    dB = torch.from_numpy(B.view(np.float16)).cuda()
    out_dt = torch.float16 if cfg["out"] == "f16" else torch.float32
    dC = torch.empty((M, N), dtype=out_dt, device="cuda")
    plan = pkg.Plan(M, N, K, out=cfg["out"], variant=args.variant, pipe_depth=args.depth,
                    block_n=args.block_n, group_m=args.group_m, stream_k=args.stream_k,
                    k_order=args.k_order, block_k=args.block_k)
    stream = torch.cuda.Stream()
    sh = stream.cuda_stream

    for _ in range(args.warmup):
        plan.run(dA.data_ptr(), dB.data_ptr(), dC.data_ptr(), sh)
    torch.cuda.synchronize()
    if plan.device_status() != 0:
        raise SystemExit("warm-up failed: " + pkg.gemm_last_error())

    if args.graph and args.l2_flush:
        raise SystemExit("--graph and --l2-flush cannot be combined")
    graph = None
    if args.graph:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for _ in range(args.steps):
                plan.run(dA.data_ptr(), dB.data_ptr(), dC.data_ptr(), sh)
        graph.replay()  # one untimed replay
        torch.cuda.synchronize()
    scratch = None
    if args.l2_flush:
        l2 = torch.cuda.get_device_properties(local_rank).L2_cache_size
        scratch = torch.empty(2 * l2 // 4, dtype=torch.int32, device="cuda")
    sampler = ClockSampler(local_rank)
    sampler.start()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    sampler.mark_start()
    # The K launches run back to back between two events: an event recorded
    # between two launches would serialise them and hide the overlap of one
    # launch's set-up with the previous launch's tail (programmatic dependent
    # launch).  Only the L2-flush mode brackets each launch with events, to
    # leave the flushes out of the launches' time.
    with torch.cuda.stream(stream):
        t_start.record(stream)
        if graph is not None:
            graph.replay()
        elif scratch is None:
            for _ in range(args.steps):
                plan.run(dA.data_ptr(), dB.data_ptr(), dC.data_ptr(), sh)
        else:
            for i in range(args.steps):
                scratch.fill_(i)  # evicts A, B and C from L2 (outside the launch's events)
                ev[i][0].record(stream)
                plan.run(dA.data_ptr(), dB.data_ptr(), dC.data_ptr(), sh)
                ev[i][1].record(stream)
        t_end.record(stream)
    torch.cuda.synchronize()
    sampler.mark_end()
    barrier()
    clocks = sampler.stop()
    if plan.device_status() != 0:
        raise SystemExit("timed run failed: " + pkg.gemm_last_error())
    total_ms = t_start.elapsed_time(t_end)
    if scratch is not None:
        # the timed region also holds the flushes: the step time is the
        # launches' own time
        launch_ms = [a.elapsed_time(b) for a, b in ev]
        total_ms = sum(launch_ms)
    else:
        launch_ms = [total_ms / args.steps] * args.steps
    total_ms = max_over_ranks(total_ms, dist, "cuda")

    # Outside the timed region: each launch alone between its own two events
    # (informational; such launches cannot overlap their neighbours).
    single_ms = []
    if graph is None and scratch is None:
        n1 = min(args.steps, 20)
        ev1 = ev[:n1]
        with torch.cuda.stream(stream):
            for a, b in ev1:
                a.record(stream)
                plan.run(dA.data_ptr(), dB.data_ptr(), dC.data_ptr(), sh)
                b.record(stream)
        torch.cuda.synchronize()
        if plan.device_status() != 0:
            raise SystemExit("per-launch pass failed: " + pkg.gemm_last_error())
        single_ms = [a.elapsed_time(b) for a, b in ev1]

    flops, nbytes = algorithmic(cfg)
    ms_per_step = total_ms / args.steps
    value = whole_job_rate(world, flops, args.steps, total_ms)
    avg_launch_s = statistics.mean(launch_ms) * 1e-3

    # ------------------------------------------ clock pass (informational)
    # Outside the timed region: the same plan back to back for about a
    # second, long enough for nvidia-smi's 20 ms samples to show the SM clock
    # and power under this load (the timed region itself is shorter than a
    # few sampling periods at 8192^3).
    clock_pass = None
    if args.clock_pass_seconds > 0 and graph is None:
        n_pass = max(8, int(args.clock_pass_seconds * 1e3 / max(ms_per_step, 1e-3)))
        cs = ClockSampler(local_rank)
        cs.start()
        p0 = torch.cuda.Event(enable_timing=True)
        p1 = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        cs.mark_start()
        with torch.cuda.stream(stream):
            p0.record(stream)
            for _ in range(n_pass):
                plan.run(dA.data_ptr(), dB.data_ptr(), dC.data_ptr(), sh)
            p1.record(stream)
        torch.cuda.synchronize()
        cs.mark_end()
        pass_clocks = cs.stop()
        if plan.device_status() != 0:
            raise SystemExit("clock pass failed: " + pkg.gemm_last_error())
        clock_pass = (pass_clocks, n_pass, p0.elapsed_time(p1))

    # --------------------------------------------------- end to end, host buffers
    e2e = None
    if not args.no_e2e:
        hA = torch.from_numpy(A.view(np.float16)).pin_memory()
        hB = torch.from_numpy(B.view(np.float16)).pin_memory()
        hC = torch.empty((M, N), dtype=out_dt).pin_memory()
        e2e_steps = max(3, min(args.steps, 10))
        for _ in range(2):
            plan.run_host(hA.data_ptr(), hB.data_ptr(), hC.data_ptr(), sh)
        barrier()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(e2e_steps):
            plan.run_host(hA.data_ptr(), hB.data_ptr(), hC.data_ptr(), sh)
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(e0.elapsed_time(e1), dist, "cuda")
        e2e = {"value": whole_job_rate(world, flops, e2e_steps, e2e_ms), "unit": "TFLOP/s",
               "h2d_bytes_per_step": int(A.nbytes + B.nbytes),
               "d2h_bytes_per_step": int(hC.numel() * hC.element_size()),
               "steps": e2e_steps, "ms_per_step": e2e_ms / e2e_steps,
               "api": "gemm_run_host (pinned host buffers; copies, kernel and sync inside)"}
    plan_desc = plan.describe()
    pcfg = plan.config()
    plan.close()

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return

    peaks, peak_kind = load_peaks()
    memory_bound = cfg["name"].startswith("gemm_skinny")
    out_tag = "f16" if cfg["out"] == "f16" else "f32"
    if pcfg["variant"] in (7, 8):
        kernel_key = "k_ws2<%s%s%s>" % (out_tag, ",dynamic" if pcfg["variant"] == 8 else "",
                                        ",k128" if pcfg["block_k"] == 128 else "")
    else:
        kernel_key = "k_ws<%d,%s,%s>" % (pcfg["block_n"], out_tag,
                                          "persistent" if pcfg["variant"] == 5 else
                                          "v%d" % pcfg["variant"])
    traffic = load_traffic(cfg["name"], kernel_key)
    if memory_bound:
        achieved = nbytes / avg_launch_s / 1e9
        peak = float(peaks["hbm_gbs"])
        roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "traffic": traffic,
                "peak_source": "%s hbm_gbs (copy)" % peak_kind}
    else:
        achieved = flops / avg_launch_s / 1e12
        # A long timed region (or one the power limiter throttled) is measured
        # against the sustained figure, a short one against the burst figure.
        sustained = total_ms > 200.0 or "sw_power_cap" in clocks.get("reasons", [])
        key = "bf16_tflops_sustained" if sustained else "bf16_tflops"
        peak = float(peaks.get(key, peaks["bf16_tflops"]))
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "traffic": traffic,
                "peak_source": "%s %s (%s; fp16 dense rate = bf16 rate)"
                               % (peak_kind, key, "sustained: timed region %.0f ms%s"
                                  % (total_ms, ", sw_power_cap seen" if "sw_power_cap" in
                                     clocks.get("reasons", []) else "") if sustained
                                  else "burst: timed region %.0f ms" % total_ms),
                "frac_of_burst_peak": achieved / float(peaks["bf16_tflops"])}
    roof["algorithmic_per_launch"] = flops if not memory_bound else nbytes
    roof["avg_launch_ms"] = avg_launch_s * 1e3
    if not memory_bound:
        roof["frac_of_nominal"] = achieved / NOMINAL_F16_TFLOPS
    if clock_pass is not None:
        sms = torch.cuda.get_device_properties(local_rank).multi_processor_count
        clock_pass = clock_pass_record(clock_pass[0], clock_pass[1], clock_pass[2], flops, peaks,
                                       memory_bound, nbytes, sms)
    if clocks.get("sm_mhz"):
        # SM cycles of one step at the clock sampled around the timed region
        roof["cycles_per_step_at_sampled_clock"] = ms_per_step * 1e-3 * clocks["sm_mhz"] * 1e6

    cpu = None
    if not args.no_cpu_baseline:
        fps, threads, rows, secs, _ = time_oracle(cfg, args.cpu_seconds)
        cpu = {"value": fps / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
               "sample": "%d of %d rows of C (all %d columns, K=%d), fp64 accumulate, %.1f s"
                         % (rows, M, N, K, secs)}

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f16 (fp32 accumulate)", "data": "synthetic",
        "config": {"workload": cfg["name"], "M": M, "N": N, "K": K, "out": cfg["out"],
                   "operands": "%s seed %d" % (cfg["dist"], cfg["seed"]),
                   "l2": ("flushed: a 2 x L2 scratch write before every launch (cold)"
                          if args.l2_flush else
                          "no flush: A+B+C exceed the L2" if M * K * 2 + N * K * 2 > 130e6
                          else "operands fit in L2 (warm)"),
                   "launch": "one CUDA graph of the K launches" if args.graph
                   else "K host launches, each bracketed by events" if args.l2_flush
                   else "K host launches back to back",
                   "plan": plan_desc},
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": args.steps,
        "clocks": clocks,
        "clock_pass": clock_pass,
    }
    if single_ms:
        line["single_launch_median"] = {
            "value": flops / (statistics.median(single_ms) * 1e-3) / 1e12, "unit": "TFLOP/s",
            "launches": len(single_ms),
            "note": "each launch between its own two events, outside the timed region"}
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
