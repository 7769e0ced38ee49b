"""Time the library's default plan against torch.matmul (cuBLAS) on the
workloads, in one process, on the same stream and the same seeded operands.

    python -m tma_pipelined_tensor_fp16_gb300.vs_torch [--configs gemm_4096,ragged]
        [--shapes 2048x2048x2048,6144x6144x6144] [--rounds 5] [--iters 20]
        [--mode single|b2b|both]

`--shapes` replaces the workloads by GEMMs of the given M x N x K with
fp16 output and uniform[-1, 1] operands from seed 7.

A measurement tool only: torch.matmul is the comparison arm, never part of
the library's path.  fp16 output compares against `torch.matmul(A, B.T)`;
fp32 output against `torch.mm(A, B.T, out_dtype=torch.float32)`.

Modes (each repeated over `rounds` interleaved rounds, median reported):
* single: after 3 warm-up launches, `iters` launches each between its own two
  CUDA events on the launch stream;
* b2b: `iters` launches back to back between two events (the library's
  launches overlap their set-up with the previous launch's tail).
Prints one JSON line per workload and mode.
"""
import argparse
import json
import os
import statistics
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def _time_single(fn, stream, iters):
    import torch
    for _ in range(3):
        fn()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(iters)]
    torch.cuda.synchronize()
    for a, b in ev:
        a.record(stream)
        fn()
        b.record(stream)
    torch.cuda.synchronize()
    return statistics.median(a.elapsed_time(b) for a, b in ev)


def _time_b2b(fn, stream, iters):
    import torch
    for _ in range(3):
        fn()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record(stream)
    for _ in range(iters):
        fn()
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / iters


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--configs", default="")
    ap.add_argument("--shapes", default="")
    ap.add_argument("--rounds", type=int, default=5)
    ap.add_argument("--iters", type=int, default=20)
    ap.add_argument("--mode", default="both", choices=["single", "b2b", "both"])
    a = ap.parse_args(argv)

    import numpy as np
    import torch

    from . import binding, build, inputs
    build.build()
    cfgs = [c for c in inputs.CONFIGS
            if not a.configs or any(x in c["name"] for x in a.configs.split(","))]
    if a.shapes:
        cfgs = []
        for sh in a.shapes.split(","):
            M, N, K = (int(x) for x in sh.split("x"))
            cfgs.append(dict(name="gemm_%dx%dx%d_f16out" % (M, N, K), M=M, N=N, K=K, out="f16",
                             dist="uniform", seed=7))
    stream = torch.cuda.Stream()
    modes = ["single", "b2b"] if a.mode == "both" else [a.mode]
    for cfg in cfgs:
        M, N, K = cfg["M"], cfg["N"], cfg["K"]
        A, B = inputs.make_operands(M, N, K, cfg["dist"], cfg["seed"])
        dA = torch.from_numpy(A.view(np.float16)).cuda()
        dB = torch.from_numpy(B.view(np.float16)).cuda()
        f16 = cfg["out"] == "f16"
        dt = torch.float16 if f16 else torch.float32
        C = torch.empty((M, N), dtype=dt, device="cuda")
        T = torch.empty((M, N), dtype=dt, device="cuda") if f16 else None
        plan = binding.Plan(M, N, K, out=cfg["out"])
        sh = stream.cuda_stream
        BT = dB.t()

        def ours():
            plan.run(dA.data_ptr(), dB.data_ptr(), C.data_ptr(), sh)

        def theirs():
            with torch.cuda.stream(stream):
                if f16:
                    torch.matmul(dA, BT, out=T)
                else:
                    torch.mm(dA, BT, out_dtype=torch.float32)

        flops = 2.0 * M * N * K
        nbytes = 2.0 * (M * K + N * K) + C.element_size() * M * N
        iters = a.iters if M * N * K >= 2 ** 30 else 5 * a.iters
        for mode in modes:
            timer = _time_single if mode == "single" else _time_b2b
            ours_ms, theirs_ms = [], []
            for _ in range(a.rounds):
                ours_ms.append(timer(ours, stream, iters))
                theirs_ms.append(timer(theirs, stream, iters))
            if plan.device_status() != 0:
                raise SystemExit("library run failed: " + binding.last_error())
            o, t = statistics.median(ours_ms), statistics.median(theirs_ms)
            print(json.dumps({
                "workload": cfg["name"], "mode": mode, "plan": plan.describe(),
                "ours_us": o * 1e3, "torch_us": t * 1e3,
                "ours_tflops": flops / (o * 1e-3) / 1e12, "torch_tflops": flops / (t * 1e-3) / 1e12,
                "ours_gbs": nbytes / (o * 1e-3) / 1e9, "torch_gbs": nbytes / (t * 1e-3) / 1e9,
                "ours_over_torch": t / o, "rounds": a.rounds, "iters": iters}), flush=True)
        plan.close()


if __name__ == "__main__":
    main()
