"""Sweep the kernel variants, tile widths and pipeline depths on one workload.

    python -m tma_pipelined_tensor_fp16_gb300.sweep --config gemm_8192 \
        [--variants persistent,ws_pipelined] [--depths 2,3,4] [--block-n 64,128,256] \
        [--iters 20] [--rounds 1] [--out results.jsonl] [--shape M,N,K]

Prints one JSON line per configuration: the plan, the shared memory it needs
(or why it does not fit), and the median / mean TFLOP/s and GB/s of its
launches, timed with CUDA events on the launch stream: `rounds` passes over
all configurations, each timing `iters` launches after 3 warm-up launches.  This is the PIPE_DEPTH-versus-shared-memory trade-off measured on
the device ("GEMM II -- pipelining with TMA", Step 5: deeper rings hide more
latency; tilus "Multi-Stage Software Pipelining": deeper pipelines force
smaller tiles).
"""
import argparse
import json
import os
import statistics
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--config", default="gemm_8192x8192x8192_f16out")
    ap.add_argument("--variants", default="sync_tiled,tma_serial,pipelined,persistent_lockstep,"
                                          "ws_pipelined,persistent")
    ap.add_argument("--depths", default="1,2,3,4,5,6,7,8")
    ap.add_argument("--block-n", default="64,128,256")
    ap.add_argument("--stream-k", default="auto", help="comma list of auto,off,on")
    ap.add_argument("--group-m", default="0", help="comma list of raster group heights")
    ap.add_argument("--l2-policy", default="0", help="comma list of L2 load policies 0..3")
    ap.add_argument("--k-order", default="auto", help="comma list of auto,up,snake")
    ap.add_argument("--block-k", default="0", help="comma list of stage K extents 0,64,128")
    ap.add_argument("--iters", type=int, default=20)
    ap.add_argument("--cooldown", type=float, default=0.0,
                    help="seconds of idle GPU before each configuration's timing")
    ap.add_argument("--rounds", type=int, default=1,
                    help="interleaved rounds over all configurations")
    ap.add_argument("--out", default="")
    ap.add_argument("--shape", default="",
                    help="M,N,K overriding the workload's shape (same operand recipe and output)")
    a = ap.parse_args(argv)

    import numpy as np
    import torch

    from . import binding, build, inputs
    build.build()
    cfg = dict(next(c for c in inputs.CONFIGS if a.config in c["name"]))
    if a.shape:
        cfg["M"], cfg["N"], cfg["K"] = (int(x) for x in a.shape.split(","))
        cfg["name"] = "%s@%dx%dx%d" % (cfg["name"], cfg["M"], cfg["N"], cfg["K"])
    M, N, K = cfg["M"], cfg["N"], cfg["K"]
    A, B = inputs.make_operands(M, N, K, cfg["dist"], cfg["seed"])
    dA = torch.from_numpy(A.view(np.float16)).cuda()
    dB = torch.from_numpy(B.view(np.float16)).cuda()
    dC = torch.empty((M, N), dtype=torch.float16 if cfg["out"] == "f16" else torch.float32,
                     device="cuda")
    flops = 2.0 * M * N * K
    nbytes = 2.0 * (M * K + N * K) + dC.element_size() * M * N
    stream = torch.cuda.Stream()
    sink = open(a.out, "a") if a.out else None
    plans = []
    for variant in a.variants.split(","):
        for bn in [int(x) for x in a.block_n.split(",")]:
            depths = [int(x) for x in a.depths.split(",")]
            if variant in ("sync_tiled", "tma_serial"):
                depths = [1]
            for d, sk, gm, l2, ko, bk in [(d, sk, gm, l2, ko, bk) for d in depths
                                          for sk in a.stream_k.split(",")
                                          for gm in [int(x) for x in a.group_m.split(",")]
                                          for l2 in [int(x) for x in a.l2_policy.split(",")]
                                          for ko in a.k_order.split(",")
                                          for bk in [int(x) for x in a.block_k.split(",")]]:
                rec = {"workload": cfg["name"], "variant": variant, "block_n": bn, "depth": d,
                       "stream_k": sk, "group_m": gm, "l2_policy": l2, "k_order": ko,
                       "block_k": bk}
                try:
                    plan = binding.Plan(M, N, K, out=cfg["out"], variant=variant, block_n=bn,
                                        pipe_depth=d, stream_k=sk, group_m=gm, l2_policy=l2,
                                        k_order=ko, block_k=bk)
                except binding.GemmError as e:
                    rec["error"] = str(e)
                    _emit(rec, sink)
                    continue
                rec["plan"] = plan.describe()
                plans.append((rec, plan, []))
    args = (dA.data_ptr(), dB.data_ptr(), dC.data_ptr(), stream.cuda_stream)
    # Rounds interleave the configurations so that slow drifts of the clock
    # (power and temperature) fall on all of them alike.
    for _ in range(a.rounds):
        for rec, plan, ms in plans:
            if a.cooldown > 0:
                import time
                torch.cuda.synchronize()
                time.sleep(a.cooldown)
            for _ in range(3):
                plan.run(*args)
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(a.iters)]
            torch.cuda.synchronize()
            for e0, e1 in ev:
                e0.record(stream)
                plan.run(*args)
                e1.record(stream)
            torch.cuda.synchronize()
            ms.extend(e0.elapsed_time(e1) for e0, e1 in ev)
    for rec, plan, ms in plans:
        rec.update({
            "status": plan.device_status(),
            "launches": len(ms),
            "ms_median": statistics.median(ms), "ms_min": min(ms),
            "tflops_median": flops / (statistics.median(ms) * 1e-3) / 1e12,
            "tflops_mean": flops / (statistics.mean(ms) * 1e-3) / 1e12,
            "gbs_median": nbytes / (statistics.median(ms) * 1e-3) / 1e9,
        })
        plan.close()
        _emit(rec, sink)
    if sink:
        sink.close()


def _emit(rec, sink):
    line = json.dumps(rec)
    print(line, flush=True)
    if sink:
        sink.write(line + "\n")


if __name__ == "__main__":
    main()
