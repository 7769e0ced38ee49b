"""Device timeline of one GEMM: the prologue / steady-state / drain of the stage
ring, measured with globaltimer stamps recorded by the kernel itself
(gemm_set_trace).

    python -m tma_pipelined_tensor_fp16_gb300.timeline --config gemm_8192 \
        [--variant persistent_2cta] [--warmup 5] [--gantt 8] [--json out.json]

Prints a JSON summary: the kernel span; per CTA the prologue (set-up done ->
first MMA issued: ring fill and first-load latency), the steady state (first
to last MMA issued), the drain (last MMA issued -> CTA done: the last tile's
epilogue and teardown); the spread of CTA finish times; per unit the MMA
issue span, the gap between consecutive units' MMAs, the wait for a free
accumulator and the epilogue duration.  `--gantt n` also draws n CTAs as text
lanes (`L` loads in flight, `M` MMAs issuing, `E` epilogue).

The pages model this timeline with a fixed load and MMA time per tile ("GEMM
II -- pipelining with TMA", the interactive pipeline Gantt) and ask a design to
write its three phases down ("B200 Tma Pipeline Designer", the three-phase
timeline); this records the real one.
"""
import argparse
import json
import os
import statistics
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

WORDS = 10
H_START, H_END, H_SMID, H_UNITS = 0, 1, 2, 3
(U_TILE, U_LOAD_FIRST, U_LOAD_LAST, U_ACC_FREE, U_MMA_FIRST, U_MMA_LAST, U_EPI_START, U_EPI_END,
 U_FULL_WAIT, U_EMPTY_WAIT) = range(10)


def record(M, N, K, out, dist, seed, warmup=5, units=64, **opts):
    """Run one traced GEMM; return (trace array [grid, units+1, 8] uint64, plan config)."""
    import numpy as np
    import torch

    from . import binding, build, inputs
    build.build()
    A, B = inputs.make_operands(M, N, K, dist, seed)
    dA = torch.from_numpy(A.view(np.float16)).cuda()
    dB = torch.from_numpy(B.view(np.float16)).cuda()
    C = torch.empty((M, N), dtype=torch.float16 if out == "f16" else torch.float32, device="cuda")
    plan = binding.Plan(M, N, K, out=out, **opts)
    cfg = plan.config()
    for _ in range(warmup):
        plan(dA, dB, C)
    buf = torch.zeros(cfg["grid"] * (units + 1) * WORDS, dtype=torch.int64, device="cuda")
    plan.set_trace(buf.data_ptr(), units)
    plan(dA, dB, C)
    torch.cuda.synchronize()
    if plan.device_status() != 0:
        raise RuntimeError("traced run failed: " + binding.last_error())
    plan.set_trace(None, 0)
    plan.close()
    tr = buf.cpu().numpy().view(np.uint64).reshape(cfg["grid"], units + 1, WORDS)
    return tr, cfg


def ran(tr):
    """Indices of the CTAs that ran: under the dynamic schedule most CTAs of
    the grid are cancelled before they start and leave their records zero."""
    return [b for b in range(tr.shape[0]) if int(tr[b, 0, H_START]) != 0]


def summarize(tr, cfg):
    import numpy as np
    live = ran(tr)
    grid = len(live)
    t0 = int(tr[live, 0, H_START].min())
    rel = lambda x: (int(x) - t0) / 1000.0  # us
    ctas = []
    units_all = []
    for b in live:
        h = tr[b, 0]
        n = int(h[H_UNITS])
        us = tr[b, 1:1 + min(n, tr.shape[1] - 1)]
        mma = [u for u in us if u[U_MMA_FIRST] and u[U_MMA_LAST]]
        c = {"cta": b, "sm": int(h[H_SMID]), "start": rel(h[H_START]), "end": rel(h[H_END]),
             "units": n}
        if mma:
            c["prologue"] = rel(mma[0][U_MMA_FIRST]) - c["start"]
            c["steady"] = rel(mma[-1][U_MMA_LAST]) - rel(mma[0][U_MMA_FIRST])
            c["drain"] = c["end"] - rel(mma[-1][U_MMA_LAST])
            for i, u in enumerate(mma):
                d = {"mma_span": (int(u[U_MMA_LAST]) - int(u[U_MMA_FIRST])) / 1000.0,
                     "mma_full_wait": int(u[U_FULL_WAIT]) / 1000.0,
                     "load_lead": (int(u[U_MMA_FIRST]) - int(u[U_LOAD_FIRST])) / 1000.0
                     if u[U_LOAD_FIRST] else None}
                if i > 0:
                    prev = mma[i - 1]
                    d["mma_gap"] = (int(u[U_MMA_FIRST]) - int(prev[U_MMA_LAST])) / 1000.0
                    d["acc_wait"] = (int(u[U_ACC_FREE]) - int(prev[U_MMA_LAST])) / 1000.0
                units_all.append(d)
        ep = [u for u in us if u[U_EPI_START] and u[U_EPI_END]]
        if ep:
            c["epilogue_avg"] = statistics.mean((int(u[U_EPI_END]) - int(u[U_EPI_START])) / 1000.0
                                                for u in ep)
        ctas.append(c)
    span = max(c["end"] for c in ctas)
    ends = sorted(c["end"] for c in ctas)
    busy = sum(c["end"] - c["start"] for c in ctas) / (grid * span)

    def stats(key, src):
        v = [x[key] for x in src if x.get(key) is not None]
        if not v:
            return None
        return {"min": min(v), "median": statistics.median(v), "max": max(v),
                "mean": statistics.mean(v)}

    return {
        "plan": {k: cfg[k] for k in ("variant", "block_m", "block_n", "pipe_depth", "grid",
                                     "num_tiles", "k_blocks", "sk_tiles")},
        "ctas_ran": grid,
        "span_us": span,
        "cta_busy_fraction": busy,
        "cta_end_us": {"min": ends[0], "median": ends[len(ends) // 2], "max": ends[-1]},
        "prologue_us": stats("prologue", ctas),
        "steady_us": stats("steady", ctas),
        "drain_us": stats("drain", ctas),
        "epilogue_us": stats("epilogue_avg", ctas),
        "unit_mma_span_us": stats("mma_span", units_all),
        "unit_mma_full_wait_us": stats("mma_full_wait", units_all),
        "producer_empty_wait_us_per_unit": stats("empty_wait", [
            {"empty_wait": int(u[U_EMPTY_WAIT]) / 1000.0}
            for b in live for u in tr[b, 1:1 + min(int(tr[b, 0, H_UNITS]),
                                                                  tr.shape[1] - 1)]
            if u[U_LOAD_FIRST]]),
        "unit_mma_gap_us": stats("mma_gap", units_all),
        "unit_acc_wait_us": stats("acc_wait", units_all),
        "unit_first_load_lead_us": stats("load_lead", units_all),
        "mma_issue_fraction": sum(u["mma_span"] for u in units_all) /
        (span * len([c for c in ctas if "steady" in c])) if units_all else None,
    }


def gantt(tr, ctas_to_show, width=120):
    live = ran(tr)
    t0 = int(tr[live, 0, 0].min())
    t1 = int(tr[live, 0, 1].max())
    scale = (t1 - t0) / width
    lines = []
    for b in ctas_to_show:
        row = [" "] * width

        def paint(a, z, ch):
            if not a or not z:
                return
            i0 = int((int(a) - t0) / scale)
            i1 = max(i0 + 1, int((int(z) - t0) / scale))
            for i in range(max(0, i0), min(width, i1)):
                if row[i] == " " or ch == "M":
                    row[i] = ch
        n = int(tr[b, 0, H_UNITS])
        for u in tr[b, 1:1 + min(n, tr.shape[1] - 1)]:
            paint(u[U_LOAD_FIRST], u[U_LOAD_LAST], "L")
            paint(u[U_EPI_START], u[U_EPI_END], "E")
            paint(u[U_MMA_FIRST], u[U_MMA_LAST], "M")
        lines.append("cta %4d |%s|" % (b, "".join(row)))
    lines.append("          0 us%s%.1f us" % (" " * (width - 12), (t1 - t0) / 1000.0))
    return "\n".join(lines)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--config", default="gemm_8192x8192x8192_f16out")
    ap.add_argument("--variant", default="auto")
    ap.add_argument("--depth", type=int, default=0)
    ap.add_argument("--stream-k", default="auto")
    ap.add_argument("--l2-policy", type=int, default=0)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--gantt", type=int, default=0)
    ap.add_argument("--json", default="")
    a = ap.parse_args(argv)
    from . import inputs
    cfg = next(c for c in inputs.CONFIGS if a.config in c["name"])
    tr, pcfg = record(cfg["M"], cfg["N"], cfg["K"], cfg["out"], cfg["dist"], cfg["seed"],
                      warmup=a.warmup, variant=a.variant, pipe_depth=a.depth,
                      stream_k=a.stream_k, l2_policy=a.l2_policy)
    s = summarize(tr, pcfg)
    s["workload"] = cfg["name"]
    print(json.dumps(s, indent=1))
    if a.gantt:
        live = ran(tr)
        step = max(1, len(live) // a.gantt)
        print(gantt(tr, live[::step][:a.gantt]))
    if a.json:
        with open(a.json, "w") as f:
            json.dump(s, f, indent=1)


if __name__ == "__main__":
    main()
