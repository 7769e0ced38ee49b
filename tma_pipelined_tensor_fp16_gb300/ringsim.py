"""Host-side model of the stage-ring protocols (``include/ringsim.h``).

A discrete-event model of the load / MMA / epilogue handshake, built from
``sim/ringsim.cpp`` into ``libringsim.so`` with the host C++ compiler.  Two
uses:

* protocol checking, with faults injected on the host (a wrong byte budget,
  a budget announced several times, a missed phase flip, phases reset per
  persistent tile, an early refill, an epilogue that does not wait, and for
  the response ring of the dynamic tile schedule a wrong reader count or a
  missing re-arm): the model reports the deadlock or the first read of
  incomplete data;
* the timing model of "GEMM II -- pipelining with TMA" (the interactive
  pipeline Gantt: serial vs prefetch, PIPE_DEPTH, K tiles, load : MMA cost),
  as makespan, tensor-core idle fraction, back-to-back MMAs and loads in
  flight.

    python -m tma_pipelined_tensor_fp16_gb300.ringsim [--depth 2] [--k-tiles 8] [--load-mma 1.2]
    python -m tma_pipelined_tensor_fp16_gb300.ringsim --clc
"""
import argparse
import ctypes
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "sim", "ringsim.cpp")
HEADER = os.path.join(os.path.dirname(HERE), "include", "ringsim.h")
LIB_PATH = os.path.join(HERE, "libringsim.so")

LOCKSTEP, WARP_SPEC, PAIR, CLC = 0, 1, 2, 3
(OK, DEADLOCK, EARLY_READ, OVERWRITE, EXTRA_ARRIVAL, BAD_ARG) = range(6)
STATUS_NAMES = {OK: "ok", DEADLOCK: "deadlock", EARLY_READ: "early read", OVERWRITE: "overwrite",
                EXTRA_ARRIVAL: "extra arrival", BAD_ARG: "bad argument"}


class RingsimConfig(ctypes.Structure):
    _fields_ = [("protocol", ctypes.c_int), ("depth", ctypes.c_int), ("k_tiles", ctypes.c_int),
                ("tiles", ctypes.c_int), ("accumulators", ctypes.c_int),
                ("load_time", ctypes.c_double), ("mma_time", ctypes.c_double),
                ("epilogue_time", ctypes.c_double), ("issue_latency", ctypes.c_double),
                ("stage_bytes", ctypes.c_longlong), ("chunks", ctypes.c_int),
                ("bytes_delta", ctypes.c_longlong), ("announce_times", ctypes.c_int),
                ("skip_phase_flip", ctypes.c_int), ("reset_phase_per_tile", ctypes.c_int),
                ("refill_before_mma", ctypes.c_int), ("epilogue_no_wait", ctypes.c_int),
                ("clc_slots", ctypes.c_int),
                ("clc_latency", ctypes.c_double), ("clc_readers_delta", ctypes.c_int),
                ("clc_no_rearm", ctypes.c_int), ("clc_rearm_after_release", ctypes.c_int),
                ("clc_request_late", ctypes.c_int)]


class RingsimResult(ctypes.Structure):
    _fields_ = [("status", ctypes.c_int), ("makespan", ctypes.c_double),
                ("mma_busy", ctypes.c_double), ("idle_fraction", ctypes.c_double),
                ("mma_back_to_back", ctypes.c_int), ("max_loads_in_flight", ctypes.c_int),
                ("stages_consumed", ctypes.c_int), ("tiles_stored", ctypes.c_int),
                ("roles_unique", ctypes.c_int), ("detail", ctypes.c_char * 256),
                ("response_wait", ctypes.c_double), ("request_wait", ctypes.c_double),
                ("responses_read", ctypes.c_int)]


def _cxx():
    return os.environ.get("CXX") or shutil.which("g++") or shutil.which("c++") or "g++"


def build(force=False):
    """Compile libringsim.so next to this file (host C++ only)."""
    newest = max(os.path.getmtime(SRC), os.path.getmtime(HEADER))
    if not force and os.path.exists(LIB_PATH) and os.path.getmtime(LIB_PATH) >= newest:
        return LIB_PATH
    tmp = LIB_PATH + ".tmp%d" % os.getpid()
    cmd = [_cxx(), "-std=c++17", "-O2", "-fPIC", "-shared", "-fvisibility=hidden",
           "-I", os.path.dirname(HEADER), "-o", tmp, SRC]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("ringsim build failed:\n%s%s" % (r.stdout, r.stderr))
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


_lib = None


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(LIB_PATH)
        L.ringsim_run.restype = ctypes.c_int
        L.ringsim_run.argtypes = [ctypes.POINTER(RingsimConfig), ctypes.POINTER(RingsimResult)]
        L.ringsim_byte_trace.restype = None
        L.ringsim_byte_trace.argtypes = [ctypes.c_longlong, ctypes.c_longlong,
                                         ctypes.POINTER(ctypes.c_longlong)]
        _lib = L
    return _lib


DEFAULTS = dict(protocol=WARP_SPEC, depth=4, k_tiles=8, tiles=1, accumulators=2, load_time=1.2,
                mma_time=1.0, epilogue_time=0.0, issue_latency=0.0,
                stage_bytes=(128 * 64 + 128 * 64) * 2, chunks=2, bytes_delta=0,
                announce_times=1, skip_phase_flip=0, reset_phase_per_tile=0,
                refill_before_mma=0, epilogue_no_wait=0, clc_slots=4, clc_latency=0.5, clc_readers_delta=0,
                clc_no_rearm=0, clc_rearm_after_release=0, clc_request_late=0)


def run(**kw):
    """Run one configuration (keyword arguments as in ringsim_config; the
    protocol may be given as "lockstep", "warp_spec", "pair" or "clc"); returns
    a dict."""
    args = dict(DEFAULTS)
    unknown = set(kw) - set(args)
    if unknown:
        raise TypeError("unknown ringsim option(s): %s" % sorted(unknown))
    args.update(kw)
    if isinstance(args["protocol"], str):
        args["protocol"] = {"lockstep": LOCKSTEP, "warp_spec": WARP_SPEC,
                            "pair": PAIR, "clc": CLC}[args["protocol"]]
    cfg = RingsimConfig(**args)
    res = RingsimResult()
    lib().ringsim_run(ctypes.byref(cfg), ctypes.byref(res))
    out = {n: getattr(res, n) for n, _ in RingsimResult._fields_ if n != "detail"}
    out["detail"] = res.detail.decode()
    out["status_name"] = STATUS_NAMES.get(res.status, "?")
    return out


def byte_trace(bytes_a, bytes_b):
    """[(pending arrivals, pending bytes, phase completed)] after the
    expect_tx and after each of the two copies."""
    buf = (ctypes.c_longlong * 9)()
    lib().ringsim_byte_trace(bytes_a, bytes_b, buf)
    return [tuple(int(buf[3 * i + j]) for j in range(3)) for i in range(3)]


def gantt(mode="prefetch", depth=2, k_tiles=8, load_mma=1.2):
    """The pipeline Gantt of "GEMM II": one tile's K loop, a fixed load time
    (load_mma x the MMA time) per tile of K and a unit MMA time; serial is
    Step 4 (a ring of one stage: load, wait, MMA, wait), prefetch is Step 5
    (loads run PIPE_DEPTH ahead).  Each K tile is one copy here, so the loads
    in flight count K tiles."""
    d = 1 if mode == "serial" else depth
    r = run(protocol=LOCKSTEP, depth=d, k_tiles=k_tiles, tiles=1, load_time=load_mma,
            mma_time=1.0, epilogue_time=0.0, chunks=1)
    return {"mode": mode, "depth": d, "k_tiles": k_tiles, "load_mma": load_mma,
            "status": r["status_name"], "makespan": r["makespan"],
            "tensor_idle": r["idle_fraction"], "mma_back_to_back": bool(r["mma_back_to_back"]),
            "loads_in_flight_max": r["max_loads_in_flight"] // 2}


def clc_table(slots=(1, 2, 4), latencies=(0.5, 4.0, 12.0), tiles=17, k_tiles=8,
              epilogue_time=6.0):
    """The dynamic schedule's response ring: for each slot count and response
    latency (in MMA times per K block; a tile is k_tiles of them), the
    makespan of `tiles` tiles and the time the requester waited for a free
    slot and for responses, with requests at the start of each tile."""
    rows = []
    for n in slots:
        for lat in latencies:
            r = run(protocol=CLC, clc_slots=n, clc_latency=lat, tiles=tiles,
                    k_tiles=k_tiles, depth=4, load_time=1.2, mma_time=1.0,
                    epilogue_time=epilogue_time)
            rows.append({"slots": n, "latency": lat, "status": r["status_name"],
                         "makespan": r["makespan"], "request_wait": r["request_wait"],
                         "response_wait": r["response_wait"]})
    return rows


def clc_miscount_onset(slots=(1, 2, 4, 8), limit=400):
    """Tiles per cluster after which a response ring whose empty barriers
    count one reader too few first fails (overwrite or deadlock)."""
    out = []
    for n in slots:
        onset = None
        for tiles in range(1, limit + 1):
            r = run(protocol=CLC, clc_slots=n, tiles=tiles, k_tiles=8, depth=4,
                    load_time=1.2, mma_time=1.0, epilogue_time=6.0, clc_readers_delta=-1)
            if r["status_name"] != "ok":
                onset = (tiles, r["status_name"])
                break
        out.append({"slots": n, "onset": onset})
    return out


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--depth", type=int, default=2)
    ap.add_argument("--k-tiles", type=int, default=8)
    ap.add_argument("--load-mma", type=float, default=1.2)
    ap.add_argument("--clc", action="store_true",
                    help="the dynamic schedule's response ring instead of the pipeline Gantt")
    a = ap.parse_args()
    if a.clc:
        print("response ring, 17 tiles of %d K blocks (times in MMA times per K block)"
              % a.k_tiles)
        for row in clc_table(k_tiles=a.k_tiles):
            print("slots %d  latency %5.1f  %-8s makespan %7.1f  request wait %6.1f  "
                  "response wait %6.1f" % (row["slots"], row["latency"], row["status"],
                                            row["makespan"], row["request_wait"],
                                            row["response_wait"]))
        for row in clc_miscount_onset():
            print("one reader too few, %d slot(s): %s" % (
                row["slots"], "first fails at %d tiles (%s)" % row["onset"] if row["onset"]
                else "no failure within 400 tiles"))
        return
    for mode in ("serial", "prefetch"):
        g = gantt(mode, a.depth, a.k_tiles, a.load_mma)
        print("%-8s PIPE_DEPTH=%d K tiles=%d load:MMA=%.2f  makespan %.2f  tensor idle %.1f%%  "
              "MMA back-to-back %s  loads in flight (max) %d"
              % (mode, g["depth"], g["k_tiles"], g["load_mma"], g["makespan"],
                 100 * g["tensor_idle"], "yes" if g["mma_back_to_back"] else "no",
                 g["loads_in_flight_max"]))


if __name__ == "__main__":
    main()
