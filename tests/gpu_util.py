"""Helpers for the GPU parity tests: upload seeded operands, run one GEMM
through the C ABI, compare with the oracle under the stated tolerances.

Tolerances (written out here and used by every parity test):
* fp32 output: max |C_gpu - C_ref| <= 1e-3 * sqrt(K).
* fp16 output: per element |C_gpu - C_ref| <= 1e-2 * |C_ref| + 1e-3 * sqrt(K)
  (relative 1e-2, with an absolute floor so entries whose exact value is near
  zero are not held to a relative test they cannot meet).
* small-integer inputs: bit-exact -- the exact integer result in fp32, or its
  round-to-nearest-even fp16 encoding as computed by the oracle's own encoder.
"""
import numpy as np

import oracle


def tol_ok(got, ref, K, out):
    """Boolean array: which entries meet the tolerance."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    floor = 1e-3 * np.sqrt(K)
    if out == "f32":
        return np.abs(got - ref) <= floor
    return np.abs(got - ref) <= 1e-2 * np.abs(ref) + floor


def assert_close(got, ref, K, out, what=""):
    ok = tol_ok(got, ref, K, out)
    if not ok.all():
        bad = np.argwhere(~ok)
        i = tuple(bad[0])
        raise AssertionError(
            "%s: %d/%d entries out of tolerance; first at %s: got %r ref %r (max |err| %.4g)"
            % (what, bad.shape[0], ok.size, i, float(np.asarray(got)[i]),
               float(np.asarray(ref)[i]),
               float(np.max(np.abs(np.asarray(got, np.float64) - ref)))))


def assert_exact(got_bits_or_vals, ref, out, what=""):
    """Bit-exact comparison for integer-valued results."""
    ref = np.asarray(ref, dtype=np.float64)
    if out == "f32":
        got = np.asarray(got_bits_or_vals, dtype=np.float32).astype(np.float64)
        ok = got == ref
    else:
        got = np.asarray(got_bits_or_vals).view(np.uint16)
        ok = got == oracle.f64_to_f16(ref)
    if not ok.all():
        bad = np.argwhere(~ok)
        raise AssertionError("%s: %d/%d entries differ from the exact result; first at %s"
                             % (what, bad.shape[0], ok.size, tuple(bad[0])))


# Max-error records of the full-size comparisons, printed by the terminal
# summary hook in conftest.py: (what, entries compared, max |err|, worst
# err / allowed).
ERROR_LOG = []


def record_error(what, got, ref, K, out):
    """Log the largest error of `got` against `ref` over every entry, and the
    largest ratio of an entry's error to what the tolerance allows it."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = np.abs(got - ref)
    floor = 1e-3 * np.sqrt(K)
    allowed = floor if out == "f32" else 1e-2 * np.abs(ref) + floor
    ERROR_LOG.append((what, err.size, float(err.max()), float((err / allowed).max())))
    return float(err.max())


_FULL_REF = {}


def full_reference(cfg, dist=None, seed=None):
    """Seeded operands of workload `cfg` and the oracle's C over every entry,
    computed once per test session (about 25 s for 8192^3 on 16 host cores).
    `dist` / `seed` override the workload's own (e.g. "int" for the exact
    cases)."""
    from tma_pipelined_tensor_fp16_gb300 import inputs
    dist = dist or cfg["dist"]
    seed = cfg["seed"] if seed is None else seed
    key = (cfg["M"], cfg["N"], cfg["K"], dist, seed)
    if key not in _FULL_REF:
        A, B = inputs.make_operands(cfg["M"], cfg["N"], cfg["K"], dist, seed)
        _FULL_REF[key] = (A, B, oracle.gemm(A, B))
    return _FULL_REF[key]


def to_device(bits):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.float16)).cuda()


def run(A_bits, B_bits, out, guard_rows=0, stream=None, **opts):
    """C = A . B^T on the GPU through the C ABI.  Returns (C as numpy, guard
    rows as numpy, plan description).  C is pre-filled with NaN; the guard
    rows past the end of C must stay NaN."""
    import torch

    import tma_pipelined_tensor_fp16_gb300 as pkg
    M, K = A_bits.shape
    N = B_bits.shape[0]
    dA, dB = to_device(A_bits), to_device(B_bits)
    dt = torch.float16 if out == "f16" else torch.float32
    buf = torch.full((M + guard_rows, N), float("nan"), dtype=dt, device="cuda")
    C = buf[:M]
    plan = pkg.Plan(M, N, K, out=out, **opts)
    try:
        plan(dA, dB, C, stream=stream)
        torch.cuda.synchronize()
        st = plan.device_status()
        if st != 0:
            raise AssertionError("device status %d: %s" % (st, pkg.gemm_last_error()))
        desc = plan.describe()
    finally:
        plan.close()
    host = buf.cpu()
    if out == "f16":
        c = host[:M].numpy()
        g = host[M:].numpy()
    else:
        c = host[:M].numpy()
        g = host[M:].numpy()
    return c, g, desc


def run_repeated(A_bits, B_bits, out, reps, **opts):
    """Launch ONE plan `reps` times on one stream, refilling C with NaN on that
    stream before every launch; returns the list of outputs (numpy).  This is
    how bench.py uses a plan: per-plan device state (run epoch, status word,
    stream-K tickets, tile-schedule barriers) carries over between launches."""
    import torch

    import tma_pipelined_tensor_fp16_gb300 as pkg
    M, K = A_bits.shape
    N = B_bits.shape[0]
    dA, dB = to_device(A_bits), to_device(B_bits)
    dt = torch.float16 if out == "f16" else torch.float32
    C = torch.empty((M, N), dtype=dt, device="cuda")
    st = torch.cuda.Stream()
    plan = pkg.Plan(M, N, K, out=out, **opts)
    outs = []
    try:
        for _ in range(reps):
            with torch.cuda.stream(st):
                C.fill_(float("nan"))
            plan(dA, dB, C, stream=st)
            st.synchronize()
            s = plan.device_status()
            if s != 0:
                raise AssertionError("device status %d: %s" % (s, pkg.gemm_last_error()))
            outs.append(C.cpu().numpy())
    finally:
        plan.close()
    return outs
