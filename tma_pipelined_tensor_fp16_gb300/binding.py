"""ctypes binding of libtmagemm.so (the C ABI in include/tmagemm.h).

Argument marshalling only: every step of the GEMM runs in the library's CUDA
kernels.  If the library has not been built, or the device is not a GB300,
the calls fail loudly -- there is no fallback of any kind.
"""
import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libtmagemm.so")

GEMM_OUT_F32, GEMM_OUT_F16 = 0, 1
(GEMM_OK, GEMM_ERR_INVALID_ARG, GEMM_ERR_UNSUPPORTED, GEMM_ERR_CUDA, GEMM_ERR_TIMEOUT,
 GEMM_ERR_NO_DEVICE) = range(6)
(GEMM_VAR_AUTO, GEMM_VAR_SYNC_TILED, GEMM_VAR_TMA_SERIAL, GEMM_VAR_PIPELINED,
 GEMM_VAR_WS_PIPELINED, GEMM_VAR_PERSISTENT, GEMM_VAR_PERSISTENT_LOCKSTEP,
 GEMM_VAR_PERSISTENT_2CTA, GEMM_VAR_DYNAMIC_2CTA) = range(9)

VARIANTS = {
    "auto": GEMM_VAR_AUTO,
    "sync_tiled": GEMM_VAR_SYNC_TILED,
    "tma_serial": GEMM_VAR_TMA_SERIAL,
    "pipelined": GEMM_VAR_PIPELINED,
    "ws_pipelined": GEMM_VAR_WS_PIPELINED,
    "persistent": GEMM_VAR_PERSISTENT,
    "persistent_lockstep": GEMM_VAR_PERSISTENT_LOCKSTEP,
    "persistent_2cta": GEMM_VAR_PERSISTENT_2CTA,
    "dynamic_2cta": GEMM_VAR_DYNAMIC_2CTA,
}
VARIANT_NAMES = {v: k for k, v in VARIANTS.items()}


class gemm_options(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in
                ("variant", "pipe_depth", "block_n", "group_m", "grid", "wait_budget_ms",
                 "debug_stall", "stream_k", "l2_policy", "k_order", "block_k")]


class gemm_config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in
                ("variant", "block_m", "block_n", "block_k", "pipe_depth", "group_m", "grid",
                 "threads", "tiles_m", "tiles_n", "num_tiles", "k_blocks", "smem_bytes",
                 "tmem_cols", "tx_bytes", "dp_tiles", "sk_tiles", "sk_kb_per_worker",
                 "sk_max_contrib")] + [("workspace_bytes", ctypes.c_longlong),
                                       ("a_rows", ctypes.c_int),
                                       ("tail_halves", ctypes.c_int)]

    def as_dict(self):
        return {n: getattr(self, n) for n, _ in self._fields_}


class GemmError(RuntimeError):
    def __init__(self, status, msg):
        super().__init__("gemm status %d: %s" % (status, msg))
        self.status = status


_SIGS = {
    "gemm_create_plan": (ctypes.c_void_p, [ctypes.c_int64] * 3 + [ctypes.c_int]),
    "gemm_create_plan_ex": (ctypes.c_void_p,
                            [ctypes.c_int64] * 3 + [ctypes.c_int, ctypes.POINTER(gemm_options)]),
    "gemm_run": (ctypes.c_int, [ctypes.c_void_p] * 5),
    "gemm_run_host": (ctypes.c_int, [ctypes.c_void_p] * 5),
    "gemm_get_device_status": (ctypes.c_int, [ctypes.c_void_p]),
    "gemm_destroy": (None, [ctypes.c_void_p]),
    "gemm_last_error": (ctypes.c_char_p, []),
    "gemm_last_status": (ctypes.c_int, []),
    "gemm_plan_describe": (ctypes.c_char_p, [ctypes.c_void_p]),
    "gemm_plan_config": (ctypes.c_int, [ctypes.c_void_p, ctypes.POINTER(gemm_config)]),
    "gemm_select_config": (ctypes.c_int, [ctypes.c_int64] * 3 + [
        ctypes.c_int, ctypes.POINTER(gemm_options), ctypes.c_int, ctypes.c_int,
        ctypes.POINTER(gemm_config)]),
    "gemm_schedule_tile": (ctypes.c_int, [ctypes.POINTER(gemm_config), ctypes.c_int64,
                                          ctypes.POINTER(ctypes.c_int),
                                          ctypes.POINTER(ctypes.c_int)]),
    "gemm_sw128_offset": (ctypes.c_int64, [ctypes.c_int64, ctypes.c_int64]),
    "gemm_schedule_unit": (ctypes.c_int, [ctypes.POINTER(gemm_config), ctypes.c_int, ctypes.c_int]
                           + [ctypes.POINTER(ctypes.c_int)] * 5),
    "gemm_set_trace": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]),
    "gemm_run_noalloc": (ctypes.c_int, [ctypes.c_int64] * 3 + [ctypes.c_int] + [ctypes.c_void_p] * 4
                         + [ctypes.POINTER(ctypes.c_int)]),
}

_lib = None


def lib():
    """The loaded library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                "%s is missing: build it first (python -c 'import __graft_entry__ as g; g.build()')"
                % LIB_PATH)
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def last_error():
    return (lib().gemm_last_error() or b"").decode()


def _check(status):
    if status != GEMM_OK:
        raise GemmError(status, last_error())
    return status


STREAM_K = {"auto": 0, "off": 1, "on": 2}
K_ORDER = {"auto": 0, "up": 1, "snake": 2}


def make_options(variant="auto", pipe_depth=0, block_n=0, group_m=0, grid=0, wait_budget_ms=0,
                 debug_stall=0, stream_k="auto", l2_policy=0, k_order="auto", block_k=0):
    v = VARIANTS[variant] if isinstance(variant, str) else int(variant)
    sk = STREAM_K[stream_k] if isinstance(stream_k, str) else int(stream_k)
    ko = K_ORDER[k_order] if isinstance(k_order, str) else int(k_order)
    return gemm_options(v, pipe_depth, block_n, group_m, grid, wait_budget_ms, debug_stall, sk,
                        l2_policy, ko, block_k)


# ---- the C entry points under their own names ------------------------------

def gemm_create_plan(M, N, K, dtype_out):
    return lib().gemm_create_plan(M, N, K, dtype_out)


def gemm_create_plan_ex(M, N, K, dtype_out, opts=None):
    return lib().gemm_create_plan_ex(M, N, K, dtype_out,
                                     ctypes.byref(opts) if opts is not None else None)


def gemm_run(plan, A_ptr, B_ptr, C_ptr, stream_handle):
    return lib().gemm_run(plan, A_ptr, B_ptr, C_ptr, stream_handle)


def gemm_run_host(plan, A_ptr, B_ptr, C_ptr, stream_handle):
    return lib().gemm_run_host(plan, A_ptr, B_ptr, C_ptr, stream_handle)


def gemm_run_noalloc(M, N, K, dtype_out, A_ptr, B_ptr, C_ptr, stream_handle, want_status=True):
    """Allocation-free run of the default kernel (see include/tmagemm.h).
    Returns (status, device_status); device_status is None when the call is
    asynchronous (want_status=False)."""
    if want_status:
        ds = ctypes.c_int(-1)
        st = lib().gemm_run_noalloc(M, N, K, dtype_out, A_ptr, B_ptr, C_ptr, stream_handle,
                                    ctypes.byref(ds))
        return st, ds.value
    st = lib().gemm_run_noalloc(M, N, K, dtype_out, A_ptr, B_ptr, C_ptr, stream_handle, None)
    return st, None


def gemm_set_trace(plan, device_ptr, units_per_cta):
    return lib().gemm_set_trace(plan, device_ptr, units_per_cta)


def gemm_get_device_status(plan):
    return lib().gemm_get_device_status(plan)


def gemm_destroy(plan):
    lib().gemm_destroy(plan)


def gemm_last_error():
    return last_error()


def gemm_last_status():
    return lib().gemm_last_status()


def gemm_plan_describe(plan):
    return (lib().gemm_plan_describe(plan) or b"").decode()


def gemm_plan_config(plan):
    c = gemm_config()
    _check(lib().gemm_plan_config(plan, ctypes.byref(c)))
    return c


def gemm_select_config(M, N, K, dtype_out, opts=None, sm_count=152, smem_optin=232448):
    c = gemm_config()
    st = lib().gemm_select_config(M, N, K, dtype_out,
                                  ctypes.byref(opts) if opts is not None else None,
                                  sm_count, smem_optin, ctypes.byref(c))
    return st, c


def gemm_schedule_tile(cfg, tile):
    m, n = ctypes.c_int(), ctypes.c_int()
    st = lib().gemm_schedule_tile(ctypes.byref(cfg), tile, ctypes.byref(m), ctypes.byref(n))
    return st, m.value, n.value


def gemm_schedule_unit(cfg, worker, index):
    """(tile, kb0, kb1, contrib, ncontrib) of a worker's unit, or None past the end."""
    v = [ctypes.c_int() for _ in range(5)]
    st = lib().gemm_schedule_unit(ctypes.byref(cfg), worker, index, *[ctypes.byref(x) for x in v])
    if st == 0:
        return None
    if st != 1:
        raise GemmError(st, last_error())
    return tuple(x.value for x in v)


def gemm_worker_units(cfg, worker):
    units, i = [], 0
    while True:
        u = gemm_schedule_unit(cfg, worker, i)
        if u is None:
            return units
        units.append(u)
        i += 1


def gemm_sw128_offset(row, byte_in_row):
    return lib().gemm_sw128_offset(row, byte_in_row)


# ---- a small object wrapper --------------------------------------------------

class Plan:
    """Owns one gemm_plan.  ``run`` takes device pointers (ints) and a stream
    handle; ``__call__`` takes torch CUDA tensors."""

    def __init__(self, M, N, K, out="f16", **options):
        self.M, self.N, self.K = M, N, K
        self.out = out
        dt = GEMM_OUT_F16 if out == "f16" else GEMM_OUT_F32
        self._h = gemm_create_plan_ex(M, N, K, dt, make_options(**options))
        if not self._h:
            raise GemmError(gemm_last_status(), last_error())

    @property
    def handle(self):
        return self._h

    def describe(self):
        return gemm_plan_describe(self._h)

    def config(self):
        return gemm_plan_config(self._h).as_dict()

    def run(self, A_ptr, B_ptr, C_ptr, stream_handle=0):
        _check(gemm_run(self._h, A_ptr, B_ptr, C_ptr, stream_handle))

    def run_host(self, A_ptr, B_ptr, C_ptr, stream_handle=0):
        _check(gemm_run_host(self._h, A_ptr, B_ptr, C_ptr, stream_handle))

    def device_status(self):
        return gemm_get_device_status(self._h)

    def set_trace(self, device_ptr, units_per_cta):
        _check(gemm_set_trace(self._h, device_ptr, units_per_cta))

    def __call__(self, A, B, C, stream=None):
        """C = A . B^T for torch CUDA tensors (A: M x K fp16, B: N x K fp16,
        C: M x N fp16/fp32, all contiguous)."""
        import torch
        for name, t in (("A", A), ("B", B), ("C", C)):
            if not t.is_cuda or not t.is_contiguous():
                raise ValueError("%s must be a contiguous CUDA tensor" % name)
        if A.dtype != torch.float16 or B.dtype != torch.float16:
            raise TypeError("A and B must be float16")
        want = torch.float16 if self.out == "f16" else torch.float32
        if C.dtype != want:
            raise TypeError("C must be %s" % want)
        if tuple(A.shape) != (self.M, self.K) or tuple(B.shape) != (self.N, self.K) or \
                tuple(C.shape) != (self.M, self.N):
            raise ValueError("shape mismatch with the plan")
        s = stream if stream is not None else torch.cuda.current_stream(A.device)
        self.run(A.data_ptr(), B.data_ptr(), C.data_ptr(), s.cuda_stream)
        return C

    def close(self):
        if getattr(self, "_h", None):
            gemm_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
