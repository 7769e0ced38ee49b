"""CPU oracle for the dense fp16 GEMM  C = A . B^T  (fp64 accumulation).

TEST INFRASTRUCTURE.  Only the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import this package.  The product path (the
CUDA library and its Python binding) never imports, links or calls it, and the
two share no code.

The arithmetic lives in ``oracle.c`` (plain C, compiled by ``build.py``); this
module only marshals numpy arrays into it.  Conventions:

* ``A``: M x K fp16, row-major, passed as a ``uint16`` array of bit patterns
  (or ``float16``).
* ``B``: N x K fp16 ("K-major": row n holds the K values of column n of B^T).
* result: M x N ``float64``, row-major,
  ``C[m, n] = sum_k A[m, k] * B[n, k]`` summed in ascending k in fp64.

The operand layout follows "GEMM II -- pipelining with TMA", Step 4 (the A tile
is loaded at {m, k} and the B tile at {n, k}, each BLK x BLK_K); the fp32
accumulate and the narrowing to the output dtype follow the same page's
baseline paragraph and its TMA-store epilogue.
"""
import ctypes
import os

import numpy as np

from . import build as _build

_LIB = None


def _lib():
    global _LIB
    if _LIB is None:
        # ORACLE_LIB points the tests' planted-mistake checks at a mutated copy.
        path = os.environ.get("ORACLE_LIB") or _build.build()
        lib = ctypes.CDLL(path)
        i64, u16p, f64p, i64p = (ctypes.c_int64, ctypes.POINTER(ctypes.c_uint16),
                                  ctypes.POINTER(ctypes.c_double),
                                  ctypes.POINTER(ctypes.c_int64))
        lib.oracle_f16_to_f64.argtypes = [ctypes.c_uint16]
        lib.oracle_f16_to_f64.restype = ctypes.c_double
        lib.oracle_f64_to_f16.argtypes = [ctypes.c_double]
        lib.oracle_f64_to_f16.restype = ctypes.c_uint16
        lib.oracle_decode_f16.argtypes = [i64, u16p, f64p]
        lib.oracle_decode_f16.restype = None
        lib.oracle_encode_f16.argtypes = [i64, f64p, u16p]
        lib.oracle_encode_f16.restype = None
        lib.oracle_gemm_f16.argtypes = [i64, i64, i64, u16p, u16p, f64p, ctypes.c_int]
        lib.oracle_gemm_f16.restype = ctypes.c_int
        lib.oracle_gemm_rows_f16.argtypes = [i64, i64, i64, u16p, u16p, f64p, i64, i64,
                                             ctypes.c_int]
        lib.oracle_gemm_rows_f16.restype = ctypes.c_int
        lib.oracle_gemm_entries_f16.argtypes = [i64, i64, i64, u16p, u16p, i64, i64p, i64p,
                                                f64p]
        lib.oracle_gemm_entries_f16.restype = ctypes.c_int
        _LIB = lib
    return _LIB


def _u16(x):
    x = np.ascontiguousarray(x)
    if x.dtype == np.float16:
        x = x.view(np.uint16)
    if x.dtype != np.uint16:
        raise TypeError("fp16 operands must be float16 or uint16 bit patterns, got %s" % x.dtype)
    return x


def _ptr(x, ctype):
    return x.ctypes.data_as(ctypes.POINTER(ctype))


def default_threads() -> int:
    """Host threads the oracle uses by default: every core this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def f16_to_f64(bits):
    """Decode fp16 bit patterns (any shape) to float64, exactly."""
    b = _u16(bits)
    out = np.empty(b.shape, dtype=np.float64)
    _lib().oracle_decode_f16(b.size, _ptr(b, ctypes.c_uint16), _ptr(out, ctypes.c_double))
    return out


def f64_to_f16(x):
    """Round float64 values (any shape) to fp16 bit patterns, nearest-even."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.uint16)
    _lib().oracle_encode_f16(x.size, _ptr(x, ctypes.c_double), _ptr(out, ctypes.c_uint16))
    return out


def _check(A, B):
    A, B = _u16(A), _u16(B)
    if A.ndim != 2 or B.ndim != 2 or A.shape[1] != B.shape[1]:
        raise ValueError("need A (M x K) and B (N x K) with the same K, got %s and %s"
                         % (A.shape, B.shape))
    return A, B


def gemm(A, B, threads=None):
    """Full C = A . B^T as an M x N float64 array."""
    A, B = _check(A, B)
    M, K = A.shape
    N = B.shape[0]
    C = np.empty((M, N), dtype=np.float64)
    rc = _lib().oracle_gemm_f16(M, N, K, _ptr(A, ctypes.c_uint16), _ptr(B, ctypes.c_uint16),
                                _ptr(C, ctypes.c_double), threads or default_threads())
    if rc != 0:
        raise RuntimeError("oracle_gemm_f16 failed (%d)" % rc)
    return C


def gemm_rows(A, B, m_begin, m_end, threads=None):
    """Rows [m_begin, m_end) of C = A . B^T as a (m_end - m_begin) x N float64 array."""
    A, B = _check(A, B)
    M, K = A.shape
    N = B.shape[0]
    C = np.empty((max(m_end - m_begin, 0), N), dtype=np.float64)
    rc = _lib().oracle_gemm_rows_f16(M, N, K, _ptr(A, ctypes.c_uint16),
                                     _ptr(B, ctypes.c_uint16), _ptr(C, ctypes.c_double),
                                     m_begin, m_end, threads or default_threads())
    if rc != 0:
        raise RuntimeError("oracle_gemm_rows_f16 failed (%d)" % rc)
    return C


def gemm_entries(A, B, rows, cols):
    """C[rows[i], cols[i]] for each i, as a float64 vector."""
    A, B = _check(A, B)
    M, K = A.shape
    N = B.shape[0]
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    if rows.shape != cols.shape:
        raise ValueError("rows and cols must have the same shape")
    out = np.empty(rows.shape, dtype=np.float64)
    rc = _lib().oracle_gemm_entries_f16(M, N, K, _ptr(A, ctypes.c_uint16),
                                        _ptr(B, ctypes.c_uint16), rows.size,
                                        _ptr(rows, ctypes.c_int64), _ptr(cols, ctypes.c_int64),
                                        _ptr(out, ctypes.c_double))
    if rc != 0:
        raise IndexError("gemm_entries: index out of range")
    return out
