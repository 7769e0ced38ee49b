"""Seeded synthetic GEMM operands, shared by the CUDA path's tests/benchmark and
the oracle's tests.

This module holds none of the GEMM's arithmetic: it only turns a seed into fp16
operand bit patterns.  Neither the CUDA library nor the oracle imports it; the
callers pass its arrays to both.

Stream: SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
generators", OOPSLA 2014; the constants are those of its published reference
generator).  Output i of the stream for seed s is

    z   = s + (i + 1) * 0x9E3779B97F4A7C15          (mod 2^64)
    z   = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9
    z   = (z ^ (z >> 27)) * 0x94D049BB133111EB
    out = z ^ (z >> 31)

Fill order: one stream per seed; A (M x K, row-major) first, then B (N x K,
row-major) continuing the same stream.

Distributions (values are rounded to fp16, nearest-even, before either side
sees them, so both paths consume identical bits):

* ``uniform``: u = (out >> 40) is a 24-bit integer; value = u * 2^-23 - 1, which
  lies in [-1, 1) and is exact in fp32; then fp32 -> fp16.
* ``normal``: Box-Muller on two consecutive outputs:
  u1 = ((out0 >> 40) + 1) * 2^-24 in (0, 1],  u2 = (out1 >> 40) * 2^-24 in [0, 1);
  value = sqrt(-2 ln u1) * cos(2 pi u2) in fp64, then fp32, then fp16.
* ``int``: small integers in {-2, ..., 2}: value = ((out >> 40) * 5 >> 24) - 2.
* ``ones``, ``zeros``: constants (no stream).
"""
import numpy as np

GOLDEN_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_MIX1 = np.uint64(0xBF58476D1CE4E5B9)
_MIX2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22


def splitmix64(seed: int, start: int, count: int) -> np.ndarray:
    """Outputs start .. start+count-1 of the SplitMix64 stream for ``seed``."""
    out = np.empty(count, dtype=np.uint64)
    s = np.uint64(seed & 0xFFFFFFFFFFFFFFFF)
    with np.errstate(over="ignore"):
        for c0 in range(0, count, _CHUNK):
            n = min(_CHUNK, count - c0)
            i = np.arange(start + c0 + 1, start + c0 + 1 + n, dtype=np.uint64)
            z = s + i * GOLDEN_GAMMA
            z = (z ^ (z >> np.uint64(30))) * _MIX1
            z = (z ^ (z >> np.uint64(27))) * _MIX2
            out[c0:c0 + n] = z ^ (z >> np.uint64(31))
    return out


def _draws_per_value(dist: str) -> int:
    return 2 if dist == "normal" else 1


def _values(dist: str, seed: int, start: int, count: int) -> np.ndarray:
    """``count`` fp16 values (as float16) of distribution ``dist``, taking stream
    outputs from position ``start`` on."""
    if dist == "ones":
        return np.ones(count, dtype=np.float16)
    if dist == "zeros":
        return np.zeros(count, dtype=np.float16)
    out = np.empty(count, dtype=np.float16)
    per = _draws_per_value(dist)
    for c0 in range(0, count, _CHUNK):
        n = min(_CHUNK, count - c0)
        x = splitmix64(seed, start + c0 * per, n * per)
        if dist == "uniform":
            u = (x >> np.uint64(40)).astype(np.float32)
            v = u * np.float32(2.0 ** -23) - np.float32(1.0)
            out[c0:c0 + n] = v.astype(np.float16)
        elif dist == "normal":
            x = x.reshape(n, 2)
            u1 = ((x[:, 0] >> np.uint64(40)).astype(np.float64) + 1.0) * 2.0 ** -24
            u2 = (x[:, 1] >> np.uint64(40)).astype(np.float64) * 2.0 ** -24
            v = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)
            out[c0:c0 + n] = v.astype(np.float32).astype(np.float16)
        elif dist == "int":
            u = x >> np.uint64(40)
            v = ((u * np.uint64(5)) >> np.uint64(24)).astype(np.int64) - 2
            out[c0:c0 + n] = v.astype(np.float16)
        else:
            raise ValueError("unknown distribution %r" % dist)
    return out


def make_operands(M: int, N: int, K: int, dist: str = "uniform", seed: int = 0):
    """(A, B) as uint16 fp16 bit patterns: A is M x K row-major, B is N x K row-major."""
    per = _draws_per_value(dist)
    a = _values(dist, seed, 0, M * K).reshape(M, K)
    b = _values(dist, seed, M * K * per, N * K).reshape(N, K)
    return a.view(np.uint16), b.view(np.uint16)


def identity_b(N: int, K: int) -> np.ndarray:
    """B with B[n][k] = 1 if n == k else 0 (N x K), as fp16 bits; then A.B^T = A
    restricted to its first N columns (exactly)."""
    b = np.zeros((N, K), dtype=np.float16)
    r = np.arange(min(N, K))
    b[r, r] = 1.0
    return b.view(np.uint16)


def permutation_b(N: int, seed: int) -> np.ndarray:
    """B with B[n][k] = 1 iff k == perm[n] (N x N) for a seeded permutation, as
    fp16 bits, plus the permutation; then (A.B^T)[m][n] = A[m][perm[n]]."""
    keys = splitmix64(seed, 0, N)
    perm = np.argsort(keys, kind="stable").astype(np.int64)
    b = np.zeros((N, N), dtype=np.float16)
    b[np.arange(N), perm] = 1.0
    return b.view(np.uint16), perm


# The five workloads the method is measured on: shape, output dtype, operand
# distribution and seed.
CONFIGS = [
    dict(name="gemm_256x256x256_f32out", M=256, N=256, K=256, out="f32", dist="uniform", seed=0),
    dict(name="gemm_4096x4096x4096_f16out", M=4096, N=4096, K=4096, out="f16", dist="uniform",
         seed=1),
    dict(name="gemm_8192x8192x8192_f16out", M=8192, N=8192, K=8192, out="f16", dist="uniform",
         seed=2),
    dict(name="gemm_ragged_4000x3000x5000_f32out", M=4000, N=3000, K=5000, out="f32",
         dist="normal", seed=3),
    dict(name="gemm_skinny_64x16384x16384_f16out", M=64, N=16384, K=16384, out="f16",
         dist="uniform", seed=4),
]
