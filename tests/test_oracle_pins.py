"""Pins for the CPU oracle: each test checks the oracle against something other
than itself -- exact rational brute force, closed forms, integer arithmetic,
library routines (numpy's IEEE half conversion, numpy's fp64 matmul) -- chosen
so that a dropped term, a wrong sign or index, or a transposed operand fails at
least one of them (``test_oracle_mutants.py`` plants such mistakes and checks
that these pins catch every one).

What the oracle computes is the plain definition of the method's result,
C = A . B^T with A (M x K) and B (N x K) both K-contiguous ("GEMM II --
pipelining with TMA", Step 4: A tile at {m, k}, B tile at {n, k}), summed in
fp64 over fp16 inputs ("GEMM II", baseline paragraph: fp32 accumulate; the
oracle keeps the higher-precision sum the tolerance is measured against).
"""
import math
from fractions import Fraction

import numpy as np
import pytest

import oracle
from tma_pipelined_tensor_fp16_gb300 import inputs

ALL_BITS = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)


# ----------------------------------------------------------------- fp16 codec

def test_decode_all_65536_patterns_match_ieee_half():
    got = oracle.f16_to_f64(ALL_BITS)
    ref = ALL_BITS.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # signed zeros and infinities keep their sign
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def test_decode_known_values():
    # 0x3c00 = 1, 0xc000 = -2, 0x7bff = 65504 (largest finite), 0x0001 = 2^-24
    # (smallest subnormal), 0x0400 = 2^-14 (smallest normal), 0x3555 ~ 1/3.
    d = dict(zip([0x3C00, 0xC000, 0x7BFF, 0x0001, 0x0400, 0x3555, 0x8000],
                 [1.0, -2.0, 65504.0, 2.0 ** -24, 2.0 ** -14, 0.333251953125, -0.0]))
    got = oracle.f16_to_f64(np.array(list(d), dtype=np.uint16))
    assert list(got) == list(d.values())


def test_encode_roundtrips_every_finite_half():
    ref = ALL_BITS.view(np.float16).astype(np.float64)
    fin = np.isfinite(ref)
    back = oracle.f64_to_f16(ref[fin])
    assert np.array_equal(back, ALL_BITS[fin])


def test_encode_matches_ieee_rne_on_random_doubles():
    rng = np.random.default_rng(12345)
    # log-uniform magnitudes spanning subnormals to overflow, both signs
    mag = np.exp2(rng.uniform(-27.0, 17.0, size=2_000_000))
    x = mag * rng.choice([-1.0, 1.0], size=mag.size)
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(oracle.f64_to_f16(x), ref)


def test_encode_ties_and_edges():
    cases = [
        (1.0 + 2.0 ** -11, 0x3C00),            # tie between 1 and 1+2^-10 -> even (1)
        (1.0 + 3 * 2.0 ** -11, 0x3C02),        # tie -> even significand 2
        (1.0 + 2.0 ** -11 + 2.0 ** -40, 0x3C01),  # just above the tie -> up
        (2.0 ** -25, 0x0000),                  # half the smallest subnormal -> even (0)
        (3 * 2.0 ** -25, 0x0002),              # 1.5 quanta -> 2
        (65504.0, 0x7BFF),
        (65519.99, 0x7BFF),
        (65520.0, 0x7C00),                     # halfway to 2^16 -> even -> inf
        (-65520.0, 0xFC00),
        (-0.0, 0x8000),
        (2.0 ** -14 - 2.0 ** -25, 0x0400),     # rounds up into the smallest normal
        (1e300, 0x7C00),
    ]
    x = np.array([c[0] for c in cases])
    want = np.array([c[1] for c in cases], dtype=np.uint16)
    assert np.array_equal(oracle.f64_to_f16(x), want)
    assert oracle.f64_to_f16(np.array([np.nan]))[0] & 0x7C00 == 0x7C00


# ------------------------------------------------------------- GEMM, brute force

def _exact(Abits, Bbits):
    """Exact C = A.B^T over rationals: fp16 values are dyadic, so this has no
    rounding at all."""
    fa = [[Fraction(float(v)) for v in row] for row in Abits.view(np.float16).astype(np.float64)]
    fb = [[Fraction(float(v)) for v in row] for row in Bbits.view(np.float16).astype(np.float64)]
    return [[sum((x * y for x, y in zip(ra, rb)), Fraction(0)) for rb in fb] for ra in fa]


@pytest.mark.parametrize("M,N,K,dist,seed", [
    (1, 1, 1, "uniform", 7), (1, 5, 3, "uniform", 8), (5, 1, 9, "normal", 9),
    (3, 7, 2, "uniform", 10), (9, 4, 17, "normal", 11), (6, 6, 33, "uniform", 12),
    (2, 3, 64, "normal", 13),
])
def test_gemm_matches_exact_rational_result(M, N, K, dist, seed):
    A, B = inputs.make_operands(M, N, K, dist, seed)
    ex = _exact(A, B)
    got = oracle.gemm(A, B, threads=3)
    absab = np.abs(A.view(np.float16).astype(np.float64)) @ np.abs(
        B.view(np.float16).astype(np.float64)).T
    # fp64 summation bound: |err| <= K * 2^-53 * sum|a||b|
    bound = K * 2.0 ** -53 * absab
    for m in range(M):
        for n in range(N):
            assert abs(Fraction(got[m, n]) - ex[m][n]) <= Fraction(bound[m, n]), (m, n)


@pytest.mark.parametrize("M,N,K", [(4, 7, 5), (7, 3, 16), (1, 9, 2)])
def test_entries_and_rows_match_exact_rational_result(M, N, K):
    A, B = inputs.make_operands(M, N, K, "normal", 99)
    ex = _exact(A, B)
    rows, cols = np.meshgrid(np.arange(M), np.arange(N), indexing="ij")
    ent = oracle.gemm_entries(A, B, rows.ravel(), cols.ravel()).reshape(M, N)
    part = oracle.gemm_rows(A, B, 1, M, threads=2)
    for m in range(M):
        for n in range(N):
            assert abs(Fraction(ent[m, n]) - ex[m][n]) <= Fraction(K * 2.0 ** -53 * 64.0)
            if m >= 1:
                assert part[m - 1, n] == ent[m, n]


def test_gemm_close_to_numpy_fp64_matmul():
    A, B = inputs.make_operands(37, 53, 301, "normal", 21)
    a = A.view(np.float16).astype(np.float64)
    b = B.view(np.float16).astype(np.float64)
    ref = a @ b.T
    bound = 2 * 301 * 2.0 ** -53 * (np.abs(a) @ np.abs(b).T)
    assert np.all(np.abs(oracle.gemm(A, B) - ref) <= bound)


# ------------------------------------------------------------------ closed forms

@pytest.mark.parametrize("M,N,K", [(3, 5, 1), (17, 9, 256), (2, 3, 5000), (1, 2, 16384)])
def test_all_ones_gives_K_everywhere(M, N, K):
    A, B = inputs.make_operands(M, N, K, "ones", 0)
    C = oracle.gemm(A, B)
    assert np.all(C == float(K))


def test_identity_b_gives_a():
    M, K = 33, 48
    A, _ = inputs.make_operands(M, 1, K, "uniform", 5)
    C = oracle.gemm(A, inputs.identity_b(K, K))
    assert np.array_equal(C, A.view(np.float16).astype(np.float64))


def test_identity_b_wider_k_gives_leading_columns():
    M, N, K = 5, 8, 24
    A, _ = inputs.make_operands(M, 1, K, "normal", 6)
    C = oracle.gemm(A, inputs.identity_b(N, K))
    assert np.array_equal(C, A.view(np.float16).astype(np.float64)[:, :N])


def test_permutation_b_permutes_columns_of_a():
    # A transposed B operand would give A[m, perm^-1[n]] instead: caught here.
    M, N = 11, 40
    A, _ = inputs.make_operands(M, 1, N, "uniform", 31)
    Bp, perm = inputs.permutation_b(N, 77)
    assert not np.array_equal(perm, np.argsort(perm))  # not an involution
    C = oracle.gemm(A, Bp)
    assert np.array_equal(C, A.view(np.float16).astype(np.float64)[:, perm])


# --------------------------------------------------------------- integer inputs

@pytest.mark.parametrize("M,N,K,seed", [(37, 29, 300, 1), (64, 16, 5000, 2), (8, 130, 8, 3)])
def test_small_integer_inputs_are_exact(M, N, K, seed):
    A, B = inputs.make_operands(M, N, K, "int", seed)
    ai = A.view(np.float16).astype(np.int64)
    bi = B.view(np.float16).astype(np.int64)
    assert set(np.unique(ai)) <= {-2, -1, 0, 1, 2}
    exact = ai @ bi.T  # integer arithmetic: no rounding anywhere
    assert np.array_equal(oracle.gemm(A, B), exact.astype(np.float64))


def test_small_integer_fp16_rounding_of_exact_sums():
    # The fp16-output reference is RNE(exact integer); check the oracle's
    # rounding of such sums against numpy's IEEE half conversion.
    A, B = inputs.make_operands(16, 16, 4096, "int", 4)
    C = oracle.gemm(A, B)
    assert np.array_equal(oracle.f64_to_f16(C), C.astype(np.float16).view(np.uint16))


def test_int_distribution_is_roughly_uniform_over_five_values():
    A, _ = inputs.make_operands(200, 1, 500, "int", 9)
    vals, counts = np.unique(A.view(np.float16).astype(np.int64), return_counts=True)
    assert list(vals) == [-2, -1, 0, 1, 2]
    assert counts.min() > 0.18 * A.size and counts.max() < 0.22 * A.size


# ----------------------------------------------------------- input generators

def test_splitmix64_vectorised_matches_scalar_definition():
    mask = (1 << 64) - 1

    def scalar(seed, n):
        out, s = [], seed
        for _ in range(n):
            s = (s + 0x9E3779B97F4A7C15) & mask
            z = s
            z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & mask
            z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & mask
            out.append(z ^ (z >> 31))
        return out

    for seed in (0, 1, 2**63 + 5):
        assert [int(v) for v in inputs.splitmix64(seed, 0, 50)] == scalar(seed, 50)
    # a window starting mid-stream equals the same slice of the full stream
    full = inputs.splitmix64(3, 0, 100)
    assert np.array_equal(inputs.splitmix64(3, 40, 60), full[40:])


def test_uniform_and_normal_ranges_and_moments():
    A, B = inputs.make_operands(300, 200, 1000, "uniform", 1)
    a = A.view(np.float16).astype(np.float64)
    assert a.min() >= -1.0 and a.max() <= 1.0
    assert abs(a.mean()) < 0.01 and abs(a.var() - 1 / 3) < 0.01
    A, _ = inputs.make_operands(300, 1, 1000, "normal", 3)
    a = A.view(np.float16).astype(np.float64)
    assert abs(a.mean()) < 0.01 and abs(a.std() - 1.0) < 0.01
    # B continues the stream after A: it is not a copy of A's first rows
    A, B = inputs.make_operands(4, 4, 64, "uniform", 2)
    assert not np.array_equal(A, B)
