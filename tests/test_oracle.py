"""Pins for the CPU oracle, independent of the oracle's own code.

Each check compares the oracle against something it does not share code with:
numpy's IEEE conversions, exact rational arithmetic (fractions.Fraction),
closed forms (identity, permutation, rank-1), exact integer arithmetic, and a
float64 library matmul on shapes where a transposed or mis-indexed operand
would change the answer.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle

RNG = np.random.default_rng(1234)


def f16_bits(a):
    return np.asarray(a, dtype=np.float16).view(np.uint16)


def rand_f16(shape, rng=RNG):
    return f16_bits(rng.uniform(-1, 1, size=shape))


# ---- formats -------------------------------------------------------------


def test_f16_decode_all_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.f16_to_f64(bits)
    want = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    # signed zeros keep their sign
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(want[~nan]))


def test_bf16_decode_all_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.bf16_to_f64(bits)
    want = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])


def test_f16_encode_roundtrip_and_ties():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = bits.view(np.float16).astype(np.float64)
    finite = np.isfinite(vals)
    assert np.array_equal(oracle.f64_to_f16(vals[finite]), bits[finite])
    # exact midpoints between consecutive positive finite halves: ties go to even
    pos = np.sort(vals[finite & (vals >= 0)])
    pos = np.unique(pos)
    mids = (pos[:-1] + pos[1:]) / 2.0
    want = mids.astype(np.float16).view(np.uint16)
    assert np.array_equal(oracle.f64_to_f16(mids), want)
    assert np.array_equal(oracle.f64_to_f16(-mids), want | 0x8000)


def test_f16_encode_random_and_edges():
    x = np.concatenate([
        RNG.uniform(-70000, 70000, 20000),
        RNG.uniform(-1e-4, 1e-4, 20000),           # subnormal range
        RNG.standard_normal(20000) * 10.0 ** RNG.integers(-9, 6, 20000),
        np.array([65504.0, 65519.99, 65520.0, 1e9, -1e9, 2.0 ** -25, 2.0 ** -25 * 1.0000001,
                  3 * 2.0 ** -26, np.inf, -np.inf, 0.0, -0.0]),
    ])
    got = oracle.f64_to_f16(x)
    with np.errstate(over="ignore"):
        want = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, want)
    assert oracle.f64_to_f16(np.array([np.nan]))[0] & 0x7C00 == 0x7C00


# ---- GEMM ----------------------------------------------------------------


def exact_gemm(A_bits, B_bits):
    """Brute force with exact rationals (tiny shapes only)."""
    A = [[Fraction(float(v)) for v in row] for row in A_bits.view(np.float16).astype(np.float64)]
    B = [[Fraction(float(v)) for v in row] for row in B_bits.view(np.float16).astype(np.float64)]
    M, K, N = len(A), len(B), len(B[0])
    return [[sum(A[i][k] * B[k][j] for k in range(K)) for j in range(N)] for i in range(M)]


@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (3, 5, 7), (8, 2, 4), (5, 8, 3)])
def test_gemm_brute_force_exact(M, N, K):
    A, B = rand_f16((M, K)), rand_f16((K, N))
    got = oracle.gemm(A, B)
    ref = exact_gemm(A, B)
    for i in range(M):
        for j in range(N):
            # fp64 accumulation of <= 7 exact products: within a few ulps of the exact value
            assert abs(Fraction(got[i, j]) - ref[i][j]) <= Fraction(1, 2 ** 50)


def test_gemm_identity_both_sides():
    n = 48
    B = rand_f16((n, 37))
    I = f16_bits(np.eye(n))
    assert np.array_equal(oracle.gemm(I, B), B.view(np.float16).astype(np.float64))
    A = rand_f16((29, n))
    assert np.array_equal(oracle.gemm(A, I), A.view(np.float16).astype(np.float64))


def test_gemm_permutation_rows():
    n = 40
    perm = RNG.permutation(n)
    P = np.zeros((n, n))
    P[np.arange(n), perm] = 1.0
    B = rand_f16((n, 24))
    got = oracle.gemm(f16_bits(P), B)
    assert np.array_equal(got, B.view(np.float16).astype(np.float64)[perm])


def test_gemm_rank1_closed_form():
    M, N, K = 17, 23, 64
    u = RNG.integers(-3, 4, M) * 0.5
    v = RNG.integers(-3, 4, N) * 0.25
    A = f16_bits(np.repeat(u[:, None], K, axis=1))
    B = f16_bits(np.repeat(v[None, :], K, axis=0))
    assert np.array_equal(oracle.gemm(A, B), K * np.outer(u, v))


def test_gemm_integer_exact_against_int64():
    M, N, K = 33, 47, 129
    Ai = RNG.integers(-2, 3, (M, K))
    Bi = RNG.integers(-2, 3, (K, N))
    got = oracle.gemm(f16_bits(Ai), f16_bits(Bi))
    assert np.array_equal(got, (Ai.astype(np.int64) @ Bi.astype(np.int64)).astype(np.float64))


def test_gemm_nonsquare_matches_library_matmul():
    # distinct M, N, K and non-symmetric data: a transposed operand or swapped index fails
    M, N, K = 19, 31, 53
    A, B = rand_f16((M, K)), rand_f16((K, N))
    want = A.view(np.float16).astype(np.float64) @ B.view(np.float16).astype(np.float64)
    got = oracle.gemm(A, B)
    assert np.allclose(got, want, rtol=0, atol=1e-12)


def test_gemm_rows_subset_matches_full():
    M, N, K = 64, 40, 72
    A, B = rand_f16((M, K)), rand_f16((K, N))
    full = oracle.gemm(A, B)
    rows = np.array([63, 0, 17, 17, 5])
    assert np.array_equal(oracle.gemm(A, B, rows=rows), full[rows])


def test_gemm_rows_rejects_out_of_range():
    A, B = rand_f16((4, 4)), rand_f16((4, 4))
    with pytest.raises(ValueError):
        oracle.gemm(A, B, rows=[4])


def test_gemm_empty_shapes():
    assert oracle.gemm(rand_f16((0, 5)), rand_f16((5, 3))).shape == (0, 3)
    z = oracle.gemm(np.zeros((3, 0), np.uint16), np.zeros((0, 4), np.uint16))
    assert z.shape == (3, 4) and np.all(z == 0)


def test_gemm_threads_do_not_change_bits():
    A, B = rand_f16((50, 70)), rand_f16((70, 30))
    assert np.array_equal(oracle.gemm(A, B, threads=1), oracle.gemm(A, B, threads=4))


# ---- GEMV ----------------------------------------------------------------


def bf16_bits(a):
    return torch.from_numpy(np.asarray(a, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bf16_vals(bits):
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()


def test_gemv_bf16_matches_library_dot():
    K, N = 96, 37
    x = bf16_bits(RNG.uniform(-1, 1, K))
    W = bf16_bits(RNG.uniform(-1, 1, (N, K)))
    want = bf16_vals(W) @ bf16_vals(x)
    assert np.allclose(oracle.gemv_bf16(x, W), want, rtol=0, atol=1e-12)


def test_gemv_bf16_integer_exact_and_layout():
    # W is K-major: y[n] uses row n of W.  Integer values make the sum exact.
    K, N = 64, 9
    xi = RNG.integers(-2, 3, K)
    Wi = RNG.integers(-2, 3, (N, K))
    got = oracle.gemv_bf16(bf16_bits(xi), bf16_bits(Wi))
    assert np.array_equal(got, (Wi @ xi).astype(np.float64))


def exact_q8(x_bits, q, s_bits):
    x = [Fraction(float(v)) for v in bf16_vals(x_bits)]
    s = s_bits.view(np.float16).astype(np.float64)
    N, K = q.shape
    out = []
    for n in range(N):
        tot = Fraction(0)
        for g in range(K // 32):
            part = sum(x[k] * int(q[n, k]) for k in range(32 * g, 32 * g + 32))
            tot += Fraction(float(s[n, g])) * part
        out.append(tot)
    return out


def test_gemv_q8_brute_force_exact():
    K, N = 96, 5
    x = bf16_bits(RNG.uniform(-1, 1, K))
    q = RNG.integers(-127, 128, (N, K)).astype(np.int8)
    s = f16_bits(RNG.uniform(1e-3, 1e-2, (N, K // 32)))
    got = oracle.gemv_q8(x, q, s)
    ref = exact_q8(x, q, s)
    for n in range(N):
        assert abs(Fraction(got[n]) - ref[n]) <= abs(ref[n]) * Fraction(1, 2 ** 48) + Fraction(1, 2 ** 60)


def test_gemv_q8_group_scale_closed_form():
    # q = 1, x = 1: y[n] = 32 * sum_g s[n, g].  Scales differ per group and per row,
    # so a scale taken from the wrong group or the wrong row changes the answer.
    K, N = 128, 6
    x = bf16_bits(np.ones(K))
    q = np.ones((N, K), np.int8)
    s_vals = (np.arange(N * (K // 32)).reshape(N, K // 32) + 1) * 2.0 ** -8
    got = oracle.gemv_q8(x, q, f16_bits(s_vals))
    assert np.array_equal(got, 32 * s_vals.sum(axis=1))


def test_gemv_q8_one_hot_positions():
    # a single nonzero weight at (n, k) picks x[k] * s[n, k // 32]
    K, N = 96, 4
    xv = np.arange(1, K + 1) * 2.0 ** -7
    s_vals = RNG.integers(1, 8, (N, K // 32)) * 2.0 ** -4
    for (n, k) in [(0, 0), (3, 95), (2, 33), (1, 64)]:
        q = np.zeros((N, K), np.int8)
        q[n, k] = -3
        got = oracle.gemv_q8(bf16_bits(xv), q, f16_bits(s_vals))
        want = np.zeros(N)
        want[n] = -3 * xv[k] * s_vals[n, k // 32]
        assert np.array_equal(got, want)


def test_gemv_q8_rejects_ragged_group():
    with pytest.raises(ValueError):
        oracle.gemv_q8(np.zeros(40, np.uint16), np.zeros((2, 40), np.int8), np.zeros((2, 1), np.uint16))


# ---- bf16 ----------------------------------------------------------------


def test_bf16_encode_roundtrip_ties_and_random():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = bf16_vals(bits)
    finite = np.isfinite(vals)
    assert np.array_equal(oracle.f64_to_bf16(vals[finite]), bits[finite])
    # Midpoints between consecutive positive finite bf16 values and random values,
    # against torch's conversion (nearest, ties to even).  torch converts float64
    # through float32, so every input here is exactly representable in float32:
    # then its result is a single rounding to bf16.
    pos = np.unique(vals[finite & (vals >= 0)])
    mids = (pos[:-1] + pos[1:]) / 2.0
    rnd = (RNG.standard_normal(50000) * 10.0 ** RNG.integers(-40, 38, 50000)).astype(np.float32)
    x = np.concatenate([mids, -mids, rnd[np.isfinite(rnd)].astype(np.float64),
                        np.array([3.3895313892515355e38, float(np.float32(3.4e38)), 2.0 ** -149, 2.0 ** -134,
                                  3 * 2.0 ** -135, 0.0, -0.0])])
    assert np.array_equal(x.astype(np.float32).astype(np.float64), x)
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.f64_to_bf16(x), want)


def test_gemm_bf16_matches_library_matmul_and_integers():
    M, N, K = 19, 31, 53
    A = bf16_bits(RNG.uniform(-1, 1, (M, K)))
    B = bf16_bits(RNG.uniform(-1, 1, (K, N)))
    want = bf16_vals(A) @ bf16_vals(B)
    assert np.allclose(oracle.gemm(A, B, dtype="bf16"), want, rtol=0, atol=1e-12)
    Ai = RNG.integers(-2, 3, (M, K))
    Bi = RNG.integers(-2, 3, (K, N))
    got = oracle.gemm(bf16_bits(Ai), bf16_bits(Bi), dtype="bf16")
    assert np.array_equal(got, (Ai @ Bi).astype(np.float64))
