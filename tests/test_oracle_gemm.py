"""Pins for oracle.gemm: closed forms, brute force, library routine on exact cases,
layout equivalence, the MXFP8 dequantisation and planted mistakes in the checker."""
import itertools

import numpy as np
import pytest

import synthetic
from oracle import gemm as G
from oracle import numerics as nm


def _bf16(x):
    return nm.bf16_bits_to_f64(synthetic.f64_to_bf16_bits(x))


def test_identity_gives_b():
    K = N = 96
    B = _bf16(np.random.default_rng(0).uniform(-1, 1, (K, N)))
    C, Ca = G.gemm_full(np.eye(K), B, True, K, N, K)
    assert np.array_equal(C, B)
    assert np.array_equal(Ca, np.abs(B))


@pytest.mark.parametrize("K", [1, 256, 8192])
def test_all_ones_gives_k(K):
    M, N = 3, 5
    C, Ca = G.gemm_full(np.ones((M, K)), np.ones((K, N)), True, M, N, K)
    assert np.all(C == K) and np.all(Ca == K)
    assert np.all(nm.bf16_bits_to_f64(nm.f64_to_bf16_rne(C)) == K)  # K exact in bf16


def test_k1_outer_product():
    rng = np.random.default_rng(1)
    a = _bf16(rng.uniform(-1, 1, (17, 1)))
    b = _bf16(rng.uniform(-1, 1, (1, 23)))
    C, _ = G.gemm_full(a, b, True, 17, 23, 1)
    assert np.array_equal(C, a[:, 0][:, None] * b[0][None, :])


def test_brute_force_tiny():
    rng = np.random.default_rng(2)
    for M, N, K in [(1, 1, 1), (3, 4, 5), (8, 8, 8), (7, 2, 9)]:
        A = _bf16(rng.uniform(-1, 1, (M, K)))
        B = _bf16(rng.uniform(-1, 1, (K, N)))
        C, Ca = G.gemm_full(A, B, True, M, N, K)
        for i, j in itertools.product(range(M), range(N)):
            s = 0.0
            sa = 0.0
            for k in range(K):
                s += A[i, k] * B[k, j]
                sa += abs(A[i, k]) * abs(B[k, j])
            assert C[i, j] == s and Ca[i, j] == sa


def test_numpy_matmul_on_exact_integer_inputs():
    rng = np.random.default_rng(3)
    A = rng.integers(-8, 9, (64, 80)).astype(np.float64)
    B = rng.integers(-8, 9, (80, 48)).astype(np.float64)
    C, Ca = G.gemm_full(A, B, True, 64, 48, 80)
    assert np.array_equal(C, A @ B)
    assert np.array_equal(Ca, np.abs(A) @ np.abs(B))


def test_layouts_and_entries_agree():
    rng = np.random.default_rng(4)
    M, N, K = 33, 41, 70
    A = _bf16(rng.uniform(-1, 1, (M, K)))
    B = _bf16(rng.uniform(-1, 1, (K, N)))
    C1, A1 = G.gemm_full(A, B, True, M, N, K)
    C2, A2 = G.gemm_full(A, np.ascontiguousarray(B.T), False, M, N, K)
    assert np.array_equal(C1, C2) and np.array_equal(A1, A2)
    ii = rng.integers(0, M, 50)
    jj = rng.integers(0, N, 50)
    Ce, Ae = G.gemm_entries(A, B, True, K, ii, jj)
    assert np.array_equal(Ce, C1[ii, jj]) and np.array_equal(Ae, A1[ii, jj])
    # padded leading dimensions are ignored beyond K / N
    Ap = np.zeros((M, K + 6))
    Ap[:, :K] = A
    Ap[:, K:] = 1e30
    Cp, _ = G.gemm_full(Ap, B, True, M, N, K)
    assert np.array_equal(Cp, C1)


def test_abs_bound_dominates():
    rng = np.random.default_rng(5)
    A = rng.standard_normal((20, 30))
    B = rng.standard_normal((30, 25))
    C, Ca = G.gemm_full(A, B, True, 20, 25, 30)
    assert np.all(np.abs(C) <= Ca)
    Cp, Cap = G.gemm_full(np.abs(A), np.abs(B), True, 20, 25, 30)
    assert np.array_equal(Cp, Cap)


def test_mxfp8_unit_payload_closed_form():
    M, N, K = 4, 6, 512
    qa = np.full((M, K), 0x38, np.uint8)  # 1.0
    qb = np.full((N, K), 0x38, np.uint8)
    sa = (127 + np.arange(M) - 2).astype(np.uint8)[:, None].repeat(K // 128, 1)
    sb = (127 - np.arange(N) + 3).astype(np.uint8)[:, None].repeat(K // 128, 1)
    A = G.dequant_mxfp8(qa, sa)
    B = G.dequant_mxfp8(qb, sb)
    C, _ = G.gemm_full(A, B, False, M, N, K)
    expect = K * np.ldexp(1.0, (np.arange(M)[:, None] - 2) + (-np.arange(N)[None, :] + 3))
    assert np.array_equal(C, expect)


def test_mxfp8_scale_applies_to_its_k_block_only():
    q = np.full((2, 384), 0x38, np.uint8)
    s = np.full((2, 3), 127, np.uint8)
    s[0, 1] = 130  # x8 on columns 128..255 of row 0
    A = G.dequant_mxfp8(q, s)
    assert np.all(A[0, :128] == 1) and np.all(A[0, 128:256] == 8) and np.all(A[0, 256:] == 1)
    assert np.all(A[1] == 1)


def test_checker_accepts_rounded_result_and_rejects_planted_errors():
    rng = np.random.default_rng(6)
    A = _bf16(rng.uniform(-1, 1, (64, 256)))
    B = _bf16(rng.uniform(-1, 1, (256, 64)))
    C64, Abs = G.gemm_full(A, B, True, 64, 64, 256)
    ref_bits = nm.f64_to_bf16_rne(C64)
    info = G.check(ref_bits, C64, Abs)
    assert info["frob_rel"] == 0.0
    # the same numbers accumulated in fp32 also pass
    c32 = (A.astype(np.float32) @ B.astype(np.float32)).astype(np.float64)
    G.check(nm.f64_to_bf16_rne(c32), C64, Abs)
    bad = ref_bits.copy()  # one element off by 3% of its |A|.|B| bound
    bad[3, 5] = nm.f64_to_bf16_rne(C64[3, 5] + 3e-2 * Abs[3, 5])
    with pytest.raises(AssertionError):
        G.check(bad, C64, Abs)
    with pytest.raises(AssertionError):  # a transposed result
        G.check(np.ascontiguousarray(ref_bits.T), C64, Abs)
    with pytest.raises(AssertionError):  # a dropped K block
        C_drop, _ = G.gemm_full(A[:, :192], B[:192], True, 64, 64, 192)
        G.check(nm.f64_to_bf16_rne(C_drop), C64, Abs)


def test_epilogue_identity_and_closed_form():
    rng = np.random.default_rng(8)
    C64 = rng.standard_normal((5, 7))
    Abs = np.abs(C64) + 1.0
    C1, A1 = G.epilogue(C64, Abs)
    assert np.array_equal(C1, C64) and np.array_equal(A1, Abs)
    # all-ones operands: C = alpha * K + bias[n], exact
    K = 256
    C, Ab = G.gemm_full(np.ones((3, K)), np.ones((K, 4)), True, 3, 4, K)
    bias = np.array([0.5, -1.0, 2.0, 0.0])
    Ce, Ae = G.epilogue(C, Ab, alpha=0.25, bias=bias)
    assert np.array_equal(Ce, np.tile(0.25 * K + bias, (3, 1)))
    assert np.array_equal(Ae, np.tile(0.25 * K + np.abs(bias), (3, 1)))


def test_epilogue_checker_rejects_missing_bias_or_scale():
    rng = np.random.default_rng(9)
    A = _bf16(rng.uniform(-1, 1, (32, 128)))
    B = _bf16(rng.uniform(-1, 1, (128, 48)))
    C64, Abs = G.gemm_full(A, B, True, 32, 48, 128)
    bias = rng.uniform(-4, 4, 48)
    Ce, Ae = G.epilogue(C64, Abs, alpha=-1.5, bias=bias)
    G.check(nm.f64_to_bf16_rne(Ce), Ce, Ae)
    with pytest.raises(AssertionError):  # bias dropped
        G.check(nm.f64_to_bf16_rne(-1.5 * C64), Ce, Ae)
    with pytest.raises(AssertionError):  # scale dropped
        G.check(nm.f64_to_bf16_rne(C64 + bias[None, :]), Ce, Ae)
