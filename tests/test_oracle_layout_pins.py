"""Pins for the oracle's general FP16 GEMM (transposed operands, row-major
storage, any leading dimension, optional bias).

What the pins rest on, none of it the oracle's own arithmetic:
  * the column-major special case is the column-major oracle, pinned in
    test_oracle_pins.py (same bits, same double sums);
  * transposing or re-storing an operand with numpy, with padding between
    columns, must not change any result;
  * a pure-Python triple loop over the definition on tiny inputs whose
    padding holds NaN (reading padding would show);
  * exact integer products (numpy int64 matmul) plus an integer bias;
  * closed forms: A = 0 gives the bias broadcast exactly, and a bias of 0.5
    on an exact sum of 2049 rounds once to 2050 (rounding the sum first would
    give 2048, then 2048.5 -> 2048).
"""
import itertools

import numpy as np
import pytest

import oracle
from bf16_gemm_skinny_gb300 import inputs

F16_NAN = 0x7E00


def enc(x):
    return oracle.f16_encode(np.asarray(x, np.float64).reshape(-1))


def store(mat_bits, row_major, ld, pad_bits=F16_NAN):
    """Stores the logical R x C matrix `mat_bits` (2-D uint16) with leading
    dimension `ld`; the unused part of each stride holds `pad_bits`."""
    R, C = mat_bits.shape
    if row_major:
        assert ld >= C
        buf = np.full((R, ld), pad_bits, np.uint16)
        buf[:, :C] = mat_bits
    else:
        assert ld >= R
        buf = np.full((C, ld), pad_bits, np.uint16)
        buf[:, :R] = mat_bits.T
    return buf.reshape(-1)


def logical(flat_colmajor, R, C):
    """Flat column-major R x C -> 2-D array."""
    return np.asarray(flat_colmajor).reshape(C, R).T


def operands_2d(M, N, K, dist, seed_a=1, seed_b=2):
    A, B = inputs.gemm_operands(M, N, K, dist, seed_a, seed_b)
    return logical(A, M, K), logical(B, K, N)


def call(A2, B2, transa, transb, row_major, pad_a=3, pad_b=5, **kw):
    """Stores op(A) = A2 and op(B) = B2 in the requested form and runs the oracle."""
    M, K = A2.shape
    N = B2.shape[1]
    sa = A2.T if transa else A2          # the matrix that is stored
    sb = B2.T if transb else B2
    lda = (sa.shape[1] if row_major else sa.shape[0]) + pad_a
    ldb = (sb.shape[1] if row_major else sb.shape[0]) + pad_b
    Af = store(sa, row_major, lda)
    Bf = store(sb, row_major, ldb)
    return oracle.gemm_f16_general(Af, Bf, M, N, K, lda, ldb, transa, transb, row_major, **kw)


def test_column_major_case_is_the_column_major_oracle():
    M, N, K = 67, 45, 93
    A, B = inputs.gemm_operands(M, N, K, "normal0.5", 1, 2)
    r1, o1 = oracle.gemm_f16_colmajor(A, B, M, N, K)
    r2, o2 = oracle.gemm_f16_general(A, B, M, N, K, M, K)
    assert np.array_equal(o1, o2)
    assert np.array_equal(r1, r2)


@pytest.mark.parametrize("transa,transb,row_major", list(itertools.product([0, 1], repeat=3)))
def test_every_storage_form_gives_the_same_product(transa, transb, row_major):
    """All eight forms (NN/NT/TN/TT, column- and row-major, padded strides)
    agree bit for bit with the plain column-major oracle."""
    M, N, K = 37, 29, 41
    A2, B2 = operands_2d(M, N, K, "normal0.5")
    ref0, out0 = oracle.gemm_f16_colmajor(A2.T.reshape(-1), B2.T.reshape(-1), M, N, K)
    ref, out = call(A2, B2, transa, transb, row_major)
    assert np.array_equal(out, out0)
    assert np.array_equal(ref, ref0)


def brute(A2, B2, bias=None, mode=0):
    """Pure-Python definition: C(m,n) = sum_k A(m,k) B(k,n) (+ bias), in double."""
    a = oracle.f16_decode(A2.reshape(-1)).reshape(A2.shape)
    b = oracle.f16_decode(B2.reshape(-1)).reshape(B2.shape)
    bz = None if bias is None else oracle.f16_decode(bias)
    M, K = a.shape
    N = b.shape[1]
    c = np.zeros((M, N))
    for m in range(M):
        for n in range(N):
            s = 0.0
            for k in range(K):
                s += float(a[m, k]) * float(b[k, n])
            if mode == 1:
                s += float(bz[m])
            elif mode == 2:
                s += float(bz[n])
            c[m, n] = s
    return c


@pytest.mark.parametrize("transa,transb,row_major,mode", [
    (0, 0, 0, 0), (1, 0, 0, 1), (0, 1, 0, 2), (1, 1, 0, 1), (0, 0, 1, 2), (1, 0, 1, 0), (0, 1, 1, 1), (1, 1, 1, 2)])
def test_tiny_brute_force_with_nan_padding(transa, transb, row_major, mode):
    M, N, K = 5, 4, 3
    A2, B2 = operands_2d(M, N, K, "normal0.5", 21, 22)
    bias = enc(np.linspace(-1.5, 2.0, max(M, N))) if mode else None
    ref, out = call(A2, B2, transa, transb, row_major, bias=bias, bias_mode=mode)
    want = brute(A2, B2, bias, mode)
    got = logical(ref, M, N)
    assert np.all(np.isfinite(got)), "padding was read"
    np.testing.assert_allclose(got, want, rtol=1e-14, atol=1e-14)
    assert np.array_equal(out, enc(want.T.reshape(-1)))


@pytest.mark.parametrize("transa,transb,row_major,mode", [(0, 1, 0, 2), (1, 0, 1, 1), (1, 1, 0, 2), (0, 0, 1, 1)])
def test_integer_inputs_exact(transa, transb, row_major, mode):
    """Entries in {-2..2} and an integer bias: every sum is an integer well
    inside FP16's exact range, so the result is the integer product."""
    M, N, K = 70, 52, 96
    A2, B2 = operands_2d(M, N, K, "int2", 11, 12)
    rng = np.random.default_rng(5)
    bias_i = rng.integers(-40, 41, max(M, N))
    _, out = call(A2, B2, transa, transb, row_major, bias=enc(bias_i), bias_mode=mode)
    ai = oracle.f16_decode(A2.reshape(-1)).reshape(M, K).astype(np.int64)
    bi = oracle.f16_decode(B2.reshape(-1)).reshape(K, N).astype(np.int64)
    c = ai @ bi + (bias_i[:M, None] if mode == 1 else bias_i[None, :N])
    assert np.array_equal(out, enc(c.T.reshape(-1)))


@pytest.mark.parametrize("mode", [1, 2])
def test_zero_product_gives_the_bias(mode):
    M, N, K = 6, 9, 4
    A2 = np.zeros((M, K), np.uint16)
    _, B2 = operands_2d(M, N, K, "normal0.5")
    bias = enc(np.arange(1, max(M, N) + 1) * 0.375 - 2.0)
    _, out = call(A2, B2, 0, 1, 0, bias=bias, bias_mode=mode)
    want = np.tile(bias[:M], N) if mode == 1 else np.repeat(bias[:N], M)
    assert np.array_equal(out, want)


def test_bias_joins_the_single_rounding():
    """2048 * 1 + 1 * 1 = 2049 exactly; + 0.5 = 2049.5 -> FP16 2050 (spacing 2 there)."""
    A2 = enc([2048.0, 1.0]).reshape(1, 2)
    B2 = enc([1.0, 1.0]).reshape(2, 1)
    for mode in (1, 2):
        ref, out = call(A2, B2, 0, 0, 0, bias=enc([0.5]), bias_mode=mode)
        assert ref[0] == 2049.5
        assert oracle.f16_decode(out)[0] == 2050.0
    _, out = call(A2, B2, 0, 0, 0)
    assert oracle.f16_decode(out)[0] == 2048.0   # 2049 is a tie: even significand


def test_row_and_column_selection():
    M, N, K = 40, 33, 50
    A2, B2 = operands_2d(M, N, K, "normal0.5")
    bias = enc(np.linspace(-1, 1, N))
    ref, out = call(A2, B2, 1, 1, 1, bias=bias, bias_mode=2)
    rows, cols = [0, 7, 39], [32, 1, 5]
    rs, os_ = call(A2, B2, 1, 1, 1, bias=bias, bias_mode=2, rows=rows, cols=cols)
    full = logical(out, M, N)
    assert np.array_equal(logical(os_, 3, 3), full[np.ix_(rows, cols)])
    assert np.array_equal(logical(rs, 3, 3), logical(ref, M, N)[np.ix_(rows, cols)])


def test_rejects_bad_arguments():
    A2, B2 = operands_2d(4, 4, 4, "normal0.5")
    with pytest.raises(ValueError):
        oracle.gemm_f16_general(A2.reshape(-1), B2.reshape(-1), 4, 4, 4, 8, 4)   # lda too large for A
    with pytest.raises(RuntimeError):
        oracle.gemm_f16_general(A2.T.reshape(-1), B2.T.reshape(-1), 4, 4, 4, 4, 4, bias=enc([1, 2, 3, 4]),
                                bias_mode=3)
