"""Special values through the GPU kernels, against the oracle (IEEE semantics:
the oracle computes in float64 and rounds once; NaN payloads are not compared,
only NaN-ness).

  * subnormal inputs: FP16 values down to 2^-24 and BF16 values down to 2^-133
    take part in the products (their products are far inside FP32's range);
  * subnormal outputs: sums that land in FP16's / BF16's subnormal range round
    to the right subnormal;
  * overflow: sums past the format's maximum round to +-Inf;
  * Inf and NaN inputs: Inf * 0 and Inf - Inf give NaN, Inf * x gives +-Inf.
Each case is built from small integers times powers of two, so every product
and partial sum is exact in FP32 and the comparison is bit for bit (up to NaN
payloads).
"""
import numpy as np
import pytest

import oracle
from bf16_gemm_skinny_gb300 import _native as bsk
from bf16_gemm_skinny_gb300 import build as bsk_build
from helpers import from_dev, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    import torch

    bsk_build.build()
    oracle.build()
    torch.cuda.init()
    yield bsk.load()


def same(got_bits, want_bits, decode):
    g = decode(np.asarray(got_bits).reshape(-1))
    w = decode(np.asarray(want_bits).reshape(-1))
    both_nan = np.isnan(g) & np.isnan(w)
    assert np.array_equal(np.isnan(g), np.isnan(w)), "NaN positions differ"
    ok = ~both_nan
    assert np.array_equal(np.asarray(got_bits).reshape(-1)[ok], np.asarray(want_bits).reshape(-1)[ok])


def gemm16(A, B, M, N, K):
    import torch

    C = torch.empty(M * N, dtype=torch.int16, device="cuda")
    bsk.gemm_f16_colmajor(to_dev(A), to_dev(B), C, M, N, K)
    return from_dev(C)


def enc16(x):
    return oracle.f16_encode(np.asarray(x, np.float64).reshape(-1))


def encb(x):
    return oracle.bf16_encode(np.asarray(x, np.float64).reshape(-1))


@pytest.mark.parametrize("M,N,K", [(128, 96, 64), (300, 257, 130)])
def test_fp16_subnormal_inputs_and_outputs(M, N, K):
    """A holds integers times 2^-14 .. 2^-24 (subnormals included), B small
    integers; the sums are integers times 2^-24: some subnormal, some normal."""
    rng = np.random.default_rng(41)
    a = rng.integers(-3, 4, M * K) * 2.0 ** rng.integers(-24, -13, M * K)
    b = rng.integers(-2, 3, K * N).astype(np.float64)
    A, B = enc16(a), enc16(b)
    assert np.array_equal(oracle.f16_decode(A), a) and np.array_equal(oracle.f16_decode(B), b)
    _, want = oracle.gemm_f16_colmajor(A, B, M, N, K)
    got = gemm16(A, B, M, N, K)
    same(got, want, oracle.f16_decode)
    vals = oracle.f16_decode(want)
    assert np.any((vals != 0) & (np.abs(vals) < 2.0 ** -14)), "no subnormal outputs exercised"


def test_fp16_overflow_to_infinity():
    """Rows of +-1024 against 2s sum to +-131072, past FP16's largest (65504): +-Inf;
    the other rows stay finite."""
    M, N, K = 128, 64, 64
    a2 = np.ones((M, K))
    a2[: M // 2] = 1024.0
    a2[: M // 4] = -1024.0
    b = np.full(K * N, 2.0)
    A, B = enc16(a2.T.reshape(-1)), enc16(b)    # A(m, k) at A[m + k*M]
    _, want = oracle.gemm_f16_colmajor(A, B, M, N, K)
    got = gemm16(A, B, M, N, K)
    same(got, want, oracle.f16_decode)
    w = oracle.f16_decode(want)
    assert np.all(np.isposinf(w.reshape(N, M)[:, M // 4: M // 2])) and np.all(np.isneginf(w.reshape(N, M)[:, : M // 4]))
    assert np.all(np.isfinite(w.reshape(N, M)[:, M // 2:]))


def test_fp16_inf_and_nan_propagate():
    M, N, K = 256, 64, 128
    rng = np.random.default_rng(42)
    a = rng.integers(-2, 3, M * K).astype(np.float64)
    b = rng.integers(-2, 3, K * N).astype(np.float64)
    a[5] = np.inf            # column k = 0 of A (MN-major), row 5: Inf * b(0, n)
    a[M * 3 + 7] = -np.inf   # row 7, k = 3
    a[M * 4 + 7] = np.inf    # row 7, k = 4: -Inf + Inf -> NaN where both products are finite-signed
    a[M * 9 + 11] = np.nan
    b[17 * K + 0] = 0.0      # column 17: Inf * 0 -> NaN in row 5
    A, B = enc16(a), enc16(b)
    _, want = oracle.gemm_f16_colmajor(A, B, M, N, K)
    got = gemm16(A, B, M, N, K)
    same(got, want, oracle.f16_decode)
    w = oracle.f16_decode(want)
    assert np.any(np.isnan(w)) and np.any(np.isinf(w))


@pytest.mark.parametrize("n", [1, 4, 8, 24])
def test_bf16_linear_subnormals_and_specials(n):
    """The linear layer (CUDA-core GEMV for n <= 3, tensor cores beyond): BF16
    subnormal weights with subnormal and normal results, an Inf and a NaN."""
    import torch

    M, K = 512, 256
    rng = np.random.default_rng(43 + n)
    w = rng.integers(-3, 4, M * K) * 2.0 ** rng.integers(-133, -120, M * K)   # BF16 subnormals and tiny normals
    x = rng.integers(-2, 3, n * K).astype(np.float64)
    w[10 * K + 5] = np.inf
    w[20 * K + 9] = np.nan
    W, X = encb(w), encb(x)
    finite = np.isfinite(w)
    assert np.array_equal(oracle.bf16_decode(W)[finite], w[finite])
    _, want = oracle.linear_bf16(W, X, M, K, n)
    y = torch.empty(n * M, dtype=torch.int16, device="cuda")
    bsk.gemv_bf16(to_dev(W), to_dev(X), y, M, K, n)
    same(from_dev(y), want, oracle.bf16_decode)
    vals = oracle.bf16_decode(want)
    assert np.any((vals != 0) & (np.abs(vals) < 2.0 ** -126)), "no subnormal outputs exercised"
    assert np.any(np.isnan(vals))


@pytest.mark.parametrize("n", [1, 8])
def test_bf16_linear_overflow_to_infinity(n):
    """Row 3 holds 2^126 and x is positive, so its partial sums only grow and pass
    BF16's (and FP32's) largest value: +Inf; the other rows stay finite."""
    import torch

    M, K = 256, 512
    rng = np.random.default_rng(45)
    w = rng.integers(1, 4, M * K).astype(np.float64)
    w[3 * K: 4 * K] = 2.0 ** 126
    x = rng.integers(1, 3, n * K).astype(np.float64)
    W, X = encb(w), encb(x)
    _, want = oracle.linear_bf16(W, X, M, K, n)
    y = torch.empty(n * M, dtype=torch.int16, device="cuda")
    bsk.gemv_bf16(to_dev(W), to_dev(X), y, M, K, n)
    same(from_dev(y), want, oracle.bf16_decode)
    vals = oracle.bf16_decode(want).reshape(n, M)
    assert np.all(np.isposinf(vals[:, 3])) and np.all(np.isfinite(np.delete(vals, 3, axis=1)))


def test_fp8_special_codes():
    """E5M2 Inf, E4M3 and E5M2 NaN codes, and the formats' subnormals."""
    import torch

    M, N, K = 128, 40, 256
    rng = np.random.default_rng(44)
    for fmt, flag, nan_code, inf_code in (("e4m3", bsk.FP8_E4M3, 0x7F, None), ("e5m2", bsk.FP8_E5M2, 0x7F, 0x7C)):
        A = rng.integers(0, 8, M * K).astype(np.uint8)             # +subnormals and small normals (codes 0..7)
        A |= (rng.integers(0, 2, M * K).astype(np.uint8) << 7)     # random signs
        B = rng.integers(0x30, 0x40, N * K).astype(np.uint8)       # moderate normals
        A[3 * K + 1] = nan_code
        if inf_code is not None:
            A[7 * K + 2] = inf_code
            A[9 * K + 4] = inf_code | 0x80
            A[9 * K + 5] = inf_code            # row 9: -Inf + Inf -> NaN
        _, want = oracle.gemm_fp8(A, B, M, N, K, K, K, fmt, 1.0, "f32")
        C = torch.empty(M * N, dtype=torch.int32, device="cuda")
        bsk.gemm_fp8(flag, torch.from_numpy(A).cuda(), K, torch.from_numpy(B).cuda(), K, C, M, bsk.OUT_F32, M, N,
                     K, 1.0)
        got = C.cpu().numpy().view(np.uint32)
        g = got.view(np.float32).astype(np.float64)
        w = want.view(np.float32).astype(np.float64)
        assert np.array_equal(np.isnan(g), np.isnan(w)), fmt
        ok = ~np.isnan(w)
        assert np.array_equal(got[ok], want[ok]), fmt
