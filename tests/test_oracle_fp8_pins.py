"""Pins for the oracle's FP8 GEMM (E4M3 / E5M2 inputs, FP32 accumulator, FP32
or BF16 output) and for its FP8 decoder and binary32 encoder.

What the pins rest on, none of it the oracle's own arithmetic:
  * every one of the 256 codes of each format decodes as torch's float8_e4m3fn
    / float8_e5m2 types do, plus the formats' landmark values written out;
  * the binary32 encoder agrees with numpy's float64 -> float32 cast on random
    values, ties and the edges of the range;
  * E4M3 values are exactly FP16 values, so the FP8 GEMM's exact sums equal
    the pinned FP16 oracle's on the same numbers;
  * exact integer products (numpy int64 matmul) times an exact alpha;
  * a pure-Python loop over the definition with exact rational sums;
  * closed forms where rounding once from the exact sum differs from rounding
    through FP32 first.
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle
from bf16_gemm_skinny_gb300 import inputs

FMTS = ("e4m3", "e5m2")


def torch_decode(codes, fmt):
    import torch

    dt = {"e4m3": torch.float8_e4m3fn, "e5m2": torch.float8_e5m2}[fmt]
    t = torch.from_numpy(np.ascontiguousarray(codes, np.uint8)).view(dt)
    return t.to(torch.float64).numpy()


@pytest.mark.parametrize("fmt", FMTS)
def test_decode_all_codes_match_torch(fmt):
    codes = np.arange(256, dtype=np.uint8)
    got = oracle.fp8_decode(codes, fmt)
    want = torch_decode(codes, fmt)
    assert np.array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    assert np.array_equal(got[ok], want[ok])
    assert np.array_equal(np.signbit(got[ok]), np.signbit(want[ok]))


def test_decode_landmarks():
    e4 = lambda c: float(oracle.fp8_decode(np.array([c], np.uint8), "e4m3")[0])  # noqa: E731
    e5 = lambda c: float(oracle.fp8_decode(np.array([c], np.uint8), "e5m2")[0])  # noqa: E731
    assert e4(0x38) == 1.0 and e4(0xB8) == -1.0
    assert e4(0x7E) == 448.0                       # largest E4M3
    assert e4(0x01) == 2.0 ** -9                   # smallest subnormal
    assert e4(0x08) == 2.0 ** -6                   # smallest normal
    assert e4(0x07) == 7 * 2.0 ** -9
    assert np.isnan(e4(0x7F)) and np.isnan(e4(0xFF))
    assert e4(0x78) == 256.0                       # exponent 15 is a normal binade in E4M3
    assert e5(0x3C) == 1.0
    assert e5(0x7B) == 57344.0                     # largest E5M2
    assert e5(0x7C) == np.inf and e5(0xFC) == -np.inf
    assert np.isnan(e5(0x7D))
    assert e5(0x01) == 2.0 ** -16 and e5(0x04) == 2.0 ** -14
    assert e5(0x80) == 0.0 and np.signbit(e5(0x80))


def test_f32_encoder_matches_numpy():
    rng = np.random.default_rng(3)
    x = np.concatenate([rng.standard_normal(20000) * 10.0 ** rng.integers(-40, 39, 20000),
                        [0.0, -0.0, 1.0, 3.4028234663852886e38, 1e-45, 1.4e-45, 7e-46, 2e-38]])
    got = oracle.f32_encode(x)
    want = x.astype(np.float32).view(np.uint32)
    assert np.array_equal(got, want)
    # ties to even at 1.0 (spacing 2^-23) and the overflow threshold
    t = np.array([1 + 2.0 ** -24, 1 + 3 * 2.0 ** -24, 2.0 ** 128 * (1 - 2.0 ** -25), 2.0 ** 128])
    assert list(oracle.f32_encode(t)) == [0x3F800000, 0x3F800002, 0x7F800000, 0x7F800000]
    assert oracle.f32_encode(np.array([np.nan]))[0] & 0x7FC00000 == 0x7FC00000


@pytest.mark.parametrize("fmt,alpha", [("e4m3", 1.0), ("e4m3", 0.5), ("e5m2", -2.0), ("e5m2", 0.25)])
def test_integer_inputs_exact(fmt, alpha):
    M, N, K = 37, 23, 300
    A, B = inputs.fp8_operands(M, N, K, "int2", fmt, 11, 12)
    a = oracle.fp8_decode(A, fmt).reshape(M, K).astype(np.int64)
    b = oracle.fp8_decode(B, fmt).reshape(N, K).astype(np.int64)
    c = (a @ b.T).astype(np.float64) * alpha            # C(m, n)
    ref, out = oracle.gemm_fp8(A, B, M, N, K, K, K, fmt, alpha, "f32")
    assert np.array_equal(ref, c.T.reshape(-1))
    assert np.array_equal(out, c.T.reshape(-1).astype(np.float32).view(np.uint32))


def test_e4m3_sums_equal_the_fp16_oracle():
    """E4M3 values are FP16 values: the exact sums must agree bit for bit with
    the FP16 oracle's (A K-major = transa, B K-major = no transpose)."""
    M, N, K = 41, 19, 210
    A, B = inputs.fp8_operands(M, N, K, "normal1", "e4m3", 1, 2)
    Ah = oracle.f16_encode(oracle.fp8_decode(A, "e4m3"))       # exact conversion
    Bh = oracle.f16_encode(oracle.fp8_decode(B, "e4m3"))
    ref8, _ = oracle.gemm_fp8(A, B, M, N, K, K, K, "e4m3")
    ref16, _ = oracle.gemm_f16_general(Ah, Bh, M, N, K, K, K, transa=1, transb=0)
    assert np.array_equal(ref8, ref16)


@pytest.mark.parametrize("fmt", FMTS)
def test_tiny_brute_force_with_nan_padding(fmt):
    M, N, K, pad = 4, 3, 5, 3
    rng = np.random.default_rng(9)
    vals = rng.standard_normal((M + N) * K)
    codes = inputs.to_fp8_bits(vals, fmt)
    a_codes = codes[:M * K].reshape(M, K)
    b_codes = codes[M * K:].reshape(N, K)
    nan = 0x7F
    A = np.full((M, K + pad), nan, np.uint8)
    A[:, :K] = a_codes
    B = np.full((N, K + pad), nan, np.uint8)
    B[:, :K] = b_codes
    alpha = 0.75
    ref, out = oracle.gemm_fp8(A, B, M, N, K, K + pad, K + pad, fmt, alpha, "bf16")
    av = torch_decode(a_codes.reshape(-1), fmt).reshape(M, K)
    bv = torch_decode(b_codes.reshape(-1), fmt).reshape(N, K)
    for m in range(M):
        for n in range(N):
            exact = sum(Fraction(float(av[m, k])) * Fraction(float(bv[n, k])) for k in range(K)) * Fraction(alpha)
            assert ref[m + n * M] == float(exact), (m, n)
    assert np.array_equal(out, oracle.bf16_encode(ref))


def test_single_rounding_from_the_exact_sum():
    """E5M2: 1*1 + 2^-4*2^-4 + 2^-15*2^-15 = 1 + 2^-8 + 2^-30 exactly.  BF16 of
    that is 1 + 2^-7 (0x3F81); rounding to FP32 first would give the tie
    1 + 2^-8 and then 1.0.  FP32 output: 1 + 2^-8 (0x3F808000)."""
    one, sixteenth, tiny = 0x3C, 0x2C, 0x02      # 1.0, 2^-4, 2^-15 in E5M2
    vals = oracle.fp8_decode(np.array([one, sixteenth, tiny], np.uint8), "e5m2")
    assert list(vals) == [1.0, 2.0 ** -4, 2.0 ** -15]
    A = np.array([one, sixteenth, tiny], np.uint8)
    B = A.copy()
    ref, o16 = oracle.gemm_fp8(A, B, 1, 1, 3, 3, 3, "e5m2", 1.0, "bf16")
    assert ref[0] == 1 + 2.0 ** -8 + 2.0 ** -30
    assert o16[0] == 0x3F81
    _, o32 = oracle.gemm_fp8(A, B, 1, 1, 3, 3, 3, "e5m2", 1.0, "f32")
    assert o32[0] == 0x3F808000


def test_selection_and_zero_k():
    M, N, K = 30, 20, 64
    A, B = inputs.fp8_operands(M, N, K, "normal1", "e5m2")
    ref, out = oracle.gemm_fp8(A, B, M, N, K, K, K, "e5m2", 1.0, "bf16")
    rows, cols = [0, 29, 3], [19, 0]
    rs, os_ = oracle.gemm_fp8(A, B, M, N, K, K, K, "e5m2", 1.0, "bf16", rows=rows, cols=cols)
    full = ref.reshape(N, M).T
    assert np.array_equal(rs.reshape(2, 3).T, full[np.ix_(rows, cols)])
    ref0, out0 = oracle.gemm_fp8(np.zeros(0, np.uint8), np.zeros(0, np.uint8), 3, 2, 0, 1, 1)
    assert np.all(ref0 == 0) and np.all(out0 == 0)
