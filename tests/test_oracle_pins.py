"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each check below would fail for a plausible slip in ``oracle/oracle.c``:
a wrong exponent bias or fraction width (codec checks against numpy/torch and
exhaustive round trips), double rounding or truncation (tie and
double-rounding cases, exact rational brute force), a dropped k term or an
off-by-one k range (closed-form column sums, exact brute force), a transposed
operand or wrong column-major index (identity, permutation, transpose
identity, rank-1 with distinct row/column scales), a sign error (signed
inputs everywhere).

Definitions pinned: the GEMM of "MTT S4000 GEMM 优化中的分块、尾处理与并发实战复盘"
section 2 (GEMM入门; triple loop and column-major addressing) with section 1's
FP16 in / FP16 out contract, and the linear layer Y = X W^T of the DCU
decode-GEMV article, section 6.1.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")

ALL = np.arange(65536, dtype=np.uint32).astype(np.uint16)


# --------------------------------------------------------------------------
# Independent references: numpy's float16 and torch's bfloat16
# --------------------------------------------------------------------------

def np_f16_values():
    return ALL.view(np.float16).astype(np.float64)


def torch_bf16_values():
    return torch.from_numpy(ALL.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()


def _is_nan_bits_f16(b):
    return ((b >> 10) & 0x1F) == 0x1F and (b & 0x3FF) != 0


def _is_nan_bits_bf16(b):
    return ((b >> 7) & 0xFF) == 0xFF and (b & 0x7F) != 0


def test_f16_decode_matches_numpy_exhaustive(oracle_mod):
    ours = oracle.f16_decode(ALL)
    ref = np_f16_values()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    # signed zeros decode with their sign
    assert np.signbit(ours[0x8000]) and not np.signbit(ours[0])


def test_bf16_decode_matches_torch_exhaustive(oracle_mod):
    ours = oracle.bf16_decode(ALL)
    ref = torch_bf16_values()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])


def test_f16_round_trip_exhaustive(oracle_mod):
    back = oracle.f16_encode(oracle.f16_decode(ALL))
    nan = np.array([_is_nan_bits_f16(int(b)) for b in ALL])
    assert np.array_equal(back[~nan], ALL[~nan])
    assert all(_is_nan_bits_f16(int(b)) for b in back[nan])


def test_bf16_round_trip_exhaustive(oracle_mod):
    back = oracle.bf16_encode(oracle.bf16_decode(ALL))
    nan = np.array([_is_nan_bits_bf16(int(b)) for b in ALL])
    assert np.array_equal(back[~nan], ALL[~nan])
    assert all(_is_nan_bits_bf16(int(b)) for b in back[nan])


def test_f16_encode_matches_numpy_direct_cast(oracle_mod):
    """numpy casts float64 -> float16 with one correct rounding; compare on wide random samples."""
    rng = np.random.default_rng(7)
    mags = np.ldexp(rng.uniform(1.0, 2.0, 200_000), rng.integers(-30, 18, 200_000))
    x = mags * rng.choice([-1.0, 1.0], mags.size)
    # exact midpoints between neighbouring halves, where truncation or double rounding shows
    finite = np.sort(np.unique(np_f16_values()[np.isfinite(np_f16_values())]))
    mids = (finite[:-1] + finite[1:]) / 2.0
    x = np.concatenate([x, mids, -mids, [0.0, -0.0, 65504.0, 65519.9, 65520.0, 1e6, -1e6]])
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(oracle.f16_encode(x), ref)


def _nearest_even(x: Fraction, table_vals, table_bits, frac_mask, inf_val, inf_bits):
    """Brute force round-to-nearest-even of an exact rational over a sorted value table."""
    import bisect

    if x == 0:
        return 0
    neg = x < 0
    a = -x if neg else x
    vals = table_vals + [inf_val]
    bits = table_bits + [inf_bits]
    i = bisect.bisect_left(vals, a)
    if i == len(vals):
        r = inf_bits
    elif vals[i] == a:
        r = bits[i]
    else:
        lo, hi = vals[i - 1], vals[i]
        dlo, dhi = a - lo, hi - a
        if dlo < dhi:
            r = bits[i - 1]
        elif dhi < dlo:
            r = bits[i]
        else:
            r = bits[i - 1] if (bits[i - 1] & 1) == 0 else bits[i]
    return r | (0x8000 if neg else 0)


def _positive_table(values, bits):
    keep = [(Fraction(float(v)), int(b)) for v, b in zip(values, bits)
            if np.isfinite(v) and v >= 0 and not (v == 0 and b != 0)]
    keep.sort()
    return [k[0] for k in keep], [k[1] for k in keep]


def test_bf16_encode_matches_exact_brute_force(oracle_mod):
    vals, bits = _positive_table(torch_bf16_values(), ALL)
    rng = np.random.default_rng(11)
    xs = list(np.ldexp(rng.uniform(1.0, 2.0, 3000), rng.integers(-140, 129, 3000)))
    xs += [-v for v in xs[:500]]
    # midpoints (ties) between neighbours and points just off them
    for i in rng.integers(0, len(vals) - 1, 400):
        mid = (vals[i] + vals[i + 1]) / 2
        xs += [float(mid), float(mid) * (1 + 2.0 ** -40), float(mid) * (1 - 2.0 ** -40)]
    xs = np.array(xs, np.float64)
    ours = oracle.bf16_encode(xs)
    inf_val = Fraction(2) ** 128
    for x, o in zip(xs, ours):
        want = _nearest_even(Fraction(float(x)), vals, bits, 0x7F, inf_val, 0x7F80)
        assert int(o) == want, (x, hex(int(o)), hex(want))


@pytest.mark.parametrize("x,bits", [
    (1 + 2.0 ** -11, 0x3C00),                 # tie -> even (1.0)
    (1 + 3 * 2.0 ** -11, 0x3C02),             # tie -> even (1 + 2^-9)
    (1 + 2.0 ** -11 + 2.0 ** -40, 0x3C01),    # just above the tie: no double rounding
    (2.0 ** -25, 0x0000),                     # half the smallest subnormal: tie -> 0
    (3 * 2.0 ** -25, 0x0002),                 # tie between subnormals 1 and 2 -> even
    (2.0 ** -14 - 2.0 ** -26, 0x0400),        # rounds up into the smallest normal
    (65504.0, 0x7BFF), (65519.99, 0x7BFF), (65520.0, 0x7C00), (-65520.0, 0xFC00),
])
def test_f16_encode_special_cases(oracle_mod, x, bits):
    assert int(oracle.f16_encode(np.array([x]))[0]) == bits


@pytest.mark.parametrize("x,bits", [
    (1 + 2.0 ** -8, 0x3F80),                  # tie -> even (1.0)
    (1 + 3 * 2.0 ** -8, 0x3F82),              # tie -> even
    (1 + 2.0 ** -8 + 2.0 ** -40, 0x3F81),     # going through float32 first would give 0x3F80
    (-(1 + 2.0 ** -8 + 2.0 ** -40), 0xBF81),
    (2.0 ** -134, 0x0000),                    # tie -> 0
    (3 * 2.0 ** -134, 0x0002),
    ((2 - 2.0 ** -7) * 2.0 ** 127, 0x7F7F),   # largest finite
    ((2 - 2.0 ** -8) * 2.0 ** 127, 0x7F80),   # tie above the largest finite -> Inf
])
def test_bf16_encode_special_cases(oracle_mod, x, bits):
    assert int(oracle.bf16_encode(np.array([x]))[0]) == bits


# --------------------------------------------------------------------------
# GEMM pins
# --------------------------------------------------------------------------

def f16(vals):
    return np.asarray(vals, np.float64).astype(np.float16).view(np.uint16).reshape(-1)


def colmajor(mat):
    """2-D float array -> flat column-major FP16 bits."""
    return f16(np.asarray(mat, np.float64).T.reshape(-1))


def test_gemm_identity_right_and_left(oracle_mod):
    rng = np.random.default_rng(1)
    M, K = 37, 29
    a = rng.uniform(-3, 3, (M, K))
    A = colmajor(a)
    I = colmajor(np.eye(K))
    _, C = oracle.gemm_f16_colmajor(A, I, M, K, K)
    assert np.array_equal(C, A)                      # A * I == A, bit for bit
    b = rng.uniform(-3, 3, (M, 23))
    B = colmajor(b)
    _, C2 = oracle.gemm_f16_colmajor(colmajor(np.eye(M)), B, M, 23, M)
    assert np.array_equal(C2, B)                     # I * B == B


def test_gemm_permutation_permutes_columns(oracle_mod):
    rng = np.random.default_rng(2)
    M, K = 19, 31
    a = rng.uniform(-2, 2, (M, K))
    perm = rng.permutation(K)
    P = np.zeros((K, K))
    P[perm, np.arange(K)] = 1.0                      # column n of P selects row perm[n]
    _, C = oracle.gemm_f16_colmajor(colmajor(a), colmajor(P), M, K, K)
    want = colmajor(a[:, perm])
    assert np.array_equal(C, want)


def test_gemm_rank1_closed_form(oracle_mod):
    """A(m,k) = alpha_m, B(k,n) = beta_n  =>  C(m,n) = K * alpha_m * beta_n (exactly representable)."""
    M, N, K = 6, 5, 48
    alpha = np.array([0.5, -1.0, 2.0, 0.25, -0.75, 1.5])
    beta = np.array([1.0, -0.5, 0.125, 3.0, -2.0])
    a = np.repeat(alpha[:, None], K, axis=1)
    b = np.repeat(beta[None, :], K, axis=0)
    ref, C = oracle.gemm_f16_colmajor(colmajor(a), colmajor(b), M, N, K)
    want = K * np.outer(alpha, beta)
    assert np.array_equal(ref.reshape(N, M).T, want)
    assert np.array_equal(C, colmajor(want))


def test_gemm_rank1_with_rounding(oracle_mod):
    """(1+2^-10)^2 * 3 = 3 + 3*2^-9 + 3*2^-20, which rounds once to 3 + 3*2^-9."""
    K = 3
    v = 1 + 2.0 ** -10
    ref, C = oracle.gemm_f16_colmajor(colmajor([[v] * K]), colmajor([[v]] * K), 1, 1, K)
    assert ref[0] == 3 * v * v
    assert C[0] == f16([3 + 3 * 2.0 ** -9])[0]


@pytest.mark.parametrize("K", [1, 2, 3, 4, 5, 6, 7, 11, 64, 257])
def test_gemm_closed_form_column_sum(oracle_mod, K):
    """A == 1, B(k,n) = (k mod 5) - 2 + n: each full period of k mod 5 sums to 0."""
    M, N = 4, 3
    k = np.arange(K)
    b = ((k % 5) - 2)[:, None] + np.arange(N)[None, :]
    ref, _ = oracle.gemm_f16_colmajor(colmajor(np.ones((M, K))), colmajor(b), M, N, K)
    partial = {0: 0, 1: -2, 2: -3, 3: -3, 4: -2}[K % 5]
    for n in range(N):
        assert np.all(ref[n * M:(n + 1) * M] == partial + n * K)


def _exact_f16_gemm(a, b):
    """Exact rational GEMM, rounded by brute force over every finite FP16 value."""
    vals, bits = _positive_table(np_f16_values(), ALL)
    M, K = a.shape
    N = b.shape[1]
    out = np.empty(M * N, np.uint16)
    for n in range(N):
        for m in range(M):
            s = sum((Fraction(float(a[m, k])) * Fraction(float(b[k, n])) for k in range(K)), Fraction(0))
            out[m + n * M] = _nearest_even(s, vals, bits, 0x3FF, Fraction(65536), 0x7C00)
    return out


@pytest.mark.parametrize("seed", range(6))
def test_gemm_brute_force_tiny_shapes(oracle_mod, seed):
    rng = np.random.default_rng(100 + seed)
    M, N, K = (int(v) for v in rng.integers(1, 7, 3))
    if seed % 2:
        a = rng.integers(-2, 3, (M, K)).astype(np.float64)
        b = rng.integers(-2, 3, (K, N)).astype(np.float64)
    else:
        a = rng.uniform(-1, 1, (M, K)).astype(np.float16).astype(np.float64)
        b = rng.uniform(-1, 1, (K, N)).astype(np.float16).astype(np.float64)
    _, C = oracle.gemm_f16_colmajor(colmajor(a), colmajor(b), M, N, K)
    assert np.array_equal(C, _exact_f16_gemm(a, b))


def test_gemm_transpose_identity(oracle_mod):
    """(A B)^T = B^T A^T through the column-major reinterpretation, bit for bit."""
    rng = np.random.default_rng(3)
    M, N, K = 23, 17, 41
    a = rng.uniform(-1, 1, (M, K))
    b = rng.uniform(-1, 1, (K, N))
    _, C = oracle.gemm_f16_colmajor(colmajor(a), colmajor(b), M, N, K)
    _, Ct = oracle.gemm_f16_colmajor(colmajor(b.T), colmajor(a.T), N, M, K)
    assert np.array_equal(C.reshape(N, M).T, Ct.reshape(M, N))


def test_gemm_subsets_agree_with_full(oracle_mod):
    rng = np.random.default_rng(4)
    M, N, K = 33, 21, 50
    A = colmajor(rng.uniform(-1, 1, (M, K)))
    B = colmajor(rng.uniform(-1, 1, (K, N)))
    ref, C = oracle.gemm_f16_colmajor(A, B, M, N, K)
    cols = [0, 5, 20]
    refc, Cc = oracle.gemm_f16_colmajor(A, B, M, N, K, cols=cols)
    for j, n in enumerate(cols):
        assert np.array_equal(Cc[j * M:(j + 1) * M], C[n * M:(n + 1) * M])
        assert np.array_equal(refc[j * M:(j + 1) * M], ref[n * M:(n + 1) * M])
    rows = [0, 7, 32]
    refr, Cr = oracle.gemm_f16_colmajor_rows(A, B, M, N, K, rows)
    for i, m in enumerate(rows):
        assert np.array_equal(Cr[i::len(rows)], C[m::M])


def test_gemm_integer_inputs_are_exact(oracle_mod):
    """Integer entries in {-2..2}: every sum is an integer, so ref equals the integer product."""
    rng = np.random.default_rng(5)
    M, N, K = 40, 30, 200
    a = rng.integers(-2, 3, (M, K))
    b = rng.integers(-2, 3, (K, N))
    ref, C = oracle.gemm_f16_colmajor(colmajor(a), colmajor(b), M, N, K)
    want = (a @ b).astype(np.float64)
    assert np.array_equal(ref.reshape(N, M).T, want)
    assert np.array_equal(C, colmajor(want))


def test_gemm_empty_k_gives_zero(oracle_mod):
    ref, C = oracle.gemm_f16_colmajor(np.zeros(0, np.uint16), np.zeros(0, np.uint16), 3, 2, 0)
    assert np.all(ref == 0) and np.all(C == 0)


# --------------------------------------------------------------------------
# Linear-layer pins
# --------------------------------------------------------------------------

def bf16(vals):
    t = torch.tensor(np.asarray(vals, np.float64).reshape(-1), dtype=torch.float64).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def test_linear_matches_gemm_with_n1(oracle_mod):
    """y = x W^T with n = 1 equals the column-major GEMM with A = W (transposed in memory), B = x.

    Values are small integers, exact in both FP16 and BF16, so the two double sums agree exactly.
    """
    rng = np.random.default_rng(6)
    M, K = 50, 70
    w = rng.integers(-2, 3, (M, K)).astype(np.float64)
    x = rng.integers(-2, 3, (1, K)).astype(np.float64)
    yref, _ = oracle.linear_bf16(bf16(w), bf16(x), M, K, 1)
    cref, _ = oracle.gemm_f16_colmajor(colmajor(w), colmajor(x.T), M, 1, K)
    assert np.array_equal(yref[0], cref)


def test_linear_closed_forms(oracle_mod):
    """W row j = one-hot at column j mod K picks x[t, j mod K]; a ones row sums x."""
    M, K, n = 12, 8, 3
    rng = np.random.default_rng(8)
    x = rng.standard_normal((n, K))
    xb = bf16(x)
    xv = oracle.bf16_decode(xb).reshape(n, K)
    w = np.zeros((M, K))
    w[np.arange(M), np.arange(M) % K] = 1.0
    w[K:, :] = 0.0
    w[K, :] = 1.0
    yref, y = oracle.linear_bf16(bf16(w), xb, M, K, n)
    for t in range(n):
        for j in range(K):
            assert yref[t, j] == xv[t, j]
            assert y[t, j] == xb[t * K + j]
        assert yref[t, K] == sum(Fraction(float(v)) for v in xv[t])
        assert np.all(yref[t, K + 1:] == 0)


def test_linear_brute_force_tiny(oracle_mod):
    vals, bits = _positive_table(torch_bf16_values(), ALL)
    rng = np.random.default_rng(9)
    M, K, n = 5, 7, 3
    wb = bf16(rng.standard_normal((M, K)))
    xb = bf16(rng.standard_normal((n, K)))
    wv = oracle.bf16_decode(wb).reshape(M, K)   # decoder pinned above against torch
    xv = oracle.bf16_decode(xb).reshape(n, K)
    _, y = oracle.linear_bf16(wb, xb, M, K, n)
    for t in range(n):
        for j in range(M):
            s = sum((Fraction(float(xv[t, k])) * Fraction(float(wv[j, k])) for k in range(K)), Fraction(0))
            assert int(y[t, j]) == _nearest_even(s, vals, bits, 0x7F, Fraction(2) ** 128, 0x7F80)


def test_linear_subsets_agree(oracle_mod):
    rng = np.random.default_rng(10)
    M, K, n = 40, 24, 5
    wb = bf16(rng.standard_normal((M, K)) * 0.02)
    xb = bf16(rng.standard_normal((n, K)))
    ref, y = oracle.linear_bf16(wb, xb, M, K, n)
    js = [0, 17, 39]
    refj, yj = oracle.linear_bf16(wb, xb, M, K, n, js=js)
    assert np.array_equal(yj, y[:, js]) and np.array_equal(refj, ref[:, js])
    ts = [4, 0]
    reft, yt = oracle.linear_bf16_tokens(wb, xb, M, K, n, ts)
    assert np.array_equal(yt, y[ts, :]) and np.array_equal(reft, ref[ts, :])


def test_gemm_accumulates_beyond_float32(oracle_mod):
    """32768 + 2^-20 + 2^-20 - 32768 = 2^-19 exactly; a float32 accumulator would return 0."""
    a = [[128.0, 2.0 ** -10, 2.0 ** -10, -128.0]]
    b = [[256.0], [2.0 ** -10], [2.0 ** -10], [256.0]]
    ref, C = oracle.gemm_f16_colmajor(colmajor(a), colmajor(b), 1, 1, 4)
    assert ref[0] == 2.0 ** -19
    assert C[0] == f16([2.0 ** -19])[0]


def test_linear_accumulates_beyond_float32(oracle_mod):
    w = [[128.0, 2.0 ** -10, 2.0 ** -10, -128.0]]
    x = [[256.0, 2.0 ** -10, 2.0 ** -10, 256.0]]
    ref, y = oracle.linear_bf16(bf16(w), bf16(x), 1, 4, 1)
    assert ref[0, 0] == 2.0 ** -19
    assert y[0, 0] == bf16([2.0 ** -19])[0]
