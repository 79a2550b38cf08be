"""GPU parity of gemm_fp8 (E4M3 / E5M2 inputs, FP32 accumulation, FP32 or BF16
output) against the oracle's FP8 GEMM, called through the C ABI.

Integer-valued inputs (entries in {-2..2}) with an exact alpha: every partial
sum is a small integer, so the output must equal the oracle bit for bit.
Random inputs: the same accumulation bound as the 16-bit GEMM,
|C - C_exact| <= |alpha| * 4e-3 * sqrt(K/256) * max|a| * max|b| + 1/2 ulp of
the output format, and a relative Frobenius error <= 1e-3 against the
correctly rounded exact result.  Operand padding holds the FP8 NaN code
(0x7F in both formats): reading it would show.  C starts as NaN and its
padding must be untouched afterwards.
"""
import numpy as np
import pytest

import oracle
from bf16_gemm_skinny_gb300 import _native as bsk
from bf16_gemm_skinny_gb300 import build as bsk_build
from bf16_gemm_skinny_gb300 import inputs

pytestmark = pytest.mark.gpu

NAN8 = 0x7F
NAN32 = 0x7FC00000
NAN16 = 0x7FC0
GUARD = 64
FMT = {"e4m3": 0, "e5m2": 1}
OUT = {"f32": 0, "bf16": 1}


@pytest.fixture(scope="module", autouse=True)
def lib():
    import torch

    bsk_build.build()
    oracle.build()
    torch.cuda.init()
    yield bsk.load()
    for k in bsk.OPTIONS:
        bsk.set_option(k, 0)


_CACHE = {}


def operands(M, N, K, dist, fmt):
    key = (M, N, K, dist, fmt)
    if key not in _CACHE:
        seeds = (11, 12) if dist == "int2" else (1, 2)
        A, B = inputs.fp8_operands(M, N, K, dist, fmt, *seeds)
        _CACHE[key] = (A.reshape(M, K), B.reshape(N, K))
    return _CACHE[key]


def padded(rows, ld):
    R, K = rows.shape
    buf = np.full((R, ld), NAN8, np.uint8)
    buf[:, :K] = rows
    return buf.reshape(-1)


def run(A2, B2, fmt, out, alpha=1.0, pad_a=0, pad_b=0, pad_c=0, offset=0, enqueue=False):
    """A2: M x K codes, B2: N x K codes.  Returns (C as M x N output bits, A flat, lda, B flat, ldb)."""
    import torch

    M, K = A2.shape
    N = B2.shape[0]
    lda, ldb, ldc = max(K, 1) + pad_a, max(K, 1) + pad_b, M + pad_c
    Af, Bf = padded(A2, lda), padded(B2, ldb)

    def dev(bits):
        t = torch.from_numpy(np.concatenate([np.zeros(offset, np.uint8), bits])).to("cuda")
        return t[offset:]

    Ad, Bd = dev(Af), dev(Bf)
    if out == "f32":
        buf = torch.full((N * ldc + GUARD,), NAN32, dtype=torch.int32, device="cuda")
        canary = 0x5A5A5A5A
    else:
        buf = torch.full((N * ldc + GUARD,), NAN16, dtype=torch.int16, device="cuda")
        canary = 0x5A5A
    buf[N * ldc:] = canary
    C = buf[:N * ldc]
    call = bsk.gemm_fp8_enqueue if enqueue else bsk.gemm_fp8
    call(FMT[fmt], Ad, lda, Bd, ldb, C, ldc, OUT[out], M, N, K, alpha)
    if enqueue:
        bsk.stream_check()
    torch.cuda.synchronize()
    host = buf.cpu().numpy().view(np.uint32 if out == "f32" else np.uint16)
    assert np.all(host[N * ldc:] == canary), "guard words after C were written"
    assert np.array_equal(Ad.cpu().numpy(), Af) and np.array_equal(Bd.cpu().numpy(), Bf), "an input was modified"
    full = host[:N * ldc].reshape(N, ldc)
    assert np.all(full[:, M:] == (NAN32 if out == "f32" else NAN16)), "C's padding was written"
    return full[:, :M].T, Af, lda, Bf, ldb


def want(Af, lda, Bf, ldb, M, N, K, fmt, out, alpha=1.0, rows=None, cols=None):
    ref, bits = oracle.gemm_fp8(Af, Bf, M, N, K, lda, ldb, fmt, alpha, out, rows=rows, cols=cols)
    nr = M if rows is None else len(rows)
    nc = N if cols is None else len(cols)
    return ref.reshape(nc, nr).T, bits.reshape(nc, nr).T


def decode_out(bits, out):
    if out == "f32":
        return np.asarray(bits, np.uint32).view(np.float32).astype(np.float64)
    return oracle.bf16_decode(np.asarray(bits, np.uint16).reshape(-1)).reshape(np.shape(bits))


def ulp_out(x, out):
    frac, emin = (23, -126) if out == "f32" else (7, -126)
    a = np.abs(x)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.exp2(np.maximum(e, emin) - frac)


def check(got_bits, ref, out, K, amax, bmax, alpha, label):
    got = decode_out(got_bits, out).reshape(-1)
    ref = np.asarray(ref, np.float64).reshape(-1)
    assert np.all(np.isfinite(got)), f"{label}: non-finite outputs"
    rn = ref.astype(np.float32).astype(np.float64) if out == "f32" else oracle.bf16_decode(oracle.bf16_encode(ref))
    denom = np.linalg.norm(rn)
    rel = float(np.linalg.norm(got - rn) / denom) if denom > 0 else float(np.linalg.norm(got - rn))
    assert rel <= 1e-3, f"{label}: relative Frobenius error {rel:.3e}"
    bound = abs(alpha) * 4e-3 * np.sqrt(K / 256.0) * amax * bmax + 0.5 * ulp_out(np.maximum(abs(got), abs(ref)), out)
    err = np.abs(got - ref)
    worst = int(np.argmax(err - bound))
    assert np.all(err <= bound), f"{label}: |out - exact| {err[worst]:.4g} > {bound[worst]:.4g} at {worst}"
    return rel


def absmax(codes, fmt):
    return float(np.max(np.abs(oracle.fp8_decode(codes.reshape(-1), fmt)))) if codes.size else 0.0


SHAPES = [(1, 1, 1), (17, 33, 19), (128, 128, 128), (129, 257, 129), (300, 517, 200), (1000, 777, 1030),
          (64, 8, 256), (256, 300, 64)]


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("out", ["f32", "bf16"])
@pytest.mark.parametrize("M,N,K", SHAPES)
def test_integer_inputs_bit_exact(fmt, out, M, N, K):
    A2, B2 = operands(M, N, K, "int2", fmt)
    alpha = 0.5 if out == "f32" else -2.0
    got, Af, lda, Bf, ldb = run(A2, B2, fmt, out, alpha, pad_a=16, pad_b=3, pad_c=5)
    _, bits = want(Af, lda, Bf, ldb, M, N, K, fmt, out, alpha)
    assert np.array_equal(got, bits), f"{int((got != bits).sum())} of {got.size} entries differ"


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_random_inputs_within_tolerance(fmt, out):
    M, N, K = 1000, 777, 1030
    A2, B2 = operands(M, N, K, "normal1", fmt)
    alpha = 0.03125
    got, Af, lda, Bf, ldb = run(A2, B2, fmt, out, alpha)
    ref, _ = want(Af, lda, Bf, ldb, M, N, K, fmt, out, alpha)
    check(got, ref, out, K, absmax(A2, fmt), absmax(B2, fmt), alpha, f"{fmt}->{out}")


@pytest.mark.parametrize("kernel,block_n,group_m,skc", [
    (2, 256, 2, 0), (2, 256, 5, 0), (1, 256, 3, 0), (1, 128, 1, 0), (1, 64, 7, 0), (1, 32, 2, 0),
    (1, 32, 2, 4), (1, 256, 1, 16)])
def test_result_independent_of_tile_config(kernel, block_n, group_m, skc):
    M, N, K = 1000, 777, 1030
    A2, B2 = operands(M, N, K, "int2", "e4m3")
    opts = {"gemm_kernel": kernel, "block_n": block_n, "group_m": group_m, "split_k": skc}
    for k, v in opts.items():
        bsk.set_option(k, v)
    try:
        got, Af, lda, Bf, ldb = run(A2, B2, "e4m3", "bf16")
    finally:
        for k in opts:
            bsk.set_option(k, 0)
    _, bits = want(Af, lda, Bf, ldb, M, N, K, "e4m3", "bf16")
    assert np.array_equal(got, bits)


@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_split_k_scale_and_outputs(out):
    """Split-K over clusters (forced) applies alpha once, after the partials are
    summed: integer codes with alpha 1 give the oracle's bits; random codes
    with alpha 1/32 stay within tolerance."""
    M, N, K = 700, 300, 2304
    opts = {"gemm_kernel": 1, "block_n": 64, "split_k": 8}
    for k, v in opts.items():
        bsk.set_option(k, v)
    try:
        A2, B2 = operands(M, N, K, "int2", "e4m3")
        got, Af, lda, Bf, ldb = run(A2, B2, "e4m3", out)
        _, bits = want(Af, lda, Bf, ldb, M, N, K, "e4m3", out)
        assert np.array_equal(got, bits)
        A2, B2 = operands(M, N, K, "normal1", "e4m3")
        got, Af, lda, Bf, ldb = run(A2, B2, "e4m3", out, 0.03125)
    finally:
        for k in opts:
            bsk.set_option(k, 0)
    ref, _ = want(Af, lda, Bf, ldb, M, N, K, "e4m3", out, 0.03125)
    check(got, ref, out, K, absmax(A2, "e4m3"), absmax(B2, "e4m3"), 0.03125, f"split-K e4m3->{out}")


@pytest.mark.parametrize("N", [1, 8, 16, 33, 64, 100, 128, 129])
def test_skinny_n(N):
    """Decode-like shapes: many weight rows, few tokens (narrow tiles)."""
    M, K = 1000, 640
    A2, B2 = operands(M, N, K, "int2", "e5m2")
    got, Af, lda, Bf, ldb = run(A2, B2, "e5m2", "f32")
    _, bits = want(Af, lda, Bf, ldb, M, N, K, "e5m2", "f32")
    assert np.array_equal(got, bits)


@pytest.mark.parametrize("block_m", [8, 56, 120])
@pytest.mark.parametrize("N", [8, 100])
def test_skinny_tile_heights(block_m, N):
    """Narrow tiles of block_m weight rows (the balanced schedule's heights,
    forced): bit-exact on integer inputs, and C's padding rows stay untouched."""
    M, K = 1000, 640
    A2, B2 = operands(M, N, K, "int2", "e4m3")
    bsk.set_option("block_m", block_m)
    try:
        got, Af, lda, Bf, ldb = run(A2, B2, "e4m3", "bf16", pad_a=16, pad_c=5)
    finally:
        bsk.set_option("block_m", 0)
    _, bits = want(Af, lda, Bf, ldb, M, N, K, "e4m3", "bf16")
    assert np.array_equal(got, bits)


@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_unaligned_pointers_and_strides(out):
    """Bases one byte off and leading dimensions not multiples of 16: both operands are packed."""
    M, N, K = 333, 129, 200
    A2, B2 = operands(M, N, K, "int2", "e4m3")
    got, Af, lda, Bf, ldb = run(A2, B2, "e4m3", out, 1.0, pad_a=1, pad_b=5, pad_c=1, offset=1)
    _, bits = want(Af, lda, Bf, ldb, M, N, K, "e4m3", out)
    assert np.array_equal(got, bits)


def test_force_pack_agrees():
    M, N, K = 512, 384, 512
    A2, B2 = operands(M, N, K, "normal1", "e4m3")
    base, *_ = run(A2, B2, "e4m3", "f32")
    bsk.set_option("force_pack", 1)
    try:
        other, *_ = run(A2, B2, "e4m3", "f32")
    finally:
        bsk.set_option("force_pack", 0)
    assert np.array_equal(base, other)


@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_k_zero_writes_zeros(out):
    got, *_ = run(np.zeros((37, 0), np.uint8), np.zeros((19, 0), np.uint8), "e4m3", out, 3.0, pad_c=3)
    assert np.all(got == 0)


def test_single_rounding_happens_after_fp32_accumulation():
    """1*1 + 2^-4*2^-4 + 2^-15*2^-15 (E5M2): the FP32 accumulator holds 1 + 2^-8
    (2^-30 is below its spacing), so the BF16 output is the tie 1 + 2^-8 -> 1.0
    (0x3F80), one ulp from the exact sum's rounding (0x3F81): the expected
    difference between FP32 accumulation and the exact oracle."""
    A2 = np.array([[0x3C, 0x2C, 0x02]], np.uint8)
    got, Af, lda, Bf, ldb = run(A2, A2.copy(), "e5m2", "bf16")
    assert got[0, 0] == 0x3F80
    _, bits = want(Af, lda, Bf, ldb, 1, 1, 3, "e5m2", "bf16")
    assert bits[0, 0] == 0x3F81
    got32, *_ = run(A2, A2.copy(), "e5m2", "f32")
    assert got32[0, 0] == 0x3F808000


def test_deterministic_and_enqueue_matches_blocking():
    M, N, K = 512, 384, 640
    A2, B2 = operands(M, N, K, "normal1", "e5m2")
    first, *_ = run(A2, B2, "e5m2", "bf16", 0.5)
    again, *_ = run(A2, B2, "e5m2", "bf16", 0.5, enqueue=True)
    assert np.array_equal(first, again)


@pytest.mark.parametrize("fmt,out,M,N,K", [
    ("e4m3", "bf16", 8192, 8192, 8192),    # square, CTA pairs
    ("e4m3", "f32", 34816, 16, 5120),      # FP8 weights x 16 tokens (skinny)
    ("e5m2", "bf16", 4096, 4096, 4096),
])
def test_large_sampled(fmt, out, M, N, K):
    A2, B2 = operands(M, N, K, "normal1", fmt)
    alpha = 1.0 / 64
    got, Af, lda, Bf, ldb = run(A2, B2, fmt, out, alpha)
    rows = [0, 127, 128, 1000, M - 1]
    cols = sorted({0, min(255, N - 1), min(256, N - 1), N // 2, N - 1})
    ref_r, _ = want(Af, lda, Bf, ldb, M, N, K, fmt, out, alpha, rows=rows)
    ref_c, _ = want(Af, lda, Bf, ldb, M, N, K, fmt, out, alpha, cols=cols)
    amax, bmax = absmax(A2, fmt), absmax(B2, fmt)
    check(got[rows, :], ref_r, out, K, amax, bmax, alpha, "sampled rows")
    check(got[:, cols], ref_c, out, K, amax, bmax, alpha, "sampled columns")


@pytest.mark.parametrize("M,N,K,stream_k", [(34816, 16, 5120, 0), (34816, 16, 5120, 1), (1000, 40, 4096, 2),
                                            (512, 100, 8192, 2)])
def test_stream_k_schedule(M, N, K, stream_k):
    """FP8 skinny shapes take stream-K by default (272 row tiles on the SMs);
    forced on or off, integer inputs give the oracle's bits."""
    A2, B2 = operands(M, N, K, "int2", "e4m3")
    bsk.set_option("stream_k", stream_k)
    try:
        got, Af, lda, Bf, ldb = run(A2, B2, "e4m3", "f32")
    finally:
        bsk.set_option("stream_k", 0)
    cols = sorted({0, N // 2, N - 1})
    _, bits = want(Af, lda, Bf, ldb, M, N, K, "e4m3", "f32", cols=cols)
    assert np.array_equal(got[:, cols], bits)


def test_stream_k_on_cta_pairs():
    """FP8 on CTA pairs with stream-K forced: integer inputs, the oracle's bits."""
    M, N, K = 1000, 777, 4096
    A2, B2 = operands(M, N, K, "int2", "e4m3")
    bsk.set_option("stream_k", 2)
    try:
        got, Af, lda, Bf, ldb = run(A2, B2, "e4m3", "bf16")
    finally:
        bsk.set_option("stream_k", 0)
    _, bits = want(Af, lda, Bf, ldb, M, N, K, "e4m3", "bf16")
    assert np.array_equal(got, bits)


@pytest.mark.parametrize("offset", range(16))
def test_pack_every_byte_offset(offset):
    """FP8 operands at every byte offset inside a 16-byte chunk, with odd leading
    dimensions (every line starts at another offset): the pack's aligned loads
    and byte shifts, bit for bit."""
    M, N, K = 200, 72, 131
    A2, B2 = operands(M, N, K, "int2", "e4m3")
    got, Af, lda, Bf, ldb = run(A2, B2, "e4m3", "f32", pad_a=3, pad_b=5, offset=offset)
    _, bits = want(Af, lda, Bf, ldb, M, N, K, "e4m3", "f32")
    assert np.array_equal(got, bits)


def _random_cases(count, seed):
    """Seeded shapes (M, N, K log-uniform in 1..3000, at most 2e8 multiply-adds),
    formats, output types and paddings."""
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < count:
        M, N, K = (int(np.exp(rng.uniform(0, np.log(3000)))) for _ in range(3))
        if M * N * K > 2e8:
            continue
        fmt = ("e4m3", "e5m2")[int(rng.integers(0, 2))]
        o = ("f32", "bf16")[int(rng.integers(0, 2))]
        pads = tuple(int(v) for v in rng.choice([0, 0, 1, 16, 5], 3))
        out.append((M, N, K, fmt, o, pads))
    return out


@pytest.mark.parametrize("M,N,K,fmt,out,pads", _random_cases(30, 88))
def test_random_shapes_default_plan(M, N, K, fmt, out, pads):
    """Random shapes, formats, output types and leading dimensions through the
    default plan (the pack for unaligned ones): integer codes give the oracle's
    bits, and no padding of C is written."""
    A, B = inputs.fp8_operands(M, N, K, "int2", fmt, M + 3, N + 9)
    A2, B2 = A.reshape(M, K), B.reshape(N, K)
    got, Af, lda, Bf, ldb = run(A2, B2, fmt, out, pad_a=pads[0], pad_b=pads[1], pad_c=pads[2])
    _, bits = want(Af, lda, Bf, ldb, M, N, K, fmt, out)
    assert np.array_equal(got, bits), f"{int((got != bits).sum())} of {got.size} entries differ"
