"""GPU parity of gemm_f16 (transposed operands, row-major storage, any leading
dimension, optional fused bias) against the oracle's general GEMM, called
through the C ABI.

Every stored operand has padding between its lines filled with FP16 NaN (a
read of padding would show in the result); C starts as NaN and its padding
must still hold NaN afterwards, with the guard words after it untouched.
Integer inputs (entries in {-2..2}, integer bias): bit-identical to the
oracle.  Random inputs: the tolerance in helpers.check_tolerance.
"""
import itertools

import numpy as np
import pytest

import oracle
from bf16_gemm_skinny_gb300 import _native as bsk
from bf16_gemm_skinny_gb300 import build as bsk_build
from bf16_gemm_skinny_gb300 import inputs
from helpers import CANARY, FP16_NAN, absmax_f16, check_tolerance, from_dev, poisoned, to_dev

pytestmark = pytest.mark.gpu

FORMS = list(itertools.product([0, 1], repeat=3))   # (order, transa, transb)


@pytest.fixture(scope="module", autouse=True)
def lib():
    import torch

    bsk_build.build()
    oracle.build()
    torch.cuda.init()
    yield bsk.load()
    for k in bsk.OPTIONS:
        bsk.set_option(k, 0)


def enc(x):
    return oracle.f16_encode(np.asarray(x, np.float64).reshape(-1))


def store(mat, order, ld):
    """Flat storage of the 2-D uint16 matrix `mat` in `order` with leading
    dimension `ld`; padding holds NaN."""
    R, C = mat.shape
    if order:
        buf = np.full((R, ld), FP16_NAN, np.uint16)
        buf[:, :C] = mat
    else:
        buf = np.full((C, ld), FP16_NAN, np.uint16)
        buf[:, :R] = mat.T
    return buf.reshape(-1)


def operands(M, N, K, dist, seeds=None):
    sa, sb = seeds or ((11, 12) if dist == "int2" else (1, 2))
    A, B = inputs.gemm_operands(M, N, K, dist, sa, sb)
    return A.reshape(K, M).T, B.reshape(N, K).T     # logical M x K and K x N


def layout(order, transa, transb, A2, B2, pad_a, pad_b):
    sa = A2.T if transa else A2
    sb = B2.T if transb else B2
    lda = max(1, sa.shape[1] if order else sa.shape[0]) + pad_a
    ldb = max(1, sb.shape[1] if order else sb.shape[0]) + pad_b
    return store(sa, order, lda), lda, store(sb, order, ldb), ldb


def run(order, transa, transb, A2, B2, pad_a=0, pad_b=0, pad_c=0, bias=None, mode=0, offset=0, enqueue=False):
    """Runs gemm_f16; returns (logical M x N result bits, flat A, lda, flat B, ldb)."""
    import torch

    M, K = A2.shape
    N = B2.shape[1]
    Af, lda, Bf, ldb = layout(order, transa, transb, A2, B2, pad_a, pad_b)
    ldc = (N if order else M) + pad_c
    lines = M if order else N
    n_c = lines * ldc

    def dev(bits):
        return to_dev(np.concatenate([np.zeros(offset, np.uint16), bits]))[offset:]

    Ad, Bd = dev(Af), dev(Bf)
    biasd = None if bias is None else dev(bias)
    buf, _ = poisoned(n_c + offset, FP16_NAN)
    C = buf[offset:offset + n_c]
    call = bsk.gemm_f16_enqueue if enqueue else bsk.gemm_f16
    call(order, transa, transb, Ad, lda, Bd, ldb, C, ldc, M, N, K, biasd, mode)
    if enqueue:
        bsk.stream_check()
    torch.cuda.synchronize()
    assert np.all(from_dev(buf[offset + n_c:]) == CANARY), "guard words after C were written"
    assert np.array_equal(from_dev(Ad), Af) and np.array_equal(from_dev(Bd), Bf), "an input was modified"
    full = from_dev(C).reshape(lines, ldc)
    assert np.all(full[:, (N if order else M):] == FP16_NAN), "C's padding was written"
    got = full[:, :N] if order else full[:, :M].T
    return got, Af, lda, Bf, ldb


def want(order, transa, transb, Af, lda, Bf, ldb, M, N, K, bias=None, mode=0, rows=None, cols=None):
    ref, out = oracle.gemm_f16_general(Af, Bf, M, N, K, lda, ldb, transa, transb, order, bias=bias,
                                       bias_mode=mode, rows=rows, cols=cols)
    nr = M if rows is None else len(rows)
    nc = N if cols is None else len(cols)
    return ref.reshape(nc, nr).T, out.reshape(nc, nr).T


@pytest.mark.parametrize("order,transa,transb", FORMS)
@pytest.mark.parametrize("M,N,K", [(129, 257, 65), (300, 517, 200), (64, 20, 96)])
def test_integer_inputs_bit_exact(order, transa, transb, M, N, K):
    A2, B2 = operands(M, N, K, "int2")
    got, Af, lda, Bf, ldb = run(order, transa, transb, A2, B2, pad_a=3, pad_b=8, pad_c=5)
    _, out = want(order, transa, transb, Af, lda, Bf, ldb, M, N, K)
    assert np.array_equal(got, out), f"{int((got != out).sum())} of {got.size} entries differ"


@pytest.mark.parametrize("order,transa,transb", FORMS)
def test_random_inputs_within_tolerance(order, transa, transb):
    M, N, K = 1000, 777, 1030
    A2, B2 = operands(M, N, K, "normal0.5")
    got, Af, lda, Bf, ldb = run(order, transa, transb, A2, B2, pad_a=8, pad_b=0, pad_c=16)
    ref, _ = want(order, transa, transb, Af, lda, Bf, ldb, M, N, K)
    check_tolerance(got.T.reshape(-1), ref.T.reshape(-1), "f16", K, absmax_f16(A2.reshape(-1)),
                    absmax_f16(B2.reshape(-1)), f"order={order} ta={transa} tb={transb}")


@pytest.mark.parametrize("order,transa,transb,mode", [
    (0, 0, 0, 1), (0, 0, 1, 2), (0, 1, 0, 2), (0, 1, 1, 1), (1, 0, 1, 2), (1, 0, 0, 1), (1, 1, 0, 2), (1, 1, 1, 1)])
@pytest.mark.parametrize("dist", ["int2", "normal0.5"])
def test_fused_bias(order, transa, transb, mode, dist):
    M, N, K = 333, 290, 136
    A2, B2 = operands(M, N, K, dist)
    rng = np.random.default_rng(7)
    vals = rng.integers(-40, 41, max(M, N)) if dist == "int2" else rng.normal(0, 2.0, max(M, N))
    bias = enc(vals)[:M if mode == 1 else N]
    got, Af, lda, Bf, ldb = run(order, transa, transb, A2, B2, pad_a=1, pad_b=2, pad_c=3, bias=bias, mode=mode)
    ref, out = want(order, transa, transb, Af, lda, Bf, ldb, M, N, K, bias=bias, mode=mode)
    if dist == "int2":
        assert np.array_equal(got, out)
    else:
        check_tolerance(got.T.reshape(-1), ref.T.reshape(-1), "f16", K, absmax_f16(A2.reshape(-1)),
                        absmax_f16(B2.reshape(-1)), "bias")


def test_bias_joins_the_single_rounding():
    """Exact sum 2049 (a tie in FP16) plus a bias of 0.5 rounds once to 2050."""
    A2 = enc([2048.0, 1.0]).reshape(1, 2)
    B2 = enc([1.0, 1.0]).reshape(2, 1)
    got, *_ = run(0, 0, 0, A2, B2, bias=enc([0.5]), mode=1)
    assert oracle.f16_decode(got.reshape(-1))[0] == 2050.0
    got, *_ = run(0, 0, 0, A2, B2)
    assert oracle.f16_decode(got.reshape(-1))[0] == 2048.0


@pytest.mark.parametrize("transb", [0, 1])
@pytest.mark.parametrize("kernel,block_n,group_m", [
    (2, 256, 2), (2, 256, 5), (1, 256, 3), (1, 128, 1), (1, 64, 7), (1, 32, 2)])
def test_result_independent_of_tile_config(transb, kernel, block_n, group_m):
    """CTA-pair and single-CTA kernels, every tile width (a transposed B is
    staged 64 columns at a time: block_n 32 runs as 64), several GROUP_M."""
    M, N, K = 1000, 777, 1030
    A2, B2 = operands(M, N, K, "int2")
    bsk.set_option("gemm_kernel", kernel)
    bsk.set_option("block_n", block_n)
    bsk.set_option("group_m", group_m)
    try:
        got, Af, lda, Bf, ldb = run(0, 1, transb, A2, B2, pad_a=8, pad_b=8)
    finally:
        for k in ("gemm_kernel", "block_n", "group_m"):
            bsk.set_option(k, 0)
    _, out = want(0, 1, transb, Af, lda, Bf, ldb, M, N, K)
    assert np.array_equal(got, out)


@pytest.mark.parametrize("N", [1, 8, 31, 64, 65, 128, 129, 200])
def test_skinny_n_with_transposed_b(N):
    """Skinny N takes the narrow tiles; with a transposed B the tile is at least 64 wide."""
    M, K = 777, 520
    A2, B2 = operands(M, N, K, "int2")
    got, Af, lda, Bf, ldb = run(0, 0, 1, A2, B2, pad_b=8)
    _, out = want(0, 0, 1, Af, lda, Bf, ldb, M, N, K)
    assert np.array_equal(got, out)


@pytest.mark.parametrize("order,transa,transb", [(0, 0, 1), (0, 1, 1), (1, 0, 1), (1, 1, 0)])
def test_unaligned_pointers_and_strides(order, transa, transb):
    """Bases one element off and odd leading dimensions: both operands are packed."""
    M, N, K = 333, 129, 70
    A2, B2 = operands(M, N, K, "int2")
    got, Af, lda, Bf, ldb = run(order, transa, transb, A2, B2, pad_a=1, pad_b=3, pad_c=1, offset=1)
    _, out = want(order, transa, transb, Af, lda, Bf, ldb, M, N, K)
    assert np.array_equal(got, out)


def test_force_pack_and_direct_store_agree():
    M, N, K = 1024, 640, 1040
    A2, B2 = operands(M, N, K, "normal0.5")
    base, *_ = run(0, 1, 1, A2, B2)
    for option in ("force_pack", "force_direct_store"):
        bsk.set_option(option, 1)
        try:
            other, *_ = run(0, 1, 1, A2, B2)
        finally:
            bsk.set_option(option, 0)
        assert np.array_equal(base, other), option


@pytest.mark.parametrize("mode", [0, 1, 2])
def test_k_zero_writes_the_bias(mode):
    M, N = 37, 19
    bias = enc(np.arange(max(M, N)) * 0.25 - 3.0)[:M if mode == 1 else N] if mode else None
    A2 = np.zeros((M, 0), np.uint16)
    B2 = np.zeros((0, N), np.uint16)
    got, *_ = run(0, 0, 0, A2, B2, pad_c=4, bias=bias, mode=mode)
    exp = np.zeros((M, N), np.uint16)
    if mode == 1:
        exp[:] = bias[:, None]
    elif mode == 2:
        exp[:] = bias[None, :]
    assert np.array_equal(got, exp)


def test_column_major_nn_matches_gemm_f16_colmajor():
    import torch

    M, N, K = 512, 384, 320
    A2, B2 = operands(M, N, K, "normal0.5")
    got, Af, lda, Bf, ldb = run(0, 0, 0, A2, B2)
    C = torch.empty(M * N, dtype=torch.int16, device="cuda")
    bsk.gemm_f16_colmajor(to_dev(Af), to_dev(Bf), C, M, N, K)
    assert np.array_equal(from_dev(C).reshape(N, M).T, got)


def test_enqueue_variant_matches_blocking():
    M, N, K = 512, 384, 320
    A2, B2 = operands(M, N, K, "normal0.5")
    bias = enc(np.linspace(-1, 1, N))
    a, *_ = run(1, 0, 1, A2, B2, bias=bias, mode=2, enqueue=True)
    b, *_ = run(1, 0, 1, A2, B2, bias=bias, mode=2)
    assert np.array_equal(a, b)


@pytest.mark.parametrize("order,transa,transb,M,N,K", [
    (1, 0, 1, 2048, 8192, 4096),   # row-major linear layer Y = X W^T + b (tokens x features)
    (0, 0, 1, 4096, 4096, 4096),   # column-major NT: the MN-major B on CTA pairs
    (0, 1, 0, 4096, 4096, 4096),   # column-major TN
])
def test_large_sampled(order, transa, transb, M, N, K):
    A2, B2 = operands(M, N, K, "uniform")
    bias = enc(np.random.default_rng(3).uniform(-1, 1, N))
    got, Af, lda, Bf, ldb = run(order, transa, transb, A2, B2, bias=bias, mode=2)
    rows = [0, 127, 128, 1000, M - 1]
    cols = [0, 255, 256, 3001, N - 1]
    ref_r, _ = want(order, transa, transb, Af, lda, Bf, ldb, M, N, K, bias=bias, mode=2, rows=rows)
    ref_c, _ = want(order, transa, transb, Af, lda, Bf, ldb, M, N, K, bias=bias, mode=2, cols=cols)
    amax, bmax = absmax_f16(A2.reshape(-1)), absmax_f16(B2.reshape(-1))
    check_tolerance(got[rows, :].reshape(-1), ref_r.reshape(-1), "f16", K, amax, bmax, "sampled rows")
    check_tolerance(got[:, cols].reshape(-1), ref_c.reshape(-1), "f16", K, amax, bmax, "sampled columns")


@pytest.mark.parametrize("M,pad_c", [(333, 3), (1001, 7), (1000, 8)])
def test_ragged_m_with_aligned_ldc_leaves_padding_alone(M, pad_c):
    """ldc a multiple of 8 with M not: the rows between M and ldc stay untouched."""
    N, K = 300, 64
    A2, B2 = operands(M, N, K, "int2")
    got, Af, lda, Bf, ldb = run(0, 0, 0, A2, B2, pad_c=pad_c)   # run() checks the padding
    _, out = want(0, 0, 0, Af, lda, Bf, ldb, M, N, K)
    assert np.array_equal(got, out)


@pytest.mark.parametrize("sched", [{"stream_k": 2}, {"stream_k": 2, "gemm_kernel": 1}, {"tile_sched": 2},
                                   {"split_k": 8, "gemm_kernel": 1}, {"split_k": 4, "gemm_kernel": 1, "block_n": 64}])
@pytest.mark.parametrize("order,transa,transb,mode", [
    (0, 0, 0, 1), (0, 1, 1, 2), (1, 0, 1, 2), (1, 1, 0, 1), (0, 0, 1, 0)])
def test_schedules_with_layouts_and_bias(sched, order, transa, transb, mode):
    """Stream-K (on CTA pairs and on single CTAs) and the dynamic tile order with
    every storage form and a per-row or per-column bias: the owner of a split
    tile adds the partials before the bias and the single rounding, and a
    dynamically ordered tile keeps its own bias slice.  Integer inputs and bias:
    the oracle's bits."""
    M, N, K = 700, 600, 2100
    A2, B2 = operands(M, N, K, "int2")
    bias = None
    if mode:
        vals = np.random.default_rng(9).integers(-40, 41, max(M, N))
        bias = enc(vals)[:M if mode == 1 else N]
    for k, v in sched.items():
        bsk.set_option(k, v)
    try:
        got, Af, lda, Bf, ldb = run(order, transa, transb, A2, B2, pad_a=2, pad_b=1, pad_c=3, bias=bias, mode=mode)
    finally:
        for k in sched:
            bsk.set_option(k, 0)
    _, out = want(order, transa, transb, Af, lda, Bf, ldb, M, N, K, bias=bias, mode=mode)
    assert np.array_equal(got, out), f"{int((got != out).sum())} of {got.size} entries differ"


def _random_cases(count, seed):
    """Seeded shapes, storage forms, paddings and bias modes, M, N, K log-uniform
    in 1..3000 with at most 2e8 multiply-adds."""
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < count:
        M, N, K = (int(np.exp(rng.uniform(0, np.log(3000)))) for _ in range(3))
        if M * N * K > 2e8:
            continue
        order, transa, transb = (int(v) for v in rng.integers(0, 2, 3))
        pads = tuple(int(v) for v in rng.choice([0, 0, 1, 3, 8], 3))
        out.append((M, N, K, order, transa, transb, pads, int(rng.integers(0, 3))))
    return out


@pytest.mark.parametrize("M,N,K,order,transa,transb,pads,mode", _random_cases(40, 77))
def test_random_layouts_default_plan(M, N, K, order, transa, transb, pads, mode):
    """Random shapes in every storage form, with padded leading dimensions and
    each bias mode, through the default plan: integer inputs and bias give the
    oracle's bits, and no padding of C is written."""
    A2, B2 = operands(M, N, K, "int2", seeds=(M + 5, N + 7))
    bias = None
    if mode:
        vals = np.random.default_rng(K).integers(-40, 41, max(M, N))
        bias = enc(vals)[:M if mode == 1 else N]
    got, Af, lda, Bf, ldb = run(order, transa, transb, A2, B2, pad_a=pads[0], pad_b=pads[1], pad_c=pads[2],
                                bias=bias, mode=mode)
    _, out = want(order, transa, transb, Af, lda, Bf, ldb, M, N, K, bias=bias, mode=mode)
    assert np.array_equal(got, out), f"{int((got != out).sum())} of {got.size} entries differ"


@pytest.mark.parametrize("order,transa,transb,M,N,K,sms,mode", [
    (0, 0, 0, 1000, 777, 1030, 8, 0),     # MN-major A; four pairs, several rounds of 512 x 256 tiles
    (0, 0, 0, 600, 517, 640, 8, 0),       # the second tile row's second block lies wholly past M
    (0, 1, 0, 1536, 512, 640, 6, 1),      # K-major A, per-row bias, three pairs
    (1, 0, 1, 700, 1100, 1024, 8, 2),     # the row-major linear layer X W^T + b (K-major after the swap)
    (0, 0, 0, 2304, 2560, 1024, 0, 0),
])
def test_pair_512_row_tiles(order, transa, transb, M, N, K, sms, mode):
    """CTA pairs on 512 x 256 tiles (BSK_OPT_PAIR_M = 2: two 256-row blocks per
    pair tile sharing each B slice; grids capped where needed so that the
    planner keeps CTA pairs): integer inputs, with an integer bias where
    given, match the oracle bit for bit; with every k loop ascending, random
    inputs give the bits of the 256 x 256 tiles (each output sums the same
    products in the same order)."""
    A2, B2 = operands(M, N, K, "int2")
    bias = None
    if mode:
        vals = np.random.default_rng(5).integers(-40, 41, max(M, N))
        bias = enc(vals[:M] if mode == 1 else vals[:N])
    bsk.set_option("pair_m", 2)
    bsk.set_option("num_sms", sms)
    try:
        got, Af, lda, Bf, ldb = run(order, transa, transb, A2, B2, pad_a=8, pad_b=16, pad_c=8, bias=bias, mode=mode)
    finally:
        bsk.set_option("pair_m", 0)
        bsk.set_option("num_sms", 0)
    rows = np.unique(np.r_[np.arange(0, M, 37), M - 1]) if M * N > 1 << 20 else None
    cols = np.unique(np.r_[np.arange(0, N, 41), N - 1]) if M * N > 1 << 20 else None
    _, out = want(order, transa, transb, Af, lda, Bf, ldb, M, N, K, bias=bias, mode=mode, rows=rows, cols=cols)
    sub = got if rows is None else got[np.ix_(rows, cols)]
    assert np.array_equal(sub, out), f"{int((sub != out).sum())} of {sub.size} entries differ"
    Ar, Br = operands(M, N, K, "normal0.5")
    outs = {}
    for pm in (1, 2):
        bsk.set_option("pair_m", pm)
        bsk.set_option("k_order", 1)
        bsk.set_option("num_sms", sms)
        try:
            outs[pm] = run(order, transa, transb, Ar, Br, pad_a=8, pad_b=16, pad_c=8)[0]
        finally:
            bsk.set_option("pair_m", 0)
            bsk.set_option("k_order", 0)
            bsk.set_option("num_sms", 0)
    assert np.array_equal(outs[1], outs[2])
