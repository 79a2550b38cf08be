"""GPU parity of gemv_bf16 (decode GEMV, n <= 8, and the prefill GEMM, n > 8)
against the oracle, through the C ABI."""
import numpy as np
import pytest

import oracle
from bf16_gemm_skinny_gb300 import _native as bsk
from bf16_gemm_skinny_gb300 import build as bsk_build
from bf16_gemm_skinny_gb300 import inputs
from helpers import BF16_NAN, CANARY, absmax_bf16, check_tolerance, from_dev, poisoned, to_dev

pytestmark = pytest.mark.gpu

_CACHE = {}


def operands(M, K, n, integer):
    key = (M, K, n, integer)
    if key not in _CACHE:
        if integer:
            _CACHE[key] = inputs.linear_operands(M, K, n, "int2", "int2", seed_x=11, seed_w=12)
        else:
            _CACHE[key] = inputs.linear_operands(M, K, n, "normal0.02", "normal1")
    return _CACHE[key]


@pytest.fixture(scope="module", autouse=True)
def lib():
    import torch

    bsk_build.build()
    oracle.build()
    torch.cuda.init()
    yield bsk.load()
    for k in bsk.OPTIONS:
        bsk.set_option(k, 0)


def run(W, x, M, K, n, offset=0):
    import torch

    Wd = to_dev(np.concatenate([np.zeros(offset, np.uint16), W]))[offset:]
    xd = to_dev(np.concatenate([np.zeros(offset, np.uint16), x]))[offset:]
    buf, _ = poisoned(n * M + offset, BF16_NAN)
    y = buf[offset:offset + n * M]
    bsk.gemv_bf16(Wd, xd, y, M, K, n)
    torch.cuda.synchronize()
    assert np.all(from_dev(buf[offset + n * M:]) == CANARY), "guard words after y were written"
    assert np.array_equal(from_dev(Wd), W), "W was modified"
    assert np.array_equal(from_dev(xd), x), "x was modified"
    return from_dev(y).reshape(n, M)


@pytest.mark.parametrize("n", [1, 4, 8])
def test_decode_34816x5120_full(n):
    """The decode shape at full size; every output checked."""
    M, K = 34816, 5120
    W, x = operands(M, K, n, False)
    got = run(W, x, M, K, n)
    ref, _ = oracle.linear_bf16(W, x, M, K, n)
    check_tolerance(got, ref, "bf16", K, absmax_bf16(x), absmax_bf16(W), f"gemv n={n}")


@pytest.mark.parametrize("n", [1, 4, 8])
def test_decode_34816x5120_integer_bit_exact(n):
    M, K = 34816, 5120
    W, x = operands(M, K, n, True)
    _, want = oracle.linear_bf16(W, x, M, K, n)
    assert np.array_equal(run(W, x, M, K, n), want)


@pytest.mark.parametrize("n", range(1, 9))
@pytest.mark.parametrize("M,K", [(1003, 1032), (1, 8), (33, 5120), (4096, 256)])
def test_every_token_count(n, M, K):
    W, x = operands(M, K, n, True)
    _, want = oracle.linear_bf16(W, x, M, K, n)
    assert np.array_equal(run(W, x, M, K, n), want)
    W, x = operands(M, K, n, False)
    ref, _ = oracle.linear_bf16(W, x, M, K, n)
    check_tolerance(run(W, x, M, K, n), ref, "bf16", K, absmax_bf16(x), absmax_bf16(W), f"{M}x{K} n={n}")


GEMV_KERNEL_ROWS = [(k, r) for k in (1, 2, 3) for r in (1, 2, 4, 8)] + [(4, 4), (4, 8)]


@pytest.mark.parametrize("kernel,rows", GEMV_KERNEL_ROWS)
@pytest.mark.parametrize("warps", [1, 3, 8, 16])
@pytest.mark.parametrize("n", [1, 3, 5, 8])
def test_kernels_rows_per_warp_and_block_shape(kernel, rows, warps, n):
    """Every GEMV kernel (register streaming, cp.async pipeline with FP32 or BF16 x,
    token-paired) at its rows-per-warp and block shapes gives the oracle's bits on
    integer inputs."""
    M, K = 2051, 2048
    W, x = operands(M, K, n, True)
    _, want = oracle.linear_bf16(W, x, M, K, n)
    bsk.set_option("gemv_kernel", kernel)
    bsk.set_option("gemv_rows", rows)
    bsk.set_option("gemv_warps", warps)
    try:
        got = run(W, x, M, K, n)
    finally:
        bsk.set_option("gemv_kernel", 0)
        bsk.set_option("gemv_rows", 0)
        bsk.set_option("gemv_warps", 0)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("kernel", [1, 2, 3, 4, 5])
@pytest.mark.parametrize("n", [1, 2, 4, 5, 8])
def test_all_kernels_full_decode_shape(kernel, n):
    M, K = 34816, 5120
    W, x = operands(M, K, n, False)
    ref, _ = oracle.linear_bf16(W, x, M, K, n)
    bsk.set_option("gemv_kernel", kernel)
    try:
        got = run(W, x, M, K, n)
    finally:
        bsk.set_option("gemv_kernel", 0)
    check_tolerance(got, ref, "bf16", K, absmax_bf16(x), absmax_bf16(W), f"gemv kernel={kernel} n={n}")


@pytest.mark.parametrize("M,K,n,offset", [(517, 1001, 3, 0), (517, 1001, 4, 0), (300, 4096, 8, 1), (64, 7, 1, 0)])
@pytest.mark.parametrize("kernel", [0, 1])
def test_scalar_variant(M, K, n, offset, kernel):
    """K not a multiple of 8, or unaligned pointers: the scalar CUDA-core kernel
    (kernel 1 requested, or by default for n <= 3), or by default for n >= 4
    the tensor-core path on packed operands."""
    W, x = operands(M, K, n, False)
    ref, _ = oracle.linear_bf16(W, x, M, K, n)
    bsk.set_option("gemv_kernel", kernel)
    try:
        got = run(W, x, M, K, n, offset=offset)
    finally:
        bsk.set_option("gemv_kernel", 0)
    check_tolerance(got, ref, "bf16", K, absmax_bf16(x), absmax_bf16(W), f"unaligned, kernel {kernel}")


@pytest.mark.parametrize("n", [1, 8])
def test_k_slabs(n):
    """x larger than the shared-memory budget is staged in k-slabs."""
    M, K = 301, 20000
    W, x = operands(M, K, n, True)
    _, want = oracle.linear_bf16(W, x, M, K, n)
    assert np.array_equal(run(W, x, M, K, n), want)


@pytest.mark.parametrize("kernel", [1, 2])
@pytest.mark.parametrize("M,K,n", [(1000, 520, 100), (256, 256, 9), (777, 1032, 300), (1024, 64, 4096),
                                   (3000, 2048, 12), (2048, 1024, 32), (1500, 512, 64), (1024, 5120, 128)])
def test_prefill_medium(kernel, M, K, n):
    bsk.set_option("gemm_kernel", kernel)
    try:
        _prefill_medium(M, K, n)
    finally:
        bsk.set_option("gemm_kernel", 0)


def _prefill_medium(M, K, n):
    for integer in (True, False):
        W, x = operands(M, K, n, integer)
        ref, want = oracle.linear_bf16(W, x, M, K, n)
        got = run(W, x, M, K, n)
        if integer:
            assert np.array_equal(got, want)
        else:
            check_tolerance(got, ref, "bf16", K, absmax_bf16(x), absmax_bf16(W), f"prefill {M}x{K} n={n}")


@pytest.mark.parametrize("integer", [False, True])
def test_prefill_4096x34816x5120_sampled(integer):
    """The prefill projection at full size, checked on sampled tokens and features."""
    M, K, n = 34816, 5120, 4096
    W, x = operands(M, K, n, integer)
    got = run(W, x, M, K, n)
    ts = [0, 1, 255, 256, 4095]
    reft, outt = oracle.linear_bf16_tokens(W, x, M, K, n, ts)
    js = [0, 127, 128, 20000, 34815]
    refj, outj = oracle.linear_bf16(W, x, M, K, n, js=js)
    if integer:
        assert np.array_equal(got[ts, :], outt)
        assert np.array_equal(got[:, js], outj)
    else:
        check_tolerance(got[ts, :], reft, "bf16", K, absmax_bf16(x), absmax_bf16(W), "prefill tokens")
        check_tolerance(got[:, js], refj, "bf16", K, absmax_bf16(x), absmax_bf16(W), "prefill features")


@pytest.mark.parametrize("n", [9, 16, 64, 128])
def test_skinny_34816x5120_full(n):
    """Skinny tensor-core path (8 < n <= 128: one CTA per 128 x {32,64,128} tile) at the
    decode shape, every output checked."""
    M, K = 34816, 5120
    W, x = operands(M, K, n, False)
    ref, _ = oracle.linear_bf16(W, x, M, K, n)
    check_tolerance(run(W, x, M, K, n), ref, "bf16", K, absmax_bf16(x), absmax_bf16(W), f"skinny n={n}")


@pytest.mark.parametrize("block_m", [8, 40, 64, 120, 128])
@pytest.mark.parametrize("M,K,n", [(34816, 1032, 4), (4095, 1032, 8), (1003, 640, 32), (777, 2048, 100)])
def test_skinny_tile_heights(block_m, M, K, n):
    """The tensor-core skinny path with tiles of block_m rows of W (the heights
    of the balanced schedule, forced; the MMA still computes 128 rows, of which
    only the tile's are stored): integer inputs match the oracle bit for bit,
    random ones stay within tolerance."""
    bsk.set_option("block_m", block_m)
    bsk.set_option("gemv_kernel", 5)
    try:
        W, x = operands(M, K, n, True)
        _, want = oracle.linear_bf16(W, x, M, K, n)
        assert np.array_equal(run(W, x, M, K, n), want)
        W, x = operands(M, K, n, False)
        ref, _ = oracle.linear_bf16(W, x, M, K, n)
        check_tolerance(run(W, x, M, K, n), ref, "bf16", K, absmax_bf16(x), absmax_bf16(W),
                        f"{M}x{K} n={n} block_m={block_m}")
    finally:
        bsk.set_option("block_m", 0)
        bsk.set_option("gemv_kernel", 0)


@pytest.mark.parametrize("prefetch_kb", [1, 2, 64])
@pytest.mark.parametrize("M,K,n,offset,block_m", [(34816, 5120, 4, 0, 0), (1003, 1032, 8, 1, 0), (4095, 200, 16, 0, 0),
                                                  (777, 2048, 100, 0, 0), (4095, 1032, 8, 0, 40)])
def test_skinny_prologue_prefetch_depths(prefetch_kb, M, K, n, offset, block_m):
    """The L2 prefetch of the first tile's weight rows in the prologue is a hint:
    none, the shortest and the deepest setting -- on the decode shape, a packed
    (unaligned) W, a k loop shorter than the prefetch, a ragged M and a forced
    tile height -- give the oracle's bits on integer inputs."""
    bsk.set_option("prefetch_kb", prefetch_kb)
    bsk.set_option("block_m", block_m)
    try:
        W, x = operands(M, K, n, True)
        _, want = oracle.linear_bf16(W, x, M, K, n)
        assert np.array_equal(run(W, x, M, K, n, offset), want)
    finally:
        bsk.set_option("prefetch_kb", 0)
        bsk.set_option("block_m", 0)


@pytest.mark.parametrize("M,K,n", [(1100, 640, 600), (2048, 1032, 1024)])
def test_prefill_on_512_row_pair_tiles(M, K, n):
    """The BF16 prefill product (K-major W and x) on CTA pairs with 512 x 256
    tiles forced (on 8 SMs, so that the planner keeps CTA pairs for these
    short k loops): integer inputs give the oracle's bits."""
    bsk.set_option("pair_m", 2)
    bsk.set_option("num_sms", 8)
    try:
        W, x = operands(M, K, n, True)
        _, want = oracle.linear_bf16(W, x, M, K, n)
        assert np.array_equal(run(W, x, M, K, n), want)
    finally:
        bsk.set_option("pair_m", 0)
        bsk.set_option("num_sms", 0)


def test_k_zero_and_empty():
    got = run(np.zeros(0, np.uint16), np.zeros(0, np.uint16), 50, 0, 3)
    assert np.all(got == 0)
    got = run(np.zeros(0, np.uint16), np.zeros(0, np.uint16), 50, 0, 20)
    assert np.all(got == 0)
