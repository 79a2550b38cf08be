"""GPU parity of gemm_f16_colmajor against the oracle (called through the C ABI).

Random inputs: the tolerance in helpers.check_tolerance.  Integer-valued
inputs (entries in {-2..2}): bit-identical to the oracle.  Every call also
checks that the output was fully overwritten (it starts as NaN), that the
guard words after it are untouched and that the inputs are unchanged.
"""
import numpy as np
import pytest

import oracle
from bf16_gemm_skinny_gb300 import _native as bsk
from bf16_gemm_skinny_gb300 import build as bsk_build
from bf16_gemm_skinny_gb300 import inputs
from helpers import (CANARY, FP16_NAN, absmax_f16, check_tolerance, from_dev, poisoned, to_dev)

pytestmark = pytest.mark.gpu

_CACHE = {}


def operands(M, N, K, dist):
    key = (M, N, K, dist)
    if key not in _CACHE:
        seeds = (11, 12) if dist == "int2" else (1, 2)
        _CACHE[key] = inputs.gemm_operands(M, N, K, dist, *seeds)
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


def run(A, B, M, N, K, offset=0, enqueue=False):
    """Runs the GEMM on device copies of A, B; returns C's bits.  offset > 0
    shifts all three device pointers by that many elements (unaligned bases)."""
    import torch

    Ad = to_dev(np.concatenate([np.zeros(offset, np.uint16), A]))[offset:]
    Bd = to_dev(np.concatenate([np.zeros(offset, np.uint16), B]))[offset:]
    buf, _ = poisoned(M * N + offset, FP16_NAN)
    C = buf[offset:offset + M * N]
    if enqueue:
        bsk.gemm_f16_colmajor_enqueue(Ad, Bd, C, M, N, K)
        bsk.stream_check()
    else:
        bsk.gemm_f16_colmajor(Ad, Bd, C, M, N, K)
    torch.cuda.synchronize()
    assert np.all(from_dev(buf[offset + M * N:]) == CANARY), "guard words after C were written"
    assert np.array_equal(from_dev(Ad), A), "A was modified"
    assert np.array_equal(from_dev(Bd), B), "B was modified"
    return from_dev(C)


SMALL_SHAPES = [
    (256, 256, 256),      # the 256^3 workload
    (1, 1, 1), (1, 300, 17), (17, 33, 19), (8, 8, 8), (64, 64, 64),
    (128, 256, 64), (129, 257, 65), (127, 1, 63), (300, 517, 200), (1000, 777, 1030), (640, 520, 4096),
]


@pytest.mark.parametrize("M,N,K", SMALL_SHAPES)
def test_integer_inputs_bit_exact(M, N, K):
    A, B = operands(M, N, K, "int2")
    got = run(A, B, M, N, K)
    _, want = oracle.gemm_f16_colmajor(A, B, M, N, K)
    assert np.array_equal(got, want), f"{int((got != want).sum())} of {got.size} entries differ"


@pytest.mark.parametrize("M,N,K", SMALL_SHAPES)
def test_random_inputs_within_tolerance(M, N, K):
    dist = "uniform" if (M, N, K) == (256, 256, 256) else "normal0.5"
    A, B = operands(M, N, K, dist)
    got = run(A, B, M, N, K)
    ref, _ = oracle.gemm_f16_colmajor(A, B, M, N, K)
    check_tolerance(got, ref, "f16", K, absmax_f16(A), absmax_f16(B), f"{M}x{N}x{K}")


def sampled_check(got, A, B, M, N, K, cols, rows, integer):
    refc, outc = oracle.gemm_f16_colmajor(A, B, M, N, K, cols=cols)
    got_c = np.concatenate([got[n * M:(n + 1) * M] for n in cols])
    refr, outr = oracle.gemm_f16_colmajor_rows(A, B, M, N, K, rows)
    got_r = np.concatenate([got[np.arange(N) * M + m] for m in rows])
    # oracle rows come column-major over the selected rows: entry (i, n) at i + n*len(rows)
    refr = refr.reshape(N, len(rows)).T.reshape(-1)
    outr = outr.reshape(N, len(rows)).T.reshape(-1)
    if integer:
        assert np.array_equal(got_c, outc)
        assert np.array_equal(got_r, outr)
    else:
        check_tolerance(got_c, refc, "f16", K, absmax_f16(A), absmax_f16(B), "sampled columns")
        check_tolerance(got_r, refr, "f16", K, absmax_f16(A), absmax_f16(B), "sampled rows")


@pytest.mark.parametrize("dist", ["normal0.5", "int2"])
def test_ragged_4095x4097x4100(dist):
    """Tails in M, N and K, unaligned leading dimensions (pack + masked stores),
    and a GROUP_M remainder group (32 tile rows, group 12)."""
    M, N, K = 4095, 4097, 4100
    A, B = operands(M, N, K, dist)
    bsk.set_option("group_m", 12)
    try:
        got = run(A, B, M, N, K)
    finally:
        bsk.set_option("group_m", 0)
    cols = [0, 1, 255, 256, 2047, 4095, 4096]
    rows = [0, 127, 128, 2049, 4094]
    sampled_check(got, A, B, M, N, K, cols, rows, dist == "int2")
    if dist == "int2":
        # every sum is an integer below 2^24: the exact product, full output
        a = oracle.f16_decode(A).reshape(K, M).T
        b = oracle.f16_decode(B).reshape(N, K).T
        want = oracle.f16_encode((a @ b).T.reshape(-1))
        assert np.array_equal(got, want)


@pytest.mark.parametrize("dist", ["uniform", "int2"])
def test_8192x8192x16384_sampled(dist):
    """The headline shape, in the launch configuration the benchmark times."""
    M, N, K = 8192, 8192, 16384
    A, B = operands(M, N, K, dist)
    got = run(A, B, M, N, K)
    assert np.all(np.isfinite(oracle.f16_decode(got[::997])))
    cols = [0, 255, 256, 4099, 8191]
    rows = [0, 127, 128, 5000, 8191]
    sampled_check(got, A, B, M, N, K, cols, rows, dist == "int2")


@pytest.mark.parametrize("kernel,block_n,group_m", [
    (2, 256, 8), (2, 256, 1), (2, 256, 3), (1, 256, 8), (1, 256, 3), (1, 128, 1), (1, 128, 12),
    (1, 64, 5), (1, 32, 2)])
def test_result_independent_of_tile_config(kernel, block_n, group_m):
    """CTA-pair 256x256 tiles, single-CTA 128x256 / 128x128 / 128x64 / 128x32 tiles,
    several GROUP_M: bit-identical to the oracle on integer inputs."""
    M, N, K = 1000, 777, 1030
    A, B = operands(M, N, K, "int2")
    _, want = oracle.gemm_f16_colmajor(A, B, M, N, K)
    bsk.set_option("gemm_kernel", kernel)
    bsk.set_option("block_n", block_n)
    bsk.set_option("group_m", group_m)
    try:
        got = run(A, B, M, N, K)
    finally:
        bsk.set_option("gemm_kernel", 0)
        bsk.set_option("block_n", 0)
        bsk.set_option("group_m", 0)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("M,N,K", [(256, 256, 256), (129, 257, 65), (1000, 777, 1030), (300, 517, 200),
                                   (4096, 9, 1024), (1000, 33, 520), (2000, 100, 4096)])
def test_single_cta_kernel(M, N, K):
    """The one-CTA-per-tile kernel stays correct beside the default CTA-pair kernel."""
    A, B = operands(M, N, K, "normal0.5")
    bsk.set_option("gemm_kernel", 1)
    try:
        got = run(A, B, M, N, K)
    finally:
        bsk.set_option("gemm_kernel", 0)
    ref, _ = oracle.gemm_f16_colmajor(A, B, M, N, K)
    check_tolerance(got, ref, "f16", K, absmax_f16(A), absmax_f16(B), f"single-CTA {M}x{N}x{K}")


def test_deterministic_run_to_run():
    M, N, K = 1024, 1536, 2048
    A, B = operands(M, N, K, "normal0.5")
    first = run(A, B, M, N, K)
    for _ in range(2):
        assert np.array_equal(run(A, B, M, N, K), first)


@pytest.mark.parametrize("option", ["force_pack", "force_direct_store"])
def test_pack_and_store_paths_agree(option):
    M, N, K = 1024, 640, 1040
    A, B = operands(M, N, K, "normal0.5")
    base = run(A, B, M, N, K)
    bsk.set_option(option, 1)
    try:
        other = run(A, B, M, N, K)
    finally:
        bsk.set_option(option, 0)
    assert np.array_equal(base, other)


@pytest.mark.parametrize("M,N,K", [(256, 256, 256), (333, 129, 70)])
def test_unaligned_pointers(M, N, K):
    A, B = operands(M, N, K, "normal0.5")
    got = run(A, B, M, N, K, offset=1)
    ref, _ = oracle.gemm_f16_colmajor(A, B, M, N, K)
    check_tolerance(got, ref, "f16", K, absmax_f16(A), absmax_f16(B), "unaligned")


def test_k_zero_writes_zeros():
    got = run(np.zeros(0, np.uint16), np.zeros(0, np.uint16), 37, 19, 0)
    assert np.all(got == 0)


def test_enqueue_variant_matches_blocking():
    M, N, K = 512, 384, 320
    A, B = operands(M, N, K, "normal0.5")
    assert np.array_equal(run(A, B, M, N, K, enqueue=True), run(A, B, M, N, K))


def test_watchdog_gives_up_and_library_stays_usable():
    """A wait that nothing satisfies returns BSK_ERR_TIMEOUT instead of hanging;
    the context is still healthy afterwards."""
    assert bsk.test_wait_timeout(2000) == 4
    assert "gave up" in bsk.last_error()
    test_integer_inputs_bit_exact(129, 257, 65)


def test_binding_uses_the_current_torch_stream():
    """Without an explicit stream the binding launches on torch's current stream
    (here a side stream); the work is ordered on that stream."""
    import torch

    M, N, K = 512, 384, 320
    A, B = operands(M, N, K, "int2")
    _, want = oracle.gemm_f16_colmajor(A, B, M, N, K)
    Ad, Bd = to_dev(A), to_dev(B)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        assert bsk._stream(None) == side.cuda_stream
        C = torch.full((M * N,), FP16_NAN, dtype=torch.int16, device="cuda")
        bsk.gemm_f16_colmajor_enqueue(Ad, Bd, C, M, N, K)
    side.synchronize()
    assert np.array_equal(from_dev(C), want)
    assert bsk._stream(None) == torch.cuda.current_stream().cuda_stream
    C2 = torch.empty(M * N, dtype=torch.int16, device="cuda")
    bsk.gemm_f16_colmajor_enqueue(Ad, Bd, C2, M, N, K, stream=side)
    side.synchronize()
    assert np.array_equal(from_dev(C2), want)


@pytest.mark.parametrize("M,N,K,block_n,sms", [
    (1000, 777, 1030, 128, 0), (1000, 777, 1030, 64, 0), (1000, 777, 1030, 32, 7),
    (512, 64, 4096, 64, 0),       # 4 tiles x 64 k-blocks over every SM: ~38 CTAs per tile
    (4096, 9, 1024, 32, 0), (300, 517, 64, 128, 0), (129, 257, 65, 256, 5)])
def test_stream_k_schedule(M, N, K, block_n, sms):
    """Stream-K on the one-CTA-per-tile kernel (forced): integer inputs give the
    oracle's bits whatever the split; random inputs stay within tolerance and
    repeat bit for bit."""
    A, B = operands(M, N, K, "int2")
    _, want = oracle.gemm_f16_colmajor(A, B, M, N, K)
    opts = {"gemm_kernel": 1, "block_n": block_n, "stream_k": 2, "num_sms": sms}
    for k, v in opts.items():
        bsk.set_option(k, v)
    try:
        assert np.array_equal(run(A, B, M, N, K), want)
        Ar, Br = operands(M, N, K, "normal0.5")
        got = run(Ar, Br, M, N, K)
        assert np.array_equal(run(Ar, Br, M, N, K), got)
    finally:
        for k in opts:
            bsk.set_option(k, 0)
    ref, _ = oracle.gemm_f16_colmajor(Ar, Br, M, N, K)
    check_tolerance(got, ref, "f16", K, absmax_f16(Ar), absmax_f16(Br), f"stream-K {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K,sms", [(1000, 777, 1030, 0), (4095, 4097, 4100, 0), (300, 517, 2048, 9),
                                       (2048, 1024, 8192, 0)])
def test_stream_k_on_cta_pairs(M, N, K, sms):
    """Stream-K on the CTA-pair kernel (forced): integer inputs give the oracle's
    bits; the column-major result repeats bit for bit."""
    A, B = operands(M, N, K, "int2")
    opts = {"stream_k": 2, "num_sms": sms}
    for k, v in opts.items():
        bsk.set_option(k, v)
    try:
        got = run(A, B, M, N, K)
        again = run(A, B, M, N, K)
    finally:
        for k in opts:
            bsk.set_option(k, 0)
    assert np.array_equal(got, again)
    cols = sorted({0, 1, 255, 256, N // 2, N - 1})
    rows = sorted({0, 127, 128, M // 2, M - 1})
    sampled_check(got, A, B, M, N, K, cols, rows, True)


@pytest.mark.parametrize("M,N,K", [(256, 256, 2048), (128, 128, 16384), (300, 517, 2048), (512, 512, 4096),
                                   (129, 33, 4160)])
def test_few_tiles_long_k_default_schedule(M, N, K):
    """Few tiles with a long k loop: the default plan splits each tile's k loop
    over a cluster of CTAs that add their partials through distributed shared
    memory.
    Integer inputs give the oracle's bits; random inputs stay within tolerance
    and repeat bit for bit."""
    A, B = operands(M, N, K, "int2")
    _, want = oracle.gemm_f16_colmajor(A, B, M, N, K)
    assert np.array_equal(run(A, B, M, N, K), want)
    Ar, Br = operands(M, N, K, "normal0.5")
    got = run(Ar, Br, M, N, K)
    assert np.array_equal(run(Ar, Br, M, N, K), got)
    ref, _ = oracle.gemm_f16_colmajor(Ar, Br, M, N, K)
    check_tolerance(got, ref, "f16", K, absmax_f16(Ar), absmax_f16(Br), f"few tiles {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", [
    (2048, 2048, 256),     # short k loop on many tiles: one CTA per 128 x 256 tile instead of CTA pairs
    (2304, 2560, 512),
    (2048, 2048, 2048),    # 32 k-blocks, all 128 single-CTA tiles in one wave
    (128, 8192, 2048),     # tile-starved, k loop too short to split: whole 128 x 64 tiles
    (8192, 128, 2048)])
def test_planner_regimes(M, N, K):
    """The default plan in each regime the planner tells apart gives the oracle's
    bits on integer inputs and stays within tolerance on random ones."""
    A, B = operands(M, N, K, "int2")
    _, want = oracle.gemm_f16_colmajor(A, B, M, N, K)
    assert np.array_equal(run(A, B, M, N, K), want)
    Ar, Br = operands(M, N, K, "normal0.5")
    got = run(Ar, Br, M, N, K)
    ref, _ = oracle.gemm_f16_colmajor(Ar, Br, M, N, K)
    check_tolerance(got, ref, "f16", K, absmax_f16(Ar), absmax_f16(Br), f"plan {M}x{N}x{K}")


def _random_shapes(count, seed, min_work, max_work):
    """Seeded shapes over every regime of the planner: each of M, N, K drawn
    log-uniformly from 1..8192 (K up to 16384), half of them rounded to a
    multiple of 8 (aligned C, TMA stores), with min_work..max_work multiply-adds."""
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < count:
        M, N = (int(np.exp(rng.uniform(0, np.log(8192)))) for _ in range(2))
        K = int(np.exp(rng.uniform(0, np.log(16384))))
        if rng.random() < 0.5:
            M, N, K = (max(8, (v + 7) // 8 * 8) for v in (M, N, K))
        if min_work <= M * N * K <= max_work:
            out.append((M, N, K))
    return out


@pytest.mark.parametrize("M,N,K", _random_shapes(40, 2026, 1, 6e8) + _random_shapes(20, 2027, 3e8, 4e9))
def test_random_shapes_default_plan(M, N, K):
    """Whatever plan the planner picks for a shape (CTA pairs, one-CTA tiles of
    any width, split-K over clusters, stream-K, the pack for unaligned leading
    dimensions), integer inputs give the oracle's bits in every element."""
    A, B = operands(M, N, K, "int2")
    _, want = oracle.gemm_f16_colmajor(A, B, M, N, K)
    assert np.array_equal(run(A, B, M, N, K), want), f"{M}x{N}x{K}"


@pytest.mark.parametrize("M,N,K,block_n,skc", [
    (1000, 777, 1030, 32, 2), (1000, 777, 1030, 64, 4), (1000, 777, 1030, 128, 8), (1000, 777, 1030, 256, 16),
    (129, 257, 65, 32, 8),        # 2 k-blocks over 8 CTAs: six hold empty (zero) partials
    (300, 517, 2048, 32, 16), (4095, 40, 4100, 32, 4), (64, 20, 96, 32, 2)])
def test_split_k_over_clusters(M, N, K, block_n, skc):
    """Split-K over a cluster of the one-CTA kernel (forced): every CTA leaves its
    partial in shared memory, the cluster sums each column slice in rank order
    through distributed shared memory.  Integer inputs give the oracle's bits;
    random inputs stay within tolerance and repeat bit for bit."""
    A, B = operands(M, N, K, "int2")
    Ar, Br = operands(M, N, K, "normal0.5")
    opts = {"gemm_kernel": 1, "block_n": block_n, "split_k": skc}
    for k, v in opts.items():
        bsk.set_option(k, v)
    try:
        got = run(A, B, M, N, K)
        got_r = run(Ar, Br, M, N, K)
        again = run(Ar, Br, M, N, K)
    finally:
        for k in opts:
            bsk.set_option(k, 0)
    _, want = oracle.gemm_f16_colmajor(A, B, M, N, K)
    assert np.array_equal(got, want)
    assert np.array_equal(got_r, again)
    ref, _ = oracle.gemm_f16_colmajor(Ar, Br, M, N, K)
    check_tolerance(got_r, ref, "f16", K, absmax_f16(Ar), absmax_f16(Br), f"split-K {skc} {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", [(1000, 777, 1030), (256, 256, 64), (300, 517, 200), (2304, 2560, 1024),
                                   (4095, 4097, 4100)])
def test_dynamic_tile_order_on_cta_pairs(M, N, K):
    """CTA pairs with the dynamic tile order forced (one cluster per tile launched,
    free pairs taking the tiles of clusters whose launch they cancel), from a
    single tile up to 17 x 16 tiles: integer inputs give the oracle's bits, and
    on random inputs the result equals the fixed order's bit for bit (a tile's
    sum does not depend on which pair computes it)."""
    A, B = operands(M, N, K, "int2")
    bsk.set_option("tile_sched", 2)
    try:
        got = run(A, B, M, N, K)
    finally:
        bsk.set_option("tile_sched", 0)
    cols = sorted(c for c in {0, 1, 255, 256, N // 2, N - 1} if c < N)
    rows = sorted(r for r in {0, 127, 128, M // 2, M - 1} if r < M)
    sampled_check(got, A, B, M, N, K, cols, rows, True)
    Ar, Br = operands(M, N, K, "normal0.5")
    outs = {}
    for sched in (1, 2):
        bsk.set_option("tile_sched", sched)
        try:
            outs[sched] = run(Ar, Br, M, N, K)
        finally:
            bsk.set_option("tile_sched", 0)
    assert np.array_equal(outs[1], outs[2])


@pytest.mark.parametrize("M,N,K,sms", [(4095, 4097, 4100, 0), (2304, 2560, 1024, 0), (1000, 777, 1030, 8),
                                       (300, 517, 2048, 9)])
def test_k_order_of_rounds_on_cta_pairs(M, N, K, sms):
    """CTA pairs over two or more rounds of tiles, with odd rounds running their
    k loop downwards (the default) and with every k loop ascending: integer inputs
    give the oracle's bits either way, and random inputs stay within tolerance
    and repeat bit for bit."""
    A, B = operands(M, N, K, "int2")
    Ar, Br = operands(M, N, K, "normal0.5")
    cols = sorted(c for c in {0, 1, 255, 256, 511, 512, N // 2, N - 1} if c < N)
    rows = sorted(r for r in {0, 127, 128, 255, 256, M // 2, M - 1} if r < M)
    outs = {}
    for order in (0, 1):
        bsk.set_option("num_sms", sms)
        bsk.set_option("k_order", order)
        try:
            sampled_check(run(A, B, M, N, K), A, B, M, N, K, cols, rows, True)
            outs[order] = run(Ar, Br, M, N, K)
            assert np.array_equal(run(Ar, Br, M, N, K), outs[order])
        finally:
            bsk.set_option("k_order", 0)
            bsk.set_option("num_sms", 0)
        sampled_check(outs[order], Ar, Br, M, N, K, cols, rows, False)


@pytest.mark.parametrize("sms,offset", [(1, 3), (2, 0), (5, 7)])
def test_pack_on_few_sms(sms, offset):
    """The pack on a grid capped to a few SMs: each warp streams hundreds of
    512-byte steps through its ring (many wrap-arounds, line changes inside a
    warp's range, the partial last group of every line), both operands in one
    launch; the result must equal the oracle's bit for bit."""
    M, N, K = 1001, 515, 1037
    A, B = operands(M, N, K, "int2")
    bsk.set_option("num_sms", sms)
    try:
        got = run(A, B, M, N, K, offset=offset)
    finally:
        bsk.set_option("num_sms", 0)
    _, want = oracle.gemm_f16_colmajor(A, B, M, N, K)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("offset", range(8))
def test_pack_every_base_offset(offset):
    """Bases at every 2-byte offset inside a 16-byte chunk and odd leading
    dimensions: the pack's aligned loads and shifts, bit for bit."""
    M, N, K = 257, 130, 67
    A, B = operands(M, N, K, "int2")
    got = run(A, B, M, N, K, offset=offset)
    _, want = oracle.gemm_f16_colmajor(A, B, M, N, K)
    assert np.array_equal(got, want)
