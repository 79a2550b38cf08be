"""Host-side checks that need no GPU: the library loads and exports every
symbol of include/bsk.h, the tile rasteriser is a bijection onto the tile
grid (remainder group included), argument validation rejects bad calls
before touching a device, and the option table round-trips."""
import ctypes
import os
import re

import pytest

from bf16_gemm_skinny_gb300 import _native as bsk
from bf16_gemm_skinny_gb300 import build as bsk_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    bsk_build.build()
    return bsk.load()


def header_functions(path=("include", "bsk.h")):
    text = open(os.path.join(ROOT, *path)).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?(?:int|void|long long|char)\s*\*?\s*(\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


TUNING_HEADER = ("bf16_gemm_skinny_gb300", "csrc", "bsk_tuning.h")


def test_header_declares_the_bound_symbols():
    assert header_functions() == sorted(bsk.EXPORTS)
    assert header_functions(TUNING_HEADER) == sorted(bsk.TUNING_EXPORTS)


def test_public_header_holds_no_tuning_state_or_test_hook():
    """The C ABI holds the product calls only: the process-wide options and the
    test hooks live in the internal tuning header."""
    public = header_functions()
    for name in bsk.TUNING_EXPORTS:
        assert name not in public, name
    text = open(os.path.join(ROOT, "include", "bsk.h")).read()
    assert "BSK_OPT_" not in text


def test_library_exports_every_header_symbol(lib):
    names = header_functions() + header_functions(TUNING_HEADER)
    for name in names:
        assert hasattr(lib, name), name
    out = os.popen(f"nm -D --defined-only {bsk.library_path()}").read()
    exported = set(re.findall(r" T (\w+)$", out, flags=re.M))
    missing = set(names) - exported
    assert not missing, missing


def test_version_and_status_strings(lib):
    assert bsk.version() >= 100
    for code, name in bsk.STATUS.items():
        assert lib.bsk_status_string(code).decode() == name


def tiles_of(num_m, num_n, group_m):
    return [bsk.tile_coord(t, num_m, num_n, group_m) for t in range(num_m * num_n)]


@pytest.mark.parametrize("num_m,num_n,group_m", [
    (1, 1, 1), (64, 32, 8), (32, 17, 12), (32, 17, 8), (7, 5, 3), (5, 7, 16), (272, 16, 8), (3, 100, 2),
])
def test_tile_coord_is_a_bijection(lib, num_m, num_n, group_m):
    got = tiles_of(num_m, num_n, group_m)
    assert sorted(got) == [(m, n) for m in range(num_m) for n in range(num_n)]


def test_tile_coord_group_order_and_remainder(lib):
    """Consecutive tiles walk down a group of group_m rows, then move one column;
    the last group holds num_m mod group_m rows ("Hygon 优化", 分组调度)."""
    num_m, num_n, g = 10, 4, 4
    got = tiles_of(num_m, num_n, g)
    assert got[:5] == [(0, 0), (1, 0), (2, 0), (3, 0), (0, 1)]
    tail = got[2 * g * num_n:]              # remainder group: rows 8, 9
    assert tail[:4] == [(8, 0), (9, 0), (8, 1), (9, 1)]
    assert {m for m, _ in tail} == {8, 9}


def test_tile_coord_rejects_bad_arguments(lib):
    assert bsk.tile_coord(5, 2, 2, 1) == (-1, -1)
    assert bsk.tile_coord(0, 0, 2, 1) == (-1, -1)
    assert bsk.tile_coord(0, 2, 2, 0) == (-1, -1)


FAKE = 1 << 40   # never dereferenced: validation fails before any device access


@pytest.mark.parametrize("args", [
    (FAKE, FAKE + (1 << 30), FAKE + (2 << 30), -1, 4, 4),
    (FAKE, FAKE + (1 << 30), FAKE + (2 << 30), 4, -1, 4),
    (FAKE, FAKE + (1 << 30), FAKE + (2 << 30), 4, 4, -3),
    (FAKE, FAKE + (1 << 30), None, 4, 4, 4),
    (None, FAKE + (1 << 30), FAKE + (2 << 30), 4, 4, 4),
    (FAKE, FAKE + 16, FAKE + 8, 4, 4, 4),             # C overlaps A
    (FAKE, FAKE + 4096, FAKE + 4096 + 8, 4, 4, 4),    # C overlaps B
])
def test_gemm_rejects_bad_arguments(lib, args):
    A, B, C, M, N, K = args
    assert lib.gemm_f16_colmajor(A, B, C, M, N, K, None) == 1
    assert lib.bsk_gemm_f16_colmajor_enqueue(A, B, C, M, N, K, None) == 1
    assert bsk.last_error()


@pytest.mark.parametrize("args", [
    (FAKE, FAKE + (1 << 30), FAKE + (2 << 30), -1, 4, 1),
    (FAKE, FAKE + (1 << 30), FAKE + (2 << 30), 4, 4, -1),
    (FAKE, FAKE + (1 << 30), None, 4, 4, 1),
    (FAKE, None, FAKE + (2 << 30), 4, 4, 1),
    (FAKE, FAKE + (1 << 30), FAKE + 2, 4, 4, 1),      # y overlaps W
])
def test_gemv_rejects_bad_arguments(lib, args):
    W, x, y, M, K, n = args
    assert lib.gemv_bf16(W, x, y, M, K, n, None) == 1
    assert lib.bsk_gemv_bf16_enqueue(W, x, y, M, K, n, None) == 1


G_A, G_B, G_C, G_BIAS = FAKE, FAKE + (1 << 30), FAKE + (2 << 30), FAKE + (3 << 30)


@pytest.mark.parametrize("args", [
    # order, transa, transb, A, lda, B, ldb, C, ldc, M, N, K, bias, bias_mode
    (2, 0, 0, G_A, 8, G_B, 8, G_C, 8, 8, 8, 8, None, 0),         # bad order
    (0, 2, 0, G_A, 8, G_B, 8, G_C, 8, 8, 8, 8, None, 0),         # bad transa
    (0, 0, -1, G_A, 8, G_B, 8, G_C, 8, 8, 8, 8, None, 0),        # bad transb
    (0, 0, 0, G_A, 8, G_B, 8, G_C, 8, 8, 8, 8, None, 3),         # bad bias mode
    (0, 0, 0, G_A, 8, G_B, 8, G_C, 8, 8, 8, 8, None, 1),         # bias mode without a bias
    (1, 0, 0, G_A, 8, G_B, 8, G_C, 8, 8, 8, 8, None, 2),
    (0, 0, 0, G_A, 7, G_B, 8, G_C, 8, 8, 8, 8, None, 0),         # lda < M
    (0, 1, 0, G_A, 8, G_B, 9, G_C, 9, 9, 9, 9, None, 0),         # transa: lda < K
    (0, 0, 1, G_A, 8, G_B, 8, G_C, 8, 8, 9, 8, None, 0),         # transb: ldb < N
    (0, 0, 0, G_A, 8, G_B, 8, G_C, 7, 8, 8, 8, None, 0),         # ldc < M
    (1, 0, 0, G_A, 8, G_B, 8, G_C, 7, 8, 8, 8, None, 0),         # row-major: ldc < N
    (1, 0, 0, G_A, 7, G_B, 8, G_C, 8, 8, 8, 8, None, 0),         # row-major: lda < K
    (0, 0, 0, G_A, 8, G_B, 8, G_C, 8, -1, 8, 8, None, 0),        # negative size
    (0, 0, 0, G_A, 8, G_B, 8, None, 8, 8, 8, 8, None, 0),        # C NULL
    (0, 0, 0, G_A, 8, G_B, 8, G_A + 126, 8, 8, 8, 8, None, 0),   # C overlaps A's last element
    (0, 0, 0, G_A, 8, G_B, 8, G_C, 8, 8, 8, 8, G_C + 14, 1),     # C overlaps the bias
    (0, 0, 0, G_A, 8, G_B, 8, G_C, 0, 0, 8, 8, None, 0),         # ldc 0 even for an empty C
])
def test_general_gemm_rejects_bad_arguments(lib, args):
    assert lib.gemm_f16(*args, None) == 1
    assert lib.bsk_gemm_f16_enqueue(*args, None) == 1
    assert bsk.last_error()


@pytest.mark.parametrize("args", [
    # format, A, lda, B, ldb, C, ldc, out_type, M, N, K, alpha
    (2, G_A, 64, G_B, 64, G_C, 64, 0, 64, 64, 64, 1.0),            # bad format
    (0, G_A, 64, G_B, 64, G_C, 64, 2, 64, 64, 64, 1.0),            # bad output type
    (1, G_A, 64, G_B, 64, G_C, 64, 1, 64, 64, 64, float("nan")),   # alpha not finite
    (0, G_A, 64, G_B, 64, G_C, 64, 0, 64, 64, 64, float("inf")),
    (0, G_A, 63, G_B, 64, G_C, 64, 0, 64, 64, 64, 1.0),            # lda < K
    (0, G_A, 64, G_B, 63, G_C, 64, 0, 64, 64, 64, 1.0),            # ldb < K
    (0, G_A, 64, G_B, 64, G_C, 63, 0, 64, 64, 64, 1.0),            # ldc < M
    (0, G_A, 64, G_B, 64, G_C, 64, 0, -1, 64, 64, 1.0),            # negative size
    (0, G_A, 64, G_B, 64, None, 64, 0, 64, 64, 64, 1.0),           # C NULL
    (0, None, 64, G_B, 64, G_C, 64, 0, 64, 64, 64, 1.0),           # A NULL
    (0, G_A, 64, G_B, 64, G_A + 4000, 64, 0, 64, 64, 64, 1.0),     # C overlaps A (bytes 0..4095)
    (0, G_A, 64, G_B, 64, G_B - 16 * 1024 + 4, 64, 0, 64, 64, 64, 1.0),  # FP32 C (16 KB) reaches into B
])
def test_fp8_gemm_rejects_bad_arguments(lib, args):
    assert lib.gemm_fp8(*args, None) == 1
    assert lib.bsk_gemm_fp8_enqueue(*args, None) == 1
    assert bsk.last_error()


def test_fp8_gemm_empty_output_is_a_no_op(lib):
    assert lib.gemm_fp8(0, None, 8, None, 8, None, 1, 0, 0, 5, 8, 1.0, None) == 0
    assert lib.gemm_fp8(1, None, 8, None, 8, None, 4, 1, 4, 0, 8, 1.0, None) == 0


def test_general_gemm_accepts_exact_leading_dimensions(lib):
    """Overlap is decided on the spans the strides reach: a C right after A's
    last element is not an overlap; on a machine without a GPU the call then
    fails only at the device check."""
    st = lib.gemm_f16(0, 0, 0, G_A, 8, G_B, 8, G_A + 128, 8, 8, 8, 8, None, 0, None)
    assert st in (2, 3), bsk.last_error()


def test_empty_outputs_are_no_ops_without_a_device(lib):
    assert lib.gemm_f16(0, 1, 1, None, 7, None, 5, None, 1, 0, 5, 7, None, 0, None) == 0
    assert lib.gemm_f16_colmajor(None, None, None, 0, 5, 7, None) == 0
    assert lib.gemm_f16_colmajor(None, None, None, 5, 0, 7, None) == 0
    assert lib.gemv_bf16(None, None, None, 0, 7, 1, None) == 0
    assert lib.gemv_bf16(None, None, None, 9, 7, 0, None) == 0


def test_host_buffer_calls_validate_without_a_gpu(lib):
    """Argument checks come before any CUDA call; K = 0 is the empty sum, filled on the host."""
    import numpy as np

    assert lib.gemm_f16_colmajor_host(None, None, None, -1, 4, 4, None) == 1
    assert lib.gemv_bf16_host(None, None, None, 4, 4, -2, None) == 1
    assert lib.gemm_f16_colmajor_host(None, None, None, 0, 4, 4, None) == 0
    assert lib.gemv_bf16_host(None, None, None, 4, 4, 0, None) == 0
    c = np.full(12, 0x5A5A, np.uint16)
    assert lib.gemm_f16_colmajor_host(None, None, c.ctypes.data, 3, 4, 4, None) == 1   # A, B NULL with K > 0
    a = np.ones(12, np.uint16)
    assert lib.gemm_f16_colmajor_host(a.ctypes.data, a.ctypes.data, a.ctypes.data, 3, 4, 4, None) == 1   # overlap
    assert lib.gemm_f16_colmajor_host(None, None, c.ctypes.data, 3, 4, 0, None) == 0
    assert np.all(c == 0)
    y = np.full(6, 0x5A5A, np.uint16)
    assert lib.gemv_bf16_host(None, None, y.ctypes.data, 3, 0, 2, None) == 0
    assert np.all(y == 0)


def test_options_round_trip_and_range_checks(lib):
    assert bsk.get_option("group_m") == 0
    bsk.set_option("group_m", 12)
    assert bsk.get_option("group_m") == 12
    bsk.set_option("group_m", 0)
    with pytest.raises(bsk.BskError):
        bsk.set_option("block_n", 96)
    with pytest.raises(bsk.BskError):
        bsk.set_option("gemv_rows", 3)
    for name, good, bad in (("pdl", 1, 2), ("tile_sched", 2, 3), ("stream_k", 2, 3), ("split_k", 16, 3),
                            ("prefetch_kb", 64, 65), ("k_order", 1, 2), ("pair_m", 2, 3)):
        bsk.set_option(name, good)
        assert bsk.get_option(name) == good
        bsk.set_option(name, 0)
        with pytest.raises(bsk.BskError):
            bsk.set_option(name, bad)
    assert lib.bsk_set_option(99, 1) == 1
    assert lib.bsk_set_option(len(bsk.OPTIONS) + 1, 1) == 1


@pytest.mark.parametrize("shape,kw,want", [
    # the headline product: CTA pairs on 512 x 256 tiles (a k loop of 256 blocks)
    ((8192, 8192, 16384), {}, dict(pair=1, block_n=256, pair_m=2)),
    ((6144, 6144, 8192), {}, dict(pair=1, pair_m=2)),
    # 80 k-blocks: the unhidden epilogue of 512-row tiles would cost more than they save
    ((34816, 4096, 5120), dict(a_mn_major=False), dict(pair=1, pair_m=1)),
    ((4095, 4097, 4100), {}, dict(pair=1, pair_m=1)),
    # 512-row tiles would fill the pairs worse (80 tiles in two waves against 144)
    ((2304, 4096, 8192), {}, dict(pair=1, pair_m=1)),
    # a transposed B and FP8 inputs keep 256 x 256 tiles
    ((8192, 8192, 16384), dict(b_mn_major=True), dict(pair=1, pair_m=1)),
    ((8192, 8192, 8192), dict(a_mn_major=False, fp8=True), dict(pair=1, pair_m=1)),
    # latency-bound and short-k shapes run one CTA per tile
    ((256, 256, 256), {}, dict(pair=0, block_n=32, pair_m=1)),
    ((8192, 8192, 256), {}, dict(pair=0, block_n=256)),
    # skinny decode: the tile width follows N
    ((34816, 16, 5120), dict(a_mn_major=False), dict(pair=0, block_n=32, split_k=0)),
    ((34816, 100, 5120), dict(a_mn_major=False), dict(pair=0, block_n=128)),
])
def test_planner_rules(lib, shape, kw, want):
    """The tile plan the GEMM planner picks on 152 SMs (no launch; split-K plans,
    which need the device's cluster capacity, are not considered here)."""
    plan = bsk.plan_gemm(*shape, **kw)
    assert {k: plan[k] for k in want} == want, plan


def test_planner_follows_forcing_options(lib):
    try:
        bsk.set_option("pair_m", 1)
        assert bsk.plan_gemm(8192, 8192, 16384)["pair_m"] == 1
        bsk.set_option("pair_m", 2)
        assert bsk.plan_gemm(34816, 4096, 5120, a_mn_major=False)["pair_m"] == 2
        bsk.set_option("pair_m", 0)
        bsk.set_option("tile_sched", 2)    # the dynamic order runs 256 x 256 tiles only
        plan = bsk.plan_gemm(8192, 8192, 16384)
        assert plan["dyn"] == 1 and plan["pair_m"] == 1
        bsk.set_option("tile_sched", 0)
        bsk.set_option("gemm_kernel", 1)   # one CTA per 128 x 256 tile
        assert bsk.plan_gemm(8192, 8192, 16384)["pair"] == 0
    finally:
        for k in ("pair_m", "tile_sched", "gemm_kernel"):
            bsk.set_option(k, 0)
    with pytest.raises(bsk.BskError):
        bsk.plan_gemm(0, 8, 8)


def test_watchdog_probe_validates_limit(lib):
    assert lib.bsk_test_wait_timeout(0, None) == 1
    assert lib.bsk_test_wait_timeout(20_000_000, None) == 1


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    """No fallback: a missing library is an error, not a silent CPU path."""
    monkeypatch.setattr(bsk, "_lib", None)
    monkeypatch.setattr(bsk_build, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        bsk.load()
