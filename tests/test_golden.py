"""The workload arithmetic the benchmark reports, checked against the numbers
the pages print (tests/golden/workload_arithmetic.txt, each line cited)."""
import os

import pytest

import bench

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "workload_arithmetic.txt")


def golden():
    rows = {}
    for line in open(GOLDEN, encoding="utf-8"):
        if line.startswith("#") or not line.strip():
            continue
        name, _inputs, value, tol, _src = (f.strip() for f in line.split("|"))
        rows[name] = (float(value), float(tol))
    return rows


def close(got, want, tol):
    return abs(got - want) <= tol * abs(want) + 1e-12


@pytest.fixture(scope="module")
def g():
    return golden()


def test_gemm_flop_count(g):
    want, tol = g["gemm_flops_8192x8192x16384"]
    assert bench.gemm_flops() == 2 * 8192 * 8192 * 16384
    assert close(bench.gemm_flops(), want, tol)


def test_stage_bytes(g):
    want, tol = g["stage_bytes_64x64x32"]
    assert close(bench.tile_stage_bytes(64, 64, 32), want, tol)
    # the GEMM's own stage: a 128 x 64 A slice and a 256 x 64 B slice
    assert bench.tile_stage_bytes(128, 256, 64) == 48 * 1024


def test_roofline_examples(g):
    want, tol = g["roofline_10_flop_per_byte"]
    assert close(bench.roofline(395.0, 1.206, 10.0), want, tol)
    want, tol = g["roofline_500_flop_per_byte"]
    assert close(bench.roofline(395.0, 1.206, 500.0), want, tol)
    assert bench.roofline(1e9, 1.206, 500.0) == pytest.approx(603.0)
    want, tol = g["roofline_ridge"]
    assert close(395.0 / 1.206, want, tol)


def test_decode_estimates(g):
    want, tol = g["decode_weight_io_ms"]
    assert close(54.0 / 1.206, want, tol)          # GB / (TB/s) = ms
    want, tol = g["decode_compute_ms"]
    assert close(54.0 / 395.0, want, tol)          # GFLOP / (TFLOP/s) = ms


def test_gemv_algorithmic_bytes():
    """W once + x once + y once, BF16: the figures the GEMV roofline divides by."""
    assert bench.gemv_bytes(1) == 356_595_712
    assert bench.gemv_bytes(4) == 356_835_328
    assert bench.gemv_bytes(8) == 357_154_816
