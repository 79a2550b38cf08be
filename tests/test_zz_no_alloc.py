"""gemm_f16_colmajor_noalloc: the GEMM entry point for callers that cannot
allocate device memory during a call (a process whose own allocator has
reserved all free HBM, or one held to a memory budget fixed at start-up).
It packs unaligned operands into the library's fixed 96 MiB device array
instead of a freshly allocated workspace.

The GPU test calls it through the C ABI twice in a row, on two problems that
both need packing, and checks each result against the regular
gemm_f16_colmajor with the tolerance the parity tests use (the two share
their kernels, so the results are also expected to be bit-identical).
This file is collected last so that a run stopping at the first failure has
already run every other test.
"""
import ctypes

import numpy as np
import pytest

import oracle
from bf16_gemm_skinny_gb300 import _native as bsk
from bf16_gemm_skinny_gb300 import build as bsk_build
from bf16_gemm_skinny_gb300 import inputs
from helpers import CANARY, FP16_NAN, absmax_f16, check_tolerance, from_dev, poisoned, to_dev


@pytest.fixture(scope="module")
def lib():
    bsk_build.build()
    return bsk.load()


def test_rejects_problems_beyond_the_scratch_limit(lib):
    """M = 8191 forces packing A (8192 x 8192 halves = 128 MiB > 96 MiB): refused
    before any device work, with a message naming the limit."""
    fake = 1 << 40
    rc = lib.gemm_f16_colmajor_noalloc(fake, fake + (1 << 31), fake + (1 << 32), 8191, 8, 8192, None)
    assert rc == 1
    assert "96 MiB" in bsk.last_error()


def _run(fn, A, B, M, N, K, offset):
    import torch

    Ad = to_dev(np.concatenate([np.zeros(offset, np.uint16), A]))[offset:]
    Bd = to_dev(np.concatenate([np.zeros(offset, np.uint16), B]))[offset:]
    buf, _ = poisoned(M * N + offset, FP16_NAN)
    C = buf[offset:offset + M * N]
    fn(Ad, Bd, C, M, N, K)
    torch.cuda.synchronize()
    assert np.all(from_dev(buf[offset + M * N:]) == CANARY)
    assert np.array_equal(from_dev(Ad), A) and np.array_equal(from_dev(Bd), B)
    return from_dev(C)


@pytest.mark.gpu
def test_matches_regular_entry_point_on_two_calls_in_a_row(lib):
    import torch

    torch.cuda.init()
    oracle.build()
    problems = [
        (4095, 4097, 4100, 0),   # ragged: both operands packed (~67 MB of scratch)
        (333, 129, 70, 1),       # unaligned base pointers: both operands packed
    ]
    for M, N, K, offset in problems:
        A, B = inputs.gemm_operands(M, N, K, "normal0.5")
        want = _run(bsk.gemm_f16_colmajor, A, B, M, N, K, offset)
        got = _run(bsk.gemm_f16_colmajor_noalloc, A, B, M, N, K, offset)
        check_tolerance(got, oracle.f16_decode(want), "f16", K, absmax_f16(A), absmax_f16(B),
                        f"noalloc {M}x{N}x{K}")
        assert np.array_equal(got, want)
