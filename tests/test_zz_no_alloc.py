"""gemm_f16_colmajor_noalloc: the GEMM entry point for callers that cannot
allocate device memory during a call (a process whose own allocator has
reserved all free HBM, or one held to a memory budget fixed at start-up).
Where the regular entry point allocates a workspace (to pack unaligned
operands, or for stream-K partials), it uses the library's fixed 96 MiB
device array instead.

The GPU tests call it through the C ABI:
  * twice in a row on each of several problems -- both operands packed (the
    4095 x 4097 x 4100 workload), unaligned base pointers, 16-byte-aligned
    operands that need no scratch, a skinny shape, stream-K partials in the
    array, and K = 0 -- and check
    every result against the oracle (integer-valued inputs bit for bit,
    random ones within the tolerance the parity tests use) and against the
    regular gemm_f16_colmajor (the same planner and kernels: bit-identical);
  * after a warm-up call of each kind (the first call on a device does the
    set-up, which maps the array and the kernels' code), again on every kind
    of problem, checking that device free memory, torch's allocator
    statistics and the high-water marks of the device's default memory pool
    do not move.
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


def _device_operands(A, B, M, N, offset):
    """A, B on the device `offset` elements past a 16-byte boundary, and C (poisoned,
    with guard words after it) at the same offset."""
    Ad = to_dev(np.concatenate([np.zeros(offset, np.uint16), A]))[offset:]
    Bd = to_dev(np.concatenate([np.zeros(offset, np.uint16), B]))[offset:]
    buf, _ = poisoned(M * N + offset, FP16_NAN)
    return Ad, Bd, buf


def _call(fn, Ad, Bd, buf, M, N, K, offset):
    import torch

    buf[:M * N + offset] = FP16_NAN
    C = buf[offset:offset + M * N]
    fn(Ad, Bd, C, M, N, K)
    torch.cuda.synchronize()
    assert np.all(from_dev(buf[offset + M * N:]) == CANARY), "guard words after C were written"
    return from_dev(C)


# (M, N, K, offset, distribution): what each exercises
PROBLEMS = [
    (4095, 4097, 4100, 0, "normal0.5"),   # ragged: both operands packed (~67 MB of scratch)
    (4095, 4097, 4100, 0, "int2"),
    (333, 129, 70, 1, "normal0.5"),       # unaligned base pointers: both operands packed
    (333, 129, 70, 1, "int2"),
    (256, 256, 256, 0, "uniform"),        # 16-byte aligned: no scratch at all
    (256, 256, 256, 0, "int2"),
    (1000, 24, 2056, 3, "int2"),          # skinny, unaligned
]


@pytest.mark.gpu
@pytest.mark.parametrize("M,N,K,offset,dist", PROBLEMS)
def test_matches_oracle_and_regular_entry_point_on_two_calls_in_a_row(lib, M, N, K, offset, dist):
    import torch

    torch.cuda.init()
    oracle.build()
    seeds = (11, 12) if dist == "int2" else (1, 2)
    A, B = inputs.gemm_operands(M, N, K, dist, *seeds)
    Ad, Bd, buf = _device_operands(A, B, M, N, offset)
    regular = _call(bsk.gemm_f16_colmajor, Ad, Bd, buf, M, N, K, offset)
    # columns checked against the oracle: all for the small problems, a spread
    # including the ragged last one for the large
    cols = np.arange(N) if M * N <= 1 << 20 else np.unique(np.r_[np.arange(0, N, 97), N - 1])
    ref, want_bits = oracle.gemm_f16_colmajor(A, B, M, N, K, cols=cols)
    for call in range(2):
        got = _call(bsk.gemm_f16_colmajor_noalloc, Ad, Bd, buf, M, N, K, offset)
        sub = got.reshape(N, M)[cols].reshape(-1)
        if dist == "int2":
            assert np.array_equal(sub, want_bits), f"call {call}: integer inputs differ from the oracle"
        else:
            check_tolerance(sub, ref, "f16", K, absmax_f16(A), absmax_f16(B), f"noalloc {M}x{N}x{K} call {call}")
        # same planner, same kernels: the regular entry point's bits (so within its tolerance too)
        assert np.array_equal(got, regular), f"call {call}: differs from gemm_f16_colmajor"
    assert np.array_equal(from_dev(Ad), A) and np.array_equal(from_dev(Bd), B), "an input was modified"


@pytest.mark.gpu
@pytest.mark.parametrize("M,N,K,offset", [(512, 256, 8192, 0), (1000, 24, 2056, 3)])
def test_stream_k_partials_in_the_fixed_array(lib, M, N, K, offset):
    """Stream-K forced: its FP32 partials and flags come from the fixed array (after
    the packed operands, for the unaligned problem).  Integer inputs match the
    oracle bit for bit and the regular entry point under the same option, and
    calls after the first leave device free memory unchanged."""
    import torch

    torch.cuda.init()
    oracle.build()
    A, B = inputs.gemm_operands(M, N, K, "int2", 11, 12)
    Ad, Bd, buf = _device_operands(A, B, M, N, offset)
    _, want = oracle.gemm_f16_colmajor(A, B, M, N, K)
    bsk.set_option("stream_k", 2)
    try:
        regular = _call(bsk.gemm_f16_colmajor, Ad, Bd, buf, M, N, K, offset)
        assert np.array_equal(regular, want), "regular entry point, stream-K"
        _call(bsk.gemm_f16_colmajor_noalloc, Ad, Bd, buf, M, N, K, offset)   # set-up call
        DefaultPool(torch.cuda.current_device()).reset_marks()   # returns the regular call's workspace
        torch.cuda.synchronize()
        free0, _ = torch.cuda.mem_get_info()
        for call in range(2):
            got = _call(bsk.gemm_f16_colmajor_noalloc, Ad, Bd, buf, M, N, K, offset)
            assert torch.cuda.mem_get_info()[0] == free0, f"call {call}: device free memory moved"
            assert np.array_equal(got, want), f"call {call}: differs from the oracle"
    finally:
        bsk.set_option("stream_k", 0)


@pytest.mark.gpu
def test_k_zero_writes_positive_zeros_twice(lib):
    import torch

    torch.cuda.init()
    M, N = 300, 77
    buf, _ = poisoned(M * N, FP16_NAN)
    for _ in range(2):
        buf[:M * N] = FP16_NAN
        bsk.gemm_f16_colmajor_noalloc(None, None, buf[:M * N], M, N, 0)
        torch.cuda.synchronize()
        host = from_dev(buf)
        assert np.all(host[:M * N] == 0)           # +0.0 in every element: the empty sum
        assert np.all(host[M * N:] == CANARY)


def _cudart():
    """The CUDA runtime library, for the default memory pool's statistics (None if
    it cannot be loaded here)."""
    for name in ("libcudart.so.13", "libcudart.so", "/usr/local/cuda/lib64/libcudart.so"):
        try:
            return ctypes.CDLL(name)
        except OSError:
            continue
    return None


class DefaultPool:
    """High-water marks of the current device's default (stream-ordered) memory pool."""
    RESERVED_HIGH, USED_HIGH = 6, 8   # cudaMemPoolAttrReservedMemHigh, cudaMemPoolAttrUsedMemHigh

    def __init__(self, device: int):
        self.rt = _cudart()
        self.pool = ctypes.c_void_p()
        if self.rt is not None and self.rt.cudaDeviceGetDefaultMemPool(ctypes.byref(self.pool), device) != 0:
            self.rt = None

    def reset_marks(self):
        if self.rt is None:
            return
        zero = ctypes.c_uint64(0)
        for attr in (self.RESERVED_HIGH, self.USED_HIGH):
            assert self.rt.cudaMemPoolSetAttribute(self.pool, attr, ctypes.byref(zero)) == 0
        self.rt.cudaMemPoolTrimTo(self.pool, ctypes.c_size_t(0))

    def marks(self):
        if self.rt is None:
            return None
        out = []
        for attr in (self.RESERVED_HIGH, self.USED_HIGH):
            v = ctypes.c_uint64(0)
            assert self.rt.cudaMemPoolGetAttribute(self.pool, attr, ctypes.byref(v)) == 0
            out.append(v.value)
        return tuple(out)


@pytest.mark.gpu
def test_allocates_nothing_after_set_up(lib):
    import torch

    torch.cuda.init()
    dev = torch.cuda.current_device()
    kinds = []
    for M, N, K, offset, dist in [(4095, 4097, 4100, 0, "normal0.5"), (333, 129, 70, 1, "int2"),
                                  (256, 256, 256, 0, "uniform"), (1000, 24, 2056, 3, "int2")]:
        A, B = inputs.gemm_operands(M, N, K, dist)
        kinds.append((M, N, K, offset) + _device_operands(A, B, M, N, offset))
    kz, _ = poisoned(300 * 77, FP16_NAN)
    # warm-up: the first call of each kind on this device (set-up, kernel code)
    for M, N, K, offset, Ad, Bd, buf in kinds:
        _call(bsk.gemm_f16_colmajor_noalloc, Ad, Bd, buf, M, N, K, offset)
    bsk.gemm_f16_colmajor_noalloc(None, None, kz[:300 * 77], 300, 77, 0)
    torch.cuda.synchronize()

    pool = DefaultPool(dev)
    pool.reset_marks()
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info(dev)
    torch0 = (torch.cuda.memory_allocated(dev), torch.cuda.memory_reserved(dev))
    marks0 = pool.marks()
    for rep in range(2):
        for M, N, K, offset, Ad, Bd, buf in kinds:
            C = buf[offset:offset + M * N]
            bsk.gemm_f16_colmajor_noalloc(Ad, Bd, C, M, N, K)
            free1, _ = torch.cuda.mem_get_info(dev)
            assert free1 == free0, f"device free memory moved by {free0 - free1} bytes in a {M}x{N}x{K} call"
            assert pool.marks() == marks0, f"the default memory pool was used by a {M}x{N}x{K} call"
        bsk.gemm_f16_colmajor_noalloc(None, None, kz[:300 * 77], 300, 77, 0)
        assert torch.cuda.mem_get_info(dev)[0] == free0
    assert (torch.cuda.memory_allocated(dev), torch.cuda.memory_reserved(dev)) == torch0
