"""gemm_f16_colmajor_host / gemv_bf16_host: the same results as the device
entry points (bit for bit: the same kernels), on shapes that take several
copy blocks, from pinned and from pageable host buffers, and after work that
writes the host inputs on the same stream just before the call."""
import numpy as np
import pytest

import oracle
from bf16_gemm_skinny_gb300 import _native as bsk
from bf16_gemm_skinny_gb300 import build as bsk_build
from bf16_gemm_skinny_gb300 import inputs
from helpers import from_dev, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    import torch

    bsk_build.build()
    oracle.build()
    torch.cuda.init()
    yield bsk.load()


def host_buffer(bits, pinned):
    import torch

    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.pin_memory() if pinned else t.clone()


@pytest.mark.parametrize("pinned", [True, False])
@pytest.mark.parametrize("M,N,K", [(1000, 777, 1030), (512, 10000, 4096), (4095, 4097, 4100)])
def test_gemm_host_matches_device_call(M, N, K, pinned):
    """(512, 10000, 4096): B is 78 MB, two column blocks; ragged shapes take the pack path."""
    import torch

    A, B = inputs.gemm_operands(M, N, K, "int2", 31, 32)
    Ah, Bh = host_buffer(A, pinned), host_buffer(B, pinned)
    Ch = host_buffer(np.full(M * N, 0x7E00, np.uint16), pinned)
    bsk.gemm_f16_colmajor_host(Ah, Bh, Ch, M, N, K)
    got = Ch.numpy().view(np.uint16)
    Cd = torch.empty(M * N, dtype=torch.int16, device="cuda")
    bsk.gemm_f16_colmajor(to_dev(A), to_dev(B), Cd, M, N, K)
    assert np.array_equal(got, from_dev(Cd))
    cols = sorted({0, N // 3, N // 2 + 1, N - 1})
    _, want = oracle.gemm_f16_colmajor(A, B, M, N, K, cols=cols)
    assert np.array_equal(np.concatenate([got[n * M:(n + 1) * M] for n in cols]), want)
    assert np.array_equal(Ah.numpy().view(np.uint16), A) and np.array_equal(Bh.numpy().view(np.uint16), B)


@pytest.mark.parametrize("pinned", [True, False])
@pytest.mark.parametrize("n", [1, 4, 8, 16])
def test_gemv_host_matches_device_call(n, pinned):
    """The decode shape 34816 x 5120 (356 MB of weights, six row blocks)."""
    import torch

    M, K = 34816, 5120
    W, x = inputs.linear_operands(M, K, n, "int2", "int2", seed_x=33, seed_w=34)
    Wh, xh = host_buffer(W, pinned), host_buffer(x, pinned)
    yh = host_buffer(np.full(n * M, 0x7FC0, np.uint16), pinned)
    bsk.gemv_bf16_host(Wh, xh, yh, M, K, n)
    got = yh.numpy().view(np.uint16)
    yd = torch.empty(n * M, dtype=torch.int16, device="cuda")
    bsk.gemv_bf16(to_dev(W), to_dev(x), yd, M, K, n)
    assert np.array_equal(got, from_dev(yd))
    rows = np.array([0, 5000, 17407, 17408, 30000, M - 1])
    _, want = oracle.linear_bf16(W.reshape(M, K)[rows].reshape(-1), x, rows.size, K, n)
    assert np.array_equal(got.reshape(n, M)[:, rows], want.reshape(n, rows.size))


def test_host_call_follows_earlier_work_on_its_stream():
    """A device-to-host copy into A enqueued on the stream just before the call:
    the call's copies in must see its result, not the old contents."""
    import torch

    M, N, K = 1024, 768, 512
    A, B = inputs.gemm_operands(M, N, K, "int2", 35, 36)
    A_old, _ = inputs.gemm_operands(M, N, K, "int2", 37, 38)
    Ah = host_buffer(A_old, True)
    Bh = host_buffer(B, True)
    Ch = host_buffer(np.zeros(M * N, np.uint16), True)
    Ad = to_dev(A)
    big = torch.ones(64 << 20, dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    big.mul_(2.0).add_(1.0)              # keep the stream busy so the copy below is still pending
    Ah.copy_(Ad, non_blocking=True)      # on the current stream
    bsk.gemm_f16_colmajor_host(Ah, Bh, Ch, M, N, K)
    _, want = oracle.gemm_f16_colmajor(A, B, M, N, K)
    assert np.array_equal(Ch.numpy().view(np.uint16), want)


def test_host_calls_empty_and_zero_k():
    C = np.full(6 * 5, 0x5A5A, np.uint16)
    A = np.ones(6 * 0, np.uint16)
    bsk.gemm_f16_colmajor_host(A, A, C, 6, 5, 0)
    assert np.all(C == 0)
    y = np.full(3 * 7, 0x5A5A, np.uint16)
    bsk.gemv_bf16_host(A, A, y, 7, 0, 3)
    assert np.all(y == 0)
    bsk.gemm_f16_colmajor_host(None, None, None, 0, 5, 7)
