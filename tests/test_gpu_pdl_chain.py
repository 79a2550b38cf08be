"""Programmatic dependent launch under real data dependencies.

The kernels start their prologue while the kernel before them in the stream
may still run, and read their inputs only after griddepcontrol.wait.  Here each
launch consumes the output of the launch just before it: a GEMM whose A is the
previous GEMM's C, and a GEMV whose x is the previous GEMV's y.  The second
factor of every link is a signed permutation (one +-1 per column of B, or per
row of W), so each link only reorders and negates the values before it: the
results stay exactly representable and the whole chain must equal the oracle's
bit for bit.  A stale read of an input still being written would show up as a
mismatch.
"""
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
    for k in bsk.OPTIONS:
        bsk.set_option(k, 0)


def signed_permutation(n, seed):
    """One +-1 per row and per column: P[i, perm[i]] = sign[i]."""
    rng = np.random.default_rng(seed)
    return rng.permutation(n), rng.choice([-1.0, 1.0], n)


def dense(perm, sign):
    n = perm.size
    P = np.zeros((n, n))
    P[np.arange(n), perm] = sign
    return P


@pytest.mark.parametrize("pdl", [0, 1])
@pytest.mark.parametrize("M,N,K,links", [(2048, 256, 4096, 6), (512, 512, 512, 12)])
def test_gemm_chain(M, N, K, links, pdl):
    """C_0 = A B_0 (long, so the next link's prologue overlaps it), then
    C_i = C_{i-1} P_i with P_i an N x N signed permutation (K = N for the links)."""
    import torch

    A, B0 = inputs.gemm_operands(M, N, K, "int2", 51, 52)
    Ps = [signed_permutation(N, 60 + i) for i in range(links)]
    # B[k + n*K] = P[k, n]: column-major
    Pbits = [oracle.f16_encode(dense(*P).T.reshape(-1)) for P in Ps]
    bsk.set_option("pdl", 0 if pdl else 1)
    try:
        Cs = [torch.zeros(M * N, dtype=torch.int16, device="cuda") for _ in range(links + 1)]
        Pd = [to_dev(b) for b in Pbits]
        bsk.gemm_f16_colmajor_enqueue(to_dev(A), to_dev(B0), Cs[0], M, N, K)
        for i in range(links):
            bsk.gemm_f16_colmajor_enqueue(Cs[i], Pd[i], Cs[i + 1], M, N, N)
        bsk.stream_check()
        torch.cuda.synchronize()
        got = from_dev(Cs[-1])
    finally:
        bsk.set_option("pdl", 0)
    # C_0 exactly (integer sums), rounded once by the oracle's encoder; each link
    # then moves column k of C to the column n with P[k, n] != 0, times the sign
    # (float64 products and sums of small integers are exact)
    a = oracle.f16_decode(A).reshape(K, M).T
    b = oracle.f16_decode(B0).reshape(N, K).T
    c = oracle.f16_decode(oracle.f16_encode((a @ b).T.reshape(-1))).reshape(N, M)
    for perm, sign in Ps:
        nxt = np.empty_like(c)
        # column perm[k] of the result = sign[k] * column k; the other N - 1 products
        # are zeros, and -0 + +0 = +0, so a zero result is +0 (hence the + 0.0)
        nxt[perm] = c * sign[:, None] + 0.0
        c = nxt
    assert np.array_equal(got, oracle.f16_encode(c.reshape(-1)))
    # the first link through the oracle itself, on sampled columns
    cols = [0, N // 2, N - 1]
    _, c0 = oracle.gemm_f16_colmajor(A, B0, M, N, K, cols=cols)
    want0 = oracle.f16_encode((a @ b)[:, cols].T.reshape(-1))
    assert np.array_equal(c0, want0)


@pytest.mark.parametrize("pdl", [0, 1])
@pytest.mark.parametrize("n", [1, 8])
def test_gemv_chain(n, pdl):
    """y_0 = x W_0^T (a 4096 x 5120 weight stream, so the next link's prologue
    overlaps it), then y_i = y_{i-1} P_i^T with P_i a signed permutation."""
    import torch

    M0, K = 4096, 5120
    links = 8
    W0, x = inputs.linear_operands(M0, K, n, "int2", "int2", seed_x=71, seed_w=72)
    Ps = [signed_permutation(M0, 80 + i) for i in range(links)]
    bsk.set_option("pdl", 0 if pdl else 1)
    try:
        ys = [torch.zeros(n * M0, dtype=torch.int16, device="cuda") for _ in range(links + 1)]
        Pd = [to_dev(oracle.bf16_encode(dense(*P).reshape(-1))) for P in Ps]   # W[j, k] = P[j, k]
        bsk.gemv_bf16_enqueue(to_dev(W0), to_dev(x), ys[0], M0, K, n)
        for i in range(links):
            bsk.gemv_bf16_enqueue(Pd[i], ys[i], ys[i + 1], M0, M0, n)
        bsk.stream_check()
        torch.cuda.synchronize()
        got = from_dev(ys[-1])
    finally:
        bsk.set_option("pdl", 0)
    _, y = oracle.linear_bf16(W0, x, M0, K, n)
    y = oracle.bf16_decode(y.reshape(-1)).reshape(n, M0)
    for perm, sign in Ps:
        # y_new[t, j] = sum_k y[t, k] P[j, k] = sign[j] * y[t, perm[j]] (+0 for a zero result)
        y = y[:, perm] * sign[None, :] + 0.0
    assert np.array_equal(got, oracle.bf16_encode(y.reshape(-1)))
