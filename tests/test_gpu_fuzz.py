"""Seeded fuzz through the default plans: hundreds of random problems (the
FP16 column-major GEMM, gemm_f16 in every storage form with each bias mode,
the FP8 GEMM in both formats and outputs, and gemv_bf16 for 1..160 tokens),
integer-valued inputs, every element compared with the oracle bit for bit.  Shapes are drawn log-uniform
(M, N up to 8192, K up to 16384, half of them rounded to multiples of 8), so
most are small and odd: the unaligned pack, ragged tails, every tile width,
split-K over clusters and the CTA-pair kernel all come up."""
import numpy as np
import pytest

import oracle
from bf16_gemm_skinny_gb300 import _native as bsk
from bf16_gemm_skinny_gb300 import build as bsk_build
from bf16_gemm_skinny_gb300 import inputs

pytestmark = pytest.mark.gpu

CASES = 400
MAX_WORK = 3e8   # multiply-adds per problem


@pytest.fixture(scope="module", autouse=True)
def lib():
    import torch

    bsk_build.build()
    oracle.build()
    torch.cuda.init()
    yield bsk.load()
    for k in bsk.OPTIONS:
        bsk.set_option(k, 0)


def _shape(rng):
    while True:
        M, N = (int(np.exp(rng.uniform(0, np.log(8192)))) for _ in range(2))
        K = int(np.exp(rng.uniform(0, np.log(16384))))
        if rng.random() < 0.5:
            M, N, K = (max(8, (v + 7) // 8 * 8) for v in (M, N, K))
        if M * N * K <= MAX_WORK:
            return M, N, K


def _colmajor(rng, M, N, K):
    import torch

    A, B = inputs.gemm_operands(M, N, K, "int2", int(rng.integers(1, 1000)), int(rng.integers(1, 1000)))
    C = torch.empty(M * N, dtype=torch.int16, device="cuda")
    bsk.gemm_f16_colmajor(torch.from_numpy(A.view(np.int16)).cuda(), torch.from_numpy(B.view(np.int16)).cuda(),
                          C, M, N, K)
    _, want = oracle.gemm_f16_colmajor(A, B, M, N, K)
    return np.array_equal(C.cpu().numpy().view(np.uint16), want)


def _fp8(rng, M, N, K):
    import torch

    fmt = ("e4m3", "e5m2")[int(rng.integers(0, 2))]
    out = int(rng.integers(0, 2))   # 0: FP32, 1: BF16
    A, B = inputs.fp8_operands(M, N, K, "int2", fmt, int(rng.integers(1, 1000)), int(rng.integers(1, 1000)))
    C = torch.empty(M * N, dtype=torch.int32 if out == 0 else torch.int16, device="cuda")
    bsk.gemm_fp8(0 if fmt == "e4m3" else 1, torch.from_numpy(A).cuda(), K, torch.from_numpy(B).cuda(), K, C, M, out,
                 M, N, K, 1.0)
    _, want = oracle.gemm_fp8(A, B, M, N, K, K, K, fmt, 1.0, "f32" if out == 0 else "bf16")
    got = C.cpu().numpy().view(np.uint32 if out == 0 else np.uint16)
    return np.array_equal(got, np.asarray(want).reshape(-1))


def _layout(rng, M, N, K):
    import torch

    order, ta, tb = (int(v) for v in rng.integers(0, 2, 3))
    mode = int(rng.integers(0, 3))
    A, B = inputs.gemm_operands(M, N, K, "int2", int(rng.integers(1, 1000)), int(rng.integers(1, 1000)))
    A2, B2 = A.reshape(K, M).T, B.reshape(N, K).T       # logical M x K and K x N
    sa, sb = (A2.T if ta else A2), (B2.T if tb else B2)

    def stored(mat):
        return np.ascontiguousarray(mat if order else mat.T).reshape(-1), max(1, mat.shape[1] if order else mat.shape[0])

    Af, lda = stored(sa)
    Bf, ldb = stored(sb)
    bias = None
    if mode:
        bias = oracle.f16_encode(rng.integers(-40, 41, max(M, N)).astype(np.float64))[:M if mode == 1 else N]
    C = torch.empty(M * N, dtype=torch.int16, device="cuda")
    bsk.gemm_f16(order, ta, tb, torch.from_numpy(Af.view(np.int16)).cuda(), lda,
                 torch.from_numpy(Bf.view(np.int16)).cuda(), ldb, C, N if order else M, M, N, K,
                 None if bias is None else torch.from_numpy(bias.view(np.int16)).cuda(), mode)
    _, want = oracle.gemm_f16_general(Af, Bf, M, N, K, lda, ldb, ta, tb, order, bias=bias, bias_mode=mode)
    got = C.cpu().numpy().view(np.uint16)
    got = got.reshape(M, N) if order else got.reshape(N, M).T
    return np.array_equal(got, np.asarray(want).reshape(N, M).T)


def _gemv(rng):
    """y = x W^T through gemv_bf16 (CUDA cores for n <= 3, the tensor-core GEMM
    beyond), M up to 40000, K up to 8192, n up to 160 tokens."""
    import torch

    while True:
        M = int(np.exp(rng.uniform(0, np.log(40000))))
        K = int(np.exp(rng.uniform(0, np.log(8192))))
        n = int(np.exp(rng.uniform(0, np.log(160))))
        if M * K * n <= MAX_WORK:
            break
    W, x = inputs.linear_operands(M, K, n, "int2", "int2", int(rng.integers(1, 1000)), int(rng.integers(1, 1000)))
    y = torch.empty(n * M, dtype=torch.int16, device="cuda")
    bsk.gemv_bf16(torch.from_numpy(W.view(np.int16)).cuda(), torch.from_numpy(x.view(np.int16)).cuda(), y, M, K, n)
    _, want = oracle.linear_bf16(W, x, M, K, n)
    return np.array_equal(y.cpu().numpy().view(np.uint16), want.reshape(-1)), (M, K, n)


@pytest.mark.parametrize("seed", [303])
def test_fuzz_gemv(seed):
    rng = np.random.default_rng(seed)
    fails = []
    for _ in range(150):
        ok, shape = _gemv(rng)
        if not ok:
            fails.append(shape)
    bsk.stream_check()
    assert not fails, f"{len(fails)} problems differ from the oracle, e.g. {fails[:5]}"


@pytest.mark.parametrize("seed", [101, 202])
def test_fuzz_default_plans(seed):
    rng = np.random.default_rng(seed)
    fails = []
    for _ in range(CASES // 2):
        kind = int(rng.integers(0, 3))
        M, N, K = _shape(rng)
        ok = (_colmajor, _fp8, _layout)[kind](rng, M, N, K)
        if not ok:
            fails.append((("colmajor", "fp8", "layout")[kind], M, N, K))
    bsk.stream_check()
    assert not fails, f"{len(fails)} problems differ from the oracle, e.g. {fails[:5]}"
