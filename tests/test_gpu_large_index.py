"""Sizes where element or byte offsets pass 2^31: every kernel's address
arithmetic must be 64-bit where it needs to be.  Each case keeps the host side
small -- operands are either small themselves or built on the device from a
small seeded block -- and the oracle checks sampled outputs on the same bits.
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
    torch.cuda.empty_cache()


@pytest.fixture(autouse=True)
def free_memory():
    import torch

    yield
    torch.cuda.empty_cache()


def test_gemm_output_past_2_31_elements():
    """C is 65536 x 33000 (2.16e9 elements, 4.3 GB): the last columns sit past 2^31."""
    import torch

    M, N, K = 65536, 33000, 64
    A, B = inputs.gemm_operands(M, N, K, "int2", 11, 12)
    C = torch.empty(M * N, dtype=torch.int16, device="cuda")
    bsk.gemm_f16_colmajor(to_dev(A), to_dev(B), C, M, N, K)
    cols = [0, 32767, N - 2, N - 1]
    _, want = oracle.gemm_f16_colmajor(A, B, M, N, K, cols=cols)
    got = np.concatenate([from_dev(C[n * M:(n + 1) * M]) for n in cols])
    assert np.array_equal(got, want)
    del C


@pytest.mark.parametrize("n,kernel", [(1, 0), (4, 2), (8, 0)])
def test_gemv_weights_past_2_31_elements(n, kernel):
    """W has 524291 rows of 4104 (2.15e9 elements, 4.3 GB), built on the device by
    repeating a seeded block of 4099 rows; rows past 523265 start beyond 2^31.
    Kernel 0 = default (CUDA-core for n = 1, tensor-core for n = 8), 2 = pipelined."""
    import torch

    M, K, P = 524291, 4104, 4099
    block, x = inputs.linear_operands(P, K, n, "int2", "int2", seed_x=11, seed_w=12)
    blk = to_dev(block).view(P, K)
    reps = -(-M // P)
    W = blk.repeat(reps, 1)[:M].contiguous().view(-1)
    y = torch.empty(n * M, dtype=torch.int16, device="cuda")
    bsk.set_option("gemv_kernel", kernel)
    try:
        bsk.gemv_bf16(W, to_dev(x), y, M, K, n)
    finally:
        bsk.set_option("gemv_kernel", 0)
    js = np.array([0, 1, 523264, 523265, 523266, M - 2, M - 1])
    rows = block.reshape(P, K)[js % P].reshape(-1)
    _, want = oracle.linear_bf16(rows, x, len(js), K, n)
    got = from_dev(y).reshape(n, M)[:, js]
    assert np.array_equal(got, want.reshape(n, len(js)))
    del W, y


def test_fp8_fp32_output_past_2_31_bytes():
    """FP32 C of 65536 x 16400 (4.3 GB): byte offsets past 2^32 in the stores."""
    import torch

    M, N, K = 65536, 16400, 128
    A, B = inputs.fp8_operands(M, N, K, "int2", "e4m3", 11, 12)
    C = torch.empty(M * N, dtype=torch.int32, device="cuda")
    bsk.gemm_fp8(bsk.FP8_E4M3, torch.from_numpy(A).cuda(), K, torch.from_numpy(B).cuda(), K, C, M, bsk.OUT_F32,
                 M, N, K, 1.0)
    cols = [0, N // 2, N - 1]
    _, want = oracle.gemm_fp8(A, B, M, N, K, K, K, "e4m3", 1.0, "f32", cols=cols)
    got = np.concatenate([C[n * M:(n + 1) * M].cpu().numpy().view(np.uint32) for n in cols])
    assert np.array_equal(got, want)
    del C


def test_attention_cache_past_2_31_elements():
    """A paged cache of 2700 blocks x 784 tokens x 4 KV heads x 256 (2.17e9 elements
    per K and V, 8.7 GB together); the sequence's pages are the last physical
    blocks, so every row it reads starts beyond 2^31.  The oracle sees the same
    pages compacted to blocks 0..41 (same values, same order)."""
    import math

    import torch

    nqh, nkv, hd, bs, L = 16, 4, 256, 784, 32768
    nb_seq = -(-L // bs)
    num_blocks = 2700
    per_block = bs * nkv * hd
    k_small = inputs.to_bf16_bits(inputs.draw("normal1", nb_seq * per_block, 501))
    v_small = inputs.to_bf16_bits(inputs.draw("normal1", nb_seq * per_block, 502))
    q = inputs.to_bf16_bits(inputs.draw("normal1", nqh * hd, 503))
    phys = np.arange(num_blocks - nb_seq, num_blocks, dtype=np.int32)[::-1].copy()   # reversed, at the top
    kd = torch.zeros(num_blocks * per_block, dtype=torch.int16, device="cuda")
    vd = torch.zeros(num_blocks * per_block, dtype=torch.int16, device="cuda")
    ks, vs = to_dev(k_small).view(nb_seq, per_block), to_dev(v_small).view(nb_seq, per_block)
    for i, b in enumerate(phys):
        kd[int(b) * per_block:(int(b) + 1) * per_block] = ks[i]
        vd[int(b) * per_block:(int(b) + 1) * per_block] = vs[i]
    bt = torch.from_numpy(phys).cuda()
    sl = torch.tensor([L], dtype=torch.int32, device="cuda")
    out = torch.empty(nqh * hd, dtype=torch.int16, device="cuda")
    scale = 1.0 / math.sqrt(hd)
    bsk.decode_attention_bf16(to_dev(q), kd, vd, bt, sl, out, 1, nqh, nkv, hd, bs, nb_seq, num_blocks, L, scale, 0)
    ref, _ = oracle.decode_attention_bf16(q, k_small, v_small, np.arange(nb_seq, dtype=np.int32).reshape(1, -1),
                                          np.array([L], np.int32), nqh, nkv, hd, bs, scale)
    got = oracle.bf16_decode(from_dev(out))
    # same derived bound as the attention parity tests: weights, then one BF16 rounding
    err = np.abs(got - ref.reshape(-1))
    vmax = float(np.max(np.abs(oracle.bf16_decode(v_small))))
    sum_abs = hd * float(np.max(np.abs(oracle.bf16_decode(q)))) * float(np.max(np.abs(oracle.bf16_decode(k_small)))) \
        * scale
    eps_w = hd * 2.0 ** -23 * sum_abs + 2.0 ** -21
    bound = (2 * eps_w + L * 2.0 ** -24) * vmax + 2.0 ** -8 * np.maximum(np.abs(got), np.abs(ref.reshape(-1)))
    assert np.all(err <= bound), f"max err {err.max():.3g}"
    del kd, vd
