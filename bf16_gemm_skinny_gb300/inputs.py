"""Seeded synthetic inputs for the GEMM and linear-layer workloads.

This module is shared by the tests, the smoke check, the benchmark and the
oracle's callers.  It holds none of the method's arithmetic: it draws numbers
with numpy's PCG64 generator and turns them into 16-bit patterns or FP8 codes
with library casts (numpy for FP16, torch for BF16 and FP8).  The same bit
patterns then feed both the CUDA path and the oracle.

Recipe (the pages name the shapes but give no seeds or value distributions):

* operand "A" / activations "x" use ``seed_a`` (default 1), operand "B" /
  weights "W" use ``seed_b`` (default 2); integer variants use 11 / 12;
* ``uniform``: ``rng.uniform(-1, 1)``; ``normal0.5``: ``0.5*rng.standard_normal()``;
  ``normal0.02``: ``0.02*rng.standard_normal()``; ``normal1``:
  ``rng.standard_normal()``; ``int2``: ``rng.integers(-2, 3)`` (entries in
  {-2,...,2}, every partial sum of a product is an integer);
* values are drawn in float64, in fixed chunks, then cast to FP16 (numpy) or
  to float32 and then BF16, FP8 E4M3 or FP8 E5M2 (torch's float8_e4m3fn /
  float8_e5m2 casts).
"""
from __future__ import annotations

import numpy as np

_CHUNK = 1 << 22

DISTS = ("uniform", "normal0.5", "normal0.02", "normal1", "int2")


def draw(dist: str, size: int, seed: int) -> np.ndarray:
    """``size`` float64 values from distribution ``dist`` with PCG64(``seed``)."""
    if dist not in DISTS:
        raise ValueError(f"unknown distribution {dist!r}")
    rng = np.random.Generator(np.random.PCG64(seed))
    out = np.empty(size, np.float64)
    for lo in range(0, size, _CHUNK):
        hi = min(size, lo + _CHUNK)
        m = hi - lo
        if dist == "uniform":
            out[lo:hi] = rng.uniform(-1.0, 1.0, m)
        elif dist == "normal0.5":
            out[lo:hi] = 0.5 * rng.standard_normal(m)
        elif dist == "normal0.02":
            out[lo:hi] = 0.02 * rng.standard_normal(m)
        elif dist == "normal1":
            out[lo:hi] = rng.standard_normal(m)
        else:
            out[lo:hi] = rng.integers(-2, 3, m)
    return out


def to_f16_bits(values: np.ndarray) -> np.ndarray:
    """FP16 bit patterns of ``values`` (numpy's float16 cast)."""
    out = np.empty(values.shape, np.uint16)
    flat_in = values.reshape(-1)
    flat_out = out.reshape(-1)
    for lo in range(0, flat_in.size, _CHUNK):
        hi = min(flat_in.size, lo + _CHUNK)
        flat_out[lo:hi] = flat_in[lo:hi].astype(np.float16).view(np.uint16)
    return out


def to_bf16_bits(values: np.ndarray) -> np.ndarray:
    """BF16 bit patterns of ``values`` (cast to float32, then torch's bfloat16 cast)."""
    import torch

    out = np.empty(values.shape, np.uint16)
    flat_in = values.reshape(-1)
    flat_out = out.reshape(-1)
    for lo in range(0, flat_in.size, _CHUNK):
        hi = min(flat_in.size, lo + _CHUNK)
        t = torch.from_numpy(flat_in[lo:hi].astype(np.float32)).to(torch.bfloat16)
        flat_out[lo:hi] = t.view(torch.int16).numpy().view(np.uint16)
    return out


def to_fp8_bits(values: np.ndarray, fmt: str) -> np.ndarray:
    """FP8 codes (uint8) of ``values``: cast to float32, then torch's float8 cast
    (``fmt`` 'e4m3' -> float8_e4m3fn, 'e5m2' -> float8_e5m2)."""
    import torch

    dtype = {"e4m3": torch.float8_e4m3fn, "e5m2": torch.float8_e5m2}[fmt]
    out = np.empty(values.shape, np.uint8)
    flat_in = values.reshape(-1)
    flat_out = out.reshape(-1)
    for lo in range(0, flat_in.size, _CHUNK):
        hi = min(flat_in.size, lo + _CHUNK)
        t = torch.from_numpy(flat_in[lo:hi].astype(np.float32)).to(dtype)
        flat_out[lo:hi] = t.view(torch.uint8).numpy()
    return out


def fp8_operands(M: int, N: int, K: int, dist: str, fmt: str, seed_a: int = 1, seed_b: int = 2):
    """FP8 operands of the K-major FP8 GEMM as flat uint8 arrays.

    Returns ``(A, B)`` with ``A[k + m*K]`` (M*K entries) and ``B[k + n*K]``
    (K*N entries).
    """
    A = to_fp8_bits(draw(dist, M * K, seed_a), fmt)
    B = to_fp8_bits(draw(dist, K * N, seed_b), fmt)
    return A, B


def gemm_operands(M: int, N: int, K: int, dist: str, seed_a: int = 1, seed_b: int = 2):
    """FP16 operands of the column-major GEMM as flat uint16 arrays.

    Returns ``(A, B)`` with ``A[m + k*M]`` (M*K entries) and ``B[k + n*K]``
    (K*N entries).
    """
    A = to_f16_bits(draw(dist, M * K, seed_a))
    B = to_f16_bits(draw(dist, K * N, seed_b))
    return A, B


def linear_operands(M: int, K: int, n: int, w_dist: str, x_dist: str,
                    seed_x: int = 1, seed_w: int = 2):
    """BF16 operands of y = x W^T as flat uint16 arrays: ``(W[M*K], x[n*K])`` row-major."""
    W = to_bf16_bits(draw(w_dist, M * K, seed_w))
    x = to_bf16_bits(draw(x_dist, n * K, seed_x))
    return W, x


# The five workloads: name -> description used by tests, smoke and bench.
WORKLOADS = {
    "gemm_256": dict(kind="gemm", M=256, N=256, K=256, dist="uniform"),
    "gemm_ragged": dict(kind="gemm", M=4095, N=4097, K=4100, dist="normal0.5"),
    "gemm_8192x8192x16384": dict(kind="gemm", M=8192, N=8192, K=16384, dist="uniform"),
    "gemv_34816x5120": dict(kind="linear", M=34816, K=5120, n=(1, 4, 8),
                            w_dist="normal0.02", x_dist="normal1"),
    "prefill_4096x34816x5120": dict(kind="linear", M=34816, K=5120, n=4096,
                                    w_dist="normal0.02", x_dist="normal1"),
}
