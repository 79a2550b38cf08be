"""Shared helpers for the parity tests: device transfer, output poisoning and
the tolerance of the half-precision GEMM / linear layer.

Tolerance (random inputs).  The bound on the FP32-accumulated value is
    |acc - exact| <= 4e-3 * sqrt(K/256) * max|a| * max|b|
(max|a|, max|b| are the realised maxima of the call's inputs).  The output is
that value rounded once to 16 bits, so each output element must satisfy
    |out - exact| <= 4e-3 * sqrt(K/256) * max|a| * max|b| + ulp_out(max(|out|, |exact|)) / 2
and, over the whole output, the relative Frobenius error against the
correctly rounded exact result must be <= 1e-3.  Integer-valued inputs
(entries in {-2..2}) keep every partial sum an exact integer below 2^24, so
there the output must equal the oracle's bit for bit.
"""
from __future__ import annotations

import numpy as np

import oracle

FP16_NAN = 0x7E00
BF16_NAN = 0x7FC0
CANARY = 0x5A5A


def to_dev(bits: np.ndarray, device="cuda"):
    import torch

    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device)


def poisoned(n: int, nan_bits: int, guard: int = 64, device="cuda"):
    """Device buffer of n + guard int16 values: NaN pattern then canary words.

    Returns (full_buffer, view_of_first_n)."""
    import torch

    buf = torch.full((n + guard,), nan_bits, dtype=torch.int16, device=device)
    buf[n:] = CANARY
    return buf, buf[:n]


def from_dev(t) -> np.ndarray:
    return t.detach().cpu().numpy().view(np.uint16)


def ulp(values: np.ndarray, fmt: str) -> np.ndarray:
    """Spacing of representable values at |values| in FP16 or BF16 (subnormal floor included)."""
    frac, emin = (10, -14) if fmt == "f16" else (7, -126)
    a = np.abs(values)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, emin)
    return np.ldexp(1.0, (e - frac).astype(np.int64))


def decode(bits: np.ndarray, fmt: str) -> np.ndarray:
    return oracle.f16_decode(bits) if fmt == "f16" else oracle.bf16_decode(bits)


def encode(values: np.ndarray, fmt: str) -> np.ndarray:
    return oracle.f16_encode(values) if fmt == "f16" else oracle.bf16_encode(values)


def check_tolerance(got_bits, ref, fmt: str, K: int, amax: float, bmax: float, label: str = ""):
    """Assert the random-input tolerance; returns a dict of the measured errors."""
    got = decode(np.asarray(got_bits).reshape(-1), fmt)
    ref = np.asarray(ref, np.float64).reshape(-1)
    assert np.all(np.isfinite(got)), f"{label}: non-finite outputs"
    rn = decode(encode(ref, fmt), fmt)
    diff_rn = got - rn
    denom = np.linalg.norm(rn)
    rel_frob = float(np.linalg.norm(diff_rn) / denom) if denom > 0 else float(np.linalg.norm(diff_rn))
    rel_frob_exact = float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300))
    acc_bound = 4e-3 * np.sqrt(K / 256.0) * amax * bmax
    bound = acc_bound + 0.5 * ulp(np.maximum(np.abs(got), np.abs(ref)), fmt)
    err = np.abs(got - ref)
    worst = int(np.argmax(err - bound))
    mismatches = int(np.count_nonzero(got != rn))
    stats = dict(rel_frob=rel_frob, rel_frob_vs_exact=rel_frob_exact, max_abs=float(err.max()),
                 acc_bound=float(acc_bound), mismatched_roundings=mismatches, n=int(got.size))
    assert rel_frob <= 1e-3, f"{label}: relative Frobenius error {rel_frob:.3e} > 1e-3 ({stats})"
    assert np.all(err <= bound), (f"{label}: |out - exact| = {err[worst]:.4g} > bound {bound[worst]:.4g} "
                                  f"at flat index {worst} ({stats})")
    return stats


def absmax_f16(bits) -> float:
    return float(np.max(np.abs(oracle.f16_decode(bits)))) if bits.size else 0.0


def absmax_bf16(bits) -> float:
    return float(np.max(np.abs(oracle.bf16_decode(bits)))) if bits.size else 0.0
