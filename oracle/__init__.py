"""CPU oracle for the half-precision GEMM and the BF16 linear layer.

TEST INFRASTRUCTURE ONLY.  The tests, the package smoke check and the
benchmark's CPU-baseline leg are the only code allowed to import this
package.  The product library never imports, links or runs it, and it
shares no code with the CUDA path.

The arithmetic lives in ``oracle.c`` (plain C, FP64 accumulation, own
FP16/BF16 codecs, one round-to-nearest-even at the end); this module only
compiles that file with gcc and marshals numpy arrays into it.

Definitions followed:

* DCU decode-GEMV article (forum.sourcefind.cn), sections 6.1 and 7: decode
  attention over a paged KV cache, out = softmax(scale * q K^T) V per query
  head, query head h reading KV head h / (num_q_heads / num_kv_heads).

* "MTT S4000 GEMM 优化中的分块、尾处理与并发实战复盘", section 2 (GEMM入门):
  C(m,n) = sum_k A(m,k) B(k,n), column-major A[m + k*M], B[k + n*K],
  C[m + n*M]; section 1 (规则分析): FP16 in, FP32 accumulate, FP16 out.
* DCU decode-GEMV article (forum.sourcefind.cn), sections 6.1-6.2: the
  linear layer Y = X W^T with X:[n,k], W:[m,k], Y:[n,m].

Parity pins: every function here is pinned by ``tests/test_oracle_pins.py``
(exhaustive codec checks against numpy/torch and brute force, identity and
permutation matrices, rank-1 closed forms, exact rational brute force on tiny
shapes, the transpose identity, GEMV/GEMM consistency).
"""
from __future__ import annotations

import ctypes
import os
import shutil
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into oracle/_build/liboracle.so with gcc (-O2, OpenMP if available)."""
    with _lock:
        if (not force and os.path.exists(_LIB_PATH)
                and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
            return _LIB_PATH
        os.makedirs(_BUILD_DIR, exist_ok=True)
        cc = shutil.which("gcc") or shutil.which("cc")
        if cc is None:
            raise RuntimeError("oracle: no C compiler (gcc) found")
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        base = [cc, "-O2", "-std=c11", "-fPIC", "-shared", _SRC, "-o", tmp]
        r = subprocess.run(base[:2] + ["-fopenmp"] + base[2:] + ["-lm"],
                           capture_output=True, text=True)
        if r.returncode != 0:  # no libgomp: build single-threaded
            r = subprocess.run(base + ["-lm"], capture_output=True, text=True)
            if r.returncode != 0:
                raise RuntimeError("oracle: gcc failed:\n" + r.stderr)
        os.replace(tmp, _LIB_PATH)
        return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    # A test that plants a mistake in a copy of oracle.c points this variable at
    # the copy's build, to show that the pins catch the mistake.
    path = os.environ.get("ORACLE_LIB_OVERRIDE") or build()
    lib = ctypes.CDLL(path)
    u16p = ctypes.POINTER(ctypes.c_uint16)
    f64p = ctypes.POINTER(ctypes.c_double)
    i64p = ctypes.POINTER(ctypes.c_int64)
    i64 = ctypes.c_int64
    lib.orc_f16_decode.argtypes = [ctypes.c_uint16]
    lib.orc_f16_decode.restype = ctypes.c_double
    lib.orc_bf16_decode.argtypes = [ctypes.c_uint16]
    lib.orc_bf16_decode.restype = ctypes.c_double
    lib.orc_f16_encode_rn.argtypes = [ctypes.c_double]
    lib.orc_f16_encode_rn.restype = ctypes.c_uint16
    lib.orc_bf16_encode_rn.argtypes = [ctypes.c_double]
    lib.orc_bf16_encode_rn.restype = ctypes.c_uint16
    for name in ("orc_f16_decode_n", "orc_bf16_decode_n"):
        getattr(lib, name).argtypes = [u16p, f64p, i64]
        getattr(lib, name).restype = None
    for name in ("orc_f16_encode_n", "orc_bf16_encode_n"):
        getattr(lib, name).argtypes = [f64p, u16p, i64]
        getattr(lib, name).restype = None
    lib.orc_max_threads.argtypes = []
    lib.orc_max_threads.restype = ctypes.c_int
    for name in ("orc_gemm_f16_colmajor_cols", "orc_gemm_f16_colmajor_rows"):
        getattr(lib, name).argtypes = [u16p, u16p, i64, i64, i64, i64p, i64,
                                       f64p, u16p, ctypes.c_int]
        getattr(lib, name).restype = ctypes.c_int
    for name in ("orc_linear_bf16", "orc_linear_bf16_tokens"):
        getattr(lib, name).argtypes = [u16p, u16p, i64, i64, i64, i64p, i64,
                                       f64p, u16p, ctypes.c_int]
        getattr(lib, name).restype = ctypes.c_int
    ci = ctypes.c_int
    u8p = ctypes.POINTER(ctypes.c_uint8)
    u32p = ctypes.POINTER(ctypes.c_uint32)
    lib.orc_f32_encode_n.argtypes = [f64p, u32p, i64]
    lib.orc_f32_encode_n.restype = None
    lib.orc_fp8_decode_n.argtypes = [u8p, f64p, i64, ci]
    lib.orc_fp8_decode_n.restype = None
    lib.orc_gemm_fp8.argtypes = [ci, u8p, i64, u8p, i64, i64, i64, i64, ctypes.c_double, ci,
                                 i64p, i64, i64p, i64, f64p, u32p, u16p, ci]
    lib.orc_gemm_fp8.restype = ctypes.c_int
    lib.orc_gemm_f16_general.argtypes = [ci, ci, ci, u16p, i64, u16p, i64, i64, i64, i64, u16p, ci,
                                         i64p, i64, i64p, i64, f64p, u16p, ci]
    lib.orc_gemm_f16_general.restype = ctypes.c_int
    i32p = ctypes.POINTER(ctypes.c_int32)
    lib.orc_decode_attention_bf16.argtypes = [u16p, u16p, u16p, i32p, i32p, i64, i64, i64, i64, i64, i64, i64,
                                              ctypes.c_double, f64p, u16p, ctypes.c_int]
    lib.orc_decode_attention_bf16.restype = ctypes.c_int
    _lib = lib
    return lib


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError(f"expected uint16 bit patterns, got {a.dtype}")
    return a


def _ptr(a, ctype):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def max_threads() -> int:
    """Threads an OpenMP region of the oracle uses by default (1 if built without OpenMP)."""
    return int(_load().orc_max_threads())


# --------------------------------------------------------------------------
# codecs
# --------------------------------------------------------------------------

def f16_decode(bits) -> np.ndarray:
    """FP16 bit patterns -> exact float64 values (the oracle's own decoder)."""
    b = _u16(bits)
    out = np.empty(b.shape, np.float64)
    _load().orc_f16_decode_n(_ptr(b, ctypes.c_uint16), _ptr(out, ctypes.c_double), b.size)
    return out


def bf16_decode(bits) -> np.ndarray:
    """BF16 bit patterns -> exact float64 values (the oracle's own decoder)."""
    b = _u16(bits)
    out = np.empty(b.shape, np.float64)
    _load().orc_bf16_decode_n(_ptr(b, ctypes.c_uint16), _ptr(out, ctypes.c_double), b.size)
    return out


def f16_encode(x) -> np.ndarray:
    """float64 -> FP16 bits, one round-to-nearest-even straight from double."""
    v = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(v.shape, np.uint16)
    _load().orc_f16_encode_n(_ptr(v, ctypes.c_double), _ptr(out, ctypes.c_uint16), v.size)
    return out


def bf16_encode(x) -> np.ndarray:
    """float64 -> BF16 bits, one round-to-nearest-even straight from double."""
    v = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(v.shape, np.uint16)
    _load().orc_bf16_encode_n(_ptr(v, ctypes.c_double), _ptr(out, ctypes.c_uint16), v.size)
    return out


# --------------------------------------------------------------------------
# GEMM: C(m,n) = sum_k A(m,k) B(k,n), column-major, FP16 in/out
# --------------------------------------------------------------------------

def gemm_f16_colmajor(A, B, M: int, N: int, K: int, cols=None, threads: int = 0):
    """Oracle for the column-major FP16 GEMM.

    ``A`` and ``B`` are flat uint16 arrays holding A[m + k*M] and B[k + n*K].
    Returns ``(ref, out)``: ``ref`` is the float64 sum (before rounding) and
    ``out`` the FP16 bits after one round-to-nearest-even, both flat and
    column-major with shape ``M x ncols`` (``ncols = N`` when ``cols`` is None,
    else column j holds output column ``cols[j]``).
    """
    A = _u16(A).reshape(-1)
    B = _u16(B).reshape(-1)
    if A.size != M * K or B.size != N * K:
        raise ValueError("oracle: operand sizes do not match M, N, K")
    c = None if cols is None else np.ascontiguousarray(cols, dtype=np.int64)
    nc = N if c is None else c.size
    ref = np.empty(M * nc, np.float64)
    out = np.empty(M * nc, np.uint16)
    rc = _load().orc_gemm_f16_colmajor_cols(
        _ptr(A, ctypes.c_uint16), _ptr(B, ctypes.c_uint16), M, N, K,
        _ptr(c, ctypes.c_int64), 0 if c is None else c.size,
        _ptr(ref, ctypes.c_double), _ptr(out, ctypes.c_uint16), threads)
    if rc != 0:
        raise RuntimeError(f"oracle gemm failed ({rc})")
    return ref, out


def gemm_f16_colmajor_rows(A, B, M: int, N: int, K: int, rows, threads: int = 0):
    """Oracle GEMM restricted to output rows ``rows``.

    Returns ``(ref, out)`` with shape ``len(rows) x N`` stored column-major:
    entry (i, n) at ``i + n*len(rows)``.
    """
    A = _u16(A).reshape(-1)
    B = _u16(B).reshape(-1)
    if A.size != M * K or B.size != N * K:
        raise ValueError("oracle: operand sizes do not match M, N, K")
    r = np.ascontiguousarray(rows, dtype=np.int64)
    ref = np.empty(r.size * N, np.float64)
    out = np.empty(r.size * N, np.uint16)
    rc = _load().orc_gemm_f16_colmajor_rows(
        _ptr(A, ctypes.c_uint16), _ptr(B, ctypes.c_uint16), M, N, K,
        _ptr(r, ctypes.c_int64), r.size,
        _ptr(ref, ctypes.c_double), _ptr(out, ctypes.c_uint16), threads)
    if rc != 0:
        raise RuntimeError(f"oracle gemm rows failed ({rc})")
    return ref, out


def gemm_f16_general(A, B, M: int, N: int, K: int, lda: int, ldb: int, transa: int = 0, transb: int = 0,
                     row_major: int = 0, bias=None, bias_mode: int = 0, rows=None, cols=None, threads: int = 0):
    """Oracle for the FP16 GEMM in any storage form, with an optional bias.

    C(m,n) = fp16_rn(sum_k op(A)(m,k) op(B)(k,n) + bias), op() the BLAS
    transposition flags, every stored matrix addressed column-major
    (``row_major=0``: (r,c) at r + c*ld) or row-major (``row_major=1``: (r,c)
    at c + r*ld).  ``bias_mode`` 1: bias[m], 2: bias[n] (FP16 bits).
    Returns ``(ref, out)`` for the selected rows (all M when None) x columns
    (all N when None), flat and column-major over the selection.
    """
    A = _u16(A).reshape(-1)
    B = _u16(B).reshape(-1)

    def span(r, c, ld):  # elements a stored r x c matrix reaches
        if r == 0 or c == 0:
            return 0
        return (r - 1) + (c - 1) * ld + 1 if not row_major else (c - 1) + (r - 1) * ld + 1

    ar, ac = (K, M) if transa else (M, K)
    br, bc = (N, K) if transb else (K, N)
    if A.size < span(ar, ac, lda) or B.size < span(br, bc, ldb):
        raise ValueError("oracle: operands smaller than their shapes and leading dimensions")
    bz = None
    if bias_mode:
        bz = _u16(bias).reshape(-1)
        if bz.size < (M if bias_mode == 1 else N):
            raise ValueError("oracle: bias too short")
    r = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    c = None if cols is None else np.ascontiguousarray(cols, dtype=np.int64)
    nr = M if r is None else r.size
    nc = N if c is None else c.size
    ref = np.empty(nr * nc, np.float64)
    out = np.empty(nr * nc, np.uint16)
    rc = _load().orc_gemm_f16_general(
        row_major, transa, transb, _ptr(A, ctypes.c_uint16), lda, _ptr(B, ctypes.c_uint16), ldb, M, N, K,
        _ptr(bz, ctypes.c_uint16), bias_mode,
        _ptr(r, ctypes.c_int64), 0 if r is None else r.size, _ptr(c, ctypes.c_int64), 0 if c is None else c.size,
        _ptr(ref, ctypes.c_double), _ptr(out, ctypes.c_uint16), threads)
    if rc != 0:
        raise RuntimeError(f"oracle general gemm failed ({rc})")
    return ref, out


# --------------------------------------------------------------------------
# FP8 GEMM: C(m,n) = alpha * sum_k A(m,k) B(k,n), FP32 accumulator
# --------------------------------------------------------------------------

def f32_encode(x) -> np.ndarray:
    """float64 -> binary32 bits (uint32), one round-to-nearest-even."""
    v = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(v.shape, np.uint32)
    _load().orc_f32_encode_n(_ptr(v, ctypes.c_double), _ptr(out, ctypes.c_uint32), v.size)
    return out


def fp8_decode(codes, fmt: str) -> np.ndarray:
    """FP8 codes (uint8) -> float64; fmt 'e4m3' or 'e5m2'."""
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.empty(c.shape, np.float64)
    _load().orc_fp8_decode_n(_ptr(c, ctypes.c_uint8), _ptr(out, ctypes.c_double), c.size, _fp8_flag(fmt))
    return out


def _fp8_flag(fmt: str) -> int:
    if fmt not in ("e4m3", "e5m2"):
        raise ValueError("oracle: FP8 format must be 'e4m3' or 'e5m2'")
    return 1 if fmt == "e5m2" else 0


def gemm_fp8(A, B, M: int, N: int, K: int, lda: int, ldb: int, fmt: str = "e4m3", alpha: float = 1.0,
             out: str = "f32", rows=None, cols=None, threads: int = 0):
    """Oracle for the FP8 GEMM: C(m,n) = alpha * sum_k A(m,k) B(k,n) with
    A(m,k) = A[k + m*lda] and B(k,n) = B[k + n*ldb] (uint8 codes, both K-major).

    Returns ``(ref, out_bits)`` for the selected rows x columns (all when None),
    flat and column-major over the selection: ``ref`` the float64 value after
    alpha, ``out_bits`` one RN rounding of it to FP32 (uint32 bits, out='f32')
    or BF16 (uint16 bits, out='bf16').
    """
    A = np.ascontiguousarray(A, dtype=np.uint8).reshape(-1)
    B = np.ascontiguousarray(B, dtype=np.uint8).reshape(-1)
    if out not in ("f32", "bf16"):
        raise ValueError("oracle: FP8 GEMM output must be 'f32' or 'bf16'")
    if lda < max(1, K) or ldb < max(1, K):
        raise ValueError("oracle: leading dimension below K")
    if (M and K and A.size < (M - 1) * lda + K) or (N and K and B.size < (N - 1) * ldb + K):
        raise ValueError("oracle: operands smaller than their shapes and leading dimensions")
    r = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    c = None if cols is None else np.ascontiguousarray(cols, dtype=np.int64)
    nr = M if r is None else r.size
    nc = N if c is None else c.size
    ref = np.empty(nr * nc, np.float64)
    o32 = np.empty(nr * nc, np.uint32) if out == "f32" else None
    o16 = np.empty(nr * nc, np.uint16) if out == "bf16" else None
    rc = _load().orc_gemm_fp8(
        _fp8_flag(fmt), _ptr(A, ctypes.c_uint8), lda, _ptr(B, ctypes.c_uint8), ldb, M, N, K, float(alpha),
        0 if out == "f32" else 1, _ptr(r, ctypes.c_int64), 0 if r is None else r.size,
        _ptr(c, ctypes.c_int64), 0 if c is None else c.size, _ptr(ref, ctypes.c_double),
        _ptr(o32, ctypes.c_uint32), _ptr(o16, ctypes.c_uint16), threads)
    if rc != 0:
        raise RuntimeError(f"oracle FP8 gemm failed ({rc})")
    return ref, (o32 if out == "f32" else o16)


# --------------------------------------------------------------------------
# Linear layer: Y[t,j] = sum_k X[t,k] W[j,k], BF16 in/out
# --------------------------------------------------------------------------

def linear_bf16(W, X, M: int, K: int, n: int, js=None, threads: int = 0):
    """Oracle for y = x W^T (decode GEMV when n is small, prefill GEMM when large).

    ``W`` is [M,K] row-major, ``X`` is [n,K] row-major, both uint16 BF16 bits.
    Returns ``(ref, out)`` of shape ``(n, nj)``: float64 sums and BF16 bits,
    ``nj = M`` when ``js`` is None, else column i holds output feature ``js[i]``.
    """
    W = _u16(W).reshape(-1)
    X = _u16(X).reshape(-1)
    if W.size != M * K or X.size != n * K:
        raise ValueError("oracle: operand sizes do not match M, K, n")
    j = None if js is None else np.ascontiguousarray(js, dtype=np.int64)
    nj = M if j is None else j.size
    ref = np.empty(n * nj, np.float64)
    out = np.empty(n * nj, np.uint16)
    rc = _load().orc_linear_bf16(
        _ptr(W, ctypes.c_uint16), _ptr(X, ctypes.c_uint16), M, K, n,
        _ptr(j, ctypes.c_int64), 0 if j is None else j.size,
        _ptr(ref, ctypes.c_double), _ptr(out, ctypes.c_uint16), threads)
    if rc != 0:
        raise RuntimeError(f"oracle linear failed ({rc})")
    return ref.reshape(n, nj), out.reshape(n, nj)


def linear_bf16_tokens(W, X, M: int, K: int, n: int, ts, threads: int = 0):
    """Oracle linear layer for the tokens ``ts`` only: returns arrays of shape ``(len(ts), M)``."""
    W = _u16(W).reshape(-1)
    X = _u16(X).reshape(-1)
    if W.size != M * K or X.size != n * K:
        raise ValueError("oracle: operand sizes do not match M, K, n")
    t = np.ascontiguousarray(ts, dtype=np.int64)
    ref = np.empty(t.size * M, np.float64)
    out = np.empty(t.size * M, np.uint16)
    rc = _load().orc_linear_bf16_tokens(
        _ptr(W, ctypes.c_uint16), _ptr(X, ctypes.c_uint16), M, K, n,
        _ptr(t, ctypes.c_int64), t.size,
        _ptr(ref, ctypes.c_double), _ptr(out, ctypes.c_uint16), threads)
    if rc != 0:
        raise RuntimeError(f"oracle linear tokens failed ({rc})")
    return ref.reshape(t.size, M), out.reshape(t.size, M)


# --------------------------------------------------------------------------
# Decode attention over a paged BF16 KV cache
# --------------------------------------------------------------------------

def decode_attention_bf16(q, k_cache, v_cache, block_tables, seq_lens, num_q_heads: int, num_kv_heads: int,
                          head_dim: int, block_size: int, scale: float, threads: int = 0):
    """Oracle for out = softmax(scale * q K^T) V per (sequence, query head) over a paged cache.

    ``q``: uint16 [num_seqs, num_q_heads, head_dim]; ``k_cache``/``v_cache``: uint16
    [num_blocks, block_size, num_kv_heads, head_dim]; ``block_tables``: int32
    [num_seqs, max_blocks]; ``seq_lens``: int32 [num_seqs].  Returns ``(ref, out)`` with the
    float64 result and its BF16 bits, both [num_seqs, num_q_heads, head_dim].
    """
    q = _u16(q).reshape(-1)
    kc = _u16(k_cache).reshape(-1)
    vc = _u16(v_cache).reshape(-1)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32).reshape(-1)
    num_seqs = sl.size
    max_blocks = bt.shape[1] if bt.ndim == 2 else (bt.size // max(num_seqs, 1))
    per_block = block_size * num_kv_heads * head_dim
    num_blocks = kc.size // per_block if per_block else 0
    if q.size != num_seqs * num_q_heads * head_dim or kc.size != vc.size or kc.size != num_blocks * per_block:
        raise ValueError("oracle: attention operand sizes do not match")
    ref = np.empty(num_seqs * num_q_heads * head_dim, np.float64)
    out = np.empty(num_seqs * num_q_heads * head_dim, np.uint16)
    i32 = ctypes.c_int32
    rc = _load().orc_decode_attention_bf16(
        _ptr(q, ctypes.c_uint16), _ptr(kc, ctypes.c_uint16), _ptr(vc, ctypes.c_uint16),
        _ptr(bt, i32), _ptr(sl, i32), num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
        max_blocks, num_blocks, float(scale), _ptr(ref, ctypes.c_double), _ptr(out, ctypes.c_uint16), threads)
    if rc != 0:
        raise RuntimeError(f"oracle decode attention failed ({rc})")
    shape = (num_seqs, num_q_heads, head_dim)
    return ref.reshape(shape), out.reshape(shape)
