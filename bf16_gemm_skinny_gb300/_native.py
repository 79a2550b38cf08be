"""ctypes binding of libbsk (argument marshalling only).

Each function takes CUDA tensors (any 16-bit dtype; only ``data_ptr()`` is
used) or raw device addresses as ints, plus an optional stream (a
``torch.cuda.Stream``, a raw ``cudaStream_t`` int, or None for torch's current
stream), and calls the C entry point of the same name.  A non-zero status
raises :class:`BskError`.  The library is loaded on first use; if it has not
been built, the call raises -- there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

_lock = threading.Lock()
_lib = None

STATUS = {
    0: "BSK_OK",
    1: "BSK_ERR_INVALID_ARG",
    2: "BSK_ERR_UNSUPPORTED_DEVICE",
    3: "BSK_ERR_CUDA",
    4: "BSK_ERR_TIMEOUT",
    5: "BSK_ERR_NO_MEMORY",
}

OPTIONS = {
    "group_m": 1,
    "block_n": 2,
    "force_pack": 3,
    "force_direct_store": 4,
    "gemv_rows": 5,
    "gemv_warps": 6,
    "wait_limit_us": 7,
    "num_sms": 8,
    "gemv_kernel": 9,
    "gemm_kernel": 10,
    "stream_k": 11,
    "pdl": 12,
    "tile_sched": 13,
    "block_m": 14,
    "split_k": 15,
    "prefetch_kb": 16,
    "k_order": 17,
    "pair_m": 18,
}

# Every symbol include/bsk.h (the C ABI) declares.
EXPORTS = (
    "gemm_f16_colmajor", "gemv_bf16", "bsk_gemm_f16_colmajor_enqueue", "bsk_gemv_bf16_enqueue",
    "bsk_stream_check", "bsk_last_error", "bsk_status_string", "bsk_version", "gemm_f16_colmajor_noalloc",
    "decode_attention_bf16", "bsk_decode_attention_bf16_enqueue", "gemm_f16", "bsk_gemm_f16_enqueue",
    "gemm_fp8", "bsk_gemm_fp8_enqueue", "gemm_f16_colmajor_host", "gemv_bf16_host",
)
# Tuning options and test hooks (csrc/bsk_tuning.h): exported for the tests and
# the benchmark, not part of the C ABI.
TUNING_EXPORTS = ("bsk_tile_coord", "bsk_set_option", "bsk_get_option", "bsk_test_wait_timeout", "bsk_plan_gemm")

COL_MAJOR, ROW_MAJOR = 0, 1
BIAS_NONE, BIAS_ROW, BIAS_COLUMN = 0, 1, 2
FP8_E4M3, FP8_E5M2 = 0, 1
OUT_F32, OUT_BF16 = 0, 1


class BskError(RuntimeError):
    """A libbsk call returned a non-zero status."""

    def __init__(self, status: int, message: str):
        self.status = status
        super().__init__(f"{STATUS.get(status, status)}: {message}")


def library_path() -> str:
    return _build.LIB_PATH


def load():
    """Load libbsk.so (raises if it is missing: build it with bf16_gemm_skinny_gb300.build.build())."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"libbsk.so not built ({path}); run bf16_gemm_skinny_gb300.build.build()")
        lib = ctypes.CDLL(path)
        p = ctypes.c_void_p
        i = ctypes.c_int
        for name in ("gemm_f16_colmajor", "bsk_gemm_f16_colmajor_enqueue", "gemm_f16_colmajor_noalloc",
                     "gemm_f16_colmajor_host"):
            getattr(lib, name).argtypes = [p, p, p, i, i, i, p]
            getattr(lib, name).restype = i
        for name in ("gemm_f16", "bsk_gemm_f16_enqueue"):
            getattr(lib, name).argtypes = [i, i, i, p, i, p, i, p, i, i, i, i, p, i, p]
            getattr(lib, name).restype = i
        for name in ("gemm_fp8", "bsk_gemm_fp8_enqueue"):
            getattr(lib, name).argtypes = [i, p, i, p, i, p, i, i, i, i, i, ctypes.c_float, p]
            getattr(lib, name).restype = i
        for name in ("gemv_bf16", "bsk_gemv_bf16_enqueue", "gemv_bf16_host"):
            getattr(lib, name).argtypes = [p, p, p, i, i, i, p]
            getattr(lib, name).restype = i
        for name in ("decode_attention_bf16", "bsk_decode_attention_bf16_enqueue"):
            getattr(lib, name).argtypes = [p, p, p, p, p, p, i, i, i, i, i, i, i, i, ctypes.c_float, i, p]
            getattr(lib, name).restype = i
        lib.bsk_stream_check.argtypes = [p]
        lib.bsk_stream_check.restype = i
        lib.bsk_last_error.argtypes = []
        lib.bsk_last_error.restype = ctypes.c_char_p
        lib.bsk_status_string.argtypes = [i]
        lib.bsk_status_string.restype = ctypes.c_char_p
        lib.bsk_version.argtypes = []
        lib.bsk_version.restype = i
        lib.bsk_tile_coord.argtypes = [i, i, i, i, ctypes.POINTER(i), ctypes.POINTER(i)]
        lib.bsk_tile_coord.restype = None
        lib.bsk_set_option.argtypes = [i, ctypes.c_longlong]
        lib.bsk_set_option.restype = i
        lib.bsk_get_option.argtypes = [i]
        lib.bsk_get_option.restype = ctypes.c_longlong
        lib.bsk_test_wait_timeout.argtypes = [ctypes.c_uint, p]
        lib.bsk_test_wait_timeout.restype = i
        lib.bsk_plan_gemm.argtypes = [i, i, i, i, i, i, i, ctypes.POINTER(i)]
        lib.bsk_plan_gemm.restype = i
        _lib = lib
        return lib


def _addr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if hasattr(t, "data_ptr"):
        return int(t.data_ptr())
    return int(t.ctypes.data)   # a NumPy array (host memory)


_torch = None
_raw_stream = None


def _current_stream_handle() -> int:
    """cudaStream_t of torch's current stream on the current device.  Uses torch's
    direct accessor when it has one (a plain call instead of a Stream object)."""
    global _torch, _raw_stream
    if _torch is None:
        import torch

        _torch = torch
        raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
        get_dev = getattr(torch._C, "_cuda_getDevice", None)
        if raw is not None and get_dev is not None:
            _raw_stream = lambda: raw(get_dev())  # noqa: E731
    if _raw_stream is not None:
        return int(_raw_stream())
    return int(_torch.cuda.current_stream().cuda_stream)


def _stream(stream) -> int | None:
    if stream is None:
        return _current_stream_handle()
    if isinstance(stream, int):
        return stream
    return int(stream.cuda_stream)


def last_error() -> str:
    return load().bsk_last_error().decode(errors="replace")


def _check(status: int) -> None:
    if status != 0:
        raise BskError(status, last_error())


def gemm_f16_colmajor(A, B, C, M: int, N: int, K: int, stream=None) -> None:
    """C(m,n) = sum_k A(m,k) B(k,n), column-major FP16; blocks until done."""
    _check(load().gemm_f16_colmajor(_addr(A), _addr(B), _addr(C), M, N, K, _stream(stream)))


def gemm_f16_colmajor_enqueue(A, B, C, M: int, N: int, K: int, stream=None) -> None:
    """Asynchronous variant of gemm_f16_colmajor (check with stream_check)."""
    _check(load().bsk_gemm_f16_colmajor_enqueue(_addr(A), _addr(B), _addr(C), M, N, K, _stream(stream)))


def gemm_f16(order: int, transa: int, transb: int, A, lda: int, B, ldb: int, C, ldc: int, M: int, N: int,
             K: int, bias=None, bias_mode: int = BIAS_NONE, stream=None) -> None:
    """C = op(A) op(B) (+ bias), FP16, any storage order / transposition /
    leading dimensions (CBLAS conventions); blocks until done."""
    _check(load().gemm_f16(order, transa, transb, _addr(A), lda, _addr(B), ldb, _addr(C), ldc, M, N, K,
                           _addr(bias), bias_mode, _stream(stream)))


def gemm_f16_enqueue(order: int, transa: int, transb: int, A, lda: int, B, ldb: int, C, ldc: int, M: int, N: int,
                     K: int, bias=None, bias_mode: int = BIAS_NONE, stream=None) -> None:
    """Asynchronous variant of gemm_f16 (check with stream_check)."""
    _check(load().bsk_gemm_f16_enqueue(order, transa, transb, _addr(A), lda, _addr(B), ldb, _addr(C), ldc, M, N,
                                       K, _addr(bias), bias_mode, _stream(stream)))


def gemm_fp8(fmt: int, A, lda: int, B, ldb: int, C, ldc: int, out_type: int, M: int, N: int, K: int,
             alpha: float = 1.0, stream=None) -> None:
    """C(m,n) = alpha * sum_k A(m,k) B(k,n): FP8 codes, A[k + m*lda], B[k + n*ldb],
    C column-major FP32 or BF16; blocks until done."""
    _check(load().gemm_fp8(fmt, _addr(A), lda, _addr(B), ldb, _addr(C), ldc, out_type, M, N, K, float(alpha),
                           _stream(stream)))


def gemm_fp8_enqueue(fmt: int, A, lda: int, B, ldb: int, C, ldc: int, out_type: int, M: int, N: int, K: int,
                     alpha: float = 1.0, stream=None) -> None:
    """Asynchronous variant of gemm_fp8 (check with stream_check)."""
    _check(load().bsk_gemm_fp8_enqueue(fmt, _addr(A), lda, _addr(B), ldb, _addr(C), ldc, out_type, M, N, K,
                                       float(alpha), _stream(stream)))


def gemm_f16_colmajor_noalloc(A, B, C, M: int, N: int, K: int, stream=None) -> None:
    """gemm_f16_colmajor without any device allocation: packs unaligned operands
    into the library's fixed 96 MiB scratch array instead (see include/bsk.h)."""
    _check(load().gemm_f16_colmajor_noalloc(_addr(A), _addr(B), _addr(C), M, N, K, _stream(stream)))


def gemv_bf16(W, x, y, M: int, K: int, n: int, stream=None) -> None:
    """y[t, j] = sum_k x[t, k] W[j, k], BF16; blocks until done."""
    _check(load().gemv_bf16(_addr(W), _addr(x), _addr(y), M, K, n, _stream(stream)))


def gemm_f16_colmajor_host(A, B, C, M: int, N: int, K: int, stream=None) -> None:
    """gemm_f16_colmajor on host buffers (CPU tensors or NumPy arrays; pinned ones
    overlap the copies with the computation); blocks until C holds the result."""
    _check(load().gemm_f16_colmajor_host(_addr(A), _addr(B), _addr(C), M, N, K, _stream(stream)))


def gemv_bf16_host(W, x, y, M: int, K: int, n: int, stream=None) -> None:
    """gemv_bf16 on host buffers (CPU tensors or NumPy arrays); blocks until y holds
    the result."""
    _check(load().gemv_bf16_host(_addr(W), _addr(x), _addr(y), M, K, n, _stream(stream)))


def gemv_bf16_enqueue(W, x, y, M: int, K: int, n: int, stream=None) -> None:
    """Asynchronous variant of gemv_bf16 (check with stream_check)."""
    _check(load().bsk_gemv_bf16_enqueue(_addr(W), _addr(x), _addr(y), M, K, n, _stream(stream)))


def decode_attention_bf16(q, k_cache, v_cache, block_tables, seq_lens, out, num_seqs: int, num_q_heads: int,
                          num_kv_heads: int, head_dim: int, block_size: int, max_blocks: int, num_blocks: int,
                          max_seq_len: int, softmax_scale: float, num_segments: int = 0, stream=None) -> None:
    """Split-KV decode attention over a paged BF16 cache (see include/bsk.h); blocks until done."""
    _check(load().decode_attention_bf16(_addr(q), _addr(k_cache), _addr(v_cache), _addr(block_tables),
                                        _addr(seq_lens), _addr(out), num_seqs, num_q_heads, num_kv_heads, head_dim,
                                        block_size, max_blocks, num_blocks, max_seq_len, softmax_scale,
                                        num_segments, _stream(stream)))


def decode_attention_bf16_enqueue(q, k_cache, v_cache, block_tables, seq_lens, out, num_seqs: int,
                                  num_q_heads: int, num_kv_heads: int, head_dim: int, block_size: int,
                                  max_blocks: int, num_blocks: int, max_seq_len: int, softmax_scale: float,
                                  num_segments: int = 0, stream=None) -> None:
    """Asynchronous variant of decode_attention_bf16."""
    _check(load().bsk_decode_attention_bf16_enqueue(
        _addr(q), _addr(k_cache), _addr(v_cache), _addr(block_tables), _addr(seq_lens), _addr(out), num_seqs,
        num_q_heads, num_kv_heads, head_dim, block_size, max_blocks, num_blocks, max_seq_len, softmax_scale,
        num_segments, _stream(stream)))


def stream_check(stream=None) -> None:
    _check(load().bsk_stream_check(_stream(stream)))


def tile_coord(t: int, num_m: int, num_n: int, group_m: int):
    pm, pn = ctypes.c_int(), ctypes.c_int()
    load().bsk_tile_coord(t, num_m, num_n, group_m, ctypes.byref(pm), ctypes.byref(pn))
    return pm.value, pn.value


def plan_gemm(M: int, N: int, K: int, a_mn_major: bool = True, b_mn_major: bool = False, fp8: bool = False,
              sms: int = 152) -> dict:
    """The plan a GEMM of this shape would take (test hook; launches nothing)."""
    out = (ctypes.c_int * 7)()
    _check(load().bsk_plan_gemm(M, N, K, int(a_mn_major), int(b_mn_major), int(fp8), sms, out))
    return dict(zip(("block_n", "block_m", "pair", "stream_k", "split_k", "pair_m", "dyn"), list(out)))


def set_option(name: str, value: int) -> None:
    _check(load().bsk_set_option(OPTIONS[name], int(value)))


def get_option(name: str) -> int:
    return int(load().bsk_get_option(OPTIONS[name]))


def version() -> int:
    return int(load().bsk_version())


def test_wait_timeout(limit_us: int, stream=None) -> int:
    """Runs the watchdog probe; returns the raw status (BSK_ERR_TIMEOUT = 4 expected)."""
    return int(load().bsk_test_wait_timeout(limit_us, _stream(stream)))
