/*
 * bsk.h -- C ABI of libbsk: half-precision GEMM with FP32 accumulation on one
 * NVIDIA GB300 (sm_103a), in two regimes, plus the decode attention beside them:
 *
 *   gemm_f16_colmajor  large column-major FP16 GEMM on the tcgen05 tensor cores;
 *   gemm_f16           the same GEMM with transposed operands, row-major storage,
 *                      any leading dimensions and an optional fused bias;
 *   gemm_fp8           FP8 (E4M3 / E5M2) GEMM with FP32 accumulation;
 *   gemv_bf16          BF16 linear layer y = x W^T: the HBM-bound decode GEMV for
 *                      n <= 3 tokens (CUDA cores), the tensor-core GEMM for
 *                      larger n (skinny decode batches, prefill projections);
 *   decode_attention_bf16  split-KV decode attention over a paged BF16 KV cache.
 *
 * Conventions shared by every call:
 *  - Matrix pointers are DEVICE pointers (cudaMalloc / torch CUDA tensors) to
 *    16-bit values stored as raw bit patterns (IEEE binary16 or bfloat16).
 *    The caller owns every buffer; the library never writes an input.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *  - The blocking calls return only when their work on `stream` is complete
 *    (they synchronise that stream), so results may be read right away.
 *    The *_enqueue variants only launch; call bsk_stream_check() later.
 *  - Return value: a bsk_status code (0 = success).  On failure nothing has
 *    been written to the output unless the status is BSK_ERR_CUDA or
 *    BSK_ERR_TIMEOUT, and bsk_last_error() describes the failure.
 *  - Sizes are `int` (the signature of the original contract); every size
 *    must be >= 0.  A zero output extent is a no-op; K == 0 writes +0.0
 *    to every output element (the empty sum).
 *  - Only devices of compute capability 10.3 are supported; there is no CPU
 *    fallback and no other backend.
 */
#ifndef BSK_H
#define BSK_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum bsk_status {
    BSK_OK = 0,
    BSK_ERR_INVALID_ARG = 1,        /* bad size, null pointer, or an output overlapping an input */
    BSK_ERR_UNSUPPORTED_DEVICE = 2, /* current device is not compute capability 10.3 */
    BSK_ERR_CUDA = 3,               /* a CUDA runtime/driver call or a launch failed */
    BSK_ERR_TIMEOUT = 4,            /* a device-side wait gave up (watchdog); output undefined */
    BSK_ERR_NO_MEMORY = 5           /* the pack workspace could not be allocated */
} bsk_status;

/*
 * C = A * B, column-major FP16, FP32 accumulation, FP16 output rounded to
 * nearest even.  Definition: "MTT S4000 GEMM 优化中的分块、尾处理与并发实战复盘",
 * section 2 (GEMM入门): C(m,n) = sum_k A(m,k) B(k,n), with
 *     A(m,k) = A[m + k*M]   (M x K, leading dimension M)
 *     B(k,n) = B[k + n*K]   (K x N, leading dimension K)
 *     C(m,n) = C[m + n*M]   (M x N, leading dimension M)
 * and section 1 (规则分析): FP16 in, FP32 accumulate, FP16 out, inputs left
 * unmodified, computation complete on return, no BLAS library.
 *
 * Any M, N, K >= 0 are accepted.  When A or B is not 16-byte aligned or its
 * leading dimension is not a multiple of 8 elements, the operand is first
 * copied into a library-owned, stream-ordered workspace with a padded leading
 * dimension (BSK_ERR_NO_MEMORY if that allocation fails).  C may have any
 * alignment.  C must not overlap A or B (BSK_ERR_INVALID_ARG).
 */
int gemm_f16_colmajor(const uint16_t* A, const uint16_t* B, uint16_t* C, int M, int N, int K, void* stream);

/* Storage order of every matrix of a gemm_f16 call (the CBLAS convention). */
typedef enum bsk_order {
    BSK_COL_MAJOR = 0, /* entry (r, c) of a stored matrix at P[r + c*ld] */
    BSK_ROW_MAJOR = 1  /* entry (r, c) at P[c + r*ld] */
} bsk_order;

/* Axis of the optional bias of gemm_f16. */
typedef enum bsk_bias_mode {
    BSK_BIAS_NONE = 0,
    BSK_BIAS_ROW = 1,    /* bias[m]: one value per row of C (length M) */
    BSK_BIAS_COLUMN = 2  /* bias[n]: one value per column of C (length N) */
} bsk_bias_mode;

/*
 * The FP16 GEMM of gemm_f16_colmajor in every storage form, with an optional
 * fused bias:
 *     C(m,n) = fp16_rn( sum_k op(A)(m,k) op(B)(k,n) + bias ),  FP32 accumulation,
 * where op(A) = A (transa 0, A stored M x K) or A^T (transa 1, A stored K x M),
 * op(B) = B (transb 0, B stored K x N) or B^T (transb 1, B stored N x K), every
 * stored matrix (and C, M x N) addressed in `order` (bsk_order) with its own
 * leading dimension.  The product is the one of "MTT S4000 GEMM
 * 优化中的分块、尾处理与并发实战复盘", section 2 (GEMM入门), whose
 * column-major NN form gemm_f16_colmajor is; transposition flags and row-major
 * storage follow the BLAS/CBLAS conventions.  The bias is the optional term
 * that the DCU decode-GEMV article (forum.sourcefind.cn), section 6.1, names
 * among the properties of a linear call: an FP16 vector (device pointer) of
 * length M (BSK_BIAS_ROW) or N (BSK_BIAS_COLUMN), added to the FP32
 * accumulator before the single rounding; NULL with BSK_BIAS_NONE.  (A
 * row-major linear layer Y = X W^T + b is order BSK_ROW_MAJOR, transb 1,
 * BSK_BIAS_COLUMN.)
 *
 * Leading dimensions count elements and must be at least the stored row
 * count (column-major) or column count (row-major), and >= 1.  Operands that
 * are not 16-byte aligned or whose leading dimension is not a multiple of 8
 * are packed into a stream-ordered workspace first (BSK_ERR_NO_MEMORY if that
 * fails); C may have any alignment and stride.  Only the M x N entries of C
 * are written.  K == 0 writes the bias (or +0.0).  C must not overlap A, B
 * or the bias (BSK_ERR_INVALID_ARG), nor may a flag or mode be out of range.
 * Blocking, like gemm_f16_colmajor; bsk_gemm_f16_enqueue only launches.
 */
int gemm_f16(int order, int transa, int transb, const uint16_t* A, int lda, const uint16_t* B, int ldb,
             uint16_t* C, int ldc, int M, int N, int K, const uint16_t* bias, int bias_mode, void* stream);

/* FP8 formats of gemm_fp8 (OCP 8-bit floating point). */
typedef enum bsk_fp8_format {
    BSK_FP8_E4M3 = 0, /* 1 sign, 4 exponent (bias 7), 3 fraction bits; max 448; no infinity */
    BSK_FP8_E5M2 = 1  /* 1 sign, 5 exponent (bias 15), 2 fraction bits; max 57344; IEEE-style inf/NaN */
} bsk_fp8_format;

/* Output type of gemm_fp8. */
typedef enum bsk_out_type {
    BSK_OUT_F32 = 0,  /* IEEE binary32 */
    BSK_OUT_BF16 = 1  /* bfloat16, rounded to nearest even */
} bsk_out_type;

/*
 * FP8 GEMM with FP32 accumulation: C(m,n) = out( alpha * sum_k A(m,k) B(k,n) ).
 * The FP8 row of the matrix-instruction table in "Hygon 优化" (FlagGems
 * documentation), section DUMMA 矩阵指令形状: E4M3 or E5M2 inputs, FP32
 * accumulator; the product is the GEMM of "MTT S4000 GEMM 优化中的分块、尾处理与
 * 并发实战复盘", section 2.  A and B hold the same `format` (bsk_fp8_format),
 * both K-major (the layout the FP8 tensor-core instruction reads):
 *     A(m,k) = A[k + m*lda]   (M x K, each row's K codes contiguous, lda >= K)
 *     B(k,n) = B[k + n*ldb]   (K x N, each column's K codes contiguous, ldb >= K)
 *     C(m,n) = C[m + n*ldc]   (M x N column-major, ldc >= M; elements of `out_type`)
 * (a row-major linear layer Y[T,F] = X[T,K] W[F,K]^T is A = W, B = X, M = F,
 * N = T, and C = Y row-major with ldc = F).  `alpha` (finite) scales the FP32
 * accumulator before the output conversion (a product of per-tensor scales;
 * 1.0 gives the plain product).  BSK_OUT_F32 stores the scaled accumulator;
 * BSK_OUT_BF16 rounds it once to nearest even.  K == 0 writes +0.0.
 * Operands that are not 16-byte aligned or whose leading dimension is not a
 * multiple of 16 are packed into a stream-ordered workspace first.  C must
 * not overlap A or B.  Blocking; bsk_gemm_fp8_enqueue only launches.
 */
int gemm_fp8(int format, const uint8_t* A, int lda, const uint8_t* B, int ldb, void* C, int ldc, int out_type,
             int M, int N, int K, float alpha, void* stream);

/*
 * y = x W^T in BF16 with FP32 accumulation, output rounded to nearest even.
 * Definition: DCU decode-GEMV article (forum.sourcefind.cn), section 6.1:
 *     W : [M, K] row-major   W(j,k) = W[j*K + k]   (weights, output features x input features)
 *     x : [n, K] row-major   x(t,k) = x[t*K + k]   (n tokens)
 *     y : [n, M] row-major   y(t,j) = y[t*M + j] = sum_k x(t,k) W(j,k)
 * Section 2: n = 1 is the decode GEMV, large n the prefill GEMM.
 *
 * n <= 3 runs the CUDA-core GEMV (128-bit weight stream, warp-shuffle
 * reduction); n >= 4 runs the tcgen05 GEMM with both operands K-major (tiles
 * as narrow as 128 x 32 for small n).
 * Any M, K, n >= 0 are accepted (unaligned W/x or K % 8 != 0 take a scalar
 * CUDA-core variant, or the pack workspace on the tensor-core path).  y must
 * not overlap W or x.
 */
int gemv_bf16(const uint16_t* W, const uint16_t* x, uint16_t* y, int M, int K, int n, void* stream);

/*
 * Decode attention over a paged BF16 KV cache, split along the sequence and
 * merged with a numerically stable softmax reduction.  Definition: DCU
 * decode-GEMV article (forum.sourcefind.cn), section 6.1: per query head,
 * out = softmax(scale * q K^T) V over the sequence's tokens; section 6.3: the
 * tokens are cut into contiguous segments whose local (max, sum, prob V) are
 * merged by rescaling with exp(local max - global max); section 7: query head
 * h reads KV head h / (num_q_heads / num_kv_heads).  The page omits the score
 * scale; pass it (1/sqrt(head_dim) is usual; 1.0 gives the literal formula).
 *
 *   q            [num_seqs, num_q_heads, head_dim] BF16 (device)
 *   k_cache      [num_blocks, block_size, num_kv_heads, head_dim] BF16 (device)
 *   v_cache      same layout as k_cache
 *   block_tables [num_seqs, max_blocks] int32 (device): physical block of each
 *                block_size-token chunk of a sequence
 *   seq_lens     [num_seqs] int32 (device): tokens per sequence (clamped to
 *                [0, max_seq_len]; a sequence of length 0 gives zeros)
 *   out          [num_seqs, num_q_heads, head_dim] BF16 (device)
 *   num_segments segments per sequence, 1..1024 (the page chooses 16, or 32 once
 *                max_seq_len >= 12288, for its 80-CU part); 0 = automatic: one
 *                full wave of the split kernel on this GPU, each segment >= 64 tokens
 * head_dim 64, 128 or 256; num_q_heads / num_kv_heads 1, 2, 4 or 8; q, k_cache,
 * v_cache aligned to head_dim/16 bytes.  FP32 accumulation, output rounded to
 * nearest even.  A workspace of num_seqs * num_q_heads * segments *
 * (head_dim + 2) floats is allocated in stream order.  A block-table entry
 * outside [0, num_blocks) is skipped and reported as BSK_ERR_INVALID_ARG by
 * the blocking call (or the next bsk_stream_check).
 */
int decode_attention_bf16(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                          const int32_t* block_tables, const int32_t* seq_lens, uint16_t* out, int num_seqs,
                          int num_q_heads, int num_kv_heads, int head_dim, int block_size, int max_blocks,
                          int num_blocks, int max_seq_len, float softmax_scale, int num_segments, void* stream);

/*
 * gemm_f16_colmajor for callers that cannot allocate device memory during a
 * call (for example a serving process whose own allocator reserved all free
 * HBM at start-up, or a program held to a device-memory budget fixed when it
 * started).  Same arguments, result bits and blocking behaviour as
 * gemm_f16_colmajor: the same argument checks, the same choice of tiles,
 * kernel and schedule, the same kernels.  The pages have no counterpart:
 * this entry point exists for the way the library is deployed.
 *
 * Where gemm_f16_colmajor allocates a stream-ordered workspace (to pack an
 * operand whose base is not 16-byte aligned or whose M or K is not a multiple
 * of 8, or for the FP32 partials of the stream-K schedule), this call uses a
 * fixed 96 MiB device array that is part of the library (held on every GPU
 * that loads it, until the process exits) and calls no cudaMalloc, cudaFree
 * or other allocating routine.  Calls needing more workspace than 96 MiB
 * return BSK_ERR_INVALID_ARG before any device work; aligned operands need no
 * pack at any size.
 * Set-up: the first call on each device looks up the array's device address
 * (cudaGetSymbolAddress) and loads the device code of the kernels it may
 * launch.  Under CUDA's default lazy module loading that is when the 96 MiB
 * array and the kernels' code are mapped, so the first call on a device does
 * take device memory: make it before the caller reserves the device's free
 * memory (or run with CUDA_MODULE_LOADING=EAGER), and before anything else on
 * its stream is being captured.  Later calls allocate nothing.
 * The call blocks (it reads the device status word back and synchronises
 * `stream`), so it cannot be captured into a CUDA graph.
 * All calls share the array and keep the previous call's contents in it, so
 * calls that overlap on the GPU (several streams or host threads) race:
 * serialise them.
 */
int gemm_f16_colmajor_noalloc(const uint16_t* A, const uint16_t* B, uint16_t* C, int M, int N, int K,
                              void* stream);

/*
 * gemm_f16_colmajor and gemv_bf16 on HOST buffers: A, B, C (W, x, y) are host
 * pointers with the same layouts, sizes and results as the device calls (the
 * same kernels compute them).  The call takes device memory for the operands
 * and the result in stream order (M*K + K*N + M*N, or M*K + n*K + n*M,
 * 16-bit elements), copies in, computes, copies back and returns when the
 * result is in C (y), with `stream` synchronised.  The copies run on two
 * streams of the call's own beside `stream` and overlap the work in blocks:
 * the GEMM copies A first, then B and C in column blocks (the GEMM of one
 * block runs while the next block of B comes in and the previous block of C
 * goes out); gemv_bf16_host copies x first, then W in row blocks.  The
 * copies start after the work enqueued on `stream` before the call.
 * Page-locked (pinned) host buffers let the copies overlap the computation;
 * pageable buffers give the same result, with less overlap.  The device
 * memory comes from a memory pool of the library's (one per device, created
 * on the first such call), which keeps up to 2 GiB mapped between calls so
 * that repeated calls do not map fresh memory.  K = 0 fills C
 * (y) with +0.0 on the host; M = 0, N = 0 (n = 0) do nothing.  Errors as for
 * the device calls; C (y) must not overlap an input.
 */
int gemm_f16_colmajor_host(const uint16_t* A, const uint16_t* B, uint16_t* C, int M, int N, int K, void* stream);
int gemv_bf16_host(const uint16_t* W, const uint16_t* x, uint16_t* y, int M, int K, int n, void* stream);

/*
 * Same work as gemm_f16_colmajor / gemv_bf16 / decode_attention_bf16, but asynchronous: validates the
 * arguments, launches on `stream` and returns without waiting.  A device-side
 * watchdog timeout raised by this work is reported by the next
 * bsk_stream_check() (or the next blocking call).  Buffers must stay alive
 * until the stream has passed this work.
 */
int bsk_gemm_f16_enqueue(int order, int transa, int transb, const uint16_t* A, int lda, const uint16_t* B,
                         int ldb, uint16_t* C, int ldc, int M, int N, int K, const uint16_t* bias, int bias_mode,
                         void* stream);
int bsk_gemm_fp8_enqueue(int format, const uint8_t* A, int lda, const uint8_t* B, int ldb, void* C, int ldc,
                         int out_type, int M, int N, int K, float alpha, void* stream);
int bsk_gemm_f16_colmajor_enqueue(const uint16_t* A, const uint16_t* B, uint16_t* C, int M, int N, int K,
                                  void* stream);
int bsk_gemv_bf16_enqueue(const uint16_t* W, const uint16_t* x, uint16_t* y, int M, int K, int n, void* stream);
int bsk_decode_attention_bf16_enqueue(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                                      const int32_t* block_tables, const int32_t* seq_lens, uint16_t* out,
                                      int num_seqs, int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                      int max_blocks, int num_blocks, int max_seq_len, float softmax_scale,
                                      int num_segments, void* stream);

/* Synchronise `stream`, then report BSK_ERR_CUDA for a pending CUDA error or
 * BSK_ERR_TIMEOUT if a device-side wait gave up since the last check. */
int bsk_stream_check(void* stream);

/* Message for the last non-OK status returned on this host thread ("" if none). */
const char* bsk_last_error(void);

/* Short name of a status code. */
const char* bsk_status_string(int status);

/* Library version: major*10000 + minor*100 + patch. */
int bsk_version(void);

#ifdef __cplusplus
}
#endif

#endif /* BSK_H */
