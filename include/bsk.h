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
 * started).  Same arguments, result and blocking behaviour as
 * gemm_f16_colmajor, and the same kernels.  The pages have no counterpart:
 * this entry point exists for the way the library is deployed.
 *
 * Instead of allocating a workspace when an operand must be packed (base not
 * 16-byte aligned, or M or K not a multiple of 8), it packs into a fixed
 * 96 MiB device array that is part of the library (held on every GPU that
 * loads it, until the process exits), and it calls no cudaMalloc, cudaFree or
 * other allocating routine.  Calls needing more scratch than 96 MiB return
 * BSK_ERR_INVALID_ARG; aligned operands need none at any size.
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress): make it before any stream capture on that device.
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

/*
 * Tile order of the GEMM ("Hygon 优化", section 分组调度：提高 L2 数据复用):
 * maps the flattened tile index t of a num_m x num_n tile grid to its tile
 * coordinates, visiting group_m tile rows per tile column, the last group
 * holding the remaining rows.  Host-side copy of the function the kernel
 * uses; needs no GPU.  Invalid arguments give (-1, -1).
 */
void bsk_tile_coord(int t, int num_m, int num_n, int group_m, int* pid_m, int* pid_n);

/*
 * Tuning and test options (process-wide; not thread-safe; 0 restores the
 * default).  Keys:
 *   BSK_OPT_GROUP_M          GEMM tile-row group size (default 2 for CTA pairs, 16 otherwise)
 *   BSK_OPT_BLOCK_N          GEMM tile width 32, 64, 128 or 256 (default: the smallest of
 *                            32/64/128 that covers N, else 256)
 *   BSK_OPT_FORCE_PACK       1: pack A and B even when aligned
 *   BSK_OPT_FORCE_DIRECT_STORE 1: masked register stores instead of the TMA store
 *   BSK_OPT_GEMV_ROWS        GEMV rows of W per warp: 1, 2, 4 or 8 (default by n)
 *   BSK_OPT_GEMV_WARPS       GEMV warps per CTA, 1..16 (default 16 pipelined, 8 streaming)
 *   BSK_OPT_WAIT_LIMIT_US    device-side wait limit in microseconds (default 2 s)
 *   BSK_OPT_NUM_SMS          cap on the persistent GEMM grid (default: all SMs)
 *   BSK_OPT_GEMM_KERNEL      GEMM kernel for 256-wide tiles: 1 one CTA per 128 x 256 tile,
 *                            2 CTA pairs on 256 x 256 tiles (default 2; narrower tiles
 *                            always run one CTA per 128 x BN tile)
 *   BSK_OPT_GEMV_KERNEL      kernel of gemv_bf16 for n <= 8: 1 register streaming,
 *                            2 cp.async-pipelined, 3 pipelined with x kept in BF16,
 *                            4 token-paired (n >= 5) -- the CUDA-core GEMVs -- or 5 the
 *                            tensor-core skinny GEMM (default: 1 for n <= 3, 5 for
 *                            n >= 4; a CUDA-core kernel whose buffers do not fit in
 *                            shared memory falls back to another)
 *   BSK_OPT_STREAM_K         GEMM schedule: 1 whole tiles, 2 stream-K (every SM -- or CTA
 *                            pair -- an equal share of the tile x k-block iterations of the
 *                            last wave; split tiles are summed in FP32 by the unit that
 *                            holds their first k-block), 0 automatic: stream-K on the
 *                            one-CTA-per-tile kernel when whole tiles would fill under three
 *                            quarters of the SMs and a tile has at least 32 k-blocks; whole
 *                            tiles on CTA pairs
 *   BSK_OPT_PDL              1: launch the GEMM, GEMV and attention kernels in plain stream
 *                            order; 0 (default): as programmatic dependents of the kernel
 *                            before them in the stream, so that their launch and prologue
 *                            (barrier set-up, TMEM allocation, L2 prefetch of the first
 *                            weight tiles) overlap that kernel's last CTAs.  Either way no
 *                            input is read and no output written before the earlier kernel
 *                            has completed.
 *   BSK_OPT_TILE_SCHED       tile order of the CTA-pair GEMM kernel (whole tiles): 0 or 1
 *                            fixed (pair p takes tiles p, p + P, ...), 2 dynamic (one cluster
 *                            per tile launched; a pair that is done takes the tile of a
 *                            cluster whose launch it cancels, so tiles go to the pairs that
 *                            are free first; BSK_OPT_NUM_SMS does not cap this grid)
 * Returns BSK_ERR_INVALID_ARG for an unknown key or a value out of range.
 */
enum {
    BSK_OPT_GROUP_M = 1,
    BSK_OPT_BLOCK_N = 2,
    BSK_OPT_FORCE_PACK = 3,
    BSK_OPT_FORCE_DIRECT_STORE = 4,
    BSK_OPT_GEMV_ROWS = 5,
    BSK_OPT_GEMV_WARPS = 6,
    BSK_OPT_WAIT_LIMIT_US = 7,
    BSK_OPT_NUM_SMS = 8,
    BSK_OPT_GEMV_KERNEL = 9,
    BSK_OPT_GEMM_KERNEL = 10,
    BSK_OPT_STREAM_K = 11,
    BSK_OPT_PDL = 12,
    BSK_OPT_TILE_SCHED = 13
};
int bsk_set_option(int key, long long value);
long long bsk_get_option(int key);

/*
 * Test hook for the watchdog: launches one CTA that waits on a barrier that
 * nothing completes, using the GEMM's bounded wait with a limit of
 * `limit_us` microseconds (1 .. 10,000,000).  Returns BSK_ERR_TIMEOUT when the
 * wait gave up as designed, BSK_OK never.  Blocks until the probe finished.
 */
int bsk_test_wait_timeout(unsigned int limit_us, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* BSK_H */
