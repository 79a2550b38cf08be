// bsk_internal.h -- declarations shared by the library's translation units
// (not installed, not part of the C ABI).
#pragma once

#include <atomic>
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace bsk {

// Code a kernel writes into the device status word when a bounded wait gives
// up: kDevErrTimeoutBase + the number of the wait site (0 = no error).
constexpr int kDevErrTimeoutBase = 0x100;
// Code a kernel writes when an index it reads from the caller (a block-table
// entry) is out of range; the access is skipped.
constexpr int kDevErrBadIndex = 0x200;

// Grouped ordering of output tiles ("Hygon 优化", section 分组调度：提高 L2 数据复用):
// the 2-D grid of num_m x num_n tiles is flattened so that consecutive tile
// indices walk down a group of `group_m` tile rows before moving to the next
// tile column; tiles that share a column of B (and a row of A within the
// group) run close together in time and hit in L2.  The last group holds the
// remaining num_m mod group_m rows.
__host__ __device__ inline void tile_coord(int t, int num_m, int num_n, int group_m, int* pid_m, int* pid_n)
{
    const int per_group = group_m * num_n;
    const int group = t / per_group;
    const int first_m = group * group_m;
    const int rows_left = num_m - first_m;
    const int group_rows = rows_left < group_m ? rows_left : group_m;
    const int r = t - group * per_group;
    *pid_m = first_m + r % group_rows;
    *pid_n = r / group_rows;
}

// Launches `kern` on `stream`; with `pdl` set, as a programmatic dependent of
// the kernel before it in the stream: its CTAs may be scheduled while that
// kernel's last CTAs still run, so the kernel must execute griddepcontrol.wait
// before it reads or writes any memory an earlier stream operation may touch.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream, bool pdl,
                          Args&&... args)
{
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}

// Waits until the grids this one depends on programmatically have completed and
// their memory operations are visible (returns at once without such grids).
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Lets the next programmatic dependent in the stream be scheduled now; it still
// waits for this grid's completion in its own griddep_wait().
__device__ __forceinline__ void griddep_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

using TmapEncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// Sets the message bsk_last_error() returns on this host thread.
void record_error(const char* msg);

// cuTensorMapEncodeTiled from the driver (resolved once through the runtime).
TmapEncodeFn tmap_encoder();

// Raises one kernel's dynamic shared-memory limit, once per device: a launcher
// keeps one of these in a function-local static next to the kernel it launches,
// so the attribute call is not repeated on every launch (it costs host time
// that short kernels would otherwise wait for).  (Asking every kernel for the
// largest shared-memory carveout, so that consecutive kernels need no SM
// reconfiguration, was measured on GB300 and dropped: the CUDA-core GEMV then
// ran 52.5 -> 62.3 us per launch.)
struct SmemOptIn {
    static constexpr int kMaxDevices = 128;
    std::atomic<int> done[kMaxDevices];   // bytes already allowed on each device (static storage: zero)

    cudaError_t ensure(const void* kernel, int bytes)
    {
        int dev = -1;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        const bool slot = dev >= 0 && dev < kMaxDevices;
        if (slot && done[dev].load(std::memory_order_acquire) >= bytes) return cudaSuccess;
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
        if (e == cudaSuccess && slot) done[dev].store(bytes, std::memory_order_release);
        return e;
    }
};

// Launch of the tcgen05 GEMM: C (M x N, column-major, m contiguous, leading
// dimension ldc) = A (M x K) * B (K x N) [+ bias], FP32 accumulation, FP16 or
// BF16 in/out.  A is either MN-major (A(m,k) at A[m + k*lda]) or K-major (A(m,k)
// at A[k + m*lda]); B is K-major (B(k,n) at B[k + n*ldb]) or MN-major (B(k,n)
// at B[n + k*ldb]).  A and B must be 16-byte aligned with 16-byte-multiple
// leading dimensions (the caller packs them otherwise).
// Element types of the GEMM: A and B share one input type; C has its own.
// The FP8 types run on tcgen05.mma kind::f8f6f4 with K-major A and B only.
enum GemmInType : int { kInF16 = 0, kInBF16 = 1, kInE4M3 = 2, kInE5M2 = 3 };
enum GemmOutType : int { kOutF16 = 0, kOutBF16 = 1, kOutF32 = 2 };

struct GemmLaunch {
    const void* A = nullptr;
    long long lda = 0;
    bool a_mn_major = true;
    const void* B = nullptr;
    long long ldb = 0;
    bool b_mn_major = false;  // B(k,n) at B[n + k*ldb] (FP16 only, block_n >= 64)
    void* C = nullptr;
    long long ldc = 0;
    int M = 0, N = 0, K = 0;
    int in_type = kInF16;    // GemmInType of A and B
    int out_type = kOutF16;  // GemmOutType of C
    float alpha = 1.0f;      // FP8 inputs: C = alpha * A * B (the 16-bit kernels ignore it)
    int block_n = 256;       // 32, 64, 128 or 256
    int block_m = 128;       // one-CTA kernel, K-major A, whole tiles: rows per tile (8..128, a multiple of 8)
    bool pair = true;        // block_n == 256 only: CTA-pair kernel (256 x 256 tiles over two SMs)
    int group_m = 2;         // >= 1
    bool tma_store = false;  // C 16-byte aligned with 16-byte-multiple ldc
    const uint16_t* bias = nullptr;  // optional, output precision
    int bias_mode = 0;       // 1: bias[m] per row, 2: bias[n] per column
    int num_sms = 1;         // persistent grid size cap
    bool stream_k = false;   // one-CTA-per-tile kernel only: stream-K schedule over num_sms CTAs
    float* sk_part = nullptr;  // stream-K: num_sms * block_n * 128 floats of workspace
    int* sk_flag = nullptr;    // stream-K: num_sms ints, zero before the launch
    int* status = nullptr;   // device status word
    unsigned long long wait_limit_ns = 2000000000ull;
    bool pdl = true;         // whole-tile launches: programmatic dependent of the previous kernel
    bool dyn = false;        // CTA pairs, whole tiles: dynamic tile order (one cluster per tile launched)
    int skc = 0;             // one-CTA kernel: split-K over clusters of skc CTAs (2..16, a power of two
                             // dividing block_n); 0 = off
    int prefetch_kb = 0;     // one-CTA kernel, K-major A, whole tiles: extra k-blocks of the first
                             // tile's rows prefetched into L2 in the prologue
    bool k_alternate = false;  // CTA pairs, whole tiles: odd rounds run their k loop downwards
    int pair_m = 1;          // CTA pairs, 16-bit inputs, K-major B, whole tiles in the fixed order:
                             // 256-row blocks per pair tile (1 or 2)
};

// Returns 0 on success; otherwise an error message is written to `msg`.
int launch_gemm(const GemmLaunch& g, cudaStream_t stream, char* msg, size_t msg_len);
// Clusters of `skc` CTAs of the one-CTA GEMM kernel that fit on the current
// device at once (0 if the size is not available).
int split_k_capacity(int skc);
// The FP8 part of launch_gemm (gemm_fp8.cu).
int launch_gemm_fp8(const GemmLaunch& g, cudaStream_t stream, char* msg, size_t msg_len);
// CTA pairs on 512 x 256 tiles (gemm_tcgen05_m512.cu), and its column-major FP16
// instance (for loading its code ahead of time).
int launch_gemm_pair_m512(const GemmLaunch& g, cudaStream_t stream, char* msg, size_t msg_len);
const void* gemm_pair_m512_colmajor_kernel();

// Decode GEMV / skinny GEMM on the CUDA cores: y[t, j] = sum_k x[t, k] W[j, k]
// for t < n <= 8, W [M, K] row-major, x [n, K], y [n, M] row-major, BF16.
struct GemvLaunch {
    const uint16_t* W;
    const uint16_t* x;
    uint16_t* y;
    int M, K, n;
    int rows_per_warp;    // 0 = default for n
    int warps_per_block;  // 0 = default
    int kernel;           // 0 = auto, 1 = register streaming, 2/3 = cp.async-pipelined (x FP32 / BF16),
                          // 4 = token-paired accumulators
    int num_sms;
    bool pdl;             // programmatic dependent of the previous kernel in the stream
};
int launch_gemv(const GemvLaunch& g, cudaStream_t stream, char* msg, size_t msg_len);

// Split-KV decode attention over a paged BF16 cache (see attention.cu).
struct AttnLaunch {
    const uint16_t* q;            // [num_seqs, num_q_heads, head_dim]
    const uint16_t* k_cache;      // [num_blocks, block_size, num_kv_heads, head_dim]
    const uint16_t* v_cache;
    const int32_t* block_tables;  // [num_seqs, max_blocks]
    const int32_t* seq_lens;      // [num_seqs]
    uint16_t* out;                // [num_seqs, num_q_heads, head_dim]
    float* workspace;             // num_seqs * num_q_heads * num_segments * (head_dim + 2) floats
    int num_seqs, num_q_heads, num_kv_heads, head_dim;
    int block_size, max_blocks, num_blocks, max_seq_len, num_segments;
    float scale;
    int* status;
    bool pdl = true;              // split kernel: programmatic dependent of the previous kernel
};
int launch_decode_attention(const AttnLaunch& a, cudaStream_t stream, char* msg, size_t msg_len);
// CTAs of the attention's split kernel resident per SM for this head shape (>= 1).
int attention_ctas_per_sm(int head_dim, int q_per_kv);

// One operand copy for launch_pack: `lines` lines of line_bytes bytes, line l
// read from src + l * ld_src and written to dst + l * ld_dst (bytes; dst and
// ld_dst 16-byte aligned).  The source is only read.
struct PackCopy {
    const void* src;
    long long ld_src;
    void* dst;
    long long ld_dst;
    long long line_bytes;
    long long lines;
};

// Enqueues the n (at most two) copies in one launch on `stream`, as a
// programmatic dependent of the kernel before it when pdl is set.  A wait that
// gives up after limit_ns records a timeout in `status`.  The destination's
// leading dimension must be a multiple of 16 bytes and at least line_bytes
// rounded up to 16: a line's last 16-byte chunk is stored whole.
int launch_pack(const PackCopy* copies, int n, int sms, bool pdl, int* status, unsigned long long limit_ns,
                cudaStream_t stream, char* msg, size_t msg_len);

// C(m,n) = bias[m] (mode 1), bias[n] (mode 2) or +0.0 (mode 0) for the M x N
// column-major C with leading dimension ldc: the GEMM with K == 0.
int launch_fill_bias(uint16_t* C, long long ldc, int M, int N, const uint16_t* bias, int bias_mode,
                     cudaStream_t stream, char* msg, size_t msg_len);

// A caller-provided region that replaces the GEMM's stream-ordered workspace
// (packed operands, stream-K partials and flags), and the device status word
// its kernels report a timeout in.  `ptr` is 256-byte aligned.
struct FixedScratch {
    void* ptr = nullptr;
    size_t bytes = 0;
    int* status = nullptr;
};

// The work of gemm_f16_colmajor on `stream` with its workspace taken from
// `scratch` instead of allocated: the same argument checks, the same plan
// (pack, tile width, kernel, schedule, options) and the same kernels.  A plan
// that needs more than scratch.bytes is refused with BSK_ERR_INVALID_ARG
// before anything is launched.  Allocates nothing (no pinned status word
// either: the kernels write scratch.status).  Returns a bsk_status.
int enqueue_gemm_f16_colmajor_fixed(const uint16_t* A, const uint16_t* B, uint16_t* C, int M, int N, int K,
                                    const FixedScratch& scratch, cudaStream_t stream);

// Workspace bytes gemm_f16_colmajor(A, B, C, M, N, K) spends on packed
// operands (host arithmetic only; stream-K partials come on top).
size_t gemm_f16_colmajor_pack_bytes(const uint16_t* A, const uint16_t* B, int M, int N, int K);

// Loads the device code of every kernel the column-major FP16 GEMM may launch
// (its GEMM instances; the pack and fill kernels), so that no later launch of
// them maps device memory for code under lazy module loading.  0 on success.
int preload_gemm_f16_colmajor_kernels(char* msg, size_t msg_len);
int preload_aux_kernels(char* msg, size_t msg_len);

// Test hook: one CTA waits on an mbarrier that nothing completes, with the same
// bounded wait the GEMM uses; it must give up after `limit_ns` and record a
// timeout in the status word.
int launch_wait_timeout_probe(int* status, unsigned long long limit_ns, cudaStream_t stream, char* msg,
                              size_t msg_len);

}  // namespace bsk
