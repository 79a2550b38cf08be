// api.cu -- the C ABI of libbsk: argument checks, path choice, workspace,
// launch, completion and error reporting.  No compute happens here.
//
// The host side follows the contract of "MTT S4000 GEMM 优化中的分块、尾处理与并发实战复盘",
// section 3.1 (搭代码框架): one exported entry that checks whether the fast
// path's layout requirements hold and otherwise takes a prepared path, then
// synchronises before returning.  Here the fast path is the TMA-fed tcgen05
// kernel; operands whose layout TMA cannot describe are packed into a
// workspace first (the same kernel then runs), rather than falling back to a
// second, slower GEMM.
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <climits>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <vector>

#include "bsk.h"
#include "bsk_internal.h"
#include "bsk_tuning.h"

namespace {

constexpr int kVersion = 100;   // 0.1.0

thread_local char t_err[1024] = "";

int fail(int status, const char* fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(t_err, sizeof(t_err), fmt, ap);
    va_end(ap);
    return status;
}

int fail_cuda(cudaError_t e, const char* what)
{
    return fail(BSK_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

// ----------------------------------------------------------------------------
// options
// ----------------------------------------------------------------------------
constexpr int kNumOpts = 19;
std::atomic<long long> g_opt[kNumOpts];

long long opt_or(int key, long long dflt)
{
    const long long v = g_opt[key].load(std::memory_order_relaxed);
    return v != 0 ? v : dflt;
}

constexpr long long kDefaultWaitLimitUs = 2000000;   // 2 s

// ----------------------------------------------------------------------------
// per-device state and the device status word
// ----------------------------------------------------------------------------
struct DeviceInfo {
    bool init = false;
    bool supported = false;
    int sms = 0;
    int major = 0, minor = 0;
};

constexpr int kMaxDevices = 128;
std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];
// Status word written by kernels when a bounded wait gives up: pinned,
// host-mapped memory, so the host reads it after a stream sync with no copy.
// Shared by every call of the process: a timeout is reported by the first
// check (blocking call or bsk_stream_check) that runs after it.
volatile int* g_status_host = nullptr;
int* g_status_dev = nullptr;

// Checks the current device (compute capability 10.3) and returns the SM
// count the GEMMs may use.  With `status_word` set it also creates, once per
// process, the pinned host-mapped status word the regular calls report
// device-side timeouts through (the fixed-scratch path passes false: it
// allocates nothing and brings its own status word).
int prepare_device(int* sms_out, bool status_word = true)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail_cuda(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(BSK_ERR_UNSUPPORTED_DEVICE, "device ordinal %d out of range", dev);
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceInfo& d = g_dev[dev];
    if (!d.init) {
        if ((e = cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
            return fail_cuda(e, "cudaDeviceGetAttribute");
        d.supported = (d.major == 10 && d.minor == 3);
        d.init = true;
    }
    if (!d.supported)
        return fail(BSK_ERR_UNSUPPORTED_DEVICE, "device %d has compute capability %d.%d; this library is built for 10.3 (sm_103a)",
                    dev, d.major, d.minor);
    if (status_word && g_status_host == nullptr) {
        void* h = nullptr;
        e = cudaHostAlloc(&h, 64, cudaHostAllocMapped | cudaHostAllocPortable);
        if (e != cudaSuccess) return fail_cuda(e, "cudaHostAlloc(status word)");
        std::memset(h, 0, 64);
        void* dptr = nullptr;
        e = cudaHostGetDevicePointer(&dptr, h, 0);
        if (e != cudaSuccess) return fail_cuda(e, "cudaHostGetDevicePointer(status word)");
        g_status_dev = static_cast<int*>(dptr);
        g_status_host = static_cast<volatile int*>(h);
    }
    long long cap = opt_or(BSK_OPT_NUM_SMS, d.sms);
    *sms_out = static_cast<int>(cap < d.sms ? cap : d.sms);
    return BSK_OK;
}

int check_status_word()
{
    if (g_status_host == nullptr) return BSK_OK;
    const int code = *g_status_host;
    if (code != 0) {
        *g_status_host = 0;
        if (code == bsk::kDevErrBadIndex)
            return fail(BSK_ERR_INVALID_ARG, "a block-table entry was out of range; its tokens were skipped");
        return fail(BSK_ERR_TIMEOUT, "a device-side wait gave up (site %d); the output is undefined",
                    code - bsk::kDevErrTimeoutBase);
    }
    return BSK_OK;
}

int sync_and_check(cudaStream_t s)
{
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return fail_cuda(e, "cudaStreamSynchronize");
    return check_status_word();
}

// ----------------------------------------------------------------------------
// helpers
// ----------------------------------------------------------------------------
bool overlaps(const void* a, size_t abytes, const void* b, size_t bbytes)
{
    if (abytes == 0 || bbytes == 0) return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + bbytes && b0 < a0 + abytes;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }


// Stream-ordered workspace for packed operands, freed in stream order after use.
struct Workspace {
    void* ptr = nullptr;
    cudaStream_t s = nullptr;
    ~Workspace() { release(); }
    // stream-ordered free on the stream it was taken on
    void release()
    {
        if (ptr != nullptr) cudaFreeAsync(ptr, s);
        ptr = nullptr;
    }
};

int alloc_workspace(Workspace& ws, size_t bytes, cudaStream_t s)
{
    ws.s = s;
    cudaError_t e = cudaMallocAsync(&ws.ptr, bytes, s);
    if (e != cudaSuccess) {
        cudaGetLastError();
        ws.ptr = nullptr;
        return fail(BSK_ERR_NO_MEMORY, "cudaMallocAsync(%zu bytes) for a workspace failed: %s", bytes,
                    cudaGetErrorString(e));
    }
    return BSK_OK;
}

// One GEMM as the kernels see it: C (column-major, M x N, leading dimension
// ldc) = A (M x K) * B (K x N) [+ bias].  A is MN-major (A(m,k) at
// A[m + k*lda]) or K-major (A[k + m*lda]); B is K-major (B[k + n*ldb]) or
// MN-major (B[n + k*ldb]).  Leading dimensions count elements.
struct GemmOp {
    const void* A = nullptr;
    long long lda = 0;
    bool a_mn_major = true;
    const void* B = nullptr;
    long long ldb = 0;
    bool b_mn_major = false;
    void* C = nullptr;
    long long ldc = 0;
    int M = 0, N = 0, K = 0;
    int in_type = bsk::kInF16;
    int out_type = bsk::kOutF16;
    float alpha = 1.0f;
    const uint16_t* bias = nullptr;
    int bias_mode = 0;
};

// Which operands must be packed before the TMA can read them (base not
// 16-byte aligned, or leading dimension not a multiple of 16 bytes), their
// padded leading dimensions and their workspace bytes (each rounded to 256).
struct PackPlan {
    int eb = 2;                   // element bytes of A and B
    int a_inner = 0, a_outer = 0;  // stored extents: `inner` contiguous elements in each of `outer` lines
    int b_inner = 0, b_outer = 0;
    bool a_ok = true, b_ok = true;
    long long lda_p = 0, ldb_p = 0;
    size_t a_bytes = 0, b_bytes = 0;
};

PackPlan plan_pack(const GemmOp& op)
{
    PackPlan pp;
    const bool force_pack = opt_or(BSK_OPT_FORCE_PACK, 0) != 0;
    const bool fp8 = op.in_type == bsk::kInE4M3 || op.in_type == bsk::kInE5M2;
    pp.eb = fp8 ? 1 : 2;
    const long long ld_unit = 16 / pp.eb;   // elements per 16 bytes
    pp.a_inner = op.a_mn_major ? op.M : op.K;
    pp.a_outer = op.a_mn_major ? op.K : op.M;
    pp.b_inner = op.b_mn_major ? op.N : op.K;
    pp.b_outer = op.b_mn_major ? op.K : op.N;
    pp.a_ok = !force_pack && aligned16(op.A) && (op.lda % ld_unit == 0);
    pp.b_ok = !force_pack && aligned16(op.B) && (op.ldb % ld_unit == 0);
    // a packed line starts on a 128-byte boundary (one TMA box row never
    // straddles two 128-byte L2 lines more than it must)
    const long long pad_unit = 128 / pp.eb;
    pp.lda_p = pp.a_ok ? op.lda : (pp.a_inner + pad_unit - 1) / pad_unit * pad_unit;
    pp.ldb_p = pp.b_ok ? op.ldb : (pp.b_inner + pad_unit - 1) / pad_unit * pad_unit;
    const size_t a_bytes = pp.a_ok ? 0 : static_cast<size_t>(pp.lda_p) * pp.a_outer * pp.eb;
    const size_t b_bytes = pp.b_ok ? 0 : static_cast<size_t>(pp.ldb_p) * pp.b_outer * pp.eb;
    pp.a_bytes = (a_bytes + 255) / 256 * 256;
    pp.b_bytes = (b_bytes + 255) / 256 * 256;
    return pp;
}

// The GemmOp of gemm_f16_colmajor(A, B, C, M, N, K).
GemmOp colmajor_op(const uint16_t* A, const uint16_t* B, uint16_t* C, int M, int N, int K)
{
    GemmOp op;
    op.A = A;
    op.lda = M > 1 ? M : 1;
    op.B = B;
    op.ldb = K > 1 ? K : 1;
    op.C = C;
    op.ldc = M > 1 ? M : 1;
    op.M = M;
    op.N = N;
    op.K = K;
    return op;
}

// The kernel, tile and schedule of one GEMM.  Every choice below was measured on
// GB300; the comments give the figures.
struct GemmPlan {
    int block_n = 256;      // tile width: 32, 64, 128 or 256
    int block_m = 128;      // one-CTA kernel, K-major A, one tile column: rows per tile
    bool pair = true;       // CTA-pair kernel (256 x 256 tiles over two SMs)
    bool stream_k = false;  // one-CTA kernel: stream-K schedule (workspace partials)
    int skc = 0;            // one-CTA kernel: split-K over clusters of skc CTAs
    bool dyn = false;       // CTA pairs: dynamic tile order
    int pair_m = 1;         // CTA pairs: 256-row blocks per tile (1: 256 x 256, 2: 512 x 256)
};

GemmPlan plan_gemm(const GemmOp& op, int sms)
{
    const bool fp8 = op.in_type == bsk::kInE4M3 || op.in_type == bsk::kInE5M2;
    // Tile width: the smallest of 32 / 64 / 128 covering a skinny N (one CTA per
    // tile, deep ring: the weight stream sets the pace), else 256 on CTA pairs.
    // An MN-major B is staged in 64-column swizzle atoms: at least 64 wide.
    const long long bn_opt = opt_or(BSK_OPT_BLOCK_N, 0);
    const int bn_auto = op.N <= 32 ? 32 : op.N <= 64 ? 64 : op.N <= 128 ? 128 : 256;
    int block_n = static_cast<int>(bn_opt > 0 ? bn_opt : bn_auto);
    if (op.b_mn_major && block_n < 64) block_n = 64;
    const long long gemm_kernel = opt_or(BSK_OPT_GEMM_KERNEL, 0);
    bool pair = block_n == 256 && gemm_kernel != 1;
    // Stream-K (one-CTA-per-tile kernel) when whole tiles would leave more than
    // a quarter of the SM slots idle and each tile has at least 64 k-blocks to
    // share (below that, whole tiles of the narrowest width that fits one wave).
    // A 256-wide shape whose CTA-pair tiles would fill under three quarters of
    // the pairs leaves the pairs for single CTAs from 32 k-blocks on.  Its fixed costs (workspace, flag reset, cooperative launch: about
    // 13 us of host and device time per call on GB300) outweigh the gain on
    // short problems and when the waves are already nearly full (measured: 272
    // tiles on 152 SMs 8% slower split; 4096 x 256 x 8192 13% faster split than
    // on CTA pairs before each tile's split was capped at four CTAs, 32.6 against
    // 47 us after; 256^3 and 1024^3 twice as slow).
    const long long kbs = (op.K + (fp8 ? 127LL : 63LL)) / (fp8 ? 128 : 64);
    const long long sk_opt = opt_or(BSK_OPT_STREAM_K, 0);
    auto fill = [&](long long tiles, long long slots) {
        const long long waves = (tiles + slots - 1) / slots;
        return static_cast<double>(tiles) / static_cast<double>(waves * slots);
    };
    const long long m_tiles = (op.M + 127LL) / 128;
    // Few tiles and a short k loop (too short to share out as stream-K): the
    // call's time is latency -- launch, first loads, one tile's MMAs, the
    // epilogue -- so narrower tiles on single CTAs spread it over more SMs.
    // 256^3 on GB300, calls back to back: 7.9 us per call on one CTA pair,
    // 5.2 us on 128 x 128 tiles, 4.5 us on 128 x 64 tiles (8 CTAs), 4.2 us on
    // 128 x 32 tiles (16 CTAs).  128 x 32 tiles are taken while they fit in one
    // wave (0.3 us faster than 128 x 64 from 256^3 to 640^3 and 1024 x 256 x
    // 1024; 1024^3 would need two waves of them: 12.3 against 8.3 us).
    if (pair && gemm_kernel == 0 && bn_opt == 0 && kbs < 32) {
        const long long pair_tiles = ((op.M + 255LL) / 256) * ((op.N + 255LL) / 256);
        if (pair_tiles * 4 <= (sms / 2 > 0 ? sms / 2 : 1)) {
            pair = false;
            block_n = !op.b_mn_major && m_tiles * ((op.N + 31LL) / 32) <= sms ? 32 : 64;
        }
    }
    // Short k loops: one CTA per 128 x 256 tile finishes before CTA pairs when a
    // tile has at most 8 k-blocks, or at most 32 with all single-CTA tiles in one
    // wave (GB300, calls back to back, pairs / single CTAs: 8192^2 x 256 57.2 /
    // 50.5 us, 8192^2 x 512 63.1 / 57.0, 4096^2 x 512 22.0 / 19.6, 2048^2 x 1024
    // 11.8 / 10.6, 2048^2 x 2048 16.7 / 15.5; 8192^2 x 1024 84.0 / 89.5 and
    // 4096^2 x 1024 27.4 / 27.4 stay on pairs).
    if (pair && gemm_kernel == 0 && bn_opt == 0) {
        const long long single_tiles = m_tiles * ((op.N + 255LL) / 256);
        if (kbs <= 8 || (kbs <= 32 && single_tiles <= sms)) pair = false;
    }
    if (pair && gemm_kernel == 0 && sk_opt != 1 && kbs >= 32) {
        const long long pair_tiles = ((op.M + 255LL) / 256) * ((op.N + 255LL) / 256);
        if (fill(pair_tiles, sms / 2 > 0 ? sms / 2 : 1) < 0.75) pair = false;
    }
    bool stream_k = false;
    if (!pair && sk_opt != 1) {
        const long long tiles = m_tiles * ((op.N + block_n - 1LL) / block_n);
        const bool starved = fill(tiles, sms) < 0.75;
        // Split only k loops of 64 k-blocks or more: at 32 its fixed costs and the
        // owners' fix-up outweigh the gain (calls back to back on GB300, split
        // against whole narrow tiles: 128 x 512 x 2048 20.6 / 12.0 us, 512 x 512 x
        // 2048 21.4 / 12.1, 2048 x 512 x 2048 24.9 / 12.9, 8192 x 128 x 2048 21.1 /
        // 12.9; at K = 4096 they are even, from K = 8192 on the split wins).
        stream_k = sk_opt == 2 || (starved && kbs >= 64);
        if (!stream_k && starved && bn_opt == 0 && gemm_kernel == 0) {
            // whole tiles: the narrowest whose grid still fits in one wave
            for (int bn = op.b_mn_major ? 64 : 32; bn < block_n; bn *= 2) {
                if (m_tiles * ((op.N + bn - 1LL) / bn) <= sms) {
                    block_n = bn;
                    break;
                }
            }
        }
    } else if (pair && sk_opt != 1) {
        // CTA pairs: whole waves first, the last (partial) wave shared -- on
        // request only.  The pair kernel runs under the power cap, so idle SMs in
        // a partial wave cost little; interleaved A/B on GB300 (stream-K time over
        // whole-tile time): 8192^2 x 16384 0.987, 4096^2 x 16384 0.944, at
        // K = 8192 or less 0.99 - 1.025, the ragged 4095 x 4097 x 4100 1.06 and
        // 4096 x 1024 x 4096 1.43 (fixed costs); inside a benchmark step of
        // GEMM + GEMVs the 8192^2 x 16384 gain did not show.
        stream_k = sk_opt == 2;
    }
    // Split-K over a cluster (one-CTA kernel): each tile's k loop is cut among a
    // cluster of 2..16 CTAs that sum their FP32 partials through distributed
    // shared memory -- no workspace, no flags, no cooperative launch.  For a
    // tile-starved problem the plan with the least estimated time wins, from a
    // model fitted to calls back to back on GB300: one CTA streams (128 + BN)
    // 128-byte operand rows per k-block at about 80 GB/s (1.6 ns a row); a
    // whole-tile launch costs about 4.3 us beyond that, a split one 5.0 us plus
    // 31 ns per column of its tile (the partial, the barriers, the sums) and
    // 0.5 us more for clusters of 16.  The largest cluster whose tiles all fit
    // on the device at once is taken for each width.  Measured (us, plan
    // chosen / whole tiles or stream-K): 128 x 128 x 16384 10.6 / 31.0, 128 x
    // 512 x 16384 13.1 / 39.3, 256 x 1024 x 8192 16.9 / 29.3, 1024 x 256 x 4096
    // 11.8 / 24.0, 128 x 512 x 2048 8.1 / 12.5; 128 x 8192 x 2048 stays on
    // whole tiles (13.4; the best split 15.1).
    int skc = 0;
    const long long skc_opt = opt_or(BSK_OPT_SPLIT_K, 0);
    if (!pair && skc_opt >= 2) {
        skc = static_cast<int>(skc_opt);
        stream_k = false;
    } else if (!pair && skc_opt == 0 && sk_opt == 0 && gemm_kernel == 0 && bn_opt == 0 && op.M > 0 && op.N > 0) {
        const long long tiles_now = m_tiles * ((op.N + block_n - 1LL) / block_n);
        if (fill(tiles_now, sms) < 0.75) {
            auto row_ns = [](long long bn) { return (128 + bn) * 16 / 10; };   // per k-block
            long long best = stream_k ? -1 : 4300 + kbs * ((tiles_now + sms - 1) / sms) * row_ns(block_n);
            for (int bn = op.b_mn_major ? 64 : 32; bn <= 256; bn *= 2) {
                const long long tiles = m_tiles * ((op.N + bn - 1LL) / bn);
                for (int sz = 16; sz >= 2; sz /= 2) {
                    if (kbs / sz < 2 || tiles > bsk::split_k_capacity(sz)) continue;
                    const long long est = 5000 + 31LL * bn + (sz == 16 ? 500 : 0) + (kbs + sz - 1) / sz * row_ns(bn);
                    if (best < 0 || est < best) {
                        best = est;
                        block_n = bn;
                        skc = sz;
                    }
                    break;
                }
            }
            if (skc > 1) stream_k = false;
        }
    }
    // Tile order on CTA pairs (whole tiles): fixed unless the dynamic order --
    // one cluster per tile launched, a free pair taking the tile of a cluster
    // whose launch it cancels -- is requested.  Interleaved A/B on GB300
    // (dynamic time over fixed): 8192^2 x 16384 1.00, 8192^3 0.98, the prefill
    // shape 1.00, 4095 x 4097 x 4100 and 8192^2 x 4096 1.03.
    const bool dyn = pair && !stream_k && opt_or(BSK_OPT_TILE_SCHED, 0) == 2;
    // Tile height of the one-CTA kernel on a K-major A with one tile column (the
    // skinny decode shapes): 128 rows, or fewer on request.  Heights that leave
    // every CTA the fewest rows -- the 34816-row decode weight as 291 tiles of
    // 120 rows on 146 CTAs, 240 rows each, instead of 272 tiles of 128 on 136
    // CTAs -- measured 1.2 us slower per launch on GB300 (n = 4 and 8, chains of
    // 24 launches: 59.2 / 58.6 us against 57.8 / 57.4), so they are not the
    // default.
    // CTA pairs on 512 x 256 tiles (16-bit inputs, K-major B, whole tiles in the
    // fixed order): each CTA stages 256 rows of A, so every B slice in shared
    // memory feeds two MMAs and a k step moves 48 KB per SM for twice the MMAs of
    // a 256 x 256 tile's 32 KB, which relieves the shared memory (at 256 x 256 its
    // bandwidth is the limit).  The one accumulator leaves the epilogue of a tile
    // unhidden, so long k loops only.  GB300, 16-bit, calls back to back (256 x
    // 256 / 512 x 256 tiles): 8192^2 x 16384 1853-1856 / 1924-1926 TFLOP/s, for 3 s
    // under the power cap 1610-1611 / 1672-1673 (SM clock 1470-1477 / 1530 MHz);
    // 8192^3 1829-1841 / 1869-1874; 34816 x 4096 x 5120 (80 k-blocks) 0.753 / 0.783 ms.
    int pair_m = 1;
    const long long pm_opt = opt_or(BSK_OPT_PAIR_M, 0);
    if (pair && !stream_k && !dyn && !op.b_mn_major && !fp8 && pm_opt != 1) {
        if (pm_opt == 2) {
            pair_m = 2;
        } else if (kbs >= 128) {
            const long long pairs = sms / 2 > 0 ? sms / 2 : 1;
            const long long n_tiles = (op.N + 255LL) / 256;
            const double fill256 = fill(((op.M + 255LL) / 256) * n_tiles, pairs);
            const double fill512 = fill(((op.M + 511LL) / 512) * n_tiles, pairs);
            if (fill512 >= fill256 - 0.02) pair_m = 2;
        }
    }
    int block_m = 128;
    const long long bm_opt = opt_or(BSK_OPT_BLOCK_M, 0);
    if (!pair && !stream_k && !op.a_mn_major && (op.N + block_n - 1LL) / block_n == 1 && bm_opt > 0)
        block_m = static_cast<int>(bm_opt);
    GemmPlan plan;
    plan.block_n = block_n;
    plan.block_m = block_m;
    plan.pair = pair;
    plan.stream_k = stream_k;
    plan.skc = skc;
    plan.dyn = dyn;
    plan.pair_m = pair_m;
    return plan;
}

// Runs the tcgen05 GEMM on operands in any layout TMA may not take directly:
// an operand whose base is not 16-byte aligned or whose leading dimension is
// not a multiple of 16 bytes is packed into a stream-ordered workspace (or
// into `fixed`, when given).
int run_gemm(const GemmOp& op, int sms, cudaStream_t s, const bsk::FixedScratch* fixed = nullptr)
{
    const PackPlan pp = plan_pack(op);
    const int eb = pp.eb;
    const int a_inner = pp.a_inner, a_outer = pp.a_outer, b_inner = pp.b_inner, b_outer = pp.b_outer;
    const bool a_ok = pp.a_ok, b_ok = pp.b_ok;
    const long long lda_p = pp.lda_p, ldb_p = pp.ldb_p;
    const size_t a_bytes = pp.a_bytes, b_bytes = pp.b_bytes;

    const GemmPlan plan = plan_gemm(op, sms);
    const int block_n = plan.block_n;
    const bool stream_k = plan.stream_k;

    // one slot per CTA: block_n x 128 FP32 (CTA pairs: each CTA's 128 rows of a 256-wide tile)
    const size_t sk_part_bytes = stream_k ? static_cast<size_t>(sms) * block_n * 128 * sizeof(float) : 0;
    const size_t sk_flag_bytes = stream_k ? static_cast<size_t>(sms) * sizeof(int) : 0;

    Workspace ws;
    const void* Ause = op.A;
    const void* Buse = op.B;
    float* sk_part = nullptr;
    int* sk_flag = nullptr;
    char msg[512] = "";
    const size_t ws_bytes = a_bytes + b_bytes + sk_part_bytes + sk_flag_bytes;
    if (ws_bytes > 0) {
        uint8_t* base = nullptr;
        if (fixed != nullptr) {
            if (ws_bytes > fixed->bytes)
                return fail(BSK_ERR_INVALID_ARG,
                            "this problem needs %zu bytes of workspace (packed operands%s), more than the fixed "
                            "%zu-byte (%zu MiB) scratch array; pass 16-byte-aligned operands with 16-byte-multiple "
                            "leading dimensions (no pack) or use the allocating entry point",
                            ws_bytes, stream_k ? " and stream-K partials" : "", fixed->bytes, fixed->bytes >> 20);
            base = static_cast<uint8_t*>(fixed->ptr);
        } else {
            int st = alloc_workspace(ws, ws_bytes, s);
            if (st != BSK_OK) return st;
            base = static_cast<uint8_t*>(ws.ptr);
        }
        // the operands that need it are copied to a 16-byte-multiple leading
        // dimension in the workspace, both in one launch
        bsk::PackCopy copies[2];
        int n_copies = 0;
        if (!a_ok) {
            copies[n_copies++] = {op.A, op.lda * eb, base, lda_p * eb, static_cast<long long>(a_inner) * eb, a_outer};
            Ause = base;
        }
        if (!b_ok) {
            copies[n_copies++] = {op.B, op.ldb * eb, base + a_bytes, ldb_p * eb, static_cast<long long>(b_inner) * eb,
                                  b_outer};
            Buse = base + a_bytes;
        }
        if (n_copies > 0 &&
            bsk::launch_pack(copies, n_copies, sms, opt_or(BSK_OPT_PDL, 0) != 1,
                             fixed != nullptr ? fixed->status : g_status_dev,
                             static_cast<unsigned long long>(opt_or(BSK_OPT_WAIT_LIMIT_US, kDefaultWaitLimitUs)) * 1000ull,
                             s, msg, sizeof(msg)))
            return fail(BSK_ERR_CUDA, "%s", msg);
        if (stream_k) {
            sk_part = reinterpret_cast<float*>(base + a_bytes + b_bytes);
            sk_flag = reinterpret_cast<int*>(base + a_bytes + b_bytes + sk_part_bytes);
            cudaError_t e = cudaMemsetAsync(sk_flag, 0, sk_flag_bytes, s);
            if (e != cudaSuccess) return fail_cuda(e, "cudaMemsetAsync(stream-K flags)");
        }
    }

    bsk::GemmLaunch g;
    g.A = Ause;
    g.lda = lda_p;
    g.a_mn_major = op.a_mn_major;
    g.B = Buse;
    g.ldb = ldb_p;
    g.b_mn_major = op.b_mn_major;
    g.C = op.C;
    g.ldc = op.ldc;
    g.M = op.M;
    g.N = op.N;
    g.K = op.K;
    g.in_type = op.in_type;
    g.out_type = op.out_type;
    g.alpha = op.alpha;
    g.bias = op.bias_mode != 0 ? op.bias : nullptr;
    g.bias_mode = op.bias_mode;
    g.block_n = plan.block_n;
    g.block_m = plan.block_m;
    g.pair = plan.pair;
    g.stream_k = plan.stream_k;
    g.sk_part = sk_part;
    g.sk_flag = sk_flag;
    g.skc = plan.skc;
    // Tile-row group ("Hygon 优化", section 分组调度).  CTA pairs: 8.  Measured on
    // GB300 on 8192^2 x 16384, one launch (cold L2): DRAM reads 4.54 / 4.35 /
    // 2.34 / 3.46 GB for GROUP_M 2 / 4 / 8 / 16, 1.235 / 1.238 / 1.169 / 1.204
    // ms; back to back for seconds under the 1.4 kW cap every setting does the
    // same work per SM cycle and 8 runs at the highest clock: 1580 / 1631 /
    // 1644 / 1622 TFLOP/s.  One CTA per tile: 16.
    g.group_m = static_cast<int>(opt_or(BSK_OPT_GROUP_M, g.pair && g.block_n == 256 ? 8 : 16));
    // TMA store of C: 16-byte aligned base and ldc, and M a multiple of 8.  With
    // a ragged M the store's clipping was seen to write up to the end of the
    // last 16-byte unit, i.e. into C's padding rows when ldc > M.
    // FP32 outputs always take the coalesced direct stores (32 lanes x 4 bytes).
    g.tma_store = op.out_type != bsk::kOutF32 && aligned16(op.C) && (op.ldc % 8 == 0) && (op.M % 8 == 0) &&
                  opt_or(BSK_OPT_FORCE_DIRECT_STORE, 0) == 0;
    g.num_sms = sms;
    g.status = fixed != nullptr ? fixed->status : g_status_dev;
    g.wait_limit_ns = static_cast<unsigned long long>(opt_or(BSK_OPT_WAIT_LIMIT_US, kDefaultWaitLimitUs)) * 1000ull;
    g.pdl = opt_or(BSK_OPT_PDL, 0) != 1;
    g.dyn = plan.dyn;
    // One-CTA kernel with a K-major A (the skinny decode weight): while a launch
    // waits for the kernel before it, its epilogue warps prefetch 16 more
    // k-blocks of their first tile's rows into L2, using the DRAM bandwidth the
    // earlier kernel's last CTAs leave idle.  34816 x 5120 on GB300, per launch
    // (off / 4 / 8 / 16 / 32 k-blocks), chains of 24 back to back: n = 4 57.3-57.8
    // / 57.4-57.5 / 57.0-57.3 / 56.7 / 56.5-56.8 us, n = 8 57.7-58.2 / 57.7-57.9 /
    // 57.2-57.4 / 56.3-56.5 / 57.0; one launch after a GEMM: the same within 1 us
    // up to 16, 1-2 us slower at 32 (the prefetches then delay the first loads).
    const long long pf_opt = opt_or(BSK_OPT_PREFETCH_KB, 0);
    g.prefetch_kb = static_cast<int>(pf_opt == 0 ? 16 : pf_opt == 1 ? 0 : pf_opt);
    // CTA pairs: odd rounds of whole tiles run their k loop from the top, so a
    // round starts on the A panels' k-slices the round before it read last (still
    // in L2).  8192^2 x 16384 on GB300, back to back for 3 s under the 1.4 kW
    // cap, two interleaved pairs of runs: 1612.7 / 1616.5 TFLOP/s at 1447 / 1455
    // MHz against 1597.7 / 1598.8 at 1425 / 1432 always ascending; DRAM reads of
    // one launch 2.23 / 2.28 GB against 2.31 / 2.54; single launches the same
    // within their spread.  Each tile still has one fixed summation order.
    g.k_alternate = opt_or(BSK_OPT_K_ORDER, 0) != 1;
    g.pair_m = plan.pair_m;
    if (bsk::launch_gemm(g, s, msg, sizeof(msg))) return fail(BSK_ERR_CUDA, "%s", msg);
    return BSK_OK;
}

// Elements a stored matrix with `outer` lines of `inner` elements, `ld` apart, reaches.
long long span_elems(long long inner, long long outer, long long ld)
{
    if (inner == 0 || outer == 0) return 0;
    return (outer - 1) * ld + inner;
}

// The general FP16 GEMM on column-major storage (row-major calls are mapped
// onto it by the caller): C = op(A) op(B) [+ bias].
int enqueue_gemm_general(int transa, int transb, const uint16_t* A, long long lda, const uint16_t* B,
                         long long ldb, uint16_t* C, long long ldc, int M, int N, int K, const uint16_t* bias,
                         int bias_mode, void* stream, const bsk::FixedScratch* fixed = nullptr)
{
    if (M < 0 || N < 0 || K < 0) return fail(BSK_ERR_INVALID_ARG, "negative size (M=%d N=%d K=%d)", M, N, K);
    if ((transa != 0 && transa != 1) || (transb != 0 && transb != 1))
        return fail(BSK_ERR_INVALID_ARG, "transa/transb must be 0 or 1 (got %d, %d)", transa, transb);
    if (bias_mode < 0 || bias_mode > 2) return fail(BSK_ERR_INVALID_ARG, "bias_mode must be 0, 1 or 2 (got %d)", bias_mode);
    if (bias_mode != 0 && bias == nullptr) return fail(BSK_ERR_INVALID_ARG, "bias_mode %d needs a bias vector", bias_mode);
    // stored shapes: A is M x K (transa 0) or K x M (transa 1), B is K x N or N x K
    const long long a_rows = transa ? K : M, a_cols = transa ? M : K;
    const long long b_rows = transb ? N : K, b_cols = transb ? K : N;
    if (lda < (a_rows > 1 ? a_rows : 1) || ldb < (b_rows > 1 ? b_rows : 1) || ldc < (M > 1 ? M : 1))
        return fail(BSK_ERR_INVALID_ARG, "leading dimension too small (lda=%lld ldb=%lld ldc=%lld for M=%d N=%d K=%d, "
                    "transa=%d transb=%d)", lda, ldb, ldc, M, N, K, transa, transb);
    if (M == 0 || N == 0) return BSK_OK;
    const size_t a_bytes = static_cast<size_t>(span_elems(a_rows, a_cols, lda)) * 2;
    const size_t b_bytes = static_cast<size_t>(span_elems(b_rows, b_cols, ldb)) * 2;
    const size_t c_bytes = static_cast<size_t>(span_elems(M, N, ldc)) * 2;
    const size_t bias_bytes = bias_mode == 0 ? 0 : static_cast<size_t>(bias_mode == 1 ? M : N) * 2;
    if (C == nullptr) return fail(BSK_ERR_INVALID_ARG, "C is NULL");
    if (K > 0 && (A == nullptr || B == nullptr)) return fail(BSK_ERR_INVALID_ARG, "A or B is NULL");
    if (overlaps(C, c_bytes, A, K > 0 ? a_bytes : 0) || overlaps(C, c_bytes, B, K > 0 ? b_bytes : 0) ||
        overlaps(C, c_bytes, bias, bias_bytes))
        return fail(BSK_ERR_INVALID_ARG, "C overlaps an input");
    const long long tiles = ((M + 127LL) / 128) * ((N + 127LL) / 128);
    if (tiles > INT_MAX) return fail(BSK_ERR_INVALID_ARG, "problem too large (%lld tiles)", tiles);
    int sms = 0;
    int st = prepare_device(&sms, fixed == nullptr);
    if (st != BSK_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (K == 0) {
        char msg[512] = "";
        if (bsk::launch_fill_bias(C, ldc, M, N, bias, bias_mode, s, msg, sizeof(msg)))
            return fail(BSK_ERR_CUDA, "%s", msg);
        return BSK_OK;
    }
    GemmOp op;
    op.A = A;
    op.lda = lda;
    op.a_mn_major = transa == 0;
    op.B = B;
    op.ldb = ldb;
    op.b_mn_major = transb == 1;
    op.C = C;
    op.ldc = ldc;
    op.M = M;
    op.N = N;
    op.K = K;
    op.bias = bias;
    op.bias_mode = bias_mode;
    return run_gemm(op, sms, s, fixed);
}

int enqueue_gemm_f16_cblas(int order, int transa, int transb, const uint16_t* A, int lda, const uint16_t* B,
                           int ldb, uint16_t* C, int ldc, int M, int N, int K, const uint16_t* bias,
                           int bias_mode, void* stream)
{
    if (order == BSK_COL_MAJOR)
        return enqueue_gemm_general(transa, transb, A, lda, B, ldb, C, ldc, M, N, K, bias, bias_mode, stream);
    if (order != BSK_ROW_MAJOR) return fail(BSK_ERR_INVALID_ARG, "order must be BSK_COL_MAJOR or BSK_ROW_MAJOR");
    // Row-major C (M x N) is column-major C^T (N x M) = op(B)^T op(A)^T, and a
    // row-major stored matrix is the column-major store of its transpose: swap
    // the operands and their flags, and the bias's axis.
    if (bias_mode < 0 || bias_mode > 2) return fail(BSK_ERR_INVALID_ARG, "bias_mode must be 0, 1 or 2 (got %d)", bias_mode);
    const int swapped_mode = bias_mode == 1 ? 2 : bias_mode == 2 ? 1 : 0;
    return enqueue_gemm_general(transb, transa, B, ldb, A, lda, C, ldc, N, M, K, bias, swapped_mode, stream);
}

int enqueue_gemm_fp8(int format, const uint8_t* A, int lda, const uint8_t* B, int ldb, void* C, int ldc,
                     int out_type, int M, int N, int K, float alpha, void* stream)
{
    if (M < 0 || N < 0 || K < 0) return fail(BSK_ERR_INVALID_ARG, "negative size (M=%d N=%d K=%d)", M, N, K);
    if (format != BSK_FP8_E4M3 && format != BSK_FP8_E5M2)
        return fail(BSK_ERR_INVALID_ARG, "format must be BSK_FP8_E4M3 or BSK_FP8_E5M2 (got %d)", format);
    if (out_type != BSK_OUT_F32 && out_type != BSK_OUT_BF16)
        return fail(BSK_ERR_INVALID_ARG, "out_type must be BSK_OUT_F32 or BSK_OUT_BF16 (got %d)", out_type);
    if (!std::isfinite(alpha)) return fail(BSK_ERR_INVALID_ARG, "alpha must be finite");
    if (lda < (K > 1 ? K : 1) || ldb < (K > 1 ? K : 1) || ldc < (M > 1 ? M : 1))
        return fail(BSK_ERR_INVALID_ARG, "leading dimension too small (lda=%d ldb=%d ldc=%d for M=%d N=%d K=%d)", lda,
                    ldb, ldc, M, N, K);
    if (M == 0 || N == 0) return BSK_OK;
    const size_t ob = out_type == BSK_OUT_F32 ? 4 : 2;
    const size_t a_bytes = static_cast<size_t>(span_elems(K, M, lda));
    const size_t b_bytes = static_cast<size_t>(span_elems(K, N, ldb));
    const size_t c_bytes = static_cast<size_t>(span_elems(M, N, ldc)) * ob;
    if (C == nullptr) return fail(BSK_ERR_INVALID_ARG, "C is NULL");
    if (K > 0 && (A == nullptr || B == nullptr)) return fail(BSK_ERR_INVALID_ARG, "A or B is NULL");
    if (overlaps(C, c_bytes, A, K > 0 ? a_bytes : 0) || overlaps(C, c_bytes, B, K > 0 ? b_bytes : 0))
        return fail(BSK_ERR_INVALID_ARG, "C overlaps an input");
    const long long tiles = ((M + 127LL) / 128) * ((N + 127LL) / 128);
    if (tiles > INT_MAX) return fail(BSK_ERR_INVALID_ARG, "problem too large (%lld tiles)", tiles);
    int sms = 0;
    int st = prepare_device(&sms);
    if (st != BSK_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (K == 0) {
        cudaError_t e = cudaMemset2DAsync(C, static_cast<size_t>(ldc) * ob, 0, static_cast<size_t>(M) * ob, N, s);
        return e == cudaSuccess ? BSK_OK : fail_cuda(e, "cudaMemset2DAsync");
    }
    GemmOp op;
    op.A = A;
    op.lda = lda;
    op.a_mn_major = false;
    op.B = B;
    op.ldb = ldb;
    op.b_mn_major = false;
    op.C = C;
    op.ldc = ldc;
    op.M = M;
    op.N = N;
    op.K = K;
    op.in_type = format == BSK_FP8_E5M2 ? bsk::kInE5M2 : bsk::kInE4M3;
    op.out_type = out_type == BSK_OUT_F32 ? bsk::kOutF32 : bsk::kOutBF16;
    op.alpha = alpha;
    return run_gemm(op, sms, s);
}

int enqueue_gemm_f16(const uint16_t* A, const uint16_t* B, uint16_t* C, int M, int N, int K, void* stream)
{
    return enqueue_gemm_general(0, 0, A, M > 1 ? M : 1, B, K > 1 ? K : 1, C, M > 1 ? M : 1, M, N, K, nullptr, 0,
                                stream);
}

int enqueue_gemv_bf16(const uint16_t* W, const uint16_t* x, uint16_t* y, int M, int K, int n, void* stream)
{
    if (M < 0 || K < 0 || n < 0) return fail(BSK_ERR_INVALID_ARG, "negative size (M=%d K=%d n=%d)", M, K, n);
    if (M == 0 || n == 0) return BSK_OK;
    const size_t w_bytes = static_cast<size_t>(M) * K * 2, x_bytes = static_cast<size_t>(n) * K * 2;
    const size_t y_bytes = static_cast<size_t>(n) * M * 2;
    if (y == nullptr) return fail(BSK_ERR_INVALID_ARG, "y is NULL");
    if (K > 0 && (W == nullptr || x == nullptr)) return fail(BSK_ERR_INVALID_ARG, "W or x is NULL");
    if (overlaps(y, y_bytes, W, w_bytes) || overlaps(y, y_bytes, x, x_bytes))
        return fail(BSK_ERR_INVALID_ARG, "y overlaps an input");
    const long long tiles = ((M + 127LL) / 128) * ((n + 127LL) / 128);
    if (tiles > INT_MAX) return fail(BSK_ERR_INVALID_ARG, "problem too large (%lld tiles)", tiles);
    int sms = 0;
    int st = prepare_device(&sms);
    if (st != BSK_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (K == 0) {
        cudaError_t e = cudaMemsetAsync(y, 0, y_bytes, s);
        return e == cudaSuccess ? BSK_OK : fail_cuda(e, "cudaMemsetAsync");
    }
    // n <= 3: the CUDA-core GEMV.  From n = 4 on the tensor-core skinny GEMM
    // (128 x 32 tiles, deep TMA ring) streams W faster: the CUDA-core kernels
    // become FMA- and issue-bound as the token count grows.  Measured on GB300 at
    // 34816 x 5120 in chains of back-to-back launches: n = 3 56.0 vs 57.9 us,
    // n = 4 59.5 vs 57.7 us (best CUDA-core configuration vs tensor cores),
    // n = 8 75.0 vs 57.4 us.
    const long long gemv_kernel = opt_or(BSK_OPT_GEMV_KERNEL, 0);
    const bool cuda_core = n <= 8 && (gemv_kernel == 0 ? n <= 3 : gemv_kernel != 5);
    if (cuda_core) {
        bsk::GemvLaunch g;
        g.W = W;
        g.x = x;
        g.y = y;
        g.M = M;
        g.K = K;
        g.n = n;
        g.rows_per_warp = static_cast<int>(opt_or(BSK_OPT_GEMV_ROWS, 0));
        g.warps_per_block = static_cast<int>(opt_or(BSK_OPT_GEMV_WARPS, 0));
        g.kernel = static_cast<int>(opt_or(BSK_OPT_GEMV_KERNEL, 0));
        g.num_sms = sms;
        g.pdl = opt_or(BSK_OPT_PDL, 0) != 1;
        char msg[512] = "";
        if (bsk::launch_gemv(g, s, msg, sizeof(msg))) return fail(BSK_ERR_CUDA, "%s", msg);
        return BSK_OK;
    }
    // Prefill: Y^T (M x n, column-major == y row-major) = W (K-major) * x^T (K-major).
    GemmOp op;
    op.A = W;
    op.lda = K;
    op.a_mn_major = false;
    op.B = x;
    op.ldb = K;
    op.b_mn_major = false;
    op.C = y;
    op.ldc = M;
    op.M = M;
    op.N = n;
    op.K = K;
    op.in_type = bsk::kInBF16;
    op.out_type = bsk::kOutBF16;
    return run_gemm(op, sms, s);
}

int enqueue_decode_attention(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                             const int32_t* block_tables, const int32_t* seq_lens, uint16_t* out, int num_seqs,
                             int num_q_heads, int num_kv_heads, int head_dim, int block_size, int max_blocks,
                             int num_blocks, int max_seq_len, float softmax_scale, int num_segments, void* stream)
{
    if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || block_size <= 0 || max_blocks <= 0 ||
        num_blocks <= 0 || max_seq_len < 0)
        return fail(BSK_ERR_INVALID_ARG, "bad attention sizes (seqs=%d q_heads=%d kv_heads=%d block_size=%d "
                    "max_blocks=%d num_blocks=%d max_seq_len=%d)", num_seqs, num_q_heads, num_kv_heads, block_size,
                    max_blocks, num_blocks, max_seq_len);
    if (num_q_heads % num_kv_heads != 0)
        return fail(BSK_ERR_INVALID_ARG, "num_q_heads (%d) is not a multiple of num_kv_heads (%d)", num_q_heads,
                    num_kv_heads);
    if (num_seqs > 65535 || num_kv_heads > 65535)
        return fail(BSK_ERR_INVALID_ARG, "num_seqs and num_kv_heads must be at most 65535");
    const int group = num_q_heads / num_kv_heads;
    if (group != 1 && group != 2 && group != 4 && group != 8)
        return fail(BSK_ERR_INVALID_ARG, "query heads per KV head must be 1, 2, 4 or 8 (got %d)", group);
    if (head_dim != 64 && head_dim != 128 && head_dim != 256)
        return fail(BSK_ERR_INVALID_ARG, "head_dim must be 64, 128 or 256 (got %d)", head_dim);
    if (static_cast<long long>(max_seq_len) > static_cast<long long>(max_blocks) * block_size)
        return fail(BSK_ERR_INVALID_ARG, "max_seq_len %d exceeds max_blocks * block_size", max_seq_len);
    if (num_segments < 0 || num_segments > 1024)
        return fail(BSK_ERR_INVALID_ARG, "num_segments %d out of range (0 = automatic, else 1..1024)", num_segments);
    if (!(softmax_scale == softmax_scale) || softmax_scale == INFINITY || softmax_scale == -INFINITY)
        return fail(BSK_ERR_INVALID_ARG, "softmax_scale must be finite");
    if (num_seqs == 0) return BSK_OK;
    if (!q || !k_cache || !v_cache || !block_tables || !seq_lens || !out)
        return fail(BSK_ERR_INVALID_ARG, "a pointer argument is NULL");
    const size_t row_align = static_cast<size_t>(head_dim) * 2 / 32;   // bytes each lane loads
    const uintptr_t mask = row_align - 1;
    if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k_cache) |
         reinterpret_cast<uintptr_t>(v_cache)) & mask)
        return fail(BSK_ERR_INVALID_ARG, "q, k_cache and v_cache must be %zu-byte aligned", row_align);
    const size_t q_bytes = static_cast<size_t>(num_seqs) * num_q_heads * head_dim * 2;
    const size_t cache_bytes = static_cast<size_t>(num_blocks) * block_size * num_kv_heads * head_dim * 2;
    if (overlaps(out, q_bytes, q, q_bytes) || overlaps(out, q_bytes, k_cache, cache_bytes) ||
        overlaps(out, q_bytes, v_cache, cache_bytes))
        return fail(BSK_ERR_INVALID_ARG, "out overlaps an input");
    int sms = 0;
    int st = prepare_device(&sms);
    if (st != BSK_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // Segments: as given (16 / 32 is the page's rule for its 80-CU part), else enough
    // CTAs for about two per SM on this GPU, each segment at least 64 tokens long.
    int segs = num_segments;
    if (segs <= 0) {
        const long long heads = static_cast<long long>(num_seqs) * num_kv_heads;
        // one full wave of the split kernel: as many CTAs as fit on the SMs
        const long long per_sm = bsk::attention_ctas_per_sm(head_dim, num_q_heads / num_kv_heads);
        long long want = (per_sm * sms + heads - 1) / heads;
        const long long cap = (max_seq_len + 63) / 64;
        if (want > cap) want = cap;
        if (want < 1) want = 1;
        if (want > 1024) want = 1024;
        segs = static_cast<int>(want);
    }
    Workspace ws;
    const size_t ws_bytes = static_cast<size_t>(num_seqs) * num_q_heads * segs * (head_dim + 2) * sizeof(float);
    st = alloc_workspace(ws, ws_bytes, s);
    if (st != BSK_OK) return st;
    bsk::AttnLaunch a;
    a.q = q;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.block_tables = block_tables;
    a.seq_lens = seq_lens;
    a.out = out;
    a.workspace = static_cast<float*>(ws.ptr);
    a.num_seqs = num_seqs;
    a.num_q_heads = num_q_heads;
    a.num_kv_heads = num_kv_heads;
    a.head_dim = head_dim;
    a.block_size = block_size;
    a.max_blocks = max_blocks;
    a.num_blocks = num_blocks;
    a.max_seq_len = max_seq_len;
    a.num_segments = segs;
    a.scale = softmax_scale;
    a.status = g_status_dev;
    a.pdl = opt_or(BSK_OPT_PDL, 0) != 1;
    char msg[512] = "";
    if (bsk::launch_decode_attention(a, s, msg, sizeof(msg))) return fail(BSK_ERR_CUDA, "%s", msg);
    return BSK_OK;
}

// ---------------------------------------------------------------------------
// Entry points on host buffers.  The library copies the operands to the
// device, computes and copies the result back in blocks, so that the copy of
// one block in, the computation of the block before it and the copy of the
// block before that out run at the same time, on three streams: host ->
// device, the caller's stream, device -> host.  The link between host and
// device is the bound of such a call; the blocks hide the computation and the
// copy back behind the copy in.
// ---------------------------------------------------------------------------
class HostPipe {
  public:
    HostPipe() = default;
    HostPipe(const HostPipe&) = delete;
    HostPipe& operator=(const HostPipe&) = delete;
    ~HostPipe()
    {
        for (cudaEvent_t e : events_) cudaEventDestroy(e);
        if (in_ != nullptr) cudaStreamDestroy(in_);
        if (out_ != nullptr) cudaStreamDestroy(out_);
    }
    int init()
    {
        cudaError_t e = cudaStreamCreateWithFlags(&in_, cudaStreamNonBlocking);
        if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&out_, cudaStreamNonBlocking);
        return e == cudaSuccess ? BSK_OK : fail_cuda(e, "cudaStreamCreateWithFlags");
    }
    cudaStream_t in() const { return in_; }
    cudaStream_t out() const { return out_; }
    // Makes `waiter` wait for the work enqueued on `from` so far.
    int order(cudaStream_t from, cudaStream_t waiter)
    {
        cudaEvent_t ev = nullptr;
        cudaError_t e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
        if (e != cudaSuccess) return fail_cuda(e, "cudaEventCreateWithFlags");
        events_.push_back(ev);
        if ((e = cudaEventRecord(ev, from)) != cudaSuccess) return fail_cuda(e, "cudaEventRecord");
        if ((e = cudaStreamWaitEvent(waiter, ev, 0)) != cudaSuccess) return fail_cuda(e, "cudaStreamWaitEvent");
        return BSK_OK;
    }

  private:
    cudaStream_t in_ = nullptr, out_ = nullptr;
    std::vector<cudaEvent_t> events_;
};

// Device memory of the host-buffer calls: a memory pool of the library's per
// device (not the caller's default pool) that keeps up to kHostPoolKeep bytes
// mapped between calls, so that a call does not map fresh memory each time.
constexpr unsigned long long kHostPoolKeep = 2ull << 30;

int host_pool(cudaMemPool_t* out)
{
    static std::mutex mu;
    static cudaMemPool_t pools[bsk::SmemOptIn::kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail_cuda(e, "cudaGetDevice");
    if (dev < 0 || dev >= bsk::SmemOptIn::kMaxDevices) return fail(BSK_ERR_UNSUPPORTED_DEVICE, "device %d", dev);
    std::lock_guard<std::mutex> lock(mu);
    if (pools[dev] == nullptr) {
        cudaMemPoolProps props = {};
        props.allocType = cudaMemAllocationTypePinned;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = dev;
        cudaMemPool_t pool = nullptr;
        if ((e = cudaMemPoolCreate(&pool, &props)) != cudaSuccess) return fail_cuda(e, "cudaMemPoolCreate");
        unsigned long long keep = kHostPoolKeep;
        if ((e = cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep)) != cudaSuccess) {
            cudaMemPoolDestroy(pool);
            return fail_cuda(e, "cudaMemPoolSetAttribute");
        }
        pools[dev] = pool;
    }
    *out = pools[dev];
    return BSK_OK;
}

int alloc_host_call_workspace(Workspace& ws, size_t bytes, cudaStream_t s)
{
    cudaMemPool_t pool = nullptr;
    int st = host_pool(&pool);
    if (st != BSK_OK) return st;
    ws.s = s;
    cudaError_t e = cudaMallocFromPoolAsync(&ws.ptr, bytes, pool, s);
    if (e != cudaSuccess) {
        cudaGetLastError();
        ws.ptr = nullptr;
        return fail(BSK_ERR_NO_MEMORY, "cudaMallocFromPoolAsync(%zu bytes) failed: %s", bytes, cudaGetErrorString(e));
    }
    return BSK_OK;
}

// Blocks of a streamed operand of `bytes`: about 32 MB each, 1 to 16 (measured on
// GB300: 32 MB blocks 7.5% faster than 64 MB on the 8192^2 x 16384 GEMM, whose
// last block's compute and copy back are the part the copies in cannot hide).
int pipe_blocks(size_t bytes)
{
    const size_t per = 32ull << 20;
    const size_t b = (bytes + per - 1) / per;
    return static_cast<int>(b < 1 ? 1 : (b > 16 ? 16 : b));
}

// C = A B (column-major FP16, as gemm_f16_colmajor) on host buffers: A goes
// to the device first, then B and C in column blocks (a column block of a
// column-major matrix is one contiguous range).
int run_gemm_f16_host(const uint16_t* A, const uint16_t* B, uint16_t* C, int M, int N, int K, cudaStream_t s)
{
    if (M < 0 || N < 0 || K < 0) return fail(BSK_ERR_INVALID_ARG, "negative size (M=%d N=%d K=%d)", M, N, K);
    if (M == 0 || N == 0) return BSK_OK;
    const size_t a_bytes = static_cast<size_t>(M) * K * 2, b_bytes = static_cast<size_t>(K) * N * 2;
    const size_t c_bytes = static_cast<size_t>(M) * N * 2;
    if (C == nullptr) return fail(BSK_ERR_INVALID_ARG, "C is NULL");
    if (K > 0 && (A == nullptr || B == nullptr)) return fail(BSK_ERR_INVALID_ARG, "A or B is NULL");
    if (K > 0 && (overlaps(C, c_bytes, A, a_bytes) || overlaps(C, c_bytes, B, b_bytes)))
        return fail(BSK_ERR_INVALID_ARG, "C overlaps an input");
    if (K == 0) {   // the empty sum
        std::memset(C, 0, c_bytes);
        return BSK_OK;
    }
    int sms = 0;
    int st = prepare_device(&sms);
    if (st != BSK_OK) return st;
    const size_t a_pad = (a_bytes + 255) / 256 * 256, b_pad = (b_bytes + 255) / 256 * 256;
    Workspace ws;
    if ((st = alloc_host_call_workspace(ws, a_pad + b_pad + c_bytes, s)) != BSK_OK) return st;
    uint8_t* base = static_cast<uint8_t*>(ws.ptr);
    uint16_t* dA = reinterpret_cast<uint16_t*>(base);
    uint16_t* dB = reinterpret_cast<uint16_t*>(base + a_pad);
    uint16_t* dC = reinterpret_cast<uint16_t*>(base + a_pad + b_pad);
    HostPipe hp;
    if ((st = hp.init()) != BSK_OK) return st;
    // the copies start after the caller's earlier work on `s` (which may be
    // writing the host buffers) and after the workspace allocation
    if ((st = hp.order(s, hp.in())) != BSK_OK || (st = hp.order(s, hp.out())) != BSK_OK) return st;
    cudaError_t e = cudaMemcpyAsync(dA, A, a_bytes, cudaMemcpyHostToDevice, hp.in());
    if (e != cudaSuccess) return fail_cuda(e, "cudaMemcpyAsync(A)");
    const int blocks = pipe_blocks(b_bytes);
    const long long nb = ((static_cast<long long>(N) + blocks - 1) / blocks + 255) / 256 * 256;
    for (long long n0 = 0; n0 < N && st == BSK_OK; n0 += nb) {
        const long long n1 = n0 + nb < N ? n0 + nb : N;
        e = cudaMemcpyAsync(dB + n0 * K, B + n0 * K, static_cast<size_t>(n1 - n0) * K * 2, cudaMemcpyHostToDevice,
                            hp.in());
        if (e != cudaSuccess) {
            st = fail_cuda(e, "cudaMemcpyAsync(B block)");
            break;
        }
        if ((st = hp.order(hp.in(), s)) != BSK_OK) break;
        st = enqueue_gemm_general(0, 0, dA, M, dB + n0 * K, K, dC + n0 * M, M, M, static_cast<int>(n1 - n0), K,
                                  nullptr, 0, s);
        if (st != BSK_OK) break;
        if ((st = hp.order(s, hp.out())) != BSK_OK) break;
        e = cudaMemcpyAsync(C + n0 * M, dC + n0 * M, static_cast<size_t>(n1 - n0) * M * 2, cudaMemcpyDeviceToHost,
                            hp.out());
        if (e != cudaSuccess) st = fail_cuda(e, "cudaMemcpyAsync(C block)");
    }
    // join both copy streams before the workspace is released and the call returns
    const int j1 = hp.order(hp.in(), s), j2 = hp.order(hp.out(), s);
    ws.release();
    const int sync = sync_and_check(s);
    if (st != BSK_OK) return st;
    if (j1 != BSK_OK) return j1;
    if (j2 != BSK_OK) return j2;
    return sync;
}

// y = x W^T (BF16, as gemv_bf16) on host buffers: x goes to the device first,
// then W in row blocks; each block's outputs (n rows of its width) come back
// with one strided copy into y.
int run_gemv_bf16_host(const uint16_t* W, const uint16_t* x, uint16_t* y, int M, int K, int n, cudaStream_t s)
{
    if (M < 0 || K < 0 || n < 0) return fail(BSK_ERR_INVALID_ARG, "negative size (M=%d K=%d n=%d)", M, K, n);
    if (M == 0 || n == 0) return BSK_OK;
    const size_t w_bytes = static_cast<size_t>(M) * K * 2, x_bytes = static_cast<size_t>(n) * K * 2;
    const size_t y_bytes = static_cast<size_t>(n) * M * 2;
    if (y == nullptr) return fail(BSK_ERR_INVALID_ARG, "y is NULL");
    if (K > 0 && (W == nullptr || x == nullptr)) return fail(BSK_ERR_INVALID_ARG, "W or x is NULL");
    if (K > 0 && (overlaps(y, y_bytes, W, w_bytes) || overlaps(y, y_bytes, x, x_bytes)))
        return fail(BSK_ERR_INVALID_ARG, "y overlaps an input");
    if (K == 0) {   // the empty sum
        std::memset(y, 0, y_bytes);
        return BSK_OK;
    }
    int sms = 0;
    int st = prepare_device(&sms);
    if (st != BSK_OK) return st;
    const size_t w_pad = (w_bytes + 255) / 256 * 256, x_pad = (x_bytes + 255) / 256 * 256;
    Workspace ws;
    if ((st = alloc_host_call_workspace(ws, w_pad + x_pad + y_bytes, s)) != BSK_OK) return st;
    uint8_t* base = static_cast<uint8_t*>(ws.ptr);
    uint16_t* dW = reinterpret_cast<uint16_t*>(base);
    uint16_t* dx = reinterpret_cast<uint16_t*>(base + w_pad);
    uint16_t* dy = reinterpret_cast<uint16_t*>(base + w_pad + x_pad);
    HostPipe hp;
    if ((st = hp.init()) != BSK_OK) return st;
    if ((st = hp.order(s, hp.in())) != BSK_OK || (st = hp.order(s, hp.out())) != BSK_OK) return st;
    cudaError_t e = cudaMemcpyAsync(dx, x, x_bytes, cudaMemcpyHostToDevice, hp.in());
    if (e != cudaSuccess) return fail_cuda(e, "cudaMemcpyAsync(x)");
    const int blocks = pipe_blocks(w_bytes);
    const long long mb = ((static_cast<long long>(M) + blocks - 1) / blocks + 127) / 128 * 128;
    for (long long m0 = 0; m0 < M && st == BSK_OK; m0 += mb) {
        const long long m1 = m0 + mb < M ? m0 + mb : M;
        const long long rows = m1 - m0;
        e = cudaMemcpyAsync(dW + m0 * K, W + m0 * K, static_cast<size_t>(rows) * K * 2, cudaMemcpyHostToDevice,
                            hp.in());
        if (e != cudaSuccess) {
            st = fail_cuda(e, "cudaMemcpyAsync(W block)");
            break;
        }
        if ((st = hp.order(hp.in(), s)) != BSK_OK) break;
        // this block's outputs, n x rows, contiguous at dy + n * m0
        uint16_t* dyb = dy + static_cast<long long>(n) * m0;
        if ((st = enqueue_gemv_bf16(dW + m0 * K, dx, dyb, static_cast<int>(rows), K, n, s)) != BSK_OK) break;
        if ((st = hp.order(s, hp.out())) != BSK_OK) break;
        e = cudaMemcpy2DAsync(y + m0, static_cast<size_t>(M) * 2, dyb, static_cast<size_t>(rows) * 2,
                              static_cast<size_t>(rows) * 2, static_cast<size_t>(n), cudaMemcpyDeviceToHost, hp.out());
        if (e != cudaSuccess) st = fail_cuda(e, "cudaMemcpy2DAsync(y block)");
    }
    const int j1 = hp.order(hp.in(), s), j2 = hp.order(hp.out(), s);
    ws.release();
    const int sync = sync_and_check(s);
    if (st != BSK_OK) return st;
    if (j1 != BSK_OK) return j1;
    if (j2 != BSK_OK) return j2;
    return sync;
}

}  // namespace

namespace bsk {

size_t gemm_f16_colmajor_pack_bytes(const uint16_t* A, const uint16_t* B, int M, int N, int K)
{
    if (M <= 0 || N <= 0 || K <= 0) return 0;
    const PackPlan pp = plan_pack(colmajor_op(A, B, nullptr, M, N, K));
    return pp.a_bytes + pp.b_bytes;
}

int enqueue_gemm_f16_colmajor_fixed(const uint16_t* A, const uint16_t* B, uint16_t* C, int M, int N, int K,
                                    const FixedScratch& scratch, cudaStream_t stream)
{
    return enqueue_gemm_general(0, 0, A, M > 1 ? M : 1, B, K > 1 ? K : 1, C, M > 1 ? M : 1, M, N, K, nullptr, 0,
                                stream, &scratch);
}

void record_error(const char* msg)
{
    snprintf(t_err, sizeof(t_err), "%s", msg);
}

TmapEncodeFn tmap_encoder()
{
    static TmapEncodeFn fn = []() -> TmapEncodeFn {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        return reinterpret_cast<TmapEncodeFn>(p);
    }();
    return fn;
}

}  // namespace bsk

extern "C" {

int gemm_f16_colmajor(const uint16_t* A, const uint16_t* B, uint16_t* C, int M, int N, int K, void* stream)
{
    int st = enqueue_gemm_f16(A, B, C, M, N, K, stream);
    if (st != BSK_OK) return st;
    if (M == 0 || N == 0) return BSK_OK;
    return sync_and_check(static_cast<cudaStream_t>(stream));
}

int gemv_bf16(const uint16_t* W, const uint16_t* x, uint16_t* y, int M, int K, int n, void* stream)
{
    int st = enqueue_gemv_bf16(W, x, y, M, K, n, stream);
    if (st != BSK_OK) return st;
    if (M == 0 || n == 0) return BSK_OK;
    return sync_and_check(static_cast<cudaStream_t>(stream));
}

int gemm_f16(int order, int transa, int transb, const uint16_t* A, int lda, const uint16_t* B, int ldb,
             uint16_t* C, int ldc, int M, int N, int K, const uint16_t* bias, int bias_mode, void* stream)
{
    int st = enqueue_gemm_f16_cblas(order, transa, transb, A, lda, B, ldb, C, ldc, M, N, K, bias, bias_mode, stream);
    if (st != BSK_OK) return st;
    if (M == 0 || N == 0) return BSK_OK;
    return sync_and_check(static_cast<cudaStream_t>(stream));
}

int bsk_gemm_f16_enqueue(int order, int transa, int transb, const uint16_t* A, int lda, const uint16_t* B,
                         int ldb, uint16_t* C, int ldc, int M, int N, int K, const uint16_t* bias, int bias_mode,
                         void* stream)
{
    return enqueue_gemm_f16_cblas(order, transa, transb, A, lda, B, ldb, C, ldc, M, N, K, bias, bias_mode, stream);
}

int gemm_fp8(int format, const uint8_t* A, int lda, const uint8_t* B, int ldb, void* C, int ldc, int out_type,
             int M, int N, int K, float alpha, void* stream)
{
    int st = enqueue_gemm_fp8(format, A, lda, B, ldb, C, ldc, out_type, M, N, K, alpha, stream);
    if (st != BSK_OK) return st;
    if (M == 0 || N == 0) return BSK_OK;
    return sync_and_check(static_cast<cudaStream_t>(stream));
}

int bsk_gemm_fp8_enqueue(int format, const uint8_t* A, int lda, const uint8_t* B, int ldb, void* C, int ldc,
                         int out_type, int M, int N, int K, float alpha, void* stream)
{
    return enqueue_gemm_fp8(format, A, lda, B, ldb, C, ldc, out_type, M, N, K, alpha, stream);
}

int bsk_gemm_f16_colmajor_enqueue(const uint16_t* A, const uint16_t* B, uint16_t* C, int M, int N, int K,
                                  void* stream)
{
    return enqueue_gemm_f16(A, B, C, M, N, K, stream);
}

int bsk_gemv_bf16_enqueue(const uint16_t* W, const uint16_t* x, uint16_t* y, int M, int K, int n, void* stream)
{
    return enqueue_gemv_bf16(W, x, y, M, K, n, stream);
}

int gemm_f16_colmajor_host(const uint16_t* A, const uint16_t* B, uint16_t* C, int M, int N, int K, void* stream)
{
    return run_gemm_f16_host(A, B, C, M, N, K, static_cast<cudaStream_t>(stream));
}

int gemv_bf16_host(const uint16_t* W, const uint16_t* x, uint16_t* y, int M, int K, int n, void* stream)
{
    return run_gemv_bf16_host(W, x, y, M, K, n, static_cast<cudaStream_t>(stream));
}

int decode_attention_bf16(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                          const int32_t* block_tables, const int32_t* seq_lens, uint16_t* out, int num_seqs,
                          int num_q_heads, int num_kv_heads, int head_dim, int block_size, int max_blocks,
                          int num_blocks, int max_seq_len, float softmax_scale, int num_segments, void* stream)
{
    int st = enqueue_decode_attention(q, k_cache, v_cache, block_tables, seq_lens, out, num_seqs, num_q_heads,
                                      num_kv_heads, head_dim, block_size, max_blocks, num_blocks, max_seq_len,
                                      softmax_scale, num_segments, stream);
    if (st != BSK_OK || num_seqs == 0) return st;
    return sync_and_check(static_cast<cudaStream_t>(stream));
}

int bsk_decode_attention_bf16_enqueue(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                                      const int32_t* block_tables, const int32_t* seq_lens, uint16_t* out,
                                      int num_seqs, int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                      int max_blocks, int num_blocks, int max_seq_len, float softmax_scale,
                                      int num_segments, void* stream)
{
    return enqueue_decode_attention(q, k_cache, v_cache, block_tables, seq_lens, out, num_seqs, num_q_heads,
                                    num_kv_heads, head_dim, block_size, max_blocks, num_blocks, max_seq_len,
                                    softmax_scale, num_segments, stream);
}

int bsk_stream_check(void* stream)
{
    return sync_and_check(static_cast<cudaStream_t>(stream));
}

const char* bsk_last_error(void) { return t_err; }

const char* bsk_status_string(int status)
{
    switch (status) {
    case BSK_OK: return "BSK_OK";
    case BSK_ERR_INVALID_ARG: return "BSK_ERR_INVALID_ARG";
    case BSK_ERR_UNSUPPORTED_DEVICE: return "BSK_ERR_UNSUPPORTED_DEVICE";
    case BSK_ERR_CUDA: return "BSK_ERR_CUDA";
    case BSK_ERR_TIMEOUT: return "BSK_ERR_TIMEOUT";
    case BSK_ERR_NO_MEMORY: return "BSK_ERR_NO_MEMORY";
    default: return "BSK_ERR_UNKNOWN";
    }
}

int bsk_version(void) { return kVersion; }

void bsk_tile_coord(int t, int num_m, int num_n, int group_m, int* pid_m, int* pid_n)
{
    int pm = -1, pn = -1;
    if (num_m > 0 && num_n > 0 && group_m > 0 && t >= 0 && static_cast<long long>(num_m) * num_n > t)
        bsk::tile_coord(t, num_m, num_n, group_m, &pm, &pn);
    if (pid_m) *pid_m = pm;
    if (pid_n) *pid_n = pn;
}

int bsk_plan_gemm(int M, int N, int K, int a_mn_major, int b_mn_major, int fp8, int sms, int* plan)
{
    if (plan == nullptr || M < 1 || N < 1 || K < 1 || sms < 2)
        return fail(BSK_ERR_INVALID_ARG, "plan query: sizes and SM count must be positive (sms >= 2), plan non-NULL");
    GemmOp op;
    op.M = M;
    op.N = N;
    op.K = K;
    op.a_mn_major = a_mn_major != 0;
    op.b_mn_major = b_mn_major != 0;
    op.in_type = fp8 ? bsk::kInE4M3 : bsk::kInF16;
    op.out_type = fp8 ? bsk::kOutBF16 : bsk::kOutF16;
    const GemmPlan p = plan_gemm(op, sms);
    plan[0] = p.block_n;
    plan[1] = p.block_m;
    plan[2] = p.pair ? 1 : 0;
    plan[3] = p.stream_k ? 1 : 0;
    plan[4] = p.skc;
    plan[5] = p.pair_m;
    plan[6] = p.dyn ? 1 : 0;
    return BSK_OK;
}

int bsk_set_option(int key, long long value)
{
    if (key < 1 || key >= kNumOpts) return fail(BSK_ERR_INVALID_ARG, "unknown option key %d", key);
    bool ok = true;
    switch (key) {
    case BSK_OPT_GROUP_M: ok = value >= 0 && value <= 65536; break;
    case BSK_OPT_BLOCK_N: ok = value == 0 || value == 32 || value == 64 || value == 128 || value == 256; break;
    case BSK_OPT_FORCE_PACK:
    case BSK_OPT_FORCE_DIRECT_STORE: ok = value == 0 || value == 1; break;
    case BSK_OPT_GEMV_ROWS: ok = value == 0 || value == 1 || value == 2 || value == 4 || value == 8; break;
    case BSK_OPT_GEMV_WARPS: ok = value >= 0 && value <= 16; break;
    case BSK_OPT_GEMV_KERNEL: ok = value >= 0 && value <= 5; break;
    case BSK_OPT_GEMM_KERNEL: ok = value >= 0 && value <= 2; break;
    case BSK_OPT_STREAM_K: ok = value >= 0 && value <= 2; break;
    case BSK_OPT_PDL: ok = value == 0 || value == 1; break;
    case BSK_OPT_TILE_SCHED: ok = value >= 0 && value <= 2; break;
    case BSK_OPT_BLOCK_M: ok = value >= 0 && value <= 128 && value % 8 == 0; break;
    case BSK_OPT_SPLIT_K: ok = value == 0 || value == 1 || value == 2 || value == 4 || value == 8 || value == 16; break;
    case BSK_OPT_PREFETCH_KB: ok = value >= 0 && value <= 64; break;
    case BSK_OPT_K_ORDER: ok = value == 0 || value == 1; break;
    case BSK_OPT_PAIR_M: ok = value >= 0 && value <= 2; break;
    case BSK_OPT_WAIT_LIMIT_US: ok = value >= 0 && value <= 60000000; break;
    case BSK_OPT_NUM_SMS: ok = value >= 0 && value <= 100000; break;
    default: ok = false;
    }
    if (!ok) return fail(BSK_ERR_INVALID_ARG, "value %lld out of range for option %d", value, key);
    g_opt[key].store(value, std::memory_order_relaxed);
    return BSK_OK;
}

long long bsk_get_option(int key)
{
    if (key < 1 || key >= kNumOpts) return -1;
    return g_opt[key].load(std::memory_order_relaxed);
}

int bsk_test_wait_timeout(unsigned int limit_us, void* stream)
{
    if (limit_us < 1 || limit_us > 10000000u) return fail(BSK_ERR_INVALID_ARG, "limit_us out of range");
    int sms = 0;
    int st = prepare_device(&sms);
    if (st != BSK_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    st = sync_and_check(s);   // start from a clean status word
    if (st != BSK_OK) return st;
    char msg[512] = "";
    if (bsk::launch_wait_timeout_probe(g_status_dev, static_cast<unsigned long long>(limit_us) * 1000ull, s, msg,
                                       sizeof(msg)))
        return fail(BSK_ERR_CUDA, "%s", msg);
    return sync_and_check(s);
}

}  // extern "C"
