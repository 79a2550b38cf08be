// noalloc.cu -- gemm_f16_colmajor_noalloc: the column-major FP16 GEMM for
// callers that must not allocate device memory at call time.
//
// Who needs it: a serving process that reserves all free HBM for weights and
// KV cache when it starts (its own allocator owns every byte, so a
// cudaMalloc/cudaMallocAsync inside a library call would fail or fragment
// that reservation), and programs that run under a hard device-memory budget
// fixed at start-up and forbid allocator traffic afterwards.  The regular
// entry point allocates a stream-ordered workspace whenever an operand has
// to be packed (base not 16-byte aligned, or leading dimension not a multiple
// of 8 elements); this variant packs into a fixed array that is part of the
// library image instead, and calls no allocating routine.
//
// The scratch array is a file-scope __device__ variable of kNoAllocScratchBytes
// (96 MiB).  Every GPU that loads this library's device code holds it until
// the process exits.  Calls whose packed operands need more than that are
// rejected with BSK_ERR_INVALID_ARG; calls with 16-byte-aligned operands and
// leading dimensions need no scratch at all, whatever their size.
//
// All calls of a process share the one array (and the status word below), and
// the array keeps whatever the last call left in it.  Two calls that overlap
// on the GPU (different streams, or different host threads) race on it: issue
// them on one stream or otherwise serialise them.
//
// Set-up: the first call on each device resolves the device addresses of the
// scratch array and of the status word with cudaGetSymbolAddress (in host code
// the variables' names only stand in for them).  Make that first call on a
// device before any stream capture begins on it.
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdio>
#include <mutex>

#include "bsk.h"
#include "bsk_internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = 96ull << 20;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];
// Device status word of this entry point: a bounded wait that gives up writes
// a nonzero code here.  Cleared before every launch.
static __device__ __align__(16) int g_noalloc_status[4];

struct NoAllocDevice {
    bool ready = false;
    bool supported = false;
    int sms = 0;
    unsigned char* scratch = nullptr;
    int* status = nullptr;
};

constexpr int kMaxDevices = 128;
std::mutex g_mu;
NoAllocDevice g_devs[kMaxDevices];

int fail(int status, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
int fail(int status, const char* fmt, ...)
{
    char buf[1024];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    bsk::record_error(buf);
    return status;
}

int fail_cuda(cudaError_t e, const char* what)
{
    return fail(BSK_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

// Once per device, with that device current: check it and look up the device
// addresses of the scratch array and the status word.
int setup_current_device(NoAllocDevice** out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail_cuda(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(BSK_ERR_UNSUPPORTED_DEVICE, "device ordinal %d out of range", dev);
    std::lock_guard<std::mutex> lk(g_mu);
    NoAllocDevice& d = g_devs[dev];
    if (!d.ready) {
        int major = 0, minor = 0;
        if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
            return fail_cuda(e, "cudaDeviceGetAttribute");
        d.supported = (major == 10 && minor == 3);
        if (!d.supported)
            return fail(BSK_ERR_UNSUPPORTED_DEVICE, "device %d has compute capability %d.%d; this library is built for 10.3",
                        dev, major, minor);
        void* p = nullptr;
        if ((e = cudaGetSymbolAddress(&p, g_noalloc_scratch)) != cudaSuccess)
            return fail_cuda(e, "cudaGetSymbolAddress(scratch)");
        d.scratch = static_cast<unsigned char*>(p);
        if ((e = cudaGetSymbolAddress(&p, g_noalloc_status)) != cudaSuccess)
            return fail_cuda(e, "cudaGetSymbolAddress(status word)");
        d.status = static_cast<int*>(p);
        d.ready = true;
    }
    if (!d.supported) return fail(BSK_ERR_UNSUPPORTED_DEVICE, "device %d is not compute capability 10.3", dev);
    *out = &d;
    return BSK_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool overlaps(const void* a, size_t abytes, const void* b, size_t bbytes)
{
    if (abytes == 0 || bbytes == 0) return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + bbytes && b0 < a0 + abytes;
}
long long round_up8(long long v) { return (v + 7) / 8 * 8; }

long long option_or(int key, long long dflt)
{
    const long long v = bsk_get_option(key);
    return v > 0 ? v : dflt;
}

}  // namespace

extern "C" int gemm_f16_colmajor_noalloc(const uint16_t* A, const uint16_t* B, uint16_t* C, int M, int N, int K,
                                         void* stream)
{
    if (M < 0 || N < 0 || K < 0) return fail(BSK_ERR_INVALID_ARG, "negative size (M=%d N=%d K=%d)", M, N, K);
    if (M == 0 || N == 0) return BSK_OK;
    const size_t a_bytes = static_cast<size_t>(M) * K * 2, b_bytes = static_cast<size_t>(K) * N * 2;
    const size_t c_bytes = static_cast<size_t>(M) * N * 2;
    if (C == nullptr) return fail(BSK_ERR_INVALID_ARG, "C is NULL");
    if (K > 0 && (A == nullptr || B == nullptr)) return fail(BSK_ERR_INVALID_ARG, "A or B is NULL");
    if (overlaps(C, c_bytes, A, a_bytes) || overlaps(C, c_bytes, B, b_bytes))
        return fail(BSK_ERR_INVALID_ARG, "C overlaps an input");
    const long long tiles = ((M + 127LL) / 128) * ((N + 127LL) / 128);
    if (tiles > 0x7FFFFFFFLL) return fail(BSK_ERR_INVALID_ARG, "problem too large (%lld tiles)", tiles);

    // Scratch needed for packing (same layout as the regular entry point).
    const bool force_pack = bsk_get_option(BSK_OPT_FORCE_PACK) == 1;
    const bool a_ok = !force_pack && aligned16(A) && (M % 8 == 0);
    const bool b_ok = !force_pack && aligned16(B) && (K % 8 == 0);
    const long long lda_p = a_ok ? M : round_up8(M);
    const long long ldb_p = b_ok ? K : round_up8(K);
    size_t a_pack = a_ok || K == 0 ? 0 : static_cast<size_t>(lda_p) * K * 2;
    const size_t b_pack = b_ok || K == 0 ? 0 : static_cast<size_t>(ldb_p) * N * 2;
    a_pack = (a_pack + 255) / 256 * 256;
    if (a_pack + b_pack > kNoAllocScratchBytes)
        return fail(BSK_ERR_INVALID_ARG,
                    "gemm_f16_colmajor_noalloc: packing these operands needs %zu bytes of scratch, more than its "
                    "fixed %zu-byte (96 MiB) array; use gemm_f16_colmajor, or pass 16-byte-aligned operands with "
                    "M and K multiples of 8 (no scratch needed)",
                    a_pack + b_pack, kNoAllocScratchBytes);

    NoAllocDevice* d = nullptr;
    int st = setup_current_device(&d);
    if (st != BSK_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (K == 0) {
        if ((e = cudaMemsetAsync(C, 0, c_bytes, s)) != cudaSuccess) return fail_cuda(e, "cudaMemsetAsync");
        if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return fail_cuda(e, "cudaStreamSynchronize");
        return BSK_OK;
    }
    if ((e = cudaMemsetAsync(d->status, 0, sizeof(int), s)) != cudaSuccess)
        return fail_cuda(e, "cudaMemsetAsync(status word)");

    char msg[512] = "";
    const uint16_t* Ause = A;
    const uint16_t* Buse = B;
    bsk::PackCopy copies[2];
    int n_copies = 0;
    if (!a_ok) {
        uint16_t* Ap = reinterpret_cast<uint16_t*>(d->scratch);
        copies[n_copies++] = {A, M * 2LL, Ap, lda_p * 2LL, M * 2LL, K};
        Ause = Ap;
    }
    if (!b_ok) {
        uint16_t* Bp = reinterpret_cast<uint16_t*>(d->scratch + a_pack);
        copies[n_copies++] = {B, K * 2LL, Bp, ldb_p * 2LL, K * 2LL, N};
        Buse = Bp;
    }
    if (n_copies > 0 && bsk::launch_pack(copies, n_copies, d->sms, option_or(BSK_OPT_PDL, 0) != 1, s, msg,
                                         sizeof(msg)))
        return fail(BSK_ERR_CUDA, "%s", msg);
    bsk::GemmLaunch g;
    g.A = Ause;
    g.lda = lda_p;
    g.a_mn_major = true;
    g.B = Buse;
    g.ldb = ldb_p;
    g.C = C;
    g.ldc = M;
    g.M = M;
    g.N = N;
    g.K = K;
    g.in_type = bsk::kInF16;
    g.out_type = bsk::kOutF16;
    // Tile width: the smallest of 32 / 64 / 128 covering a skinny N (one CTA per
    // tile, deep ring: the weight stream sets the pace), else 256 on CTA pairs.
    const long long bn_opt = option_or(BSK_OPT_BLOCK_N, 0);
    const int bn_auto = N <= 32 ? 32 : N <= 64 ? 64 : N <= 128 ? 128 : 256;
    g.block_n = static_cast<int>(bn_opt > 0 ? bn_opt : bn_auto);
    g.pair = g.block_n == 256 && option_or(BSK_OPT_GEMM_KERNEL, 2) == 2;
    // Tile-row group: measured best on GB300 for 8192^3-class and prefill shapes.
    g.group_m = static_cast<int>(option_or(BSK_OPT_GROUP_M, g.pair && g.block_n == 256 ? 2 : 16));
    g.tma_store = aligned16(C) && (M % 8 == 0) && bsk_get_option(BSK_OPT_FORCE_DIRECT_STORE) != 1;
    const long long cap = option_or(BSK_OPT_NUM_SMS, d->sms);
    g.num_sms = static_cast<int>(cap < d->sms ? cap : d->sms);
    g.status = d->status;
    g.wait_limit_ns = static_cast<unsigned long long>(option_or(BSK_OPT_WAIT_LIMIT_US, 2000000)) * 1000ull;
    g.pdl = option_or(BSK_OPT_PDL, 0) != 1;
    g.dyn = g.pair && option_or(BSK_OPT_TILE_SCHED, 0) == 2;   // tile order on CTA pairs: fixed unless requested
    if (bsk::launch_gemm(g, s, msg, sizeof(msg))) return fail(BSK_ERR_CUDA, "%s", msg);

    int code = 0;
    if ((e = cudaMemcpyAsync(&code, d->status, sizeof(int), cudaMemcpyDeviceToHost, s)) != cudaSuccess)
        return fail_cuda(e, "cudaMemcpyAsync(status word)");
    if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return fail_cuda(e, "cudaStreamSynchronize");
    if (code != 0)
        return fail(BSK_ERR_TIMEOUT, "a device-side wait gave up (site %d); the output is undefined",
                    code - bsk::kDevErrTimeoutBase);
    return BSK_OK;
}
