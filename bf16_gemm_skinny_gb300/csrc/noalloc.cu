// noalloc.cu -- gemm_f16_colmajor_noalloc: the column-major FP16 GEMM for
// callers that must not allocate device memory at call time.
//
// Who needs it: a serving process that reserves all free HBM for weights and
// KV cache when it starts (its own allocator owns every byte, so a
// cudaMalloc/cudaMallocAsync inside a library call would fail or fragment
// that reservation), and programs that run under a hard device-memory budget
// fixed at start-up and forbid allocator traffic afterwards.  The regular
// entry point allocates a stream-ordered workspace whenever it packs an
// operand (base not 16-byte aligned, or leading dimension not a multiple of 8
// elements) or runs the stream-K schedule (FP32 partials and flags); this
// variant takes that workspace from a fixed array that is part of the library
// image instead, and calls no allocating routine.  Everything else -- the
// argument checks, the plan (pack, tile width, kernel, schedule, tuning
// options) and the kernels -- is the regular entry point's, so the two give
// the same result bits for the same call.
//
// The scratch array is a file-scope __device__ variable of kNoAllocScratchBytes
// (96 MiB).  Every GPU that loads this library's device code holds it until
// the process exits.  Calls whose workspace would exceed it are rejected with
// BSK_ERR_INVALID_ARG before any device work; calls with 16-byte-aligned
// operands and leading dimensions need no pack, whatever their size.
//
// All calls of a process share the one array (and the status word below), and
// the array keeps whatever the last call left in it.  Two calls that overlap
// on the GPU (different streams, or different host threads) race on it: issue
// them from one thread or otherwise serialise them.  (The call blocks until
// its stream has finished it, so one thread's calls never overlap.)
//
// Set-up, by the first call on each device (with that device current): the
// device addresses of the scratch array and of the status word are looked up
// with cudaGetSymbolAddress (in host code the variables' names only stand in
// for them), and the device code of every kernel this entry point may launch
// is loaded.  Under CUDA's default lazy module loading that first call is
// where the 96 MiB array and the kernels' code are mapped, so it does take
// device memory once: make it before the caller reserves the device's free
// memory (or set CUDA_MODULE_LOADING=EAGER, which maps them when the library
// is loaded), and before anything else on its stream is being captured.
// Every later call allocates nothing.  The call blocks: it copies the status
// word to the host and synchronises its stream before returning, so it cannot
// be recorded into a CUDA graph.
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdio>
#include <mutex>

#include "bsk.h"
#include "bsk_internal.h"
#include "bsk_tuning.h"

namespace {

constexpr size_t kNoAllocScratchBytes = 96ull << 20;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];
// Device status word of this entry point: a bounded wait that gives up writes
// a nonzero code here.  Cleared before every launch.
static __device__ __align__(16) int g_noalloc_status[4];

struct NoAllocDevice {
    bool ready = false;
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

// Once per device, with that device current: check it, look up the device
// addresses of the scratch array and the status word, and load the kernels'
// device code.
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
            (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess)
            return fail_cuda(e, "cudaDeviceGetAttribute");
        if (!(major == 10 && minor == 3))
            return fail(BSK_ERR_UNSUPPORTED_DEVICE, "device %d has compute capability %d.%d; this library is built for 10.3",
                        dev, major, minor);
        void* p = nullptr;
        if ((e = cudaGetSymbolAddress(&p, g_noalloc_scratch)) != cudaSuccess)
            return fail_cuda(e, "cudaGetSymbolAddress(scratch)");
        d.scratch = static_cast<unsigned char*>(p);
        if ((e = cudaGetSymbolAddress(&p, g_noalloc_status)) != cudaSuccess)
            return fail_cuda(e, "cudaGetSymbolAddress(status word)");
        d.status = static_cast<int*>(p);
        char msg[512] = "";
        if (bsk::preload_gemm_f16_colmajor_kernels(msg, sizeof(msg)) || bsk::preload_aux_kernels(msg, sizeof(msg)))
            return fail(BSK_ERR_CUDA, "%s", msg);
        d.ready = true;
    }
    *out = &d;
    return BSK_OK;
}

}  // namespace

extern "C" int gemm_f16_colmajor_noalloc(const uint16_t* A, const uint16_t* B, uint16_t* C, int M, int N, int K,
                                         void* stream)
{
    if (M < 0 || N < 0 || K < 0) return fail(BSK_ERR_INVALID_ARG, "negative size (M=%d N=%d K=%d)", M, N, K);
    if (M == 0 || N == 0) return BSK_OK;
    // The packed operands alone past the array's size: refused before the
    // device is touched (the regular planner repeats the check with the
    // stream-K partials included).
    const size_t pack = bsk::gemm_f16_colmajor_pack_bytes(A, B, M, N, K);
    if (pack > kNoAllocScratchBytes)
        return fail(BSK_ERR_INVALID_ARG,
                    "gemm_f16_colmajor_noalloc: packing these operands needs %zu bytes of scratch, more than its "
                    "fixed %zu-byte (96 MiB) array; use gemm_f16_colmajor, or pass 16-byte-aligned operands with "
                    "M and K multiples of 8 (no scratch needed)",
                    pack, kNoAllocScratchBytes);

    NoAllocDevice* d = nullptr;
    int st = setup_current_device(&d);
    if (st != BSK_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if ((e = cudaMemsetAsync(d->status, 0, sizeof(int), s)) != cudaSuccess)
        return fail_cuda(e, "cudaMemsetAsync(status word)");
    bsk::FixedScratch scratch;
    scratch.ptr = d->scratch;
    scratch.bytes = kNoAllocScratchBytes;
    scratch.status = d->status;
    st = bsk::enqueue_gemm_f16_colmajor_fixed(A, B, C, M, N, K, scratch, s);
    if (st != BSK_OK) return st;

    int code = 0;
    if ((e = cudaMemcpyAsync(&code, d->status, sizeof(int), cudaMemcpyDeviceToHost, s)) != cudaSuccess)
        return fail_cuda(e, "cudaMemcpyAsync(status word)");
    if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return fail_cuda(e, "cudaStreamSynchronize");
    if (code != 0)
        return fail(BSK_ERR_TIMEOUT, "a device-side wait gave up (site %d); the output is undefined",
                    code - bsk::kDevErrTimeoutBase);
    return BSK_OK;
}
