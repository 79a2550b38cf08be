// aux_kernels.cu -- the operand pack kernel and the bounded-wait test probe.
#include <algorithm>
#include <cstdio>

#include "bsk_internal.h"
#include "ptx.cuh"

namespace bsk {
namespace {

// The 16 bytes that start `m` bytes into `lo` (lo followed by hi, little-endian).
__device__ __forceinline__ uint4 realign16(const uint4& lo, const uint4& hi, unsigned m)
{
    const unsigned r = (m & 3u) * 8u;   // bit shift inside a word
    uint32_t v0, v1, v2, v3, v4;        // words m/4 .. m/4 + 4 of the 32 bytes
    switch (m >> 2) {
    case 0: v0 = lo.x; v1 = lo.y; v2 = lo.z; v3 = lo.w; v4 = hi.x; break;
    case 1: v0 = lo.y; v1 = lo.z; v2 = lo.w; v3 = hi.x; v4 = hi.y; break;
    case 2: v0 = lo.z; v1 = lo.w; v2 = hi.x; v3 = hi.y; v4 = hi.z; break;
    default: v0 = lo.w; v1 = hi.x; v2 = hi.y; v3 = hi.z; v4 = hi.w; break;
    }
    return make_uint4(__funnelshift_r(v0, v1, r), __funnelshift_r(v1, v2, r), __funnelshift_r(v2, v3, r),
                      __funnelshift_r(v3, v4, r));
}

// One operand's copy as the kernel sees it: `lines` lines of line_bytes bytes,
// each cut into `pieces` pieces of piece_bytes (a multiple of 16; the last
// piece of a line may be shorter), numbered line by line: unit u is piece
// u % pieces of line u / pieces.
struct PackJob {
    const uint8_t* src;
    long long ld_src;          // bytes from one source line to the next
    uint8_t* dst;              // 16-byte aligned
    long long ld_dst;          // bytes, a multiple of 16, at least line_bytes rounded up to 16
    long long line_bytes;
    long long piece_bytes;
    long long pieces;          // per line
    long long units;           // pieces x lines
    unsigned blocks;           // CTAs working on this job
};

constexpr int kPackThreads = 256;
constexpr int kPackBufs = 4;                     // pieces in flight per CTA
constexpr int kPackPiece = 8192;                 // longest piece, bytes
constexpr int kPackBufBytes = kPackPiece + 32;   // a piece's aligned cover plus the chunk read past it
constexpr int kPackCtasPerSm = 4;
constexpr int kSitePack = 0x20;                  // wait site reported on a timeout

// dst line l = src line l, byte for byte, for up to two operands in one launch
// (the first j0.blocks CTAs take job 0, the rest job 1).  The TMA needs
// 16-byte aligned bases and leading dimensions; the pack gives unaligned
// operands that shape in a workspace without touching the caller's buffers
// ("MTT S4000 GEMM 优化中的分块、尾处理与并发实战复盘", section 1: inputs may not be modified).
//
// Each CTA takes a contiguous range of units (line pieces).  For each, one
// thread issues a bulk copy of the piece's 16-byte-aligned cover -- from the
// aligned chunk holding its first byte to the end of the chunk holding its
// last, so no byte outside the pages the piece touches is read -- into one of
// kPackBufs shared-memory buffers, completing on that buffer's mbarrier, so
// kPackBufs pieces per CTA are in flight.  Once a piece has landed, thread t
// writes output chunks t, t + 256, ...: chunk c is the 16 bytes that start m
// bytes into buffer chunk c (m = the piece's offset from a 16-byte boundary),
// shifted out of buffer chunks c and c + 1, with one aligned 16-byte store.  A
// line's last chunk may carry up to 15 bytes past the line's end into the
// destination's padding (its leading dimension is rounded up to 16 bytes; the
// GEMM's tensor maps never read the padding).  Every wait is bounded.
__global__ void __launch_bounds__(kPackThreads, kPackCtasPerSm)
    pack_kernel(PackJob j0, PackJob j1, int* status, unsigned long long limit_ns)
{
    __shared__ __align__(128) uint8_t buf[kPackBufs][kPackBufBytes];
    __shared__ __align__(8) uint64_t bars[kPackBufs];
    __shared__ uint32_t abort_flag;
    if (threadIdx.x == 0) {
        for (int i = 0; i < kPackBufs; ++i) mbar_init(smem_u32(&bars[i]), 1);
        abort_flag = 0u;
        fence_mbar_init();
    }
    __syncthreads();
    griddep_wait();               // the source may be the previous kernel's output
    griddep_launch_dependents();  // the GEMM's prologue may start; it waits for this grid's completion
    const bool second = blockIdx.x >= j0.blocks;
    const PackJob& j = second ? j1 : j0;
    const long long b = second ? blockIdx.x - j0.blocks : blockIdx.x;
    const long long u0 = j.units * b / j.blocks;
    const long long n = j.units * (b + 1) / j.blocks - u0;

    // source start, destination start and length of unit u
    auto piece = [&](long long u, const uint8_t*& s, uint8_t*& d, long long& len) {
        const long long line = u / j.pieces;
        const long long off = (u - line * j.pieces) * j.piece_bytes;
        s = j.src + line * j.ld_src + off;
        d = j.dst + line * j.ld_dst + off;
        len = j.line_bytes - off < j.piece_bytes ? j.line_bytes - off : j.piece_bytes;
    };
    // thread 0: unit u0 + i into buffer i % kPackBufs
    auto issue = [&](long long i) {
        const uint8_t* s;
        uint8_t* d;
        long long len;
        piece(u0 + i, s, d, len);
        const uintptr_t a = reinterpret_cast<uintptr_t>(s);
        const uintptr_t lo = a & ~static_cast<uintptr_t>(15);
        const uintptr_t hi = (a + static_cast<uintptr_t>(len) + 15) & ~static_cast<uintptr_t>(15);
        const uint32_t bar = smem_u32(&bars[i % kPackBufs]);
        mbar_arrive_expect_tx(bar, static_cast<uint32_t>(hi - lo));
        bulk_load(smem_u32(buf[i % kPackBufs]), reinterpret_cast<const void*>(lo), static_cast<uint32_t>(hi - lo), bar);
    };
    if (threadIdx.x == 0)
        for (long long i = 0; i < n && i < kPackBufs; ++i) issue(i);

    const WaitCtl wc{&abort_flag, status, limit_ns};
    long long i = 0;
    for (; i < n; ++i) {
        const int bi = static_cast<int>(i % kPackBufs);
        const bool ok = mbar_wait(smem_u32(&bars[bi]), static_cast<uint32_t>(i / kPackBufs) & 1u, wc, kSitePack);
        if (!__syncthreads_and(ok)) break;
        const uint8_t* s;
        uint8_t* d;
        long long len;
        piece(u0 + i, s, d, len);
        const unsigned m = static_cast<unsigned>(reinterpret_cast<uintptr_t>(s) & 15u);
        const uint4* sb = reinterpret_cast<const uint4*>(buf[bi]);
        const unsigned chunks = static_cast<unsigned>((len + 15) / 16);
        for (unsigned c = threadIdx.x; c < chunks; c += kPackThreads) {
            const uint4 lo = sb[c];
            *reinterpret_cast<uint4*>(d + 16ull * c) = m == 0u ? lo : realign16(lo, sb[c + 1], m);
        }
        __syncthreads();   // every thread has read the buffer before it is refilled
        if (threadIdx.x == 0 && i + kPackBufs < n) {
            fence_proxy_async_smem();
            issue(i + kPackBufs);
        }
    }
    if (i < n && threadIdx.x == 0) {
        // abort: the copies issued and not consumed must land before the CTA exits
        uint32_t never = 0u;
        const WaitCtl wc_drain{&never, status, limit_ns};
        const long long issued = n < i + kPackBufs ? n : i + kPackBufs;
        for (long long k = i; k < issued; ++k)
            mbar_wait(smem_u32(&bars[k % kPackBufs]), static_cast<uint32_t>(k / kPackBufs) & 1u, wc_drain, kSitePack);
    }
}

// C(m,n) = bias value (or +0.0) for m < M, n < N, C(m,n) at C[m + n*ldc]: the
// K == 0 case of the GEMM (an empty sum plus the bias, already in the output
// format, so no rounding happens).
__global__ void __launch_bounds__(256)
    fill_bias_kernel(uint16_t* __restrict__ C, long long ldc, int M, int N, const uint16_t* __restrict__ bias,
                     int bias_mode)
{
    const long long total = static_cast<long long>(M) * N;
    const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
    for (long long e = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; e < total; e += stride) {
        const long long n = e / M;
        const long long m = e - n * M;
        uint16_t v = 0;
        if (bias_mode == 1) v = bias[m];
        else if (bias_mode == 2) v = bias[n];
        C[m + n * ldc] = v;
    }
}

// One CTA waits on an mbarrier that nobody arrives on.  The wait is the
// GEMM's bounded wait; it must give up after limit_ns and record a timeout.
__global__ void wait_timeout_probe_kernel(int* status, unsigned long long limit_ns)
{
    __shared__ __align__(8) uint64_t bar;
    __shared__ uint32_t abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        abort_flag = 0u;
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        const WaitCtl wc{&abort_flag, status, limit_ns};
        mbar_wait(smem_u32(&bar), 0u, wc, 0x7F);
    }
    __syncthreads();
}

}  // namespace

int preload_aux_kernels(char* msg, size_t msg_len)
{
    const void* kernels[] = {reinterpret_cast<const void*>(pack_kernel), reinterpret_cast<const void*>(fill_bias_kernel)};
    for (const void* k : kernels) {
        cudaFuncAttributes attr;
        const cudaError_t e = cudaFuncGetAttributes(&attr, k);
        if (e != cudaSuccess) {
            snprintf(msg, msg_len, "cudaFuncGetAttributes (pack/fill kernel): %s", cudaGetErrorString(e));
            return 1;
        }
    }
    return 0;
}

int launch_pack(const PackCopy* copies, int n, int sms, bool pdl, int* status, unsigned long long limit_ns,
                cudaStream_t stream, char* msg, size_t msg_len)
{
    PackJob jobs[2] = {};
    int nj = 0;
    for (int i = 0; i < n; ++i) {
        const PackCopy& c = copies[i];
        if (c.line_bytes <= 0 || c.lines <= 0) continue;
        if (nj == 2) {
            snprintf(msg, msg_len, "pack: at most two copies per launch");
            return 1;
        }
        if ((reinterpret_cast<uintptr_t>(c.dst) & 15u) != 0 || (c.ld_dst & 15) != 0 ||
            c.ld_dst < (c.line_bytes + 15) / 16 * 16) {
            snprintf(msg, msg_len, "pack: destination not 16-byte aligned or its leading dimension too small");
            return 1;
        }
        PackJob& j = jobs[nj++];
        j.src = static_cast<const uint8_t*>(c.src);
        j.ld_src = c.ld_src;
        j.dst = static_cast<uint8_t*>(c.dst);
        j.ld_dst = c.ld_dst;
        j.line_bytes = c.line_bytes;
        // pieces of equal length (multiples of 16), at most kPackPiece bytes each
        j.pieces = (c.line_bytes + kPackPiece - 1) / kPackPiece;
        j.piece_bytes = ((c.line_bytes + j.pieces - 1) / j.pieces + 15) / 16 * 16;
        j.units = j.pieces * c.lines;
    }
    if (nj == 0) return 0;
    // persistent grid, split between the jobs by their bytes (at least one CTA
    // each, no more CTAs than units)
    const unsigned long long total = static_cast<unsigned long long>(sms > 0 ? sms : 1) * kPackCtasPerSm;
    const double w0 = static_cast<double>(jobs[0].line_bytes) * static_cast<double>(jobs[0].units / jobs[0].pieces);
    const double w1 = nj > 1 ? static_cast<double>(jobs[1].line_bytes) * static_cast<double>(jobs[1].units / jobs[1].pieces)
                             : 0.0;
    unsigned long long b0 = nj > 1 ? static_cast<unsigned long long>(static_cast<double>(total) * w0 / (w0 + w1) + 0.5)
                                   : total;
    if (b0 < 1) b0 = 1;
    unsigned long long b1 = nj > 1 ? (total > b0 ? total - b0 : 1ull) : 0ull;
    b0 = std::min<unsigned long long>(b0, static_cast<unsigned long long>(jobs[0].units));
    b1 = std::min<unsigned long long>(b1, nj > 1 ? static_cast<unsigned long long>(jobs[1].units) : 0ull);
    jobs[0].blocks = static_cast<unsigned>(b0);
    jobs[1].blocks = static_cast<unsigned>(b1);
    static SmemOptIn attrs;
    cudaError_t e = attrs.ensure(reinterpret_cast<const void*>(pack_kernel), 0);
    if (e == cudaSuccess)
        e = launch_kernel(pack_kernel, dim3(static_cast<unsigned>(b0 + b1)), dim3(kPackThreads), 0, stream, pdl,
                          jobs[0], jobs[1], status, limit_ns);
    if (e != cudaSuccess) {
        snprintf(msg, msg_len, "pack launch failed: %s", cudaGetErrorString(e));
        return 1;
    }
    return 0;
}

int launch_fill_bias(uint16_t* C, long long ldc, int M, int N, const uint16_t* bias, int bias_mode,
                     cudaStream_t stream, char* msg, size_t msg_len)
{
    const long long total = static_cast<long long>(M) * N;
    if (total <= 0) return 0;
    long long grid = (total + 255) / 256;
    if (grid > 4096) grid = 4096;
    static SmemOptIn attrs;
    cudaError_t e = attrs.ensure(reinterpret_cast<const void*>(fill_bias_kernel), 0);
    if (e == cudaSuccess) {
        fill_bias_kernel<<<static_cast<unsigned>(grid), 256, 0, stream>>>(C, ldc, M, N, bias, bias_mode);
        e = cudaGetLastError();
    }
    if (e != cudaSuccess) {
        snprintf(msg, msg_len, "fill launch failed: %s", cudaGetErrorString(e));
        return 1;
    }
    return 0;
}

int launch_wait_timeout_probe(int* status, unsigned long long limit_ns, cudaStream_t stream, char* msg,
                              size_t msg_len)
{
    wait_timeout_probe_kernel<<<1, 32, 0, stream>>>(status, limit_ns);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        snprintf(msg, msg_len, "probe launch failed: %s", cudaGetErrorString(e));
        return 1;
    }
    return 0;
}

}  // namespace bsk
