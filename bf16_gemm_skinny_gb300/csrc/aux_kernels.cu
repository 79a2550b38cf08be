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

constexpr int kPackThreads = 256;                // warp 0: producer (one lane); warps 1..7: consumers
constexpr int kPackConsumers = kPackThreads - 32;
constexpr int kPackBufs = 6;                     // pieces in flight per CTA
constexpr int kPackPiece = 8704;                 // longest piece, bytes (an 8200-byte line is one piece)
constexpr int kPackBufBytes = kPackPiece + 32;   // a piece's aligned cover plus the chunk read past it
constexpr int kPackSmem = kPackBufs * kPackBufBytes + 2 * kPackBufs * 8 + 16;
constexpr int kPackCtasPerSm = 4;
constexpr int kSitePack = 0x20;                  // wait site reported on a timeout

// dst line l = src line l, byte for byte, for up to two operands in one launch
// (the first j0.blocks CTAs take job 0, the rest job 1).  The TMA needs
// 16-byte aligned bases and leading dimensions; the pack gives unaligned
// operands that shape in a workspace without touching the caller's buffers
// ("MTT S4000 GEMM 优化中的分块、尾处理与并发实战复盘", section 1: inputs may not be modified).
//
// Each CTA takes a contiguous range of units (line pieces) through a ring of
// kPackBufs shared-memory buffers, each with a "full" and an "empty" mbarrier.
// One lane of warp 0 (the producer) issues, for each unit, a bulk copy of the
// piece's 16-byte-aligned cover -- from the aligned chunk holding its first
// byte to the end of the chunk holding its last, so no byte outside the pages
// the piece touches is read -- completing on the buffer's full barrier, as
// soon as the consumers have released the buffer.  The source is read with an
// evict-first L2 policy: it is read once, and the packed copy, which the GEMM
// reads next, should stay in L2.  Warps 1..7 (the consumers) wait for a
// buffer, and consumer thread t writes output chunks t, t + 224, ...: chunk c
// is the 16 bytes that start m bytes into buffer chunk c (m = the piece's
// offset from a 16-byte boundary), shifted out of buffer chunks c and c + 1,
// with one aligned 16-byte store; each warp then arrives on the buffer's empty
// barrier.  A line's last chunk may carry up to 15 bytes past the line's end
// into the destination's padding (its leading dimension is rounded up to 16
// bytes; the GEMM's tensor maps never read the padding).  Every wait is
// bounded; on a timeout the producer waits for its copies in flight before the
// CTA exits.
__global__ void __launch_bounds__(kPackThreads, kPackCtasPerSm)
    pack_kernel(PackJob j0, PackJob j1, int* status, unsigned long long limit_ns)
{
    extern __shared__ __align__(128) uint8_t pack_smem[];
    uint8_t* const bufs = pack_smem;
    const uint32_t full0 = smem_u32(pack_smem + kPackBufs * kPackBufBytes);
    const uint32_t empty0 = full0 + 8 * kPackBufs;
    volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(pack_smem + kPackBufs * kPackBufBytes +
                                                                          16 * kPackBufs);
    if (threadIdx.x == 0) {
        for (int i = 0; i < kPackBufs; ++i) {
            mbar_init(full0 + 8 * i, 1);
            mbar_init(empty0 + 8 * i, kPackConsumers / 32);
        }
        *abort_flag = 0u;
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

    // A cursor over this CTA's units: the unit's source and destination starts
    // and length, advanced without division (one division per CTA, for the start).
    struct Cursor {
        const uint8_t* s;
        uint8_t* d;
        long long off;   // offset of the piece in its line
        long long len;
    };
    const long long line0 = u0 / j.pieces;
    const long long off0 = (u0 - line0 * j.pieces) * j.piece_bytes;
    const Cursor start{j.src + line0 * j.ld_src + off0, j.dst + line0 * j.ld_dst + off0, off0,
                       j.line_bytes - off0 < j.piece_bytes ? j.line_bytes - off0 : j.piece_bytes};
    auto advance = [&](Cursor& c) {
        if (c.off + j.piece_bytes < j.line_bytes) {
            c.off += j.piece_bytes;
            c.s += j.piece_bytes;
            c.d += j.piece_bytes;
        } else {   // next line
            c.s += j.ld_src - c.off;
            c.d += j.ld_dst - c.off;
            c.off = 0;
        }
        c.len = j.line_bytes - c.off < j.piece_bytes ? j.line_bytes - c.off : j.piece_bytes;
    };
    const WaitCtl wc{abort_flag, status, limit_ns};
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (warp == 0) {
        if (lane == 0) {
            const uint64_t read_once = l2_policy_evict_first();
            long long issued = 0;
            bool ok = true;
            Cursor cur = start;
            int bi = 0;
            uint32_t ph = 0;   // parity of the empty-barrier phase to wait for, once the ring has wrapped
            for (; issued < n; ++issued) {
                if (issued >= kPackBufs && !mbar_wait(empty0 + 8 * bi, ph, wc, kSitePack)) {
                    ok = false;
                    break;
                }
                const uintptr_t a = reinterpret_cast<uintptr_t>(cur.s);
                const uintptr_t lo = a & ~static_cast<uintptr_t>(15);
                const uintptr_t hi = (a + static_cast<uintptr_t>(cur.len) + 15) & ~static_cast<uintptr_t>(15);
                mbar_arrive_expect_tx(full0 + 8 * bi, static_cast<uint32_t>(hi - lo));
                bulk_load_hint(smem_u32(bufs + bi * kPackBufBytes), reinterpret_cast<const void*>(lo),
                               static_cast<uint32_t>(hi - lo), full0 + 8 * bi, read_once);
                advance(cur);
                if (++bi == kPackBufs) {
                    bi = 0;
                    if (issued + 1 > kPackBufs) ph ^= 1u;
                }
            }
            if (!ok) {
                // abort: the copies of the last issued units may still be landing in
                // this CTA's shared memory; wait for them (bounded) before exiting
                uint32_t never = 0u;
                const WaitCtl wc_drain{&never, status, limit_ns};
                for (long long k = issued > kPackBufs ? issued - kPackBufs : 0; k < issued; ++k)
                    mbar_wait(full0 + 8 * (k % kPackBufs), static_cast<uint32_t>(k / kPackBufs) & 1u, wc_drain,
                              kSitePack);
            }
        }
    } else {
        const unsigned t = threadIdx.x - 32;
        Cursor cur = start;
        int bi = 0;
        uint32_t ph = 0;
        for (long long i = 0; i < n; ++i) {
            const bool ok = mbar_wait(full0 + 8 * bi, ph, wc, kSitePack);
            if (!__all_sync(0xffffffffu, ok)) break;
            const unsigned m = static_cast<unsigned>(reinterpret_cast<uintptr_t>(cur.s) & 15u);
            const uint4* sb = reinterpret_cast<const uint4*>(bufs + bi * kPackBufBytes);
            const unsigned chunks = static_cast<unsigned>((cur.len + 15) / 16);
            uint4* out = reinterpret_cast<uint4*>(cur.d);
            if (m == 0u) {
                for (unsigned c = t; c < chunks; c += kPackConsumers) out[c] = sb[c];
            } else {
                for (unsigned c = t; c < chunks; c += kPackConsumers) out[c] = realign16(sb[c], sb[c + 1], m);
            }
            __syncwarp();   // the warp has read the buffer
            if (lane == 0) mbar_arrive(empty0 + 8 * bi);
            advance(cur);
            if (++bi == kPackBufs) {
                bi = 0;
                ph ^= 1u;
            }
        }
    }
    __syncthreads();
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
    static SmemOptIn smem_opt;
    cudaError_t e = smem_opt.ensure(reinterpret_cast<const void*>(pack_kernel), kPackSmem);
    if (e == cudaSuccess)
        e = launch_kernel(pack_kernel, dim3(static_cast<unsigned>(b0 + b1)), dim3(kPackThreads),
                          static_cast<size_t>(kPackSmem), stream, pdl, jobs[0], jobs[1], status, limit_ns);
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
    fill_bias_kernel<<<static_cast<unsigned>(grid), 256, 0, stream>>>(C, ldc, M, N, bias, bias_mode);
    cudaError_t e = cudaGetLastError();
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
