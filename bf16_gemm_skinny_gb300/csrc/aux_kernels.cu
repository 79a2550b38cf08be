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

// One operand's copy as the kernel sees it: `lines` lines of line_bytes bytes.
// A step is 32 consecutive 16-byte groups of one line (512 bytes, one per
// lane; the last group of a line may be partial, and lanes past the line's
// end idle), numbered line by line.
struct PackJob {
    const uint8_t* src;
    long long ld_src;          // bytes from one source line to the next
    uint8_t* dst;              // 16-byte aligned
    long long ld_dst;          // bytes, a multiple of 16
    unsigned line_bytes;
    unsigned steps_per_line;
    unsigned steps;            // steps_per_line x lines, below 2^31
    unsigned blocks;           // CTAs working on this job
};

constexpr int kPackThreads = 256;
constexpr int kPackWarps = kPackThreads / 32;
constexpr int kPackStages = 8;        // cp.async ring depth per warp
constexpr int kPackCtasPerSm = 4;

__device__ __forceinline__ void pack_cp_async16(uint32_t dst, const void* src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void pack_cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void pack_cp_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// A cursor over a warp's steps: the current line's source and destination
// starts and the step within the line.
struct PackCursor {
    const uint8_t* s;
    uint8_t* d;
    unsigned k;
    __device__ __forceinline__ void next(unsigned steps_per_line, long long ld_src, long long ld_dst)
    {
        if (++k == steps_per_line) {
            k = 0;
            s += ld_src;
            d += ld_dst;
        }
    }
};

// dst line l = src line l, byte for byte, for up to two operands in one launch
// (the first job.blocks CTAs take job 0, the rest job 1).  The TMA needs
// 16-byte aligned bases and leading dimensions; the pack gives unaligned
// operands that shape in a workspace without touching the caller's buffers
// ("MTT S4000 GEMM 优化中的分块、尾处理与并发实战复盘", section 1: inputs may not be modified).
//
// Each warp takes a contiguous range of steps.  A step's 32 groups start m
// bytes past a 16-byte boundary (m is the line's, the same for the whole
// warp), so they span 33 aligned source chunks: lane l copies chunk l with
// cp.async and lane 31 also chunk 32, each only if it holds bytes of a full
// group (so no copy reaches a page the line does not touch).  The chunks go
// through a per-warp ring of kPackStages steps in shared memory, so each SM
// keeps its warps' next seven steps of reads in flight.  After its own
// copies land (wait_group), a __syncwarp lets lane l read chunk l + 1 of its
// neighbour; the two chunks are shifted into place and stored with one
// aligned 16-byte store.  A second __syncwarp keeps the slot from being
// refilled before every lane has read it.  The partial last group of a line
// is copied byte by byte.
__global__ void __launch_bounds__(kPackThreads, kPackCtasPerSm) pack_kernel(PackJob j0, PackJob j1)
{
    __shared__ __align__(16) uint4 ring[kPackWarps][kPackStages][33];
    griddep_wait();               // the source may be the previous kernel's output
    griddep_launch_dependents();  // the GEMM's prologue may start; it waits for this grid's completion
    const bool second = blockIdx.x >= j0.blocks;
    const uint8_t* const src = second ? j1.src : j0.src;
    uint8_t* const dst = second ? j1.dst : j0.dst;
    const long long ld_src = second ? j1.ld_src : j0.ld_src;
    const long long ld_dst = second ? j1.ld_dst : j0.ld_dst;
    const unsigned line_bytes = second ? j1.line_bytes : j0.line_bytes;
    const unsigned spl = second ? j1.steps_per_line : j0.steps_per_line;
    const unsigned steps = second ? j1.steps : j0.steps;
    const unsigned blocks = second ? j1.blocks : j0.blocks;
    const unsigned b = second ? blockIdx.x - j0.blocks : blockIdx.x;
    const unsigned warp = threadIdx.x >> 5, lane = threadIdx.x & 31u;
    const unsigned long long nw = static_cast<unsigned long long>(blocks) * kPackWarps;
    const unsigned long long w = static_cast<unsigned long long>(b) * kPackWarps + warp;
    const unsigned s0 = static_cast<unsigned>(steps * w / nw);
    const unsigned n = static_cast<unsigned>(steps * (w + 1) / nw) - s0;
    const unsigned off = lane * 16u;   // the lane's group within a step, in bytes
    const unsigned line0 = s0 / spl;
    PackCursor in{src + line0 * ld_src, dst + line0 * ld_dst, s0 % spl};
    PackCursor out = in;

    auto issue = [&](int slot) {
        const unsigned g = in.k * 512u + off;
        const uintptr_t a = reinterpret_cast<uintptr_t>(in.s) + g;
        const unsigned m = static_cast<unsigned>(a & 15u);
        const uint8_t* chunk = reinterpret_cast<const uint8_t*>(a & ~static_cast<uintptr_t>(15));
        // chunk `lane` holds the start of this lane's group and, when m > 0, the
        // end of the previous lane's group
        const bool full = g + 16u <= line_bytes;
        if (full || (m != 0u && lane != 0u && g <= line_bytes))
            pack_cp_async16(smem_u32(&ring[warp][slot][lane]), chunk);
        if (lane == 31u && m != 0u && full) pack_cp_async16(smem_u32(&ring[warp][slot][32]), chunk + 16);
        pack_cp_commit();
        in.next(spl, ld_src, ld_dst);
    };

#pragma unroll
    for (int t = 0; t < kPackStages - 1; ++t) {
        if (static_cast<unsigned>(t) < n) issue(t);
        else pack_cp_commit();
    }
    int slot = 0;
    for (unsigned i = 0; i < n; ++i) {
        // the slot consumed last iteration takes the step kPackStages - 1 ahead
        const int ahead = slot == 0 ? kPackStages - 1 : slot - 1;
        if (i + (kPackStages - 1) < n) issue(ahead);
        else pack_cp_commit();
        pack_cp_wait<kPackStages - 1>();   // this lane's copies of step i have landed
        __syncwarp();                      // ... and so have its neighbours'
        const unsigned g = out.k * 512u + off;
        const uint8_t* sp = out.s + g;
        if (g + 16u <= line_bytes) {
            const unsigned m = static_cast<unsigned>(reinterpret_cast<uintptr_t>(sp) & 15u);
            const uint4 lo = ring[warp][slot][lane];
            *reinterpret_cast<uint4*>(out.d + g) = m == 0u ? lo : realign16(lo, ring[warp][slot][lane + 1], m);
        } else if (g < line_bytes) {
            for (unsigned t = 0; t < line_bytes - g; ++t) out.d[g + t] = sp[t];
        }
        __syncwarp();                      // every lane has read the slot before it is refilled
        out.next(spl, ld_src, ld_dst);
        slot = slot == kPackStages - 1 ? 0 : slot + 1;
    }
    pack_cp_wait<0>();   // the trailing (empty) groups
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

int launch_pack(const PackCopy* copies, int n, int sms, bool pdl, cudaStream_t stream, char* msg, size_t msg_len)
{
    PackJob jobs[2] = {};
    int nj = 0;
    auto flush = [&]() -> int {
        // persistent grid, split between the jobs by their steps (at least one
        // CTA each, no more than one warp per step)
        const unsigned long long per_cta = kPackWarps;
        const unsigned long long u0 = jobs[0].steps, u1 = nj > 1 ? jobs[1].steps : 0ull;
        const unsigned long long total = static_cast<unsigned long long>(sms > 0 ? sms : 1) * kPackCtasPerSm;
        unsigned long long b0 = nj > 1 ? (total * u0 + (u0 + u1) / 2) / (u0 + u1) : total;
        if (b0 < 1) b0 = 1;
        unsigned long long b1 = nj > 1 ? (total > b0 ? total - b0 : 1ull) : 0ull;
        b0 = std::min(b0, (u0 + per_cta - 1) / per_cta);
        b1 = std::min(b1, (u1 + per_cta - 1) / per_cta);
        jobs[0].blocks = static_cast<unsigned>(b0);
        jobs[1].blocks = static_cast<unsigned>(b1);
        cudaError_t e = launch_kernel(pack_kernel, dim3(static_cast<unsigned>(b0 + b1)), dim3(kPackThreads), 0,
                                      stream, pdl, jobs[0], jobs[1]);
        nj = 0;
        jobs[0] = PackJob{};
        jobs[1] = PackJob{};
        if (e != cudaSuccess) {
            snprintf(msg, msg_len, "pack launch failed: %s", cudaGetErrorString(e));
            return 1;
        }
        return 0;
    };
    for (int i = 0; i < n; ++i) {
        const PackCopy& c = copies[i];
        if (c.line_bytes <= 0 || c.lines <= 0) continue;
        if (c.line_bytes > (1LL << 31)) {
            snprintf(msg, msg_len, "pack: line of %lld bytes is too long", c.line_bytes);
            return 1;
        }
        const unsigned long long spl = (static_cast<unsigned long long>(c.line_bytes) + 511) / 512;
        // keep each job's step count below 2^31 (32-bit step arithmetic in the kernel)
        const long long lines_per_job = static_cast<long long>(std::max(1ull, (1ull << 31) / spl - 1));
        for (long long l0 = 0; l0 < c.lines; l0 += lines_per_job) {
            const long long nl = std::min(lines_per_job, c.lines - l0);
            PackJob& j = jobs[nj++];
            j.src = static_cast<const uint8_t*>(c.src) + l0 * c.ld_src;
            j.ld_src = c.ld_src;
            j.dst = static_cast<uint8_t*>(c.dst) + l0 * c.ld_dst;
            j.ld_dst = c.ld_dst;
            j.line_bytes = static_cast<unsigned>(c.line_bytes);
            j.steps_per_line = static_cast<unsigned>(spl);
            j.steps = static_cast<unsigned>(spl * static_cast<unsigned long long>(nl));
            if (nj == 2 && flush()) return 1;
        }
    }
    if (nj > 0 && flush()) return 1;
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
