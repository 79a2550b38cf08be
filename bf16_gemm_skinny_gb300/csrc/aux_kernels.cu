// aux_kernels.cu -- the operand pack kernel and the bounded-wait test probe.
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

// dst[i + j*ld_dst] = src[i + j*ld_src] for i < inner, j < outer.  The TMA
// needs 16-byte aligned bases and leading dimensions; the pack gives unaligned
// operands that shape in a workspace without touching the caller's buffers
// ("MTT S4000 GEMM 优化中的分块、尾处理与并发实战复盘", section 1: inputs may not be modified).
// Grid: x over 16-byte groups of a line, y over lines (grid-stride).  The
// destination lines are 16-byte aligned (base and ld_dst), so each full group
// is one 16-byte store.  A source group at any byte offset is read as the
// aligned 16-byte chunk holding its first byte and, unless the offset is 0,
// the next chunk, then shifted into place (two aligned loads, the second the
// neighbouring thread's first, instead of one load per element).  Both chunks
// hold bytes of the group, so neither reaches a page the line does not touch.
// The last, partial group of a line is copied element by element.
template <typename T>
__global__ void __launch_bounds__(256)
    pack_kernel(const T* __restrict__ src, long long ld_src, T* __restrict__ dst, long long ld_dst, int inner,
                int outer)
{
    constexpr int V = 16 / static_cast<int>(sizeof(T));
    const long long i0 = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) * V;
    if (i0 >= inner) return;
    const bool full = i0 + V <= inner;
    for (long long j = blockIdx.y; j < outer; j += gridDim.y) {
        const T* s = src + j * ld_src + i0;
        T* d = dst + j * ld_dst + i0;
        if (full) {
            const uintptr_t a = reinterpret_cast<uintptr_t>(s);
            const uint4* chunk = reinterpret_cast<const uint4*>(a & ~static_cast<uintptr_t>(15));
            const unsigned m = static_cast<unsigned>(a & 15u);
            const uint4 lo = chunk[0];
            *reinterpret_cast<uint4*>(d) = m == 0u ? lo : realign16(lo, chunk[1], m);
        } else {
            for (long long t = 0; i0 + t < inner; ++t) d[t] = s[t];
        }
    }
}

template <typename T>
int launch_pack_t(const T* src, long long ld_src, T* dst, long long ld_dst, int inner, int outer, cudaStream_t stream,
                  char* msg, size_t msg_len)
{
    if (inner <= 0 || outer <= 0) return 0;
    constexpr int V = 16 / static_cast<int>(sizeof(T));
    const long long groups = (static_cast<long long>(inner) + V - 1) / V;
    const unsigned gx = static_cast<unsigned>((groups + 255) / 256);
    const unsigned gy = static_cast<unsigned>(outer < 65535 ? outer : 65535);
    pack_kernel<T><<<dim3(gx, gy, 1), 256, 0, stream>>>(src, ld_src, dst, ld_dst, inner, outer);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        snprintf(msg, msg_len, "pack launch failed: %s", cudaGetErrorString(e));
        return 1;
    }
    return 0;
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

int launch_pack(const uint16_t* src, long long ld_src, uint16_t* dst, long long ld_dst, int inner, int outer,
                cudaStream_t stream, char* msg, size_t msg_len)
{
    return launch_pack_t<uint16_t>(src, ld_src, dst, ld_dst, inner, outer, stream, msg, msg_len);
}

int launch_pack_8bit(const uint8_t* src, long long ld_src, uint8_t* dst, long long ld_dst, int inner, int outer,
                     cudaStream_t stream, char* msg, size_t msg_len)
{
    return launch_pack_t<uint8_t>(src, ld_src, dst, ld_dst, inner, outer, stream, msg, msg_len);
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
