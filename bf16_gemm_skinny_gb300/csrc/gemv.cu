// gemv.cu -- decode GEMV / skinny GEMM on the CUDA cores: y = x W^T, n <= 8 tokens.
//
// DCU decode-GEMV article (forum.sourcefind.cn): section 6.1 fixes the shapes
// (X:[n,k], W:[m,k], Y:[n,m], all row-major) and section 6.2 the work split:
// every output Y[t, j] is an independent dot product of W's row j with X's row
// t over the whole k range, so the tiling runs along the output dimension m.
// Sections 2-5: with n this small the arithmetic intensity is ~n FLOP/byte and
// the time is the HBM stream of W; tensor cores do not help, the goal is to
// keep enough bytes in flight.
//
// Design:
//  * x (n x K, small) is converted to FP32 once per CTA into shared memory;
//    with K too large for shared memory it is staged in k-slabs.
//  * each warp owns R consecutive rows of W; lane l reads 16-byte chunks
//    l, l+32, ... of those rows (128-bit, fully coalesced, L1 bypassed), U
//    chunks deep, so a warp keeps U*R*512 bytes of W in flight;
//  * the 8 BF16 values of a chunk are widened to FP32 by a 16-bit shift (a
//    bfloat16 is the upper half of a binary32) and multiplied into FP32
//    accumulators with packed two-lane FMAs (fma.rn.f32x2);
//  * the R*n partial sums of a warp are reduced by a butterfly that halves the
//    value set at each shuffle step (R*n-1 shuffles instead of 5*R*n), and
//    each result is rounded once to BF16 (round to nearest even).
// A scalar variant handles K not a multiple of 8 or unaligned pointers.
#include <cuda_bf16.h>

#include <cstdio>

#include "bsk_internal.h"

namespace bsk {
namespace {

__device__ __forceinline__ uint4 ld_stream_16B(const uint4* p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// bf16 pair in one 32-bit word -> the two FP32 values (element 0 = low half).
__device__ __forceinline__ float2 bf16x2_to_f32x2(uint32_t w)
{
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c)
{
    unsigned long long d;
    const unsigned long long ua = *reinterpret_cast<unsigned long long*>(&a);
    const unsigned long long ub = *reinterpret_cast<unsigned long long*>(&b);
    const unsigned long long uc = *reinterpret_cast<unsigned long long*>(&c);
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(ua), "l"(ub), "l"(uc));
    return *reinterpret_cast<float2*>(&d);
}

__host__ __device__ constexpr int next_pow2(int v)
{
    int p = 1;
    while (p < v) p <<= 1;
    return p;
}

__host__ __device__ constexpr int log2_int(int v)
{
    int l = 0;
    while ((1 << l) < v) ++l;
    return l;
}

// Butterfly reduce-scatter over the 32 lanes of a warp.  On entry every lane
// holds V partial values; on exit lane l holds, in v[0 .. max(V/32,1)-1], the
// warp-wide sums of the original indices given by result_index().
template <int V>
__device__ __forceinline__ void warp_reduce_scatter(float (&v)[V], int lane)
{
    constexpr int kSteps = log2_int(V) < 5 ? log2_int(V) : 5;
#pragma unroll
    for (int s = 0; s < kSteps; ++s) {
        const int off = 16 >> s;
        const int half = V >> (s + 1);
        const bool upper = (lane & off) != 0;
#pragma unroll
        for (int i = 0; i < half; ++i) {
            const float send = upper ? v[i] : v[i + half];
            const float keep = upper ? v[i + half] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
        }
    }
#pragma unroll
    for (int s = kSteps; s < 5; ++s) v[0] += __shfl_xor_sync(0xffffffffu, v[0], 16 >> s);
}

// Original index held in v[i] by lane `lane` after warp_reduce_scatter<V>.
template <int V>
__device__ __forceinline__ int result_index(int lane, int i)
{
    constexpr int kSteps = log2_int(V) < 5 ? log2_int(V) : 5;
    int idx = i;
#pragma unroll
    for (int s = 0; s < kSteps; ++s)
        if (lane & (16 >> s)) idx += V >> (s + 1);
    return idx;
}

template <int V>
__device__ __forceinline__ bool result_owner(int lane)
{
    // for V < 32 the low 5 - log2(V) lane bits only carry copies
    constexpr int kSteps = log2_int(V) < 5 ? log2_int(V) : 5;
    constexpr int kDupMask = (1 << (5 - kSteps)) - 1;
    return (lane & kDupMask) == 0;
}

// x (n rows of K BF16) -> FP32 in shared memory, chunks [c0, c1) of 8 values.
// Layout (float4 units): values 0-3 of chunk c of token t at xs4[(2t)*slab8 + c],
// values 4-7 at xs4[(2t+1)*slab8 + c], so that lanes reading consecutive
// chunks touch consecutive 16-byte words (no bank conflicts).
template <int NT>
__device__ __forceinline__ void stage_x(const uint4* __restrict__ x4, int K8, int c0, int c1, float4* xs4, int slab8)
{
    const int nchunk = c1 - c0;
    for (int i = threadIdx.x; i < NT * nchunk; i += blockDim.x) {
        const int t = i / nchunk;
        const int c = i - t * nchunk;
        const uint4 v = x4[static_cast<long long>(t) * K8 + c0 + c];
        const float2 f0 = bf16x2_to_f32x2(v.x), f1 = bf16x2_to_f32x2(v.y);
        const float2 f2 = bf16x2_to_f32x2(v.z), f3 = bf16x2_to_f32x2(v.w);
        xs4[static_cast<long long>(2 * t) * slab8 + c] = make_float4(f0.x, f0.y, f1.x, f1.y);
        xs4[static_cast<long long>(2 * t + 1) * slab8 + c] = make_float4(f2.x, f2.y, f3.x, f3.y);
    }
}

template <int NT, int R, int U>
__global__ void __launch_bounds__(256)
    gemv_bf16_kernel(const uint4* __restrict__ W4, const uint4* __restrict__ x4, __nv_bfloat16* __restrict__ y,
                     int M, int K8, int slab8)
{
    extern __shared__ float4 xs4[];
    constexpr int V = next_pow2(R * NT);

    const int lane = threadIdx.x & 31;
    const int warps = blockDim.x >> 5;
    const int num_groups = (M + R - 1) / R;
    const bool single_slab = slab8 >= K8;

    if (single_slab) {
        stage_x<NT>(x4, K8, 0, K8, xs4, slab8);
        __syncthreads();
    }

    // Block-uniform loop over rounds so that k-slab staging can synchronise.
    for (int base = blockIdx.x * warps; base < num_groups; base += gridDim.x * warps) {
        const int g = base + (threadIdx.x >> 5);
        const bool active = g < num_groups;
        const int row0 = g * R;
        float2 acc[R][NT];
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int t = 0; t < NT; ++t) acc[r][t] = make_float2(0.f, 0.f);

        for (int s0 = 0; s0 < K8; s0 += slab8) {
            const int s1 = (s0 + slab8 < K8) ? s0 + slab8 : K8;
            if (!single_slab) {
                __syncthreads();
                stage_x<NT>(x4, K8, s0, s1, xs4, slab8);
                __syncthreads();
            }
            if (!active) continue;
            for (int c = s0 + lane; c < s1; c += 32 * U) {
                uint4 w[U][R];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int cc = c + 32 * u;
#pragma unroll
                    for (int r = 0; r < R; ++r) {
                        const bool ok = cc < s1 && row0 + r < M;
                        w[u][r] = ok ? ld_stream_16B(W4 + static_cast<long long>(row0 + r) * K8 + cc)
                                     : make_uint4(0u, 0u, 0u, 0u);
                    }
                }
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int cc = c + 32 * u;
                    if (cc >= s1) break;
                    float2 wf[R][4];
#pragma unroll
                    for (int r = 0; r < R; ++r) {
                        wf[r][0] = bf16x2_to_f32x2(w[u][r].x);
                        wf[r][1] = bf16x2_to_f32x2(w[u][r].y);
                        wf[r][2] = bf16x2_to_f32x2(w[u][r].z);
                        wf[r][3] = bf16x2_to_f32x2(w[u][r].w);
                    }
                    const float4* xp = xs4 + (cc - s0);
#pragma unroll
                    for (int t = 0; t < NT; ++t) {
                        const float4 xa = xp[static_cast<long long>(2 * t) * slab8];
                        const float4 xb = xp[static_cast<long long>(2 * t + 1) * slab8];
                        const float2 x0 = make_float2(xa.x, xa.y), x1 = make_float2(xa.z, xa.w);
                        const float2 x2 = make_float2(xb.x, xb.y), x3 = make_float2(xb.z, xb.w);
#pragma unroll
                        for (int r = 0; r < R; ++r) {
                            acc[r][t] = ffma2(wf[r][0], x0, acc[r][t]);
                            acc[r][t] = ffma2(wf[r][1], x1, acc[r][t]);
                            acc[r][t] = ffma2(wf[r][2], x2, acc[r][t]);
                            acc[r][t] = ffma2(wf[r][3], x3, acc[r][t]);
                        }
                    }
                }
            }
        }
        if (!active) continue;

        float v[V];
#pragma unroll
        for (int i = 0; i < V; ++i) v[i] = 0.f;
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int t = 0; t < NT; ++t) v[r * NT + t] = acc[r][t].x + acc[r][t].y;
        warp_reduce_scatter<V>(v, lane);
        if (result_owner<V>(lane)) {
            constexpr int kHeld = V >= 32 ? V / 32 : 1;
#pragma unroll
            for (int i = 0; i < kHeld; ++i) {
                const int idx = result_index<V>(lane, i);
                if (idx < R * NT) {
                    const int r = idx / NT;
                    const int t = idx - r * NT;
                    if (row0 + r < M) y[static_cast<long long>(t) * M + row0 + r] = __float2bfloat16_rn(v[i]);
                }
            }
        }
    }
}

// Scalar variant: any K, any alignment.  One warp per output row.
template <int NT>
__global__ void __launch_bounds__(256)
    gemv_bf16_scalar_kernel(const uint16_t* __restrict__ W, const uint16_t* __restrict__ x,
                            __nv_bfloat16* __restrict__ y, int M, int K)
{
    const int lane = threadIdx.x & 31;
    const long long warp0 = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const long long nwarps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
    for (long long j = warp0; j < M; j += nwarps) {
        float acc[NT];
#pragma unroll
        for (int t = 0; t < NT; ++t) acc[t] = 0.f;
        for (int k = lane; k < K; k += 32) {
            const float w = __uint_as_float(static_cast<uint32_t>(W[j * K + k]) << 16);
#pragma unroll
            for (int t = 0; t < NT; ++t)
                acc[t] = fmaf(w, __uint_as_float(static_cast<uint32_t>(x[static_cast<long long>(t) * K + k]) << 16),
                              acc[t]);
        }
#pragma unroll
        for (int t = 0; t < NT; ++t) {
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) acc[t] += __shfl_xor_sync(0xffffffffu, acc[t], off);
        }
        if (lane == 0) {
#pragma unroll
            for (int t = 0; t < NT; ++t) y[static_cast<long long>(t) * M + j] = __float2bfloat16_rn(acc[t]);
        }
    }
}

template <int NT, int R, int U>
int launch_vec(const GemvLaunch& g, cudaStream_t stream, char* msg, size_t msg_len)
{
    auto kern = gemv_bf16_kernel<NT, R, U>;
    const int K8 = g.K / 8;
    const int threads = 32 * (g.warps_per_block > 0 ? g.warps_per_block : 8);
    // x in FP32: NT * slab8 * 32 bytes; keep it within 192 KB (k-slabs beyond that)
    const long long budget = 192 * 1024;
    long long slab8 = budget / (32LL * NT);
    if (slab8 >= K8) slab8 = K8;
    if (slab8 < 1) slab8 = 1;
    const size_t smem = static_cast<size_t>(NT) * slab8 * 32;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) {
        snprintf(msg, msg_len, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
        return 1;
    }
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, smem);
    if (e != cudaSuccess || per_sm < 1) per_sm = 1;
    const long long groups = (g.M + R - 1) / R;
    const long long need = (groups + threads / 32 - 1) / (threads / 32);
    long long grid = static_cast<long long>(g.num_sms) * per_sm;
    if (grid > need) grid = need;
    if (grid < 1) grid = 1;
    kern<<<static_cast<unsigned>(grid), threads, smem, stream>>>(
        reinterpret_cast<const uint4*>(g.W), reinterpret_cast<const uint4*>(g.x),
        reinterpret_cast<__nv_bfloat16*>(g.y), g.M, K8, static_cast<int>(slab8));
    e = cudaGetLastError();
    if (e != cudaSuccess) {
        snprintf(msg, msg_len, "GEMV launch failed: %s", cudaGetErrorString(e));
        return 1;
    }
    return 0;
}

template <int NT>
int launch_scalar(const GemvLaunch& g, cudaStream_t stream, char* msg, size_t msg_len)
{
    const int threads = 256;
    long long grid = (static_cast<long long>(g.M) * 32 + threads - 1) / threads;
    const long long cap = static_cast<long long>(g.num_sms) * 8;
    if (grid > cap) grid = cap;
    if (grid < 1) grid = 1;
    gemv_bf16_scalar_kernel<NT><<<static_cast<unsigned>(grid), threads, 0, stream>>>(
        g.W, g.x, reinterpret_cast<__nv_bfloat16*>(g.y), g.M, g.K);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        snprintf(msg, msg_len, "GEMV launch failed: %s", cudaGetErrorString(e));
        return 1;
    }
    return 0;
}

// Rows per warp (R) and chunks in flight per lane (U) for each token count.
template <int NT>
int launch_vec_rows(const GemvLaunch& g, int rows, cudaStream_t stream, char* msg, size_t msg_len)
{
    switch (rows) {
    case 1: return launch_vec<NT, 1, 4>(g, stream, msg, msg_len);
    case 2: return launch_vec<NT, 2, (NT <= 4 ? 4 : 2)>(g, stream, msg, msg_len);
    case 4: return launch_vec<NT, 4, (NT <= 2 ? 4 : 2)>(g, stream, msg, msg_len);
    case 8: return launch_vec<NT, 8, (NT <= 2 ? 2 : 1)>(g, stream, msg, msg_len);
    default:
        snprintf(msg, msg_len, "unsupported rows_per_warp %d (1, 2, 4 or 8)", rows);
        return 1;
    }
}

constexpr int default_rows(int n) { return n <= 2 ? 8 : 4; }

}  // namespace

int launch_gemv(const GemvLaunch& g, cudaStream_t stream, char* msg, size_t msg_len)
{
    const bool vec = (g.K % 8 == 0) && (reinterpret_cast<uintptr_t>(g.W) % 16 == 0) &&
                     (reinterpret_cast<uintptr_t>(g.x) % 16 == 0);
    const int rows = g.rows_per_warp > 0 ? g.rows_per_warp : default_rows(g.n);
    if (vec) {
        switch (g.n) {
        case 1: return launch_vec_rows<1>(g, rows, stream, msg, msg_len);
        case 2: return launch_vec_rows<2>(g, rows, stream, msg, msg_len);
        case 3: return launch_vec_rows<3>(g, rows, stream, msg, msg_len);
        case 4: return launch_vec_rows<4>(g, rows, stream, msg, msg_len);
        case 5: return launch_vec_rows<5>(g, rows, stream, msg, msg_len);
        case 6: return launch_vec_rows<6>(g, rows, stream, msg, msg_len);
        case 7: return launch_vec_rows<7>(g, rows, stream, msg, msg_len);
        case 8: return launch_vec_rows<8>(g, rows, stream, msg, msg_len);
        default: break;
        }
    } else {
        switch (g.n) {
        case 1: return launch_scalar<1>(g, stream, msg, msg_len);
        case 2: return launch_scalar<2>(g, stream, msg, msg_len);
        case 3: return launch_scalar<3>(g, stream, msg, msg_len);
        case 4: return launch_scalar<4>(g, stream, msg, msg_len);
        case 5: return launch_scalar<5>(g, stream, msg, msg_len);
        case 6: return launch_scalar<6>(g, stream, msg, msg_len);
        case 7: return launch_scalar<7>(g, stream, msg, msg_len);
        case 8: return launch_scalar<8>(g, stream, msg, msg_len);
        default: break;
        }
    }
    snprintf(msg, msg_len, "GEMV kernel takes 1..8 tokens, got %d", g.n);
    return 1;
}

}  // namespace bsk
