// gemv.cu -- decode GEMV / skinny GEMM on the CUDA cores: y = x W^T, n <= 8 tokens
// (by default gemv_bf16 runs n <= 3 here and larger n on the tensor cores).
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

__device__ __forceinline__ void prefetch_l2(const void* p)
{
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// bf16 pair in one 32-bit word -> the two FP32 values (element 0 = low half).
// A bfloat16 is the upper half of a binary32, so each value is a byte
// permutation with zero low bytes (prmt keeps this on the integer pipe).
__device__ __forceinline__ float2 bf16x2_to_f32x2(uint32_t w)
{
    uint32_t lo, hi;
    asm("prmt.b32 %0, %1, 0, 0x1044;" : "=r"(lo) : "r"(w));
    asm("prmt.b32 %0, %1, 0, 0x3244;" : "=r"(hi) : "r"(w));
    return make_float2(__uint_as_float(lo), __uint_as_float(hi));
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

    // Until griddep_wait() the kernel before this one in the stream may still be
    // running: only L2 prefetches of this warp's first W chunks (coherent, they
    // deliver nothing to the thread) go out before it.
    {
        const int g0 = blockIdx.x * warps + (threadIdx.x >> 5);
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int c = lane + 32 * u;
                if (g0 < num_groups && g0 * R + r < M && c < K8)
                    prefetch_l2(W4 + static_cast<long long>(g0 * R + r) * K8 + c);
            }
    }
    griddep_wait();
    griddep_launch_dependents();

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

// ---------------------------------------------------------------------------
// Pipelined variant (x fits in shared memory next to the W ring).
//
// Each warp streams its rows through a private ring of D stages in shared
// memory with cp.async (16 bytes per lane per row per stage), so the bytes in
// flight (D-1 stages of R rows x 512 bytes per warp) do not depend on
// registers or on where the warp is in its arithmetic.  The warp's whole
// work -- all its row groups, each of ceil(K8/32) steps -- is one linear
// stream of steps, so the copies for the next row group start while the
// current one is still being reduced.  Each lane reads back only the
// 16-byte pieces it copied itself, so cp.async.wait_group is the only
// synchronisation needed.  Lanes past the end of a row (or rows past M)
// copy zero bytes, which zero-fills the slot.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src, uint32_t src_bytes)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// x (n rows of K BF16) into shared memory, whole K.  XF32: FP32, values 0-3 of
// chunk c of token t at xs4[(2t)*K8 + c], values 4-7 at xs4[(2t+1)*K8 + c];
// otherwise the raw BF16 chunk at xs4[t*K8 + c].
template <int NT, bool XF32>
__device__ __forceinline__ void stage_x_whole(const uint4* __restrict__ x4, int K8, uint4* xs4)
{
    for (int i = threadIdx.x; i < NT * K8; i += blockDim.x) {
        const int t = i / K8;
        const int c = i - t * K8;
        const uint4 v = x4[i];
        if constexpr (XF32) {
            const float2 f0 = bf16x2_to_f32x2(v.x), f1 = bf16x2_to_f32x2(v.y);
            const float2 f2 = bf16x2_to_f32x2(v.z), f3 = bf16x2_to_f32x2(v.w);
            reinterpret_cast<float4*>(xs4)[static_cast<long long>(2 * t) * K8 + c] =
                make_float4(f0.x, f0.y, f1.x, f1.y);
            reinterpret_cast<float4*>(xs4)[static_cast<long long>(2 * t + 1) * K8 + c] =
                make_float4(f2.x, f2.y, f3.x, f3.y);
        } else {
            xs4[static_cast<long long>(t) * K8 + c] = v;
        }
    }
}

template <int NT, int R, int D, bool XF32>
__global__ void __launch_bounds__(512, 1)
    gemv_bf16_pipe_kernel(const uint4* __restrict__ W4, const uint4* __restrict__ x4, __nv_bfloat16* __restrict__ y,
                          int M, int K8, int groups_per_warp)
{
    extern __shared__ uint4 smem4[];
    constexpr int V = next_pow2(R * NT);
    constexpr uint32_t kSlotBytes = R * 512u;       // one stage of one warp: R rows x 32 lanes x 16 B
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int warps = blockDim.x >> 5;
    const int x_words = NT * K8 * (XF32 ? 2 : 1);
    uint4* xs4 = smem4;
    uint4* ring = smem4 + x_words + warp * D * R * 32;
    const uint32_t ring_s = static_cast<uint32_t>(__cvta_generic_to_shared(ring)) + lane * 16u;

    griddep_wait();
    griddep_launch_dependents();
    stage_x_whole<NT, XF32>(x4, K8, xs4);
    __syncthreads();

    const int num_groups = (M + R - 1) / R;
    const int g_begin = (blockIdx.x * warps + warp) * groups_per_warp;
    int g_count = num_groups - g_begin;
    if (g_count > groups_per_warp) g_count = groups_per_warp;
    if (g_count <= 0) return;
    const int steps = (K8 + 31) >> 5;
    const long long row_stride = K8;                 // uint4 per row

    // Issue cursor: the next (group, step) whose copies go out, and its ring slot.
    int i_g = 0, i_s = 0, i_slot = 0;
    const uint4* i_ptr = W4 + static_cast<long long>(g_begin) * R * row_stride + lane;
    int i_rows = M - g_begin * R;
    auto issue = [&]() {
        if (i_g < g_count) {
            const uint32_t dst = ring_s + static_cast<uint32_t>(i_slot) * kSlotBytes;
            const bool kok = i_s * 32 + lane < K8;
            if (kok && i_rows >= R) {
#pragma unroll
                for (int r = 0; r < R; ++r) cp_async_16(dst + r * 512u, i_ptr + r * row_stride, 16u);
            } else {
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const bool ok = kok && r < i_rows;
                    cp_async_16(dst + r * 512u, ok ? i_ptr + r * row_stride : W4, ok ? 16u : 0u);
                }
            }
            i_ptr += 32;
            if (++i_s == steps) {
                i_s = 0;
                ++i_g;
                i_ptr += R * row_stride - static_cast<long long>(steps) * 32;
                i_rows -= R;
            }
            if (++i_slot == D) i_slot = 0;
        }
        cp_async_commit();
    };

#pragma unroll
    for (int q = 0; q < D - 1; ++q) issue();

    int c_slot = 0;
    for (int gi = 0; gi < g_count; ++gi) {
        float2 acc[R][NT];
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int t = 0; t < NT; ++t) acc[r][t] = make_float2(0.f, 0.f);

        for (int st = 0; st < steps; ++st) {
            issue();
            cp_async_wait<D - 1>();
            const int c = st * 32 + lane;
            if (c < K8) {
                const uint4* slot = ring + c_slot * (R * 32) + lane;
                float2 wf[R][4];
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const uint4 w = slot[r * 32];
                    wf[r][0] = bf16x2_to_f32x2(w.x);
                    wf[r][1] = bf16x2_to_f32x2(w.y);
                    wf[r][2] = bf16x2_to_f32x2(w.z);
                    wf[r][3] = bf16x2_to_f32x2(w.w);
                }
#pragma unroll
                for (int t = 0; t < NT; ++t) {
                    // rows innermost: consecutive FMAs update different accumulators
                    if constexpr (XF32) {
                        const float4* xt = reinterpret_cast<const float4*>(xs4) + 2 * t * K8 + c;
                        const float4 xa = xt[0];
                        const float4 xb = xt[K8];
                        const float2 xp[4] = {make_float2(xa.x, xa.y), make_float2(xa.z, xa.w),
                                              make_float2(xb.x, xb.y), make_float2(xb.z, xb.w)};
#pragma unroll
                        for (int q = 0; q < 4; ++q)
#pragma unroll
                            for (int r = 0; r < R; ++r) acc[r][t] = ffma2(wf[r][q], xp[q], acc[r][t]);
                    } else {
                        const uint4 xv = xs4[t * K8 + c];
                        const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const float2 xp = bf16x2_to_f32x2(xw[q]);
#pragma unroll
                            for (int r = 0; r < R; ++r) acc[r][t] = ffma2(wf[r][q], xp, acc[r][t]);
                        }
                    }
                }
            }
            if (++c_slot == D) c_slot = 0;
        }

        const int row0 = (g_begin + gi) * R;
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
    cp_async_wait<0>();
}

// ---------------------------------------------------------------------------
// Token-paired variant for 5..8 tokens (padded to 8).
//
// With many tokens the FP32 FMAs, not HBM, set the pace; the accumulators of
// the pipelined kernel are paired over k (two per row and token), which caps
// the rows per warp at 4 within the register budget.  Here each fma.rn.f32x2
// updates the accumulators of two tokens of one row, {w, w} * {x_t, x_t+1},
// so R = 8 rows take 32 accumulator registers and every widened x pair is
// reused by 8 rows.  x is staged token-interleaved: for chunk c and element e
// (0..7), the 8 tokens' BF16 values form one 16-byte slot, placed at slot
// e ^ (c & 7) so that lanes reading consecutive chunks spread over the banks.
// ---------------------------------------------------------------------------
template <int NT>
__device__ __forceinline__ void stage_x_token_interleaved(const uint16_t* __restrict__ x, int K, int K8, uint4* xs4)
{
    for (int i = threadIdx.x; i < K8 * 8; i += blockDim.x) {
        const int c = i >> 3;
        const int e = i & 7;
        const int k = c * 8 + e;
        uint32_t w[4];
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            const uint32_t lo = (2 * p < NT) ? x[static_cast<long long>(2 * p) * K + k] : 0u;
            const uint32_t hi = (2 * p + 1 < NT) ? x[static_cast<long long>(2 * p + 1) * K + k] : 0u;
            w[p] = lo | (hi << 16);
        }
        xs4[c * 8 + (e ^ (c & 7))] = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// bf16 value in the low (HI = false) or high half of a word -> {v, v}.
template <bool HI>
__device__ __forceinline__ float2 bf16_dup(uint32_t w)
{
    uint32_t v;
    if constexpr (HI) {
        asm("prmt.b32 %0, %1, 0, 0x3244;" : "=r"(v) : "r"(w));
    } else {
        asm("prmt.b32 %0, %1, 0, 0x1044;" : "=r"(v) : "r"(w));
    }
    return make_float2(__uint_as_float(v), __uint_as_float(v));
}

template <int NT, int R, int D>
__global__ void __launch_bounds__(512, 1)
    gemv_bf16_tokpair_kernel(const uint4* __restrict__ W4, const uint16_t* __restrict__ x,
                             __nv_bfloat16* __restrict__ y, int M, int K, int groups_per_warp)
{
    static_assert(NT >= 1 && NT <= 8, "token-paired kernel takes up to 8 tokens");
    extern __shared__ uint4 smem4[];
    constexpr int V = next_pow2(R * 8);
    constexpr uint32_t kSlotBytes = R * 512u;
    const int K8 = K >> 3;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int warps = blockDim.x >> 5;
    uint4* xs4 = smem4;
    uint4* ring = smem4 + K8 * 8 + warp * D * R * 32;
    const uint32_t ring_s = static_cast<uint32_t>(__cvta_generic_to_shared(ring)) + lane * 16u;

    griddep_wait();
    griddep_launch_dependents();
    stage_x_token_interleaved<NT>(x, K, K8, xs4);
    __syncthreads();

    const int num_groups = (M + R - 1) / R;
    const int g_begin = (blockIdx.x * warps + warp) * groups_per_warp;
    int g_count = num_groups - g_begin;
    if (g_count > groups_per_warp) g_count = groups_per_warp;
    if (g_count <= 0) return;
    const int steps = (K8 + 31) >> 5;
    const long long row_stride = K8;

    int i_g = 0, i_s = 0, i_slot = 0;
    const uint4* i_ptr = W4 + static_cast<long long>(g_begin) * R * row_stride + lane;
    int i_rows = M - g_begin * R;
    auto issue = [&]() {
        if (i_g < g_count) {
            const uint32_t dst = ring_s + static_cast<uint32_t>(i_slot) * kSlotBytes;
            const bool kok = i_s * 32 + lane < K8;
            if (kok && i_rows >= R) {
#pragma unroll
                for (int r = 0; r < R; ++r) cp_async_16(dst + r * 512u, i_ptr + r * row_stride, 16u);
            } else {
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const bool ok = kok && r < i_rows;
                    cp_async_16(dst + r * 512u, ok ? i_ptr + r * row_stride : W4, ok ? 16u : 0u);
                }
            }
            i_ptr += 32;
            if (++i_s == steps) {
                i_s = 0;
                ++i_g;
                i_ptr += R * row_stride - static_cast<long long>(steps) * 32;
                i_rows -= R;
            }
            if (++i_slot == D) i_slot = 0;
        }
        cp_async_commit();
    };

#pragma unroll
    for (int q = 0; q < D - 1; ++q) issue();

    int c_slot = 0;
    for (int gi = 0; gi < g_count; ++gi) {
        float2 acc[R][4];   // acc[r][p] = {row r . token 2p, row r . token 2p+1}
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int p = 0; p < 4; ++p) acc[r][p] = make_float2(0.f, 0.f);

        for (int st = 0; st < steps; ++st) {
            issue();
            cp_async_wait<D - 1>();
            const int c = st * 32 + lane;
            if (c < K8) {
                const uint4* slot = ring + c_slot * (R * 32) + lane;
                uint4 w[R];
#pragma unroll
                for (int r = 0; r < R; ++r) w[r] = slot[r * 32];
                const uint4* xc = xs4 + c * 8;
                const int sw = c & 7;
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const uint4 xv = xc[e ^ sw];
                    const float2 xp[4] = {bf16x2_to_f32x2(xv.x), bf16x2_to_f32x2(xv.y), bf16x2_to_f32x2(xv.z),
                                          bf16x2_to_f32x2(xv.w)};
#pragma unroll
                    for (int r = 0; r < R; ++r) {
                        const uint32_t word = (e >> 1) == 0 ? w[r].x : (e >> 1) == 1 ? w[r].y
                                            : (e >> 1) == 2 ? w[r].z : w[r].w;
                        const float2 wd = (e & 1) ? bf16_dup<true>(word) : bf16_dup<false>(word);
#pragma unroll
                        for (int p = 0; p < (NT + 1) / 2; ++p) acc[r][p] = ffma2(wd, xp[p], acc[r][p]);
                    }
                }
            }
            if (++c_slot == D) c_slot = 0;
        }

        const int row0 = (g_begin + gi) * R;
        float v[V];
#pragma unroll
        for (int i = 0; i < V; ++i) v[i] = 0.f;
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                v[r * 8 + 2 * p] = acc[r][p].x;
                v[r * 8 + 2 * p + 1] = acc[r][p].y;
            }
        warp_reduce_scatter<V>(v, lane);
        if (result_owner<V>(lane)) {
            constexpr int kHeld = V >= 32 ? V / 32 : 1;
#pragma unroll
            for (int i = 0; i < kHeld; ++i) {
                const int idx = result_index<V>(lane, i);
                const int r = idx >> 3;
                const int t = idx & 7;
                if (r < R && t < NT && row0 + r < M)
                    y[static_cast<long long>(t) * M + row0 + r] = __float2bfloat16_rn(v[i]);
            }
        }
    }
    cp_async_wait<0>();
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
    griddep_wait();
    griddep_launch_dependents();
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
    const int threads = 32 * (g.warps_per_block > 0 && g.warps_per_block <= 8 ? g.warps_per_block : 8);
    // x in FP32: NT * slab8 * 32 bytes; keep it within 192 KB (k-slabs beyond that)
    const long long budget = 192 * 1024;
    long long slab8 = budget / (32LL * NT);
    if (slab8 >= K8) slab8 = K8;
    if (slab8 < 1) slab8 = 1;
    const size_t smem = static_cast<size_t>(NT) * slab8 * 32;
    static SmemOptIn smem_opt;
    cudaError_t e = smem_opt.ensure(reinterpret_cast<const void*>(kern), static_cast<int>(smem));
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
    e = launch_kernel(kern, dim3(static_cast<unsigned>(grid)), dim3(threads), smem, stream, g.pdl,
                      reinterpret_cast<const uint4*>(g.W), reinterpret_cast<const uint4*>(g.x),
                      reinterpret_cast<__nv_bfloat16*>(g.y), g.M, K8, static_cast<int>(slab8));
    if (e == cudaSuccess) e = cudaGetLastError();
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
    cudaError_t e = launch_kernel(gemv_bf16_scalar_kernel<NT>, dim3(static_cast<unsigned>(grid)), dim3(threads), 0,
                                  stream, g.pdl, g.W, g.x, reinterpret_cast<__nv_bfloat16*>(g.y), g.M, g.K);
    if (e == cudaSuccess) e = cudaGetLastError();
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

constexpr int kPipeMaxSmem = 232448;   // 227 KB per CTA

// Shared memory of the pipelined kernel: x (FP32 or BF16) + one ring per warp.
constexpr long long pipe_smem(int NT, int R, int D, bool xf32, int K8, int warps)
{
    return static_cast<long long>(NT) * K8 * (xf32 ? 32 : 16) + static_cast<long long>(warps) * D * R * 512;
}

// Returns 1 and sets *status if the pipelined kernel ran (or failed to launch), 0 if it does not fit.
template <int NT, int R, int D, bool XF32>
int try_launch_pipe(const GemvLaunch& g, cudaStream_t stream, char* msg, size_t msg_len, int* status,
                    int min_warps)
{
    const int K8 = g.K / 8;
    const long long groups = (static_cast<long long>(g.M) + R - 1) / R;
    // Warps per CTA (one CTA per SM): the requested count, else the count in
    // [min_warps, 16] that fits in shared memory and leaves the fewest idle warp
    // slots when every warp takes the same number of row groups.
    int warps = 0;
    if (g.warps_per_block > 0) {
        if (pipe_smem(NT, R, D, XF32, K8, g.warps_per_block) <= kPipeMaxSmem) warps = g.warps_per_block;
    } else {
        double best = -1.0;
        for (int w = 16; w >= min_warps; --w) {
            if (pipe_smem(NT, R, D, XF32, K8, w) > kPipeMaxSmem) continue;
            const long long slots = static_cast<long long>(g.num_sms) * w;
            const long long per = (groups + slots - 1) / slots;
            const double eff = static_cast<double>(groups) / static_cast<double>(per * slots);
            if (eff > best + 1e-9) {
                best = eff;
                warps = w;
            }
        }
    }
    if (warps == 0) return 0;
    const long long smem = pipe_smem(NT, R, D, XF32, K8, warps);
    auto kern = gemv_bf16_pipe_kernel<NT, R, D, XF32>;
    static SmemOptIn smem_opt;
    cudaError_t e = smem_opt.ensure(reinterpret_cast<const void*>(kern), static_cast<int>(smem));
    if (e != cudaSuccess) {
        snprintf(msg, msg_len, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
        *status = 1;
        return 1;
    }
    // Same number of row groups for every warp: size the grid to the work.
    const long long max_warps = static_cast<long long>(g.num_sms) * warps;
    const long long per_warp = (groups + max_warps - 1) / max_warps;
    const long long warps_needed = (groups + per_warp - 1) / per_warp;
    const long long grid = (warps_needed + warps - 1) / warps;
    e = launch_kernel(kern, dim3(static_cast<unsigned>(grid)), dim3(warps * 32), static_cast<size_t>(smem), stream,
                      g.pdl, reinterpret_cast<const uint4*>(g.W), reinterpret_cast<const uint4*>(g.x),
                      reinterpret_cast<__nv_bfloat16*>(g.y), g.M, K8, static_cast<int>(per_warp));
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) {
        snprintf(msg, msg_len, "GEMV launch failed: %s", cudaGetErrorString(e));
        *status = 1;
        return 1;
    }
    *status = 0;
    return 1;
}

// Pipelined kernel with R rows per warp: x in FP32 when that leaves room for at
// least 8 warps (or the requested count), else x in BF16 (converted per use).
template <int NT, int R, int D>
int try_launch_pipe_rows(const GemvLaunch& g, cudaStream_t stream, char* msg, size_t msg_len, int* status)
{
    const int min_warps = g.warps_per_block > 0 ? g.warps_per_block : 8;
    if (g.kernel != 3) {
        if (try_launch_pipe<NT, R, D, true>(g, stream, msg, msg_len, status, min_warps)) return 1;
    }
    return try_launch_pipe<NT, R, D, false>(g, stream, msg, msg_len, status, min_warps);
}

// Token-paired kernel: x (K8 x 8 slots of 16 bytes) + one ring per warp.
template <int NT, int R, int D>
int try_launch_tokpair(const GemvLaunch& g, cudaStream_t stream, char* msg, size_t msg_len, int* status)
{
    const int K8 = g.K / 8;
    const long long x_bytes = static_cast<long long>(K8) * 128;
    const long long per_warp_ring = static_cast<long long>(D) * R * 512;
    const long long groups = (static_cast<long long>(g.M) + R - 1) / R;
    int warps = 0;
    if (g.warps_per_block > 0) {
        if (x_bytes + g.warps_per_block * per_warp_ring <= kPipeMaxSmem) warps = g.warps_per_block;
    } else {
        double best = -1.0;
        for (int w = 16; w >= 8; --w) {
            if (x_bytes + w * per_warp_ring > kPipeMaxSmem) continue;
            const long long slots = static_cast<long long>(g.num_sms) * w;
            const long long per = (groups + slots - 1) / slots;
            const double eff = static_cast<double>(groups) / static_cast<double>(per * slots);
            if (eff > best + 1e-9) {
                best = eff;
                warps = w;
            }
        }
    }
    if (warps == 0) return 0;
    const long long smem = x_bytes + warps * per_warp_ring;
    auto kern = gemv_bf16_tokpair_kernel<NT, R, D>;
    static SmemOptIn smem_opt;
    cudaError_t e = smem_opt.ensure(reinterpret_cast<const void*>(kern), static_cast<int>(smem));
    if (e != cudaSuccess) {
        snprintf(msg, msg_len, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
        *status = 1;
        return 1;
    }
    const long long max_warps = static_cast<long long>(g.num_sms) * warps;
    const long long per_warp = (groups + max_warps - 1) / max_warps;
    const long long warps_needed = (groups + per_warp - 1) / per_warp;
    const long long grid = (warps_needed + warps - 1) / warps;
    e = launch_kernel(kern, dim3(static_cast<unsigned>(grid)), dim3(warps * 32), static_cast<size_t>(smem), stream,
                      g.pdl, reinterpret_cast<const uint4*>(g.W), g.x, reinterpret_cast<__nv_bfloat16*>(g.y), g.M,
                      g.K, static_cast<int>(per_warp));
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) {
        snprintf(msg, msg_len, "GEMV launch failed: %s", cudaGetErrorString(e));
        *status = 1;
        return 1;
    }
    *status = 0;
    return 1;
}

// Kernel choice for the aligned path.  Measured on the 34816 x 5120 decode
// shape: n <= 3 streams fastest from registers (the arithmetic is light and
// the loads of U chunks per lane keep HBM busy; 4 rows per warp for n <= 2,
// 2 rows for n = 3, whose 3 x 4 accumulators per row leave fewer registers
// for loads in flight); at n = 4 the cp.async ring keeps loads in flight
// while the arithmetic runs (x in FP32); for n >= 5 the FMAs dominate and
// the token-paired kernel does the fewest instructions per weight.  (By
// default gemv_bf16 sends n >= 4 to the tensor cores.)
template <int NT>
int launch_vec_any(const GemvLaunch& g, cudaStream_t stream, char* msg, size_t msg_len)
{
    const int kernel = g.kernel != 0 ? g.kernel : (NT <= 3 ? 1 : (NT <= 4 ? 2 : 4));
    if (kernel == 4) {
        const int rows = g.rows_per_warp > 0 ? g.rows_per_warp : 8;
        int status = 0;
        int ran = 0;
        switch (rows) {
        case 4: ran = try_launch_tokpair<NT, 4, 3>(g, stream, msg, msg_len, &status); break;
        case 8: ran = try_launch_tokpair<NT, 8, 2>(g, stream, msg, msg_len, &status); break;
        default:
            snprintf(msg, msg_len, "token-paired GEMV takes rows_per_warp 4 or 8, got %d", rows);
            return 1;
        }
        if (ran) return status;
        if (g.kernel == 4) {
            snprintf(msg, msg_len, "token-paired GEMV does not fit in shared memory for K=%d", g.K);
            return 1;
        }
    }
    const int rows = g.rows_per_warp > 0 ? g.rows_per_warp : (kernel == 1 && NT == 3 ? 2 : 4);
    if (kernel == 2 || kernel == 3 || (kernel == 4)) {
        GemvLaunch gk = g;
        gk.kernel = kernel == 4 ? 3 : kernel;
        int status = 0;
        int ran = 0;
        switch (rows) {
        case 1: ran = try_launch_pipe_rows<NT, 1, 8>(gk, stream, msg, msg_len, &status); break;
        case 2: ran = try_launch_pipe_rows<NT, 2, 5>(gk, stream, msg, msg_len, &status); break;
        case 4: ran = try_launch_pipe_rows<NT, 4, 3>(gk, stream, msg, msg_len, &status); break;
        case 8: ran = try_launch_pipe_rows<NT, 8, 3>(gk, stream, msg, msg_len, &status); break;
        default:
            snprintf(msg, msg_len, "unsupported rows_per_warp %d (1, 2, 4 or 8)", rows);
            return 1;
        }
        if (ran) return status;
        if (g.kernel == 2 || g.kernel == 3) {
            snprintf(msg, msg_len, "pipelined GEMV does not fit in shared memory for K=%d, n=%d", g.K, NT);
            return 1;
        }
    }
    return launch_vec_rows<NT>(g, rows, stream, msg, msg_len);
}

}  // namespace

int launch_gemv(const GemvLaunch& g, cudaStream_t stream, char* msg, size_t msg_len)
{
    const bool vec = (g.K % 8 == 0) && (reinterpret_cast<uintptr_t>(g.W) % 16 == 0) &&
                     (reinterpret_cast<uintptr_t>(g.x) % 16 == 0);
    if (vec) {
        switch (g.n) {
        case 1: return launch_vec_any<1>(g, stream, msg, msg_len);
        case 2: return launch_vec_any<2>(g, stream, msg, msg_len);
        case 3: return launch_vec_any<3>(g, stream, msg, msg_len);
        case 4: return launch_vec_any<4>(g, stream, msg, msg_len);
        case 5: return launch_vec_any<5>(g, stream, msg, msg_len);
        case 6: return launch_vec_any<6>(g, stream, msg, msg_len);
        case 7: return launch_vec_any<7>(g, stream, msg, msg_len);
        case 8: return launch_vec_any<8>(g, stream, msg, msg_len);
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
