// attention.cu -- decode attention over a paged BF16 KV cache, split along the
// sequence ("split-KV") and merged with a numerically stable softmax reduction.
//
// DCU decode-GEMV article (forum.sourcefind.cn):
//   section 6.1: for one query head, scores[1,L] = Q K^T, prob = softmax(scores),
//     out[1,D] = prob V, with K/V kept as paged blocks [block, token_in_block,
//     kv_head, head_dim];
//   section 6.3: the sequence is cut into contiguous segments; each segment
//     computes its own Q K^T, local maximum, local softmax denominator and local
//     prob V; the segments cannot simply be added, so a final step rescales each
//     segment's sums by exp(local max - global max) and normalises once;
//   section 7: 16 query heads over 4 KV heads, head_dim 256, page size 784;
//     16 segments, or 32 once the longest sequence reaches 12,288 tokens.
//
// Kernel 1 (one CTA per segment x KV head x sequence): the CTA owns the G query
// heads that read its KV head.  Each lane holds head_dim/32 consecutive
// elements of every q, k and v row; warps take tokens in turn, T at a time,
// compute the G dot products with warp shuffles and keep an online softmax
// state (running max m, sum l, unnormalised output o) per head in base-2
// (scores pre-multiplied by scale * log2 e).  The warps' states are combined in
// shared memory and the segment's (m, l, o) go to a workspace.
// Kernel 2 (one CTA per query head x sequence) merges the segments:
//   M = max_s m_s,  L = sum_s l_s 2^(m_s - M),  out = sum_s o_s 2^(m_s - M) / L.
// A block-table entry out of range is recorded in the status word and its
// tokens are skipped (no out-of-range read).
#include <cuda_bf16.h>

#include <cmath>
#include <cstdio>

#include "bsk_internal.h"

namespace bsk {
namespace {

constexpr int kAttnWarps = 8;
constexpr int kAttnTokens = 4;   // tokens per warp per iteration (loads in flight)

template <int EPL>
struct RowVec;   // EPL bf16 values per lane
template <>
struct RowVec<8> {
    using T = uint4;
};
template <>
struct RowVec<4> {
    using T = uint2;
};
template <>
struct RowVec<2> {
    using T = uint32_t;
};

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

template <int EPL>
__device__ __forceinline__ void widen(const typename RowVec<EPL>::T& v, float (&f)[EPL])
{
    if constexpr (EPL == 8) {
        f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x); f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
        f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z); f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
    } else if constexpr (EPL == 4) {
        f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x); f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
    } else {
        f[0] = bf16_lo(v); f[1] = bf16_hi(v);
    }
}

template <int EPL>
__device__ __forceinline__ typename RowVec<EPL>::T zero_vec()
{
    if constexpr (EPL == 8) {
        return make_uint4(0u, 0u, 0u, 0u);
    } else if constexpr (EPL == 4) {
        return make_uint2(0u, 0u);
    } else {
        return 0u;
    }
}

struct AttnParams {
    const uint16_t* q;
    const uint16_t* k;
    const uint16_t* v;
    const int32_t* block_tables;
    const int32_t* seq_lens;
    float* partial;          // [num_seqs, num_q_heads, num_segments, HD + 2]
    int num_q_heads, num_kv_heads;
    int block_size, max_blocks, num_blocks, max_seq_len, num_segments;
    float scale_log2;        // softmax scale * log2(e)
    int* status;
};

template <int HD, int G>
__global__ void __launch_bounds__(kAttnWarps * 32)
    attn_split_kernel(const AttnParams p)
{
    constexpr int EPL = HD / 32;
    using Vec = typename RowVec<EPL>::T;
    const int seg = blockIdx.x;
    const int kvh = blockIdx.y;
    const int seq = blockIdx.z;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    __shared__ float s_m[kAttnWarps][G];
    __shared__ float s_l[kAttnWarps][G];
    extern __shared__ float s_o[];   // [kAttnWarps][G][HD]

    int L = p.seq_lens[seq];
    L = L < 0 ? 0 : (L > p.max_seq_len ? p.max_seq_len : L);
    const int seg_len = (L + p.num_segments - 1) / p.num_segments;
    const int t0 = seg * seg_len;
    const int t1 = (t0 + seg_len < L) ? t0 + seg_len : L;

    // this lane's slice of the G query rows, pre-scaled into the base-2 domain
    float qf[G][EPL];
#pragma unroll
    for (int j = 0; j < G; ++j) {
        const Vec qv = *reinterpret_cast<const Vec*>(
            p.q + (static_cast<long long>(seq) * p.num_q_heads + kvh * G + j) * HD + lane * EPL);
        widen<EPL>(qv, qf[j]);
#pragma unroll
        for (int e = 0; e < EPL; ++e) qf[j][e] *= p.scale_log2;
    }

    float m[G], l[G], o[G][EPL];
#pragma unroll
    for (int j = 0; j < G; ++j) {
        m[j] = -INFINITY;
        l[j] = 0.f;
#pragma unroll
        for (int e = 0; e < EPL; ++e) o[j][e] = 0.f;
    }

    const int32_t* bt = p.block_tables + static_cast<long long>(seq) * p.max_blocks;
    constexpr int T = kAttnTokens;
    constexpr int V = T * G;   // scores per iteration, index u * G + j
    // Warps take T-token chunks of the segment in turn; within a chunk the
    // block and in-block offset advance incrementally (one division per chunk).
    for (int c0 = t0 + warp * T; c0 < t1; c0 += kAttnWarps * T) {
        Vec kv[T], vv[T];
        bool ok[T];
        int bi = c0 / p.block_size;
        int off = c0 - bi * p.block_size;
#pragma unroll
        for (int u = 0; u < T; ++u) {
            const int t = c0 + u;
            ok[u] = t < t1;
            kv[u] = zero_vec<EPL>();
            vv[u] = zero_vec<EPL>();
            if (ok[u]) {
                const int blk = bt[bi];
                if (blk < 0 || blk >= p.num_blocks) {
                    if (lane == 0) *reinterpret_cast<volatile int*>(p.status) = kDevErrBadIndex;
                    ok[u] = false;
                } else {
                    const long long row =
                        ((static_cast<long long>(blk) * p.block_size + off) * p.num_kv_heads + kvh) * HD + lane * EPL;
                    kv[u] = *reinterpret_cast<const Vec*>(p.k + row);
                    vv[u] = *reinterpret_cast<const Vec*>(p.v + row);
                }
            }
            if (++off == p.block_size) {
                off = 0;
                ++bi;
            }
        }
        // partial dot products, then a butterfly that leaves each lane pair one
        // full score, then a broadcast of all V scores to every lane
        float sc[V];
#pragma unroll
        for (int u = 0; u < T; ++u) {
            float kf[EPL];
            widen<EPL>(kv[u], kf);
#pragma unroll
            for (int j = 0; j < G; ++j) {
                float d = 0.f;
#pragma unroll
                for (int e = 0; e < EPL; ++e) d = fmaf(qf[j][e], kf[e], d);
                sc[u * G + j] = d;
            }
        }
        float red[V];
#pragma unroll
        for (int i = 0; i < V; ++i) red[i] = sc[i];
        constexpr int kSteps = V >= 32 ? 5 : (V >= 16 ? 4 : (V >= 8 ? 3 : (V >= 4 ? 2 : (V >= 2 ? 1 : 0))));
#pragma unroll
        for (int st = 0; st < kSteps; ++st) {
            const int offs = 16 >> st;
            const int half = V >> (st + 1);
            const bool upper = (lane & offs) != 0;
#pragma unroll
            for (int i = 0; i < half; ++i) {
                const float send = upper ? red[i] : red[i + half];
                const float keep = upper ? red[i + half] : red[i];
                red[i] = keep + __shfl_xor_sync(0xffffffffu, send, offs);
            }
        }
#pragma unroll
        for (int st = kSteps; st < 5; ++st) red[0] += __shfl_xor_sync(0xffffffffu, red[0], 16 >> st);
        // lane holding score i: its bits map to lane bits 4, 3, ... from the top
#pragma unroll
        for (int i = 0; i < V; ++i) {
            int src = 0;
#pragma unroll
            for (int st = 0; st < kSteps; ++st)
                if (i & (V >> (st + 1))) src |= 16 >> st;
            sc[i] = __shfl_sync(0xffffffffu, red[0], src);
        }
        // online softmax, once per T tokens; rescale only when the max moves
#pragma unroll
        for (int j = 0; j < G; ++j) {
            float cm = -INFINITY;
#pragma unroll
            for (int u = 0; u < T; ++u)
                if (ok[u]) cm = fmaxf(cm, sc[u * G + j]);
            if (cm == -INFINITY) continue;
            if (cm > m[j]) {
                const float corr = exp2f(m[j] - cm);
                l[j] *= corr;
#pragma unroll
                for (int e = 0; e < EPL; ++e) o[j][e] *= corr;
                m[j] = cm;
            }
#pragma unroll
            for (int u = 0; u < T; ++u) {
                const float pu = ok[u] ? exp2f(sc[u * G + j] - m[j]) : 0.f;
                l[j] += pu;
                float vf[EPL];
                widen<EPL>(vv[u], vf);
#pragma unroll
                for (int e = 0; e < EPL; ++e) o[j][e] = fmaf(pu, vf[e], o[j][e]);
            }
        }
    }

    // combine the warps' states
    if (lane == 0) {
#pragma unroll
        for (int j = 0; j < G; ++j) {
            s_m[warp][j] = m[j];
            s_l[warp][j] = l[j];
        }
    }
#pragma unroll
    for (int j = 0; j < G; ++j)
#pragma unroll
        for (int e = 0; e < EPL; ++e) s_o[(warp * G + j) * HD + lane * EPL + e] = o[j][e];
    __syncthreads();

    float* out = p.partial +
                 ((static_cast<long long>(seq) * p.num_q_heads + kvh * G) * p.num_segments + seg) * (HD + 2);
    const long long head_stride = static_cast<long long>(p.num_segments) * (HD + 2);
    for (int i = threadIdx.x; i < G * HD; i += blockDim.x) {
        const int j = i / HD;
        const int e = i - j * HD;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kAttnWarps; ++w) M = fmaxf(M, s_m[w][j]);
        float O = 0.f, Lsum = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < kAttnWarps; ++w) {
                const float f = exp2f(s_m[w][j] - M);
                O = fmaf(f, s_o[(w * G + j) * HD + e], O);
                Lsum = fmaf(f, s_l[w][j], Lsum);
            }
        }
        float* dst = out + j * head_stride;
        dst[2 + e] = O;
        if (e == 0) {
            dst[0] = M;
            dst[1] = Lsum;
        }
    }
}

template <int HD>
__global__ void __launch_bounds__(256)
    attn_merge_kernel(const float* __restrict__ partial, __nv_bfloat16* __restrict__ out, int num_segments)
{
    const int head = blockIdx.x;   // seq * num_q_heads + q head
    const float* base = partial + static_cast<long long>(head) * num_segments * (HD + 2);
    float M = -INFINITY;
    for (int s = 0; s < num_segments; ++s) M = fmaxf(M, base[static_cast<long long>(s) * (HD + 2)]);
    float Lsum = 0.f;
    if (M != -INFINITY)
        for (int s = 0; s < num_segments; ++s) {
            const float* ps = base + static_cast<long long>(s) * (HD + 2);
            Lsum = fmaf(exp2f(ps[0] - M), ps[1], Lsum);
        }
    for (int e = threadIdx.x; e < HD; e += blockDim.x) {
        float O = 0.f;
        if (M != -INFINITY)
            for (int s = 0; s < num_segments; ++s) {
                const float* ps = base + static_cast<long long>(s) * (HD + 2);
                O = fmaf(exp2f(ps[0] - M), ps[2 + e], O);
            }
        out[static_cast<long long>(head) * HD + e] = __float2bfloat16_rn(Lsum > 0.f ? O / Lsum : 0.f);
    }
}

template <int HD, int G>
int launch_split(const AttnLaunch& a, const AttnParams& p, cudaStream_t stream, char* msg, size_t msg_len)
{
    const size_t smem = static_cast<size_t>(kAttnWarps) * G * HD * sizeof(float);
    auto kern = attn_split_kernel<HD, G>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) {
        snprintf(msg, msg_len, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
        return 1;
    }
    dim3 grid(a.num_segments, a.num_kv_heads, a.num_seqs);
    kern<<<grid, kAttnWarps * 32, smem, stream>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) {
        snprintf(msg, msg_len, "attention launch failed: %s", cudaGetErrorString(e));
        return 1;
    }
    const int merge_threads = HD < 256 ? HD : 256;
    attn_merge_kernel<HD><<<a.num_seqs * a.num_q_heads, merge_threads, 0, stream>>>(
        p.partial, reinterpret_cast<__nv_bfloat16*>(a.out), a.num_segments);
    e = cudaGetLastError();
    if (e != cudaSuccess) {
        snprintf(msg, msg_len, "attention merge launch failed: %s", cudaGetErrorString(e));
        return 1;
    }
    return 0;
}

template <int HD>
int launch_hd(const AttnLaunch& a, const AttnParams& p, cudaStream_t stream, char* msg, size_t msg_len)
{
    switch (a.num_q_heads / a.num_kv_heads) {
    case 1: return launch_split<HD, 1>(a, p, stream, msg, msg_len);
    case 2: return launch_split<HD, 2>(a, p, stream, msg, msg_len);
    case 4: return launch_split<HD, 4>(a, p, stream, msg, msg_len);
    case 8: return launch_split<HD, 8>(a, p, stream, msg, msg_len);
    default:
        snprintf(msg, msg_len, "query heads per KV head must be 1, 2, 4 or 8");
        return 1;
    }
}

}  // namespace

int launch_decode_attention(const AttnLaunch& a, cudaStream_t stream, char* msg, size_t msg_len)
{
    AttnParams p;
    p.q = a.q;
    p.k = a.k_cache;
    p.v = a.v_cache;
    p.block_tables = a.block_tables;
    p.seq_lens = a.seq_lens;
    p.partial = a.workspace;
    p.num_q_heads = a.num_q_heads;
    p.num_kv_heads = a.num_kv_heads;
    p.block_size = a.block_size;
    p.max_blocks = a.max_blocks;
    p.num_blocks = a.num_blocks;
    p.max_seq_len = a.max_seq_len;
    p.num_segments = a.num_segments;
    p.scale_log2 = a.scale * 1.4426950408889634f;   // log2(e)
    p.status = a.status;
    switch (a.head_dim) {
    case 64: return launch_hd<64>(a, p, stream, msg, msg_len);
    case 128: return launch_hd<128>(a, p, stream, msg, msg_len);
    case 256: return launch_hd<256>(a, p, stream, msg, msg_len);
    default:
        snprintf(msg, msg_len, "head_dim must be 64, 128 or 256, got %d", a.head_dim);
        return 1;
    }
}

}  // namespace bsk
