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
// heads that read its KV head.  Its warps take tokens in turn, 8 at a time,
// streamed through a per-warp cp.async ring in shared memory; the G x 8 scores
// of a chunk come from tensor-core MMAs (BF16 products, FP32 sums), and an
// online softmax state (running max m, sum l, unnormalised output o) per head
// is kept in base 2 (scores multiplied by scale * log2 e); each lane holds
// head_dim/32 consecutive elements of every head's output.  The warps' states
// are combined in shared memory and the segment's (m, l, o) go to a workspace.
// Kernel 2 (one CTA per query head x sequence x 32 output elements) merges the
// segments:
//   M = max_s m_s,  L = sum_s l_s 2^(m_s - M),  out = sum_s o_s 2^(m_s - M) / L.
// A block-table entry out of range is recorded in the status word and its
// tokens are skipped (no out-of-range read).
#include <cuda_bf16.h>

#include <cmath>
#include <cstdio>

#include "bsk_internal.h"

namespace bsk {
namespace {

constexpr int kAttnWarps = 4;
constexpr int kAttnTokens = 8;   // tokens per warp per ring stage: the N of the score MMA
constexpr int kAttnStages = 3;   // cp.async ring depth per warp

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

// bf16 pair in one 32-bit word -> the two FP32 values (element 0 = low half):
// a bfloat16 is the upper half of a binary32 (byte permutations, integer pipe).
__device__ __forceinline__ float2 bf16x2_to_f32x2(uint32_t w)
{
    uint32_t lo, hi;
    asm("prmt.b32 %0, %1, 0, 0x1044;" : "=r"(lo) : "r"(w));
    asm("prmt.b32 %0, %1, 0, 0x3244;" : "=r"(hi) : "r"(w));
    return make_float2(__uint_as_float(lo), __uint_as_float(hi));
}

// Packed two-lane FP32 FMA: {a.x*b.x + c.x, a.y*b.y + c.y}, each rounded once.
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c)
{
    unsigned long long d;
    const unsigned long long ua = *reinterpret_cast<unsigned long long*>(&a);
    const unsigned long long ub = *reinterpret_cast<unsigned long long*>(&b);
    const unsigned long long uc = *reinterpret_cast<unsigned long long*>(&c);
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(ua), "l"(ub), "l"(uc));
    return *reinterpret_cast<float2*>(&d);
}

// 2^x for x <= 0 (a softmax weight): the hardware approximation, one
// instruction; 2^-inf = +0.
__device__ __forceinline__ float exp2_weight(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// The EPL/2 bf16 pairs of one lane's row slice, widened.
template <int EPL>
__device__ __forceinline__ void widen2(const uint8_t* src, float2 (&f)[EPL / 2])
{
    const typename RowVec<EPL>::T v = *reinterpret_cast<const typename RowVec<EPL>::T*>(src);
    const uint32_t* w = reinterpret_cast<const uint32_t*>(&v);
#pragma unroll
    for (int i = 0; i < EPL / 2; ++i) f[i] = bf16x2_to_f32x2(w[i]);
}

__device__ __forceinline__ uint32_t smem_addr(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Asynchronous global -> shared copy of BYTES (4, 8 or 16); src_bytes = 0
// copies nothing and zero-fills the destination.
template <int BYTES>
__device__ __forceinline__ void cp_async(uint32_t dst, const void* src, uint32_t src_bytes)
{
    if constexpr (BYTES == 16) {
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
                     : "memory");
    } else {
        asm volatile("cp.async.ca.shared.global [%0], [%1], %2, %3;" ::"r"(dst), "l"(src), "n"(BYTES),
                     "r"(src_bytes)
                     : "memory");
    }
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

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

// Shared memory of the split kernel: the warps' cp.async rings, reused after
// the token loop for the warps' (unnormalised) outputs.  Rows of a stage are
// stored with their 16-byte chunks permuted (chunk c of row r at c ^ (r & 7))
// so that the eight rows an ldmatrix reads at once fall in distinct banks.
template <int HD, int G>
struct SplitSmem {
    static constexpr int kRow = HD * 2;                          // bytes of one K or V row
    static constexpr int kStage = 2 * kAttnTokens * kRow;        // T K rows, then T V rows
    static constexpr int kWarpRing = kAttnStages * kStage;
    static constexpr int kRing = kAttnWarps * kWarpRing;
    static constexpr int kOut = kAttnWarps * G * HD * 4;
    static constexpr int kBytes = kRing > kOut ? kRing : kOut;
};

// Byte offset of byte b of row r inside a stage.
template <int ROW>
__device__ __forceinline__ uint32_t swz(int r, int b)
{
    return static_cast<uint32_t>(r * ROW + ((((b >> 4) ^ (r & 7)) << 4) | (b & 15)));
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

// D (16 x 8, FP32) += A (16 x 16, BF16, row-major) * B (16 x 8, BF16, column-major).
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Each warp streams its chunks (T = 8 tokens each; the warps take chunks in
// turn) through a private D-stage ring in shared memory: the copies for chunk
// i+D-1 are issued before chunk i is consumed.  Each lane copies its own slice
// (head_dim/32 values) of every K and V row.
//
// Scores on the tensor cores: S (heads x 8 tokens) = Q (heads x head_dim) K^T
// as head_dim/16 mma.sync m16n8k16 steps, the G query heads as rows 0..G-1 of
// A (held in registers for the whole kernel), the chunk's K rows as B (loaded
// with ldmatrix).  BF16 products are exact and the sums are FP32, as before.
// Lane 4g + c then holds head g's scores for tokens 2c, 2c+1: the four lanes of
// a head find the chunk max, the head's new running max, the weights
// 2^(s - max), their sum and the rescale factor of the old sums, and put the
// weights and factors in shared memory.  The output update stays on the CUDA
// cores in FP32: every lane owns head_dim/32 values of each head's output and
// adds weight x V row (packed FMAs) for the chunk's tokens.
template <int HD, int G>
__global__ void __launch_bounds__(kAttnWarps * 32, 2)
    attn_split_kernel(const AttnParams p)
{
    constexpr int EPL = HD / 32;
    constexpr int LB = EPL * 2;   // bytes per lane per row
    constexpr int T = kAttnTokens;
    constexpr int D = kAttnStages;
    constexpr int KS = HD / 16;   // MMA k-steps
    using SM = SplitSmem<HD, G>;
    static_assert(G <= 8, "at most 8 query heads per KV head (rows of the score MMA)");
    static_assert(KS % 2 == 0, "k-steps are loaded two at a time");
    static_assert(kAttnStages * kAttnTokens <= 32, "the stages' token-validity bits share one 32-bit word");
    const int seg = blockIdx.x;
    const int kvh = blockIdx.y;
    const int seq = blockIdx.z;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int gq = lane >> 2;      // MMA group: the head this lane's scores belong to
    const int cq = lane & 3;       // position in the group: tokens 2cq, 2cq+1

    __shared__ float s_m[kAttnWarps][G];
    __shared__ float s_l[kAttnWarps][G];
    __shared__ float s_f[kAttnWarps][G];   // combine: each warp's weight per head
    __shared__ float s_hm[G], s_hl[G];      // combine: each head's max and sum
    // weights of the chunk and rescale factors, each stored twice ({w, w}): the
    // packed FMAs of the output update take them as pairs straight from memory
    __shared__ __align__(16) float2 s_p[kAttnWarps][T][G];
    __shared__ __align__(16) float2 s_c[kAttnWarps][G];
    extern __shared__ __align__(16) uint8_t smem[];
    // This kernel is a programmatic dependent of the kernel before it in the
    // stream: nothing is read before that kernel has completed.  The merge
    // kernel launched after this one may be scheduled from now on; it waits on
    // the device for this grid to complete before reading anything.
    griddep_wait();
    griddep_launch_dependents();

    int L = p.seq_lens[seq];
    L = L < 0 ? 0 : (L > p.max_seq_len ? p.max_seq_len : L);
    const int seg_len = (L + p.num_segments - 1) / p.num_segments;
    const int t0 = seg * seg_len;
    const int t1 = (t0 + seg_len < L) ? t0 + seg_len : L;

    // A fragments of the query rows: lane (g, c) holds q[g][16s + 2c, +1] and
    // q[g][16s + 2c + 8, +9] for every k-step s (rows 8..15 of A are zero)
    uint32_t qa[KS][2];
    {
        const uint32_t* qrow = reinterpret_cast<const uint32_t*>(
            p.q + (static_cast<long long>(seq) * p.num_q_heads + kvh * G + (gq < G ? gq : 0)) * HD);
#pragma unroll
        for (int k = 0; k < KS; ++k) {
            qa[k][0] = gq < G ? qrow[8 * k + cq] : 0u;
            qa[k][1] = gq < G ? qrow[8 * k + 4 + cq] : 0u;
        }
    }

    constexpr int P = EPL / 2;
    float m_h = -INFINITY, l_h = 0.f;   // running max and sum of head gq (lanes of a head agree)
    float2 o[G][P];
#pragma unroll
    for (int j = 0; j < G; ++j)
#pragma unroll
        for (int e = 0; e < P; ++e) o[j][e] = make_float2(0.f, 0.f);

    const int32_t* bt = p.block_tables + static_cast<long long>(seq) * p.max_blocks;
    const long long tok_stride = static_cast<long long>(p.num_kv_heads) * HD;   // elements between tokens
    const long long head_off = static_cast<long long>(kvh) * HD + lane * EPL;
    uint8_t* wring = smem + warp * SM::kWarpRing;   // this warp's ring
    const uint32_t ring = smem_addr(wring);
    // this lane's slice of row r (< 8) of a stage, and of row 8 + r, relative to
    // row 0 and row 8: slice_off[r] (the row offset r * kRow included)
    uint32_t slice_off[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) slice_off[r] = swz<SM::kRow>(r, lane * LB);
    constexpr int kChunkStep = kAttnWarps * T;
    const int first = t0 + warp * T;
    const int nch = first < t1 ? (t1 - first + kChunkStep - 1) / kChunkStep : 0;

    // Copies chunk i of this warp into ring stage `st`; returns the mask of its
    // tokens that exist (inside the segment, with a valid block).
    auto issue = [&](int i, int st) -> uint32_t {
        const int c0 = first + i * kChunkStep;
        int bi = c0 / p.block_size;
        int off = c0 - bi * p.block_size;
        const uint32_t dst0 = ring + st * SM::kStage;
        if (c0 + T <= t1 && off + T <= p.block_size) {
            // the usual case: the whole chunk inside one page and the segment
            const int blk = bt[bi];
            if (blk >= 0 && blk < p.num_blocks) {
                const long long row = (static_cast<long long>(blk) * p.block_size + off) * tok_stride + head_off;
                const uint16_t* ks = p.k + row;
                const uint16_t* vs = p.v + row;
#pragma unroll
                for (int u = 0; u < T; ++u) {
                    cp_async<LB>(dst0 + slice_off[u], ks, LB);
                    cp_async<LB>(dst0 + T * SM::kRow + slice_off[u], vs, LB);
                    ks += tok_stride;
                    vs += tok_stride;
                }
                cp_async_commit();
                return (1u << T) - 1u;
            }
        }
        uint32_t bits = 0;
#pragma unroll
        for (int u = 0; u < T; ++u) {
            const int t = c0 + u;
            bool ok = t < t1;
            const uint16_t* ks = p.k;
            const uint16_t* vs = p.v;
            if (ok) {
                const int blk = bt[bi];
                if (blk < 0 || blk >= p.num_blocks) {
                    if (lane == 0) *reinterpret_cast<volatile int*>(p.status) = kDevErrBadIndex;
                    ok = false;
                } else {
                    const long long row = (static_cast<long long>(blk) * p.block_size + off) * tok_stride + head_off;
                    ks = p.k + row;
                    vs = p.v + row;
                }
            }
            cp_async<LB>(dst0 + slice_off[u], ks, ok ? LB : 0u);
            cp_async<LB>(dst0 + T * SM::kRow + slice_off[u], vs, ok ? LB : 0u);
            bits |= (ok ? 1u : 0u) << u;
            if (++off == p.block_size) {
                off = 0;
                ++bi;
            }
        }
        cp_async_commit();
        return bits;
    };

    constexpr uint32_t kMask = (1u << T) - 1u;
    uint32_t vbits = 0;   // validity of the tokens held by each stage: bits [st*T, st*T+T)
#pragma unroll
    for (int i = 0; i < D - 1; ++i) {
        uint32_t b = 0;
        if (i < nch) {
            b = issue(i, i);
        } else {
            cp_async_commit();
        }
        vbits |= b << (i * T);
    }

    for (int i = 0; i < nch; ++i) {
        const int st = i % D;
        const int in = i + D - 1;
        const int sn = in % D;
        uint32_t b = 0;
        if (in < nch) {
            b = issue(in, sn);
        } else {
            cp_async_commit();
        }
        vbits = (vbits & ~(kMask << (sn * T))) | (b << (sn * T));
        cp_async_wait<D - 1>();   // chunk i has landed (this lane's copies) ...
        __syncwarp();             // ... and every lane's: the score MMA reads all of them
        const uint32_t okb = (vbits >> (st * T)) & kMask;
        const uint32_t stage = ring + st * SM::kStage;

        // scores: head_dim/16 MMA steps, B fragments (K rows) two steps per ldmatrix
        float sd[4] = {0.f, 0.f, 0.f, 0.f};
        {
            // two accumulators (even and odd k-steps) halve the chain of dependent MMAs
            float se[4] = {0.f, 0.f, 0.f, 0.f};
            const int tk = lane & 7;   // the K row (token) this lane addresses for ldmatrix
#pragma unroll
            for (int k = 0; k + 1 < KS; k += 2) {
                const int chunk = 2 * k + (lane >> 3);   // 16-byte chunk: 8 dims each
                uint32_t b0, b1, b2, b3;
                ldmatrix_x4(stage + tk * SM::kRow + (((chunk ^ tk) & (HD / 8 - 1)) << 4), b0, b1, b2, b3);
                mma_bf16_16816(sd, qa[k][0], 0u, qa[k][1], 0u, b0, b1);
                mma_bf16_16816(se, qa[k + 1][0], 0u, qa[k + 1][1], 0u, b2, b3);
            }
            sd[0] += se[0];
            sd[1] += se[1];
        }
        // softmax arithmetic in the lanes of each head (lane 4g + c: tokens 2c, 2c+1)
        const bool v0 = ((okb >> (2 * cq)) & 1u) != 0;
        const bool v1 = ((okb >> (2 * cq + 1)) & 1u) != 0;
        const float s0 = v0 ? sd[0] * p.scale_log2 : -INFINITY;
        const float s1 = v1 ? sd[1] * p.scale_log2 : -INFINITY;
        float cm = fmaxf(s0, s1);
        cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, 1));
        cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, 2));
        const float m_new = fmaxf(m_h, cm);
        const float p0 = v0 ? exp2_weight(s0 - m_new) : 0.f;
        const float p1 = v1 ? exp2_weight(s1 - m_new) : 0.f;
        const float corr = m_new == -INFINITY ? 1.f : exp2_weight(m_h - m_new);
        float ps = p0 + p1;
        ps += __shfl_xor_sync(0xffffffffu, ps, 1);
        ps += __shfl_xor_sync(0xffffffffu, ps, 2);
        l_h = l_h * corr + ps;
        m_h = m_new;
        if (gq < G) {
            s_p[warp][2 * cq][gq] = make_float2(p0, p0);
            s_p[warp][2 * cq + 1][gq] = make_float2(p1, p1);
            if (cq == 0) s_c[warp][gq] = make_float2(corr, corr);
        }
        __syncwarp();
        // output update: rescale, then weight x V row for each token of the chunk
        const float2 z2 = make_float2(0.f, 0.f);
#pragma unroll
        for (int j = 0; j < G; ++j) {
            const float2 c2 = s_c[warp][j];
#pragma unroll
            for (int e = 0; e < P; ++e) o[j][e] = ffma2(c2, o[j][e], z2);
        }
        const uint8_t* vstage = wring + st * SM::kStage + T * SM::kRow;
#pragma unroll
        for (int u = 0; u < T; ++u) {
            if (!(okb & (1u << u))) continue;
            float2 vf[P];
            widen2<EPL>(vstage + slice_off[u], vf);
#pragma unroll
            for (int j = 0; j < G; ++j) {
                const float2 p2 = s_p[warp][u][j];
#pragma unroll
                for (int e = 0; e < P; ++e) o[j][e] = ffma2(p2, vf[e], o[j][e]);
            }
        }
        __syncwarp();   // s_p and the stage are free for the next chunk
    }
    cp_async_wait<0>();   // the trailing (empty) groups; the ring is reused below

    // combine the warps' states (the ring area now holds the warps' outputs)
    __syncthreads();
    float* s_o = reinterpret_cast<float*>(smem);   // [kAttnWarps][G][HD]
    if (gq < G && cq == 0) {
        s_m[warp][gq] = m_h;
        s_l[warp][gq] = l_h;
    }
#pragma unroll
    for (int j = 0; j < G; ++j) {
        // this lane's EPL consecutive values of head j, in 16-byte (or 8-byte) stores
        float* dst = s_o + (warp * G + j) * HD + lane * EPL;
        if constexpr (EPL % 4 == 0) {
#pragma unroll
            for (int e = 0; e < P; e += 2)
                *reinterpret_cast<float4*>(dst + 2 * e) = make_float4(o[j][e].x, o[j][e].y, o[j][e + 1].x, o[j][e + 1].y);
        } else {
#pragma unroll
            for (int e = 0; e < P; ++e) *reinterpret_cast<float2*>(dst + 2 * e) = o[j][e];
        }
    }
    __syncthreads();
    // per head: M = max_w m_w, the warps' weights 2^(m_w - M) and L = sum_w w l_w,
    // once (G threads), for the CTA's outputs below
    if (threadIdx.x < G) {
        const int j = threadIdx.x;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kAttnWarps; ++w) M = fmaxf(M, s_m[w][j]);
        float Lsum = 0.f;
#pragma unroll
        for (int w = 0; w < kAttnWarps; ++w) {
            const float f = M == -INFINITY ? 0.f : exp2f(s_m[w][j] - M);
            s_f[w][j] = f;
            Lsum = fmaf(f, s_l[w][j], Lsum);
        }
        s_hm[j] = M;
        s_hl[j] = Lsum;
    }
    __syncthreads();

    float* out = p.partial +
                 ((static_cast<long long>(seq) * p.num_q_heads + kvh * G) * p.num_segments + seg) * (HD + 2);
    const long long head_stride = static_cast<long long>(p.num_segments) * (HD + 2);
    for (int i = threadIdx.x; i < G * HD; i += blockDim.x) {
        const int j = i / HD;
        const int e = i - j * HD;
        float O = 0.f;
#pragma unroll
        for (int w = 0; w < kAttnWarps; ++w) O = fmaf(s_f[w][j], s_o[(w * G + j) * HD + e], O);
        float* dst = out + j * head_stride;
        dst[2 + e] = O;
        if (e == 0) {
            dst[0] = s_hm[j];
            dst[1] = s_hl[j];
        }
    }
}

// Block-wide reductions for the merge kernel (blockDim.x a multiple of 32, <= 1024).
__device__ __forceinline__ float block_max(float v, float* s_red)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    if (lane == 0) s_red[warp] = v;
    __syncthreads();
    float r = -INFINITY;
    for (int w = 0; w < nw; ++w) r = fmaxf(r, s_red[w]);
    __syncthreads();
    return r;
}

__device__ __forceinline__ float block_sum(float v, float* s_red)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    if (lane == 0) s_red[warp] = v;
    __syncthreads();
    float r = 0.f;
    for (int w = 0; w < nw; ++w) r += s_red[w];
    __syncthreads();
    return r;
}

constexpr int kMergeWarps = 8;
constexpr int kMergeLoads = 16;   // o_s loads in flight per lane

// One CTA per (query head x sequence, 32 output elements).  It is launched as
// a programmatic dependent of the split kernel, so it may be scheduled while
// the split kernel's last CTAs still run; griddepcontrol.wait holds it until
// that grid has completed and its partials are visible.  Then, in one round of
// loads, each thread fetches (m_s, l_s) of its segments and the o_s[e] its warp
// sums (every 8th segment, the CTA's 32 elements, one per lane).  M = max_s
// m_s, weights w_s = 2^(m_s - M) (in shared memory), L = sum_s w_s l_s; each
// warp sums w_s o_s[e] and the eight partial sums are added: out[e] = sum / L.
template <int HD>
__global__ void __launch_bounds__(kMergeWarps * 32)
    attn_merge_kernel(const float* __restrict__ partial, __nv_bfloat16* __restrict__ out, int num_segments)
{
    extern __shared__ float s_w[];   // [num_segments]
    __shared__ float s_red[32];
    __shared__ float s_acc[kMergeWarps][32];
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int head = blockIdx.x;   // seq * num_q_heads + q head
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    constexpr int kThreads = kMergeWarps * 32;
    constexpr int kPerThread = 1024 / kThreads;   // num_segments <= 1024
    const float* base = partial + static_cast<long long>(head) * num_segments * (HD + 2);
    const int e = blockIdx.y * 32 + lane;
    const float* po = base + 2 + e;
    // the first kMergeLoads of this warp's o_s[e], loaded together with (m_s, l_s)
    float v0[kMergeLoads];
#pragma unroll
    for (int u = 0; u < kMergeLoads; ++u) {
        const int s = warp + u * kMergeWarps;
        v0[u] = s < num_segments ? po[static_cast<long long>(s) * (HD + 2)] : 0.f;
    }
    float ms[kPerThread], ls[kPerThread];
#pragma unroll
    for (int i = 0; i < kPerThread; ++i) {
        const int s = threadIdx.x + i * kThreads;
        ms[i] = -INFINITY;
        ls[i] = 0.f;
        if (s < num_segments) {
            ms[i] = base[static_cast<long long>(s) * (HD + 2)];
            ls[i] = base[static_cast<long long>(s) * (HD + 2) + 1];
        }
    }
    float mx = -INFINITY;
#pragma unroll
    for (int i = 0; i < kPerThread; ++i) mx = fmaxf(mx, ms[i]);
    const float M = block_max(mx, s_red);
    float lsum = 0.f;
#pragma unroll
    for (int i = 0; i < kPerThread; ++i) {
        const int s = threadIdx.x + i * kThreads;
        if (s < num_segments) {
            const float w = M == -INFINITY ? 0.f : exp2f(ms[i] - M);
            s_w[s] = w;
            lsum = fmaf(w, ls[i], lsum);
        }
    }
    const float Lsum = block_sum(lsum, s_red);   // its barriers also publish s_w
    float O = 0.f;
#pragma unroll
    for (int u = 0; u < kMergeLoads; ++u) {
        const int s = warp + u * kMergeWarps;
        if (s < num_segments) O = fmaf(s_w[s], v0[u], O);
    }
    for (int s0 = warp + kMergeWarps * kMergeLoads; s0 < num_segments; s0 += kMergeWarps * kMergeLoads) {
        float v[kMergeLoads];
#pragma unroll
        for (int u = 0; u < kMergeLoads; ++u) {
            const int s = s0 + u * kMergeWarps;
            v[u] = s < num_segments ? po[static_cast<long long>(s) * (HD + 2)] : 0.f;
        }
#pragma unroll
        for (int u = 0; u < kMergeLoads; ++u) {
            const int s = s0 + u * kMergeWarps;
            if (s < num_segments) O = fmaf(s_w[s], v[u], O);
        }
    }
    s_acc[warp][lane] = O;
    __syncthreads();
    if (warp == 0) {
        float sum = 0.f;
#pragma unroll
        for (int w = 0; w < kMergeWarps; ++w) sum += s_acc[w][lane];
        out[static_cast<long long>(head) * HD + e] = __float2bfloat16_rn(Lsum > 0.f ? sum / Lsum : 0.f);
    }
}

template <int HD, int G>
int launch_split(const AttnLaunch& a, const AttnParams& p, cudaStream_t stream, char* msg, size_t msg_len)
{
    const int smem = SplitSmem<HD, G>::kBytes;
    auto kern = attn_split_kernel<HD, G>;
    static SmemOptIn smem_opt;
    cudaError_t e = smem_opt.ensure(reinterpret_cast<const void*>(kern), smem);
    if (e != cudaSuccess) {
        snprintf(msg, msg_len, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
        return 1;
    }
    dim3 grid(a.num_segments, a.num_kv_heads, a.num_seqs);
    e = launch_kernel(kern, grid, dim3(kAttnWarps * 32), static_cast<size_t>(smem), stream, a.pdl, p);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) {
        snprintf(msg, msg_len, "attention launch failed: %s", cudaGetErrorString(e));
        return 1;
    }
    // The merge is a programmatic dependent of the split kernel: it may be
    // scheduled before the split grid has finished and waits on the device.
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.num_seqs * a.num_q_heads, HD / 32, 1);
    cfg.blockDim = dim3(kMergeWarps * 32, 1, 1);
    cfg.dynamicSmemBytes = a.num_segments * sizeof(float);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, attn_merge_kernel<HD>, static_cast<const float*>(p.partial),
                           reinterpret_cast<__nv_bfloat16*>(a.out), a.num_segments);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) {
        snprintf(msg, msg_len, "attention merge launch failed: %s", cudaGetErrorString(e));
        return 1;
    }
    return 0;
}

// CTAs of the split kernel that fit on one SM (its shared memory and
// registers), queried once per instance and device.
template <int HD, int G>
int split_ctas_per_sm()
{
    static std::atomic<int> cached[SmemOptIn::kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= SmemOptIn::kMaxDevices) dev = -1;
    int n = dev >= 0 ? cached[dev].load(std::memory_order_acquire) : 0;
    if (n > 0) return n;
    const int smem = SplitSmem<HD, G>::kBytes;
    auto kern = attn_split_kernel<HD, G>;
    static SmemOptIn smem_opt;
    if (smem_opt.ensure(reinterpret_cast<const void*>(kern), smem) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kAttnWarps * 32, smem) != cudaSuccess || n < 1) {
        cudaGetLastError();
        return 1;
    }
    if (dev >= 0) cached[dev].store(n, std::memory_order_release);
    return n;
}

template <int HD>
int ctas_per_sm_hd(int group)
{
    switch (group) {
    case 1: return split_ctas_per_sm<HD, 1>();
    case 2: return split_ctas_per_sm<HD, 2>();
    case 4: return split_ctas_per_sm<HD, 4>();
    case 8: return split_ctas_per_sm<HD, 8>();
    default: return 1;
    }
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

int attention_ctas_per_sm(int head_dim, int q_per_kv)
{
    switch (head_dim) {
    case 64: return ctas_per_sm_hd<64>(q_per_kv);
    case 128: return ctas_per_sm_hd<128>(q_per_kv);
    case 256: return ctas_per_sm_hd<256>(q_per_kv);
    default: return 1;
    }
}

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
