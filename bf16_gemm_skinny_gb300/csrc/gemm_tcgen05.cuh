// gemm_tcgen05.cuh -- persistent, warp-specialised tcgen05 GEMM kernels for
// sm_103a, shared by the translation units that instantiate them (the 16-bit
// GEMMs in gemm_tcgen05.cu, the FP8 GEMMs in gemm_fp8.cu).
//
// Computes C = A * B with FP32 accumulation in tensor memory and one rounding
// to the output type in the epilogue ("MTT S4000 GEMM 优化中的分块、尾处理与并发实战复盘",
// section 1: FP16 in, FP32 accumulate, FP16 out; section 2: the column-major
// addressing A(m,k) = A[m + k*M], B(k,n) = B[k + n*K], C(m,n) = C[m + n*M]).
// The FP8 instances (E4M3 or E5M2 in, FP32 accumulate: the FP8 row of the
// matrix-instruction table in "Hygon 优化", section DUMMA 矩阵指令形状) run the
// same pipeline on tcgen05.mma kind::f8f6f4: a stage still holds one 128-byte
// k row per operand row (128 FP8 values), and each MMA still reads 32 bytes of
// it (32 FP8 values instead of 16 half values).
//
// Structure (one CTA per SM, 192 threads):
//   warp 0      TMA producer: fills a STAGES-deep ring of (A, B) k-slices
//               ("Hygon 优化", section 软件流水线: overlap the k-loop loads with
//               the MMAs; the per-stage bytes are (BM + BN) * BK * element size).
//   warp 1      allocates TMEM and issues tcgen05.mma from one thread; each
//               stage's smem slot is released by tcgen05.commit when its MMAs
//               have read it.
//   warps 2..5  epilogue: tcgen05.ld of the FP32 accumulator, optional bias or
//               scale, rounding to the output type, store to C (TMA store for
//               16-bit outputs with 16-byte-aligned C, else masked stores).
//               There is no FP32 intermediate matrix and no separate conversion
//               kernel.
// The accumulator is double-buffered in TMEM (2 x BN columns) so the epilogue
// of tile i overlaps the mainloop of tile i+1.  Tiles are visited in the
// grouped (GROUP_M) order of "Hygon 优化", section 分组调度.
//
// Schedules (the same roles walk the same sequence of (tile, k-blocks)):
//   * whole tiles, fixed: unit u of U (a CTA, or a CTA pair) takes tiles
//     u, u + U, ... in the grouped order;
//   * stream-K: whole waves as above, then the last wave's (tile, k-block)
//     iterations shared evenly; the unit holding a split tile's first k-block
//     adds the others' FP32 partials (workspace slots released by GPU-scope
//     flags) in unit order; the launch is cooperative;
//   * dynamic order (CTA pairs): one cluster per tile launched; a pair that is
//     done takes the tile of a cluster whose launch it cancels (cluster launch
//     control), the answers passed to every role through a small ring.
// Whole-tile launches are programmatic dependents of the kernel before them:
// the prologue (barriers, TMEM, tensor-map and L2 prefetches) runs first and
// griddepcontrol.wait comes before any global read or write.
//
// Tails: TMA zero-fills the parts of a box outside the tensor (M, N and K
// tails contribute zero products; a zero byte is +0 in both FP8 formats) and
// the TMA store / masked store drop rows and columns outside C ("Hygon 优化",
// section DUMMA 矩阵指令形状, on tail masks).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdio>
#include <type_traits>

#include "bsk_internal.h"
#include "ptx.cuh"

namespace bsk {
namespace {

constexpr int kBM = 128;      // tile rows (TMEM lanes), one MMA of M = 128
constexpr int kRowBytes = 128;  // k per stage: one 128-byte swizzle row (64 16-bit or 128 8-bit values)
constexpr int kMmaBytes = 32;   // k bytes per tcgen05.mma: 16 values of kind::f16, 32 of kind::f8f6f4
constexpr int kThreads = 192;

// Per-type constants of one kernel instance.
template <int IN, int OUT>
struct Types {
    static constexpr bool kFp8 = IN == kInE4M3 || IN == kInE5M2;
    static constexpr int kElemBytes = kFp8 ? 1 : 2;
    static constexpr int kBK = kRowBytes / kElemBytes;   // k values per stage
    static constexpr int kOutBytes = OUT == kOutF32 ? 4 : 2;
    static_assert(kFp8 || OUT == IN, "16-bit inputs produce the same 16-bit type");
    __host__ __device__ static constexpr uint32_t idesc(bool a_mn, bool b_mn, int m, int n)
    {
        return kFp8 ? idesc_f8f6f4(IN == kInE5M2 ? 1u : 0u, IN == kInE5M2 ? 1u : 0u, m, n)
                    : idesc_f16(IN == kInBF16, a_mn, b_mn, m, n);
    }
};
constexpr int kEpiWarps = 4;
constexpr int kEpiBox = 32;   // epilogue chunk: 32 rows x 32 columns per warp

template <int BN>
struct Cfg {
    // ring depth: as many stages as fit next to the epilogue buffers
    static constexpr int kStages = BN == 256 ? 4 : BN == 128 ? 6 : BN == 64 ? 8 : 10;
    static constexpr int kABytes = kBM * kRowBytes;
    static constexpr int kBBytes = BN * kRowBytes;
    static constexpr int kStageBytes = kABytes + kBBytes;
    static constexpr int kEpiBufBytes = kEpiBox * kEpiBox * 2;
    static constexpr int kEpiBufs = 2;   // staging buffers per epilogue warp
    static constexpr int kEpiBytes = kEpiWarps * kEpiBufs * kEpiBufBytes;
    static constexpr int kTmemCols = 2 * BN;
    static constexpr int kNumBars = 2 * kStages + 5;
    static constexpr int kBarBytes = 256;
    static constexpr int kSmemBytes = 1024 + kStages * kStageBytes + kEpiBytes + kBarBytes;
    static_assert(kNumBars * 8 + 8 <= kBarBytes, "barrier area too small");
    static_assert(kSmemBytes <= 232448, "shared memory budget exceeded");
};

struct Params {
    int M, N, K;
    // Rows of C per tile: 128 (the MMA's M), or fewer -- a multiple of 8 -- in
    // the balanced schedule of the one-CTA kernel with a K-major A, where every
    // CTA gets the same number of rows (the rows past `bm` that the MMA still
    // computes come from stale shared memory and are not stored).
    int bm;
    int num_m, num_n, num_tiles, num_kb;
    int group_m;
    void* C;
    long long ldc;
    int tma_store;
    const uint16_t* bias;   // optional, output precision: bias[m] (mode 1) or bias[n] (mode 2)
    int bias_mode;
    float alpha;            // FP8 inputs: scale of the FP32 accumulator
    // Stream-K schedule: the first sk_dp_tiles tiles (whole waves) go to the
    // units (CTAs, or CTA pairs) whole, unit + j * G, so that the tiles in flight
    // together stay neighbours in the GROUP_M order; the remaining tiles'
    // I = (num_tiles - sk_dp_tiles) * num_kb (tile, k-block) iterations are then
    // shared out: unit c of G takes [c*I/G, (c+1)*I/G) in tile order.  A tile
    // split between units is finished by the unit that holds its first
    // k-block; the others leave FP32 partials in their slots (one per CTA).
    int sk;                 // 1: stream-K, 0: whole tiles, unit + j * units
    int sk_dp_tiles;        // tiles handed out whole first (a multiple of the unit count)
    long long sk_iters;     // (num_tiles - sk_dp_tiles) * num_kb
    float* sk_part;         // [gridDim.x][tile width][128]: a CTA's 128 rows of a tile, column-major
    int* sk_flag;           // [gridDim.x], zero at launch: set once a CTA's slot is written
    int* status;
    unsigned long long wait_limit_ns;
    // CTA pairs, whole tiles: 1 = dynamic tile order (the grid holds one cluster
    // per tile; later tiles come from clusters whose launch is cancelled)
    int dyn;
    // One-CTA kernel: split-K over a cluster of skc CTAs (0 = off).  CTA r of
    // the cluster takes k-blocks [r*kb/skc, (r+1)*kb/skc) of tile blockIdx.x /
    // skc, leaves its FP32 partial in its own shared memory, and after a
    // cluster barrier sums columns [r*BN/skc, (r+1)*BN/skc) of the tile over
    // all skc partials (in rank order) and stores them.
    int skc;
    // One-CTA kernel, K-major A, whole tiles: the epilogue warps prefetch k-blocks
    // [2, 2 + pf_kb) of their first tile's A rows into L2 before the dependency wait.
    // CTA pairs, whole tiles: with rev_round = R > 0 the tiles of odd rounds
    // (tile / R odd; R = the pairs of the fixed order) run their k loop from the
    // last k-block down, so that a round starts on the A panels' k-slices the
    // round before it read last, which are still in L2.
    int rev_round;
    const uint8_t* a_rows;  // A's first row
    long long a_ld_bytes;   // bytes between A's rows
    int pf_kb;
};

// The work of one unit (a CTA, or a CTA pair) of `units` as a sequence of
// segments (tile, k-blocks [kb0, kb1)).
struct SegCursor {
    long long tile;       // whole-tile phase: next tile (step `step`) while < dp_end
    long long dp_end;
    long long pos, end;   // shared phase: iteration range, counted from the first shared tile
    int step;
};

__device__ __forceinline__ SegCursor seg_first(const Params& p, int unit, int units)
{
    if (p.skc > 1) {
        const long long base = static_cast<long long>(unit / p.skc) * p.num_kb;
        const long long r = unit % p.skc;
        return {0, 0, base + r * p.num_kb / p.skc, base + (r + 1) * p.num_kb / p.skc, 1};
    }
    if (p.sk) {
        return {static_cast<long long>(unit), static_cast<long long>(p.sk_dp_tiles),
                static_cast<long long>(unit) * p.sk_iters / units,
                static_cast<long long>(unit + 1) * p.sk_iters / units, units};
    }
    return {static_cast<long long>(unit), static_cast<long long>(p.num_tiles), 0, 0, units};
}

__device__ __forceinline__ bool seg_next(const Params& p, SegCursor& c, int& tile, int& kb0, int& kb1)
{
    if (c.tile < c.dp_end) {
        tile = static_cast<int>(c.tile);
        kb0 = 0;
        kb1 = p.num_kb;
        c.tile += c.step;
        return true;
    }
    if (c.pos >= c.end) return false;
    const int rel = static_cast<int>(c.pos / p.num_kb);
    const long long t0 = static_cast<long long>(rel) * p.num_kb;
    const long long e = c.end < t0 + p.num_kb ? c.end : t0 + p.num_kb;
    tile = p.sk_dp_tiles + rel;
    kb0 = static_cast<int>(c.pos - t0);
    kb1 = static_cast<int>(e - t0);
    c.pos = e;
    return true;
}

// The unit whose stream-K share holds iteration i of the shared phase: the
// largest c with c*I/G <= i.
__device__ __forceinline__ int sk_unit_of(const Params& p, long long i, int units)
{
    return static_cast<int>(((i + 1) * static_cast<long long>(units) + p.sk_iters - 1) / p.sk_iters) - 1;
}

// Stream-K fix-up: adds to r[j] the FP32 partials that CTAs first .. last left
// for this lane's row, column j of the current 32-column chunk (p0 points at
// CTA 0's slot entry for the chunk's first column; slots are `slot` floats
// apart, columns 128 floats).  The slots are read four at a time so that
// their loads are in flight together; the sums are taken in slot order.
__device__ __forceinline__ void add_partials(uint32_t (&r)[32], const float* p0, long long slot, int first, int last)
{
    for (int q = first; q <= last; q += 4) {
        float v[4][32];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            if (q + u <= last) {
                const float* pq = p0 + static_cast<long long>(q + u) * slot;
#pragma unroll
                for (int j = 0; j < 32; ++j) v[u][j] = pq[j * kBM];
            }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            if (q + u <= last) {
#pragma unroll
                for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) + v[u][j]);
            }
        }
    }
}

// Identifiers of the waits, reported in the status word on a timeout.
enum WaitSite {
    kSiteProducerEmpty = 1,
    kSiteMmaTmemEmpty = 2,
    kSiteMmaFull = 3,
    kSiteEpilogueTmemFull = 4,
    kSiteMmaDrain = 5,
    kSiteProducerDrain = 6,
    kSiteStreamKPartial = 7,
    kSiteSchedFull = 8,
    kSiteSchedEmpty = 9,
};

// Dynamic tile order of the CTA-pair kernel (Params::dyn).  Cluster c of the
// grid starts on tile c; each later tile of a pair is the tile of a cluster
// whose launch the hardware cancels on request (cluster launch control), so
// tiles go to whichever pairs are free first instead of a fixed share per
// pair.  The even CTA's producer makes one request per tile, into a ring of
// kSched response slots that both CTAs receive.  Every role of both CTAs reads
// each response after its CTA's sched_full barrier completes, then hands the
// slot back on the even CTA's sched_empty barrier, which needs kSchedReaders
// arrivals before the slot is reused.
constexpr int kSched = 4;
// even CTA: producer, MMA issuer, epilogue warps; odd CTA: producer, epilogue warps
constexpr int kSchedReaders = 2 + 2 * kEpiWarps + 1;

// Tile of iteration `it` under the dynamic order: 1 with *tile set, 0 when the
// pair has no tile left, -1 on a timeout.  For it > 0, *slot is the response
// slot read, which the caller hands back.
__device__ __forceinline__ int dyn_tile(int it, uint32_t resp0, uint32_t sched_full0, const WaitCtl& wc, int* tile,
                                        int* slot)
{
    if (it == 0) {
        *tile = static_cast<int>(blockIdx.x >> 1);
        return 1;
    }
    const int u = it - 1;
    const int s = u % kSched;
    *slot = s;
    if (!mbar_wait(sched_full0 + 8 * s, static_cast<uint32_t>(u / kSched) & 1u, wc, kSiteSchedFull)) return -1;
    int first_x = 0;
    if (!clc_query(resp0 + 16 * s, &first_x)) return 0;
    *tile = first_x >> 1;
    return 1;
}

// One rounding of the FP32 accumulator to a 16-bit output type.
template <int OUT>
__device__ __forceinline__ uint16_t round_out(uint32_t acc_bits)
{
    const float v = __uint_as_float(acc_bits);
    if constexpr (OUT == kOutBF16) {
        return __bfloat16_as_ushort(__float2bfloat16_rn(v));
    } else {
        return __half_as_ushort(__float2half_rn(v));
    }
}

// Masked column-major stores of one lane's row m, columns n0..n0+31 (rows at
// or past m_end -- the end of C or of the tile -- store nothing).  The lanes of
// a warp hold consecutive rows, so each store instruction writes 32 adjacent
// elements of one column.  The column address advances by a running pointer
// and the column bound is tested once per 32 columns: the epilogue warps share
// their schedulers with the producer and the MMA issuer, and per-element
// 64-bit index arithmetic (about 15 instructions per element) slowed the
// tensor pipe's feed (measured on 4096^3: 99 us against 88 us with TMA stores;
// the tensor pipe busy 74% instead of 85% of active cycles).
template <int OUT>
__device__ __forceinline__ void store_row(const uint32_t (&r)[32], const Params& p, int m, int n0, int m_end)
{
    if (m >= m_end) return;
    const int ncols = p.N - n0;
    using E = typename std::conditional<OUT == kOutF32, uint32_t, uint16_t>::type;
    E* q = reinterpret_cast<E*>(p.C) + (static_cast<long long>(m) + static_cast<long long>(n0) * p.ldc);
    const long long step = p.ldc;
    auto value = [&](int j) -> E {
        if constexpr (OUT == kOutF32) {
            return r[j];
        } else {
            return round_out<OUT>(r[j]);
        }
    };
    if (ncols >= 32) {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            *q = value(j);
            q += step;
        }
    } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            if (j < ncols) *q = value(j);
            q += step;
        }
    }
}

// Epilogue arithmetic on one lane's 32 accumulators before the rounding: the
// FP8 scale, or the bias of the 16-bit GEMM.
template <int IN, int OUT>
__device__ __forceinline__ void finish_acc(uint32_t (&r)[32], const Params& p, int m, int n0);

template <int OUT>
__device__ __forceinline__ float bias_value(const uint16_t* bias, int i)
{
    const uint16_t b = bias[i];
    if constexpr (OUT == kOutBF16) {
        return __uint_as_float(static_cast<uint32_t>(b) << 16);
    } else {
        return __half2float(__ushort_as_half(b));
    }
}

// Adds the bias to the FP32 accumulators of row m, columns n0..n0+31, before the
// one rounding to the output type.
template <int OUT>
__device__ __forceinline__ void add_bias(uint32_t (&r)[32], const Params& p, int m, int n0)
{
    if (p.bias_mode == 1) {
        if (m < p.M) {
            const float b = bias_value<OUT>(p.bias, m);
#pragma unroll
            for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) + b);
        }
    } else if (p.bias_mode == 2) {
#pragma unroll
        for (int j = 0; j < 32; ++j)
            if (n0 + j < p.N) r[j] = __float_as_uint(__uint_as_float(r[j]) + bias_value<OUT>(p.bias, n0 + j));
    }
}

template <int IN, int OUT>
__device__ __forceinline__ void finish_acc(uint32_t (&r)[32], const Params& p, int m, int n0)
{
    if constexpr (Types<IN, OUT>::kFp8) {
        if (p.alpha != 1.0f) {
#pragma unroll
            for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) * p.alpha);
        }
    } else {
        if (p.bias_mode != 0) add_bias<OUT>(r, p, m, n0);
    }
}

template <bool FP8>
__device__ __forceinline__ void mma_issue(uint32_t d_tmem, uint64_t ad, uint64_t bd, uint32_t idesc, uint32_t acc)
{
    if constexpr (FP8) {
        mma_f8f6f4(d_tmem, ad, bd, idesc, acc);
    } else {
        mma_f16(d_tmem, ad, bd, idesc, acc);
    }
}

template <bool FP8>
__device__ __forceinline__ void mma_issue_pair(uint32_t d_tmem, uint64_t ad, uint64_t bd, uint32_t idesc,
                                               uint32_t acc)
{
    if constexpr (FP8) {
        mma_f8f6f4_pair(d_tmem, ad, bd, idesc, acc);
    } else {
        mma_f16_pair(d_tmem, ad, bd, idesc, acc);
    }
}

template <int BN, bool A_MN, bool B_MN, int IN, int OUT>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tcgen05_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmC, const Params p)
{
    using Cf = Cfg<BN>;
    constexpr int S = Cf::kStages;
    using Ty = Types<IN, OUT>;
    constexpr uint32_t kIdesc = Ty::idesc(A_MN, B_MN, kBM, BN);
    static_assert(!B_MN || BN % 64 == 0, "an MN-major B needs whole 64-column swizzle atoms");
    static_assert(!Ty::kFp8 || (!A_MN && !B_MN), "FP8 operands are K-major");

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    uint8_t* sA = smem;
    uint8_t* sB = sA + S * Cf::kABytes;
    uint8_t* sEpi = sB + S * Cf::kBBytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sEpi + Cf::kEpiBytes);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + Cf::kNumBars);
    volatile uint32_t* abort_flag = tmem_slot + 1;

    const uint32_t full0 = smem_u32(bars);            // S barriers: stage loaded
    const uint32_t empty0 = full0 + 8 * S;            // S barriers: stage consumed
    const uint32_t tfull0 = empty0 + 8 * S;           // 2 barriers: accumulator ready
    const uint32_t tempty0 = tfull0 + 16;             // 2 barriers: accumulator drained
    const uint32_t drain_bar = tempty0 + 16;          // abort path: MMAs finished

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull0 + 8 * a, 1);
            mbar_init(tempty0 + 8 * a, kEpiWarps);
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0u;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
        if (p.tma_store) prefetch_tmap(&tmC);
        if (p.sk == 0 && p.skc <= 1 && static_cast<int>(blockIdx.x) < p.num_tiles) {
            // The first tile's first two stages into L2 while the kernel before
            // this one may still be running (a prefetch is coherent: nothing
            // reaches shared memory before griddep_wait below).  Two, not the
            // whole ring: the TMA unit works through the prefetches before the
            // real loads, and a launch with nothing to overlap waits for them.
            // Measured on the 34816 x 5120 decode shape (n = 4 and 8), first data
            // after the prologue 4.5-5.6 us with the whole ring prefetched, 1.9-2.4
            // us with two stages, kernel span 61-62 -> 59-60 us.
            int pm, pn;
            tile_coord(static_cast<int>(blockIdx.x), p.num_m, p.num_n, p.group_m, &pm, &pn);
            constexpr int kPrefetchStages = S < 2 ? S : 2;
            const int kbs = p.num_kb < kPrefetchStages ? p.num_kb : kPrefetchStages;
            for (int kb = 0; kb < kbs; ++kb) {
                const int k0 = kb * Ty::kBK;
                if constexpr (A_MN) {
                    tma_prefetch_l2_2d(&tmA, pm * kBM, k0);
                    tma_prefetch_l2_2d(&tmA, pm * kBM + 64, k0);
                } else {
                    tma_prefetch_l2_2d(&tmA, k0, pm * p.bm);
                }
                if constexpr (B_MN) {
#pragma unroll
                    for (int j = 0; j < BN / 64; ++j) tma_prefetch_l2_2d(&tmB, pn * BN + 64 * j, k0);
                } else {
                    tma_prefetch_l2_2d(&tmB, k0, pn * BN);
                }
            }
        }
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), Cf::kTmemCols);
        tmem_relinquish_alloc_permit();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    if constexpr (!A_MN) {
        // K-major A (the skinny decode weight): the epilogue warps, idle until the
        // first accumulator, prefetch the next pf_kb k-blocks of their first
        // tile's rows into L2 -- one 128-byte line per row and k-block, by the
        // load units, so the TMA unit's queue stays free for the real loads.
        // Like the producer's prefetch above this reads nothing into the SM.
        if (warp >= 2 && p.pf_kb > 0 && p.sk == 0 && p.skc <= 1 && static_cast<int>(blockIdx.x) < p.num_tiles) {
            int pm, pn;
            tile_coord(static_cast<int>(blockIdx.x), p.num_m, p.num_n, p.group_m, &pm, &pn);
            const int row = pm * p.bm + (static_cast<int>(threadIdx.x) - 64);
            constexpr int kFirst = S < 2 ? S : 2;
            const int kb_end = p.num_kb < kFirst + p.pf_kb ? p.num_kb : kFirst + p.pf_kb;
            if (row < p.M && row < (pm + 1) * p.bm) {
                const uint8_t* r = p.a_rows + static_cast<long long>(row) * p.a_ld_bytes;
                for (int kb = kFirst; kb < kb_end; ++kb) prefetch_l2(r + static_cast<long long>(kb) * kRowBytes);
            }
        }
    }
    // The prologue touched only shared memory, TMEM and the parameters; global
    // memory is read and written only once the kernel before this one in the
    // stream has completed (a no-op unless launched as its dependent).
    griddep_wait();
    griddep_launch_dependents();
    const WaitCtl wc{abort_flag, p.status, p.wait_limit_ns};
    // Waits on the abort path ignore the abort flag but keep the time limit.
    uint32_t never = 0u;
    const WaitCtl wc_drain{&never, p.status, p.wait_limit_ns};
    // bytes a stage's loads deliver: a K-major A box is p.bm rows of 128 bytes
    const uint32_t stage_tx = (A_MN ? Cf::kABytes : p.bm * kRowBytes) + Cf::kBBytes;

    if (warp == 0) {
        // ------------------------------------------------------------------
        // TMA producer
        // ------------------------------------------------------------------
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            long long issued = 0;
            bool ok = true;
            SegCursor cur = seg_first(p, blockIdx.x, gridDim.x);
            int tile, kb0, kb1;
            while (ok && seg_next(p, cur, tile, kb0, kb1)) {
                int pm, pn;
                tile_coord(tile, p.num_m, p.num_n, p.group_m, &pm, &pn);
                const int m0 = pm * p.bm;
                const int n0 = pn * BN;
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!mbar_wait(empty0 + 8 * stage, phase ^ 1u, wc, kSiteProducerEmpty)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = full0 + 8 * stage;
                    mbar_arrive_expect_tx(fb, stage_tx);
                    const uint32_t a_dst = smem_u32(sA + stage * Cf::kABytes);
                    const uint32_t b_dst = smem_u32(sB + stage * Cf::kBBytes);
                    const int k0 = kb * Ty::kBK;
                    if constexpr (A_MN) {
                        // two 64(m) x 64(k) boxes: m is the 128-byte swizzle row
                        tma_load_2d(a_dst, &tmA, fb, m0, k0);
                        tma_load_2d(a_dst + Cf::kABytes / 2, &tmA, fb, m0 + 64, k0);
                    } else {
                        tma_load_2d(a_dst, &tmA, fb, k0, m0);   // 128-byte k row x 128(m) box
                    }
                    if constexpr (B_MN) {
#pragma unroll
                        for (int i = 0; i < BN / 64; ++i)   // 64(n) x 64(k) boxes, 8 KB apart
                            tma_load_2d(b_dst + i * 8192, &tmB, fb, n0 + 64 * i, k0);
                    } else {
                        tma_load_2d(b_dst, &tmB, fb, k0, n0);    // 128-byte k row x BN(n) box
                    }
                    ++issued;
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) {
                // Abort: let the loads already issued land before the CTA can exit.
                const long long pending = issued < S ? issued : S;
                for (long long j = 1; j <= pending; ++j) {
                    const int s = (stage - static_cast<int>(j) + S) % S;
                    const uint32_t ph = (stage - static_cast<int>(j) < 0) ? (phase ^ 1u) : phase;
                    mbar_wait(full0 + 8 * s, ph, wc_drain, kSiteProducerDrain);
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------------
        // MMA issuer (one thread)
        // ------------------------------------------------------------------
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            bool issued_any = false;
            SegCursor cur = seg_first(p, blockIdx.x, gridDim.x);
            int tile, kb0, kb1;
            for (int it = 0; seg_next(p, cur, tile, kb0, kb1); ++it) {
                const int acc = it & 1;
                const uint32_t aph = static_cast<uint32_t>(it >> 1) & 1u;
                if (!mbar_wait(tempty0 + 8 * acc, aph ^ 1u, wc, kSiteMmaTmemEmpty)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!mbar_wait(full0 + 8 * stage, phase, wc, kSiteMmaFull)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint32_t a_base = smem_u32(sA + stage * Cf::kABytes);
                    const uint32_t b_base = smem_u32(sB + stage * Cf::kBBytes);
#pragma unroll
                    for (int kk = 0; kk < kRowBytes / kMmaBytes; ++kk) {
                        // MN-major A: 16 k-rows of 128 bytes per MMA, the two 64-element
                        // m blocks 8 KB apart; K-major operands: 32 bytes along the row.
                        const uint64_t ad = A_MN ? smem_desc_sw128(a_base + kk * 2048, Cf::kABytes / 2, 1024)
                                                 : smem_desc_sw128(a_base + kk * 32, 16, 1024);
                        const uint64_t bd = B_MN ? smem_desc_sw128(b_base + kk * 2048, 8192, 1024)
                                                 : smem_desc_sw128(b_base + kk * 32, 16, 1024);
                        mma_issue<Ty::kFp8>(d_tmem, ad, bd, kIdesc, (kb != kb0 || kk != 0) ? 1u : 0u);
                    }
                    mma_commit(empty0 + 8 * stage);
                    issued_any = true;
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                mma_commit(tfull0 + 8 * acc);
            }
            if (!ok && issued_any) {
                // Abort: every MMA issued so far must finish before TMEM is freed.
                mma_commit(drain_bar);
                mbar_wait(drain_bar, 0u, wc_drain, kSiteMmaDrain);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------------
        // Epilogue: TMEM -> registers -> 16-bit -> C
        // ------------------------------------------------------------------
        const int quarter = warp & 3;             // TMEM lanes this warp may read
        const int ew = warp - 2;                  // owner of kEpiBufs staging buffers
        uint8_t* ebuf = sEpi + ew * Cf::kEpiBufs * Cf::kEpiBufBytes;
        // Staging buffers are taken in turn over all of this warp's TMA stores,
        // tiles included (a 32-wide tile has one store per tile): the buffer of
        // the store kEpiBufs before is free once at most kEpiBufs - 1 stores are
        // still reading.
        int staged = 0;
        SegCursor cur = seg_first(p, blockIdx.x, gridDim.x);
        int tile, kb0, kb1;
        for (int it = 0; seg_next(p, cur, tile, kb0, kb1); ++it) {
            const int acc = it & 1;
            const uint32_t aph = static_cast<uint32_t>(it >> 1) & 1u;
            bool ok = mbar_wait(tfull0 + 8 * acc, aph, wc, kSiteEpilogueTmemFull);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after_sync();
            int pm, pn;
            tile_coord(tile, p.num_m, p.num_n, p.group_m, &pm, &pn);
            const int m0 = pm * p.bm + quarter * 32;
            const int n0 = pn * BN;
            // rows of C this warp stores: its 32 TMEM lanes, clipped to the tile and to C
            const int tile_end = pm * p.bm + p.bm;
            const int m_end = tile_end < p.M ? tile_end : p.M;
            // the TMA store writes all 32 rows of a box (clipped at M only)
            const bool whole_quarter = m0 + 32 <= tile_end;
            const uint32_t t_row = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                                   static_cast<uint32_t>(acc * BN);
            // Stream-K roles: a segment that does not start the tile leaves its
            // partial in this CTA's slot; one that starts it but does not end it
            // adds the slots of the CTAs holding the rest of the tile.
            const bool to_slot = p.sk && kb0 != 0;
            int q_last = static_cast<int>(blockIdx.x);
            if (p.sk && kb0 == 0 && kb1 != p.num_kb) {
                q_last = sk_unit_of(p, static_cast<long long>(tile - p.sk_dp_tiles + 1) * p.num_kb - 1, gridDim.x);
                bool fok = true;
                for (int q = static_cast<int>(blockIdx.x) + 1; fok && q <= q_last; ++q)
                    fok = flag_wait_acquire(p.sk_flag + q, wc, kSiteStreamKPartial);
                (void)__all_sync(0xffffffffu, fok);   // on a timeout the status word is set; the output is undefined
            }
#pragma unroll 1
            for (int c = 0; c < BN / 32; ++c) {
                uint32_t r[32];
                tmem_ld_32x32b_x32(t_row + c * 32, r);
                tmem_ld_wait();
                if (c == BN / 32 - 1) {
                    // all of this accumulator is in registers: hand TMEM back to the MMA warp
                    tc_fence_before_sync();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(tempty0 + 8 * acc);
                }
                const long long slot_col = static_cast<long long>(c * 32) * kBM + quarter * 32 + lane;
                if (p.skc > 1) {
                    // split-K over the cluster: the partial stays in this CTA's shared
                    // memory ([column][128 rows] FP32 over the ring, whose stages the
                    // MMAs have finished reading)
                    if (c == 0) fence_proxy_async_smem();
                    float* part = reinterpret_cast<float*>(smem) + slot_col;
#pragma unroll
                    for (int j = 0; j < 32; ++j) part[j * kBM] = __uint_as_float(r[j]);
                    continue;
                }
                if (to_slot) {
                    float* ps = p.sk_part + static_cast<long long>(blockIdx.x) * BN * kBM + slot_col;
#pragma unroll
                    for (int j = 0; j < 32; ++j) ps[j * kBM] = __uint_as_float(r[j]);
                    continue;
                }
                add_partials(r, p.sk_part + slot_col, static_cast<long long>(BN) * kBM, static_cast<int>(blockIdx.x) + 1,
                             q_last);
                finish_acc<IN, OUT>(r, p, m0 + lane, n0 + c * 32);
                if (Ty::kOutBytes == 2 && p.tma_store && whole_quarter) {
                    uint8_t* buf = ebuf + (staged++ % Cf::kEpiBufs) * Cf::kEpiBufBytes;
                    if (lane == 0) bulk_wait_group_read<Cf::kEpiBufs - 1>();   // the store that used `buf` has read it
                    __syncwarp();
                    uint16_t* b16 = reinterpret_cast<uint16_t*>(buf);
#pragma unroll
                    for (int j = 0; j < 32; ++j) b16[j * 32 + lane] = round_out<OUT>(r[j]);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&tmC, smem_u32(buf), m0, n0 + c * 32);
                        bulk_commit_group();
                    }
                } else {
                    store_row<OUT>(r, p, m0 + lane, n0 + c * 32, m_end);
                }
            }
            if (to_slot) {
                // every epilogue warp's part of the slot is written before the flag is released
                __threadfence();
                asm volatile("bar.sync 1, %0;" ::"n"(kEpiWarps * 32) : "memory");
                if (warp == 2 && lane == 0) flag_set_release(p.sk_flag + blockIdx.x);
            }
        }
        if (lane == 0) bulk_wait_group<0>();
        __syncwarp();
    }

    if (p.skc > 1) {
        // Split-K over the cluster.  A CTA whose share of k-blocks is empty holds
        // a zero partial.  Barrier 1: every CTA's partial is in its shared memory.
        SegCursor cur = seg_first(p, blockIdx.x, gridDim.x);
        if (cur.pos >= cur.end && warp >= 2) {
            float* part = reinterpret_cast<float*>(smem);
            for (int i = threadIdx.x - 64; i < BN * kBM; i += kEpiWarps * 32) part[i] = 0.f;
        }
        cluster_sync();
        if (warp >= 2) {
            // Columns [rank * BN/skc, (rank+1) * BN/skc) of the tile, summed over the
            // cluster's partials in rank order.  Work items are 4 rows of one column
            // (16 bytes of each partial); a thread takes every 128th item and keeps 16
            // loads in flight: 4 items x 4 partials at a time in clusters of 2 or 4,
            // one item x all partials in clusters of 8 or 16 (fewer items, more
            // partials each).
            const int rank = static_cast<int>(cluster_ctarank());
            const int cols = BN / p.skc;
            const int items = cols * (kBM / 4);
            const int t = threadIdx.x - 64;
            int pm, pn;
            tile_coord(static_cast<int>(blockIdx.x) / p.skc, p.num_m, p.num_n, p.group_m, &pm, &pn);
            const uint32_t part0 = smem_u32(smem);
            using E = typename std::conditional<OUT == kOutF32, uint32_t, uint16_t>::type;
            auto offset = [&](int i) {
                return static_cast<uint32_t>(((rank * cols + i / (kBM / 4)) * kBM + (i % (kBM / 4)) * 4) * 4);
            };
            auto add4 = [](float4& a, const float4& x) {
                a.x += x.x;
                a.y += x.y;
                a.z += x.z;
                a.w += x.w;
            };
            // bias or FP8 scale, one rounding, and the four rows' stores of item i
            auto emit = [&](int i, const float4& acc) {
                const int n = pn * BN + rank * cols + i / (kBM / 4);
                const int m_first = pm * kBM + (i % (kBM / 4)) * 4;
                const float v4[4] = {acc.x, acc.y, acc.z, acc.w};
                if (n >= p.N) return;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int m = m_first + e;
                    if (m >= p.M) break;
                    float v = v4[e];
                    if constexpr (Ty::kFp8) {
                        if (p.alpha != 1.0f) v *= p.alpha;
                    } else {
                        if (p.bias_mode == 1) v += bias_value<OUT>(p.bias, m);
                        else if (p.bias_mode == 2) v += bias_value<OUT>(p.bias, n);
                    }
                    E* dst = reinterpret_cast<E*>(p.C) + (static_cast<long long>(m) + static_cast<long long>(n) * p.ldc);
                    if constexpr (OUT == kOutF32) {
                        *dst = __float_as_uint(v);
                    } else {
                        *dst = round_out<OUT>(__float_as_uint(v));
                    }
                }
            };
            if (p.skc >= 8) {
                for (int i = t; i < items; i += kEpiWarps * 32) {
                    const uint32_t off = offset(i);
                    float4 x[16];
#pragma unroll
                    for (int q = 0; q < 16; ++q)
                        if (q < p.skc) x[q] = ld_shared_cluster_v4(mapa_shared(part0 + off, q));
                    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                    for (int q = 0; q < 16; ++q)
                        if (q < p.skc) add4(acc, x[q]);
                    emit(i, acc);
                }
            } else {
                for (int i0 = t; i0 < items; i0 += 4 * kEpiWarps * 32) {
                    float4 acc[4];
                    uint32_t off[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
                        off[u] = offset(i0 + u * kEpiWarps * 32);
                    }
                    float4 x[4][4];
#pragma unroll
                    for (int u = 0; u < 4; ++u)
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            if (i0 + u * kEpiWarps * 32 < items && q < p.skc)
                                x[u][q] = ld_shared_cluster_v4(mapa_shared(part0 + off[u], q));
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        if (i0 + u * kEpiWarps * 32 >= items) continue;
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            if (q < p.skc) add4(acc[u], x[u][q]);
                        emit(i0 + u * kEpiWarps * 32, acc[u]);
                    }
                }
            }
        }
        // Barrier 2: no CTA leaves while a peer may still read its shared memory.
        cluster_sync();
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, Cf::kTmemCols);
    }
}

// ---------------------------------------------------------------------------
// CTA-pair variant (tcgen05 .cta_group::2).  A cluster of two CTAs on two SMs
// computes a 256 x 256 tile: CTA r of the pair stages rows [128r, 128r+128) of
// the tile's A slice and rows [128r, 128r+128) of its B slice (the n range), so
// each SM loads and stores 32 KB per 64-deep k step instead of 48 KB, and the
// ring holds 6 stages instead of 4.  One thread of the even CTA issues the
// 256 x 256 x 16 MMAs, which read both CTAs' halves and leave each CTA's 128
// accumulator rows in its own TMEM.
//   * both CTAs' TMA loads signal the even CTA's "full" barrier, which the even
//     CTA's producer arms with the bytes of both halves;
//   * the MMA's commits arrive on the "empty" and "accumulator full" barriers of
//     both CTAs (multicast);
//   * each CTA's epilogue warps hand the accumulator back by arriving on the even
//     CTA's "accumulator empty" barrier (8 arrivals).
// ---------------------------------------------------------------------------
template <int MB>
struct PairCfg {
    static_assert(MB == 1 || MB == 2, "one or two 256-row blocks per pair tile");
    static constexpr int kStages = MB == 1 ? 6 : 4;
    static constexpr int kBlockABytes = kBM * kRowBytes;   // this CTA's 128 rows of one A block
    static constexpr int kABytes = MB * kBlockABytes;
    static constexpr int kBBytes = kBM * kRowBytes;        // this CTA's 128 rows of B
    static constexpr int kStageBytes = kABytes + kBBytes;  // 32 / 48 KB; the pair moves twice that per stage
    static constexpr int kEpiBufBytes = kEpiBox * kEpiBox * 2;
    static constexpr int kEpiBytes = kEpiWarps * 2 * kEpiBufBytes;
    static constexpr int kTile = 256;                      // pair tile is 256 * MB rows x 256 columns
    // MB = 1: two 256-column accumulators (the epilogue of one tile overlaps the
    // next tile's MMAs); MB = 2: one accumulator of two 256-column blocks
    static constexpr int kAccBufs = MB == 1 ? 2 : 1;
    static constexpr int kTmemCols = 2 * kTile;
    static constexpr int kNumBars = 2 * kStages + 5;
    // barriers, TMEM slot + abort flag, then the dynamic order's 2 x kSched
    // barriers and kSched 16-byte response slots
    static constexpr int kSchedBarOffset = kNumBars * 8 + 8;
    static constexpr int kSchedRespOffset = (kSchedBarOffset + 2 * kSched * 8 + 15) / 16 * 16;
    static constexpr int kBarBytes = 512;
    static constexpr int kSmemBytes = 1024 + kStages * kStageBytes + kEpiBytes + kBarBytes;
    static_assert(kSchedRespOffset + kSched * 16 <= kBarBytes, "barrier area too small");
    static_assert(kSmemBytes <= 232448, "shared memory budget exceeded");
};

template <bool A_MN, bool B_MN, int IN, int OUT, int MB>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tcgen05_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                             const __grid_constant__ CUtensorMap tmC, const Params p)
{
    using Cf = PairCfg<MB>;
    constexpr int S = Cf::kStages;
    constexpr int T = Cf::kTile;
    constexpr int TM = T * MB;   // rows of C per pair tile
    using Ty = Types<IN, OUT>;
    constexpr uint32_t kIdesc = Ty::idesc(A_MN, B_MN, 2 * kBM, T);
    static_assert(!Ty::kFp8 || (!A_MN && !B_MN), "FP8 operands are K-major");

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    uint8_t* sA = smem;
    uint8_t* sB = sA + S * Cf::kABytes;
    uint8_t* sEpi = sB + S * Cf::kBBytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sEpi + Cf::kEpiBytes);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + Cf::kNumBars);
    volatile uint32_t* abort_flag = tmem_slot + 1;

    const uint32_t full0 = smem_u32(bars);
    const uint32_t empty0 = full0 + 8 * S;
    const uint32_t tfull0 = empty0 + 8 * S;
    const uint32_t tempty0 = tfull0 + 16;
    const uint32_t drain_bar = tempty0 + 16;
    const uint32_t sched_full0 = full0 + Cf::kSchedBarOffset;    // kSched barriers: response landed
    const uint32_t sched_empty0 = sched_full0 + 8 * kSched;     // kSched barriers: response read by all
    const uint32_t resp0 = full0 + Cf::kSchedRespOffset;         // kSched 16-byte responses

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const int pair = blockIdx.x >> 1;
    const int num_pairs = gridDim.x >> 1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull0 + 8 * a, 1);
            mbar_init(tempty0 + 8 * a, 2 * kEpiWarps);
        }
        mbar_init(drain_bar, 1);
        for (int q = 0; q < kSched; ++q) {
            mbar_init(sched_full0 + 8 * q, 1);
            mbar_init(sched_empty0 + 8 * q, kSchedReaders);
        }
        *abort_flag = 0u;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
        if (p.tma_store) prefetch_tmap(&tmC);
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_u32(tmem_slot), Cf::kTmemCols);
        tmem_relinquish_alloc_permit_pair();
    }
    // Both CTAs' barriers are initialised and the TMEM columns allocated before
    // any CTA signals its peer.
    tc_fence_before_sync();
    cluster_sync();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    // The prologue touched only shared memory, TMEM and the parameters; global
    // memory is read and written only once the kernel before this one in the
    // stream has completed (a no-op unless launched as its dependent).
    griddep_wait();
    griddep_launch_dependents();
    const uint32_t leader_full0 = mapa_shared(full0, 0);
    const uint32_t leader_tempty0 = mapa_shared(tempty0, 0);
    const uint32_t leader_sched_empty0 = mapa_shared(sched_empty0, 0);
    const WaitCtl wc{abort_flag, p.status, p.wait_limit_ns};
    uint32_t never = 0u;
    const WaitCtl wc_drain{&never, p.status, p.wait_limit_ns};

    if (warp == 0) {
        // ------------------------------------------------------------------
        // TMA producer (both CTAs): this CTA's halves of A and B
        // ------------------------------------------------------------------
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            long long issued = 0;
            bool ok = true;
            int armed = 0, read = 0;   // dynamic order: responses this CTA expects / has read
            SegCursor cur = seg_first(p, pair, num_pairs);
            int tile = 0, kb0 = 0, kb1 = 0;
            for (int it = 0; ok; ++it) {
                if (p.dyn) {
                    int slot = 0;
                    const int r = dyn_tile(it, resp0, sched_full0, wc, &tile, &slot);
                    if (r < 0) {
                        ok = false;
                        break;
                    }
                    if (it > 0) {
                        ++read;
                        mbar_arrive_remote(leader_sched_empty0 + 8 * slot);
                    }
                    if (r == 0) break;
                    kb0 = 0;
                    kb1 = p.num_kb;
                    // ask for the pair's next tile now, so that the answer is in by the
                    // time this tile's k-blocks are issued
                    const int q = it % kSched;
                    if (leader && !mbar_wait_cluster(sched_empty0 + 8 * q, ((it / kSched) & 1) ^ 1u, wc,
                                                     kSiteSchedEmpty)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(sched_full0 + 8 * q, 16);
                    ++armed;
                    if (leader) clc_try_cancel_multicast(resp0 + 16 * q, sched_full0 + 8 * q);
                } else if (!seg_next(p, cur, tile, kb0, kb1)) {
                    break;
                }
                int pm, pn;
                tile_coord(tile, p.num_m, p.num_n, p.group_m, &pm, &pn);
                const int m0 = pm * TM + static_cast<int>(rank) * kBM;   // this CTA's rows of A block 0
                const int n0 = pn * T + static_cast<int>(rank) * kBM;
                const bool rev = p.rev_round > 0 && kb0 == 0 && kb1 == p.num_kb && ((tile / p.rev_round) & 1);
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!mbar_wait(empty0 + 8 * stage, phase ^ 1u, wc, kSiteProducerEmpty)) {
                        ok = false;
                        break;
                    }
                    if (leader) mbar_arrive_expect_tx(full0 + 8 * stage, 2 * Cf::kStageBytes);
                    const uint32_t fb = leader_full0 + 8 * stage;
                    const uint32_t a_dst = smem_u32(sA + stage * Cf::kABytes);
                    const uint32_t b_dst = smem_u32(sB + stage * Cf::kBBytes);
                    const int k0 = (rev ? kb0 + kb1 - 1 - kb : kb) * Ty::kBK;
#pragma unroll
                    for (int b = 0; b < MB; ++b) {   // A block b: rows m0 + b * 256 of this CTA's half
                        const uint32_t ab = a_dst + b * Cf::kBlockABytes;
                        if constexpr (A_MN) {
                            tma_load_2d_pair(ab, &tmA, fb, m0 + b * T, k0);
                            tma_load_2d_pair(ab + Cf::kBlockABytes / 2, &tmA, fb, m0 + b * T + 64, k0);
                        } else {
                            tma_load_2d_pair(ab, &tmA, fb, k0, m0 + b * T);
                        }
                    }
                    if constexpr (B_MN) {
                        tma_load_2d_pair(b_dst, &tmB, fb, n0, k0);            // 64(n) x 64(k)
                        tma_load_2d_pair(b_dst + 8192, &tmB, fb, n0 + 64, k0);
                    } else {
                        tma_load_2d_pair(b_dst, &tmB, fb, k0, n0);
                    }
                    ++issued;
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (armed > read) {
                // A response is still on its way into this CTA's shared memory
                // (abort path): wait (bounded) until it has landed.
                const int u = armed - 1;
                mbar_wait(sched_full0 + 8 * (u % kSched), static_cast<uint32_t>(u / kSched) & 1u, wc_drain,
                          kSiteSchedFull);
            }
            if (!ok && leader) {
                // Abort: the even CTA's full barriers count both CTAs' bytes; wait
                // (bounded) until the loads already armed have landed.
                const long long pending = issued < S ? issued : S;
                for (long long j = 1; j <= pending; ++j) {
                    const int s = (stage - static_cast<int>(j) + S) % S;
                    const uint32_t ph = (stage - static_cast<int>(j) < 0) ? (phase ^ 1u) : phase;
                    mbar_wait(full0 + 8 * s, ph, wc_drain, kSiteProducerDrain);
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------------
        // MMA issuer: one thread of the even CTA
        // ------------------------------------------------------------------
        if (lane == 0 && leader) {
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            bool issued_any = false;
            SegCursor cur = seg_first(p, pair, num_pairs);
            int tile = 0, kb0 = 0, kb1 = 0;
            for (int it = 0;; ++it) {
                if (p.dyn) {
                    int slot = 0;
                    const int r = dyn_tile(it, resp0, sched_full0, wc, &tile, &slot);
                    if (r < 0) {
                        ok = false;
                        break;
                    }
                    if (it > 0) mbar_arrive_remote(leader_sched_empty0 + 8 * slot);
                    if (r == 0) break;
                    kb0 = 0;
                    kb1 = p.num_kb;
                } else if (!seg_next(p, cur, tile, kb0, kb1)) {
                    break;
                }
                const int acc = it % Cf::kAccBufs;
                const uint32_t aph = static_cast<uint32_t>(it / Cf::kAccBufs) & 1u;
                if (!mbar_wait_cluster(tempty0 + 8 * acc, aph ^ 1u, wc, kSiteMmaTmemEmpty)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                // accumulator of A block b: TMEM columns (acc + b) * 256 (one of acc, b is 0)
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * T);
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!mbar_wait(full0 + 8 * stage, phase, wc, kSiteMmaFull)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint32_t a_base = smem_u32(sA + stage * Cf::kABytes);
                    const uint32_t b_base = smem_u32(sB + stage * Cf::kBBytes);
#pragma unroll
                    for (int kk = 0; kk < kRowBytes / kMmaBytes; ++kk) {
                        const uint64_t bd = B_MN ? smem_desc_sw128(b_base + kk * 2048, 8192, 1024)
                                                 : smem_desc_sw128(b_base + kk * 32, 16, 1024);
#pragma unroll
                        for (int b = 0; b < MB; ++b) {   // the blocks share this k-step's B slice
                            const uint32_t ab = a_base + b * Cf::kBlockABytes;
                            const uint64_t ad = A_MN ? smem_desc_sw128(ab + kk * 2048, Cf::kBlockABytes / 2, 1024)
                                                     : smem_desc_sw128(ab + kk * 32, 16, 1024);
                            mma_issue_pair<Ty::kFp8>(d_tmem + static_cast<uint32_t>(b * T), ad, bd, kIdesc,
                                                     (kb != kb0 || kk != 0) ? 1u : 0u);
                        }
                    }
                    mma_commit_pair_multicast(empty0 + 8 * stage, 0x3);
                    issued_any = true;
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                mma_commit_pair_multicast(tfull0 + 8 * acc, 0x3);
            }
            if (!ok && issued_any) {
                mma_commit_pair_multicast(drain_bar, 0x1);
                mbar_wait(drain_bar, 0u, wc_drain, kSiteMmaDrain);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------------
        // Epilogue (both CTAs): this CTA's 128 rows of each 256-row block of the tile
        // ------------------------------------------------------------------
        const int quarter = warp & 3;
        const int ew = warp - 2;
        uint8_t* ebuf = sEpi + ew * 2 * Cf::kEpiBufBytes;
        int staged = 0;   // TMA stores of this warp so far: buffer staged % 2
        SegCursor cur = seg_first(p, pair, num_pairs);
        int tile = 0, kb0 = 0, kb1 = 0;
        for (int it = 0;; ++it) {
            if (p.dyn) {
                int slot = 0;
                int r = dyn_tile(it, resp0, sched_full0, wc, &tile, &slot);
                r = __reduce_min_sync(0xffffffffu, r);
                __syncwarp();   // every lane has read the response before it is handed back
                if (it > 0 && r >= 0 && lane == 0) mbar_arrive_remote(leader_sched_empty0 + 8 * slot);
                if (r <= 0) break;
                kb0 = 0;
                kb1 = p.num_kb;
            } else if (!seg_next(p, cur, tile, kb0, kb1)) {
                break;
            }
            const int acc = it % Cf::kAccBufs;
            const uint32_t aph = static_cast<uint32_t>(it / Cf::kAccBufs) & 1u;
            bool ok = mbar_wait(tfull0 + 8 * acc, aph, wc, kSiteEpilogueTmemFull);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after_sync();
            int pm, pn;
            tile_coord(tile, p.num_m, p.num_n, p.group_m, &pm, &pn);
            const int m0 = pm * TM + static_cast<int>(rank) * kBM + quarter * 32;   // in A block 0
            const int n0 = pn * T;
            const uint32_t t_row = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                                   static_cast<uint32_t>(acc * T);
            // Stream-K roles, as in the one-CTA kernel; slots and flags are per CTA
            // (pair * 2 + rank), each holding this CTA's 128 rows of the tile.
            const bool to_slot = p.sk && kb0 != 0;
            const int my_slot = pair * 2 + static_cast<int>(rank);
            int q_last = pair;
            if (p.sk && kb0 == 0 && kb1 != p.num_kb) {
                q_last = sk_unit_of(p, static_cast<long long>(tile - p.sk_dp_tiles + 1) * p.num_kb - 1, num_pairs);
                bool fok = true;
                for (int q = pair + 1; fok && q <= q_last; ++q)
                    fok = flag_wait_acquire(p.sk_flag + q * 2 + static_cast<int>(rank), wc, kSiteStreamKPartial);
                (void)__all_sync(0xffffffffu, fok);   // on a timeout the status word is set; the output is undefined
            }
#pragma unroll 1
            for (int cb = 0; cb < MB * (T / 32); ++cb) {
                const int b = cb / (T / 32);   // A block of the chunk (stream-K runs with MB = 1)
                const int c = cb % (T / 32);
                const int mb = m0 + b * T;
                uint32_t r[32];
                tmem_ld_32x32b_x32(t_row + b * T + c * 32, r);
                tmem_ld_wait();
                if (cb == MB * (T / 32) - 1) {
                    tc_fence_before_sync();
                    __syncwarp();
                    if (lane == 0) mbar_arrive_remote(leader_tempty0 + 8 * acc);
                }
                const long long slot_col = static_cast<long long>(c * 32) * kBM + quarter * 32 + lane;
                if (to_slot) {
                    float* ps = p.sk_part + static_cast<long long>(my_slot) * T * kBM + slot_col;
#pragma unroll
                    for (int j = 0; j < 32; ++j) ps[j * kBM] = __uint_as_float(r[j]);
                    continue;
                }
                if (mb >= p.M) continue;   // all 32 rows past the end of C: nothing to store
                // slot of CTA (pair q, rank): (q * 2 + rank) * T * kBM
                add_partials(r, p.sk_part + static_cast<long long>(rank) * T * kBM + slot_col, 2LL * T * kBM, pair + 1,
                             q_last);
                finish_acc<IN, OUT>(r, p, mb + lane, n0 + c * 32);
                if (Ty::kOutBytes == 2 && p.tma_store) {
                    uint8_t* buf = ebuf + (staged++ & 1) * Cf::kEpiBufBytes;
                    if (lane == 0) bulk_wait_group_read<1>();
                    __syncwarp();
                    uint16_t* b16 = reinterpret_cast<uint16_t*>(buf);
#pragma unroll
                    for (int j = 0; j < 32; ++j) b16[j * 32 + lane] = round_out<OUT>(r[j]);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&tmC, smem_u32(buf), mb, n0 + c * 32);
                        bulk_commit_group();
                    }
                } else {
                    store_row<OUT>(r, p, mb + lane, n0 + c * 32, p.M);
                }
            }
            if (to_slot) {
                __threadfence();
                asm volatile("bar.sync 1, %0;" ::"n"(kEpiWarps * 32) : "memory");
                if (warp == 2 && lane == 0) flag_set_release(p.sk_flag + my_slot);
            }
        }
        if (lane == 0) bulk_wait_group<0>();
        __syncwarp();
    }

    // Neither CTA may leave while its peer can still read its shared memory or
    // arrive on its barriers.
    tc_fence_before_sync();
    cluster_sync();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc_pair(tmem_base, Cf::kTmemCols);
    }
}

inline CUtensorMapDataType tmap_type(int type_code)
{
    return type_code == kInBF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
           : type_code == kInF16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
}

// 2-D tiled tensor map; `dtype` one of tmap_type()'s results.
inline bool encode_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, unsigned long long dim0,
                      unsigned long long dim1, unsigned long long stride1_bytes, unsigned box0, unsigned box1,
                      CUtensorMapSwizzle swz, char* msg, size_t msg_len)
{
    TmapEncodeFn enc = tmap_encoder();
    if (enc == nullptr) {
        snprintf(msg, msg_len, "cuTensorMapEncodeTiled is not available from the driver");
        return false;
    }
    const cuuint64_t dims[2] = {dim0, dim1};
    const cuuint64_t strides[1] = {stride1_bytes};
    const cuuint32_t box[2] = {box0, box1};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, dtype, 2,
                     const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        snprintf(msg, msg_len, "cuTensorMapEncodeTiled failed (%d) for dims %llu x %llu, stride %llu B, box %u x %u",
                 static_cast<int>(r), dim0, dim1, stride1_bytes, box0, box1);
        return false;
    }
    return true;
}

// Tensor maps of A, B (128-byte swizzled k rows or 64 x 64 MN-major boxes) and
// C (16-bit outputs stored by TMA only).  `rows_a` is the height of a K-major
// A box (the tile's rows), `rows_b` the B box height.
template <int IN, int OUT, bool A_MN, bool B_MN>
bool encode_operands(const GemmLaunch& g, int rows_a, int rows_b, CUtensorMap* tmA, CUtensorMap* tmB,
                     CUtensorMap* tmC, char* msg, size_t msg_len)
{
    using Ty = Types<IN, OUT>;
    const CUtensorMapDataType dt = tmap_type(IN);
    const unsigned long long eb = Ty::kElemBytes;
    const bool ok_a = A_MN ? encode_2d(tmA, dt, g.A, g.M, g.K, g.lda * eb, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B, msg,
                                       msg_len)
                           : encode_2d(tmA, dt, g.A, g.K, g.M, g.lda * eb, Ty::kBK, rows_a,
                                       CU_TENSOR_MAP_SWIZZLE_128B, msg, msg_len);
    if (!ok_a) return false;
    const bool ok_b = B_MN ? encode_2d(tmB, dt, g.B, g.N, g.K, g.ldb * eb, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B, msg,
                                       msg_len)
                           : encode_2d(tmB, dt, g.B, g.K, g.N, g.ldb * eb, Ty::kBK, rows_b,
                                       CU_TENSOR_MAP_SWIZZLE_128B, msg, msg_len);
    if (!ok_b) return false;
    if (Ty::kOutBytes == 2 && g.tma_store) {
        const CUtensorMapDataType dc = OUT == kOutBF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                       : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
        if (!encode_2d(tmC, dc, g.C, g.M, g.N, g.ldc * 2ull, kEpiBox, kEpiBox, CU_TENSOR_MAP_SWIZZLE_NONE, msg,
                       msg_len))
            return false;
    } else {
        *tmC = *tmA;   // unused by the kernel
    }
    return true;
}

template <int BN, bool A_MN, bool B_MN, int IN, int OUT>
int launch_instance(const GemmLaunch& g, cudaStream_t stream, char* msg, size_t msg_len)
{
    using Cf = Cfg<BN>;
    using Ty = Types<IN, OUT>;
    // Tile rows: 128, or the balanced height the planner chose (K-major A,
    // whole tiles only).
    const int bm = (!A_MN && !g.stream_k && g.skc <= 1 && g.block_m >= 8 && g.block_m <= kBM && g.block_m % 8 == 0)
                       ? g.block_m
                       : kBM;
    CUtensorMap tmA, tmB, tmC;
    if (!encode_operands<IN, OUT, A_MN, B_MN>(g, bm, BN, &tmA, &tmB, &tmC, msg, msg_len)) return 1;

    Params p;
    p.M = g.M;
    p.N = g.N;
    p.K = g.K;
    p.bm = bm;
    p.num_m = (g.M + bm - 1) / bm;
    p.num_n = (g.N + BN - 1) / BN;
    p.num_tiles = p.num_m * p.num_n;
    p.num_kb = (g.K + Ty::kBK - 1) / Ty::kBK;
    p.group_m = g.group_m < 1 ? 1 : g.group_m;
    p.C = g.C;
    p.ldc = g.ldc;
    p.tma_store = (Ty::kOutBytes == 2 && g.tma_store) ? 1 : 0;
    p.bias = g.bias;
    p.bias_mode = g.bias != nullptr ? g.bias_mode : 0;
    p.alpha = g.alpha;
    p.status = g.status;
    p.wait_limit_ns = g.wait_limit_ns;
    p.dyn = 0;
    p.skc = 0;
    p.rev_round = 0;
    p.a_rows = static_cast<const uint8_t*>(g.A);
    p.a_ld_bytes = g.lda * Ty::kElemBytes;
    p.pf_kb = A_MN ? 0 : g.prefetch_kb;

    auto kern = gemm_tcgen05_kernel<BN, A_MN, B_MN, IN, OUT>;
    static SmemOptIn smem_opt;
    cudaError_t e = smem_opt.ensure(reinterpret_cast<const void*>(kern), Cf::kSmemBytes);
    if (e != cudaSuccess) {
        snprintf(msg, msg_len, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
        return 1;
    }
    if (g.skc > 1) {
        // Split-K: one cluster of skc CTAs per tile (no workspace, no flags).
        int skc = g.skc;
        p.sk = 0;
        p.sk_dp_tiles = 0;
        p.sk_iters = 0;
        p.sk_part = nullptr;
        p.sk_flag = nullptr;
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        cudaLaunchConfig_t cfg = {};
        cfg.blockDim = dim3(kThreads, 1, 1);
        cfg.dynamicSmemBytes = Cf::kSmemBytes;
        cfg.stream = stream;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        // Clusters of this kernel that fit on the device at once, per cluster size
        // (queried once per device).  A size whose clusters would not all fit in
        // one wave is halved while that makes them fit: one wave of smaller
        // clusters finishes before two waves of larger ones (GB300, one CTA per
        // SM: 76 clusters of 2, 36 of 4, 15 of 8, 7 of 16).
        static std::atomic<int> fit_cache[SmemOptIn::kMaxDevices][5];
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= SmemOptIn::kMaxDevices) dev = -1;
        auto fits = [&](int size) {
            int lg = 0;
            while ((1 << lg) < size) ++lg;
            int n = dev >= 0 ? fit_cache[dev][lg].load(std::memory_order_acquire) : 0;
            if (n > 0) return n;
            if (size > 8 && cudaFuncSetAttribute(reinterpret_cast<const void*>(kern),
                                                 cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) {
                cudaGetLastError();
                return 0;
            }
            attr[0].val.clusterDim.x = static_cast<unsigned>(size);
            cfg.gridDim = dim3(static_cast<unsigned>(size), 1, 1);
            n = 0;
            if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
                cudaGetLastError();
                n = 0;
            }
            if (n > 0 && dev >= 0) fit_cache[dev][lg].store(n, std::memory_order_release);
            return n;
        };
        while (skc > 2 && fits(skc) < p.num_tiles) skc /= 2;
        p.skc = skc;
        attr[0].val.clusterDim.x = static_cast<unsigned>(skc);
        cfg.gridDim = dim3(static_cast<unsigned>(p.num_tiles) * static_cast<unsigned>(skc), 1, 1);
        cfg.numAttrs = g.pdl ? 2 : 1;
        e = cudaLaunchKernelEx(&cfg, kern, tmA, tmB, tmC, p);
        if (e == cudaSuccess) e = cudaGetLastError();
        if (e != cudaSuccess) {
            snprintf(msg, msg_len, "GEMM (split-K, clusters of %d) launch failed: %s", skc, cudaGetErrorString(e));
            return 1;
        }
        return 0;
    }
    int grid = 0;
    p.sk = 0;
    p.sk_dp_tiles = 0;
    p.sk_iters = 0;
    p.sk_part = nullptr;
    p.sk_flag = nullptr;
    if (g.stream_k && g.sk_part != nullptr && g.sk_flag != nullptr) {
        // Every SM takes an equal share of the (tile, k-block) iterations.  The CTAs
        // of a split tile wait on one another, so they must all be resident: the
        // launch is cooperative (it fails rather than run them in waves).
        p.sk = 1;
        grid = g.num_sms;
        p.sk_dp_tiles = (p.num_tiles / grid) * grid;
        if (p.sk_dp_tiles == p.num_tiles) p.sk_dp_tiles -= grid;   // keep one wave to share
        p.sk_iters = static_cast<long long>(p.num_tiles - p.sk_dp_tiles) * p.num_kb;
        if (grid > p.sk_iters) grid = static_cast<int>(p.sk_iters);
        if (p.sk_dp_tiles == 0) {
            // Few tiles: the CTA that finishes a split tile adds the others' FP32
            // partials one after another, so each tile is shared by at most four
            // CTAs, each with at least 8 k-blocks.  256 x 256 x 2048 (2 tiles of
            // 32 k-blocks): 64 CTAs of one k-block each took 114 us per call.
            const long long split = p.num_kb / 8 < 1 ? 1 : (p.num_kb / 8 > 4 ? 4 : p.num_kb / 8);
            const long long cap = static_cast<long long>(p.num_tiles) * split;
            if (grid > cap) grid = static_cast<int>(cap);
        }
        p.sk_part = g.sk_part;
        p.sk_flag = g.sk_flag;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeCooperative;
        attr[0].val.cooperative = 1;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(grid, 1, 1);
        cfg.blockDim = dim3(kThreads, 1, 1);
        cfg.dynamicSmemBytes = Cf::kSmemBytes;
        cfg.stream = stream;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, kern, tmA, tmB, tmC, p);
        if (e == cudaSuccess) e = cudaGetLastError();
        if (e != cudaSuccess) {
            snprintf(msg, msg_len, "GEMM (stream-K) launch failed: %s", cudaGetErrorString(e));
            return 1;
        }
        return 0;
    }
    // Every CTA gets the same number of tiles (the last wave is not left partial).
    const int per_cta = (p.num_tiles + g.num_sms - 1) / g.num_sms;
    grid = (p.num_tiles + per_cta - 1) / per_cta;
    e = launch_kernel(kern, dim3(grid), dim3(kThreads), Cf::kSmemBytes, stream, g.pdl, tmA, tmB, tmC, p);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) {
        snprintf(msg, msg_len, "GEMM launch failed: %s", cudaGetErrorString(e));
        return 1;
    }
    return 0;
}

template <bool A_MN, bool B_MN, int IN, int OUT, int MB = 1>
int launch_pair_instance(const GemmLaunch& g, cudaStream_t stream, char* msg, size_t msg_len)
{
    using Cf = PairCfg<MB>;
    using Ty = Types<IN, OUT>;
    if (MB != 1 && (g.stream_k || g.dyn)) {
        snprintf(msg, msg_len, "GEMM (CTA pair): 512-row tiles run whole tiles in the fixed order only");
        return 1;
    }
    CUtensorMap tmA, tmB, tmC;
    if (!encode_operands<IN, OUT, A_MN, B_MN>(g, kBM, kBM, &tmA, &tmB, &tmC, msg, msg_len)) return 1;
    Params p;
    p.M = g.M;
    p.bm = kBM;
    p.N = g.N;
    p.K = g.K;
    p.num_m = (g.M + Cf::kTile * MB - 1) / (Cf::kTile * MB);
    p.num_n = (g.N + Cf::kTile - 1) / Cf::kTile;
    p.num_tiles = p.num_m * p.num_n;
    p.num_kb = (g.K + Ty::kBK - 1) / Ty::kBK;
    p.group_m = g.group_m < 1 ? 1 : g.group_m;
    p.C = g.C;
    p.ldc = g.ldc;
    p.tma_store = (Ty::kOutBytes == 2 && g.tma_store) ? 1 : 0;
    p.bias = g.bias;
    p.bias_mode = g.bias != nullptr ? g.bias_mode : 0;
    p.alpha = g.alpha;
    p.sk = 0;
    p.sk_dp_tiles = 0;
    p.sk_iters = 0;
    p.sk_part = nullptr;
    p.sk_flag = nullptr;
    p.status = g.status;
    p.wait_limit_ns = g.wait_limit_ns;
    p.dyn = 0;
    p.skc = 0;
    p.rev_round = 0;
    p.a_rows = nullptr;
    p.a_ld_bytes = 0;
    p.pf_kb = 0;

    auto kern = gemm_tcgen05_pair_kernel<A_MN, B_MN, IN, OUT, MB>;
    static SmemOptIn smem_opt;
    cudaError_t e = smem_opt.ensure(reinterpret_cast<const void*>(kern), Cf::kSmemBytes);
    if (e != cudaSuccess) {
        snprintf(msg, msg_len, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
        return 1;
    }
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = Cf::kSmemBytes;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // Co-resident clusters of this instance: a property of the kernel and the
    // device, queried once per device.
    static std::atomic<int> max_clusters[SmemOptIn::kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= SmemOptIn::kMaxDevices) dev = -1;
    int clusters = dev >= 0 ? max_clusters[dev].load(std::memory_order_acquire) : 0;
    if (clusters < 1) {
        if (cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg) != cudaSuccess || clusters < 1) {
            cudaGetLastError();
            clusters = g.num_sms / 2;
        } else if (dev >= 0) {
            max_clusters[dev].store(clusters, std::memory_order_release);
        }
    }
    if (clusters > g.num_sms / 2) clusters = g.num_sms / 2;
    if (clusters < 1) clusters = 1;
    if (g.stream_k && g.sk_part != nullptr && g.sk_flag != nullptr) {
        // Every co-resident pair takes an equal share of the (tile, k-block)
        // iterations; pairs wait on one another, so the launch is cooperative.
        p.sk = 1;
        p.sk_dp_tiles = (p.num_tiles / clusters) * clusters;
        if (p.sk_dp_tiles == p.num_tiles) p.sk_dp_tiles -= clusters;   // keep one wave to share
        p.sk_iters = static_cast<long long>(p.num_tiles - p.sk_dp_tiles) * p.num_kb;
        const int pairs = static_cast<long long>(clusters) < p.sk_iters ? clusters : static_cast<int>(p.sk_iters);
        p.rev_round = g.k_alternate ? pairs : 0;
        p.sk_part = g.sk_part;
        p.sk_flag = g.sk_flag;
        cudaLaunchAttribute attr2[2];
        attr2[0] = attr[0];
        attr2[1].id = cudaLaunchAttributeCooperative;
        attr2[1].val.cooperative = 1;
        cfg.attrs = attr2;
        cfg.numAttrs = 2;
        cfg.gridDim = dim3(2 * pairs, 1, 1);
        e = cudaLaunchKernelEx(&cfg, kern, tmA, tmB, tmC, p);
        if (e == cudaSuccess) e = cudaGetLastError();
        if (e != cudaSuccess) {
            snprintf(msg, msg_len, "GEMM (CTA pair, stream-K) launch failed: %s", cudaGetErrorString(e));
            return 1;
        }
        return 0;
    }
    const int per_pair = (p.num_tiles + clusters - 1) / clusters;
    const int pairs = (p.num_tiles + per_pair - 1) / per_pair;
    p.rev_round = g.k_alternate ? pairs : 0;   // the dynamic order keeps the fixed order's rounds
    cfg.gridDim = dim3(2 * pairs, 1, 1);
    if (g.dyn) {
        // one cluster per tile: the resident clusters take the tiles of those
        // whose launch they cancel (the kernel's dynamic order)
        p.dyn = 1;
        cfg.gridDim = dim3(2 * static_cast<unsigned>(p.num_tiles), 1, 1);
    }
    cudaLaunchAttribute attr_pdl[2];
    attr_pdl[0] = attr[0];
    attr_pdl[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr_pdl[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr_pdl;
    cfg.numAttrs = g.pdl ? 2 : 1;
    e = cudaLaunchKernelEx(&cfg, kern, tmA, tmB, tmC, p);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) {
        snprintf(msg, msg_len, "GEMM (CTA pair) launch failed: %s", cudaGetErrorString(e));
        return 1;
    }
    return 0;
}

}  // namespace
}  // namespace bsk
