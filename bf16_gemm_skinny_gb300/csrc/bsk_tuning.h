/*
 * bsk_tuning.h -- tuning options and test hooks of libbsk.
 *
 * These entry points are exported from libbsk.so for the library's own tests
 * and benchmark.  They are not part of the C ABI in include/bsk.h: the
 * options are process-wide state that changes which kernel, tile width, tile
 * order and schedule every later call of every thread uses, and the hooks
 * exist only to check the library.  A program built on include/bsk.h needs
 * none of them; every option's default is the measured best choice.
 */
#ifndef BSK_TUNING_H
#define BSK_TUNING_H

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Tile order of the GEMM ("Hygon 优化", section 分组调度：提高 L2 数据复用):
 * maps the flattened tile index t of a num_m x num_n tile grid to its tile
 * coordinates, visiting group_m tile rows per tile column, the last group
 * holding the remaining rows.  Host-side copy of the function the kernel
 * uses; needs no GPU.  Invalid arguments give (-1, -1).
 */
void bsk_tile_coord(int t, int num_m, int num_n, int group_m, int* pid_m, int* pid_n);

/*
 * Tuning and test options (process-wide; not thread-safe; 0 restores the
 * default).  Keys:
 *   BSK_OPT_GROUP_M          GEMM tile-row group size (default 8 for CTA pairs, 16 otherwise)
 *   BSK_OPT_BLOCK_N          GEMM tile width 32, 64, 128 or 256 (default: the smallest of
 *                            32/64/128 that covers N, else 256)
 *   BSK_OPT_FORCE_PACK       1: pack A and B even when aligned
 *   BSK_OPT_FORCE_DIRECT_STORE 1: masked register stores instead of the TMA store
 *   BSK_OPT_GEMV_ROWS        GEMV rows of W per warp: 1, 2, 4 or 8 (default by n)
 *   BSK_OPT_GEMV_WARPS       GEMV warps per CTA, 1..16 (default 16 pipelined, 8 streaming)
 *   BSK_OPT_WAIT_LIMIT_US    device-side wait limit in microseconds (default 2 s)
 *   BSK_OPT_NUM_SMS          cap on the persistent GEMM grid (default: all SMs)
 *   BSK_OPT_GEMM_KERNEL      GEMM kernel for 256-wide tiles: 1 one CTA per 128 x 256 tile,
 *                            2 CTA pairs on 256 x 256 tiles (default 2; narrower tiles
 *                            always run one CTA per 128 x BN tile)
 *   BSK_OPT_GEMV_KERNEL      kernel of gemv_bf16 for n <= 8: 1 register streaming,
 *                            2 cp.async-pipelined, 3 pipelined with x kept in BF16,
 *                            4 token-paired (n >= 5) -- the CUDA-core GEMVs -- or 5 the
 *                            tensor-core skinny GEMM (default: 1 for n <= 3, 5 for
 *                            n >= 4; a CUDA-core kernel whose buffers do not fit in
 *                            shared memory falls back to another)
 *   BSK_OPT_STREAM_K         GEMM schedule: 1 whole tiles (no automatic split of any kind),
 *                            2 stream-K (every SM -- or CTA pair -- an equal share of the
 *                            tile x k-block iterations of the last wave; split tiles are
 *                            summed in FP32 by the unit that holds their first k-block),
 *                            0 automatic: on the one-CTA-per-tile kernel, when whole tiles
 *                            would fill under three quarters of the SMs, split-K over a
 *                            cluster where its estimated time is lowest, else stream-K if a
 *                            tile has at least 64 k-blocks; whole tiles on CTA pairs
 *   BSK_OPT_PDL              1: launch the GEMM, GEMV and attention kernels in plain stream
 *                            order; 0 (default): as programmatic dependents of the kernel
 *                            before them in the stream, so that their launch and prologue
 *                            (barrier set-up, TMEM allocation, L2 prefetch of the first
 *                            weight tiles) overlap that kernel's last CTAs.  Either way no
 *                            input is read and no output written before the earlier kernel
 *                            has completed.
 *   BSK_OPT_TILE_SCHED       tile order of the CTA-pair GEMM kernel (whole tiles): 0 or 1
 *                            fixed (pair p takes tiles p, p + P, ...), 2 dynamic (one cluster
 *                            per tile launched; a pair that is done takes the tile of a
 *                            cluster whose launch it cancels, so tiles go to the pairs that
 *                            are free first; BSK_OPT_NUM_SMS does not cap this grid)
 *   BSK_OPT_BLOCK_M          rows per tile of the one-CTA GEMM kernel with a K-major A and a
 *                            single tile column (the skinny decode shapes): 8..128, a
 *                            multiple of 8 (default 128; other shapes always use 128)
 *   BSK_OPT_SPLIT_K          split-K over a cluster of the one-CTA GEMM kernel: 0 automatic
 *                            (tile-starved problems), 1 off, 2 / 4 / 8 / 16 force that cluster
 *                            size (one-CTA kernel, whole tiles; 16 needs a non-portable cluster)
 *   BSK_OPT_PREFETCH_KB      one-CTA GEMM kernel with a K-major A (the skinny decode shapes):
 *                            k-blocks of the first tile's A rows that the epilogue warps
 *                            prefetch into L2 while the launch waits for the kernel before
 *                            it, beyond the two stages the producer prefetches: 0 automatic
 *                            (16), 1 none, 2..64 that many
 *   BSK_OPT_K_ORDER          k order of the CTA-pair GEMM's whole tiles: 0 automatic (odd
 *                            rounds of tiles descending, so a round starts on the k-slices
 *                            the round before it left in L2), 1 always ascending
 *   BSK_OPT_PAIR_M           rows of a CTA-pair tile (16-bit inputs, K-major B, whole tiles in
 *                            the fixed order): 0 automatic, 1 256 x 256 tiles, 2 512 x 256
 *                            tiles (each CTA stages 256 rows of A; every B slice feeds two
 *                            MMAs; one accumulator, so the epilogue no longer overlaps the
 *                            next tile's MMAs)
 * Returns BSK_ERR_INVALID_ARG for an unknown key or a value out of range.
 */
enum {
    BSK_OPT_GROUP_M = 1,
    BSK_OPT_BLOCK_N = 2,
    BSK_OPT_FORCE_PACK = 3,
    BSK_OPT_FORCE_DIRECT_STORE = 4,
    BSK_OPT_GEMV_ROWS = 5,
    BSK_OPT_GEMV_WARPS = 6,
    BSK_OPT_WAIT_LIMIT_US = 7,
    BSK_OPT_NUM_SMS = 8,
    BSK_OPT_GEMV_KERNEL = 9,
    BSK_OPT_GEMM_KERNEL = 10,
    BSK_OPT_STREAM_K = 11,
    BSK_OPT_PDL = 12,
    BSK_OPT_TILE_SCHED = 13,
    BSK_OPT_BLOCK_M = 14,
    BSK_OPT_SPLIT_K = 15,
    BSK_OPT_PREFETCH_KB = 16,
    BSK_OPT_K_ORDER = 17,
    BSK_OPT_PAIR_M = 18
};
int bsk_set_option(int key, long long value);
long long bsk_get_option(int key);

/*
 * Test hook: the plan gemm_f16 / gemm_fp8 would take for an M x N x K product
 * (column-major storage; a_mn_major / b_mn_major as the kernels see the
 * operands; fp8 nonzero for E4M3 inputs) on `sms` SMs under the current
 * options, written to plan[0..6]: tile width, tile height of the one-CTA
 * kernel, CTA pairs (0/1), stream-K (0/1), split-K cluster size (0 = none),
 * 256-row blocks per pair tile (1/2), dynamic tile order (0/1).  Split-K plans
 * depend on how many clusters fit on the current device: without a device
 * none is considered.  Launches nothing.
 */
int bsk_plan_gemm(int M, int N, int K, int a_mn_major, int b_mn_major, int fp8, int sms, int* plan);

/*
 * Test hook for the watchdog: launches one CTA that waits on a barrier that
 * nothing completes, using the GEMM's bounded wait with a limit of
 * `limit_us` microseconds (1 .. 10,000,000).  Returns BSK_ERR_TIMEOUT when the
 * wait gave up as designed, BSK_OK never.  Blocks until the probe finished.
 */
int bsk_test_wait_timeout(unsigned int limit_us, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* BSK_TUNING_H */
