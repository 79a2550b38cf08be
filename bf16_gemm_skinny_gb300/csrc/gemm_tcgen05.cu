// gemm_tcgen05.cu -- instances and dispatch of the 16-bit tcgen05 GEMMs
// (FP16 in/out with any operand majorness, BF16 in/out with an MN- or K-major
// A); the kernels are in gemm_tcgen05.cuh, the FP8 instances in gemm_fp8.cu.
#include "gemm_tcgen05.cuh"

namespace bsk {
namespace {

// B MN-major (a transposed B) is instantiated for FP16 only.
template <int BN>
int dispatch_single(const GemmLaunch& g, cudaStream_t stream, char* msg, size_t msg_len)
{
    const bool bf16 = g.in_type == kInBF16;
    if (g.b_mn_major) {
        if constexpr (BN >= 64) {
            if (bf16) {
                snprintf(msg, msg_len, "a transposed B operand is supported for FP16 only");
                return 1;
            }
            return g.a_mn_major ? launch_instance<BN, true, true, kInF16, kOutF16>(g, stream, msg, msg_len)
                                : launch_instance<BN, false, true, kInF16, kOutF16>(g, stream, msg, msg_len);
        } else {
            snprintf(msg, msg_len, "a transposed B operand needs block_n >= 64");
            return 1;
        }
    }
    if (g.a_mn_major)
        return bf16 ? launch_instance<BN, true, false, kInBF16, kOutBF16>(g, stream, msg, msg_len)
                    : launch_instance<BN, true, false, kInF16, kOutF16>(g, stream, msg, msg_len);
    return bf16 ? launch_instance<BN, false, false, kInBF16, kOutBF16>(g, stream, msg, msg_len)
                : launch_instance<BN, false, false, kInF16, kOutF16>(g, stream, msg, msg_len);
}

int dispatch_pair(const GemmLaunch& g, cudaStream_t stream, char* msg, size_t msg_len)
{
    const bool bf16 = g.in_type == kInBF16;
    if (g.b_mn_major) {
        if (bf16) {
            snprintf(msg, msg_len, "a transposed B operand is supported for FP16 only");
            return 1;
        }
        return g.a_mn_major ? launch_pair_instance<true, true, kInF16, kOutF16>(g, stream, msg, msg_len)
                            : launch_pair_instance<false, true, kInF16, kOutF16>(g, stream, msg, msg_len);
    }
    if (g.a_mn_major)
        return bf16 ? launch_pair_instance<true, false, kInBF16, kOutBF16>(g, stream, msg, msg_len)
                    : launch_pair_instance<true, false, kInF16, kOutF16>(g, stream, msg, msg_len);
    return bf16 ? launch_pair_instance<false, false, kInBF16, kOutBF16>(g, stream, msg, msg_len)
                : launch_pair_instance<false, false, kInF16, kOutF16>(g, stream, msg, msg_len);
}

}  // namespace

int preload_gemm_f16_colmajor_kernels(char* msg, size_t msg_len)
{
    // the instances gemm_f16_colmajor may pick: MN-major A, K-major B, FP16 in
    // and out, on CTA pairs or one CTA per 128 x BN tile
    const void* kernels[] = {
        reinterpret_cast<const void*>(gemm_tcgen05_pair_kernel<true, false, kInF16, kOutF16, 1>),
        gemm_pair_m512_colmajor_kernel(),
        reinterpret_cast<const void*>(gemm_tcgen05_kernel<256, true, false, kInF16, kOutF16>),
        reinterpret_cast<const void*>(gemm_tcgen05_kernel<128, true, false, kInF16, kOutF16>),
        reinterpret_cast<const void*>(gemm_tcgen05_kernel<64, true, false, kInF16, kOutF16>),
        reinterpret_cast<const void*>(gemm_tcgen05_kernel<32, true, false, kInF16, kOutF16>),
    };
    for (const void* k : kernels) {
        cudaFuncAttributes attr;
        const cudaError_t e = cudaFuncGetAttributes(&attr, k);
        if (e != cudaSuccess) {
            snprintf(msg, msg_len, "cudaFuncGetAttributes (GEMM kernel): %s", cudaGetErrorString(e));
            return 1;
        }
    }
    return 0;
}

int split_k_capacity(int skc)
{
    // Every instance of the one-CTA kernel takes one SM (its ring fills the
    // shared memory), so the count is the same for all: queried once per device
    // and size on one instance.
    static std::atomic<int> cache[SmemOptIn::kMaxDevices][5];
    if (skc < 1 || skc > 16 || (skc & (skc - 1)) != 0) return 0;
    int lg = 0;
    while ((1 << lg) < skc) ++lg;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= SmemOptIn::kMaxDevices) dev = -1;
    int n = dev >= 0 ? cache[dev][lg].load(std::memory_order_acquire) : 0;
    if (n > 0) return n;
    using Cf = Cfg<32>;
    auto kern = gemm_tcgen05_kernel<32, true, false, kInF16, kOutF16>;
    static SmemOptIn smem_opt;
    if (smem_opt.ensure(reinterpret_cast<const void*>(kern), Cf::kSmemBytes) != cudaSuccess ||
        (skc > 8 && cudaFuncSetAttribute(reinterpret_cast<const void*>(kern),
                                         cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)) {
        cudaGetLastError();
        return 0;
    }
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(skc);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(skc), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = Cf::kSmemBytes;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    if (n > 0 && dev >= 0) cache[dev][lg].store(n, std::memory_order_release);
    return n;
}

int launch_gemm(const GemmLaunch& g, cudaStream_t stream, char* msg, size_t msg_len)
{
    if (g.in_type == kInE4M3 || g.in_type == kInE5M2) return launch_gemm_fp8(g, stream, msg, msg_len);
    if (g.in_type != kInF16 && g.in_type != kInBF16) {
        snprintf(msg, msg_len, "unknown input type %d", g.in_type);
        return 1;
    }
    if (g.out_type != g.in_type) {
        snprintf(msg, msg_len, "16-bit GEMMs produce their input type");
        return 1;
    }
    if (g.block_n == 256 && g.pair && g.pair_m == 2 && !g.stream_k && !g.dyn && !g.b_mn_major)
        return launch_gemm_pair_m512(g, stream, msg, msg_len);
    switch (g.block_n) {
    case 256: return g.pair ? dispatch_pair(g, stream, msg, msg_len) : dispatch_single<256>(g, stream, msg, msg_len);
    case 128: return dispatch_single<128>(g, stream, msg, msg_len);
    case 64: return dispatch_single<64>(g, stream, msg, msg_len);
    case 32: return dispatch_single<32>(g, stream, msg, msg_len);
    default:
        snprintf(msg, msg_len, "unsupported block_n %d (32, 64, 128 or 256)", g.block_n);
        return 1;
    }
}

}  // namespace bsk
