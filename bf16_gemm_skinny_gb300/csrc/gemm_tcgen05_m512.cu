// gemm_tcgen05_m512.cu -- instances of the CTA-pair GEMM on 512 x 256 tiles
// (two 256-row blocks per pair tile, 16-bit inputs, K-major B).  Each CTA
// stages 256 rows of A and 128 rows of B per k step, and every B slice in
// shared memory feeds two MMAs; the kernels are in gemm_tcgen05.cuh.  A
// separate translation unit, so that the build compiles it in parallel.
#include "gemm_tcgen05.cuh"

namespace bsk {

int launch_gemm_pair_m512(const GemmLaunch& g, cudaStream_t stream, char* msg, size_t msg_len)
{
    if (g.b_mn_major || (g.in_type != kInF16 && g.in_type != kInBF16) || g.out_type != g.in_type) {
        snprintf(msg, msg_len, "512-row pair tiles take 16-bit inputs with a K-major B");
        return 1;
    }
    const bool bf16 = g.in_type == kInBF16;
    if (g.a_mn_major)
        return bf16 ? launch_pair_instance<true, false, kInBF16, kOutBF16, 2>(g, stream, msg, msg_len)
                    : launch_pair_instance<true, false, kInF16, kOutF16, 2>(g, stream, msg, msg_len);
    return bf16 ? launch_pair_instance<false, false, kInBF16, kOutBF16, 2>(g, stream, msg, msg_len)
                : launch_pair_instance<false, false, kInF16, kOutF16, 2>(g, stream, msg, msg_len);
}

const void* gemm_pair_m512_colmajor_kernel()
{
    return reinterpret_cast<const void*>(gemm_tcgen05_pair_kernel<true, false, kInF16, kOutF16, 2>);
}

}  // namespace bsk
