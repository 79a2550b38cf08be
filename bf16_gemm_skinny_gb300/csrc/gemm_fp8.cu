// gemm_fp8.cu -- instances and dispatch of the FP8 tcgen05 GEMMs: A and B both
// E4M3 or both E5M2, K-major, FP32 accumulation, C = alpha * A * B stored as
// FP32 or rounded once to BF16 (the FP8 row of the matrix-instruction table in
// "Hygon 优化", section DUMMA 矩阵指令形状: FP8 inputs, FP32 accumulator).
// The kernels are the ones of gemm_tcgen05.cuh on tcgen05.mma kind::f8f6f4.
#include "gemm_tcgen05.cuh"

namespace bsk {
namespace {

template <int IN, int OUT>
int dispatch_fp8(const GemmLaunch& g, cudaStream_t stream, char* msg, size_t msg_len)
{
    switch (g.block_n) {
    case 256:
        return g.pair ? launch_pair_instance<false, false, IN, OUT>(g, stream, msg, msg_len)
                      : launch_instance<256, false, false, IN, OUT>(g, stream, msg, msg_len);
    case 128: return launch_instance<128, false, false, IN, OUT>(g, stream, msg, msg_len);
    case 64: return launch_instance<64, false, false, IN, OUT>(g, stream, msg, msg_len);
    case 32: return launch_instance<32, false, false, IN, OUT>(g, stream, msg, msg_len);
    default:
        snprintf(msg, msg_len, "unsupported block_n %d (32, 64, 128 or 256)", g.block_n);
        return 1;
    }
}

}  // namespace

int launch_gemm_fp8(const GemmLaunch& g, cudaStream_t stream, char* msg, size_t msg_len)
{
    if (g.a_mn_major || g.b_mn_major) {
        snprintf(msg, msg_len, "FP8 operands must be K-major");
        return 1;
    }
    if (g.bias != nullptr) {
        snprintf(msg, msg_len, "the FP8 GEMM takes no bias");
        return 1;
    }
    const bool e5m2 = g.in_type == kInE5M2;
    if (g.out_type == kOutF32)
        return e5m2 ? dispatch_fp8<kInE5M2, kOutF32>(g, stream, msg, msg_len)
                    : dispatch_fp8<kInE4M3, kOutF32>(g, stream, msg, msg_len);
    if (g.out_type == kOutBF16)
        return e5m2 ? dispatch_fp8<kInE5M2, kOutBF16>(g, stream, msg, msg_len)
                    : dispatch_fp8<kInE4M3, kOutBF16>(g, stream, msg, msg_len);
    snprintf(msg, msg_len, "FP8 GEMM output type %d is not FP32 or BF16", g.out_type);
    return 1;
}

}  // namespace bsk
