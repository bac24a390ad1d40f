// Instantiations of the persistent kernel for an activation on an fp32 D
// (ReLU, GELU), compiled apart from the plain epilogue for a parallel build.

#include "mp_kernel.cuh"

namespace mp {

cudaError_t launch_poly_gemm_act_f32(const cudaLaunchConfig_t& cfg, bool pair, int epi, const dev::Params& p) {
    switch (epi) {
        case 1: return launch_poly_gemm<1>(cfg, pair, p);
        case 2: return launch_poly_gemm<2>(cfg, pair, p);
        case 9: return launch_poly_gemm<9>(cfg, pair, p);    // lean (bit 3)
        case 10: return launch_poly_gemm<10>(cfg, pair, p);
        default: return cudaErrorInvalidValue;
    }
}

bool set_poly_gemm_smem_act_f32() {
    return set_poly_gemm_smem<1>() && set_poly_gemm_smem<2>() && set_poly_gemm_smem<9>() && set_poly_gemm_smem<10>();
}

}  // namespace mp
