// Instantiations of the persistent kernel for a bf16 D (no activation, ReLU,
// GELU), compiled apart from the plain epilogue for a parallel build.

#include "mp_kernel.cuh"

namespace mp {

cudaError_t launch_poly_gemm_bf16(const cudaLaunchConfig_t& cfg, bool pair, int epi, const dev::Params& p) {
    switch (epi) {
        case 4: return launch_poly_gemm<4>(cfg, pair, p);
        case 5: return launch_poly_gemm<5>(cfg, pair, p);
        case 6: return launch_poly_gemm<6>(cfg, pair, p);
        case 12: return launch_poly_gemm<12>(cfg, pair, p);  // lean (bit 3)
        case 13: return launch_poly_gemm<13>(cfg, pair, p);
        case 14: return launch_poly_gemm<14>(cfg, pair, p);
        default: return cudaErrorInvalidValue;
    }
}

bool set_poly_gemm_smem_bf16() {
    return set_poly_gemm_smem<4>() && set_poly_gemm_smem<5>() && set_poly_gemm_smem<6>() && set_poly_gemm_smem<12>() &&
           set_poly_gemm_smem<13>() && set_poly_gemm_smem<14>();
}

}  // namespace mp
