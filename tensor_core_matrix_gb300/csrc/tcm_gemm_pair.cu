// tcm_gemm_pair.cu -- CTA-pair (cta_group::2, 256-row tile) instantiations of
// the tcgen05 GEMM kernel (tcm_gemm_kernel.cuh).
#include "tcm_gemm_kernel.cuh"

namespace tcm {

cudaError_t launch_gemm_pair(const GemmConfig &cfg, const CUtensorMap &tmA, const CUtensorMap &tmB,
                             const GemmParams &p, int grid, cudaStream_t stream)
{
    if (cfg.bn != 256) return cudaErrorInvalidValue;
    // 6 stages (a 7-stage ring measured no faster)
    if (cfg.kind == 0) return launch_one<0, 256, 6, 2>(tmA, tmB, p, grid, stream);
    if (cfg.kind == 1) return launch_one<1, 256, 6, 2>(tmA, tmB, p, grid, stream);
    return cudaErrorInvalidValue;
}

} // namespace tcm
