// tcm_gemm_pair.cu -- CTA-pair (cta_group::2, 256-row tile) instantiations of
// the tcgen05 GEMM kernel (tcm_gemm_kernel.cuh).
#include "tcm_gemm_kernel.cuh"

namespace tcm {

cudaError_t launch_gemm_pair(const GemmConfig &cfg, const CUtensorMap &tmA, const CUtensorMap &tmB,
                             const GemmParams &p, int grid, cudaStream_t stream)
{
    if (cfg.bn != 256) return cudaErrorInvalidValue;
    const bool deep = cfg.stages == 7;
    if (cfg.kind == 0)
        return deep ? launch_one<0, 256, 7, 2>(tmA, tmB, p, grid, stream)
                    : launch_one<0, 256, 6, 2>(tmA, tmB, p, grid, stream);
    if (cfg.kind == 1)
        return deep ? launch_one<1, 256, 7, 2>(tmA, tmB, p, grid, stream)
                    : launch_one<1, 256, 6, 2>(tmA, tmB, p, grid, stream);
    return cudaErrorInvalidValue;
}

} // namespace tcm
