// tcm_gemm_pair.cu -- CTA-pair (cta_group::2, 256-row tile) instantiations of
// the tcgen05 GEMM kernel (tcm_gemm_kernel.cuh).
#include "tcm_gemm_kernel.cuh"

namespace tcm {

cudaError_t launch_gemm_pair(const GemmConfig &cfg, const CUtensorMap &tmA, const CUtensorMap &tmB,
                             const GemmParams &p, int grid, cudaStream_t stream)
{
    if (cfg.bn != 256 || cfg.katoms != 2) return cudaErrorInvalidValue;
    // 3 stages of two 128-byte K atoms (192 KB): against 6 stages of one atom, the same ring
    // bytes with half the barrier waits and commits, 0.5-2 % faster (a 7-stage single-atom
    // ring measured no faster than 6)
    if (cfg.kind == 0) return launch_one<0, 256, 3, 2, 1, 2>(tmA, tmB, p, grid, stream);
    if (cfg.kind == 1) return launch_one<1, 256, 3, 2, 1, 2>(tmA, tmB, p, grid, stream);
    return cudaErrorInvalidValue;
}

} // namespace tcm
