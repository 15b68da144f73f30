// tcm_gemm_pair.cu -- CTA-pair (cta_group::2, 256-row tile) instantiations of
// the tcgen05 GEMM kernel (tcm_gemm_kernel.cuh).
#include "tcm_gemm_kernel.cuh"

namespace tcm {

cudaError_t launch_gemm_pair(const GemmConfig &cfg, const CUtensorMap &tmA, const CUtensorMap &tmB,
                             const GemmParams &p, int grid, cudaStream_t stream)
{
    if (cfg.bn != 256) return cudaErrorInvalidValue;
    // 16-bit operands: 6 stages of one 128-byte K atom (a 7-stage ring measured no faster;
    // 3 stages of two atoms took ~2 % more cycles at 8192^3).  8-bit operands: 3 stages of
    // two atoms (192 KB, the same ring bytes), eight MMAs per barrier wait and commit:
    // E4M3 8192^3 1 %, 4096^3 3 % faster than 6 x 1.
    if (cfg.kind == 0 && cfg.katoms == 1) return launch_one<0, 256, 6, 2>(tmA, tmB, p, grid, stream);
    if (cfg.kind == 1 && cfg.katoms == 2) return launch_one<1, 256, 3, 2, 1, 2>(tmA, tmB, p, grid, stream);
    return cudaErrorInvalidValue;
}

} // namespace tcm
