// tcm_gemm_ksplit.cu -- K-split-cluster instantiations of the tcgen05 GEMM
// kernel (tcm_gemm_kernel.cuh): 2 or 4 single-CTA tiles share K, partial sums
// reduced through distributed shared memory.
#include "tcm_gemm_kernel.cuh"

namespace tcm {

cudaError_t launch_gemm_ksplit(const GemmConfig &cfg, const CUtensorMap &tmA, const CUtensorMap &tmB,
                               const GemmParams &p, int grid, cudaStream_t stream)
{
    if (cfg.cta_group != 1) return cudaErrorInvalidValue;
#define TCM_KSPLIT(KIND)                                                                                            \
    if (cfg.bn == 32 && cfg.ksplit == 2 && cfg.katoms == 2)                                                         \
        return launch_one<KIND, 32, 5, 1, 2, 2>(tmA, tmB, p, grid, stream);                                          \
    if (cfg.bn == 32 && cfg.ksplit == 2) return launch_one<KIND, 32, 10, 1, 2>(tmA, tmB, p, grid, stream);          \
    if (cfg.bn == 32 && cfg.ksplit == 4) return launch_one<KIND, 32, 8, 1, 4>(tmA, tmB, p, grid, stream);           \
    if (cfg.bn == 64 && cfg.ksplit == 2) return launch_one<KIND, 64, 8, 1, 2>(tmA, tmB, p, grid, stream);           \
    if (cfg.bn == 64 && cfg.ksplit == 4) return launch_one<KIND, 64, 5, 1, 4>(tmA, tmB, p, grid, stream);
    if (cfg.kind == 0) { TCM_KSPLIT(0) }
    if (cfg.kind == 1) { TCM_KSPLIT(1) }
#undef TCM_KSPLIT
    return cudaErrorInvalidValue;
}

} // namespace tcm
