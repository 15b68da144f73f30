// tcm_gemm.cu -- single-CTA instantiations of the tcgen05 GEMM kernel and the
// dispatch over all dense variants (the kernel itself is in tcm_gemm_kernel.cuh).
#include "tcm_gemm_kernel.cuh"

namespace tcm {

cudaError_t launch_gemm(const GemmConfig &cfg, const CUtensorMap &tmA, const CUtensorMap &tmB,
                        const GemmParams &p, int grid, cudaStream_t stream)
{
    if (cfg.ksplit > 1) return launch_gemm_ksplit(cfg, tmA, tmB, p, grid, stream);
    if (cfg.cta_group == 2) return launch_gemm_pair(cfg, tmA, tmB, p, grid, stream);
#define TCM_DISPATCH(KIND)                                                                                          \
    switch (cfg.bn) {                                                                                               \
    case 256: return launch_one<KIND, 256, 4, 1>(tmA, tmB, p, grid, stream);                                        \
    case 128: return launch_one<KIND, 128, 6, 1>(tmA, tmB, p, grid, stream);                                        \
    case 64: return launch_one<KIND, 64, 8, 1>(tmA, tmB, p, grid, stream);                                          \
    case 32:                                                                                                        \
        return cfg.katoms == 2 ? launch_one<KIND, 32, 5, 1, 1, 2>(tmA, tmB, p, grid, stream)                        \
                               : launch_one<KIND, 32, 10, 1>(tmA, tmB, p, grid, stream);                            \
    default: return cudaErrorInvalidValue;                                                                          \
    }
    if (cfg.kind == 0) { TCM_DISPATCH(0) }
    if (cfg.kind == 1) { TCM_DISPATCH(1) }
#undef TCM_DISPATCH
    return cudaErrorInvalidValue;
}

} // namespace tcm
