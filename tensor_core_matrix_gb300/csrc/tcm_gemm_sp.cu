// tcm_gemm_sp.cu -- GEMM with a 2:4 structured-sparse A on tcgen05.mma.sp.
//
// "NVIDIA MMA", section "稠密乘法与 2:4 结构化稀疏乘法": only A is sparse (two
// kept values of every four along K plus their positions), B, C and D stay
// dense, and a sparse instruction covers twice the logical K of the dense
// one; section "SM100：tcgen05.mma": the `.sp` form reads its metadata from
// tensor memory ([sp-meta-tmem]).
//
// Same pipeline as the dense kernel (tcm_gemm.cu), with these differences:
//   * one stage covers 128 logical K: A_comp 128 rows x 64 kept values
//     (128 bytes, one swizzle atom) and B BN_CTA rows x 128 values (two
//     128-byte atoms);
//   * four tcgen05.mma.sp per stage, logical K = 32 each (A +32 bytes, B
//     +64 bytes per instruction);
//   * two groups of four warps (6..9, 10..13) move the metadata into tensor
//     memory, alternating stages so that one group's store-and-signal
//     latency overlaps the other's.  The library
//     layout keeps, per row, one 32-bit word per 32 logical K (8 nibbles
//     i0 | i1 << 2).  The MMA reads, for each 16-row block, lane 16a+8s+r:
//     bits 0..15 = nibbles 4s..4s+3 of row 16a+r, bits 16..31 = the same
//     nibbles of row 16a+8+r.  Each thread owns one row, so the lane word is
//     its own word combined with the word of row (row ^ 8), fetched with one
//     shuffle.  The words go to TMEM with tcgen05.st, then the warps signal
//     `meta_full` for the issuer.  Each MMA reads its metadata from a column
//     whose index is a multiple of 4 (stride 4 between the MMAs of a stage).
//     Rows or K beyond the matrix get positions {0,1} (their A values are
//     zero-filled by TMA, so any valid positions give zero).
#include "tcm_kernel_common.cuh"

namespace tcm {

constexpr int META_GROUPS = 2;  // metadata warpgroups; group g handles the items i with i % 2 == g
constexpr int SP_THREADS = 32 * (2 + 4 + 4 * META_GROUPS); // warps 0 TMA, 1 MMA, 2-5 epilogue, 6.. metadata
constexpr int META_WARPS = 4;   // warps per metadata group (one per TMEM lane quadrant)
constexpr uint32_t META_FILL = 0x44444444u; // every group: positions {0, 1}
constexpr int META_AHEAD = 8;               // metadata items fetched ahead of use

template <int BN_CTA, int STAGES>
struct SpSmem {
    static constexpr int B_STAGE = 2 * BN_CTA * TILE_K_BYTES; // two 128-byte atoms of K
    static constexpr int A_OFF = 0;
    static constexpr int B_OFF = STAGES * A_STAGE_BYTES;
    static constexpr int BAR_OFF = B_OFF + STAGES * B_STAGE;
    static constexpr int NUM_BARS = 3 * STAGES + 5; // full, empty, meta_full, tfull[2], tempty[2], drain
    static constexpr int MISC_OFF = BAR_OFF + NUM_BARS * 8;
    static constexpr int BYTES = MISC_OFF + 16;
    static constexpr int ALLOC = BYTES + 1024;
};

__device__ __forceinline__ void mma_sp_f16_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t meta_tmem,
                                               uint32_t idesc, uint32_t accumulate)
{
    asm volatile(
        "{\n"
        ".reg .pred p;\n"
        "setp.ne.b32 p, %5, 0;\n"
        "tcgen05.mma.sp.cta_group::2.kind::f16 [%0], %1, %2, [%3], %4, p;\n"
        "}\n" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(meta_tmem), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Library metadata words of one row for logical K [128*kb, 128*kb + 128).
__device__ __forceinline__ void load_meta4(const GemmParams &p, int row, int kb, uint32_t (&w)[4])
{
#pragma unroll
    for (int j = 0; j < 4; ++j) w[j] = META_FILL;
    if (row >= p.kM) return;
    const long long first = static_cast<long long>(kb) * 4;
    const uint32_t *src = p.meta + static_cast<long long>(row) * p.meta_ld + first;
    if (first + 4 <= p.meta_ld && (reinterpret_cast<uintptr_t>(src) & 15u) == 0) {
        const uint4 v = __ldg(reinterpret_cast<const uint4 *>(src));
        w[0] = v.x, w[1] = v.y, w[2] = v.z, w[3] = v.w;
    } else {
#pragma unroll
        for (int j = 0; j < 4; ++j)
            if (first + j < p.meta_ld) w[j] = __ldg(src + j);
    }
}

// Row of D (and of A) that metadata item i of this CTA's walk belongs to.
template <int CG>
__device__ __forceinline__ int meta_row(const GemmParams &p, long long i, int first_tile, int num_clusters,
                                        uint32_t rank, int row_in_tile)
{
    const int t = first_tile + static_cast<int>(i / p.num_kb) * num_clusters;
    int mb, nb;
    tile_coords(p, t, mb, nb);
    return mb * (BM * CG) + static_cast<int>(rank) * BM + row_in_tile;
}

// BN: N extent of the (pair) tile; CG: CTA group (see the dense kernel);
// NACC: accumulators in tensor memory (2 lets the epilogue overlap the next tile).
template <int BN, int STAGES, int CG, int NACC>
__global__ void __launch_bounds__(SP_THREADS, 1)
    gemm_sp_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, const GemmParams p)
{
    constexpr int BN_CTA = BN / CG;
    using L = SpSmem<BN_CTA, STAGES>;
    static_assert(L::ALLOC <= 227 * 1024, "shared memory ring too large");
    static_assert(BN % 32 == 0 && BN_CTA <= 256, "tile width");
    static_assert(STAGES % META_GROUPS == 0, "each metadata group owns whole stages");
    // accumulators at power-of-two columns, then 16 metadata columns per stage
    constexpr uint32_t ACC_STRIDE = BN <= 128 ? 128u : 256u;
    constexpr uint32_t META_COL = ACC_STRIDE * NACC;
    constexpr uint32_t META_STAGE_COLS = 16;
    static_assert(META_COL + META_STAGE_COLS * STAGES <= 512, "tensor memory budget");
    constexpr uint32_t TMEM_COLS = META_COL + META_STAGE_COLS * STAGES <= 256 ? 256 : 512;
    constexpr uint32_t STAGE_TX = CG * (A_STAGE_BYTES + L::B_STAGE);

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    const uint32_t sbase = smem_u32(smem);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L::BAR_OFF);
    uint64_t *empty = full + STAGES;
    uint64_t *meta_full = empty + STAGES;
    uint64_t *tfull = meta_full + STAGES;
    uint64_t *tempty = tfull + 2;
    uint64_t *drain = tempty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::MISC_OFF);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::MISC_OFF + 4);

    const int warp = __shfl_sync(0xffffffffu, static_cast<int>(threadIdx.x >> 5), 0);
    const int lane = threadIdx.x & 31;
    const uint32_t rank = CG == 2 ? cluster_ctarank() : 0u;
    const bool leader = rank == 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, 1);
            mbar_init(meta_full + s, META_WARPS * CG);
        }
        for (int a = 0; a < NACC; ++a) {
            mbar_init(tfull + a, 1);
            mbar_init(tempty + a, EPI_WARPS * CG);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 1) {
        if (CG == 2) {
            tmem_alloc_pair(tmem_slot, TMEM_COLS);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(tmem_slot, TMEM_COLS);
            tmem_relinquish();
        }
    }
    tc_fence_before();
    __syncthreads();
    if (CG == 2) cluster_sync();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    const Waiter w{abort_flag, p.timeout_ns, p.status};
    const int cluster_id = static_cast<int>(blockIdx.x) / CG;
    const int num_clusters = static_cast<int>(gridDim.x) / CG;
    const int first_tile = p.tile_begin + cluster_id;

    if (warp == 0) {
        if (lane == 0) {
            const uint32_t full_cluster0 = CG == 2 ? mapa_shared(smem_u32(full), 0) : smem_u32(full);
            int stage = 0;
            uint32_t phase = 0;
            long long issued = 0;
            bool ok = true;
            for (int t = first_tile; ok && t < p.tile_end; t += num_clusters) {
                int mb, nb;
                tile_coords(p, t, mb, nb);
                const int a_row = mb * (BM * CG) + static_cast<int>(rank) * BM;
                const int b_row = nb * BN + static_cast<int>(rank) * BN_CTA;
                for (int kb = 0; kb < p.num_kb; ++kb) {
                    if (!wait_bar<CG>(empty + stage, phase ^ 1u, w, SITE_LOAD_EMPTY, true)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sa = sbase + L::A_OFF + stage * A_STAGE_BYTES;
                    const uint32_t sb = sbase + L::B_OFF + stage * L::B_STAGE;
                    const int ka = kb * 64;   // kept values of A per stage
                    const int kl = kb * 128;  // logical K of B per stage
                    if (CG == 2) {
                        if (leader) mbar_arrive_expect_tx(full + stage, STAGE_TX);
                        const uint32_t fb = full_cluster0 + static_cast<uint32_t>(stage) * 8u;
                        tma_load_2d_pair(sa, &tmA, fb, ka, a_row);
                        tma_load_2d_pair(sb, &tmB, fb, kl, b_row);
                        tma_load_2d_pair(sb + BN_CTA * TILE_K_BYTES, &tmB, fb, kl + 64, b_row);
                    } else {
                        mbar_arrive_expect_tx(full + stage, STAGE_TX);
                        tma_load_2d(sa, &tmA, full + stage, ka, a_row);
                        tma_load_2d(sb, &tmB, full + stage, kl, b_row);
                        tma_load_2d(sb + BN_CTA * TILE_K_BYTES, &tmB, full + stage, kl + 64, b_row);
                    }
                    ++issued;
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            for (int s = 0; s < STAGES; ++s) {
                const long long n = issued > s ? (issued - s + STAGES - 1) / STAGES : 0;
                if (n == 0) continue;
                const uint32_t last = static_cast<uint32_t>((n - 1) & 1);
                if (leader) wait_bar<CG>(full + s, last, w, SITE_DRAIN, false);
                else wait_bar<CG>(empty + s, last, w, SITE_DRAIN, false);
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            int local = 0;
            for (int t = first_tile; ok && t < p.tile_end; t += num_clusters, ++local) {
                const int acc = local % NACC;
                const uint32_t acc_phase = (local / NACC) & 1;
                if (!wait_bar<CG>(tempty + acc, acc_phase ^ 1u, w, SITE_MMA_ACC_EMPTY, true)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc) * ACC_STRIDE;
                for (int kb = 0; kb < p.num_kb; ++kb) {
                    if (!wait_bar<CG>(full + stage, phase, w, SITE_MMA_FULL, true) ||
                        !wait_bar<CG>(meta_full + stage, phase, w, SITE_MMA_META, true)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t ad = sdesc_kmajor_sw128(sbase + L::A_OFF + stage * A_STAGE_BYTES);
                    const uint32_t sb = sbase + L::B_OFF + stage * L::B_STAGE;
                    const uint64_t bd0 = sdesc_kmajor_sw128(sb);
                    const uint64_t bd1 = sdesc_kmajor_sw128(sb + BN_CTA * TILE_K_BYTES);
                    const uint32_t meta_t = tmem_base + META_COL + static_cast<uint32_t>(stage) * META_STAGE_COLS;
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        // A: +32 bytes (16 kept values) per MMA; B: +64 bytes (32 logical K) within its atom
                        const uint64_t bd = (k < 2 ? bd0 : bd1) + 4 * (k & 1);
                        const uint32_t accum = (kb > 0 || k > 0) ? 1u : 0u;
                        if (CG == 2) mma_sp_f16_pair(d_tmem, ad + 2 * k, bd, meta_t + 4 * k, p.idesc, accum);
                        else mma_sp_f16(d_tmem, ad + 2 * k, bd, meta_t + 4 * k, p.idesc, accum);
                    }
                    if (CG == 2) mma_commit_pair(empty + stage, 0x3);
                    else mma_commit(empty + stage);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                if (CG == 2) mma_commit_pair(tfull + acc, 0x3);
                else mma_commit(tfull + acc);
            }
            if (CG == 2) mma_commit_pair(drain, 0x1);
            else mma_commit(drain);
            wait_bar<CG>(drain, 0, w, SITE_DRAIN, false);
        }
    } else if (warp < 2 + EPI_WARPS) {
        const int quad = warp & 3;
        const int row_in_tile = quad * 32 + lane;
        const float scale = p.alpha;
        const uint32_t tempty_cluster0 = CG == 2 ? mapa_shared(smem_u32(tempty), 0) : 0u;
        int local = 0;
        for (int t = first_tile; t < p.tile_end; t += num_clusters, ++local) {
            const int acc = local % NACC;
            const uint32_t acc_phase = (local / NACC) & 1;
            int ok = 1;
            if (lane == 0) ok = wait_bar<CG>(tfull + acc, acc_phase, w, SITE_EPI_ACC_FULL, true);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            tc_fence_after();
            int mb, nb;
            tile_coords(p, t, mb, nb);
            const int row = mb * (BM * CG) + static_cast<int>(rank) * BM + row_in_tile;
            const uint32_t tbase = tmem_base + static_cast<uint32_t>(acc) * ACC_STRIDE + (static_cast<uint32_t>(quad * 32) << 16);
#pragma unroll 1
            for (int c = 0; c < BN; c += 32) {
                uint32_t r[32];
                if (p.num_kb > 0) {
                    tmem_ld_32x32b_x32(tbase + c, r);
                    tmem_ld_wait();
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j) r[j] = 0u;
                }
                if (c + 32 >= BN) {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        if (CG == 2) mbar_arrive_cluster(tempty_cluster0 + static_cast<uint32_t>(acc) * 8u);
                        else mbar_arrive(tempty + acc);
                    }
                }
                epilogue_row32(p, scale, row, nb * BN + c, r);
            }
        }
    } else {
        // metadata warps: TMEM lanes 32*quad .. +31 <- this CTA's rows.  The
        // (tile, k-block) items are walked in the issuer's order; group g takes
        // items g, g+2, g+4 ... (STAGES is even, so each group owns a fixed set
        // of stages).  Each item's words are fetched META_AHEAD items of the
        // group early into a register ring so the global-memory latency
        // overlaps the stages in between.
        const int quad = warp & 3;
        const int group = (warp - 2 - EPI_WARPS) / META_WARPS;
        const int row_in_tile = quad * 32 + lane;
        const uint32_t meta_full_cluster0 = CG == 2 ? mapa_shared(smem_u32(meta_full), 0) : 0u;
        const bool upper = (lane & 8) != 0; // s of lane 16a + 8s + r
        const int my_tiles = first_tile < p.tile_end ? (p.tile_end - 1 - first_tile) / num_clusters + 1 : 0;
        const long long items = static_cast<long long>(my_tiles) * p.num_kb;
        uint32_t ring[META_AHEAD][4];
#pragma unroll
        for (int u = 0; u < META_AHEAD; ++u) {
            const long long i = group + static_cast<long long>(META_GROUPS) * u;
            if (i < items) load_meta4(p, meta_row<CG>(p, i, first_tile, num_clusters, rank, row_in_tile), static_cast<int>(i % p.num_kb), ring[u]);
        }
        bool ok = true;
        for (long long base = group; ok && base < items; base += static_cast<long long>(META_GROUPS) * META_AHEAD) {
#pragma unroll
            for (int u = 0; u < META_AHEAD; ++u) {
                const long long i = base + static_cast<long long>(META_GROUPS) * u;
                if (!ok || i >= items) break;
                const int stage = static_cast<int>(i % STAGES);
                const uint32_t phase = static_cast<uint32_t>((i / STAGES) & 1);
                int okw = 1;
                if (lane == 0) okw = wait_bar<CG>(empty + stage, phase ^ 1u, w, SITE_META_EMPTY, true);
                okw = __shfl_sync(0xffffffffu, okw, 0);
                if (!okw) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                uint32_t hw[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint32_t other = __shfl_xor_sync(0xffffffffu, ring[u][j], 8);
                    hw[j] = upper ? ((other >> 16) | (ring[u][j] & 0xFFFF0000u)) : ((ring[u][j] & 0xFFFFu) | (other << 16));
                }
                const long long next = i + static_cast<long long>(META_GROUPS) * META_AHEAD;
                if (next < items) load_meta4(p, meta_row<CG>(p, next, first_tile, num_clusters, rank, row_in_tile), static_cast<int>(next % p.num_kb), ring[u]);
                const uint32_t mcol = tmem_base + META_COL + static_cast<uint32_t>(stage) * META_STAGE_COLS +
                                      (static_cast<uint32_t>(quad * 32) << 16);
#pragma unroll
                for (int j = 0; j < 4; ++j) tmem_st_32x32b_x1(mcol + 4 * j, hw[j]);
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if (CG == 2) mbar_arrive_cluster(meta_full_cluster0 + static_cast<uint32_t>(stage) * 8u);
                    else mbar_arrive(meta_full + stage);
                }
            }
        }
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (CG == 2) cluster_sync();
    if (warp == 1) {
        tc_fence_after();
        if (CG == 2) tmem_dealloc_pair(tmem_base, TMEM_COLS);
        else tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

template <int BN, int STAGES, int CG, int NACC>
static cudaError_t launch_sp_one(const CUtensorMap &a, const CUtensorMap &b, const GemmParams &p, int grid,
                                 cudaStream_t stream)
{
    using L = SpSmem<BN / CG, STAGES>;
    auto kern = gemm_sp_kernel<BN, STAGES, CG, NACC>;
    static std::atomic<unsigned long long> smem_limit_set{0};
    cudaError_t e = ensure_max_smem(reinterpret_cast<const void *>(kern), L::ALLOC, smem_limit_set);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(SP_THREADS, 1, 1);
    cfg.dynamicSmemBytes = L::ALLOC;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CG;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, a, b, p);
}

cudaError_t launch_gemm_sp(const GemmConfig &cfg, const CUtensorMap &tmA, const CUtensorMap &tmB,
                           const GemmParams &p, int grid, cudaStream_t stream)
{
    if (cfg.cta_group == 2 && cfg.bn == 256) return launch_sp_one<256, 4, 2, 1>(tmA, tmB, p, grid, stream);
    if (cfg.cta_group == 2 && cfg.bn == 128) return launch_sp_one<128, 6, 2, 2>(tmA, tmB, p, grid, stream);
    if (cfg.cta_group == 1 && cfg.bn == 128) return launch_sp_one<128, 4, 1, 2>(tmA, tmB, p, grid, stream);
    return cudaErrorInvalidValue;
}

} // namespace tcm
