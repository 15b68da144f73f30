// tcm_gemm_mx.cu -- block-scaled FP8 GEMM (MXFP8: E4M3/E5M2 elements, one E8M0
// scale per 32 consecutive K elements of every row of A and of B) on
// tcgen05.mma.kind::mxf8f6f4.block_scale.
//
// "NVIDIA MMA", section "SM100：tcgen05.mma": the block-scaled form reads the
// scales of A and B from tensor memory ([scale-A-tmem], [scale-B-tmem]) and
// computes D = C + sum_g (A_{q,g} S_{A,g}) (B_{q,g} S_{B,g}), each K block's
// partial sum scaled before it is accumulated; section "MXFP4 与 NVFP4": MX
// formats carry UE8M0 scales per block of 32.
//
// Pipeline as the dense kernel (TMA ring of 128-byte K stages = 128 FP8
// values, four MMAs of K = 32 per stage, one thread issuing, TMEM
// accumulators, tcgen05.ld epilogue), plus four warps that put the scales
// into tensor memory.  The scales have a ring of their own, decoupled from
// the operand ring: SF_CHUNKS chunks of four K blocks each (16 K blocks of
// look-ahead), filled one chunk per handshake, so the issuing thread waits
// for scales once per four K blocks and normally finds them already there.
//
// Scale layout in tensor memory (established on the GPU by a decoding probe,
// every (row, MMA) traced to its source; 0 mismatches): the scale of operand
// row r for the MMA whose scale-factor id is j is byte j of TMEM column
// (base + r / 32), lane r % 32 of the 32-lane quadrant the output row belongs
// to -- the same 32 x 4-column block is read by all four quadrants, so every
// warp of a group writes its own copy.  One 32-bit word therefore holds the
// four scales of a stage (ids 0..3 = its four MMAs), which is exactly the
// library layout's 4 consecutive bytes of a row (scales are row-major,
// K/32 per row).
#include "tcm_kernel_common.cuh"

namespace tcm {

constexpr int MX_THREADS = 32 * (2 + 4 + 4);     // TMA, MMA, 4 epilogue, 4 scale warps
constexpr uint32_t MX_SCALE_ONE = 0x7F7F7F7Fu;   // four E8M0 codes 127 = 1.0
constexpr int SF_CHUNKS = 4;                     // scale ring: chunks of four K blocks
constexpr uint32_t SF_KB_COLS = 16;              // per K block: A at +0..3, B at +8..15
constexpr uint32_t SF_CHUNK_COLS = 4 * SF_KB_COLS;
constexpr uint32_t SF_RING_COLS = SF_CHUNKS * SF_CHUNK_COLS; // 256

template <int BN, int STAGES>
struct MxSmem {
    static constexpr int B_STAGE = BN * TILE_K_BYTES;
    static constexpr int A_OFF = 0;
    static constexpr int B_OFF = STAGES * A_STAGE_BYTES;
    static constexpr int BAR_OFF = B_OFF + STAGES * B_STAGE;
    // full, empty, sf_full, sf_empty, tfull[2], tempty[2], drain
    static constexpr int NUM_BARS = 2 * STAGES + 2 * SF_CHUNKS + 5;
    static constexpr int MISC_OFF = BAR_OFF + NUM_BARS * 8;
    static constexpr int BYTES = MISC_OFF + 16;
    static constexpr int ALLOC = BYTES + 1024;
};

__device__ __forceinline__ void mma_mx(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                       uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate)
{
    asm volatile(
        "{\n"
        ".reg .pred p;\n"
        "setp.ne.b32 p, %6, 0;\n"
        "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale [%0], %1, %2, %3, [%4], [%5], p;\n"
        "}\n" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_mx_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                            uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate)
{
    asm volatile(
        "{\n"
        ".reg .pred p;\n"
        "setp.ne.b32 p, %6, 0;\n"
        "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale [%0], %1, %2, %3, [%4], [%5], p;\n"
        "}\n" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

// The sixteen scale codes of row `row` (of `rows` rows) for K blocks
// [kb0, kb0 + 4) of 128 values each, as four words (word j = K block kb0 + j,
// byte i of it = the i-th 32-element block).  Missing rows and blocks read 1.0.
__device__ __forceinline__ uint4 load_scales16(const uint8_t *scales, long long ld, int row, int rows, int kb0)
{
    uint4 v = make_uint4(MX_SCALE_ONE, MX_SCALE_ONE, MX_SCALE_ONE, MX_SCALE_ONE);
    if (row >= rows) return v;
    const long long first = static_cast<long long>(kb0) * 4;
    const uint8_t *src = scales + static_cast<long long>(row) * ld + first;
    if (first + 16 <= ld && (reinterpret_cast<uintptr_t>(src) & 15u) == 0) return __ldg(reinterpret_cast<const uint4 *>(src));
    uint32_t w[4] = {MX_SCALE_ONE, MX_SCALE_ONE, MX_SCALE_ONE, MX_SCALE_ONE};
#pragma unroll
    for (int b = 0; b < 16; ++b)
        if (first + b < ld) w[b / 4] = (w[b / 4] & ~(0xFFu << (8 * (b % 4)))) | (static_cast<uint32_t>(__ldg(src + b)) << (8 * (b % 4)));
    return make_uint4(w[0], w[1], w[2], w[3]);
}

__device__ __forceinline__ uint32_t word_of(const uint4 &v, int j)
{
    return j == 0 ? v.x : (j == 1 ? v.y : (j == 2 ? v.z : v.w));
}

// BN: N extent of the (pair) tile; CG: 1 = one CTA per 128 x BN tile, 2 = a CTA
// pair per 256 x BN tile (each CTA loads 128 rows of A and BN/2 rows of B).
template <int BN, int STAGES, int NACC, int CG>
__global__ void __launch_bounds__(MX_THREADS, 1)
    gemm_mx_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, const GemmParams p)
{
    constexpr int BN_CTA = BN / CG;
    using L = MxSmem<BN_CTA, STAGES>;
    static_assert(L::ALLOC <= 227 * 1024, "shared memory ring too large");
    static_assert(BN == 128 || BN == 256, "tile width");
    constexpr int SFB_COLS = BN / 32;
    constexpr uint32_t ACC_STRIDE = BN;                 // BN is a power of two here
    constexpr uint32_t SF_COL = ACC_STRIDE * NACC;      // then the scale ring
    static_assert(SF_COL + SF_RING_COLS <= 512, "tensor memory budget");
    constexpr uint32_t TMEM_COLS = 512;
    constexpr uint32_t STAGE_TX = CG * (A_STAGE_BYTES + L::B_STAGE);

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    const uint32_t sbase = smem_u32(smem);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L::BAR_OFF);
    uint64_t *empty = full + STAGES;
    uint64_t *sf_full = empty + STAGES;
    uint64_t *sf_empty = sf_full + SF_CHUNKS;
    uint64_t *tfull = sf_empty + SF_CHUNKS;
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
        }
        for (int c = 0; c < SF_CHUNKS; ++c) {
            mbar_init(sf_full + c, 4 * CG);
            mbar_init(sf_empty + c, 1);
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
    const int first_tile = p.tile_begin + static_cast<int>(blockIdx.x) / CG;
    const int step = static_cast<int>(gridDim.x) / CG;

    if (warp == 0) {
        if (lane == 0) {
            const uint32_t full_cluster0 = CG == 2 ? mapa_shared(smem_u32(full), 0) : 0u;
            int stage = 0;
            uint32_t phase = 0;
            long long issued = 0;
            bool ok = true;
            for (int t = first_tile; ok && t < p.tile_end; t += step) {
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
                    if (CG == 2) {
                        if (leader) mbar_arrive_expect_tx(full + stage, STAGE_TX);
                        const uint32_t fb = full_cluster0 + static_cast<uint32_t>(stage) * 8u;
                        tma_load_2d_pair(sa, &tmA, fb, kb * 128, a_row);
                        tma_load_2d_pair(sb, &tmB, fb, kb * 128, b_row);
                    } else {
                        mbar_arrive_expect_tx(full + stage, STAGE_TX);
                        tma_load_2d(sa, &tmA, full + stage, kb * 128, a_row);
                        tma_load_2d(sb, &tmB, full + stage, kb * 128, b_row);
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
            int chunk = 0;
            uint32_t chunk_phase = 0;
            bool ok = true;
            int local = 0;
            for (int t = first_tile; ok && t < p.tile_end; t += step, ++local) {
                const int acc = local % NACC;
                const uint32_t acc_phase = (local / NACC) & 1;
                if (!wait_bar<CG>(tempty + acc, acc_phase ^ 1u, w, SITE_MMA_ACC_EMPTY, true)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc) * ACC_STRIDE;
                for (int kb = 0; kb < p.num_kb; ++kb) {
                    if (((kb & 3) == 0 && !wait_bar<CG>(sf_full + chunk, chunk_phase, w, SITE_MMA_META, true)) ||
                        !wait_bar<CG>(full + stage, phase, w, SITE_MMA_FULL, true)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t ad = sdesc_kmajor_sw128(sbase + L::A_OFF + stage * A_STAGE_BYTES);
                    const uint64_t bd = sdesc_kmajor_sw128(sbase + L::B_OFF + stage * L::B_STAGE);
                    const uint32_t sf = tmem_base + SF_COL + static_cast<uint32_t>(chunk) * SF_CHUNK_COLS +
                                        static_cast<uint32_t>(kb & 3) * SF_KB_COLS;
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        // scale-factor ids: byte k of the stage's scale words (A bits [29,31), B bits [4,6))
                        const uint32_t idesc = p.idesc | (static_cast<uint32_t>(k) << 29) | (static_cast<uint32_t>(k) << 4);
                        const uint32_t accum = (kb > 0 || k > 0) ? 1u : 0u;
                        if (CG == 2) mma_mx_pair(d_tmem, ad + 2 * k, bd + 2 * k, idesc, sf, sf + 8, accum);
                        else mma_mx(d_tmem, ad + 2 * k, bd + 2 * k, idesc, sf, sf + 8, accum);
                    }
                    if (CG == 2) mma_commit_pair(empty + stage, 0x3);
                    else mma_commit(empty + stage);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                    if ((kb & 3) == 3 || kb + 1 == p.num_kb) {
                        if (CG == 2) mma_commit_pair(sf_empty + chunk, 0x3);
                        else mma_commit(sf_empty + chunk);
                        if (++chunk == SF_CHUNKS) {
                            chunk = 0;
                            chunk_phase ^= 1u;
                        }
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
        const uint32_t tempty_cluster0 = CG == 2 ? mapa_shared(smem_u32(tempty), 0) : 0u;
        int local = 0;
        for (int t = first_tile; t < p.tile_end; t += step, ++local) {
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
                epilogue_row32(p, p.alpha, row, nb * BN + c, r);
            }
        }
    } else {
        // Scale warps, one per TMEM lane quadrant (each quadrant reads its own
        // copy).  Chunk q of this CTA's sequence -- K blocks [4j, 4j + 4) of one
        // tile -- goes to ring slot q % SF_CHUNKS.  Per row one 16-byte load
        // holds the scales of all four K blocks; the loads of the next chunk are
        // issued before the wait for its slot, so their latency overlaps it.
        // Per K block of the chunk the warp writes word (kb % 4) of each row:
        // A rows into columns +0..3, B rows into +8..8 + BN/32 - 1.
        const int quad = warp & 3;
        const uint32_t lanebase = static_cast<uint32_t>(quad * 32) << 16;
        const uint32_t sf_full_cluster0 = CG == 2 ? mapa_shared(smem_u32(sf_full), 0) : 0u;
        const int a_row0 = static_cast<int>(rank) * BM + lane;
        uint4 sa[4], sb[SFB_COLS];
        int chunk = 0;
        uint32_t chunk_phase = 0;
        long long used = 0;
        bool ok = true;
        for (int t = first_tile; ok && t < p.tile_end; t += step) {
            int mb, nb;
            tile_coords(p, t, mb, nb);
            for (int kb0 = 0; kb0 < p.num_kb; kb0 += 4) {
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    sa[c] = load_scales16(p.sfa, p.sf_ld, mb * (BM * CG) + a_row0 + 32 * c, p.kM, kb0);
#pragma unroll
                for (int c = 0; c < SFB_COLS; ++c)
                    sb[c] = load_scales16(p.sfb, p.sf_ld, nb * BN + 32 * c + lane, p.kN, kb0);
                int okw = 1;
                if (lane == 0) okw = wait_bar<CG>(sf_empty + chunk, chunk_phase ^ 1u, w, SITE_META_EMPTY, true);
                okw = __shfl_sync(0xffffffffu, okw, 0);
                if (!okw) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t col = tmem_base + SF_COL + static_cast<uint32_t>(chunk) * SF_CHUNK_COLS + lanebase;
                const int nk = min(4, p.num_kb - kb0);
                for (int j = 0; j < nk; ++j) {
                    uint32_t wa[4], wb[SFB_COLS];
#pragma unroll
                    for (int c = 0; c < 4; ++c) wa[c] = word_of(sa[c], j);
#pragma unroll
                    for (int c = 0; c < SFB_COLS; ++c) wb[c] = word_of(sb[c], j);
                    const uint32_t cj = col + static_cast<uint32_t>(j) * SF_KB_COLS;
                    tmem_st_32x32b_x4(cj, wa);
                    if constexpr (SFB_COLS == 8) tmem_st_32x32b_x8(cj + 8, wb);
                    else tmem_st_32x32b_x4(cj + 8, wb);
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if (CG == 2) mbar_arrive_cluster(sf_full_cluster0 + static_cast<uint32_t>(chunk) * 8u);
                    else mbar_arrive(sf_full + chunk);
                }
                ++used;
                if (++chunk == SF_CHUNKS) {
                    chunk = 0;
                    chunk_phase ^= 1u;
                }
            }
        }
        // Wait for the MMA's release of every slot used, so that no commit is
        // still in flight towards this CTA's barriers when it exits.
        if (lane == 0 && ok) {
            for (int c = 0; c < SF_CHUNKS; ++c) {
                const long long n = used > c ? (used - c + SF_CHUNKS - 1) / SF_CHUNKS : 0;
                if (n > 0) wait_bar<CG>(sf_empty + c, static_cast<uint32_t>((n - 1) & 1), w, SITE_DRAIN, false);
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

template <int BN, int STAGES, int NACC, int CG>
static cudaError_t launch_mx_one(const CUtensorMap &a, const CUtensorMap &b, const GemmParams &p, int grid,
                                 cudaStream_t stream)
{
    using L = MxSmem<BN / CG, STAGES>;
    auto kern = gemm_mx_kernel<BN, STAGES, NACC, CG>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(MX_THREADS, 1, 1);
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

cudaError_t launch_gemm_mx(const GemmConfig &cfg, const CUtensorMap &tmA, const CUtensorMap &tmB,
                           const GemmParams &p, int grid, cudaStream_t stream)
{
    if (cfg.cta_group == 2) return cfg.bn == 256 ? launch_mx_one<256, 6, 1, 2>(tmA, tmB, p, grid, stream)
                                                 : cudaErrorInvalidValue;
    if (cfg.bn == 256) return launch_mx_one<256, 4, 1, 1>(tmA, tmB, p, grid, stream);
    if (cfg.bn == 128) return launch_mx_one<128, 6, 2, 1>(tmA, tmB, p, grid, stream);
    return cudaErrorInvalidValue;
}

} // namespace tcm
