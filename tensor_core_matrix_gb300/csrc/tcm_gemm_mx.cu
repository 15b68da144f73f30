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
// accumulators, tcgen05.ld epilogue), plus two groups of four warps that put
// each stage's scales into tensor memory (each group owns half of the
// stages of the ring).
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

constexpr int MX_GROUPS = 2;
constexpr int MX_THREADS = 32 * (2 + 4 + 4 * MX_GROUPS); // TMA, MMA, 4 epilogue, 2 x 4 scale warps
constexpr uint32_t MX_SCALE_ONE = 0x7F7F7F7Fu;           // four E8M0 codes 127 = 1.0

template <int BN, int STAGES>
struct MxSmem {
    static constexpr int B_STAGE = BN * TILE_K_BYTES;
    static constexpr int A_OFF = 0;
    static constexpr int B_OFF = STAGES * A_STAGE_BYTES;
    static constexpr int BAR_OFF = B_OFF + STAGES * B_STAGE;
    static constexpr int NUM_BARS = 3 * STAGES + 5; // full, empty, sf_full, tfull[2], tempty[2], drain
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

template <int BN, int STAGES, int NACC>
__global__ void __launch_bounds__(MX_THREADS, 1)
    gemm_mx_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, const GemmParams p)
{
    using L = MxSmem<BN, STAGES>;
    static_assert(L::ALLOC <= 227 * 1024, "shared memory ring too large");
    static_assert(BN == 128 || BN == 256, "tile width");
    static_assert(STAGES % MX_GROUPS == 0, "each scale group owns whole stages");
    constexpr int SFB_COLS = BN / 32;
    constexpr uint32_t ACC_STRIDE = BN;                 // BN is a power of two here
    constexpr uint32_t SF_COL = ACC_STRIDE * NACC;      // then 16 scale columns per stage
    constexpr uint32_t SF_STAGE_COLS = 16;              // A at +0..3, B at +8..8+SFB_COLS-1
    static_assert(SF_COL + SF_STAGE_COLS * STAGES <= 512, "tensor memory budget");
    constexpr uint32_t TMEM_COLS = 512;
    constexpr uint32_t STAGE_TX = A_STAGE_BYTES + L::B_STAGE;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    const uint32_t sbase = smem_u32(smem);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L::BAR_OFF);
    uint64_t *empty = full + STAGES;
    uint64_t *sf_full = empty + STAGES;
    uint64_t *tfull = sf_full + STAGES;
    uint64_t *tempty = tfull + 2;
    uint64_t *drain = tempty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::MISC_OFF);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::MISC_OFF + 4);

    const int warp = __shfl_sync(0xffffffffu, static_cast<int>(threadIdx.x >> 5), 0);
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, 1);
            mbar_init(sf_full + s, 4);
        }
        for (int a = 0; a < NACC; ++a) {
            mbar_init(tfull + a, 1);
            mbar_init(tempty + a, EPI_WARPS);
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
        tmem_alloc(tmem_slot, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    const Waiter w{abort_flag, p.timeout_ns, p.status};
    const int first_tile = p.tile_begin + static_cast<int>(blockIdx.x);
    const int step = static_cast<int>(gridDim.x);

    if (warp == 0) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            long long issued = 0;
            bool ok = true;
            for (int t = first_tile; ok && t < p.tile_end; t += step) {
                int mb, nb;
                tile_coords(p, t, mb, nb);
                for (int kb = 0; kb < p.num_kb; ++kb) {
                    if (!wait_bar<1>(empty + stage, phase ^ 1u, w, SITE_LOAD_EMPTY, true)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(full + stage, STAGE_TX);
                    tma_load_2d(sbase + L::A_OFF + stage * A_STAGE_BYTES, &tmA, full + stage, kb * 128, mb * BM);
                    tma_load_2d(sbase + L::B_OFF + stage * L::B_STAGE, &tmB, full + stage, kb * 128, nb * BN);
                    ++issued;
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            for (int s = 0; s < STAGES; ++s) {
                const long long n = issued > s ? (issued - s + STAGES - 1) / STAGES : 0;
                if (n > 0) wait_bar<1>(full + s, static_cast<uint32_t>((n - 1) & 1), w, SITE_DRAIN, false);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            int local = 0;
            for (int t = first_tile; ok && t < p.tile_end; t += step, ++local) {
                const int acc = local % NACC;
                const uint32_t acc_phase = (local / NACC) & 1;
                if (!wait_bar<1>(tempty + acc, acc_phase ^ 1u, w, SITE_MMA_ACC_EMPTY, true)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc) * ACC_STRIDE;
                for (int kb = 0; kb < p.num_kb; ++kb) {
                    if (!wait_bar<1>(full + stage, phase, w, SITE_MMA_FULL, true) ||
                        !wait_bar<1>(sf_full + stage, phase, w, SITE_MMA_META, true)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t ad = sdesc_kmajor_sw128(sbase + L::A_OFF + stage * A_STAGE_BYTES);
                    const uint64_t bd = sdesc_kmajor_sw128(sbase + L::B_OFF + stage * L::B_STAGE);
                    const uint32_t sf = tmem_base + SF_COL + static_cast<uint32_t>(stage) * SF_STAGE_COLS;
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        // scale-factor ids: byte k of the stage's scale words (A bits [29,31), B bits [4,6))
                        const uint32_t idesc = p.idesc | (static_cast<uint32_t>(k) << 29) | (static_cast<uint32_t>(k) << 4);
                        mma_mx(d_tmem, ad + 2 * k, bd + 2 * k, idesc, sf, sf + 8, (kb > 0 || k > 0) ? 1u : 0u);
                    }
                    mma_commit(empty + stage);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                mma_commit(tfull + acc);
            }
            mma_commit(drain);
            wait_bar<1>(drain, 0, w, SITE_DRAIN, false);
        }
    } else if (warp < 2 + EPI_WARPS) {
        const int quad = warp & 3;
        const int row_in_tile = quad * 32 + lane;
        int local = 0;
        for (int t = first_tile; t < p.tile_end; t += step, ++local) {
            const int acc = local % NACC;
            const uint32_t acc_phase = (local / NACC) & 1;
            int ok = 1;
            if (lane == 0) ok = wait_bar<1>(tfull + acc, acc_phase, w, SITE_EPI_ACC_FULL, true);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            tc_fence_after();
            int mb, nb;
            tile_coords(p, t, mb, nb);
            const int row = mb * BM + row_in_tile;
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
                    if (lane == 0) mbar_arrive(tempty + acc);
                }
                epilogue_row32(p, p.alpha, row, nb * BN + c, r);
            }
        }
    } else {
        // Scale warps.  Group g owns stages [g*S/2, (g+1)*S/2) of the S-stage ring
        // and handles, in order, every (tile, K block) item that lands in one of
        // its stages -- so it never skips a use of its stages and its parity
        // waits are never two phases ahead.  Per row it loads 16 bytes at a time:
        // the scales of K blocks 4q .. 4q+3 (one load per row for up to four
        // items), issued before the wait for the item's free stage so the
        // latency overlaps that wait.  Per item it writes word (kb % 4) of each
        // row into the stage's scale columns of its own lane quadrant (every
        // quadrant reads its own copy).
        const int quad = warp & 3;
        const int group = (warp - 2 - EPI_WARPS) / 4;
        constexpr int OWN = STAGES / MX_GROUPS;
        const int s_lo = group * OWN;
        const uint32_t lanebase = static_cast<uint32_t>(quad * 32) << 16;
        const int my_tiles = first_tile < p.tile_end ? (p.tile_end - 1 - first_tile) / step + 1 : 0;
        const long long items = static_cast<long long>(my_tiles) * p.num_kb;
        long long cached = -1;
        uint4 sa[4], sb[SFB_COLS];
        bool ok = true;
        for (long long i = 0; ok && i < items; ++i) {
            const int stage = static_cast<int>(i % STAGES);
            if (stage < s_lo || stage >= s_lo + OWN) continue;
            const int tl = static_cast<int>(i / p.num_kb);
            const int kb = static_cast<int>(i % p.num_kb);
            const long long key = static_cast<long long>(tl) * p.num_kb + (kb & ~3);
            if (key != cached) {
                int mb, nb;
                tile_coords(p, first_tile + tl * step, mb, nb);
#pragma unroll
                for (int c = 0; c < 4; ++c) sa[c] = load_scales16(p.sfa, p.sf_ld, mb * BM + 32 * c + lane, p.kM, kb & ~3);
#pragma unroll
                for (int c = 0; c < SFB_COLS; ++c)
                    sb[c] = load_scales16(p.sfb, p.sf_ld, nb * BN + 32 * c + lane, p.kN, kb & ~3);
                cached = key;
            }
            const uint32_t phase = static_cast<uint32_t>((i / STAGES) & 1);
            int okw = 1;
            if (lane == 0) okw = wait_bar<1>(empty + stage, phase ^ 1u, w, SITE_META_EMPTY, true);
            okw = __shfl_sync(0xffffffffu, okw, 0);
            if (!okw) {
                ok = false;
                break;
            }
            tc_fence_after();
            const int j = kb & 3;
            uint32_t wa[4], wb[SFB_COLS];
#pragma unroll
            for (int c = 0; c < 4; ++c) wa[c] = word_of(sa[c], j);
#pragma unroll
            for (int c = 0; c < SFB_COLS; ++c) wb[c] = word_of(sb[c], j);
            const uint32_t col = tmem_base + SF_COL + static_cast<uint32_t>(stage) * SF_STAGE_COLS + lanebase;
            tmem_st_32x32b_x4(col, wa);
            if constexpr (SFB_COLS == 8) tmem_st_32x32b_x8(col + 8, wb);
            else tmem_st_32x32b_x4(col + 8, wb);
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(sf_full + stage);
        }
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

template <int BN, int STAGES, int NACC>
static cudaError_t launch_mx_one(const CUtensorMap &a, const CUtensorMap &b, const GemmParams &p, int grid,
                                 cudaStream_t stream)
{
    using L = MxSmem<BN, STAGES>;
    auto kern = gemm_mx_kernel<BN, STAGES, NACC>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC);
    if (e != cudaSuccess) return e;
    kern<<<grid, MX_THREADS, L::ALLOC, stream>>>(a, b, p);
    return cudaGetLastError();
}

cudaError_t launch_gemm_mx(const GemmConfig &cfg, const CUtensorMap &tmA, const CUtensorMap &tmB,
                           const GemmParams &p, int grid, cudaStream_t stream)
{
    if (cfg.bn == 256) return launch_mx_one<256, 4, 1>(tmA, tmB, p, grid, stream);
    if (cfg.bn == 128) return launch_mx_one<128, 6, 2>(tmA, tmB, p, grid, stream);
    return cudaErrorInvalidValue;
}

} // namespace tcm
