// tcm_gemm_i8.cu -- exact INT8 x INT8 -> INT32 GEMM (with .satfinite) on the bf16
// tensor path.
//
// "NVIDIA MMA", section "SM100：tcgen05.mma" lists kind::i8 (8-bit integer operands,
// 32-bit integer accumulator); ptxas does not accept it for sm_103a.  Section
// "Ampere：FP16/BF16 与整数 MMA 基线" gives the integer semantics: the exact sum,
// saturated (.satfinite) to the 32-bit range.  This file computes exactly that on
// the kind::f16 tensor path:
//   * every int8 value is exact in bf16 (8 significant bits), and every product of
//     two is an integer of magnitude <= 2^14, exact in fp32;
//   * a sum of at most 1024 such products is an integer of magnitude <= 2^24, so
//     the fp32 accumulator holds every partial sum of a 1024-long K chunk exactly;
//   * the kernel therefore accumulates each chunk of 16 K blocks (1024 K) in a fresh
//     fp32 TMEM accumulator (two alternate, so the MMAs of chunk c+1 run while chunk c
//     is drained), and the epilogue warps convert each drained chunk to int32 and add
//     it into per-thread int32 sums held in registers;
//   * at the end of a tile, + C with a saturating add.
// Sums stay below 2^31 in magnitude while K <= 131071 (16384 * 131071 < 2^31), the
// limit of the entry point; + C then saturates (add.sat.s32: the clamp of the exact
// int32 + int32 sum).
//
// The operands are converted to bf16 first, into a caller workspace (i8_to_bf16_kernel,
// rows of K rounded up to 64 elements, zero-padded): the tensor core reads bf16 from
// shared memory, and converting in shared memory would double the shared-memory traffic
// of a kernel that is already bound by it.
//
// Tiles: 256 x 256 CTA pairs (cta_group::2), the dense kernel's 128-byte-swizzled TMA
// ring and single-thread MMA issue; ten warps: 0 loader, 1 MMA issuer, 2..9 epilogue
// (two per TMEM lane quadrant, 128 columns each, 128 int32 sums per thread).
#include <cuda_bf16.h>

#include "tcm_kernel_common.cuh"

namespace tcm {

constexpr int I8_EPI_WARPS = 8;
constexpr int I8_THREADS = 32 * (2 + I8_EPI_WARPS);
constexpr int I8_CHUNK_KB = 16; // 64-element K blocks per fp32 chunk (1024 K)
constexpr int I8_STAGES = 6;

// a + b clamped to the int32 range (add.sat.s32: exact for any two int32 values)
__device__ __forceinline__ int32_t add_sat(int32_t a, int32_t b)
{
    int32_t r;
    asm("add.sat.s32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// int8 -> bf16 (exact): rows x K values of pitch lds (bytes) into rows of ldo elements,
// zero from K to ldo.  One thread per 8 output elements (one 16-byte store).
__global__ void __launch_bounds__(256) i8_to_bf16_kernel(const int8_t *__restrict__ src, int64_t K, int64_t lds,
                                                         uint4 *__restrict__ dst, int64_t ldo)
{
    const int64_t row = blockIdx.y;
    const int64_t c8 = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (c8 * 8 >= ldo) return;
    const int8_t *s = src + row * lds + c8 * 8;
    uint32_t w[4];
#pragma unroll
    for (int h = 0; h < 4; ++h) {
        const int64_t k = c8 * 8 + 2 * h;
        const float lo = k < K ? static_cast<float>(s[2 * h]) : 0.f;
        const float hi = k + 1 < K ? static_cast<float>(s[2 * h + 1]) : 0.f;
        const __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
        w[h] = *reinterpret_cast<const uint32_t *>(&b);
    }
    dst[(row * ldo) / 8 + c8] = make_uint4(w[0], w[1], w[2], w[3]);
}

__global__ void __launch_bounds__(I8_THREADS, 1)
    gemm_i8_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, const GemmParams p)
{
    constexpr int BN = 256, CG = 2, BN_CTA = BN / CG, STAGES = I8_STAGES;
    using L = Smem<BN_CTA, STAGES>;
    static_assert(L::ALLOC <= 227 * 1024, "shared memory ring too large");
    constexpr uint32_t TMEM_COLS = 512; // two fp32 chunk accumulators of 256 columns
    constexpr uint32_t STAGE_TX = CG * (L::A_STAGE + L::B_STAGE);
    constexpr int EPI_COLS = BN / (I8_EPI_WARPS / 4); // 128 columns per epilogue warp
    const unsigned long long clk0 = clock64();          // clock probe (CTA 0, thread 0 only)
    const unsigned long long gt0 = globaltimer_ns();

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    const uint32_t sbase = smem_u32(smem);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L::BAR_OFF);
    uint64_t *empty = full + STAGES;
    uint64_t *tfull = empty + STAGES;
    uint64_t *tempty = tfull + 2;
    uint64_t *drain = tempty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::MISC_OFF);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::MISC_OFF + 4);

    const int warp = __shfl_sync(0xffffffffu, static_cast<int>(threadIdx.x >> 5), 0);
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull + a, 1);
            mbar_init(tempty + a, I8_EPI_WARPS * CG);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0 && p.num_kb > 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 1) {
        tmem_alloc_pair(tmem_slot, TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    const Waiter w{abort_flag, p.timeout_ns, p.status};
    const int first_tile = p.tile_begin + static_cast<int>(blockIdx.x) / CG;
    const int num_clusters = static_cast<int>(gridDim.x) / CG;

    if (warp == 0) {
        if (lane == 0) {
            const uint32_t full_cluster0 = mapa_shared(smem_u32(full), 0);
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
                    // test hook: the launch's first stage is never loaded (its waits time out)
                    if (!(p.fault_inject & FAULT_SKIP_FIRST_LOAD) || issued != 0) {
                        const uint32_t sa = sbase + L::A_OFF + stage * L::A_STAGE;
                        const uint32_t sb = sbase + L::B_OFF + stage * L::B_STAGE;
                        if (leader) mbar_arrive_expect_tx(full + stage, STAGE_TX);
                        const uint32_t fb = full_cluster0 + static_cast<uint32_t>(stage) * 8u;
                        tma_load_2d_pair(sa, &tmA, fb, kb * 64, a_row);
                        tma_load_2d_pair(sb, &tmB, fb, kb * 64, b_row);
                    }
                    ++issued;
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            // no copy may still be landing when the CTA exits (see the dense kernel)
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
            // chunk g (over all tiles of this pair) accumulates in TMEM columns 256 (g % 2) ..
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            long long g = 0;
            for (int t = first_tile; ok && t < p.tile_end; t += num_clusters) {
                for (int c0 = 0; ok && c0 < p.num_kb; c0 += I8_CHUNK_KB, ++g) {
                    const int acc = static_cast<int>(g & 1);
                    if (!wait_bar<CG>(tempty + acc, static_cast<uint32_t>((g >> 1) & 1) ^ 1u, w, SITE_MMA_ACC_EMPTY,
                                      true)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
                    const int c1 = min(c0 + I8_CHUNK_KB, p.num_kb);
                    for (int kb = c0; kb < c1; ++kb) {
                        if (!wait_bar<CG>(full + stage, phase, w, SITE_MMA_FULL, true)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint64_t ad = sdesc_kmajor_sw128(sbase + L::A_OFF + stage * L::A_STAGE);
                        const uint64_t bd = sdesc_kmajor_sw128(sbase + L::B_OFF + stage * L::B_STAGE);
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            mma_f16_pair(d_tmem, ad + 2 * k, bd + 2 * k, p.idesc, (kb > c0 || k > 0) ? 1u : 0u);
                        mma_commit_pair(empty + stage, 0x3);
                        if (++stage == STAGES) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                    if (!ok) break;
                    mma_commit_pair(tfull + acc, 0x3);
                }
            }
            mma_commit_pair(drain, 0x1);
            wait_bar<CG>(drain, 0, w, SITE_DRAIN, false);
        }
    } else {
        // Epilogue warp: TMEM lane quadrant warp % 4 (tile rows 32q .. 32q + 31), columns
        // c_lo .. c_lo + 127; lane l owns row 32q + l.
        const int quad = warp & 3;
        const int c_lo = ((warp - 2) / 4) * EPI_COLS;
        const int row_in_tile = quad * 32 + lane;
        const uint32_t tempty_cluster0 = mapa_shared(smem_u32(tempty), 0);
        const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
        bool ok = true;
        long long g = 0;
        for (int t = first_tile; ok && t < p.tile_end; t += num_clusters) {
            int32_t sum[EPI_COLS];
#pragma unroll
            for (int j = 0; j < EPI_COLS; ++j) sum[j] = 0;
            for (int c0 = 0; c0 < p.num_kb; c0 += I8_CHUNK_KB, ++g) {
                const int acc = static_cast<int>(g & 1);
                int got = 1;
                if (lane == 0) got = wait_bar<CG>(tfull + acc, static_cast<uint32_t>((g >> 1) & 1), w, SITE_EPI_ACC_FULL, true);
                if (!__shfl_sync(0xffffffffu, got, 0)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t tb = tmem_base + static_cast<uint32_t>(acc * BN + c_lo) + lane_off;
#pragma unroll
                for (int piece = 0; piece < EPI_COLS / 16; ++piece) {
                    uint32_t r[16];
                    tmem_ld_32x32b_x16(tb + static_cast<uint32_t>(piece * 16), r);
                    tmem_ld_wait();
                    // each chunk value is an integer of magnitude <= 2^24: exact in fp32
#pragma unroll
                    for (int j = 0; j < 16; ++j) sum[piece * 16 + j] += __float2int_rn(__uint_as_float(r[j]));
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(tempty_cluster0 + static_cast<uint32_t>(acc) * 8u);
            }
            if (!ok) break;
            int mb, nb;
            tile_coords(p, t, mb, nb);
            const int row = mb * (BM * CG) + static_cast<int>(rank) * BM + row_in_tile;
            if (row >= p.kM) continue;
            int32_t *drow = static_cast<int32_t *>(p.D) + static_cast<long long>(row) * p.ldd;
            const int32_t *crow =
                p.C ? static_cast<const int32_t *>(p.C) + static_cast<long long>(row) * p.ldc : nullptr;
            // + C with saturation (.satfinite), four columns per 16-byte access
            const int col_base = nb * BN + c_lo;
            const bool full_row = col_base + EPI_COLS <= p.kN;
#pragma unroll
            for (int q = 0; q < EPI_COLS / 4; ++q) {
                const int col = col_base + 4 * q;
                if (full_row) {
                    int4 v = make_int4(sum[4 * q], sum[4 * q + 1], sum[4 * q + 2], sum[4 * q + 3]);
                    if (crow) {
                        const int4 c = *reinterpret_cast<const int4 *>(crow + col);
                        v = make_int4(add_sat(v.x, c.x), add_sat(v.y, c.y), add_sat(v.z, c.z), add_sat(v.w, c.w));
                    }
                    *reinterpret_cast<int4 *>(drow + col) = v;
                } else {
#pragma unroll
                    for (int h = 0; h < 4; ++h)
                        if (col + h < p.kN) drow[col + h] = crow ? add_sat(sum[4 * q + h], crow[col + h]) : sum[4 * q + h];
                }
            }
        }
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    cluster_sync();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, TMEM_COLS);
    }
    clock_probe_add(p, clk0, gt0);
}

cudaError_t launch_i8_to_bf16(const int8_t *src, int64_t rows, int64_t K, int64_t lds, void *dst, int64_t ldo,
                              cudaStream_t stream)
{
    if (rows == 0) return cudaSuccess;
    const dim3 grid(static_cast<unsigned>((ldo / 8 + 255) / 256), static_cast<unsigned>(rows), 1);
    i8_to_bf16_kernel<<<grid, 256, 0, stream>>>(src, K, lds, static_cast<uint4 *>(dst), ldo);
    return cudaGetLastError();
}

cudaError_t launch_gemm_i8(const CUtensorMap &tmA, const CUtensorMap &tmB, const GemmParams &p, int grid,
                           cudaStream_t stream)
{
    using L = Smem<128, I8_STAGES>;
    static std::atomic<unsigned long long> smem_limit_set{0};
    cudaError_t e = ensure_max_smem(reinterpret_cast<const void *>(gemm_i8_kernel), L::ALLOC, smem_limit_set);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(I8_THREADS, 1, 1);
    cfg.dynamicSmemBytes = L::ALLOC;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, gemm_i8_kernel, tmA, tmB, p);
}

} // namespace tcm
