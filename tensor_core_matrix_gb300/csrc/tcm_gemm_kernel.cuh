// tcm_gemm_kernel.cuh -- the persistent tcgen05 GEMM kernel for sm_103a
// (template; instantiated by tcm_gemm.cu, tcm_gemm_pair.cu, tcm_gemm_ksplit.cu).
//
// Computes, per output tile, D = alpha*sA*sB * sum_k A[m,k] B[n,k] + beta*C + bias
// ("NVIDIA MMA", sections "从 FMA 到 MMA，再到 GEMM" and "输入/累加/输出"):
// GEMM = many MMAs + data movement + a K loop + an epilogue.
//
// One CTA per SM (persistent), 192 threads in three roles:
//   warp 0        loader: one thread issues TMA copies of the A tile
//                 (128 x 128 bytes of K) and the B tile (BN x 128 bytes)
//                 into a STAGES-deep ring of 128-byte-swizzled shared
//                 memory, gated by full/empty mbarriers (the producer /
//                 consumer queue of "Tensor Core 三种调用层次", section 6).
//   warp 1        MMA issuer: allocates tensor memory, and one thread issues
//                 four tcgen05.mma per stage (32 bytes of K each: K=16 for
//                 f16/bf16, K=32 for E4M3/E5M2), accumulating fp32 in TMEM;
//                 tcgen05.commit frees the stage and, at the end of a tile,
//                 hands the accumulator to the epilogue ("NVIDIA MMA",
//                 section "SM100：tcgen05.mma").
//   warps 2..5    epilogue: tcgen05.ld of the accumulator (warp w reads TMEM
//                 lanes 32*(w%4)..+31, one output row per thread), scale,
//                 + beta*C, + bias, round-to-nearest cast, vector stores.
// Two TMEM accumulators (2*BN columns) let the epilogue of one tile overlap
// the main loop of the next.  Tiles are assigned statically: CTA b takes
// tiles b, b+grid, b+2*grid ... in a grouped order so that tiles running at
// the same time share rows of A and columns of B in L2.
//
// Every mbarrier wait is bounded by a global-timer limit; on expiry the
// waiting thread records {TIMEOUT, site} in the device status words, raises
// a CTA-wide abort flag that the other roles poll, and all roles wind down:
// the loader waits (bounded) for its in-flight copies, the issuer for its
// in-flight MMAs, and tensor memory is freed before the CTA exits.
#pragma once

#include "tcm_kernel_common.cuh"

namespace tcm {

// Offset, in a K-split partial-sum buffer, of 16-byte piece j of the 32
// columns starting at c of tile row `row`, for slot `slot` (one slot per
// contributing CTA).  Each thread owns one 128-byte row segment per 32
// columns; its pieces are rotated by (row % 8) to spread shared-memory banks.
template <int BN>
__device__ __forceinline__ uint32_t red_offset(int slot, int row, int c, int j)
{
    return static_cast<uint32_t>(slot * (BM * BN * 4) + row * BN * 4 + c * 4 + ((j ^ (row & 7)) * 16));
}

// Tail K split (two parts): the workspace slot of split tile j for CTA `rank` of the pair,
// the helper part's 128 x BN fp32 partial sums as the byte image of its shared-memory
// staging (red_offset layout, rows bank-swizzled).
template <int CG, int BN>
__device__ __forceinline__ float *part_slot(const GemmParams &p, int j, uint32_t rank)
{
    return p.ws_part + (static_cast<size_t>(j) * CG + rank) * (BM * BN);
}

// KIND: 0 = kind::f16, 1 = kind::f8f6f4.  BN: N extent of the (pair) tile.
// CG: 1 = one CTA computes a 128 x BN tile; 2 = a cluster of two CTAs
// computes a 256 x BN tile with cta_group::2 (each CTA loads its own 128
// rows of A and BN/2 rows of B, the even CTA issues the MMAs).
// KS: with CG = 1, a cluster of KS CTAs shares each tile: CTA r accumulates
// the K blocks [num_kb*r/KS, num_kb*(r+1)/KS) in its own TMEM; CTAs 1..KS-1
// push their fp32 partial accumulators into CTA 0's shared memory (DSMEM),
// and CTA 0 adds them in rank order (a fixed order, so results do not depend
// on timing) before the epilogue.  This keeps every SM streaming when a
// problem has fewer tiles than the GPU has SMs (skinny M after the swap).
// KATOMS: 128-byte K atoms per stage.  Single-CTA tiles of width 32 use two (each weight
// row a longer contiguous run per stage: skinny, HBM-bound shapes); CTA pairs with 8-bit
// operands use two (eight MMAs per barrier wait and commit, same ring bytes).
// Work units (unit_coords): whole tiles, and -- when p.split == 2 -- the two K halves
// of each tile of the last, partly filled round (CTA pairs only).  That round is each
// CTA's last unit, so its shared-memory ring is idle by then: the helper half stages its
// fp32 accumulator there (128 x BN per CTA), bulk-copies the image to its workspace slot
// and release-adds 1 to the slot's counter; the owner half waits (bounded) for the
// counter, bulk-copies the image into its own ring and adds it before its epilogue.
// Such launches are cooperative, so every pair is resident and the waits end.
// (Register loads of the partials, chunk by chunk, cost the owner ~15 us of L2
// latency at 4096^3; one bulk copy each way does not.)
template <int KIND, int BN, int STAGES, int CG, int KS, int KATOMS = 1>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, const GemmParams p)
{
    const unsigned long long clk0 = clock64(); // clock probe (CTA 0, thread 0 only)
    const unsigned long long gt0 = globaltimer_ns();
    constexpr int RED_SLOT = BM * BN * 4; // one CTA's fp32 partial tile
    using L = Smem<BN / CG, STAGES, (KS - 1) * RED_SLOT, KATOMS>;
    static_assert(CG == 1 || CG == 2, "CTA group of 1 or 2");
    static_assert(KS == 1 || (CG == 1 && (KS == 2 || KS == 4)), "K split of 2 or 4 CTAs, single-CTA tiles only");
    static_assert(BN % 32 == 0 && BN >= 32 && BN <= 256, "BN must be a multiple of 32 in [32, 256]");
    static_assert(L::ALLOC <= 227 * 1024, "shared memory ring too large");
    constexpr uint32_t TMEM_COLS = 2 * BN < 32 ? 32 : 2 * BN;
    constexpr int KB_ELEMS = KIND == 1 ? 128 : 64; // K elements per stage (128 bytes)
    constexpr int BN_CTA = BN / CG;                  // rows of B this CTA loads
    constexpr uint32_t STAGE_TX = CG * (L::A_STAGE + L::B_STAGE);
    // packed FP4 operands land as 128 bytes per row but count 64 (the packed bytes)
    const uint32_t stage_tx = p.stage_tx ? p.stage_tx : STAGE_TX;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    const uint32_t sbase = smem_u32(smem);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L::BAR_OFF);
    uint64_t *empty = full + STAGES;
    uint64_t *tfull = empty + STAGES;
    uint64_t *tempty = tfull + 2;
    uint64_t *drain = tempty + 2;
    uint64_t *red_full = drain + 1;
    uint64_t *red_empty = drain + 2;
    uint64_t *part_full = drain + 3;   // tail K split: the helper's partial sums landed in the ring
    uint64_t *part_staged = drain + 4; // tail K split: every epilogue warp staged its rows
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::MISC_OFF);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::MISC_OFF + 4);
    constexpr bool CLUSTERED = CG == 2 || KS > 1;

    const int warp = __shfl_sync(0xffffffffu, static_cast<int>(threadIdx.x >> 5), 0);
    const int lane = threadIdx.x & 31;
    const uint32_t crank = CLUSTERED ? cluster_ctarank() : 0u;
    const uint32_t rank = CG == 2 ? crank : 0u;  // position in a CTA pair
    const int krank = KS > 1 ? static_cast<int>(crank) : 0; // position in a K split
    const bool leader = rank == 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull + a, 1);
            mbar_init(tempty + a, EPI_WARPS * CG);
        }
        mbar_init(drain, 1);
        mbar_init(part_full, 1);
        mbar_init(part_staged, EPI_WARPS);
        if constexpr (KS > 1) {
            mbar_init(red_full, (KS - 1) * EPI_WARPS);
            mbar_init(red_empty, EPI_WARPS);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0 && p.num_kb > 0) { // K == 0: the maps are not encoded
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
    if (CLUSTERED) cluster_sync();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    const Waiter w{abort_flag, p.timeout_ns, p.status};
    const int cluster_id = static_cast<int>(blockIdx.x) / (CG * KS);
    const int num_clusters = static_cast<int>(gridDim.x) / (CG * KS);
    const int first_tile = p.tile_begin + cluster_id;
    // K-split clusters: this CTA's share of each tile's K blocks (else a unit's own range)
    const int kb0 = static_cast<int>((static_cast<long long>(p.num_kb) * krank) / KS);
    const int kb1 = static_cast<int>((static_cast<long long>(p.num_kb) * (krank + 1)) / KS);

    if (warp == 0) {
        if (lane == 0) {
            // leader's full barrier, addressed through the cluster window when paired
            const uint32_t full_cluster0 = CG == 2 ? mapa_shared(smem_u32(full), 0) : smem_u32(full);
            int stage = 0;
            uint32_t phase = 0;
            long long issued = 0;
            bool ok = true;
            for (int t = first_tile; ok && t < p.tile_end; t += num_clusters) {
                const Unit u = unit_coords(p, t);
                const int ukb0 = KS > 1 ? kb0 : u.kb0, ukb1 = KS > 1 ? kb1 : u.kb1;
                const int a_row = u.mb * (BM * CG) + static_cast<int>(rank) * BM;
                const int b_row = u.nb * BN + static_cast<int>(rank) * BN_CTA;
                for (int kb = ukb0; kb < ukb1; ++kb) {
                    if (!wait_bar<CG>(empty + stage, phase ^ 1u, w, SITE_LOAD_EMPTY, true)) {
                        ok = false;
                        break;
                    }
                    if (!(p.fault_inject & FAULT_SKIP_FIRST_LOAD) || issued != 0) {
                        const uint32_t sa = sbase + L::A_OFF + stage * L::A_STAGE;
                        const uint32_t sb = sbase + L::B_OFF + stage * L::B_STAGE;
                        if (CG == 2) {
                            if (leader) mbar_arrive_expect_tx(full + stage, stage_tx);
                            const uint32_t fb = full_cluster0 + static_cast<uint32_t>(stage) * 8u;
#pragma unroll
                            for (int a = 0; a < KATOMS; ++a) {
                                tma_load_2d_pair(sa + a * A_STAGE_BYTES, &tmA, fb, (kb * KATOMS + a) * KB_ELEMS, a_row);
                                tma_load_2d_pair(sb + a * BN_CTA * TILE_K_BYTES, &tmB, fb, (kb * KATOMS + a) * KB_ELEMS,
                                                 b_row);
                            }
                        } else {
                            mbar_arrive_expect_tx(full + stage, stage_tx);
#pragma unroll
                            for (int a = 0; a < KATOMS; ++a)
                                tma_load_2d(sa + a * A_STAGE_BYTES, &tmA, full + stage, (kb * KATOMS + a) * KB_ELEMS, a_row);
#pragma unroll
                            for (int a = 0; a < KATOMS; ++a)
                                tma_load_2d(sb + a * BN_CTA * TILE_K_BYTES, &tmB, full + stage,
                                            (kb * KATOMS + a) * KB_ELEMS, b_row);
                        }
                    }
                    ++issued;
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            // No copy may still be landing in shared memory when the CTA exits.
            // The CTA that owns the full barriers waits for the last phase of
            // each stage's full barrier (all its bytes landed); the odd CTA of a
            // pair, whose copies complete on the even CTA's barriers, waits until
            // the MMA has released the last use of every stage instead.
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
                const int acc = local & 1;
                const uint32_t acc_phase = (local >> 1) & 1;
                const uint32_t idesc = p.idesc;
                const Unit u = unit_coords(p, t);
                const int ukb0 = KS > 1 ? kb0 : u.kb0, ukb1 = KS > 1 ? kb1 : u.kb1;
                if (!wait_bar<CG>(tempty + acc, acc_phase ^ 1u, w, SITE_MMA_ACC_EMPTY, true)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
                for (int kb = ukb0; kb < ukb1; ++kb) {
                    if (!wait_bar<CG>(full + stage, phase, w, SITE_MMA_FULL, true)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int a = 0; a < KATOMS; ++a) {
                        const uint64_t ad =
                            sdesc_kmajor_sw128(sbase + L::A_OFF + stage * L::A_STAGE + a * A_STAGE_BYTES);
                        const uint64_t bd =
                            sdesc_kmajor_sw128(sbase + L::B_OFF + stage * L::B_STAGE + a * BN_CTA * TILE_K_BYTES);
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            // +32 bytes of K per instruction = +2 in the descriptor's address field
                            const uint32_t accum = (kb > ukb0 || a > 0 || k > 0) ? 1u : 0u;
                            if (CG == 2) {
                                if (KIND == 1) mma_f8_pair(d_tmem, ad + 2 * k, bd + 2 * k, idesc, accum);
                                else mma_f16_pair(d_tmem, ad + 2 * k, bd + 2 * k, idesc, accum);
                            } else {
                                if (KIND == 1) mma_f8(d_tmem, ad + 2 * k, bd + 2 * k, idesc, accum);
                                else mma_f16(d_tmem, ad + 2 * k, bd + 2 * k, idesc, accum);
                            }
                        }
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
            // Every MMA issued by this thread completes before tensor memory is freed.
            if (CG == 2) mma_commit_pair(drain, 0x1);
            else mma_commit(drain);
            wait_bar<CG>(drain, 0, w, SITE_DRAIN, false);
        }
    } else {
        const int quad = warp & 3; // TMEM lanes 32*quad .. 32*quad+31
        const int row_in_tile = quad * 32 + lane;
        const float scale = p.alpha * (p.a_scale ? *p.a_scale : 1.f) * (p.b_scale ? *p.b_scale : 1.f);
        // the issuer's "accumulator free" barrier lives in the even CTA
        const uint32_t tempty_cluster0 = CG == 2 ? mapa_shared(smem_u32(tempty), 0) : 0u;
        // K split: partial sums of CTA r go to slot r-1 of CTA 0's buffer (red_offset)
        uint32_t red_cluster0 = 0u, red_full_cluster0 = 0u;
        if constexpr (KS > 1) {
            red_cluster0 = mapa_shared(sbase + L::RED_OFF, 0);
            red_full_cluster0 = mapa_shared(smem_u32(red_full), 0);
        }

        if (p.prefetch_c && (KS == 1 || krank == 0) && first_tile < p.tile_end) {
            // one unit per CTA: pull this lane's C row segment into L2 while the MMAs run
            const Unit u = unit_coords(p, first_tile);
            const int row = u.mb * (BM * CG) + static_cast<int>(rank) * BM + row_in_tile;
            const int col0 = u.nb * BN;
            if (u.part == 0 && row < p.kM && col0 < p.kN) {
                const int es = p.out_fmt == OUT_F32 ? 4 : (p.out_fmt == OUT_BF16 || p.out_fmt == OUT_F16) ? 2 : 1;
                const int bytes = min(BN, p.kN - col0) * es;
                const char *c = static_cast<const char *>(p.C) + (static_cast<long long>(row) * p.ldc + col0) * es;
                for (int off = 0; off < bytes; off += 128) prefetch_l2(c + off);
                prefetch_l2(c + bytes - 1);
            }
        }
        int local = 0;
        float amax_local = 0.f; // max |y| of this lane's outputs (when p.amax is set)
        for (int t = first_tile; t < p.tile_end; t += num_clusters, ++local) {
            const int acc = local & 1;
            const uint32_t acc_phase = (local >> 1) & 1;
            int ok = 1;
            if (lane == 0) ok = wait_bar<CG>(tfull + acc, acc_phase, w, SITE_EPI_ACC_FULL, true);
            if constexpr (KS > 1) {
                if (lane == 0 && ok) {
                    // others: the leader has consumed the previous tile's partials; leader: all partials are in
                    if (krank > 0) ok = bounded_wait<CG, true>(red_empty, (local & 1) ^ 1u, w, SITE_RED_EMPTY, true);
                    else ok = bounded_wait<CG, true>(red_full, local & 1, w, SITE_RED_FULL, true);
                }
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            tc_fence_after();
            const Unit u = unit_coords(p, t);
            const bool has_acc = KS > 1 ? kb1 > kb0 : u.kb1 > u.kb0;
            const int row = u.mb * (BM * CG) + static_cast<int>(rank) * BM + row_in_tile;
            const uint32_t tbase = tmem_base + static_cast<uint32_t>(acc * BN) + (static_cast<uint32_t>(quad * 32) << 16);
            const bool helper = CG == 2 && u.part > 0;
            const bool owner = CG == 2 && u.j >= 0 && u.part == 0;
            constexpr uint32_t PART_BYTES = BM * BN * 4;
            constexpr uint32_t PART_PIECE = 16384;
            static_assert(CG == 1 || PART_BYTES <= STAGES * (L::A_STAGE + L::B_STAGE), "partial sums fit the ring");
            bool add_parts = false;
            if (owner) {
                int got = 1;
                if (warp == 2 && lane == 0) {
                    // the helper CTA's image is in the workspace: bring it into this CTA's ring
                    got = wait_count(p.ws_flag + u.j * CG + static_cast<int>(rank), 1, w, SITE_PART_WAIT);
                    if (got) {
                        fence_proxy_async_global();
                        mbar_arrive_expect_tx(part_full, PART_BYTES);
                        const uint8_t *src = reinterpret_cast<const uint8_t *>(part_slot<CG, BN>(p, u.j, rank));
                        for (uint32_t q = 0; q < PART_BYTES; q += PART_PIECE)
                            bulk_load_g2s(sbase + q, src + q, PART_PIECE, smem_u32(part_full));
                    }
                }
                if (lane == 0 && got) got = wait_bar<CG>(part_full, 0, w, SITE_PART_WAIT, true);
                add_parts = __shfl_sync(0xffffffffu, got, 0) != 0;
            }
#pragma unroll 1
            for (int c = 0; c < BN; c += 32) {
                uint32_t r[32];
                if (has_acc) {
                    tmem_ld_32x32b_x32(tbase + c, r);
                    tmem_ld_wait();
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j) r[j] = 0u;
                }
                if (c + 32 >= BN) {
                    // last chunk read: hand the accumulator back to the issuer before storing
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        if (CG == 2) mbar_arrive_cluster(tempty_cluster0 + static_cast<uint32_t>(acc) * 8u);
                        else mbar_arrive(tempty + acc);
                    }
                }
                if constexpr (KS > 1) {
                    if (krank > 0) {
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            st_cluster_v4(red_cluster0 + red_offset<BN>(krank - 1, row_in_tile, c, j), r[4 * j],
                                          r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]);
                        continue;
                    }
                    float sum[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) sum[j] = __uint_as_float(r[j]);
#pragma unroll 1
                    for (int slot = 0; slot < KS - 1; ++slot) {
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const float4 v =
                                *reinterpret_cast<const float4 *>(smem + L::RED_OFF + red_offset<BN>(slot, row_in_tile, c, j));
                            sum[4 * j] += v.x, sum[4 * j + 1] += v.y, sum[4 * j + 2] += v.z, sum[4 * j + 3] += v.w;
                        }
                    }
#pragma unroll
                    for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(sum[j]);
                }
                if (helper) {
                    // stage the partial sums in the idle ring, rows bank-swizzled
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        *reinterpret_cast<uint4 *>(smem + red_offset<BN>(0, row_in_tile, c, j)) =
                            make_uint4(r[4 * j], r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]);
                    continue;
                }
                if (add_parts) {
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const float4 v = *reinterpret_cast<const float4 *>(smem + red_offset<BN>(0, row_in_tile, c, j));
                        r[4 * j] = __float_as_uint(__uint_as_float(r[4 * j]) + v.x);
                        r[4 * j + 1] = __float_as_uint(__uint_as_float(r[4 * j + 1]) + v.y);
                        r[4 * j + 2] = __float_as_uint(__uint_as_float(r[4 * j + 2]) + v.z);
                        r[4 * j + 3] = __float_as_uint(__uint_as_float(r[4 * j + 3]) + v.w);
                    }
                }
                const float m = epilogue_row32(p, scale, row, u.nb * BN + c, r);
                if (p.amax) amax_local = amax_combine(amax_local, m);
            }
            if (helper) {
                // publish: the staged image to the workspace in one bulk copy, then the counter
                // (every wait here is bounded: the first epilogue warp waits for the others)
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(part_staged);
                if (warp == 2 && lane == 0 && wait_bar<CG>(part_staged, 0, w, SITE_PART_WAIT, true)) {
                    uint8_t *dst = reinterpret_cast<uint8_t *>(part_slot<CG, BN>(p, u.j, rank));
                    for (uint32_t q = 0; q < PART_BYTES; q += PART_PIECE) bulk_store_s2g(dst + q, sbase + q, PART_PIECE);
                    bulk_commit_wait_all();
                    fence_proxy_async_global();
                    if (!(p.fault_inject & FAULT_SKIP_PUBLISH))
                        red_release_gpu_add(p.ws_flag + u.j * CG + static_cast<int>(rank), 1);
                }
            }
            if constexpr (KS > 1) {
                __syncwarp();
                if (lane == 0) {
                    if (krank > 0) {
                        mbar_arrive_cluster_release(red_full_cluster0); // partials of this tile are in CTA 0
                    } else {
                        // the buffer may be refilled: one arrival per other CTA
                        for (int q = 1; q < KS; ++q)
                            mbar_arrive_cluster_release(mapa_shared(smem_u32(red_empty), static_cast<uint32_t>(q)));
                    }
                }
            }
        }
        if (p.amax) amax_flush(p.amax, amax_local);
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (CLUSTERED) cluster_sync(); // peers' shared memory and TMEM stay alive until the cluster is done
    if (warp == 1) {
        tc_fence_after();
        if (CG == 2) tmem_dealloc_pair(tmem_base, TMEM_COLS);
        else tmem_dealloc(tmem_base, TMEM_COLS);
    }
    clock_probe_add(p, clk0, gt0);
}

template <int KIND, int BN, int STAGES, int CG, int KS = 1, int KATOMS = 1>
inline cudaError_t launch_one(const CUtensorMap &a, const CUtensorMap &b, const GemmParams &p, int grid,
                              cudaStream_t stream)
{
    using L = Smem<BN / CG, STAGES, (KS - 1) * BM * BN * 4, KATOMS>;
    auto kern = gemm_kernel<KIND, BN, STAGES, CG, KS, KATOMS>;
    static std::atomic<unsigned long long> smem_limit_set{0};
    cudaError_t e = ensure_max_smem(reinterpret_cast<const void *>(kern), L::ALLOC, smem_limit_set);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(NUM_THREADS, 1, 1);
    cfg.dynamicSmemBytes = L::ALLOC;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CG * KS;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    // owners of split tiles wait for helper pairs: all CTAs must be resident at once
    attr[1].id = cudaLaunchAttributeCooperative;
    attr[1].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = p.split > 1 ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, kern, a, b, p);
}

} // namespace tcm
