// tcm_gemm.cu -- the persistent tcgen05 GEMM kernel for sm_103a.
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
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "tcm_internal.h"
#include "tcm_ptx.cuh"

namespace tcm {

constexpr int BM = 128;
constexpr int TILE_K_BYTES = 128; // one 128-byte swizzle atom of K per stage
constexpr int A_STAGE_BYTES = BM * TILE_K_BYTES;
constexpr int NUM_THREADS = 192;
constexpr int EPI_WARPS = 4;
constexpr unsigned long long kMaxSpin = 1ull << 34;

template <int BN, int STAGES>
struct Smem {
    static constexpr int B_STAGE = BN * TILE_K_BYTES;
    static constexpr int A_OFF = 0;
    static constexpr int B_OFF = STAGES * A_STAGE_BYTES;
    static constexpr int BAR_OFF = B_OFF + STAGES * B_STAGE;
    static constexpr int NUM_BARS = 2 * STAGES + 5; // full, empty, tfull[2], tempty[2], drain
    static constexpr int MISC_OFF = BAR_OFF + NUM_BARS * 8;
    static constexpr int BYTES = MISC_OFF + 16;
    static constexpr int ALLOC = BYTES + 1024; // slack to align the base to 1024
};

struct Waiter {
    volatile int *abort_flag;
    unsigned long long timeout_ns;
    int *status;
};

__device__ __forceinline__ void record_timeout(const Waiter &w, int site)
{
    *w.abort_flag = 1;
    if (atomicCAS(w.status, DEV_OK, DEV_TIMEOUT) == DEV_OK) atomicExch(w.status + 1, site);
}

// Wait for phase `parity` of `bar`; false if the CTA is aborting or the limit expired.
__device__ __noinline__ bool bounded_wait(uint64_t *bar, uint32_t parity, const Waiter &w, int site, bool honour_abort)
{
    const uint32_t addr = smem_u32(bar);
    if (mbar_try_wait(addr, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (unsigned long long it = 1; it < kMaxSpin; ++it) {
        if (mbar_try_wait(addr, parity)) return true;
        if ((it & 31ull) == 0) {
            if (honour_abort && *w.abort_flag) return false;
            if (globaltimer_ns() - t0 > w.timeout_ns) break;
        }
    }
    record_timeout(w, site);
    return false;
}

__device__ __forceinline__ void tile_coords(const GemmParams &p, int t, int &mb, int &nb)
{
    const int group = p.group_m * p.tiles_n;
    const int gid = t / group;
    const int first = gid * p.group_m;
    const int gm = min(p.tiles_m - first, p.group_m);
    const int r = t - gid * group;
    mb = first + r % gm;
    nb = r / gm;
}

__device__ __forceinline__ float ld_elem(const void *base, long long i, int fmt)
{
    if (fmt == OUT_BF16) return __bfloat162float(static_cast<const __nv_bfloat16 *>(base)[i]);
    if (fmt == OUT_F16) return __half2float(static_cast<const __half *>(base)[i]);
    return static_cast<const float *>(base)[i];
}

__device__ __forceinline__ void st_elem(void *base, long long i, int fmt, float v)
{
    if (fmt == OUT_BF16) static_cast<__nv_bfloat16 *>(base)[i] = __float2bfloat16_rn(v);
    else if (fmt == OUT_F16) static_cast<__half *>(base)[i] = __float2half_rn(v);
    else static_cast<float *>(base)[i] = v;
}

// 32 consecutive elements starting at a 16-byte-aligned address.
__device__ __forceinline__ void ld32(const void *base, long long i, int fmt, float (&v)[32])
{
    if (fmt == OUT_F32) {
        const float4 *q = reinterpret_cast<const float4 *>(static_cast<const float *>(base) + i);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float4 x = q[j];
            v[4 * j] = x.x, v[4 * j + 1] = x.y, v[4 * j + 2] = x.z, v[4 * j + 3] = x.w;
        }
    } else {
        const uint4 *q = reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(base) + i);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint4 x = q[j];
            const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                if (fmt == OUT_BF16) {
                    const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162 *>(&w[h]);
                    v[8 * j + 2 * h] = __low2float(b), v[8 * j + 2 * h + 1] = __high2float(b);
                } else {
                    const __half2 b = *reinterpret_cast<const __half2 *>(&w[h]);
                    v[8 * j + 2 * h] = __low2float(b), v[8 * j + 2 * h + 1] = __high2float(b);
                }
            }
        }
    }
}

__device__ __forceinline__ void st32(void *base, long long i, int fmt, const float (&v)[32])
{
    if (fmt == OUT_F32) {
        float4 *q = reinterpret_cast<float4 *>(static_cast<float *>(base) + i);
#pragma unroll
        for (int j = 0; j < 8; ++j) q[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
    } else {
        uint4 *q = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(base) + i);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            uint32_t w[4];
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                if (fmt == OUT_BF16) {
                    const __nv_bfloat162 b = __floats2bfloat162_rn(v[8 * j + 2 * h], v[8 * j + 2 * h + 1]);
                    w[h] = *reinterpret_cast<const uint32_t *>(&b);
                } else {
                    const __half2 b = __floats2half2_rn(v[8 * j + 2 * h], v[8 * j + 2 * h + 1]);
                    w[h] = *reinterpret_cast<const uint32_t *>(&b);
                }
            }
            q[j] = make_uint4(w[0], w[1], w[2], w[3]);
        }
    }
}

// Epilogue of 32 accumulator columns of one kernel row: out = scale*acc + beta*C + bias.
__device__ __forceinline__ void epilogue_row32(const GemmParams &p, float scale, int row, int col0,
                                               const uint32_t (&r)[32])
{
    if (row >= p.kM) return;
    float v[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = scale * __uint_as_float(r[j]);
    if (!p.swap_ab) {
        const long long doff = static_cast<long long>(row) * p.ldd + col0;
        if (col0 + 32 <= p.kN) {
            if (p.beta != 0.f) {
                float c[32];
                ld32(p.C, static_cast<long long>(row) * p.ldc + col0, p.out_fmt, c);
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = fmaf(p.beta, c[j], v[j]);
            }
            if (p.bias) {
                float b[32];
                ld32(p.bias, col0, p.out_fmt, b);
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] += b[j];
            }
            st32(p.D, doff, p.out_fmt, v);
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const int col = col0 + j;
                if (col < p.kN) {
                    float x = v[j];
                    if (p.beta != 0.f)
                        x = fmaf(p.beta, ld_elem(p.C, static_cast<long long>(row) * p.ldc + col, p.out_fmt), x);
                    if (p.bias) x += ld_elem(p.bias, col, p.out_fmt);
                    st_elem(p.D, doff + j, p.out_fmt, x);
                }
            }
        }
    } else {
        // kernel row = column n of D, kernel column = row m of D
        const float b = p.bias ? ld_elem(p.bias, row, p.out_fmt) : 0.f;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            const int m = col0 + j;
            if (m < p.kN) {
                float x = v[j];
                if (p.beta != 0.f) x = fmaf(p.beta, ld_elem(p.C, static_cast<long long>(m) * p.ldc + row, p.out_fmt), x);
                x += b;
                st_elem(p.D, static_cast<long long>(m) * p.ldd + row, p.out_fmt, x);
            }
        }
    }
}

template <int KIND, int BN, int STAGES>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, const GemmParams p)
{
    using L = Smem<BN, STAGES>;
    static_assert(BN % 32 == 0 && BN >= 32 && BN <= 256, "BN must be a multiple of 32 in [32, 256]");
    static_assert(L::ALLOC <= 227 * 1024, "shared memory ring too large");
    constexpr uint32_t TMEM_COLS = 2 * BN < 32 ? 32 : 2 * BN;
    constexpr int KB_ELEMS = KIND == 1 ? 128 : 64; // K elements per stage (128 bytes)

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

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, 1);
        }
        for (int a = 0; a < 2; ++a) {
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
                    if (!bounded_wait(empty + stage, phase ^ 1u, w, SITE_LOAD_EMPTY, true)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(full + stage, A_STAGE_BYTES + L::B_STAGE);
                    tma_load_2d(sbase + L::A_OFF + stage * A_STAGE_BYTES, &tmA, full + stage, kb * KB_ELEMS, mb * BM);
                    tma_load_2d(sbase + L::B_OFF + stage * L::B_STAGE, &tmB, full + stage, kb * KB_ELEMS, nb * BN);
                    ++issued;
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            // No copy may still be landing in shared memory when the CTA exits.
            for (int s = 0; s < STAGES; ++s) {
                const long long n = issued > s ? (issued - s + STAGES - 1) / STAGES : 0;
                if (n > 0) bounded_wait(full + s, static_cast<uint32_t>((n - 1) & 1), w, SITE_DRAIN, false);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            int local = 0;
            for (int t = first_tile; ok && t < p.tile_end; t += step, ++local) {
                const int acc = local & 1;
                const uint32_t acc_phase = (local >> 1) & 1;
                if (!bounded_wait(tempty + acc, acc_phase ^ 1u, w, SITE_MMA_ACC_EMPTY, true)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
                for (int kb = 0; kb < p.num_kb; ++kb) {
                    if (!bounded_wait(full + stage, phase, w, SITE_MMA_FULL, true)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t ad = sdesc_kmajor_sw128(sbase + L::A_OFF + stage * A_STAGE_BYTES);
                    const uint64_t bd = sdesc_kmajor_sw128(sbase + L::B_OFF + stage * L::B_STAGE);
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        // +32 bytes of K per instruction = +2 in the descriptor's address field
                        const uint32_t accum = (kb > 0 || k > 0) ? 1u : 0u;
                        if (KIND == 1) mma_f8(d_tmem, ad + 2 * k, bd + 2 * k, p.idesc, accum);
                        else mma_f16(d_tmem, ad + 2 * k, bd + 2 * k, p.idesc, accum);
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
            // Every MMA issued by this thread completes before tensor memory is freed.
            mma_commit(drain);
            bounded_wait(drain, 0, w, SITE_DRAIN, false);
        }
    } else {
        const int quad = warp & 3; // TMEM lanes 32*quad .. 32*quad+31
        const int row_in_tile = quad * 32 + lane;
        const float scale = p.alpha * (p.a_scale ? *p.a_scale : 1.f) * (p.b_scale ? *p.b_scale : 1.f);
        int local = 0;
        for (int t = first_tile; t < p.tile_end; t += step, ++local) {
            const int acc = local & 1;
            const uint32_t acc_phase = (local >> 1) & 1;
            int ok = 1;
            if (lane == 0) ok = bounded_wait(tfull + acc, acc_phase, w, SITE_EPI_ACC_FULL, true);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            tc_fence_after();
            int mb, nb;
            tile_coords(p, t, mb, nb);
            const int row = mb * BM + row_in_tile;
            const uint32_t tbase = tmem_base + static_cast<uint32_t>(acc * BN) + (static_cast<uint32_t>(quad * 32) << 16);
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
                    // last chunk read: hand the accumulator back to the issuer before storing
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(tempty + acc);
                }
                epilogue_row32(p, scale, row, nb * BN + c, r);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

template <int KIND, int BN, int STAGES>
static cudaError_t launch_one(const CUtensorMap &a, const CUtensorMap &b, const GemmParams &p, int grid,
                              cudaStream_t stream)
{
    using L = Smem<BN, STAGES>;
    auto kern = gemm_kernel<KIND, BN, STAGES>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC);
    if (e != cudaSuccess) return e;
    kern<<<grid, NUM_THREADS, L::ALLOC, stream>>>(a, b, p);
    return cudaGetLastError();
}

template <int BN, int STAGES>
static size_t smem_of() { return Smem<BN, STAGES>::ALLOC; }

size_t gemm_smem_bytes(const GemmConfig &cfg)
{
    switch (cfg.bn) {
    case 256: return smem_of<256, 4>();
    case 128: return smem_of<128, 6>();
    case 64: return smem_of<64, 8>();
    default: return smem_of<32, 10>();
    }
}

cudaError_t launch_gemm(const GemmConfig &cfg, const CUtensorMap &tmA, const CUtensorMap &tmB,
                        const CUtensorMap * /*tmMeta*/, const GemmParams &p, int grid, cudaStream_t stream)
{
#define TCM_DISPATCH(KIND)                                                                                          \
    switch (cfg.bn) {                                                                                               \
    case 256: return launch_one<KIND, 256, 4>(tmA, tmB, p, grid, stream);                                           \
    case 128: return launch_one<KIND, 128, 6>(tmA, tmB, p, grid, stream);                                           \
    case 64: return launch_one<KIND, 64, 8>(tmA, tmB, p, grid, stream);                                             \
    case 32: return launch_one<KIND, 32, 10>(tmA, tmB, p, grid, stream);                                            \
    default: return cudaErrorInvalidValue;                                                                          \
    }
    if (cfg.kind == 0) { TCM_DISPATCH(0) }
    if (cfg.kind == 1) { TCM_DISPATCH(1) }
#undef TCM_DISPATCH
    return cudaErrorInvalidValue;
}

} // namespace tcm
