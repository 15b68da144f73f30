// tcm_kernel_common.cuh -- pieces shared by the dense and the 2:4-sparse
// tcgen05 GEMM kernels: shared-memory ring layout, bounded mbarrier waits
// that record a device status instead of hanging, the grouped tile order,
// and the epilogue (alpha*sA*sB*acc + beta*C + bias, activation, amax,
// RNE cast -- saturating for FP8 outputs -- and stores).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "tcm_internal.h"
#include "tcm_ptx.cuh"

namespace tcm {

constexpr int BM = 128;
constexpr int TILE_K_BYTES = 128; // one 128-byte swizzle atom of K per stage
constexpr int A_STAGE_BYTES = BM * TILE_K_BYTES;
constexpr int NUM_THREADS = 192;
constexpr int EPI_WARPS = 4;
constexpr unsigned long long kMaxSpin = 1ull << 34;

// KATOMS: 128-byte K atoms per stage (each atom is a separate SW128 tile).
template <int BN, int STAGES, int RED_BYTES = 0, int KATOMS = 1>
struct Smem {
    static constexpr int A_STAGE = KATOMS * A_STAGE_BYTES;
    static constexpr int B_STAGE = KATOMS * BN * TILE_K_BYTES;
    static constexpr int A_OFF = 0;
    static constexpr int B_OFF = STAGES * A_STAGE;
    static constexpr int RED_OFF = B_OFF + STAGES * B_STAGE; // K-split partial sums (leader CTA)
    static constexpr int BAR_OFF = RED_OFF + RED_BYTES;
    // full, empty, tfull[2], tempty[2], drain, red_full, red_empty, part_full, part_staged
    static constexpr int NUM_BARS = 2 * STAGES + 9;
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
template <bool ACQ_CLUSTER>
__device__ __forceinline__ bool poll_bar(uint32_t addr, uint32_t parity)
{
    if constexpr (ACQ_CLUSTER) return mbar_try_wait_acq_cluster(addr, parity);
    else return mbar_try_wait(addr, parity);
}

// Wait for phase `parity` of `bar`; false if the CTA is aborting or the limit expired.
// ACQ_CLUSTER: acquire at cluster scope, for barriers whose arrivals publish
// generic shared-memory data written by another CTA of the cluster.
template <int CG, bool ACQ_CLUSTER = false>
__device__ __noinline__ bool bounded_wait(uint64_t *bar, uint32_t parity, const Waiter &w, int site, bool honour_abort)
{
    const uint32_t addr = smem_u32(bar);
    if (poll_bar<ACQ_CLUSTER>(addr, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (unsigned long long it = 1; it < kMaxSpin; ++it) {
        if (poll_bar<ACQ_CLUSTER>(addr, parity)) return true;
        if ((it & 31ull) == 0) {
            if (honour_abort && *w.abort_flag) return false;
            if (globaltimer_ns() - t0 > w.timeout_ns) break;
        }
    }
    record_timeout(w, site);
    return false;
}

__device__ __forceinline__ int ld_acquire_gpu(const int *addr)
{
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(addr) : "memory");
    return v;
}

// Wait until the counter in global memory written by other CTAs reaches `target`; false
// if the CTA is aborting or the limit expired (then the timeout is recorded at `site`).
static __device__ __noinline__ bool wait_count(const int *counter, int target, const Waiter &w, int site)
{
    const uint64_t t0 = globaltimer_ns();
    for (unsigned long long it = 0; it < kMaxSpin; ++it) {
        if (ld_acquire_gpu(counter) >= target) return true;
        if ((it & 31ull) == 0) {
            if (*w.abort_flag) return false;
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

// Work unit u of a launch: a whole tile (u < split_begin), or part `part` of the `split`
// K parts of tile split_begin + j of the last, partly filled round (j = (u - split_begin) /
// split).  Splitting that round over K lets more CTA pairs share it at full tile width:
// at 8192^3 with 76 pairs, the 36 leftover 256 x 256 tiles become 72 part-K units, so
// the launch takes ~13.6 tile times instead of 14.  Part 0 owns the tile: it adds the
// other parts' fp32 partial sums (in part order) before its epilogue.  With two parts the
// owner takes p.split_kb stages, more than half: the helper finishes first and its
// partial sums are published by the time the owner's own MMAs end.
struct Unit {
    int mb, nb;   // the tile's row and column block
    int kb0, kb1; // stages (K blocks x katoms) of this unit
    int part;     // 0: whole tile or owner of a split tile; 1 .. split-1: helper
    int j;        // index of a split tile among the split ones; -1 for a whole tile
};

__device__ __forceinline__ Unit unit_coords(const GemmParams &p, int u)
{
    Unit r;
    int t = u;
    r.part = 0;
    r.j = -1;
    r.kb0 = 0;
    r.kb1 = p.num_kb;
    if (u >= p.split_begin) {
        const int q = u - p.split_begin;
        r.j = q / p.split;
        r.part = q - r.j * p.split;
        t = p.split_begin + r.j;
        if (p.split == 2) {
            r.kb0 = r.part == 0 ? 0 : p.split_kb;
            r.kb1 = r.part == 0 ? p.split_kb : p.num_kb;
        } else {
            r.kb0 = static_cast<int>((static_cast<long long>(p.num_kb) * r.part) / p.split);
            r.kb1 = static_cast<int>((static_cast<long long>(p.num_kb) * (r.part + 1)) / p.split);
        }
    }
    tile_coords(p, t, r.mb, r.nb);
    return r;
}

// Clock probe: CTA 0's SM cycles and global-timer nanoseconds from its start to its end.
__device__ __forceinline__ void clock_probe_add(const GemmParams &p, unsigned long long c0, unsigned long long g0)
{
    if (p.clock_probe && blockIdx.x == 0 && threadIdx.x == 0) {
        const unsigned long long c1 = clock64();
        const unsigned long long g1 = globaltimer_ns();
        atomicAdd(p.clock_probe, c1 - c0);
        atomicAdd(p.clock_probe + 1, g1 - g0);
        atomicAdd(p.clock_probe + 2, 1ull);
    }
}

__device__ __forceinline__ float ld_elem(const void *base, long long i, int fmt)
{
    if (fmt == OUT_BF16) return __bfloat162float(static_cast<const __nv_bfloat16 *>(base)[i]);
    if (fmt == OUT_F16) return __half2float(static_cast<const __half *>(base)[i]);
    return static_cast<const float *>(base)[i];
}

__device__ __forceinline__ __nv_fp8_interpretation_t fp8_kind(int fmt)
{
    return fmt == OUT_E4M3 ? __NV_E4M3 : __NV_E5M2;
}

// Two values, round to nearest even with saturation to the largest finite FP8 value.
__device__ __forceinline__ uint32_t fp8x2(float lo, float hi, int fmt)
{
    return static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, fp8_kind(fmt)));
}

__device__ __forceinline__ void st_elem(void *base, long long i, int fmt, float v)
{
    if (fmt == OUT_BF16) static_cast<__nv_bfloat16 *>(base)[i] = __float2bfloat16_rn(v);
    else if (fmt == OUT_F16) static_cast<__half *>(base)[i] = __float2half_rn(v);
    else if (fmt == OUT_F32) static_cast<float *>(base)[i] = v;
    else static_cast<uint8_t *>(base)[i] = __nv_cvt_float_to_fp8(v, __NV_SATFINITE, fp8_kind(fmt));
}

__device__ __forceinline__ float activate(float v, int act)
{
    if (act == ACT_RELU) return v > 0.f ? v : 0.f;
    if (act == ACT_GELU) return 0.5f * v * (1.f + erff(v * 0.70710678118654752f));
    return v;
}

// max(m, |x|) that keeps a NaN once seen (fmaxf would drop it).
__device__ __forceinline__ float amax_combine(float m, float x)
{
    const float a = fabsf(x);
    return (a > m || a != a) ? a : m;
}

// Warp-wide amax of the per-lane maxima, max-combined into *amax as fp32 bits
// (non-negative floats order like their bit patterns; a NaN is above +inf).
__device__ __forceinline__ void amax_flush(float *amax, float m)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = amax_combine(m, __shfl_xor_sync(0xffffffffu, m, o));
    if ((threadIdx.x & 31) == 0) atomicMax(reinterpret_cast<unsigned int *>(amax), __float_as_uint(m));
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
    if (fmt == OUT_E4M3 || fmt == OUT_E5M2) {
        uint4 *q = reinterpret_cast<uint4 *>(static_cast<uint8_t *>(base) + i);
        uint32_t w[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) w[j] = fp8x2(v[4 * j], v[4 * j + 1], fmt) | (fp8x2(v[4 * j + 2], v[4 * j + 3], fmt) << 16);
        q[0] = make_uint4(w[0], w[1], w[2], w[3]);
        q[1] = make_uint4(w[4], w[5], w[6], w[7]);
    } else if (fmt == OUT_F32) {
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

// Epilogue of 32 accumulator columns of one kernel row:
//   y = act(scale*acc + beta*C + bias), stored as y * RN32(1 / d_scale) in the output format.
// Returns max |y| over the stored elements when p.amax is set (else 0).
__device__ __forceinline__ float epilogue_row32(const GemmParams &p, float scale, int row, int col0,
                                                const uint32_t (&r)[32])
{
    float m = 0.f;
    if (row >= p.kM) return m;
    // D = y * r with r = 1 / d_scale rounded once to fp32 (a division per element would
    // double the cost of the fused FP8 epilogue: measured 1408 against ~3000 TFLOP/s)
    const float inv_d = p.d_scale ? __frcp_rn(*p.d_scale) : 1.f;
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
                ld32(p.bias, col0, p.bias_fmt, b);
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] += b[j];
            }
            if (p.act != ACT_NONE) {
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = activate(v[j], p.act);
            }
            if (p.amax) {
#pragma unroll
                for (int j = 0; j < 32; ++j) m = amax_combine(m, v[j]);
            }
            if (p.d_scale) {
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] *= inv_d;
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
                    if (p.bias) x += ld_elem(p.bias, col, p.bias_fmt);
                    x = activate(x, p.act);
                    if (p.amax) m = amax_combine(m, x);
                    st_elem(p.D, doff + j, p.out_fmt, p.d_scale ? x * inv_d : x);
                }
            }
        }
    } else {
        // kernel row = column n of D, kernel column = row m of D
        const float b = p.bias ? ld_elem(p.bias, row, p.bias_fmt) : 0.f;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            const int mm = col0 + j;
            if (mm < p.kN) {
                float x = v[j];
                if (p.beta != 0.f) x = fmaf(p.beta, ld_elem(p.C, static_cast<long long>(mm) * p.ldc + row, p.out_fmt), x);
                x += b;
                x = activate(x, p.act);
                if (p.amax) m = amax_combine(m, x);
                st_elem(p.D, static_cast<long long>(mm) * p.ldd + row, p.out_fmt, p.d_scale ? x * inv_d : x);
            }
        }
    }
    return m;
}

// Wait on a barrier of this CTA (arrivals may come from the peer CTA of a pair).
// The first test is inline: a phase that has already completed costs no call
// (measured: an out-of-line call on every stage of the issuing thread's loop
// left the tensor pipe idle a quarter of the time).
template <int CG>
__device__ __forceinline__ bool wait_bar(uint64_t *bar, uint32_t parity, const Waiter &w, int site, bool honour_abort)
{
    if (mbar_try_wait(smem_u32(bar), parity)) return true;
    return bounded_wait<CG>(bar, parity, w, site, honour_abort);
}

} // namespace tcm
