// tcm_sparse.cu -- 2:4 structured-sparsity compress / decompress kernels.
//
// Format ("NVIDIA MMA", section "稠密乘法与 2:4 结构化稀疏乘法"): along K
// every group of 4 logical positions keeps 2 values and their positions
// (the page's example: [a0,0,0,a3] -> values [a0,a3], metadata [0,3]);
// positions are ascending as mma.sp::ordered_metadata requires (section
// "Ampere：FP16/BF16 与整数 MMA 基线").  Kept: the two largest magnitudes,
// ties to the lower position.  Nibble = i0 | i1 << 2; eight nibbles per
// uint32, group g at bits 4*(g%8) of word g/8 of its row.
//
// Decompress: one thread per metadata word (32 logical values).  The op is a pure
// selection on 16-bit codes: magnitudes are compared as the integer value
// of the code without its sign bit, which orders finite binary16 and
// bfloat16 values exactly as their absolute values.
#include "tcm_internal.h"

namespace tcm {

// Value at position q (0..3) of a group, by selects (no indexed register array,
// which would go through local memory).
__device__ __forceinline__ uint16_t at4(const uint16_t (&v)[4], int q)
{
    return q == 0 ? v[0] : (q == 1 ? v[1] : (q == 2 ? v[2] : v[3]));
}

__device__ __forceinline__ uint32_t pick_group(const uint16_t (&v)[4], uint16_t &k0, uint16_t &k1)
{
    uint32_t mag[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) mag[q] = v[q] & 0x7FFFu;
    // first position of the largest magnitude
    int first = 0;
    uint32_t best = mag[0];
#pragma unroll
    for (int q = 1; q < 4; ++q)
        if (mag[q] > best) best = mag[q], first = q;
    // first position of the largest magnitude among the other three
    int second = -1;
    uint32_t best2 = 0;
#pragma unroll
    for (int q = 0; q < 4; ++q)
        if (q != first && (second < 0 || mag[q] > best2)) best2 = mag[q], second = q;
    const int i0 = first < second ? first : second;
    const int i1 = first < second ? second : first;
    k0 = at4(v, i0);
    k1 = at4(v, i1);
    return static_cast<uint32_t>(i0) | (static_cast<uint32_t>(i1) << 2);
}

// Compress: a "chunk" is 8 logical values of one row (one 16-byte load, two
// groups); chunk c of the matrix is row c / (K/8).  Thread t of T handles
// chunks t, t+T, t+2T, t+3T: its four loads are issued before any is used,
// and each load instruction of a warp reads 512 contiguous bytes.  Per chunk
// the thread writes its 4 kept values (8 bytes) and two nibbles; the 4 lanes
// whose chunks make up one metadata word (32 logical values) OR their bytes
// together with shuffles and the first of them stores the word.  K % 32 == 0
// and T % 4 == 0 keep those 4 chunks in one row and in one aligned lane quad.
constexpr int CMP_CHUNKS = 4;

__global__ void __launch_bounds__(256) sp_compress16_kernel(int64_t M, int64_t K, const uint16_t *__restrict__ A,
                                                            int64_t lda, uint16_t *__restrict__ Ac,
                                                            uint32_t *__restrict__ meta)
{
    const int64_t per_row = K / 8;
    const int64_t total = M * per_row;
    const int64_t T = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const int64_t t = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
    const int lane = threadIdx.x & 31;
    uint4 x[CMP_CHUNKS];
#pragma unroll
    for (int j = 0; j < CMP_CHUNKS; ++j) {
        const int64_t c = t + j * T;
        if (c < total) {
            const int64_t m = c / per_row;
            x[j] = __ldg(reinterpret_cast<const uint4 *>(A + m * lda + (c - m * per_row) * 8));
        } else {
            x[j] = make_uint4(0, 0, 0, 0);
        }
    }
#pragma unroll
    for (int j = 0; j < CMP_CHUNKS; ++j) {
        const int64_t c = t + j * T;
        const bool live = c < total;
        const int64_t m = c / per_row;
        const int64_t cc = c - m * per_row;
        const uint32_t u[4] = {x[j].x, x[j].y, x[j].z, x[j].w};
        uint16_t out[4];
        uint32_t byte = 0;
#pragma unroll
        for (int g = 0; g < 2; ++g) {
            const uint16_t grp[4] = {static_cast<uint16_t>(u[2 * g] & 0xFFFFu), static_cast<uint16_t>(u[2 * g] >> 16),
                                     static_cast<uint16_t>(u[2 * g + 1] & 0xFFFFu),
                                     static_cast<uint16_t>(u[2 * g + 1] >> 16)};
            byte |= pick_group(grp, out[2 * g], out[2 * g + 1]) << (4 * g);
        }
        if (live) {
            uint2 o;
            o.x = static_cast<uint32_t>(out[0]) | (static_cast<uint32_t>(out[1]) << 16);
            o.y = static_cast<uint32_t>(out[2]) | (static_cast<uint32_t>(out[3]) << 16);
            *reinterpret_cast<uint2 *>(Ac + m * (K / 2) + cc * 4) = o;
        }
        uint32_t word = live ? byte << (8 * (lane & 3)) : 0u;
        word |= __shfl_xor_sync(0xffffffffu, word, 1);
        word |= __shfl_xor_sync(0xffffffffu, word, 2);
        if (live && (lane & 3) == 0) meta[m * (K / 32) + cc / 4] = word;
    }
}

__global__ void __launch_bounds__(256) sp_decompress16_kernel(int64_t M, int64_t K, const uint16_t *__restrict__ Ac,
                                                              const uint32_t *__restrict__ meta,
                                                              uint16_t *__restrict__ A, int64_t lda)
{
    const int64_t words_per_row = K / 32;
    const int64_t total = M * words_per_row;
    for (int64_t w = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; w < total;
         w += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t m = w / words_per_row;
        const int64_t c = w - m * words_per_row;
        const uint32_t word = __ldg(meta + w);
        const uint4 *src = reinterpret_cast<const uint4 *>(Ac + m * (K / 2) + c * 16);
        uint16_t kept[16];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const uint4 x = __ldg(src + j);
            const uint32_t u[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                kept[8 * j + 2 * h] = static_cast<uint16_t>(u[h] & 0xFFFFu);
                kept[8 * j + 2 * h + 1] = static_cast<uint16_t>(u[h] >> 16);
            }
        }
        uint16_t v[32];
#pragma unroll
        for (int g = 0; g < 8; ++g) {
            const uint32_t nib = (word >> (4 * g)) & 0xFu;
            const uint32_t i0 = nib & 3u, i1 = nib >> 2;
#pragma unroll
            for (int q = 0; q < 4; ++q)
                v[4 * g + q] = q == static_cast<int>(i0) ? kept[2 * g] : (q == static_cast<int>(i1) ? kept[2 * g + 1] : 0);
        }
        uint4 *dst = reinterpret_cast<uint4 *>(A + m * lda + c * 32);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            uint32_t u[4];
#pragma unroll
            for (int h = 0; h < 4; ++h)
                u[h] = static_cast<uint32_t>(v[8 * j + 2 * h]) | (static_cast<uint32_t>(v[8 * j + 2 * h + 1]) << 16);
            dst[j] = make_uint4(u[0], u[1], u[2], u[3]);
        }
    }
}

static int grid_for(int64_t work)
{
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t blocks = (work + 255) / 256;
    const int64_t cap = static_cast<int64_t>(sms > 0 ? sms : 1) * 8;
    return static_cast<int>(blocks < cap ? (blocks > 0 ? blocks : 1) : cap);
}

cudaError_t launch_sp_compress(int64_t M, int64_t K, int elem_bytes, const void *A, int64_t lda, void *Ac,
                               uint32_t *meta, cudaStream_t stream)
{
    if (elem_bytes != 2) return cudaErrorInvalidValue;
    const int64_t work = M * (K / 8); // chunks of 8 logical values
    if (work == 0) return cudaSuccess;
    const int64_t blocks = (work + 256 * CMP_CHUNKS - 1) / (256 * CMP_CHUNKS);
    if (blocks > 0x7FFFFFFF) return cudaErrorInvalidValue;
    sp_compress16_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
        M, K, static_cast<const uint16_t *>(A), lda, static_cast<uint16_t *>(Ac), meta);
    return cudaGetLastError();
}

cudaError_t launch_sp_decompress(int64_t M, int64_t K, int elem_bytes, const void *Ac, const uint32_t *meta, void *A,
                                 int64_t lda, cudaStream_t stream)
{
    if (elem_bytes != 2) return cudaErrorInvalidValue;
    const int64_t work = M * (K / 32);
    if (work == 0) return cudaSuccess;
    sp_decompress16_kernel<<<grid_for(work), 256, 0, stream>>>(M, K, static_cast<const uint16_t *>(Ac), meta,
                                                                static_cast<uint16_t *>(A), lda);
    return cudaGetLastError();
}

} // namespace tcm
