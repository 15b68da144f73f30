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
// One thread owns one metadata word, i.e. 32 logical elements (64 bytes) of
// a row: four 16-byte loads in, two 16-byte stores and one word out, so a
// warp moves 2 KiB of contiguous input per step.  The op is a pure
// selection on 16-bit codes: magnitudes are compared as the integer value
// of the code without its sign bit, which orders finite binary16 and
// bfloat16 values exactly as their absolute values.
#include "tcm_internal.h"

namespace tcm {

__device__ __forceinline__ uint32_t pick_group(const uint16_t (&v)[4], uint16_t &k0, uint16_t &k1)
{
    uint32_t mag[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) mag[q] = v[q] & 0x7FFFu;
    int first = 0;
#pragma unroll
    for (int q = 1; q < 4; ++q)
        if (mag[q] > mag[first]) first = q;
    int second = first == 0 ? 1 : 0;
#pragma unroll
    for (int q = 0; q < 4; ++q)
        if (q != first && mag[q] > mag[second]) second = q;
    const int i0 = first < second ? first : second;
    const int i1 = first < second ? second : first;
    k0 = v[i0];
    k1 = v[i1];
    return static_cast<uint32_t>(i0) | (static_cast<uint32_t>(i1) << 2);
}

__global__ void __launch_bounds__(256) sp_compress16_kernel(int64_t M, int64_t K, const uint16_t *__restrict__ A,
                                                            int64_t lda, uint16_t *__restrict__ Ac,
                                                            uint32_t *__restrict__ meta)
{
    const int64_t words_per_row = K / 32;
    const int64_t total = M * words_per_row;
    for (int64_t w = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; w < total;
         w += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t m = w / words_per_row;
        const int64_t c = w - m * words_per_row;
        const uint4 *src = reinterpret_cast<const uint4 *>(A + m * lda + c * 32);
        uint16_t v[32];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint4 x = __ldg(src + j);
            const uint32_t u[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                v[8 * j + 2 * h] = static_cast<uint16_t>(u[h] & 0xFFFFu);
                v[8 * j + 2 * h + 1] = static_cast<uint16_t>(u[h] >> 16);
            }
        }
        uint32_t word = 0;
        uint16_t out[16];
#pragma unroll
        for (int g = 0; g < 8; ++g) {
            const uint16_t grp[4] = {v[4 * g], v[4 * g + 1], v[4 * g + 2], v[4 * g + 3]};
            word |= pick_group(grp, out[2 * g], out[2 * g + 1]) << (4 * g);
        }
        uint4 *dst = reinterpret_cast<uint4 *>(Ac + m * (K / 2) + c * 16);
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            uint32_t u[4];
#pragma unroll
            for (int h = 0; h < 4; ++h)
                u[h] = static_cast<uint32_t>(out[8 * j + 2 * h]) | (static_cast<uint32_t>(out[8 * j + 2 * h + 1]) << 16);
            dst[j] = make_uint4(u[0], u[1], u[2], u[3]);
        }
        meta[w] = word;
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
    const int64_t work = M * (K / 32);
    if (work == 0) return cudaSuccess;
    sp_compress16_kernel<<<grid_for(work), 256, 0, stream>>>(M, K, static_cast<const uint16_t *>(A), lda,
                                                              static_cast<uint16_t *>(Ac), meta);
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
