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

// Kept positions and values of one group of four 16-bit codes (v0 | v1 << 16,
// v2 | v3 << 16).  Each position q gets the key (|code| << 2) | (3 - q):
// keys are distinct, and a larger key means a larger magnitude or, for equal
// magnitudes, a lower position -- so the two largest keys are exactly the two
// kept positions with ties going to the lower one.  The top two of four keys
// take seven integer min / max operations; no branches, no indexed arrays.
__device__ __forceinline__ uint32_t pick_group(uint32_t lo, uint32_t hi, uint32_t &kept)
{
    const uint32_t k0 = ((lo & 0x7FFFu) << 2) | 3u;
    const uint32_t k1 = (((lo >> 16) & 0x7FFFu) << 2) | 2u;
    const uint32_t k2 = ((hi & 0x7FFFu) << 2) | 1u;
    const uint32_t k3 = (((hi >> 16) & 0x7FFFu) << 2) | 0u;
    const uint32_t a = max(k0, k1), b = min(k0, k1), c = max(k2, k3), d = min(k2, k3);
    const uint32_t top = max(a, c);
    const uint32_t second = max(min(a, c), max(b, d));
    const uint32_t qa = 3u - (top & 3u), qb = 3u - (second & 3u);
    const uint32_t i0 = min(qa, qb), i1 = max(qa, qb);
    const uint64_t grp = static_cast<uint64_t>(lo) | (static_cast<uint64_t>(hi) << 32);
    const uint32_t v0 = static_cast<uint32_t>(grp >> (16u * i0)) & 0xFFFFu;
    const uint32_t v1 = static_cast<uint32_t>(grp >> (16u * i1)) & 0xFFFFu;
    kept = v0 | (v1 << 16);
    return i0 | (i1 << 2);
}

// Compress: a "chunk" is 8 logical values of a row (one 16-byte load, two
// groups).  Block (x, y) handles chunks [x*1024, x*1024 + 1024) of rows y,
// y + gridDim.y, ...; thread t takes chunks t, t+256, t+512, t+768 of that
// range, issuing the four loads before using any, and each warp load reads
// 512 contiguous bytes.  Per chunk it writes its 4 kept values (8 bytes) and
// two nibbles; the 4 lanes whose chunks form one metadata word (32 logical
// values) OR their bytes with shuffles and the first stores the word.  K % 32
// == 0 keeps those 4 chunks in one row and in one aligned lane quad.
constexpr int CMP_CHUNKS = 4;
constexpr int CMP_SEG = 256 * CMP_CHUNKS; // chunks per block and row

__global__ void __launch_bounds__(256) sp_compress16_kernel(int64_t M, int64_t K, const uint16_t *__restrict__ A,
                                                            int64_t lda, uint16_t *__restrict__ Ac,
                                                            uint32_t *__restrict__ meta)
{
    const int per_row = static_cast<int>(K / 8);
    const int lane = threadIdx.x & 31;
    const int c_first = static_cast<int>(blockIdx.x) * CMP_SEG + static_cast<int>(threadIdx.x);
    for (int64_t m = blockIdx.y; m < M; m += gridDim.y) {
        const uint16_t *arow = A + m * lda;
        uint2 *crow = reinterpret_cast<uint2 *>(Ac + m * (K / 2));
        uint32_t *mrow = meta + m * (K / 32);
        uint4 x[CMP_CHUNKS];
#pragma unroll
        for (int j = 0; j < CMP_CHUNKS; ++j) {
            const int c = c_first + 256 * j;
            x[j] = c < per_row ? __ldg(reinterpret_cast<const uint4 *>(arow) + c) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int j = 0; j < CMP_CHUNKS; ++j) {
            const int c = c_first + 256 * j;
            uint32_t k0, k1;
            const uint32_t byte = pick_group(x[j].x, x[j].y, k0) | (pick_group(x[j].z, x[j].w, k1) << 4);
            if (c < per_row) crow[c] = make_uint2(k0, k1);
            uint32_t word = byte << (8 * (lane & 3));
            word |= __shfl_xor_sync(0xffffffffu, word, 1);
            word |= __shfl_xor_sync(0xffffffffu, word, 2);
            if (c < per_row && (lane & 3) == 0) mrow[c >> 2] = word;
        }
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
    if (M == 0 || K == 0) return cudaSuccess;
    const int64_t segs = (K / 8 + CMP_SEG - 1) / CMP_SEG;
    const dim3 grid(static_cast<unsigned>(segs), static_cast<unsigned>(M < 65535 ? M : 65535), 1);
    sp_compress16_kernel<<<grid, 256, 0, stream>>>(M, K, static_cast<const uint16_t *>(A), lda,
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

namespace tcm {

// Hardware-ordered 2:4 metadata (see tcm_sp_meta_pack in tcm.h): one thread per
// lane L of one stage's 2 KB block.  Block (t, kb) holds, at byte 16 L + 4 k, the
// word the stage's sparse MMA k reads for lane L = 16a + 8s + r: bits 0..15 =
// nibbles 4s..4s+3 of row 16a + r's word for logical K block q = 4 kb + k, bits
// 16..31 = the same of row 16a + 8 + r.  Rows past M and K blocks past K/32 read
// 0x44444444 (positions {0, 1}; their A values are zero).
// vec: every row holds whole stages of 4 words (qn % 4 == 0) at a 16-byte-aligned base.
__global__ void __launch_bounds__(256) sp_meta_pack_kernel(const uint32_t *__restrict__ meta, int64_t M,
                                                           int64_t qn, int64_t kbs, int64_t total, bool vec,
                                                           uint4 *__restrict__ out)
{
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= total) return;
    const int64_t lane = i & 127;
    const int64_t stage = i >> 7; // t * kbs + kb
    const int64_t kb = stage % kbs;
    const int64_t t = stage / kbs;
    const int64_t a = lane >> 4, s = (lane >> 3) & 1, r = lane & 7;
    const int64_t r0 = t * 128 + 16 * a + r, r1 = r0 + 8;
    const uint32_t fill = 0x44444444u;
    const int64_t q0 = kb * 4;
    uint32_t m0[4], m1[4];
    if (vec) { // the stage's four words of each row in one 16-byte load
        const uint4 v0 = r0 < M ? __ldg(reinterpret_cast<const uint4 *>(meta + r0 * qn + q0)) : make_uint4(fill, fill, fill, fill);
        const uint4 v1 = r1 < M ? __ldg(reinterpret_cast<const uint4 *>(meta + r1 * qn + q0)) : make_uint4(fill, fill, fill, fill);
        m0[0] = v0.x; m0[1] = v0.y; m0[2] = v0.z; m0[3] = v0.w;
        m1[0] = v1.x; m1[1] = v1.y; m1[2] = v1.z; m1[3] = v1.w;
    } else {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            m0[k] = (r0 < M && q0 + k < qn) ? __ldg(meta + r0 * qn + q0 + k) : fill;
            m1[k] = (r1 < M && q0 + k < qn) ? __ldg(meta + r1 * qn + q0 + k) : fill;
        }
    }
    uint32_t w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k)
        w[k] = s == 0 ? ((m0[k] & 0xFFFFu) | (m1[k] << 16)) : ((m0[k] >> 16) | (m1[k] & 0xFFFF0000u));
    out[i] = make_uint4(w[0], w[1], w[2], w[3]);
}

cudaError_t launch_sp_meta_pack(const uint32_t *meta, int64_t M, int64_t K, uint8_t *out, cudaStream_t stream)
{
    const int64_t qn = K / 32;
    const int64_t kbs = (K + 127) / 128;
    const int64_t total = ((M + 127) / 128) * kbs * 128;
    if (total == 0) return cudaSuccess;
    const bool vec = qn % 4 == 0 && (reinterpret_cast<uintptr_t>(meta) & 15u) == 0;
    sp_meta_pack_kernel<<<static_cast<unsigned>((total + 255) / 256), 256, 0, stream>>>(meta, M, qn, kbs, total, vec,
                                                                                       reinterpret_cast<uint4 *>(out));
    return cudaGetLastError();
}

} // namespace tcm
