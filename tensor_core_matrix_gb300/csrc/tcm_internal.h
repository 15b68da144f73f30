// tcm_internal.h -- declarations shared by the library's translation units
// (kernel launchers and the C-ABI layer).  Not installed; not part of the ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>
#include <atomic>

namespace tcm {

// Output / C / bias element formats; values equal the public tcm_dtype codes.
enum OutFmt : int { OUT_BF16 = 0, OUT_F16 = 1, OUT_F32 = 2, OUT_E4M3 = 3, OUT_E5M2 = 4 };

// Epilogue activations; values equal the public tcm_activation codes.
enum Act : int { ACT_NONE = 0, ACT_RELU = 1, ACT_GELU = 2 };

// Device-status codes and the wait sites that can record a timeout.
enum DevCode : int { DEV_OK = 0, DEV_TIMEOUT = 5 };
enum WaitSite : int {
    SITE_LOAD_EMPTY = 1,
    SITE_MMA_FULL = 2,
    SITE_MMA_ACC_EMPTY = 3,
    SITE_EPI_ACC_FULL = 4,
    SITE_DRAIN = 5,
    SITE_MMA_META = 6,   // sparse: issuer waiting for a stage's metadata in TMEM
    SITE_META_EMPTY = 7, // sparse: metadata warps waiting for a free stage
    SITE_RED_FULL = 8,   // K-split: leader waiting for the other CTAs' partial sums
    SITE_RED_EMPTY = 9,  // K-split: CTA waiting for the leader to consume its previous partials
    SITE_PART_WAIT = 10, // tail K split: the tile's owner waiting for the other parts' partial sums
};

// Everything a GEMM kernel needs besides its tensor maps.  "Kernel" rows and
// columns (kM x kN) are the rows of the TMA "A" operand and of the "B"
// operand; with swap_ab the kernel computes D^T (kernel row = D column).
struct GemmParams {
    int kM, kN, K;            // kernel-space problem (K = logical K)
    int num_kb;               // stages of the tile loop (K blocks of 128 bytes x katoms)
    int tiles_m, tiles_n, num_tiles;
    int group_m;              // rasterisation: tiles of this many row blocks share B in L2
    int tile_begin, tile_end; // the range of work units this launch covers (see split_begin)
    int split_begin;          // units below are whole tiles (unit = tile index); from here on each
                              // tile of the last, partly filled round is `split` K parts
    int split;                // K parts per tile of that round (1: none)
    int split_kb;             // split == 2: stages of part 0 (the owner); part 1 has the rest
    float *ws_part;           // split > 1: fp32 partial accumulators of parts 1 .. split-1
    int *ws_flag;             // split > 1: per (tail tile, CTA of the pair): epilogue warps done storing
    void *D;
    long long ldd;
    const void *C;
    long long ldc;
    const void *bias;
    const float *a_scale;
    const float *b_scale;
    float alpha, beta;
    int out_fmt;
    int bias_fmt;             // bias element format (bf16 when the output is FP8)
    int act;                  // Act applied after the bias
    const float *d_scale;     // FP8 output: dequantisation factor of D (D = y / d_scale); null = 1
    float *amax;              // if set: max |y| over the launch, max-combined as fp32 bits
    int swap_ab;
    int prefetch_c;           // one round of tiles with C: the epilogue pulls its C rows into L2 first
    uint32_t stage_tx;        // bytes a stage's TMA loads complete (all CTAs of a pair); 0 = from the tile sizes
    unsigned long long *clock_probe; // if set: CTA 0 adds its SM cycles, global-timer ns and 1 to [0..2]
    uint32_t idesc;
    unsigned long long timeout_ns;
    int *status;              // device status word pair {code, site}
    int fault_inject;         // test hook (FaultBits); 0 in normal launches
    const uint32_t *meta;     // sparse: 2:4 metadata, kM x meta_ld words (library layout)
    long long meta_ld;        // sparse: words per metadata row (K / 32)
};

// Test hook bits: make a pipeline wait run out without touching memory.
enum FaultBits : int {
    FAULT_SKIP_FIRST_LOAD = 1, // the loader never issues (nor announces) its first stage
    FAULT_SKIP_PUBLISH = 2,    // tail K split: helper parts never count their stored partials
};

// Which kernel variant a launch uses.
struct GemmConfig {
    int kind;      // 0 = kind::f16, 1 = kind::f8f6f4, 2 = sparse kind::f16 (canonical metadata
                   // staged by TMA, K % 128 == 0), 3 = MXFP8, 4 = NVFP4, 5 = sparse kind::f16
                   // (hardware-ordered metadata), 6 = MXFP4, 7 = sparse kind::f16 (canonical
                   // metadata loaded by the writer warps, any K % 32 == 0)
    int bn;        // N tile (columns of the accumulator)
    int cta_group; // 1 = one CTA per 128-row tile, 2 = CTA pair per 256-row tile
    int stages;    // 0 = the variant's default ring depth
    int ksplit;    // CTAs of a cluster that split each tile's K range (1, 2 or 4; needs cta_group 1)
    int katoms;    // 128-byte K atoms per stage (1, or 2 for 32-wide single-CTA tiles)
};

cudaError_t launch_gemm(const GemmConfig &cfg, const CUtensorMap &tmA, const CUtensorMap &tmB,
                        const GemmParams &p, int grid, cudaStream_t stream);


cudaError_t launch_gemm_pair(const GemmConfig &cfg, const CUtensorMap &tmA, const CUtensorMap &tmB,
                             const GemmParams &p, int grid, cudaStream_t stream);
cudaError_t launch_gemm_ksplit(const GemmConfig &cfg, const CUtensorMap &tmA, const CUtensorMap &tmB,
                               const GemmParams &p, int grid, cudaStream_t stream);

// Tensor maps of a block-scaled GEMM: the FP8 operands (as for the dense
// kernel) and the blocked scale arrays viewed as (atoms x 32) rows of 16 bytes.
struct MxMaps {
    CUtensorMap a, b, sa, sb;
};

cudaError_t launch_gemm_mx(const GemmConfig &cfg, const MxMaps &maps, const GemmParams &p, int grid,
                           cudaStream_t stream);
// canonical 2:4 metadata (M x K/32 words) -> the sparse MMA's tensor-memory order, 2 KB per MMA block
cudaError_t launch_sp_meta_pack(const uint32_t *meta, int64_t M, int64_t K, uint8_t *out, cudaStream_t stream);
// rows x nblk row-major scale codes -> blocked atoms (pad = the format's code of 1.0)
cudaError_t launch_mx_pack_scales(const uint8_t *src, int64_t rows, int64_t nblk, uint32_t pad, uint8_t *dst,
                                  cudaStream_t stream);


cudaError_t launch_sp_compress(int64_t M, int64_t K, int elem_bytes, const void *A, int64_t lda, void *Ac,
                               uint32_t *meta, cudaStream_t stream);
cudaError_t launch_sp_decompress(int64_t M, int64_t K, int elem_bytes, const void *Ac, const uint32_t *meta, void *A,
                                 int64_t lda, cudaStream_t stream);

// INT8 GEMM on the bf16 tensor path: int8 -> bf16 rows (zero-padded to ldo), then the chunked pair kernel
cudaError_t launch_i8_to_bf16(const int8_t *src, int64_t rows, int64_t K, int64_t lds, void *dst, int64_t ldo,
                              cudaStream_t stream);
cudaError_t launch_gemm_i8(const CUtensorMap &tmA, const CUtensorMap &tmB, const GemmParams &p, int grid,
                           cudaStream_t stream);

int *device_status_ptr(); // address of this device's status words (per current device)

// Raise a kernel's dynamic shared-memory limit once per device instead of on every
// launch; `done` is the launching function's own flag word (bit d = device d, d < 64).
inline cudaError_t ensure_max_smem(const void *kern, int bytes, std::atomic<unsigned long long> &done)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = 1ull << (dev & 63);
    if (done.load(std::memory_order_acquire) & bit) return cudaSuccess;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_acq_rel);
    return e;
}

} // namespace tcm
