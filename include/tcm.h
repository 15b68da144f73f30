/*
 * tcm.h -- C ABI of the GB300 (sm_103a) tensor-core GEMM library (libtcm.so).
 *
 * The library computes the tiled tensor-core GEMM of the pages
 *   "NVIDIA MMA" (rainlin-net.pages.dev/llm-inference/nvidia-mma), section
 *   "从 FMA 到 MMA，再到 GEMM":  D[m,n] = sum_k A[m,k] B[k,n] + C[m,n],
 * with the input / accumulator / output stages of section "输入/累加/输出"
 * (narrow inputs, fp32 accumulator, epilogue scale / bias / cast), and the
 * 2:4 structured-sparse-A form of section "稠密乘法与 2:4 结构化稀疏乘法".
 * Layout follows the ".row.col" convention of "CUDA 014 - MMA 指令的用法详解"
 * (blog-9y3.pages.dev/posts/cuda/mma/), section "MMA 指令的格式": A is
 * row-major, B is column-major -- stored as N rows of K contiguous elements
 * ("K-major"), the N x K storage that the same page's ldmatrix section
 * loads without a transpose.
 *
 * General conventions (every entry point):
 *  - All matrix / vector pointers are CALLER-OWNED DEVICE memory on the
 *    current CUDA device.  The library never frees or retains them.
 *  - Work is enqueued asynchronously on `stream` (NULL = legacy default
 *    stream).  A return of TCM_OK means "validated and launched"; results
 *    are ready once the stream reaches that point.
 *  - Argument errors are detected on the host BEFORE anything is launched
 *    and return TCM_ERR_INVALID_ARG / TCM_ERR_UNSUPPORTED /
 *    TCM_ERR_MISALIGNED; in that case no device memory is touched.
 *  - Device-side failures (a pipeline wait that exceeded its time limit) do
 *    not trap: the kernel records a code and returns; read it with
 *    tcm_get_device_status().
 *  - Element codes: bf16, f16 (IEEE binary16), f32 (IEEE binary32),
 *    e4m3 (OCP FP8 E4M3, finite max 448), e5m2 (OCP FP8 E5M2).
 *  - Base pointers must be 16-byte aligned and every leading dimension, in
 *    bytes, a multiple of 16 (tensor-memory-accelerator rule), otherwise
 *    TCM_ERR_MISALIGNED.
 *  - The library allocates no device memory on any call path.
 */
#ifndef TCM_H
#define TCM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t; declared here so this header needs no CUDA include. */
typedef struct CUstream_st *tcm_stream_t;

typedef enum {
    TCM_OK = 0,
    TCM_ERR_INVALID_ARG = 1, /* null pointer, negative size, ld < row length, ... */
    TCM_ERR_UNSUPPORTED = 2, /* dtype combination or shape class not implemented */
    TCM_ERR_MISALIGNED = 3,  /* base pointer or leading dimension not 16-byte aligned */
    TCM_ERR_CUDA = 4,        /* a CUDA runtime / driver call failed (launch, attribute, ...) */
    TCM_ERR_TIMEOUT = 5      /* a device-side wait exceeded its limit (see tcm_get_device_status) */
} tcm_status;

typedef enum {
    TCM_BF16 = 0,
    TCM_F16 = 1,
    TCM_F32 = 2,
    TCM_E4M3 = 3,
    TCM_E5M2 = 4,
    TCM_E2M1 = 5 /* OCP FP4: s | e(2, bias 1) | m(1), packed two per byte, element 2i in the low nibble */
} tcm_dtype;

/* Activation of the fused epilogue (tcm_gemm_fused). */
typedef enum {
    TCM_ACT_NONE = 0,
    TCM_ACT_RELU = 1, /* max(y, 0); NaN -> 0 */
    TCM_ACT_GELU = 2  /* y * Phi(y) = 0.5 y (1 + erf(y / sqrt 2)), with the device erff */
} tcm_activation;

/*
 * tcm_gemm -- D = alpha * (A . B) + beta * C
 *
 * Definition: "NVIDIA MMA", section "从 FMA 到 MMA，再到 GEMM"
 * (D_{m,n} = sum_k A_{m,k} B_{k,n} + C_{m,n}); accumulation in fp32 as in
 * section "输入/累加/输出"; the output cast is round-to-nearest-even.
 *
 *  M, N, K    problem size; M, N >= 1, K >= 0 (K == 0 gives beta*C; A and B
 *             are then not read, and their pointers are not checked).
 *  in_dtype   TCM_BF16 or TCM_F16 for both A and B (the FP8 types go
 *             through tcm_gemm_ex, which carries their scales).
 *  A          M x K, row-major, leading dimension K (densely packed).
 *  B          K x N column-major == N rows of K, leading dimension K.
 *  C          M x N row-major, leading dimension N, dtype = out_dtype;
 *             may be NULL iff beta == 0.  C may alias D exactly.
 *  D          M x N row-major, leading dimension N, dtype out_dtype
 *             (TCM_BF16, TCM_F16 or TCM_F32).
 *  Results are within 1e-5 * |alpha| * sum_k |a_mk b_kn| + one rounding of the
 *  output type of the exact value.
 */
tcm_status tcm_gemm(int64_t M, int64_t N, int64_t K, tcm_dtype in_dtype,
                    const void *A, const void *B, const void *C, void *D,
                    float alpha, float beta, tcm_dtype out_dtype, tcm_stream_t stream);

/*
 * tcm_gemm_ex -- D = alpha * sA * sB * (A . B) + beta * C + bias
 *
 * The epilogue chain of "NVIDIA MMA", section "输入/累加/输出"
 * (FP8 A x FP8 B -> FP32 accumulator -> scale / bias / cast -> output),
 * read as: scale, then + beta*C, then + bias[n], then one RNE cast.
 *
 *  a_dtype, b_dtype  (bf16,bf16), (f16,f16), or any pair of {e4m3, e5m2, e2m1}
 *                    (section "SM100：tcgen05.mma" table: kind::f8f6f4 lets A
 *                    and B differ, e.g. FP4 x FP8; section "量化配置如何映射到 MMA":
 *                    W4A8 on Blackwell is bare FP4 x bare FP8).  Other pairs:
 *                    TCM_ERR_UNSUPPORTED.  An E2M1 operand needs K % 128 == 0
 *                    (else TCM_ERR_UNSUPPORTED), its pitch a multiple of 64
 *                    elements and its base 32-byte aligned (else
 *                    TCM_ERR_MISALIGNED).
 *  lda, ldb          row pitches in ELEMENTS of A (M x K) and of B (N x K);
 *                    lda, ldb >= K (an E2M1 row of lda elements is lda/2 bytes).
 *  ldc, ldd          row pitches in elements of C and D; >= N.
 *  a_scale, b_scale  DEVICE pointers to one fp32 each (per-tensor
 *                    dequantisation factors: real value = stored value *
 *                    scale), or NULL for 1.0.
 *  bias              DEVICE pointer to N elements of out_dtype, or NULL.
 *  out_dtype         TCM_BF16, TCM_F16 or TCM_F32; C has the same dtype.
 */
tcm_status tcm_gemm_ex(int64_t M, int64_t N, int64_t K,
                       tcm_dtype a_dtype, const void *A, int64_t lda,
                       tcm_dtype b_dtype, const void *B, int64_t ldb,
                       const void *C, int64_t ldc, void *D, int64_t ldd,
                       tcm_dtype out_dtype, float alpha, float beta,
                       const float *a_scale, const float *b_scale, const void *bias,
                       tcm_stream_t stream);

/*
 * tcm_gemm_ex_ws -- tcm_gemm_ex with a caller-provided device workspace, which lets
 * the persistent kernel balance its last round.  The CTA pairs of the kernel take
 * 256 x 256 output tiles in rounds; when the last round is only partly filled
 * (e.g. 8192^3: 1024 tiles = 13 rounds of 76 pairs + 36 tiles) and at most half
 * full, and K is long enough for it to pay (at least 64 K blocks of 128 bytes),
 * each of its tiles is split into two parts along K, computed by two pairs
 * at once: the second part stores its fp32 partial sums in the workspace and the
 * first adds them before the epilogue.  The first part takes a few K blocks more
 * than half (9 when K allows; 10 for 8-bit operands, whose stages hold two
 * 128-byte blocks), so that the second part's sums are published by the
 * time the first part's own products are done.  Same results as tcm_gemm_ex up to the
 * order of the fp32 accumulation (integer-valued sums stay exact).
 *  workspace        DEVICE memory, 16-byte aligned, caller-owned, at least
 *                   tcm_gemm_workspace_bytes(M, N, K, a_dtype, b_dtype) bytes
 *                   (else TCM_ERR_INVALID_ARG); NULL with workspace_bytes 0 gives
 *                   tcm_gemm_ex.  Its contents are scratch: the call zeroes its
 *                   counters on `stream` first.  Two calls that may run at the same
 *                   time on the GPU must not share a workspace.
 *  other arguments  as tcm_gemm_ex.
 * A launch that splits tiles is cooperative (all its CTAs resident at once); the
 * wait of part 0 for the other parts is bounded like every pipeline wait (site 10).
 *
 * tcm_gemm_workspace_bytes -- bytes of workspace tcm_gemm_ex_ws uses for this
 * problem on the current device (0: no split; -1: arguments tcm_gemm_ex would
 * reject).  Depends on the device's SM count and on tcm_set_config_override.
 * Host only.
 */
tcm_status tcm_gemm_ex_ws(int64_t M, int64_t N, int64_t K,
                          tcm_dtype a_dtype, const void *A, int64_t lda,
                          tcm_dtype b_dtype, const void *B, int64_t ldb,
                          const void *C, int64_t ldc, void *D, int64_t ldd,
                          tcm_dtype out_dtype, float alpha, float beta,
                          const float *a_scale, const float *b_scale, const void *bias,
                          void *workspace, int64_t workspace_bytes, tcm_stream_t stream);
int64_t tcm_gemm_workspace_bytes(int64_t M, int64_t N, int64_t K, tcm_dtype a_dtype, tcm_dtype b_dtype);

/*
 * tcm_gemm_ex_builtin_ws -- tcm_gemm_ex_ws for callers that cannot allocate device
 * memory.  The pages have no counterpart: this is a service of the library.
 *
 * Some callers have no way to provide tcm_gemm_ex_ws's workspace: code that runs
 * inside another framework's device-memory manager, where every allocation must go
 * through that manager, or a latency-critical path where cudaMalloc (which may
 * synchronise the device) is not allowed.  This entry point takes the same
 * arguments as tcm_gemm_ex (the caller still passes A, B, C, D, scales and bias)
 * and allocates nothing: its workspace is a 10 MiB array inside the library, one
 * copy on every GPU that loads the library, held until the process exits.
 *  - Size limit: a problem whose tcm_gemm_workspace_bytes exceeds 10 MiB
 *    (10485760 bytes) returns TCM_ERR_UNSUPPORTED before anything is launched.
 *    On a 152-SM GB300 no problem needs more than about 9.5 MiB.
 *  - Set-up: the first call on a device looks up that device's copy of the array
 *    (with the device current); make that first call before any stream capture.
 *  - Sharing: every call on a device uses the same array, which keeps the last
 *    call's contents; each call clears what must start at zero (its counters) on
 *    `stream` before its kernel.  Calls that may run at the same time on the GPU
 *    (different streams without ordering between them) race on the array and
 *    must not be made; calls ordered on one stream are safe.
 * Results are those of tcm_gemm_ex_ws with a workspace of its own.
 */
tcm_status tcm_gemm_ex_builtin_ws(int64_t M, int64_t N, int64_t K,
                                  tcm_dtype a_dtype, const void *A, int64_t lda,
                                  tcm_dtype b_dtype, const void *B, int64_t ldb,
                                  const void *C, int64_t ldc, void *D, int64_t ldd,
                                  tcm_dtype out_dtype, float alpha, float beta,
                                  const float *a_scale, const float *b_scale, const void *bias,
                                  tcm_stream_t stream);

/*
 * tcm_gemm_fused -- tcm_gemm_ex with the rest of the epilogue chain:
 *   y   = act(alpha * sA * sB * (A . B) + beta * C + bias)
 *   D   = y * r, r = 1 / d_scale rounded once to fp32 (round to nearest even), then
 *         cast to out_dtype (FP8: round to nearest even, saturating to the largest
 *         finite value; 16/32-bit: RNE, d_scale not used)
 *   amax = max over all M x N outputs of |y| (before the division and the cast)
 *
 * "NVIDIA MMA", section "输入/累加/输出": the epilogue does scale / bias /
 * activation / cast, and FP8 outputs feed the next layer, whose per-tensor
 * scale comes from the amax of this one (delayed scaling).
 *  a_dtype .. bias   as tcm_gemm_ex, except: out_dtype may also be TCM_E4M3 or
 *                    TCM_E5M2, and then beta must be 0 (TCM_ERR_UNSUPPORTED
 *                    otherwise: there is no FP8 C) and bias is bf16[N].
 *                    ldd * sizeof(out) must be a multiple of 16.
 *  act               TCM_ACT_NONE, TCM_ACT_RELU or TCM_ACT_GELU; else
 *                    TCM_ERR_INVALID_ARG.
 *  d_scale           DEVICE pointer to one fp32 (dequantisation factor of D:
 *                    real value ~= stored value * d_scale), or NULL for 1.0.
 *                    Read only for FP8 outputs; D is y times its rounded
 *                    reciprocal (one reciprocal per launch, not one division
 *                    per element).
 *  The device product y * r is rounded to fp32 before the FP8 cast.
 *  amax              DEVICE pointer to one fp32, 4-byte aligned, or NULL.  The
 *                    call sets it to 0 on `stream` before the GEMM, then to the
 *                    maximum |y| (NaN if any y is NaN).
 */
tcm_status tcm_gemm_fused(int64_t M, int64_t N, int64_t K,
                          tcm_dtype a_dtype, const void *A, int64_t lda,
                          tcm_dtype b_dtype, const void *B, int64_t ldb,
                          const void *C, int64_t ldc, void *D, int64_t ldd,
                          tcm_dtype out_dtype, float alpha, float beta,
                          const float *a_scale, const float *b_scale, const void *bias,
                          tcm_activation act, const float *d_scale, float *amax,
                          tcm_stream_t stream);

/*
 * tcm_sp_compress -- prune a logical M x K matrix to 2:4 along K and compress it.
 *
 * Format: "NVIDIA MMA", section "稠密乘法与 2:4 结构化稀疏乘法" (each group of
 * 4 logical positions along K keeps 2 values plus their positions; the
 * worked example [a0,0,0,a3] -> values [a0,a3], metadata [0,3]) and
 * section "Ampere ..." (ordered metadata: positions ascending).
 * Selection: the two largest |v| of each group, ties to the lower position.
 *
 *  dtype      TCM_BF16 or TCM_F16.
 *  A          logical M x K row-major, pitch lda elements (lda >= K); K % 32 == 0.
 *  A_comp     output, M x K/2 row-major (pitch K/2): group g's kept values
 *             at columns 2g (lower position) and 2g+1.
 *  meta       output, M x K/32 uint32 row-major: group g's nibble
 *             (i0 | i1 << 2, i0 < i1) at bits 4*(g % 8) of word g/8.
 * Bit-exact: a pure selection, no arithmetic on the values.
 */
tcm_status tcm_sp_compress(int64_t M, int64_t K, tcm_dtype dtype,
                           const void *A, int64_t lda, void *A_comp, uint32_t *meta,
                           tcm_stream_t stream);

/*
 * tcm_sp_decompress -- inverse of tcm_sp_compress: writes the logical M x K
 * matrix (pitch lda) with +0 at the two dropped positions of every group.
 * `meta` must hold ascending nibbles as written by tcm_sp_compress.
 */
tcm_status tcm_sp_decompress(int64_t M, int64_t K, tcm_dtype dtype,
                             const void *A_comp, const uint32_t *meta, void *A, int64_t lda,
                             tcm_stream_t stream);

/*
 * tcm_gemm_sp -- D = alpha * (A' . B) + beta * C with A' the 2:4-sparse
 * logical matrix given by (A_comp, meta) in the tcm_sp_compress format.
 *
 * "NVIDIA MMA", section "稠密乘法与 2:4 结构化稀疏乘法": only A is compressed;
 * B, C and D are dense; shapes are stated on the logical K.
 *  dtype      TCM_BF16 or TCM_F16 (A_comp and B); K % 32 == 0.
 *  A_comp     M x K/2 row-major, meta M x K/32 uint32 (as tcm_sp_compress),
 *             both 16-byte aligned.
 *  B, C, D    as in tcm_gemm.
 * The kernel reads `meta` in this canonical layout and puts each stage's words
 * into the sparse MMA's tensor-memory order itself (the order described below
 * for tcm_sp_meta_pack), so no second metadata buffer is needed; the result is
 * bit-identical to tcm_gemm_sp_tc on the packed copy of the same metadata.
 * When K % 128 == 0 each stage's words (16 bytes of each row) are staged in
 * shared memory by TMA together with A and B; otherwise the kernel's metadata
 * threads load them from global memory.
 */
tcm_status tcm_gemm_sp(int64_t M, int64_t N, int64_t K, tcm_dtype dtype,
                       const void *A_comp, const uint32_t *meta, const void *B,
                       const void *C, void *D, float alpha, float beta,
                       tcm_dtype out_dtype, tcm_stream_t stream);

/*
 * Hardware-ordered 2:4 metadata.  "NVIDIA MMA", section "SM100：tcgen05.mma":
 * the sparse MMA reads its metadata from tensor memory; this layout is that
 * tensor-memory order (established on the GPU by a decoding probe), so the
 * kernel moves it in with one vector load and one tensor-memory store per
 * lane and stage instead of assembling it.
 *
 * For 128-row tile t and 128-logical-K stage kb a 2048-byte block at byte
 * offset (t * KBS + kb) * 2048, KBS = ceil(K / 128), holds for every lane
 * L = 16a + 8s + r (0 <= L < 128) at bytes 16 L + 4 k .. 16 L + 4 k + 3 the
 * word that the stage's MMA k (logical K 32, i.e. canonical word q = 4 kb + k
 * of each row) reads for lane L:
 *   bits  0..15 = nibbles 4s .. 4s+3 of row 128t + 16a + r's word q,
 *   bits 16..31 = the same nibbles of row 128t + 16a + 8 + r's word q.
 * Rows past M and words past K/32 read 0x44444444 (positions {0, 1}).
 *
 * tcm_sp_meta_tc_bytes -- ceil(M/128) * ceil(K/128) * 2048 (the size of the
 * canonical metadata, rounded up to whole tiles and stages); -1 if M < 0,
 * K < 0 or K % 32 != 0.  Host only.
 * tcm_sp_meta_pack -- write that layout from the canonical metadata of
 * tcm_sp_compress (M x K/32 uint32, device) into meta_tc (device, 16-byte
 * aligned, tcm_sp_meta_tc_bytes(M, K) bytes).  Bit-exact; asynchronous.
 * tcm_gemm_sp_tc -- tcm_gemm_sp with the metadata in this layout (same
 * arguments, same results).
 */
int64_t tcm_sp_meta_tc_bytes(int64_t M, int64_t K);
tcm_status tcm_sp_meta_pack(int64_t M, int64_t K, const uint32_t *meta, void *meta_tc, tcm_stream_t stream);
tcm_status tcm_gemm_sp_tc(int64_t M, int64_t N, int64_t K, tcm_dtype dtype,
                          const void *A_comp, const void *meta_tc, const void *B,
                          const void *C, void *D, float alpha, float beta,
                          tcm_dtype out_dtype, tcm_stream_t stream);

/*
 * tcm_gemm_mx -- block-scaled GEMM in an MX format, MXFP8 or MXFP4:
 *   D = alpha * sum_g (A_g * 2^(sa_g - 127)) . (B_g * 2^(sb_g - 127)) + beta * C + bias
 *
 * "NVIDIA MMA", section "SM100：tcgen05.mma" (block-scaled form: each K block's
 * partial sum is scaled by the A and B block scales before it is accumulated)
 * and section "MXFP4 与 NVFP4" (MX formats: one UE8M0 scale per 32 elements;
 * kernels follow a scale layout contract, which is the blocked layout below).
 *  a_dtype, b_dtype  MXFP8: TCM_E4M3 or TCM_E5M2 (any pair).  MXFP4: both TCM_E2M1
 *                    (packed two per byte, element 2i in the low nibble; section "MXFP4
 *                    与 NVFP4": MXFP4 = E2M1 elements with a UE8M0 scale per 32), then K
 *                    must be a multiple of 256 (else TCM_ERR_INVALID_ARG).  E2M1 with an
 *                    FP8 type: TCM_ERR_UNSUPPORTED.
 *  A                 M x K row-major (pitch K), B N x K (pitch K): the elements (E2M1:
 *                    rows of K/2 bytes).
 *  a_scales          E8M0 scale codes (value 2^(code - 127); 255 is NaN) of the
 *                    32-element blocks of the rows of A, in the BLOCKED layout
 *                    written by tcm_mx_pack_scales (tcm_mx_scales_bytes(M, K)
 *                    bytes); b_scales likewise for the N rows of B.
 *  K                 a multiple of 32.
 *  C, D, bias        as in tcm_gemm_ex with packed pitches (C, D: N; bias: N).
 * All pointers 16-byte aligned; N * sizeof(out) a multiple of 16.
 */
tcm_status tcm_gemm_mx(int64_t M, int64_t N, int64_t K,
                       tcm_dtype a_dtype, const void *A, const uint8_t *a_scales,
                       tcm_dtype b_dtype, const void *B, const uint8_t *b_scales,
                       const void *C, void *D, float alpha, float beta, const void *bias,
                       tcm_dtype out_dtype, tcm_stream_t stream);

/*
 * Blocked scale layout of tcm_gemm_mx.  For `rows` rows of K elements
 * (K % 32 == 0) the codes of row r, 32-block j (row-major code index
 * r * K/32 + j) live in 512-byte atoms, one per 128 rows x 4 blocks:
 *   atom (t, k) = (r / 128, j / 4) at byte (t * KT + k) * 512, KT = ceil(K / 128),
 *   byte inside the atom: (r % 32) * 16 + ((r / 32) % 4) * 4 + j % 4.
 * Positions of rows >= rows or blocks >= K/32 hold code 127 (1.0).  This is
 * the tensor-memory scale layout of the block-scaled tcgen05.mma, one atom per
 * 32 x 128-bit tcgen05.cp.
 *
 * tcm_mx_scales_bytes -- size of the blocked array: ceil(rows/128) *
 * ceil(K/128) * 512; -1 if rows < 0, K < 0 or K % 32 != 0.  Host only.
 */
int64_t tcm_mx_scales_bytes(int64_t rows, int64_t K);

/*
 * tcm_mx_pack_scales -- write the blocked layout from row-major codes.
 *  scales  device, rows x K/32 uint8 row-major (pitch K/32), caller-owned.
 *  packed  device, tcm_mx_scales_bytes(rows, K) bytes, 16-byte aligned, caller-owned.
 * Bit-exact (a permutation plus the 127 padding).  rows == 0 or K == 0 launches
 * nothing.  Asynchronous on `stream`.
 */
tcm_status tcm_mx_pack_scales(int64_t rows, int64_t K, const uint8_t *scales, uint8_t *packed,
                              tcm_stream_t stream);

/*
 * tcm_gemm_nvfp4 -- block-scaled FP4 GEMM (NVFP4):
 *   D = alpha * sum_g (A_g * sa_g) . (B_g * sb_g) + beta * C + bias
 * with A (M x K) and B (N x K) in FP4 E2M1 and one UE4M3 scale per 16
 * consecutive K elements of every row; alpha carries the product of the two
 * per-tensor fp32 scales of the NVFP4 format.
 *
 * "NVIDIA MMA", section "SM100：tcgen05.mma" (kind::mxf4nvf4: MXFP4 or NVFP4,
 * each K block's partial sum scaled before accumulation) and section
 * "MXFP4 与 NVFP4" (NVFP4: E2M1 elements, UE4M3 scale per 16 elements);
 * section "量化配置如何映射到 MMA": W4A4 NVFP4 x NVFP4 -> FP32.
 *  A, B              packed E2M1, two per byte (element 2i in the low nibble),
 *                    rows of K/2 bytes; K a multiple of 256 (else
 *                    TCM_ERR_INVALID_ARG).
 *  a_scales, b_scales  UE4M3 codes (E4M3 without sign; 0x7F is NaN) in the
 *                    blocked layout of tcm_nvfp4_pack_scales
 *                    (tcm_nvfp4_scales_bytes(rows, K) bytes).
 *  C, D, bias, alpha, beta, out_dtype  as tcm_gemm_mx.
 */
tcm_status tcm_gemm_nvfp4(int64_t M, int64_t N, int64_t K,
                          const void *A, const uint8_t *a_scales,
                          const void *B, const uint8_t *b_scales,
                          const void *C, void *D, float alpha, float beta, const void *bias,
                          tcm_dtype out_dtype, tcm_stream_t stream);

/*
 * NVFP4 scales use the same 512-byte atoms as tcm_gemm_mx with 16-element
 * blocks: the code of row r, block j (row-major index r * K/16 + j) is at
 * atom (r / 128, j / 4) = byte offset (t * KT + k) * 512 with KT = ceil(K / 64),
 * byte (r % 32) * 16 + ((r / 32) % 4) * 4 + j % 4 inside it; padding holds
 * 0x38 (1.0).  One atom is the tensor-memory scale operand of one K = 64
 * block-scaled MMA (scale_vec::4X; probed on the GPU).
 *
 * tcm_nvfp4_scales_bytes -- ceil(rows/128) * ceil(K/64) * 512; -1 if rows < 0,
 * K < 0 or K % 16 != 0.  Host only.
 * tcm_nvfp4_pack_scales -- blocked layout from row-major codes (rows x K/16,
 * device, caller-owned) into `packed` (device, 16-byte aligned, caller-owned);
 * bit-exact; asynchronous on `stream`.
 */
int64_t tcm_nvfp4_scales_bytes(int64_t rows, int64_t K);
tcm_status tcm_nvfp4_pack_scales(int64_t rows, int64_t K, const uint8_t *scales, uint8_t *packed,
                                 tcm_stream_t stream);

/*
 * tcm_gemm_i8 -- D = satfinite_int32(A . B + C) for signed 8-bit A and B, exact.
 *
 * "NVIDIA MMA", section "SM100：tcgen05.mma" lists kind::i8 (8-bit integer operands,
 * 32-bit integer accumulator) and section "Ampere：FP16/BF16 与整数 MMA 基线" the
 * integer semantics (.satfinite: the result clamped to the int32 range instead of
 * wrapping).  ptxas does not accept kind::i8 for sm_103a, so this runs on the bf16
 * tensor path with the same results: int8 values are exact in bf16, and every 1024-long
 * K chunk is accumulated in fp32 on its own (its partial sums are integers below 2^24,
 * exact), converted to int32 and added; + C saturates.
 *  M, N >= 1; 0 <= K <= 131071 (else TCM_ERR_UNSUPPORTED: the int32 sums of A . B
 *              alone then cannot overflow).
 *  A           M x K int8, row pitch lda bytes (>= K, any alignment).
 *  B           N x K int8 (the K x N operand stored K-major), pitch ldb bytes (>= K).
 *  C           M x N int32, pitch ldc elements (multiple of 4, base 16-byte aligned), or NULL.
 *  D           M x N int32, pitch ldd elements (multiple of 4, base 16-byte aligned).
 *  workspace   DEVICE memory, 16-byte aligned, at least tcm_gemm_i8_workspace_bytes(M, N, K)
 *              bytes (the bf16 copies of A and B, rows of K rounded up to 64); scratch.
 * Three launches on `stream`: the two conversions and the GEMM (256 x 256 CTA-pair tiles).
 *
 * tcm_gemm_i8_workspace_bytes -- (M + N) * ceil(K / 64) * 64 * 2; -1 if the sizes are
 * rejected.  Host only.
 */
int64_t tcm_gemm_i8_workspace_bytes(int64_t M, int64_t N, int64_t K);
tcm_status tcm_gemm_i8(int64_t M, int64_t N, int64_t K, const int8_t *A, int64_t lda,
                       const int8_t *B, int64_t ldb, const int32_t *C, int64_t ldc,
                       int32_t *D, int64_t ldd, void *workspace, int64_t workspace_bytes,
                       tcm_stream_t stream);

/*
 * tcm_get_device_status -- synchronise `stream`, then report the first
 * device-side failure recorded since the last tcm_clear_device_status():
 * *code = TCM_OK or TCM_ERR_TIMEOUT, *site = which pipeline wait gave up
 * (1 = loader waiting for a free stage, 2 = MMA issuer waiting for data,
 * 3 = MMA issuer waiting for a free accumulator, 4 = epilogue waiting for
 * an accumulator, 5 = drain at exit, 6 = MMA issuer waiting for a stage's
 * scales or sparse metadata, 7 = sparse metadata writer waiting for a free
 * stage, 10 = tcm_gemm_ex_ws part 0 waiting for the other parts' partial sums).
 * Returns TCM_ERR_CUDA if the
 * synchronisation itself failed.  Either output pointer may be NULL.
 */
tcm_status tcm_get_device_status(tcm_stream_t stream, int32_t *code, int32_t *site);

/* Reset the recorded device status of the current device to TCM_OK (synchronous). */
tcm_status tcm_clear_device_status(void);

/*
 * Limit, in nanoseconds of the GPU's global timer, for any single pipeline
 * wait inside the kernels of this library (default 2e9, i.e. 2 s; also read
 * from the environment variable TCM_TIMEOUT_NS at first use).  0 restores
 * the default.  Affects launches made after the call.
 */
void tcm_set_timeout_ns(uint64_t ns);

/*
 * Tuning / testing knob for later GEMM launches in this process (0 keeps the
 * automatic choice for that field):
 *   cta_group  1 = one CTA per 128-row tile, 2 = a CTA pair per 256-row tile
 *   tile_n     tile width in columns (dense: 32, 64, 128, 256; sparse: 128, 256)
 *   stages     depth of the shared-memory ring (the kernels provide a few
 *              depths per tile; others fall back to the default)
 *   group_m    row blocks per rasterisation group (tiles that run at the same
 *              time share rows of A and columns of B in L2)
 *   ksplit     1, 2 or 4 CTAs of a cluster sharing each tile's K range, their
 *              partial sums added through distributed shared memory (dense
 *              single-CTA tiles of width 32 or 64, e.g. skinny M)
 *   tail_split tcm_gemm_ex_ws with a workspace: 1 = never split the last round's
 *              CTA-pair tiles over K; 2 = split them whenever every pair then gets
 *              at most one part (automatic: also only when a tile has at least 64
 *              K blocks of 128 bytes, i.e. K >= 4096 for 16-bit, K >= 8192 for FP8)
 * Combinations the kernels do not provide fall back to the automatic choice.
 * Results are the same either way, up to the order of the fp32 accumulation.
 */
void tcm_set_config_override(int cta_group, int tile_n, int stages, int group_m, int ksplit, int tail_split);

/*
 * Measurement hook: while `counters` is set, every GEMM launch made afterwards
 * adds, from its first CTA, the SM clock cycles (%clock64) and global-timer
 * nanoseconds between that CTA's start and end to counters[0] and counters[1],
 * and 1 to counters[2] (atomically; DEVICE memory, three uint64, caller-owned).
 * counters[0] / counters[1] is then the SM clock in GHz during those launches.
 * NULL turns it off.  The pointer is read when a launch is made.
 */
void tcm_set_clock_probe(unsigned long long *counters);

/*
 * Test hook for the device-side failure path: with mask bit 1 set, the next
 * GEMM launch of tcm_gemm / tcm_gemm_ex / tcm_gemm_fused, tcm_gemm_mx,
 * tcm_gemm_nvfp4, tcm_gemm_sp or tcm_gemm_sp_tc (only that one) has its loader
 * skip the first shared-memory stage, so the waits for that stage run out after
 * the time limit (tcm_set_timeout_ns): the kernel records TCM_ERR_TIMEOUT at the
 * site of the first wait to give up (2: the MMA issuer or a side-data thread
 * waiting for data; 4: the epilogue waiting for the same tile; 6: the MMA
 * issuer waiting for the stage's scales or metadata in tensor memory; 7: a
 * metadata writer of tcm_gemm_sp waiting for a stage's previous MMAs), winds
 * down and returns.  With mask bit 2 set, the next tcm_gemm_ex_ws launch that
 * splits tiles has its helper parts skip announcing their partial sums, so each
 * owner's wait runs out (site 10).  D is left partly unwritten.  No memory outside the
 * kernel's own buffers is touched.
 */
void tcm_debug_fail_next_launch(int mask);

/* Human-readable name of a status code (static storage). */
const char *tcm_status_string(tcm_status status);

/* Library version, major * 10000 + minor * 100 + patch. */
int tcm_version(void);

#ifdef __cplusplus
}
#endif

#endif /* TCM_H */
