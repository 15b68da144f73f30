// tcm_gemm_mx.cu -- block-scaled GEMM (MXFP8: E4M3/E5M2 elements, one E8M0
// scale per 32 consecutive K elements of every row of A and of B, on
// tcgen05.mma.kind::mxf8f6f4.block_scale; NVFP4: packed E2M1 with UE4M3 scales
// per 16, on kind::mxf4nvf4.block_scale.scale_vec::4X), the same pipeline with
// 2:4-sparse A and hardware-ordered metadata (tcgen05.mma.sp), and the packing
// of row-major scales into the blocked layout the kernel reads.
//
// "NVIDIA MMA", section "SM100：tcgen05.mma": the block-scaled form reads the
// scales of A and B from tensor memory ([scale-A-tmem], [scale-B-tmem]) and
// computes D = C + sum_g (A_{q,g} S_{A,g}) (B_{q,g} S_{B,g}), each K block's
// partial sum scaled before it is accumulated; section "MXFP4 与 NVFP4": MX
// formats carry UE8M0 scales per block of 32; the same section notes that a
// kernel must meet a scale layout ("swizzle") contract, which the pages do not
// spell out -- the blocked layout below is this library's.
//
// Scale layout in tensor memory (established on the GPU by decoding probes,
// 0 mismatches): the scale of operand row r for the MMA whose scale-factor id
// is j is byte j of TMEM column (base + r / 32), lane r % 32 of the 32-lane
// quadrant the output row belongs to, the same 32 x 4-column block being read
// by all four quadrants.  For a CTA pair (cta_group::2, 256-row tile) each CTA
// reads the A scales of its own 128 rows and the B scales of all BN columns
// from its own tensor memory, in the same layout.
//
// tcgen05.cp.32x128b.warpx4 copies a 32-row x 16-byte shared-memory block to
// four TMEM columns of lanes 0..31 of every quadrant (row l -> lane l, bytes
// 4q..4q+3 -> column q; probed, and the cta_group::2 form issued by the even
// CTA copies each CTA's own shared memory into its own tensor memory).  So a
// 512-byte "scale atom" holding, for 128 rows and one 128-element K stage,
// byte (r % 32) * 16 + (r / 32) * 4 + j = scale of row r, 32-block j, becomes
// the MMA's scale operand with one copy.  The blocked global layout is a
// sequence of such atoms, atom (row tile t, K stage k) at byte offset
// (t * KT + k) * 512, KT = ceil(K / 128); tcm_mx_pack_scales writes it from
// row-major codes.
//
// Pipeline: the dense kernel's (TMA ring of 128-byte K stages = 128 FP8 values,
// four MMAs of K = 32 per stage, one thread issuing, TMEM accumulators).  The
// same TMA producer loads the stage's scale atoms first (in 128-byte rows: the
// atoms are contiguous, and 16-byte rows made hundreds of small TMA requests per
// stage), onto a barrier of their own (sfull), then A and B onto the stage's full
// barrier.  Copy threads
// (lane 0 of warps MX_COPY_WARP ..) copy the atoms to tensor memory
// (tcgen05.cp) as soon as they land, while A and B are still in flight, and
// commit their copies to the stage's sfready barrier; the MMA thread waits on
// sfready and full before the stage's MMAs.  Copies issued by threads other
// than the MMA thread proceed alongside the MMAs, and the issue of a copy
// costs its thread tens of cycles, so NVFP4's twelve copies per stage are
// split over three threads.  Measured at 8192^3 against one thread issuing
// the copies between its MMAs: NVFP4 2913 -> 4605 TFLOP/s, MXFP8 2597 -> 2843.
// The scale columns of a stage are rewritten only after the stage's sfull
// barrier has completed again, which the producer allows only after the MMAs
// that read them have finished.  The sparse format has no copies: four writer
// warps per CTA, one per TMEM lane quadrant, store each stage's compact
// metadata with tcgen05.st (see FMT_SP below).
//
// One accumulator of 256 columns fills half of tensor memory and the scale
// columns take part of the rest, so a 256-wide tile has a single accumulator
// buffer; for 16-bit outputs without C the epilogue converts while it drains
// tensor memory and frees it before its global stores, shortening the gap
// before the next tile's MMAs.
#include "tcm_kernel_common.cuh"

namespace tcm {

constexpr int MX_EPI_WARPS = 8; // two per TMEM lane quadrant, half the columns each
constexpr int MX_COPY_WARP = 2 + MX_EPI_WARPS; // first side-data (copy or writer) warp
constexpr int SF_ATOM = 512;                       // scales of 128 rows x one 128-value K stage

// Formats of the kernel: MX (MXFP8), NV (NVFP4), SP (2:4-sparse bf16/fp16 A,
// metadata in the hardware order -- the "side" data of a stage is then the
// sparse metadata instead of block scales).
// SPC: 2:4-sparse A with the canonical metadata of tcm_sp_compress (K % 128 == 0): TMA
// stages each stage's words of the tile's rows with its A and B, and the writer warps put
// them into the hardware order.  SPG: the same for any K % 32 == 0, the writer warps loading
// the words from global memory themselves (a row pitch that is no multiple of 16 bytes
// admits no tensor map).  The two are separate instantiations: the global-load writer
// compiled into the TMA-fed kernel cost it 2 %.
// MXF4: MXFP4, packed E2M1 with one E8M0 scale per 32 (kind::mxf4nvf4.scale_vec::2X).
enum SideFmt : int { FMT_MX = 0, FMT_NV = 1, FMT_SP = 2, FMT_SPC = 3, FMT_MXF4 = 4, FMT_SPG = 5 };
__host__ __device__ constexpr bool is_sparse(int fmt) { return fmt == FMT_SP || fmt == FMT_SPC || fmt == FMT_SPG; }
// sparse formats whose metadata TMA stages in shared memory
__host__ __device__ constexpr bool meta_by_tma(int fmt) { return fmt == FMT_SP || fmt == FMT_SPC; }
// Side-data warps per format.  MX, NV: copy warps (lane 0 of each issues the copies e
// with e % n == its index).  SP, SPC, SPG: one writer warp per TMEM lane quadrant (warp % 4).
__host__ __device__ constexpr int mx_copy_warps(int fmt)
{
    return fmt == FMT_NV ? 3 : is_sparse(fmt) ? 4 : fmt == FMT_MXF4 ? 2 : 1;
}
// scale atoms per 128-row tile per stage: MX one (4 blocks of 32 over 128 FP8 values),
// NVFP4 four (one per K = 64 MMA, blocks of 16), MXFP4 two (4 blocks of 32 each; a stage
// is 256 packed E2M1 values)
__host__ __device__ constexpr int mx_atoms_per_tile(int fmt) { return fmt == FMT_NV ? 4 : fmt == FMT_MXF4 ? 2 : 1; }
constexpr uint32_t SP_META_FILL = 0x44444444u; // positions {0, 1} in every group (rows / words past the matrix)
// TMA, MMA, epilogue (warps 2..9), copy warps
__host__ __device__ constexpr int mx_threads(int fmt) { return 32 * (2 + MX_EPI_WARPS + mx_copy_warps(fmt)); }
constexpr int SP_META_STAGE = 2048; // 128 lanes x 16 bytes: lane L's words for the stage's four MMAs

template <int BN_CTA, int BN, int STAGES, int FMT>
struct MxSmem {
    static constexpr int B_STAGE = BN_CTA * TILE_K_BYTES * (is_sparse(FMT) ? 2 : 1); // 128 logical K = 2 atoms
    static constexpr int SF_STAGE = FMT == FMT_SPG         ? 0
                                    : meta_by_tma(FMT)       ? SP_META_STAGE
                                                             : SF_ATOM * mx_atoms_per_tile(FMT) * (1 + BN / 128);
    static constexpr int A_OFF = 0;
    static constexpr int B_OFF = STAGES * A_STAGE_BYTES;
    static constexpr int SF_OFF = B_OFF + STAGES * B_STAGE;
    static constexpr int BAR_OFF = SF_OFF + STAGES * SF_STAGE;
    // full, empty, tfull[2], tempty[2], drain, sfready[STAGES], the copy threads' drain, sfull[STAGES]
    static constexpr int NUM_BARS = 4 * STAGES + 6;
    static constexpr int MISC_OFF = BAR_OFF + NUM_BARS * 8;
    static constexpr int BYTES = MISC_OFF + 16;
    static constexpr int ALLOC = BYTES + 1024;
};

// Two values rounded to nearest-even in the 16-bit output format, packed low/high.
__device__ __forceinline__ uint32_t pack2(float lo, float hi, int fmt)
{
    if (fmt == OUT_BF16) {
        const __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<const uint32_t *>(&b);
    }
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&h);
}

// Stores a warp's 32 rows (lane l holds row row0 + l, NCH 16-byte chunks of packed
// 16-bit outputs starting at column col0) so that each instruction writes whole
// 32-byte sectors: lanes 2j and 2j + 1 exchange one chunk and then write chunks
// q, q + 1 of row 2j together, then of row 2j + 1 (rows at or past kM are skipped).
// The stores are marked streaming (evict first), so that the output passing through
// L2 displaces less of A and B (measured: NVFP4 8192^3 +5 %, sparse +2.4 %).
template <int NCH>
__device__ __forceinline__ void store_rows_paired(uint16_t *D, long long ldd, int row, int kM, int col0,
                                                  const uint32_t (&packed)[4 * NCH])
{
    static_assert(NCH % 2 == 0, "chunk pairs");
    const int lane = threadIdx.x & 31;
    const bool odd = lane & 1;
    const int row_even = row - (odd ? 1 : 0);
    uint16_t *const r0 = D + static_cast<long long>(row_even) * ldd + col0;
    uint16_t *const r1 = r0 + ldd;
#pragma unroll
    for (int q = 0; q < NCH; q += 2) {
        const uint4 c0 = make_uint4(packed[4 * q], packed[4 * q + 1], packed[4 * q + 2], packed[4 * q + 3]);
        const uint4 c1 = make_uint4(packed[4 * q + 4], packed[4 * q + 5], packed[4 * q + 6], packed[4 * q + 7]);
        const uint4 send = odd ? c0 : c1; // even lane gives its chunk q + 1, odd lane its chunk q
        uint4 recv;
        recv.x = __shfl_xor_sync(0xffffffffu, send.x, 1);
        recv.y = __shfl_xor_sync(0xffffffffu, send.y, 1);
        recv.z = __shfl_xor_sync(0xffffffffu, send.z, 1);
        recv.w = __shfl_xor_sync(0xffffffffu, send.w, 1);
        const int c = 8 * (q + (odd ? 1 : 0)); // column of this lane's chunk
        if (row_even < kM) __stcs(reinterpret_cast<uint4 *>(r0 + c), odd ? recv : c0);
        if (row_even + 1 < kM) __stcs(reinterpret_cast<uint4 *>(r1 + c), odd ? c1 : recv);
    }
}

// Shared-memory descriptor of a 32-row x 16-byte block without swizzle:
// core matrices of 8 rows x 16 bytes, 128 bytes apart.
__device__ __forceinline__ uint64_t sdesc_sf_atom(uint32_t smem_addr)
{
    uint64_t d = 0;
    d |= static_cast<uint64_t>((smem_addr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>(128 >> 4) << 16;
    d |= static_cast<uint64_t>(128 >> 4) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    return d;
}

template <int CG>
__device__ __forceinline__ void tmem_cp_sf(uint32_t taddr, uint64_t sdesc)
{
    if constexpr (CG == 2)
        asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
    else
        asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

template <int CG>
__device__ __forceinline__ void mma_mx(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                       uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate)
{
    if constexpr (CG == 2)
        asm volatile(
            "{\n"
            ".reg .pred p;\n"
            "setp.ne.b32 p, %6, 0;\n"
            "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale [%0], %1, %2, %3, [%4], [%5], p;\n"
            "}\n" ::"r"(d_tmem),
            "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
            : "memory");
    else
        asm volatile(
            "{\n"
            ".reg .pred p;\n"
            "setp.ne.b32 p, %6, 0;\n"
            "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale [%0], %1, %2, %3, [%4], [%5], p;\n"
            "}\n" ::"r"(d_tmem),
            "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
            : "memory");
}

template <int CG>
__device__ __forceinline__ void mma_nvf4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate)
{
    if constexpr (CG == 2)
        asm volatile(
            "{\n"
            ".reg .pred p;\n"
            "setp.ne.b32 p, %6, 0;\n"
            "tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n"
            "}\n" ::"r"(d_tmem),
            "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
            : "memory");
    else
        asm volatile(
            "{\n"
            ".reg .pred p;\n"
            "setp.ne.b32 p, %6, 0;\n"
            "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n"
            "}\n" ::"r"(d_tmem),
            "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
            : "memory");
}

// Scale formats of the block-scaled kernel.  MX: MXFP8 (kind::mxf8f6f4, K = 32 per
// MMA, one E8M0 atom per 128 rows per stage shared by the stage's four MMAs
// through scale-factor ids 0..3).  NV: NVFP4 (kind::mxf4nvf4.scale_vec::4X, packed
// E2M1, K = 64 per MMA, one UE4M3 atom per 128 rows per MMA, scale-factor id 0).
// SP: no copies; the stage's 16 columns hold MMA k's metadata word at column 4k,
// a multiple of 4 as the sparse MMA's metadata address requires, written by the
// writer warps with tcgen05.st.
// MXF4: two atoms per tile per stage; MMA k (K = 64, blocks 2k and 2k + 1 of the stage)
// reads atom k / 2, scale-factor id 2 (k % 2) selecting bytes 2 (k % 2) .. +1 of each
// row's scale word (scale_vec::2X), the atoms laid out as NVFP4's.
template <int FMT, int SFB_ATOMS>
struct SfLayout {
    static constexpr int APT = mx_atoms_per_tile(FMT); // atoms per 128-row tile per stage
    static constexpr bool MA = APT > 1;                // NVFP4, MXFP4: several atoms per stage
    static constexpr int NCP = is_sparse(FMT) ? 0 : APT * (1 + SFB_ATOMS);  // copies per stage
    static constexpr uint32_t COLS = MA ? 4u * APT * (1u + SFB_ATOMS) : 16u; // TMEM columns per stage
    // TMEM column (within the stage) of copy e: e = tile * APT + kk, tile 0 = A, 1.. = B row tiles
    __device__ static constexpr uint32_t col(int e)
    {
        return MA ? (e < APT ? 4u * e : 4u * APT + 4u * SFB_ATOMS * static_cast<uint32_t>((e - APT) % APT) +
                                             4u * static_cast<uint32_t>((e - APT) / APT))
                  : (e == 0 ? 0u : 4u + 4u * e);
    }
    // byte offset of copy e's source within the stage's side data
    __device__ static constexpr uint32_t src(int e) { return static_cast<uint32_t>(SF_ATOM) * e; }
    // atom of the stage that MMA k reads
    __device__ static constexpr uint32_t atom(int k) { return FMT == FMT_NV ? k : FMT == FMT_MXF4 ? k / 2 : 0; }
    __device__ static constexpr uint32_t sfa(int k) { return MA ? 4u * atom(k) : 0u; }
    __device__ static constexpr uint32_t sfb(int k) { return MA ? 4u * APT + 4u * SFB_ATOMS * atom(k) : 8u; }
};

template <int CG>
__device__ __forceinline__ void tmem_cp_side(uint32_t taddr, uint32_t smem_addr)
{
    tmem_cp_sf<CG>(taddr, sdesc_sf_atom(smem_addr));
}

template <int CG>
__device__ __forceinline__ void mma_sp16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t meta_tmem,
                                         uint32_t idesc, uint32_t accumulate)
{
    if constexpr (CG == 2)
        asm volatile(
            "{\n"
            ".reg .pred p;\n"
            "setp.ne.b32 p, %5, 0;\n"
            "tcgen05.mma.sp.cta_group::2.kind::f16 [%0], %1, %2, [%3], %4, p;\n"
            "}\n" ::"r"(d_tmem),
            "l"(adesc), "l"(bdesc), "r"(meta_tmem), "r"(idesc), "r"(accumulate)
            : "memory");
    else
        asm volatile(
            "{\n"
            ".reg .pred p;\n"
            "setp.ne.b32 p, %5, 0;\n"
            "tcgen05.mma.sp.cta_group::1.kind::f16 [%0], %1, %2, [%3], %4, p;\n"
            "}\n" ::"r"(d_tmem),
            "l"(adesc), "l"(bdesc), "r"(meta_tmem), "r"(idesc), "r"(accumulate)
            : "memory");
}

// The four canonical 2:4 metadata words of `row` for 128-logical-K stage kb (words
// 4kb .. 4kb+3 of the row, tcm_sp_compress layout: qn words per row), the fill code
// for rows or words past the matrix.  vec: rows hold whole stages (qn % 4 == 0, the
// base 16-byte aligned), so the four words are one 16-byte load.
__device__ __forceinline__ uint4 sp_meta_words(const uint32_t *meta, long long qn, int rows, int row, int kb, bool vec)
{
    const long long q0 = 4ll * kb;
    if (row >= rows) return make_uint4(SP_META_FILL, SP_META_FILL, SP_META_FILL, SP_META_FILL);
    const uint32_t *src = meta + static_cast<long long>(row) * qn + q0;
    if (vec) return __ldg(reinterpret_cast<const uint4 *>(src));
    uint32_t w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) w[k] = q0 + k < qn ? __ldg(src + k) : SP_META_FILL;
    return make_uint4(w[0], w[1], w[2], w[3]);
}

template <int CG>
__device__ __forceinline__ void mma_mxf4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate)
{
    if constexpr (CG == 2)
        asm volatile(
            "{\n"
            ".reg .pred p;\n"
            "setp.ne.b32 p, %6, 0;\n"
            "tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], [%5], p;\n"
            "}\n" ::"r"(d_tmem),
            "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
            : "memory");
    else
        asm volatile(
            "{\n"
            ".reg .pred p;\n"
            "setp.ne.b32 p, %6, 0;\n"
            "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], [%5], p;\n"
            "}\n" ::"r"(d_tmem),
            "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
            : "memory");
}

// One TMA tile load onto this stage's barrier (pair: the even CTA's barrier, cluster address fb).
template <int CG>
__device__ __forceinline__ void tma_ld(uint32_t dst, const CUtensorMap *map, uint64_t *bar, uint32_t fb, int x, int y)
{
    if constexpr (CG == 2) tma_load_2d_pair(dst, map, fb, x, y);
    else tma_load_2d(dst, map, bar, x, y);
}

// BN: N extent of the (pair) tile; CG: 1 = one CTA per 128 x BN tile, 2 = a CTA
// pair per 256 x BN tile (each CTA loads 128 rows of A and BN/2 rows of B, its
// own A scale atom and all BN/128 B scale atoms).
template <int BN, int STAGES, int NACC, int CG, int FMT>
__global__ void __launch_bounds__(mx_threads(FMT), 1)
    gemm_mx_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmSA, const __grid_constant__ CUtensorMap tmSB,
                   const GemmParams p)
{
    const unsigned long long clk0 = clock64(); // clock probe (CTA 0, thread 0 only)
    const unsigned long long gt0 = globaltimer_ns();
    constexpr int BN_CTA = BN / CG;
    constexpr int SFB_ATOMS = BN / 128;
    using SF = SfLayout<FMT, SFB_ATOMS>;
    constexpr int APT = SF::APT;
    using L = MxSmem<BN_CTA, BN, STAGES, FMT>;
    static_assert(L::ALLOC <= 227 * 1024, "shared memory ring too large");
    static_assert(BN == 128 || BN == 256, "tile width");
    constexpr uint32_t ACC_STRIDE = BN;            // BN is a power of two here
    constexpr uint32_t SF_COL = ACC_STRIDE * NACC; // then SF::COLS scale columns per stage
    constexpr uint32_t SF_STAGE_COLS = SF::COLS;
    static_assert(SF_COL + SF_STAGE_COLS * STAGES <= 512, "tensor memory budget");
    constexpr uint32_t TMEM_COLS = 512;
    constexpr uint32_t STAGE_TX = CG * (A_STAGE_BYTES + L::B_STAGE); // A and B of both CTAs
    constexpr uint32_t SIDE_TX = CG * L::SF_STAGE;                     // side data of both CTAs
    constexpr int NCW = mx_copy_warps(FMT);
    constexpr int EPI_COLS = BN / (MX_EPI_WARPS / 4); // columns per epilogue warp

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    const uint32_t sbase = smem_u32(smem);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L::BAR_OFF);
    uint64_t *empty = full + STAGES;
    uint64_t *tfull = empty + STAGES;
    uint64_t *tempty = tfull + 2;
    uint64_t *drain = tempty + 2;
    uint64_t *sfready = drain + 1;       // a stage's side data copied to tensor memory
    uint64_t *cdrain = sfready + STAGES; // the copy threads' last copies done
    uint64_t *sfull = cdrain + 1;        // a stage's side data landed in shared memory
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::MISC_OFF);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::MISC_OFF + 4);

    const int warp = __shfl_sync(0xffffffffu, static_cast<int>(threadIdx.x >> 5), 0);
    const int lane = threadIdx.x & 31;
    const uint32_t rank = CG == 2 ? cluster_ctarank() : 0u;
    const bool leader = rank == 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, 1);
        }
        for (int a = 0; a < NACC; ++a) {
            mbar_init(tfull + a, 1);
            mbar_init(tempty + a, MX_EPI_WARPS * CG);
        }
        mbar_init(drain, 1);
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(sfready + s, is_sparse(FMT) ? NCW * CG : NCW); // sparse: writer warps of both CTAs
            mbar_init(sfull + s, 1);
        }
        mbar_init(cdrain, NCW);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0 && p.num_kb > 0) { // K == 0: the maps are not encoded
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        if (FMT != FMT_SPG) tma_prefetch_desc(&tmSA);
        if (!is_sparse(FMT)) tma_prefetch_desc(&tmSB);
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
    if (CG == 2) cluster_sync();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    const Waiter w{abort_flag, p.timeout_ns, p.status};
    const int first_tile = p.tile_begin + static_cast<int>(blockIdx.x) / CG;
    const int step = static_cast<int>(gridDim.x) / CG;

    if (warp == 0) {
        if (lane == 0) {
            const uint32_t full_cluster0 = CG == 2 ? mapa_shared(smem_u32(full), 0) : 0u;
            const uint32_t sfull_cluster0 = CG == 2 ? mapa_shared(smem_u32(sfull), 0) : 0u;
            const int kt = p.num_kb * APT; // scale atoms per 128-row tile along K
            // sparse metadata by TMA onto this CTA's own side-data barrier: hardware-ordered
            // blocks (SP) or canonical rows (SPC)
            constexpr bool meta_tma = meta_by_tma(FMT);
            int stage = 0;
            uint32_t phase = 0;
            long long issued = 0;
            bool ok = true;
            for (int t = first_tile; ok && t < p.tile_end; t += step) {
                int mb, nb;
                tile_coords(p, t, mb, nb);
                const int a_tile = mb * CG + static_cast<int>(rank); // 128-row tile of A
                const int a_row = a_tile * BM;
                const int b_row = nb * BN + static_cast<int>(rank) * BN_CTA;
                for (int kb = 0; kb < p.num_kb; ++kb) {
                    if (!wait_bar<CG>(empty + stage, phase ^ 1u, w, SITE_LOAD_EMPTY, true)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sa = sbase + L::A_OFF + stage * A_STAGE_BYTES;
                    const uint32_t sb = sbase + L::B_OFF + stage * L::B_STAGE;
                    const uint32_t ss = sbase + L::SF_OFF + stage * L::SF_STAGE;
                    // test hook: the first stage is never issued nor announced, so its waits run out
                    if ((p.fault_inject & FAULT_SKIP_FIRST_LOAD) && issued == 0) {
                        ++issued;
                        if (++stage == STAGES) {
                            stage = 0;
                            phase ^= 1u;
                        }
                        continue;
                    }
                    // sparse: each CTA's metadata lands on its own side-data barrier (its writer
                    // warps wait there); scales: both CTAs' atoms on the even CTA's (its copy threads)
                    if (meta_tma) mbar_arrive_expect_tx(sfull + stage, L::SF_STAGE);
                    else if (!is_sparse(FMT) && (leader || CG == 1)) mbar_arrive_expect_tx(sfull + stage, SIDE_TX);
                    if (leader || CG == 1) mbar_arrive_expect_tx(full + stage, STAGE_TX);
                    // pair: both CTAs' loads complete on the even CTA's barriers (cluster addresses)
                    const uint32_t fb = CG == 2 ? full_cluster0 + static_cast<uint32_t>(stage) * 8u : 0u;
                    const uint32_t sfb = CG == 2 ? sfull_cluster0 + static_cast<uint32_t>(stage) * 8u : 0u;
                    if constexpr (is_sparse(FMT)) {
                        // SP metadata: the tile's 2 KB block of this stage (16 rows of 128 bytes);
                        // SPC: the stage's four canonical words (16 bytes) of the tile's 128 rows
                        // (SPG: the writer warps load them themselves);
                        // compressed A: 64 kept values (128 bytes) of the stage's 128 logical K;
                        // B: two 64-value atoms
                        if constexpr (FMT == FMT_SP)
                            tma_load_2d(ss, &tmSA, sfull + stage, 0, (a_tile * p.num_kb + kb) * 16);
                        else if constexpr (FMT == FMT_SPC)
                            tma_load_2d(ss, &tmSA, sfull + stage, kb * 4, a_row);
                        tma_ld<CG>(sa, &tmA, full + stage, fb, kb * 64, a_row);
                        tma_ld<CG>(sb, &tmB, full + stage, fb, kb * 128, b_row);
                        tma_ld<CG>(sb + BN_CTA * TILE_K_BYTES, &tmB, full + stage, fb, kb * 128 + 64, b_row);
                    } else {
                        // scale atoms: 512 bytes = 4 rows of 128 bytes each in the tensor maps
                        const int ya = (a_tile * kt + kb * APT) * 4;
                        tma_ld<CG>(ss, &tmSA, sfull + stage, sfb, 0, ya);
#pragma unroll
                        for (int i = 0; i < SFB_ATOMS; ++i)
                            tma_ld<CG>(ss + SF_ATOM * APT * (1 + i), &tmSB, sfull + stage, sfb, 0,
                                       ((nb * SFB_ATOMS + i) * kt + kb * APT) * 4);
                        tma_ld<CG>(sa, &tmA, full + stage, fb, kb * 128, a_row);
                        tma_ld<CG>(sb, &tmB, full + stage, fb, kb * 128, b_row);
                    }
                    ++issued;
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            for (int s = 0; s < STAGES; ++s) {
                const long long n = issued > s ? (issued - s + STAGES - 1) / STAGES : 0;
                if (n == 0) continue;
                const uint32_t last = static_cast<uint32_t>((n - 1) & 1);
                if (leader) {
                    if (!is_sparse(FMT) || meta_tma) wait_bar<CG>(sfull + s, last, w, SITE_DRAIN, false);
                    wait_bar<CG>(full + s, last, w, SITE_DRAIN, false);
                } else {
                    // sparse: this CTA's metadata lands on its own side-data barrier
                    if (meta_tma) wait_bar<CG>(sfull + s, last, w, SITE_DRAIN, false);
                    wait_bar<CG>(empty + s, last, w, SITE_DRAIN, false);
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            // Item i = (tile, K block) in ring stage i % STAGES: wait until its data has
            // landed and the copy threads' copies of its side data have completed.
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            int local = 0;
            for (int t = first_tile; ok && t < p.tile_end; t += step, ++local) {
                const int acc = local % NACC;
                const uint32_t acc_phase = (local / NACC) & 1;
                if (!wait_bar<CG>(tempty + acc, acc_phase ^ 1u, w, SITE_MMA_ACC_EMPTY, true)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc) * ACC_STRIDE;
                for (int kb = 0; kb < p.num_kb; ++kb) {
                    if (!wait_bar<CG>(sfready + stage, phase, w, SITE_MMA_META, true) ||
                        !wait_bar<CG>(full + stage, phase, w, SITE_MMA_FULL, true)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t ad = sdesc_kmajor_sw128(sbase + L::A_OFF + stage * A_STAGE_BYTES);
                    const uint64_t bd = sdesc_kmajor_sw128(sbase + L::B_OFF + stage * L::B_STAGE);
                    const uint64_t bd1 = sdesc_kmajor_sw128(sbase + L::B_OFF + stage * L::B_STAGE + BN_CTA * TILE_K_BYTES);
                    const uint32_t sf = tmem_base + SF_COL + static_cast<uint32_t>(stage) * SF_STAGE_COLS;
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const uint32_t accum = (kb > 0 || k > 0) ? 1u : 0u;
                        if constexpr (is_sparse(FMT)) {
                            // logical K 32 per MMA: A +32 bytes (16 kept values), B +64 bytes within its
                            // atom (atom k / 2); metadata word of MMA k at column 4k
                            mma_sp16<CG>(d_tmem, ad + 2 * k, (k < 2 ? bd : bd1) + 4 * (k & 1), sf + 4u * k, p.idesc, accum);
                        } else if constexpr (FMT == FMT_NV) {
                            mma_nvf4<CG>(d_tmem, ad + 2 * k, bd + 2 * k, p.idesc, sf + SF::sfa(k), sf + SF::sfb(k), accum);
                        } else if constexpr (FMT == FMT_MXF4) {
                            // scale-factor id 2 (k % 2): bytes 2 (k % 2) .. +1 of the atom's scale words
                            const uint32_t id = 2u * static_cast<uint32_t>(k & 1);
                            const uint32_t idesc = p.idesc | (id << 29) | (id << 4);
                            mma_mxf4<CG>(d_tmem, ad + 2 * k, bd + 2 * k, idesc, sf + SF::sfa(k), sf + SF::sfb(k), accum);
                        } else {
                            // scale-factor ids: byte k of the stage's scale words (A bits [29,31), B bits [4,6))
                            const uint32_t idesc = p.idesc | (static_cast<uint32_t>(k) << 29) | (static_cast<uint32_t>(k) << 4);
                            mma_mx<CG>(d_tmem, ad + 2 * k, bd + 2 * k, idesc, sf + SF::sfa(k), sf + SF::sfb(k), accum);
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
            if (CG == 2) mma_commit_pair(drain, 0x1);
            else mma_commit(drain);
            wait_bar<CG>(drain, 0, w, SITE_DRAIN, false);
        }
    } else if (FMT == FMT_SPC && warp >= MX_COPY_WARP) {
        // Metadata writer for TMEM lane quadrant q = warp % 4 (in both CTAs of a pair).  The sparse
        // MMA reads, in TMEM lane 16a + 8s + r, bits 16s .. 16s+15 of the stage's words of tile
        // rows 16a + r (low half) and 16a + 8 + r (high half); word k goes to column 4k of the
        // stage's slot.  The stage's four canonical words of the tile's 128 rows landed in shared
        // memory with its A and B (16 bytes per row, rows past M zero), so lane L = 32q + l takes
        // rows L & ~8 and L | 8 from there; rows past M become the fill code.  The slot's
        // previous readers (the MMAs of item - STAGES) completed before the producer could
        // refill the stage.
        const int quad = warp & 3;
        const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
        const uint32_t sfready0 = CG == 2 ? mapa_shared(smem_u32(sfready), 0) : smem_u32(sfready);
        const int row_lo = (quad * 32 + lane) & ~8, row_hi = (quad * 32 + lane) | 8;
        const uint32_t sel = (lane & 8) ? 0x7632u : 0x5410u; // half s of the low row, then of the high row
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        for (int t = first_tile; ok && t < p.tile_end; t += step) {
            int mb, nb;
            tile_coords(p, t, mb, nb);
            const int rows_left = p.kM - (mb * CG + static_cast<int>(rank)) * BM;
            for (int kb = 0; kb < p.num_kb; ++kb) {
                if (!wait_bar<CG>(sfull + stage, phase, w, SITE_MMA_FULL, true)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint8_t *ss = smem + L::SF_OFF + stage * L::SF_STAGE;
                uint4 lo = *reinterpret_cast<const uint4 *>(ss + row_lo * 16);
                uint4 hi = *reinterpret_cast<const uint4 *>(ss + row_hi * 16);
                if (rows_left < BM) { // the last row tile: rows past M take the fill code
                    if (row_lo >= rows_left) lo = make_uint4(SP_META_FILL, SP_META_FILL, SP_META_FILL, SP_META_FILL);
                    if (row_hi >= rows_left) hi = make_uint4(SP_META_FILL, SP_META_FILL, SP_META_FILL, SP_META_FILL);
                }
                const uint32_t t0 = tmem_base + lane_base + SF_COL + static_cast<uint32_t>(stage) * SF_STAGE_COLS;
                tmem_st_32x32b_x1(t0, __byte_perm(lo.x, hi.x, sel));
                tmem_st_32x32b_x1(t0 + 4u, __byte_perm(lo.y, hi.y, sel));
                tmem_st_32x32b_x1(t0 + 8u, __byte_perm(lo.z, hi.z, sel));
                tmem_st_32x32b_x1(t0 + 12u, __byte_perm(lo.w, hi.w, sel));
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if (CG == 2) mbar_arrive_cluster(sfready0 + static_cast<uint32_t>(stage) * 8u);
                    else mbar_arrive(sfready + stage);
                }
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
    } else if (FMT == FMT_SPG && warp >= MX_COPY_WARP) {
        // Metadata writer as for SPC, the words from global memory: lane l loads, SPC_PREFETCH
        // stages ahead, the stage's four canonical words of its own tile row 32q + l and
        // exchanges half-words with lane l ^ 8 (the same TMEM words as above).  A slot is
        // rewritten only after its previous readers (the MMAs of item - STAGES) completed,
        // which the stage's empty barrier records.
        constexpr int SPC_PREFETCH = 4;
        const int quad = warp & 3;
        const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
        const uint32_t sfready0 = CG == 2 ? mapa_shared(smem_u32(sfready), 0) : smem_u32(sfready);
        const int my_tiles = first_tile < p.tile_end ? (p.tile_end - 1 - first_tile) / step + 1 : 0;
        const long long items = static_cast<long long>(my_tiles) * p.num_kb;
        const long long qn = p.meta_ld;
        const bool vec = (qn & 3) == 0;
        const bool upper = (lane & 8) != 0;
        const int row_in_tile = quad * 32 + lane;
        // fetch cursor: the (tile, stage) of the next item to load
        int f_t = first_tile, f_kb = 0, f_row = 0;
        long long fetched = 0;
        uint4 buf[SPC_PREFETCH];
#pragma unroll
        for (int j = 0; j < SPC_PREFETCH; ++j) {
            buf[j] = make_uint4(SP_META_FILL, SP_META_FILL, SP_META_FILL, SP_META_FILL);
            if (fetched < items) {
                if (f_kb == 0) {
                    int mb, nb;
                    tile_coords(p, f_t, mb, nb);
                    f_row = (mb * CG + static_cast<int>(rank)) * BM + row_in_tile;
                }
                buf[j] = sp_meta_words(p.meta, qn, p.kM, f_row, f_kb, vec);
                ++fetched;
                if (++f_kb == p.num_kb) f_kb = 0, f_t += step;
            }
        }
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        for (long long item = 0; ok && item < items; item += SPC_PREFETCH) {
#pragma unroll
            for (int j = 0; j < SPC_PREFETCH; ++j) {
                if (item + j >= items) break;
                const uint4 cur = buf[j];
                if (fetched < items) {
                    if (f_kb == 0) {
                        int mb, nb;
                        tile_coords(p, f_t, mb, nb);
                        f_row = (mb * CG + static_cast<int>(rank)) * BM + row_in_tile;
                    }
                    buf[j] = sp_meta_words(p.meta, qn, p.kM, f_row, f_kb, vec);
                    ++fetched;
                    if (++f_kb == p.num_kb) f_kb = 0, f_t += step;
                }
                int free_ok = 1;
                if (lane == 0) free_ok = wait_bar<CG>(empty + stage, phase ^ 1u, w, SITE_META_EMPTY, true);
                free_ok = __shfl_sync(0xffffffffu, free_ok, 0);
                if (!free_ok) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t words[4] = {cur.x, cur.y, cur.z, cur.w};
                const uint32_t t0 = tmem_base + lane_base + SF_COL + static_cast<uint32_t>(stage) * SF_STAGE_COLS;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const uint32_t other = __shfl_xor_sync(0xffffffffu, words[k], 8);
                    const uint32_t hw = upper ? ((other >> 16) | (words[k] & 0xFFFF0000u))
                                              : ((words[k] & 0xFFFFu) | (other << 16));
                    tmem_st_32x32b_x1(t0 + 4u * static_cast<uint32_t>(k), hw);
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if (CG == 2) mbar_arrive_cluster(sfready0 + static_cast<uint32_t>(stage) * 8u);
                    else mbar_arrive(sfready + stage);
                }
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
    } else if (FMT == FMT_SP && warp >= MX_COPY_WARP) {
        // Metadata writer for TMEM lane quadrant warp % 4, in both CTAs of a pair (each CTA's
        // MMA rows read their metadata from its own tensor memory): lane l loads the 16 bytes
        // of TMEM lane 32q + l (the words of the stage's four MMAs) and stores word k at
        // column 4k of the stage's slot.  The slot's previous readers (the MMAs of item -
        // STAGES) completed before the producer could refill the stage's side data.
        const int quad = warp & 3;
        const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
        const uint32_t sfready0 = CG == 2 ? mapa_shared(smem_u32(sfready), 0) : smem_u32(sfready);
        const int my_tiles = first_tile < p.tile_end ? (p.tile_end - 1 - first_tile) / step + 1 : 0;
        const long long items = static_cast<long long>(my_tiles) * p.num_kb;
        int stage = 0;
        uint32_t phase = 0;
        for (long long item = 0; item < items; ++item) {
            if (!wait_bar<CG>(sfull + stage, phase, w, SITE_MMA_FULL, true)) break;
            tc_fence_after();
            const uint4 v = *reinterpret_cast<const uint4 *>(smem + L::SF_OFF + stage * L::SF_STAGE + (quad * 32 + lane) * 16);
            const uint32_t t0 = tmem_base + lane_base + SF_COL + static_cast<uint32_t>(stage) * SF_STAGE_COLS;
            tmem_st_32x32b_x1(t0, v.x);
            tmem_st_32x32b_x1(t0 + 4u, v.y);
            tmem_st_32x32b_x1(t0 + 8u, v.z);
            tmem_st_32x32b_x1(t0 + 12u, v.w);
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (CG == 2) mbar_arrive_cluster(sfready0 + static_cast<uint32_t>(stage) * 8u);
                else mbar_arrive(sfready + stage);
            }
            if (++stage == STAGES) {
                stage = 0;
                phase ^= 1u;
            }
        }
    } else if (warp >= MX_COPY_WARP) {
        const int cw = warp - MX_COPY_WARP; // this thread issues the copies e with e % NCW == cw
        if (lane == 0 && leader) {
            const int my_tiles = first_tile < p.tile_end ? (p.tile_end - 1 - first_tile) / step + 1 : 0;
            const long long items = static_cast<long long>(my_tiles) * p.num_kb;
            int stage = 0;
            uint32_t phase = 0;
            for (long long item = 0; item < items; ++item) {
                // the stage's side data has landed; its TMEM slot's previous readers (the MMAs
                // of item - STAGES) completed before the producer could refill the stage
                if (!wait_bar<CG>(sfull + stage, phase, w, SITE_MMA_FULL, true)) break;
                tc_fence_after();
                const uint32_t ss = sbase + L::SF_OFF + stage * L::SF_STAGE;
                const uint32_t s0 = tmem_base + SF_COL + static_cast<uint32_t>(stage) * SF_STAGE_COLS;
#pragma unroll
                for (int e = 0; e < SF::NCP; ++e)
                    if (e % NCW == cw) tmem_cp_side<CG>(s0 + SF::col(e), ss + SF::src(e));
                if (CG == 2) mma_commit_pair(sfready + stage, 0x1);
                else mma_commit(sfready + stage);
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (CG == 2) mma_commit_pair(cdrain, 0x1);
            else mma_commit(cdrain);
            wait_bar<CG>(cdrain, 0, w, SITE_DRAIN, false);
        }
    } else if (warp < MX_COPY_WARP) {
        // Epilogue: warp quadrant (warp % 4) owns TMEM lanes / tile rows
        // 32q .. 32q + 31; the two warps of a quadrant split the columns.
        const int quad = warp & 3;
        const int c_lo = ((warp - 2) / 4) * EPI_COLS;
        const int row_in_tile = quad * 32 + lane;
        const uint32_t tempty_cluster0 = CG == 2 ? mapa_shared(smem_u32(tempty), 0) : 0u;
        int local = 0;
        for (int t = first_tile; t < p.tile_end; t += step, ++local) {
            const int acc = local % NACC;
            const uint32_t acc_phase = (local / NACC) & 1;
            int ok = 1;
            if (lane == 0) ok = wait_bar<CG>(tfull + acc, acc_phase, w, SITE_EPI_ACC_FULL, true);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            tc_fence_after();
            int mb, nb;
            tile_coords(p, t, mb, nb);
            const int row = mb * (BM * CG) + static_cast<int>(rank) * BM + row_in_tile;
            const uint32_t tbase = tmem_base + static_cast<uint32_t>(acc) * ACC_STRIDE + (static_cast<uint32_t>(quad * 32) << 16);
            const int col0 = nb * BN + c_lo;
            if (p.out_fmt != OUT_F32 && p.beta == 0.f && col0 + EPI_COLS <= p.kN) {
                // out = alpha * acc (+ bias), rounded once -- the same operations as
                // epilogue_row32 with beta = 0 -- packed two per register
                uint32_t packed[EPI_COLS / 2];
#pragma unroll
                for (int c = 0; c < EPI_COLS; c += 32) {
                    uint32_t r[32];
                    if (p.num_kb > 0) {
                        tmem_ld_32x32b_x32(tbase + c_lo + c, r);
                        tmem_ld_wait();
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; ++j) r[j] = 0u;
                    }
                    float v[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = p.alpha * __uint_as_float(r[j]);
                    if (p.bias) {
                        float b[32];
                        ld32(p.bias, col0 + c, p.out_fmt, b);
#pragma unroll
                        for (int j = 0; j < 32; ++j) v[j] += b[j];
                    }
#pragma unroll
                    for (int h = 0; h < 16; ++h) packed[c / 2 + h] = pack2(v[2 * h], v[2 * h + 1], p.out_fmt);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if (CG == 2) mbar_arrive_cluster(tempty_cluster0 + static_cast<uint32_t>(acc) * 8u);
                    else mbar_arrive(tempty + acc);
                }
                store_rows_paired<EPI_COLS / 8>(static_cast<uint16_t *>(p.D), p.ldd, row, p.kM, col0, packed);
                continue;
            }
#pragma unroll 1
            for (int c = c_lo; c < c_lo + EPI_COLS; c += 32) {
                uint32_t r[32];
                if (p.num_kb > 0) {
                    tmem_ld_32x32b_x32(tbase + c, r);
                    tmem_ld_wait();
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j) r[j] = 0u;
                }
                if (c + 32 >= c_lo + EPI_COLS) {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        if (CG == 2) mbar_arrive_cluster(tempty_cluster0 + static_cast<uint32_t>(acc) * 8u);
                        else mbar_arrive(tempty + acc);
                    }
                }
                epilogue_row32(p, p.alpha, row, nb * BN + c, r);
            }
        }
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (CG == 2) cluster_sync();
    if (warp == 1) {
        tc_fence_after();
        if (CG == 2) tmem_dealloc_pair(tmem_base, TMEM_COLS);
        else tmem_dealloc(tmem_base, TMEM_COLS);
    }
    clock_probe_add(p, clk0, gt0);
}

template <int BN, int STAGES, int NACC, int CG, int FMT>
static cudaError_t launch_mx_one(const MxMaps &m, const GemmParams &p, int grid, cudaStream_t stream)
{
    using L = MxSmem<BN / CG, BN, STAGES, FMT>;
    auto kern = gemm_mx_kernel<BN, STAGES, NACC, CG, FMT>;
    static_assert(mx_threads(FMT) <= 1024, "block size");
    static std::atomic<unsigned long long> smem_limit_set{0};
    cudaError_t e = ensure_max_smem(reinterpret_cast<const void *>(kern), L::ALLOC, smem_limit_set);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(mx_threads(FMT), 1, 1);
    cfg.dynamicSmemBytes = L::ALLOC;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CG;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, m.a, m.b, m.sa, m.sb, p);
}

cudaError_t launch_gemm_mx(const GemmConfig &cfg, const MxMaps &maps, const GemmParams &p, int grid,
                           cudaStream_t stream)
{
    if (cfg.kind == 5) { // 2:4-sparse A with hardware-ordered metadata
        if (cfg.cta_group == 2) {
            if (cfg.bn == 256) return launch_mx_one<256, 4, 1, 2, FMT_SP>(maps, p, grid, stream);
            if (cfg.bn == 128) return launch_mx_one<128, 5, 2, 2, FMT_SP>(maps, p, grid, stream);
            return cudaErrorInvalidValue;
        }
        if (cfg.bn == 128) return launch_mx_one<128, 4, 2, 1, FMT_SP>(maps, p, grid, stream);
        return cudaErrorInvalidValue;
    }
    if (cfg.kind == 2) { // 2:4-sparse A with canonical metadata, K % 128 == 0 (staged by TMA)
        if (cfg.cta_group == 2) {
            if (cfg.bn == 256) return launch_mx_one<256, 4, 1, 2, FMT_SPC>(maps, p, grid, stream);
            if (cfg.bn == 128) return launch_mx_one<128, 5, 2, 2, FMT_SPC>(maps, p, grid, stream);
            return cudaErrorInvalidValue;
        }
        if (cfg.bn == 128) return launch_mx_one<128, 4, 2, 1, FMT_SPC>(maps, p, grid, stream);
        return cudaErrorInvalidValue;
    }
    if (cfg.kind == 7) { // 2:4-sparse A with canonical metadata, any K % 32 == 0 (global loads)
        if (cfg.cta_group == 2) {
            if (cfg.bn == 256) return launch_mx_one<256, 4, 1, 2, FMT_SPG>(maps, p, grid, stream);
            if (cfg.bn == 128) return launch_mx_one<128, 5, 2, 2, FMT_SPG>(maps, p, grid, stream);
            return cudaErrorInvalidValue;
        }
        if (cfg.bn == 128) return launch_mx_one<128, 4, 2, 1, FMT_SPG>(maps, p, grid, stream);
        return cudaErrorInvalidValue;
    }
    if (cfg.kind == 6) { // MXFP4
        if (cfg.cta_group == 2) return cfg.bn == 256 ? launch_mx_one<256, 6, 1, 2, FMT_MXF4>(maps, p, grid, stream)
                                                     : cudaErrorInvalidValue;
        if (cfg.bn == 256) return launch_mx_one<256, 4, 1, 1, FMT_MXF4>(maps, p, grid, stream);
        if (cfg.bn == 128) return launch_mx_one<128, 6, 2, 1, FMT_MXF4>(maps, p, grid, stream);
        return cudaErrorInvalidValue;
    }
    if (cfg.kind == 4) { // NVFP4
        if (cfg.cta_group == 2) return cfg.bn == 256 ? launch_mx_one<256, 5, 1, 2, FMT_NV>(maps, p, grid, stream)
                                                     : cudaErrorInvalidValue;
        if (cfg.bn == 256) return launch_mx_one<256, 4, 1, 1, FMT_NV>(maps, p, grid, stream);
        if (cfg.bn == 128) return launch_mx_one<128, 6, 2, 1, FMT_NV>(maps, p, grid, stream);
        return cudaErrorInvalidValue;
    }
    if (cfg.cta_group == 2) return cfg.bn == 256 ? launch_mx_one<256, 6, 1, 2, FMT_MX>(maps, p, grid, stream)
                                                 : cudaErrorInvalidValue;
    if (cfg.bn == 256) return launch_mx_one<256, 4, 1, 1, FMT_MX>(maps, p, grid, stream);
    if (cfg.bn == 128) return launch_mx_one<128, 6, 2, 1, FMT_MX>(maps, p, grid, stream);
    return cudaErrorInvalidValue;
}

// ---------------------------------------------------------------- scale packing

// One thread per 16-byte row of an atom: row l of atom (t, k) holds, for the
// four rows r = 128 t + 32 q + l (q = 0..3), the four codes of blocks 4k .. 4k+3.
// Rows past `rows` and blocks past `nblk` read `pad` (the format's 1.0).
__global__ void __launch_bounds__(256) mx_pack_scales_kernel(const uint8_t *__restrict__ src, int64_t rows,
                                                             int64_t nblk, int64_t kt, int64_t total, uint32_t pad,
                                                             uint4 *__restrict__ dst)
{
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= total) return;
    const int64_t l = i & 31;
    const int64_t atom = i >> 5;
    const int64_t t = atom / kt;
    const int64_t k = atom - t * kt;
    uint32_t wv[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int64_t r = t * 128 + 32 * q + l;
        uint32_t v = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int64_t b = 4 * k + j;
            const uint32_t code = (r < rows && b < nblk) ? static_cast<uint32_t>(__ldg(src + r * nblk + b)) : pad;
            v |= code << (8 * j);
        }
        wv[q] = v;
    }
    dst[i] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
}

cudaError_t launch_mx_pack_scales(const uint8_t *src, int64_t rows, int64_t nblk, uint32_t pad, uint8_t *dst,
                                  cudaStream_t stream)
{
    const int64_t kt = (nblk + 3) / 4;
    const int64_t total = ((rows + 127) / 128) * kt * 32;
    if (total == 0) return cudaSuccess;
    const int64_t blocks = (total + 255) / 256;
    mx_pack_scales_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(src, rows, nblk, kt, total, pad,
                                                                             reinterpret_cast<uint4 *>(dst));
    return cudaGetLastError();
}

} // namespace tcm
