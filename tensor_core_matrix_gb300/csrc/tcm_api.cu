// tcm_api.cu -- the extern "C" boundary of libtcm.so (declared in include/tcm.h).
//
// Validates arguments on the host, encodes the TMA tensor maps (through the
// driver entry point cuTensorMapEncodeTiled, fetched at run time so the
// library does not link libcuda directly), picks a kernel configuration and
// launches it on the caller's stream.  No device memory is allocated here:
// the device status words are a file-scope __device__ array.
#include <atomic>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "tcm.h"
#include "tcm_internal.h"
#include "tcm_ptx.cuh"

namespace tcm {

__device__ int g_device_status[2]; // {code, site}, one copy per device

static constexpr int kMaxDevices = 64;

int *device_status_ptr()
{
    static int *ptrs[kMaxDevices] = {};
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!ptrs[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return nullptr;
        ptrs[dev] = static_cast<int *>(p);
    }
    return ptrs[dev];
}

static int sm_count()
{
    static std::atomic<int> counts[kMaxDevices] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
    int n = counts[dev].load(std::memory_order_relaxed);
    if (n == 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        counts[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

static std::atomic<unsigned long long> g_timeout_ns{0};
static std::atomic<int> g_force_cta_group{0};
static std::atomic<int> g_force_bn{0};
static std::atomic<int> g_force_stages{0};
static std::atomic<int> g_force_group_m{0};
static std::atomic<int> g_force_ksplit{0};
static std::atomic<int> g_force_split{0};
static std::atomic<unsigned long long *> g_clock_probe{nullptr};

static std::atomic<int> g_fault_once{0};

static unsigned long long timeout_ns()
{
    unsigned long long t = g_timeout_ns.load();
    if (t == 0) {
        t = 2000000000ull;
        if (const char *env = std::getenv("TCM_TIMEOUT_NS")) {
            const unsigned long long v = std::strtoull(env, nullptr, 10);
            if (v > 0) t = v;
        }
        g_timeout_ns.store(t);
    }
    return t;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// Tensor map of a K-major operand: `rows` rows of `inner` elements, pitch `ld`
// elements; tiles of box_rows x 128 bytes with 128-byte swizzling; reads
// outside the matrix return zeros.
// elem_bytes 0 = FP4 E2M1 packed two per byte: loaded with 16U4_ALIGN16B, which
// places each 16 packed values (8 bytes) at the start of a 16-byte shared-memory
// slot -- a 128-element K stage is then 128 bytes per row, the FP8 stage layout
// (the padded 8-bit container that kind::f8f6f4 reads for FP4).
static bool encode_kmajor(CUtensorMap *map, const void *base, int elem_bytes, uint64_t inner, uint64_t rows,
                          uint64_t ld, uint32_t box_rows)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const CUtensorMapDataType dt = elem_bytes == 0   ? CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B
                                   : elem_bytes == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                                     : CU_TENSOR_MAP_DATA_TYPE_UINT16;
    const cuuint64_t dims[2] = {inner, rows};
    const cuuint64_t strides[1] = {elem_bytes == 0 ? ld / 2 : ld * static_cast<uint64_t>(elem_bytes)};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(elem_bytes == 0 ? 128 : 128 / elem_bytes), box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, dt, 2, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Blocked scales (see tcm_gemm_mx.cu) as a 2-D byte tensor of 512-byte atoms, each
// atom 4 rows of 128 bytes; a box holds the box_atoms atoms of one 128-row tile in one K
// stage.
// k_per_atom: K values covered by one atom (MX 128 = 4 blocks of 32, NVFP4 64 = 4 of 16);
// box_atoms: atoms per TMA box (the atoms of one 128-row tile in one K stage).
static bool encode_sf_atoms(CUtensorMap *map, const void *base, uint64_t rows, uint64_t K, uint64_t k_per_atom,
                            uint32_t box_atoms)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    // The atoms are contiguous 512-byte blocks; the map views them as rows of 128 bytes
    // (4 per atom) so that a box of atoms moves in 128-byte requests, not 16-byte ones.
    const uint64_t atoms = ((rows + 127) / 128) * ((K + k_per_atom - 1) / k_per_atom);
    const cuuint64_t dims[2] = {128, atoms * 4};
    const cuuint64_t strides[1] = {128};
    const cuuint32_t box[2] = {128, 4u * box_atoms};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

static int elem_bytes(tcm_dtype t)
{
    switch (t) {
    case TCM_BF16: case TCM_F16: return 2;
    case TCM_F32: return 4;
    case TCM_E4M3: case TCM_E5M2: return 1;
    default: return 0; // TCM_E2M1: half a byte, handled where pitches are checked
    }
}

static bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// kind::f8f6f4 instruction-descriptor format of an 8/4-bit operand
static uint32_t f8code(uint32_t f) { return f == TCM_E5M2 ? 1u : (f == TCM_E2M1 ? 5u : 0u); }

} // namespace tcm

using namespace tcm;

extern "C" {

const char *tcm_status_string(tcm_status s)
{
    switch (s) {
    case TCM_OK: return "TCM_OK";
    case TCM_ERR_INVALID_ARG: return "TCM_ERR_INVALID_ARG";
    case TCM_ERR_UNSUPPORTED: return "TCM_ERR_UNSUPPORTED";
    case TCM_ERR_MISALIGNED: return "TCM_ERR_MISALIGNED";
    case TCM_ERR_CUDA: return "TCM_ERR_CUDA";
    case TCM_ERR_TIMEOUT: return "TCM_ERR_TIMEOUT";
    default: return "TCM_UNKNOWN_STATUS";
    }
}

int tcm_version(void) { return 100; }

void tcm_set_timeout_ns(uint64_t ns) { g_timeout_ns.store(ns); }

void tcm_set_config_override(int cta_group, int tile_n, int stages, int group_m, int ksplit, int tail_split)
{
    g_force_cta_group.store(cta_group);
    g_force_bn.store(tile_n);
    g_force_stages.store(stages);
    g_force_group_m.store(group_m);
    g_force_ksplit.store(ksplit);
    g_force_split.store(tail_split);
}

void tcm_set_clock_probe(unsigned long long *counters) { g_clock_probe.store(counters); }

void tcm_debug_fail_next_launch(int mask) { g_fault_once.store(mask); }

} // extern "C"

namespace tcm {

// Kernel variant, tile grid and work units of a dense GEMM (shared by the launch and by
// tcm_gemm_workspace_bytes, so that the size query and the launch always agree).
struct DensePlan {
    GemmConfig cfg;
    bool swap;                  // skinny M: the kernel computes D^T (weights as the 128-row operand)
    int64_t kM, kN;             // kernel-space rows and columns
    int64_t tiles_m, tiles_n, num_tiles;
    int64_t per_cluster, clusters;
    int split;                  // K parts per tile of the last, partly filled round (1: none)
    int split_kb;               // split 2: K blocks of the owner part (the helper has the rest)
    int64_t split_begin, units;
    int64_t flag_bytes, ws_bytes; // workspace: counters, then fp32 partial slots
};

static DensePlan plan_dense(int64_t M, int64_t N, int64_t K, int kind, int64_t sms, bool allow_split)
{
    DensePlan d{};
    // swap A and B for skinny M so the weight fills the 128-row MMA
    d.swap = M <= 64 && N >= 128;
    d.kM = d.swap ? N : M;
    d.kN = d.swap ? M : N;
    const int64_t kM = d.kM, kN = d.kN;
    GemmConfig &cfg = d.cfg;
    cfg.kind = kind;
    cfg.cta_group = 1;
    if (d.swap) cfg.bn = kN <= 32 ? 32 : 64;
    else if (kN <= 32) cfg.bn = 32;
    else if (kN <= 64) cfg.bn = 64;
    else if (kN <= 128) cfg.bn = 128;
    else {
        cfg.bn = 256;
        // 256 x 256 pair tiles when they still give every CTA pair work
        const int64_t pair_tiles = ((kM + 255) / 256) * ((kN + 255) / 256);
        const int64_t t128 = ((kM + 127) / 128) * ((kN + 127) / 128);
        if (kM > 128 && pair_tiles >= sms / 2) cfg.cta_group = 2;
        else if (((kM + 127) / 128) * ((kN + 255) / 256) < sms / 2 && t128 > pair_tiles) cfg.bn = 128;
    }
    // small problems (at most one 128 x 128 tile per two SMs) are latency-bound: 64-wide
    // tiles double the CTAs sharing the work (measured 512^3 with C: 7.6 against 10.4 us in
    // the kernel; 1024^3: 12.9 against 14.9 us per launch)
    if (!d.swap && cfg.bn == 128 && ((kM + 127) / 128) * ((kN + 127) / 128) <= sms / 2) cfg.bn = 64;
    const int force_cg = g_force_cta_group.load(), force_bn = g_force_bn.load();
    if (force_cg == 1 || force_cg == 2) cfg.cta_group = force_cg;
    if (force_bn == 32 || force_bn == 64 || force_bn == 128 || force_bn == 256) cfg.bn = force_bn;
    if (cfg.cta_group == 2 && (cfg.bn != 256 || d.swap)) cfg.cta_group = 1;
    cfg.stages = g_force_stages.load();
    cfg.ksplit = 1;
    const int64_t kbs = (K + (kind == 1 ? 127 : 63)) / (kind == 1 ? 128 : 64);
    {
        // K split across a cluster when single-CTA tiles leave SMs idle: pick the
        // split (1, 2, 4) whose last round of tiles is fullest, keeping >= 8 K
        // blocks per CTA; tiles of width 32 and 64 only.
        const int64_t tiles = ((kM + 127) / 128) * ((kN + cfg.bn - 1) / cfg.bn);
        if (cfg.cta_group == 1 && (cfg.bn == 32 || cfg.bn == 64)) {
            double best = 0.0;
            for (int ks = 1; ks <= 4; ks *= 2) {
                if (ks > 1 && kbs / ks < 8) break;
                const int64_t clusters = sms / ks;
                const int64_t rounds = (tiles + clusters - 1) / clusters;
                const double eff = static_cast<double>(tiles) / static_cast<double>(rounds * clusters) / (ks > 1 ? 1.02 : 1.0);
                if (eff > best + 0.05) best = eff, cfg.ksplit = ks;
            }
        }
        const int fk = g_force_ksplit.load();
        if (fk == 1 || ((fk == 2 || fk == 4) && cfg.cta_group == 1 && (cfg.bn == 32 || cfg.bn == 64))) cfg.ksplit = fk;
    }
    // two 128-byte K atoms per stage for 32-wide single-CTA tiles (the skinny,
    // HBM-bound shapes): longer contiguous reads of each weight row
    cfg.katoms = (cfg.cta_group == 1 && cfg.bn == 32 && cfg.ksplit <= 2) ? 2 : 1;
    // CTA pairs, 8-bit operands: stages of two K atoms (E4M3 8192^3 1 %, 4096^3 3 % faster than
    // one); 16-bit operands keep one (two took ~2 % more cycles at 8192^3)
    if (cfg.cta_group == 2) cfg.katoms = kind == 1 ? 2 : 1;

    d.tiles_m = (kM + 128 * cfg.cta_group - 1) / (128 * cfg.cta_group);
    d.tiles_n = (kN + cfg.bn - 1) / cfg.bn;
    d.num_tiles = d.tiles_m * d.tiles_n;
    d.per_cluster = static_cast<int64_t>(cfg.cta_group) * cfg.ksplit;
    d.clusters = sms / d.per_cluster;
    // Tail K split (CTA-pair tiles, with a workspace): the R tiles of the last, partly
    // filled round become 2R part-K units when every pair then gets at most one of them
    // (2R <= clusters).  Handing the helper part's partial sums to the owner part takes
    // ~6 us (stage, bulk store, counter; measured), so the owner takes SPLIT_SKEW_KB K
    // blocks more than half (rounded to whole stages of cfg.katoms blocks) -- ~3 us of MMA
    // at ~0.3-0.4 us per block -- and the helper's
    // sums are published about when the owner's own MMAs end; the owner then only loads
    // them (~1 us).  Measured (whole builds timed back to back): 4096^3 bf16/fp16 and
    // 2048 x 8192 x 4096 3.5 % faster than with equal halves.  Only tiles of at least
    // SPLIT_MIN_KB K blocks are split: with 32 (E4M3 4096^3) the split, skewed or not,
    // was 7-10 % slower.  tail_split 2 in the config override lowers the limit to 2
    // blocks, 1 turns the split off.
    constexpr int64_t SPLIT_MIN_KB = 64, SPLIT_SKEW_KB = 9;
    d.split = 1;
    const int64_t rem = d.num_tiles % d.clusters;
    const int fs = g_force_split.load();
    const int64_t min_kb = fs == 2 ? 2 : SPLIT_MIN_KB;
    // the parts are whole stages (cfg.katoms K blocks each)
    const int64_t stages = (kbs + cfg.katoms - 1) / cfg.katoms;
    if (allow_split && cfg.cta_group == 2 && cfg.ksplit == 1 && rem > 0 && 2 * rem <= d.clusters && kbs >= min_kb &&
        stages >= 2 && fs != 1)
        d.split = 2;
    d.split_begin = d.split > 1 ? d.num_tiles - rem : d.num_tiles;
    // owner: half the stages plus the skew (rounded to stages), leaving the helper at least one
    const int64_t skew = (SPLIT_SKEW_KB + cfg.katoms / 2) / cfg.katoms;
    d.split_kb = static_cast<int>(stages / 2 + std::min<int64_t>(skew, std::max<int64_t>(stages / 2 - 1, 0)));
    d.units = d.split_begin + (d.num_tiles - d.split_begin) * d.split;
    if (d.split > 1) {
        const int64_t nsplit = d.num_tiles - d.split_begin;
        d.flag_bytes = ((nsplit * cfg.cta_group * 4 + 255) / 256) * 256;
        d.ws_bytes = d.flag_bytes + nsplit * (d.split - 1) * cfg.cta_group * 128 * cfg.bn * 4;
    }
    return d;
}

} // namespace tcm

extern "C" {

// Dense GEMM with the full epilogue: y = act(alpha * sa * sb * acc + beta * C + bias),
// D = y / d_scale cast to out_dtype (FP8 outputs: saturating), amax = max |y|.
// tcm_gemm_ex is the act = none, 16/32-bit-output case.  With a workspace (ws,
// ws_bytes >= tcm_gemm_workspace_bytes) the last round of CTA-pair tiles may be split over K.
static tcm_status gemm_impl(int64_t M, int64_t N, int64_t K, tcm_dtype a_dtype, const void *A, int64_t lda,
                            tcm_dtype b_dtype, const void *B, int64_t ldb, const void *C, int64_t ldc, void *D,
                            int64_t ldd, tcm_dtype out_dtype, float alpha, float beta, const float *a_scale,
                            const float *b_scale, const void *bias, int act, const float *d_scale, float *amax,
                            bool fused, void *ws, int64_t ws_bytes, tcm_stream_t stream)
{
    // ---- argument checks (nothing is launched on failure)
    const bool a16 = a_dtype == TCM_BF16 || a_dtype == TCM_F16;
    const bool a8 = a_dtype == TCM_E4M3 || a_dtype == TCM_E5M2 || a_dtype == TCM_E2M1;
    const bool b8 = b_dtype == TCM_E4M3 || b_dtype == TCM_E5M2 || b_dtype == TCM_E2M1;
    int kind;
    if (a16 && b_dtype == a_dtype) kind = 0;
    else if (a8 && b8) kind = 1;
    else return TCM_ERR_UNSUPPORTED;
    const bool a4 = a_dtype == TCM_E2M1, b4 = b_dtype == TCM_E2M1;
    const bool out8 = out_dtype == TCM_E4M3 || out_dtype == TCM_E5M2;
    if (out_dtype != TCM_BF16 && out_dtype != TCM_F16 && out_dtype != TCM_F32 && !(fused && out8))
        return TCM_ERR_UNSUPPORTED;
    if (act < TCM_ACT_NONE || act > TCM_ACT_GELU) return TCM_ERR_INVALID_ARG;
    if (out8 && beta != 0.f) return TCM_ERR_UNSUPPORTED; // no FP8 C
    if ((amax && (reinterpret_cast<uintptr_t>(amax) & 3u)) || (d_scale && (reinterpret_cast<uintptr_t>(d_scale) & 3u)))
        return TCM_ERR_MISALIGNED;
    if (M < 1 || N < 1 || K < 0) return TCM_ERR_INVALID_ARG;
    if (M > INT32_MAX / 2 || N > INT32_MAX / 2 || K > INT32_MAX / 2) return TCM_ERR_UNSUPPORTED;
    if (!D) return TCM_ERR_INVALID_ARG;
    if (K > 0 && (!A || !B)) return TCM_ERR_INVALID_ARG;
    if (beta != 0.f && !C) return TCM_ERR_INVALID_ARG;
    if (lda < K || ldb < K || ldd < N || (C && ldc < N)) return TCM_ERR_INVALID_ARG;
    const int ea = elem_bytes(a_dtype), eb = elem_bytes(b_dtype), eo = elem_bytes(out_dtype);
    // A and B are not read when K == 0: their pointers and pitches are then not checked
    const bool reads_ab = K > 0;
    if ((reads_ab && (!aligned16(A) || !aligned16(B))) || !aligned16(D) || (C && !aligned16(C)) ||
        (bias && !aligned16(bias)))
        return TCM_ERR_MISALIGNED;
    if ((reads_ab && ((!a4 && (lda * ea) % 16) || (!b4 && (ldb * eb) % 16))) || (ldd * eo) % 16 ||
        (C && (ldc * eo) % 16))
        return TCM_ERR_MISALIGNED;
    // packed FP4 operands (16U4_ALIGN16B tensor maps): K a multiple of 128, rows of a
    // multiple of 32 bytes (64 elements) starting on 32-byte boundaries
    if ((a4 || b4) && K % 128 != 0) return TCM_ERR_UNSUPPORTED;
    if (reads_ab && ((a4 && (lda % 64 || (reinterpret_cast<uintptr_t>(A) & 31u))) ||
                     (b4 && (ldb % 64 || (reinterpret_cast<uintptr_t>(B) & 31u)))))
        return TCM_ERR_MISALIGNED;

    if (ws_bytes < 0 || (ws_bytes > 0 && !ws)) return TCM_ERR_INVALID_ARG;
    if (ws && !aligned16(ws)) return TCM_ERR_MISALIGNED;

    const int64_t sms = sm_count();
    if (sms <= 0) return TCM_ERR_CUDA;
    const DensePlan plan = plan_dense(M, N, K, kind, sms, ws != nullptr && ws_bytes > 0);
    const GemmConfig &cfg = plan.cfg;
    const bool swap = plan.swap;
    const int64_t kM = plan.kM, kN = plan.kN;
    if (plan.split > 1 && ws_bytes < plan.ws_bytes) return TCM_ERR_INVALID_ARG;

    // ---- tensor maps (the kernel's "A" operand is the swapped one when swap)
    const int k_elems_stage = kind == 1 ? 128 : 64;
    const uint64_t kdim = K > 0 ? static_cast<uint64_t>(K) : static_cast<uint64_t>(k_elems_stage);
    const void *opA = swap ? B : A;
    const void *opB = swap ? A : B;
    const int eA = swap ? eb : ea, eB = swap ? ea : eb;
    const int64_t ldA = swap ? ldb : lda, ldB = swap ? lda : ldb;
    CUtensorMap tmA, tmB;
    std::memset(&tmA, 0, sizeof tmA);
    std::memset(&tmB, 0, sizeof tmB);
    if (K > 0) {
        if (!encode_kmajor(&tmA, opA, eA, kdim, static_cast<uint64_t>(kM), static_cast<uint64_t>(ldA), 128))
            return TCM_ERR_CUDA;
        if (!encode_kmajor(&tmB, opB, eB, kdim, static_cast<uint64_t>(kN), static_cast<uint64_t>(ldB),
                           static_cast<uint32_t>(cfg.bn / cfg.cta_group)))
            return TCM_ERR_CUDA;
    }

    // ---- parameters and launch
    GemmParams p{};
    p.kM = static_cast<int>(kM);
    p.kN = static_cast<int>(kN);
    p.K = static_cast<int>(K);
    p.num_kb = static_cast<int>((K + k_elems_stage * cfg.katoms - 1) / (k_elems_stage * cfg.katoms));
    p.tiles_m = static_cast<int>(plan.tiles_m);
    p.tiles_n = static_cast<int>(plan.tiles_n);
    p.num_tiles = static_cast<int>(plan.num_tiles);
    // raster groups: 8 row blocks for 16-bit operands (bf16 8192^3: 11 % fewer DRAM bytes and
    // ~1 % faster than 16), 16 for 8-bit ones (E4M3 8192^3: 1.6 % faster than 8)
    p.group_m = g_force_group_m.load() > 0 ? g_force_group_m.load() : (kind == 0 ? 8 : 16);
    p.split = plan.split;
    p.split_begin = static_cast<int>(plan.split_begin);
    p.split_kb = plan.split_kb;
    if (plan.split > 1) {
        p.ws_flag = static_cast<int *>(ws);
        p.ws_part = reinterpret_cast<float *>(static_cast<uint8_t *>(ws) + plan.flag_bytes);
    }
    p.tile_begin = 0;
    p.tile_end = static_cast<int>(plan.units);
    p.D = D;
    p.ldd = ldd;
    p.C = beta != 0.f ? C : nullptr;
    p.ldc = ldc;
    p.bias = bias;
    p.a_scale = swap ? b_scale : a_scale;
    p.b_scale = swap ? a_scale : b_scale;
    p.alpha = alpha;
    p.beta = beta;
    p.out_fmt = static_cast<int>(out_dtype);
    p.bias_fmt = out8 ? OUT_BF16 : p.out_fmt;
    p.act = act;
    p.d_scale = out8 ? d_scale : nullptr;
    p.amax = amax;
    p.swap_ab = swap ? 1 : 0;
    // every CTA has one unit: its C rows can be fetched into L2 while its MMAs run (with
    // more rounds a tile's C would wait in L2 for a whole tile time, and could be evicted)
    p.prefetch_c = p.C && !swap && plan.units <= plan.clusters ? 1 : 0;
    const uint32_t fa = static_cast<uint32_t>(swap ? b_dtype : a_dtype);
    const uint32_t fb = static_cast<uint32_t>(swap ? a_dtype : b_dtype);
    // kind::f16: 0 = f16, 1 = bf16; kind::f8f6f4: 0 = E4M3, 1 = E5M2, 5 = E2M1
    const uint32_t codeA = kind == 0 ? (fa == TCM_BF16 ? 1u : 0u) : f8code(fa);
    const uint32_t codeB = kind == 0 ? (fb == TCM_BF16 ? 1u : 0u) : f8code(fb);
    p.idesc = make_idesc(codeA, codeB, 128u * static_cast<uint32_t>(cfg.cta_group), static_cast<uint32_t>(cfg.bn));
    p.clock_probe = g_clock_probe.load();
    p.timeout_ns = timeout_ns();
    p.status = device_status_ptr();
    if (!p.status) return TCM_ERR_CUDA;

    // a packed FP4 (E2M1) tile row counts 64 bytes on the barrier, not the 128 it occupies
    // in shared memory (16U4_ALIGN16B leaves an 8-byte gap after every 8 bytes)
    if (kind == 1 && (a4 || b4)) {
        const bool kA4 = swap ? b4 : a4, kB4 = swap ? a4 : b4;
        const uint32_t row_a = kA4 ? 64u : 128u, row_b = kB4 ? 64u : 128u;
        p.stage_tx = static_cast<uint32_t>(cfg.cta_group) * static_cast<uint32_t>(cfg.katoms) *
                     (row_a * 128u + row_b * static_cast<uint32_t>(cfg.bn / cfg.cta_group));
    }
    p.fault_inject = g_fault_once.exchange(0);
    const int grid = static_cast<int>((plan.units < plan.clusters ? plan.units : plan.clusters) * plan.per_cluster);
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (amax && cudaMemsetAsync(amax, 0, sizeof(float), st) != cudaSuccess) return TCM_ERR_CUDA;
    // the split tiles' counters start at zero in every launch
    if (plan.split > 1 && cudaMemsetAsync(ws, 0, static_cast<size_t>(plan.flag_bytes), st) != cudaSuccess)
        return TCM_ERR_CUDA;
    const cudaError_t e = launch_gemm(cfg, tmA, tmB, p, grid, st);
    return e == cudaSuccess ? TCM_OK : TCM_ERR_CUDA;
}

} // extern "C"

namespace tcm {

// Workspace of tcm_gemm_ex_builtin_ws, inside the library: one copy on every device that
// loads it, kept until the process exits.  10 MiB holds the largest workspace a
// 256 x 256 CTA-pair split can ask for on a GB300 (152 SMs: at most 38 split tiles of
// two 128 KB slots each, plus their counters, 9.5 MiB); larger requests are refused.
constexpr int64_t kBuiltinWsBytes = 10ll << 20;
static __device__ __align__(256) uint8_t g_builtin_ws[kBuiltinWsBytes];

// Device address of this device's copy of g_builtin_ws.  The first call on a device
// looks it up (with that device current) and keeps it; the array's name in host code
// is only a stand-in for the symbol, never a usable address.
static void *builtin_ws_ptr()
{
    static void *ptrs[kMaxDevices] = {};
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!ptrs[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_builtin_ws) != cudaSuccess) return nullptr;
        ptrs[dev] = p;
    }
    return ptrs[dev];
}

} // namespace tcm

extern "C" {

tcm_status tcm_gemm_ex_builtin_ws(int64_t M, int64_t N, int64_t K, tcm_dtype a_dtype, const void *A, int64_t lda,
                                  tcm_dtype b_dtype, const void *B, int64_t ldb, const void *C, int64_t ldc, void *D,
                                  int64_t ldd, tcm_dtype out_dtype, float alpha, float beta, const float *a_scale,
                                  const float *b_scale, const void *bias, tcm_stream_t stream)
{
    const int64_t need = tcm_gemm_workspace_bytes(M, N, K, a_dtype, b_dtype);
    if (need > kBuiltinWsBytes) return TCM_ERR_UNSUPPORTED; // larger than the built-in workspace
    void *ws = builtin_ws_ptr();
    if (!ws) return TCM_ERR_CUDA;
    return gemm_impl(M, N, K, a_dtype, A, lda, b_dtype, B, ldb, C, ldc, D, ldd, out_dtype, alpha, beta, a_scale,
                     b_scale, bias, TCM_ACT_NONE, nullptr, nullptr, false, ws, kBuiltinWsBytes, stream);
}

int64_t tcm_gemm_workspace_bytes(int64_t M, int64_t N, int64_t K, tcm_dtype a_dtype, tcm_dtype b_dtype)
{
    const bool a16 = a_dtype == TCM_BF16 || a_dtype == TCM_F16;
    const bool a8 = a_dtype == TCM_E4M3 || a_dtype == TCM_E5M2 || a_dtype == TCM_E2M1;
    const bool b8 = b_dtype == TCM_E4M3 || b_dtype == TCM_E5M2 || b_dtype == TCM_E2M1;
    int kind;
    if (a16 && b_dtype == a_dtype) kind = 0;
    else if (a8 && b8) kind = 1;
    else return -1;
    if (M < 1 || N < 1 || K < 0 || M > INT32_MAX / 2 || N > INT32_MAX / 2 || K > INT32_MAX / 2) return -1;
    const int64_t sms = sm_count();
    if (sms <= 0) return -1;
    return plan_dense(M, N, K, kind, sms, true).ws_bytes;
}

tcm_status tcm_gemm_ex(int64_t M, int64_t N, int64_t K, tcm_dtype a_dtype, const void *A, int64_t lda,
                       tcm_dtype b_dtype, const void *B, int64_t ldb, const void *C, int64_t ldc, void *D,
                       int64_t ldd, tcm_dtype out_dtype, float alpha, float beta, const float *a_scale,
                       const float *b_scale, const void *bias, tcm_stream_t stream)
{
    return gemm_impl(M, N, K, a_dtype, A, lda, b_dtype, B, ldb, C, ldc, D, ldd, out_dtype, alpha, beta, a_scale,
                     b_scale, bias, TCM_ACT_NONE, nullptr, nullptr, false, nullptr, 0, stream);
}

tcm_status tcm_gemm_ex_ws(int64_t M, int64_t N, int64_t K, tcm_dtype a_dtype, const void *A, int64_t lda,
                          tcm_dtype b_dtype, const void *B, int64_t ldb, const void *C, int64_t ldc, void *D,
                          int64_t ldd, tcm_dtype out_dtype, float alpha, float beta, const float *a_scale,
                          const float *b_scale, const void *bias, void *workspace, int64_t workspace_bytes,
                          tcm_stream_t stream)
{
    return gemm_impl(M, N, K, a_dtype, A, lda, b_dtype, B, ldb, C, ldc, D, ldd, out_dtype, alpha, beta, a_scale,
                     b_scale, bias, TCM_ACT_NONE, nullptr, nullptr, false, workspace, workspace_bytes, stream);
}

tcm_status tcm_gemm_fused(int64_t M, int64_t N, int64_t K, tcm_dtype a_dtype, const void *A, int64_t lda,
                          tcm_dtype b_dtype, const void *B, int64_t ldb, const void *C, int64_t ldc, void *D,
                          int64_t ldd, tcm_dtype out_dtype, float alpha, float beta, const float *a_scale,
                          const float *b_scale, const void *bias, tcm_activation act, const float *d_scale,
                          float *amax, tcm_stream_t stream)
{
    return gemm_impl(M, N, K, a_dtype, A, lda, b_dtype, B, ldb, C, ldc, D, ldd, out_dtype, alpha, beta, a_scale,
                     b_scale, bias, static_cast<int>(act), d_scale, amax, true, nullptr, 0, stream);
}

tcm_status tcm_gemm(int64_t M, int64_t N, int64_t K, tcm_dtype in_dtype, const void *A, const void *B,
                    const void *C, void *D, float alpha, float beta, tcm_dtype out_dtype, tcm_stream_t stream)
{
    if (in_dtype != TCM_BF16 && in_dtype != TCM_F16) return TCM_ERR_UNSUPPORTED;
    return tcm_gemm_ex(M, N, K, in_dtype, A, K, in_dtype, B, K, C, N, D, N, out_dtype, alpha, beta, nullptr, nullptr,
                       nullptr, stream);
}

static tcm_status check_sparse_shape(int64_t M, int64_t K, tcm_dtype dtype, const void *x, const void *y,
                                     const uint32_t *meta, int64_t lda)
{
    if (dtype != TCM_BF16 && dtype != TCM_F16) return TCM_ERR_UNSUPPORTED;
    if (M < 0 || K < 0 || K % 32 != 0 || lda < K) return TCM_ERR_INVALID_ARG;
    if (M > 0 && K > 0 && (!x || !y || !meta)) return TCM_ERR_INVALID_ARG;
    if ((x && !aligned16(x)) || (y && !aligned16(y)) || (meta && !aligned16(meta))) return TCM_ERR_MISALIGNED;
    if ((lda * 2) % 16) return TCM_ERR_MISALIGNED;
    return TCM_OK;
}

tcm_status tcm_sp_compress(int64_t M, int64_t K, tcm_dtype dtype, const void *A, int64_t lda, void *A_comp,
                           uint32_t *meta, tcm_stream_t stream)
{
    const tcm_status s = check_sparse_shape(M, K, dtype, A, A_comp, meta, lda);
    if (s != TCM_OK) return s;
    return launch_sp_compress(M, K, 2, A, lda, A_comp, meta, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? TCM_OK
               : TCM_ERR_CUDA;
}

tcm_status tcm_sp_decompress(int64_t M, int64_t K, tcm_dtype dtype, const void *A_comp, const uint32_t *meta, void *A,
                             int64_t lda, tcm_stream_t stream)
{
    const tcm_status s = check_sparse_shape(M, K, dtype, A, A_comp, meta, lda);
    if (s != TCM_OK) return s;
    return launch_sp_decompress(M, K, 2, A_comp, meta, A, lda, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? TCM_OK
               : TCM_ERR_CUDA;
}

int64_t tcm_sp_meta_tc_bytes(int64_t M, int64_t K)
{
    if (M < 0 || K < 0 || K % 32 != 0) return -1;
    return ((M + 127) / 128) * ((K + 127) / 128) * 2048;
}

tcm_status tcm_sp_meta_pack(int64_t M, int64_t K, const uint32_t *meta, void *meta_tc, tcm_stream_t stream)
{
    if (M < 0 || K < 0 || K % 32 != 0) return TCM_ERR_INVALID_ARG;
    if (M > INT32_MAX / 2 || K > INT32_MAX / 2) return TCM_ERR_UNSUPPORTED;
    if (M == 0 || K == 0) return TCM_OK;
    if (!meta || !meta_tc) return TCM_ERR_INVALID_ARG;
    if (!aligned16(meta_tc) || (reinterpret_cast<uintptr_t>(meta) & 3u)) return TCM_ERR_MISALIGNED;
    return launch_sp_meta_pack(meta, M, K, static_cast<uint8_t *>(meta_tc), reinterpret_cast<cudaStream_t>(stream)) ==
                   cudaSuccess
               ? TCM_OK
               : TCM_ERR_CUDA;
}

} // extern "C"

// 2:4-sparse GEMM on the block-scaled kernel's sparse formats.  canonical: `meta` is the
// M x K/32-word layout of tcm_sp_compress, which the kernel's writer warps reorder
// themselves (staged by TMA when K % 128 == 0, else loaded from global memory);
// otherwise it is the hardware-ordered layout of tcm_sp_meta_pack, loaded by TMA.
static tcm_status sparse_impl(bool canonical, int64_t M, int64_t N, int64_t K, tcm_dtype dtype, const void *A_comp,
                              const void *meta, const void *B, const void *C, void *D, float alpha, float beta,
                              tcm_dtype out_dtype, tcm_stream_t stream)
{
    if (dtype != TCM_BF16 && dtype != TCM_F16) return TCM_ERR_UNSUPPORTED;
    if (out_dtype != TCM_BF16 && out_dtype != TCM_F16 && out_dtype != TCM_F32) return TCM_ERR_UNSUPPORTED;
    if (M < 1 || N < 1 || K < 0 || K % 32 != 0) return TCM_ERR_INVALID_ARG;
    if (M > INT32_MAX / 2 || N > INT32_MAX / 2 || K > INT32_MAX / 2) return TCM_ERR_UNSUPPORTED;
    // hardware-ordered metadata rows (16 of 128 bytes per stage of 128 logical K) are
    // addressed with 32-bit coordinates
    if (!canonical && ((M + 255) / 128) * ((K + 127) / 128) * 16 > INT32_MAX) return TCM_ERR_UNSUPPORTED;
    if (!D || (K > 0 && (!A_comp || !meta || !B)) || (beta != 0.f && !C)) return TCM_ERR_INVALID_ARG;
    const int eo = elem_bytes(out_dtype);
    if ((A_comp && !aligned16(A_comp)) || (B && !aligned16(B)) || (meta && !aligned16(meta)) || !aligned16(D) ||
        (C && !aligned16(C)))
        return TCM_ERR_MISALIGNED;
    if ((N * eo) % 16) return TCM_ERR_MISALIGNED;
    const int64_t sms = sm_count();
    if (sms <= 0) return TCM_ERR_CUDA;

    GemmConfig cfg{};
    // canonical metadata: staged by TMA when its rows hold whole 16-byte stages (K % 128 == 0),
    // else loaded by the writer warps
    cfg.kind = !canonical ? 5 : K % 128 == 0 ? 2 : 7;
    cfg.ksplit = 1;
    cfg.katoms = 1;
    const int64_t pair_tiles = ((M + 255) / 256) * ((N + 255) / 256);
    cfg.cta_group = (M > 128 && N > 128 && pair_tiles >= sms / 2) ? 2 : 1;
    const int force_cg = g_force_cta_group.load();
    if (force_cg == 1 || force_cg == 2) cfg.cta_group = force_cg;
    cfg.bn = cfg.cta_group == 2 ? 256 : 128;
    if (cfg.cta_group == 2 && g_force_bn.load() == 128) cfg.bn = 128;

    MxMaps maps;
    std::memset(&maps, 0, sizeof maps);
    if (K > 0) {
        if (!encode_kmajor(&maps.a, A_comp, 2, static_cast<uint64_t>(K / 2), static_cast<uint64_t>(M),
                           static_cast<uint64_t>(K / 2), 128) ||
            !encode_kmajor(&maps.b, B, 2, static_cast<uint64_t>(K), static_cast<uint64_t>(N), static_cast<uint64_t>(K),
                           static_cast<uint32_t>(cfg.bn / cfg.cta_group)))
            return TCM_ERR_CUDA;
        if (!canonical) {
            // a stage's 2 KB of metadata (128 lanes x 16 bytes) is contiguous: one box of 16
            // rows of 128 bytes
            const uint64_t meta_rows = static_cast<uint64_t>((M + 127) / 128) * static_cast<uint64_t>((K + 127) / 128) * 16u;
            EncodeTiledFn fn = encode_fn();
            const cuuint64_t dims[2] = {128, meta_rows};
            const cuuint64_t strides[1] = {128};
            const cuuint32_t box[2] = {128, 16};
            const cuuint32_t estr[2] = {1, 1};
            if (!fn || fn(&maps.sa, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(meta), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
                return TCM_ERR_CUDA;
            maps.sb = maps.sa;
        } else if (cfg.kind == 2) {
            // library layout: each stage's four words of the tile's 128 rows (16 bytes per row)
            // as one box of a 2-D map over the M x K/32 words; rows past M read zero, which the
            // writer warps replace with the fill pattern
            EncodeTiledFn fn = encode_fn();
            const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K / 32), static_cast<cuuint64_t>(M)};
            const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K / 32) * 4u};
            const cuuint32_t box[2] = {4, 128};
            const cuuint32_t estr[2] = {1, 1};
            if (!fn || fn(&maps.sa, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void *>(meta), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
                return TCM_ERR_CUDA;
            maps.sb = maps.sa;
        }
    }
    GemmParams p{};
    p.kM = static_cast<int>(M);
    p.kN = static_cast<int>(N);
    p.K = static_cast<int>(K);
    p.num_kb = static_cast<int>((K + 127) / 128);
    p.tiles_m = static_cast<int>((M + 128 * cfg.cta_group - 1) / (128 * cfg.cta_group));
    p.tiles_n = static_cast<int>((N + cfg.bn - 1) / cfg.bn);
    p.num_tiles = p.tiles_m * p.tiles_n;
    p.group_m = g_force_group_m.load() > 0 ? g_force_group_m.load() : 16;
    p.split = 1;
    p.split_begin = p.num_tiles;
    p.tile_begin = 0;
    p.tile_end = p.num_tiles;
    p.clock_probe = g_clock_probe.load();
    p.D = D;
    p.ldd = N;
    p.C = beta != 0.f ? C : nullptr;
    p.ldc = N;
    p.bias = nullptr;
    p.a_scale = p.b_scale = nullptr;
    p.alpha = alpha;
    p.beta = beta;
    p.out_fmt = static_cast<int>(out_dtype);
    p.bias_fmt = p.out_fmt;
    p.swap_ab = 0;
    const uint32_t code = dtype == TCM_BF16 ? 1u : 0u;
    p.idesc = make_idesc(code, code, 128u * static_cast<uint32_t>(cfg.cta_group), static_cast<uint32_t>(cfg.bn)) |
              (1u << 2); // sparsity enabled
    p.timeout_ns = timeout_ns();
    p.status = device_status_ptr();
    if (!p.status) return TCM_ERR_CUDA;
    p.fault_inject = g_fault_once.exchange(0);
    if (canonical) {
        p.meta = static_cast<const uint32_t *>(meta);
        p.meta_ld = K / 32;
    }
    const int64_t clusters = sms / cfg.cta_group;
    const int grid = static_cast<int>((p.num_tiles < clusters ? p.num_tiles : clusters) * cfg.cta_group);
    const cudaError_t e = launch_gemm_mx(cfg, maps, p, grid, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? TCM_OK : TCM_ERR_CUDA;
}

extern "C" {

tcm_status tcm_gemm_sp_tc(int64_t M, int64_t N, int64_t K, tcm_dtype dtype, const void *A_comp, const void *meta_tc,
                          const void *B, const void *C, void *D, float alpha, float beta, tcm_dtype out_dtype,
                          tcm_stream_t stream)
{
    return sparse_impl(false, M, N, K, dtype, A_comp, meta_tc, B, C, D, alpha, beta, out_dtype, stream);
}

tcm_status tcm_gemm_sp(int64_t M, int64_t N, int64_t K, tcm_dtype dtype, const void *A_comp, const uint32_t *meta,
                       const void *B, const void *C, void *D, float alpha, float beta, tcm_dtype out_dtype,
                       tcm_stream_t stream)
{
    return sparse_impl(true, M, N, K, dtype, A_comp, meta, B, C, D, alpha, beta, out_dtype, stream);
}

// Block-scaled GEMM: MXFP8 (E4M3/E5M2 elements, E8M0 per 32, kind::mxf8f6f4), NVFP4
// (packed E2M1, UE4M3 per 16, kind::mxf4nvf4.scale_vec::4X) or MXFP4 (packed E2M1, E8M0
// per 32, kind::mxf4nvf4.scale_vec::2X).
enum BlockFmt { BF_MXFP8 = 0, BF_NVFP4 = 1, BF_MXFP4 = 2 };

static tcm_status block_scaled_impl(int bfmt, int64_t M, int64_t N, int64_t K, tcm_dtype a_dtype, const void *A,
                                    const uint8_t *a_scales, tcm_dtype b_dtype, const void *B, const uint8_t *b_scales,
                                    const void *C, void *D, float alpha, float beta, const void *bias,
                                    tcm_dtype out_dtype, tcm_stream_t stream)
{
    if (bfmt == BF_MXFP8) {
        const bool a8 = a_dtype == TCM_E4M3 || a_dtype == TCM_E5M2;
        const bool b8 = b_dtype == TCM_E4M3 || b_dtype == TCM_E5M2;
        if (!a8 || !b8) return TCM_ERR_UNSUPPORTED;
    }
    const bool fp4 = bfmt != BF_MXFP8; // packed E2M1 operands, 256 K values per 128-byte stage
    if (out_dtype != TCM_BF16 && out_dtype != TCM_F16 && out_dtype != TCM_F32) return TCM_ERR_UNSUPPORTED;
    const int64_t k_stage = fp4 ? 256 : 128;                  // K values per 128-byte stage
    const int64_t k_atom = bfmt == BF_NVFP4 ? 64 : 128;       // K values per scale atom
    if (M < 1 || N < 1 || K < 0 || K % (fp4 ? 256 : 32) != 0) return TCM_ERR_INVALID_ARG;
    if (M > INT32_MAX / 2 || N > INT32_MAX / 2 || K > INT32_MAX / 2) return TCM_ERR_UNSUPPORTED;
    // scale-atom rows (4 of 128 bytes per atom) are addressed with 32-bit coordinates
    if (((M + 255) / 128) * ((K + k_atom - 1) / k_atom) * 4 > INT32_MAX ||
        ((N + 255) / 128) * ((K + k_atom - 1) / k_atom) * 4 > INT32_MAX)
        return TCM_ERR_UNSUPPORTED;
    if (!D || (K > 0 && (!A || !B || !a_scales || !b_scales)) || (beta != 0.f && !C)) return TCM_ERR_INVALID_ARG;
    const int eo = elem_bytes(out_dtype);
    if ((A && !aligned16(A)) || (B && !aligned16(B)) || (a_scales && !aligned16(a_scales)) ||
        (b_scales && !aligned16(b_scales)) || !aligned16(D) || (C && !aligned16(C)) || (bias && !aligned16(bias)))
        return TCM_ERR_MISALIGNED;
    if ((N * eo) % 16) return TCM_ERR_MISALIGNED;
    const int64_t sms = sm_count();
    if (sms <= 0) return TCM_ERR_CUDA;

    GemmConfig cfg{};
    cfg.kind = bfmt == BF_NVFP4 ? 4 : bfmt == BF_MXFP4 ? 6 : 3;
    cfg.cta_group = 1;
    cfg.ksplit = 1;
    cfg.katoms = 1;
    cfg.bn = N > 128 ? 256 : 128;
    if (g_force_bn.load() == 128 || g_force_bn.load() == 256) cfg.bn = g_force_bn.load();
    // CTA pairs (256 x 256 tiles) when they still give every pair work
    if (cfg.bn == 256 && M > 128 && ((M + 255) / 256) * ((N + 255) / 256) >= sms / 2) cfg.cta_group = 2;
    if (g_force_cta_group.load() == 1 || g_force_cta_group.load() == 2) cfg.cta_group = g_force_cta_group.load();
    if (cfg.bn != 256) cfg.cta_group = 1;

    MxMaps maps;
    std::memset(&maps, 0, sizeof maps);
    if (K > 0) {
        const uint64_t uK = static_cast<uint64_t>(K);
        const uint64_t row_bytes = fp4 ? uK / 2 : uK; // packed E2M1: two values per byte
        const uint32_t box_atoms = static_cast<uint32_t>(k_stage / k_atom);
        if (!encode_kmajor(&maps.a, A, 1, row_bytes, static_cast<uint64_t>(M), row_bytes, 128) ||
            !encode_kmajor(&maps.b, B, 1, row_bytes, static_cast<uint64_t>(N), row_bytes,
                           static_cast<uint32_t>(cfg.bn / cfg.cta_group)) ||
            !encode_sf_atoms(&maps.sa, a_scales, static_cast<uint64_t>(M), uK, static_cast<uint64_t>(k_atom), box_atoms) ||
            !encode_sf_atoms(&maps.sb, b_scales, static_cast<uint64_t>(N), uK, static_cast<uint64_t>(k_atom), box_atoms))
            return TCM_ERR_CUDA;
    }
    GemmParams p{};
    p.kM = static_cast<int>(M);
    p.kN = static_cast<int>(N);
    p.K = static_cast<int>(K);
    p.num_kb = static_cast<int>((K + k_stage - 1) / k_stage);
    p.tiles_m = static_cast<int>((M + 128 * cfg.cta_group - 1) / (128 * cfg.cta_group));
    p.tiles_n = static_cast<int>((N + cfg.bn - 1) / cfg.bn);
    p.num_tiles = p.tiles_m * p.tiles_n;
    p.group_m = g_force_group_m.load() > 0 ? g_force_group_m.load() : 16;
    p.split = 1;
    p.split_begin = p.num_tiles;
    p.tile_begin = 0;
    p.tile_end = p.num_tiles;
    p.clock_probe = g_clock_probe.load();
    p.D = D;
    p.ldd = N;
    p.C = beta != 0.f ? C : nullptr;
    p.ldc = N;
    p.bias = bias;
    p.a_scale = p.b_scale = nullptr;
    p.alpha = alpha;
    p.beta = beta;
    p.out_fmt = static_cast<int>(out_dtype);
    p.bias_fmt = p.out_fmt;
    p.swap_ab = 0;
    // block-scaled instruction descriptor: [7,10) A format, [10,13) B format, [17,23) N >> 3,
    // [23] scale type, [24,29) M >> 4.  kind::mxf8f6f4: E4M3 = 0, E5M2 = 1, scale UE8M0 (1);
    // the per-MMA scale-factor ids ([4,6) B, [29,31) A) are added by the kernel.
    // kind::mxf4nvf4: E2M1 = 1; NVFP4 scale UE4M3 (0), ids 0 (probed on the GPU); MXFP4
    // scale UE8M0 (1), ids 0 or 2 (scale_vec::2X, added by the kernel).
    const uint32_t dims = ((static_cast<uint32_t>(cfg.bn) >> 3) << 17) |
                          (((128u * static_cast<uint32_t>(cfg.cta_group)) >> 4) << 24);
    if (bfmt == BF_NVFP4) p.idesc = (1u << 7) | (1u << 10) | dims;
    else if (bfmt == BF_MXFP4) p.idesc = (1u << 7) | (1u << 10) | (1u << 23) | dims;
    else
        p.idesc = ((a_dtype == TCM_E5M2 ? 1u : 0u) << 7) | ((b_dtype == TCM_E5M2 ? 1u : 0u) << 10) | (1u << 23) | dims;
    p.timeout_ns = timeout_ns();
    p.status = device_status_ptr();
    if (!p.status) return TCM_ERR_CUDA;
    p.fault_inject = g_fault_once.exchange(0);
    const int64_t clusters = sms / cfg.cta_group;
    const int grid = static_cast<int>((p.num_tiles < clusters ? p.num_tiles : clusters) * cfg.cta_group);
    const cudaError_t e = launch_gemm_mx(cfg, maps, p, grid, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? TCM_OK : TCM_ERR_CUDA;
}

tcm_status tcm_gemm_mx(int64_t M, int64_t N, int64_t K, tcm_dtype a_dtype, const void *A, const uint8_t *a_scales,
                       tcm_dtype b_dtype, const void *B, const uint8_t *b_scales, const void *C, void *D,
                       float alpha, float beta, const void *bias, tcm_dtype out_dtype, tcm_stream_t stream)
{
    const bool a4 = a_dtype == TCM_E2M1, b4 = b_dtype == TCM_E2M1;
    if (a4 != b4) return TCM_ERR_UNSUPPORTED; // E2M1 with E2M1 only (MXFP4)
    return block_scaled_impl(a4 ? BF_MXFP4 : BF_MXFP8, M, N, K, a_dtype, A, a_scales, b_dtype, B, b_scales, C, D,
                             alpha, beta, bias, out_dtype, stream);
}

tcm_status tcm_gemm_nvfp4(int64_t M, int64_t N, int64_t K, const void *A, const uint8_t *a_scales, const void *B,
                          const uint8_t *b_scales, const void *C, void *D, float alpha, float beta, const void *bias,
                          tcm_dtype out_dtype, tcm_stream_t stream)
{
    return block_scaled_impl(BF_NVFP4, M, N, K, TCM_E2M1, A, a_scales, TCM_E2M1, B, b_scales, C, D, alpha, beta,
                             bias, out_dtype, stream);
}

int64_t tcm_mx_scales_bytes(int64_t rows, int64_t K)
{
    if (rows < 0 || K < 0 || K % 32 != 0) return -1;
    return ((rows + 127) / 128) * ((K + 127) / 128) * 512;
}

tcm_status tcm_mx_pack_scales(int64_t rows, int64_t K, const uint8_t *scales, uint8_t *packed, tcm_stream_t stream)
{
    if (rows < 0 || K < 0 || K % 32 != 0) return TCM_ERR_INVALID_ARG;
    if (rows > INT32_MAX / 2 || K > INT32_MAX / 2) return TCM_ERR_UNSUPPORTED;
    if (rows == 0 || K == 0) return TCM_OK;
    if (!scales || !packed) return TCM_ERR_INVALID_ARG;
    if (!aligned16(packed)) return TCM_ERR_MISALIGNED;
    return launch_mx_pack_scales(scales, rows, K / 32, 127u, packed, reinterpret_cast<cudaStream_t>(stream)) ==
                   cudaSuccess
               ? TCM_OK
               : TCM_ERR_CUDA;
}

int64_t tcm_nvfp4_scales_bytes(int64_t rows, int64_t K)
{
    if (rows < 0 || K < 0 || K % 16 != 0) return -1;
    return ((rows + 127) / 128) * ((K + 63) / 64) * 512;
}

tcm_status tcm_nvfp4_pack_scales(int64_t rows, int64_t K, const uint8_t *scales, uint8_t *packed, tcm_stream_t stream)
{
    if (rows < 0 || K < 0 || K % 16 != 0) return TCM_ERR_INVALID_ARG;
    if (rows > INT32_MAX / 2 || K > INT32_MAX / 2) return TCM_ERR_UNSUPPORTED;
    if (rows == 0 || K == 0) return TCM_OK;
    if (!scales || !packed) return TCM_ERR_INVALID_ARG;
    if (!aligned16(packed)) return TCM_ERR_MISALIGNED;
    // padding code 0x38 = UE4M3 1.0
    return launch_mx_pack_scales(scales, rows, K / 16, 0x38u, packed, reinterpret_cast<cudaStream_t>(stream)) ==
                   cudaSuccess
               ? TCM_OK
               : TCM_ERR_CUDA;
}

// INT8: K rounded up to whole 64-element K blocks in the bf16 copies
static int64_t i8_pitch(int64_t K) { return (K + 63) / 64 * 64; }

int64_t tcm_gemm_i8_workspace_bytes(int64_t M, int64_t N, int64_t K)
{
    if (M < 1 || N < 1 || K < 0 || K > 131071) return -1;
    return (M + N) * i8_pitch(K) * 2;
}

tcm_status tcm_gemm_i8(int64_t M, int64_t N, int64_t K, const int8_t *A, int64_t lda, const int8_t *B, int64_t ldb,
                       const int32_t *C, int64_t ldc, int32_t *D, int64_t ldd, void *workspace, int64_t workspace_bytes,
                       tcm_stream_t stream)
{
    if (M < 1 || N < 1 || K < 0) return TCM_ERR_INVALID_ARG;
    if (K > 131071 || M > INT32_MAX / 2 || N > INT32_MAX / 2) return TCM_ERR_UNSUPPORTED;
    if (!D || (K > 0 && (!A || !B || !workspace)) || lda < K || ldb < K || ldd < N || (C && ldc < N))
        return TCM_ERR_INVALID_ARG;
    if (!aligned16(D) || ldd % 4 || (C && (!aligned16(C) || ldc % 4)) || (workspace && !aligned16(workspace)))
        return TCM_ERR_MISALIGNED;
    const int64_t kp = i8_pitch(K);
    if (K > 0 && workspace_bytes < (M + N) * kp * 2) return TCM_ERR_INVALID_ARG;
    const int64_t sms = sm_count();
    if (sms <= 0) return TCM_ERR_CUDA;
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    uint8_t *wa = static_cast<uint8_t *>(workspace);
    uint8_t *wb = wa ? wa + M * kp * 2 : nullptr;

    CUtensorMap tmA, tmB;
    std::memset(&tmA, 0, sizeof tmA);
    std::memset(&tmB, 0, sizeof tmB);
    if (K > 0) {
        if (!encode_kmajor(&tmA, wa, 2, static_cast<uint64_t>(kp), static_cast<uint64_t>(M), static_cast<uint64_t>(kp),
                           128) ||
            !encode_kmajor(&tmB, wb, 2, static_cast<uint64_t>(kp), static_cast<uint64_t>(N), static_cast<uint64_t>(kp),
                           128))
            return TCM_ERR_CUDA;
    }
    GemmParams p{};
    p.kM = static_cast<int>(M);
    p.kN = static_cast<int>(N);
    p.K = static_cast<int>(K);
    p.num_kb = static_cast<int>(kp / 64);
    p.tiles_m = static_cast<int>((M + 255) / 256);
    p.tiles_n = static_cast<int>((N + 255) / 256);
    p.num_tiles = p.tiles_m * p.tiles_n;
    p.group_m = g_force_group_m.load() > 0 ? g_force_group_m.load() : 16;
    p.split = 1;
    p.split_begin = p.num_tiles;
    p.tile_begin = 0;
    p.tile_end = p.num_tiles;
    p.D = D;
    p.ldd = ldd;
    p.C = C;
    p.ldc = ldc;
    p.idesc = make_idesc(1u, 1u, 256u, 256u); // bf16 x bf16, M = 256 (CTA pair), N = 256
    p.clock_probe = g_clock_probe.load();
    p.timeout_ns = timeout_ns();
    p.status = device_status_ptr();
    if (!p.status) return TCM_ERR_CUDA;
    p.fault_inject = g_fault_once.exchange(0);
    if (K > 0 && (launch_i8_to_bf16(A, M, K, lda, wa, kp, st) != cudaSuccess ||
                  launch_i8_to_bf16(B, N, K, ldb, wb, kp, st) != cudaSuccess))
        return TCM_ERR_CUDA;
    const int64_t clusters = sms / 2;
    const int grid = static_cast<int>((p.num_tiles < clusters ? p.num_tiles : clusters) * 2);
    return launch_gemm_i8(tmA, tmB, p, grid, st) == cudaSuccess ? TCM_OK : TCM_ERR_CUDA;
}

tcm_status tcm_get_device_status(tcm_stream_t stream, int32_t *code, int32_t *site)
{
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return TCM_ERR_CUDA;
    int host[2] = {0, 0};
    if (cudaMemcpyFromSymbol(host, g_device_status, sizeof host) != cudaSuccess) return TCM_ERR_CUDA;
    if (code) *code = host[0];
    if (site) *site = host[1];
    return TCM_OK;
}

tcm_status tcm_clear_device_status(void)
{
    const int zero[2] = {0, 0};
    if (cudaMemcpyToSymbol(g_device_status, zero, sizeof zero) != cudaSuccess) return TCM_ERR_CUDA;
    return TCM_OK;
}

} // extern "C"
