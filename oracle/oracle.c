/*
 * oracle.c -- plain, slow CPU oracle for the tensor-core GEMM and its
 * 2:4 structured-sparse variant.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only tests/, __graft_entry__.smoke() and bench.py's CPU
 * baseline leg use it.  It shares no code, header, table or constant with the
 * CUDA library; its dtype codes (ORC_*) are its own.
 *
 * What it computes (all arithmetic in IEEE binary64, natural k order):
 *
 *   GEMM, "NVIDIA MMA" page, section "从 FMA 到 MMA，再到 GEMM":
 *       D[m,n] = sum_k A[m,k] * B[k,n] + C[m,n]
 *   with A row-major (M x K) and B column-major, i.e. stored as N rows of K
 *   ("CUDA 014 - MMA 指令的用法详解", section "MMA 指令的格式", the .row.col
 *   modifier; the same page's ldmatrix section stores such a B as N x K).
 *
 *   Epilogue, "NVIDIA MMA" page, section "输入/累加/输出": the accumulator is
 *   a separate stage from the output; scale / bias / activation / cast are
 *   applied after the K reduction.  Reading used here (no activation):
 *       ref = alpha * sA * sB * acc + beta * C + bias[n]      (unrounded)
 *   where sA, sB are per-tensor dequantisation factors (1 for bf16/fp16).
 *
 *   2:4 sparsity, "NVIDIA MMA" page, section "稠密乘法与 2:4 结构化稀疏乘法":
 *   along K every group of 4 logical positions keeps 2 values plus their
 *   positions; the page's worked example is logical [a0,0,0,a3] -> values
 *   [a0,a3], metadata [0,3].  Section "Ampere ..." (mma.sp::ordered_metadata)
 *   requires the two positions in ascending order.  Readings where the pages
 *   are silent: keep the two largest |v|, ties to the lower index; the
 *   nibble is i0 | i1<<2; 8 nibbles per uint32 little-endian along K.
 *
 * Input element formats are decoded from their published definitions
 * (IEEE 754 binary16/binary32, bfloat16 = top half of binary32, OCP 8-bit
 * floating point E4M3 "fn" and E5M2); the page lists these types in its
 * "精度总表" table of the "NVIDIA MMA" page.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* The oracle's own element-format codes (E8M0: the UE8M0 block-scale format;
 * E2M1: 4-bit, stored two per byte, element 2i in the low nibble). */
enum { ORC_BF16 = 0, ORC_F16 = 1, ORC_F32 = 2, ORC_E4M3 = 3, ORC_E5M2 = 4, ORC_E8M0 = 5, ORC_E2M1 = 6,
       ORC_UE4M3 = 7 };

/* Width in bytes of one stored element of each format (0 = unknown). */
int orc_elem_bytes(int fmt)
{
    switch (fmt) {
    case ORC_BF16: case ORC_F16: return 2;
    case ORC_F32: return 4;
    case ORC_E4M3: case ORC_E5M2: case ORC_E8M0: case ORC_UE4M3: return 1;
    case ORC_E2M1: return 1; /* a byte holds two elements: see load_code */
    default: return 0;
    }
}

/*
 * Decode one stored code of format fmt to its exact real value.
 *   bfloat16 : s | e(8, bias 127) | m(7)
 *   binary16 : s | e(5, bias 15)  | m(10)
 *   binary32 : the C float with those bits
 *   E4M3 (OCP, "fn"): s | e(4, bias 7) | m(3); no infinities; only
 *              s.1111.111 is NaN, so e=15 with m<7 is an ordinary normal
 *              number (largest 1.75 * 2^8 = 448).
 *   E5M2 (OCP): s | e(5, bias 15) | m(2); e=31 is inf (m=0) or NaN.
 *   E8M0 (OCP MX scale): e(8), value 2^(e - 127); e = 255 is NaN.
 *   E2M1 (OCP FP4): s | e(2, bias 1) | m(1); no infinities or NaN
 *              (magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6).
 *   UE4M3 (NVFP4 block scale): E4M3 without a sign bit: e(4, bias 7) | m(3),
 *              0x7F NaN, largest 448; bit 7 unused (read as 0).
 * A zero exponent field means a subnormal: m * 2^(1 - bias - mbits).
 */
double orc_decode(uint32_t code, int fmt)
{
    int ebits, mbits, bias, sbit;
    switch (fmt) {
    case ORC_BF16: ebits = 8; mbits = 7; bias = 127; break;
    case ORC_F16: ebits = 5; mbits = 10; bias = 15; break;
    case ORC_E4M3: ebits = 4; mbits = 3; bias = 7; break;
    case ORC_UE4M3: ebits = 4; mbits = 3; bias = 7; code &= 0x7Fu; break;
    case ORC_E5M2: ebits = 5; mbits = 2; bias = 15; break;
    case ORC_E2M1: ebits = 2; mbits = 1; bias = 1; code &= 0xFu; break;
    case ORC_F32: {
        float f;
        uint32_t u = code;
        memcpy(&f, &u, sizeof f);
        return (double)f;
    }
    case ORC_E8M0:
        /* unsigned 8-bit exponent, no sign, no mantissa: 2^(e - 127); e = 255 is NaN */
        return (code & 0xFFu) == 0xFFu ? NAN : ldexp(1.0, (int)(code & 0xFFu) - 127);
    default: return NAN;
    }
    sbit = ebits + mbits;
    uint32_t m = code & ((1u << mbits) - 1u);
    uint32_t e = (code >> mbits) & ((1u << ebits) - 1u);
    double sign = ((code >> sbit) & 1u) ? -1.0 : 1.0;
    uint32_t emax = (1u << ebits) - 1u;
    if (fmt == ORC_E4M3 || fmt == ORC_UE4M3) {
        if (e == emax && m == (1u << mbits) - 1u) return NAN;
    } else if (fmt == ORC_E2M1) {
        /* every code is a number */
    } else if (e == emax) {
        return m == 0 ? sign * INFINITY : NAN;
    }
    if (e == 0) return sign * ldexp((double)m, 1 - bias - mbits);
    return sign * ldexp(1.0 + ldexp((double)m, -mbits), (int)e - bias);
}

/* Fetch code number idx of a buffer of format fmt. */
static uint32_t load_code(const void *buf, int fmt, int64_t idx)
{
    if (fmt == ORC_E2M1) {
        const uint8_t b = ((const uint8_t *)buf)[idx >> 1];
        return (idx & 1) ? (uint32_t)(b >> 4) : (uint32_t)(b & 0xFu);
    }
    switch (orc_elem_bytes(fmt)) {
    case 1: return ((const uint8_t *)buf)[idx];
    case 2: return ((const uint16_t *)buf)[idx];
    case 4: return ((const uint32_t *)buf)[idx];
    default: return 0;
    }
}

/* Decode n codes into doubles. */
int orc_decode_array(const void *src, int fmt, int64_t n, double *dst)
{
    if (orc_elem_bytes(fmt) == 0) return -1;
    for (int64_t i = 0; i < n; ++i) dst[i] = orc_decode(load_code(src, fmt, i), fmt);
    return 0;
}

/* Value of every code of a <=16-bit format: table[code] = decode(code). */
static double *decode_table(int fmt)
{
    int bytes = orc_elem_bytes(fmt);
    if (bytes != 1 && bytes != 2) return NULL;
    size_t n = fmt == ORC_E2M1 ? 16 : (size_t)1 << (8 * bytes);
    double *t = (double *)malloc(n * sizeof(double));
    if (!t) return NULL;
    for (size_t c = 0; c < n; ++c) t[c] = orc_decode((uint32_t)c, fmt);
    return t;
}

static double decoded(const void *buf, int fmt, const double *table, int64_t idx)
{
    uint32_t c = load_code(buf, fmt, idx);
    return table ? table[c] : orc_decode(c, fmt);
}

/*
 * Reference GEMM on stored codes.
 *
 * For each requested output (m, n):
 *     acc  = sum_{k=0}^{K-1} a[m,k] * b[n,k]         (fp64, natural k order)
 *     S    = sum_{k=0}^{K-1} |a[m,k] * b[n,k]|
 *     ref  = alpha * sa * sb * acc + beta * c[m,n] + bias[n]
 * a[m,k] = A[m*lda + k]   (row-major A, M x K)
 * b[n,k] = B[n*ldb + k]   (column-major B = N rows of K)
 * c[m,n] = C[m*ldc + n]   (row-major; C may be NULL, then the term is 0)
 * bias may be NULL (then 0).
 *
 * Products of two inputs of at most 11 significant bits are exact in fp64,
 * so acc differs from the exact sum only by the fp64 additions.
 *
 * If nsamp < 0 every output is computed and written row-major to
 * ref[m*N+n], S[m*N+n]; otherwise only (rows[s], cols[s]) for s < nsamp,
 * written to ref[s], S[s].  Returns 0, or -1 on a bad argument.
 */
int orc_gemm(int64_t M, int64_t N, int64_t K,
             int a_fmt, const void *A, int64_t lda,
             int b_fmt, const void *B, int64_t ldb,
             int c_fmt, const void *C, int64_t ldc,
             int bias_fmt, const void *bias,
             double alpha, double beta, double sa, double sb,
             int64_t nsamp, const int64_t *rows, const int64_t *cols,
             double *ref, double *S)
{
    if (M < 0 || N < 0 || K < 0) return -1;
    if (!orc_elem_bytes(a_fmt) || !orc_elem_bytes(b_fmt)) return -1;
    if (C && !orc_elem_bytes(c_fmt)) return -1;
    if (bias && !orc_elem_bytes(bias_fmt)) return -1;
    double *ta = decode_table(a_fmt);
    double *tb = decode_table(b_fmt);
    int64_t total = nsamp < 0 ? M * N : nsamp;
    int bad = 0;

#pragma omp parallel for schedule(dynamic, 16) reduction(| : bad)
    for (int64_t s = 0; s < total; ++s) {
        int64_t m = nsamp < 0 ? s / N : rows[s];
        int64_t n = nsamp < 0 ? s % N : cols[s];
        if (m < 0 || m >= M || n < 0 || n >= N) {
            bad = 1;
            continue;
        }
        double acc = 0.0, sabs = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            double p = decoded(A, a_fmt, ta, m * lda + k) * decoded(B, b_fmt, tb, n * ldb + k);
            acc += p;
            sabs += fabs(p);
        }
        double c = C ? orc_decode(load_code(C, c_fmt, m * ldc + n), c_fmt) : 0.0;
        double bv = bias ? orc_decode(load_code(bias, bias_fmt, n), bias_fmt) : 0.0;
        ref[s] = alpha * sa * sb * acc + beta * c + bv;
        S[s] = sabs;
    }
    free(ta);
    free(tb);
    return bad ? -1 : 0;
}

/*
 * 2:4 prune + compress of a logical row-major M x K matrix A (K % 32 == 0).
 *
 * Group g of row m is A[m, 4g .. 4g+3].  Its two kept positions i0 < i1 are
 * the two largest magnitudes, ties going to the lower index: pick the first
 * position of largest |v|, then the first position of largest |v| among the
 * other three, then order the two ascending.
 *   Ac[m*(K/2) + 2g]     = code of A[m, 4g+i0]
 *   Ac[m*(K/2) + 2g + 1] = code of A[m, 4g+i1]
 *   nibble(g) = i0 | (i1 << 2), placed at bits 4*(g % 8) of
 *   meta[m*(K/32) + g/8].
 * Values are copied as stored codes (no rounding).  Returns 0 or -1.
 */
int orc_sp_compress(int64_t M, int64_t K, int fmt, const void *A, int64_t lda,
                    void *Ac, uint32_t *meta)
{
    int bytes = orc_elem_bytes(fmt);
    if (M < 0 || K < 0 || K % 32 != 0 || bytes == 0 || lda < K) return -1;
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t w = 0; w < K / 32; ++w) meta[m * (K / 32) + w] = 0;
        for (int64_t g = 0; g < K / 4; ++g) {
            double mag[4];
            for (int q = 0; q < 4; ++q)
                mag[q] = fabs(orc_decode(load_code(A, fmt, m * lda + 4 * g + q), fmt));
            int first = 0;
            for (int q = 1; q < 4; ++q)
                if (mag[q] > mag[first]) first = q;
            int second = first == 0 ? 1 : 0;
            for (int q = 0; q < 4; ++q)
                if (q != first && mag[q] > mag[second]) second = q;
            int i0 = first < second ? first : second;
            int i1 = first < second ? second : first;
            uint32_t c0 = load_code(A, fmt, m * lda + 4 * g + i0);
            uint32_t c1 = load_code(A, fmt, m * lda + 4 * g + i1);
            int64_t o = m * (K / 2) + 2 * g;
            if (bytes == 1) {
                ((uint8_t *)Ac)[o] = (uint8_t)c0;
                ((uint8_t *)Ac)[o + 1] = (uint8_t)c1;
            } else if (bytes == 2) {
                ((uint16_t *)Ac)[o] = (uint16_t)c0;
                ((uint16_t *)Ac)[o + 1] = (uint16_t)c1;
            } else {
                ((uint32_t *)Ac)[o] = c0;
                ((uint32_t *)Ac)[o + 1] = c1;
            }
            uint32_t nib = (uint32_t)i0 | ((uint32_t)i1 << 2);
            meta[m * (K / 32) + g / 8] |= nib << (4 * (g % 8));
        }
    }
    return 0;
}

/*
 * Inverse of orc_sp_compress: A[m, 4g+q] = kept value if q is one of the
 * group's two positions, else the code 0 (+0.0).  Returns 0 or -1 (also
 * when a nibble is not ascending, i.e. i0 >= i1).
 */
int orc_sp_decompress(int64_t M, int64_t K, int fmt, const void *Ac,
                      const uint32_t *meta, void *A, int64_t lda)
{
    int bytes = orc_elem_bytes(fmt);
    if (M < 0 || K < 0 || K % 32 != 0 || bytes == 0 || lda < K) return -1;
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t g = 0; g < K / 4; ++g) {
            uint32_t nib = (meta[m * (K / 32) + g / 8] >> (4 * (g % 8))) & 0xFu;
            int i0 = (int)(nib & 3u), i1 = (int)(nib >> 2);
            if (i0 >= i1) return -1;
            int64_t o = m * (K / 2) + 2 * g;
            for (int q = 0; q < 4; ++q) {
                uint32_t c = 0;
                if (q == i0) c = load_code(Ac, fmt, o);
                if (q == i1) c = load_code(Ac, fmt, o + 1);
                int64_t d = m * lda + 4 * g + q;
                if (bytes == 1) ((uint8_t *)A)[d] = (uint8_t)c;
                else if (bytes == 2) ((uint16_t *)A)[d] = (uint16_t)c;
                else ((uint32_t *)A)[d] = c;
            }
        }
    }
    return 0;
}

/*
 * Block-scaled GEMM ("NVIDIA MMA", section "SM100：tcgen05.mma", the
 * block-scaled form): D = C + sum_g (A_{q,g} S_{A,g}) (B_{q,g} S_{B,g}), the
 * scales applied to each K block's partial sum before it enters the total.
 * Blocks are `blk` consecutive K elements; sa[m*lds_a + g] and sb[n*lds_b + g]
 * are the E8M0 scales of block g of row m of A and of row n of B.
 *     acc = sum_g 2^(sa - 127) 2^(sb - 127) sum_{k in g} a[m,k] b[n,k]
 *     S   = sum_g 2^(sa - 127) 2^(sb - 127) sum_{k in g} |a[m,k] b[n,k]|
 *     ref = alpha * acc + beta * c[m,n] + bias[n]
 * All in fp64 (block sums of at most 32 products of <= 4-bit significands
 * are exact; the power-of-two scales are exact).  nsamp / rows / cols as in
 * orc_gemm.  Returns 0 or -1.
 */
int orc_gemm_mx(int64_t M, int64_t N, int64_t K, int64_t blk, int sf_fmt,
                int a_fmt, const void *A, int64_t lda, const uint8_t *sa, int64_t lds_a,
                int b_fmt, const void *B, int64_t ldb, const uint8_t *sb, int64_t lds_b,
                int c_fmt, const void *C, int64_t ldc, int bias_fmt, const void *bias,
                double alpha, double beta,
                int64_t nsamp, const int64_t *rows, const int64_t *cols,
                double *ref, double *S)
{
    if (M < 0 || N < 0 || K < 0 || blk <= 0 || K % blk != 0) return -1;
    if (sf_fmt != ORC_E8M0 && sf_fmt != ORC_UE4M3) return -1;
    if (!orc_elem_bytes(a_fmt) || !orc_elem_bytes(b_fmt)) return -1;
    if (C && !orc_elem_bytes(c_fmt)) return -1;
    if (bias && !orc_elem_bytes(bias_fmt)) return -1;
    double *ta = decode_table(a_fmt);
    double *tb = decode_table(b_fmt);
    int64_t total = nsamp < 0 ? M * N : nsamp;
    int bad = 0;

#pragma omp parallel for schedule(dynamic, 16) reduction(| : bad)
    for (int64_t s = 0; s < total; ++s) {
        int64_t m = nsamp < 0 ? s / N : rows[s];
        int64_t n = nsamp < 0 ? s % N : cols[s];
        if (m < 0 || m >= M || n < 0 || n >= N) {
            bad = 1;
            continue;
        }
        double acc = 0.0, sabs = 0.0;
        for (int64_t g = 0; g < K / blk; ++g) {
            double part = 0.0, pabs = 0.0;
            for (int64_t k = g * blk; k < (g + 1) * blk; ++k) {
                double p = decoded(A, a_fmt, ta, m * lda + k) * decoded(B, b_fmt, tb, n * ldb + k);
                part += p;
                pabs += fabs(p);
            }
            double scale = orc_decode(sa[m * lds_a + g], sf_fmt) * orc_decode(sb[n * lds_b + g], sf_fmt);
            acc += scale * part;
            sabs += scale * pabs;
        }
        double c = C ? orc_decode(load_code(C, c_fmt, m * ldc + n), c_fmt) : 0.0;
        double bv = bias ? orc_decode(load_code(bias, bias_fmt, n), bias_fmt) : 0.0;
        ref[s] = alpha * acc + beta * c + bv;
        S[s] = sabs;
    }
    free(ta);
    free(tb);
    return bad ? -1 : 0;
}

/*
 * Fused epilogue tail, "NVIDIA MMA" page, section "输入/累加/输出": after the K
 * reduction the epilogue scales, adds the bias, applies an activation and
 * casts; an FP8 output feeds the next layer.  Readings where the page is
 * silent: the activation acts on ref = alpha*sA*sB*acc + beta*C + bias;
 *   RELU(x) = x if x > 0 else 0 (a NaN gives 0),
 *   GELU(x) = x * Phi(x) = 0.5 * x * (1 + erf(x / sqrt 2)), Phi the standard
 *             normal distribution function;
 * an FP8 output holds y * RN32(1 / d_scale) (the library's documented rule: one
 * reciprocal rounded to fp32, then a product) rounded to nearest even and saturated to
 * the format's largest finite value (E4M3 448 = 1.75 * 2^8, E5M2 57344 =
 * 1.75 * 2^15); amax = max |y| over the outputs.
 */
enum { ORC_ACT_NONE = 0, ORC_ACT_RELU = 1, ORC_ACT_GELU = 2 };

int orc_activate(int64_t n, const double *x, int act, double *y)
{
    if (act < ORC_ACT_NONE || act > ORC_ACT_GELU) return -1;
    for (int64_t i = 0; i < n; ++i) {
        const double v = x[i];
        if (act == ORC_ACT_RELU) y[i] = v > 0.0 ? v : 0.0;
        else if (act == ORC_ACT_GELU) y[i] = 0.5 * v * (1.0 + erf(v / sqrt(2.0)));
        else y[i] = v;
    }
    return 0;
}

/* The unrounded value an FP8 output element targets: y * mult, saturated, where mult is
 * the library's documented multiplier 1 / d_scale rounded to fp32 (computed exactly by
 * the caller). */
int orc_fp8_target(int64_t n, const double *y, double mult, int fmt, double *out)
{
    double top;
    if (fmt == ORC_E4M3) top = ldexp(1.75, 8);
    else if (fmt == ORC_E5M2) top = ldexp(1.75, 15);
    else return -1;
    for (int64_t i = 0; i < n; ++i) {
        const double t = y[i] * mult;
        out[i] = t > top ? top : (t < -top ? -top : t); /* a NaN passes through */
    }
    return 0;
}

/*
 * Integer GEMM, "NVIDIA MMA" page, section "Ampere：FP16/BF16 与整数 MMA 基线": signed
 * 8-bit A and B, 32-bit integer accumulator and output, .satfinite: the result is
 * clamped to the 32-bit range instead of wrapping.  Reading where the page is silent:
 * the exact sum sum_k a_mk b_nk + c_mn is formed first (64-bit, exact for any K below
 * 2^48) and clamped once at the end.  B is stored N x K (K-major) like the other GEMMs;
 * C (int32, pitch ldc) may be NULL.  Outputs (i, j) for t in [0, n) of rows[t], cols[t]
 * (all M x N in row-major order when rows == NULL) go to out[t].
 */
int orc_gemm_i8(int64_t M, int64_t N, int64_t K, const int8_t *A, int64_t lda, const int8_t *B, int64_t ldb,
                const int32_t *C, int64_t ldc, int64_t n, const int64_t *rows, const int64_t *cols, int32_t *out)
{
    if (M < 0 || N < 0 || K < 0 || lda < K || ldb < K || (C && ldc < N)) return -1;
    if (!rows && n != M * N) return -1;
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < n; ++t) {
        const int64_t i = rows ? rows[t] : t / N;
        const int64_t j = rows ? cols[t] : t % N;
        int64_t acc = 0;
        for (int64_t k = 0; k < K; ++k) acc += (int64_t)A[i * lda + k] * (int64_t)B[j * ldb + k];
        if (C) acc += C[i * ldc + j];
        if (acc > INT32_MAX) acc = INT32_MAX;
        if (acc < INT32_MIN) acc = INT32_MIN;
        out[t] = (int32_t)acc;
    }
    return 0;
}
