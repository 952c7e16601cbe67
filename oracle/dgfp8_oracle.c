/*
 * dgfp8_oracle.c -- plain CPU oracle for FP8 (E4M3) 128x128 block quantization
 * and the block-scaled NT GEMM (dense and M-grouped contiguous).
 *
 * TEST INFRASTRUCTURE. Only the tests, the smoke check and the benchmark's
 * CPU-baseline / reference leg may load this file. It shares no code, header,
 * table or constant with the CUDA library, and it never reads anything the
 * CUDA library produced unless a test hands it inputs for comparison.
 *
 * Sources (web pages about DeepGEMM; cited by page and section):
 *   [FP8-walkthrough]  lpnh.cn/news/2826317, the untitled DeepGEMM walkthrough:
 *                      §2.2 (E4M3 inputs, 128x128 blocks, scale_a*scale_b,
 *                      FP32 accumulation), §3.1 (scale = max_abs / 448, FP32
 *                      scales in their own array), §4.2 (the five quantization
 *                      steps and the round-to-nearest-even tip), §4.3 (FP64 CPU
 *                      reference), §5.4 (all-zero blocks must be special-cased).
 *   [DeepGEMM-lib]     pzsr.cn/news/21800, "DeepGEMM: GPU上的高效BLAS内核库解析":
 *                      §3.1 (NT layout; FP32 scales, or packed UE8M0 powers of
 *                      two), §2.3/§3.2 (M-grouped GEMM for MoE experts), §4.1
 *                      (fp8_gemm_nt(c, a, b, a_sf, b_sf) argument order).
 *
 * Readings where the pages leave a step open:
 *   - E4M3 is the OCP "fn" layout: s.eeee.mmm, bias 7, no infinities, codes
 *     0x7F/0xFF are NaN; the pages fix only "E4M3" and "max 448".
 *   - "divide each element by scale" is IEEE binary32 division x / s rounded to
 *     nearest, then a second rounding to E4M3 (nearest, ties to even mantissa),
 *     saturating to +-448 (the amax element can land a hair above 448).
 *   - The sign of zero is kept: a negative input that rounds to zero gives 0x80.
 *   - An all-zero block, or one whose amax/448 underflows to 0 in FP32, gets
 *     scale 1.0 (so every code is a signed zero).
 *   - Power-of-two (UE8M0) scales: the FP32 scale is rounded UP to the next
 *     power of two, then clamped to >= 2^-127 (the smallest UE8M0 value), so
 *     |x / s| never exceeds 448.
 *   - GEMM: C[i,j] = sum over 128-wide K blocks kb of
 *       sa[i/128, kb] * sb[j/128, kb] * sum_{k in kb} dec(qa[i,k]) * dec(qb[j,k])
 *     evaluated in double. The inner sum is exact in double (products of two
 *     E4M3 values have at most 8 significant bits and span 2^-18..2^17.6, so a
 *     128-term sum needs at most ~43 bits).
 *
 * Build: gcc -O2 -std=c11 -fopenmp -ffp-contract=off -shared -fPIC (no
 * fast-math: the division and comparisons below must be IEEE).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_BLOCK 128   /* [FP8-walkthrough] §2.2, §4.2 step 1: 128x128 blocks */
#define ORACLE_E4M3_MAX 448.0 /* [FP8-walkthrough] §3.1: largest E4M3 magnitude */

/* ------------------------------------------------------------------------- */
/* E4M3 decoding, written from the OCP E4M3 bit layout.                      */
/* ------------------------------------------------------------------------- */

/* Value of one E4M3 code; NaN for the two NaN codes 0x7F and 0xFF. */
static double e4m3_decode_one(unsigned code)
{
    const unsigned sign = (code >> 7) & 1u;
    const unsigned e = (code >> 3) & 0xFu;
    const unsigned m = code & 0x7u;
    double mag;
    if (e == 0xFu && m == 0x7u)
        return NAN;
    if (e == 0)
        mag = ldexp((double)m / 8.0, -6);          /* subnormal: m/8 * 2^-6 */
    else
        mag = ldexp(1.0 + (double)m / 8.0, (int)e - 7);
    return sign ? -mag : mag;
}

static double g_table[256];
static int g_table_ready = 0;

static void table_init(void)
{
    if (g_table_ready)
        return;
    for (unsigned c = 0; c < 256; ++c)
        g_table[c] = e4m3_decode_one(c);
    g_table_ready = 1;
}

/* Fill out[256] with the decode table. */
void oracle_e4m3_table(double *out)
{
    table_init();
    memcpy(out, g_table, sizeof(g_table));
}

/* ------------------------------------------------------------------------- */
/* Round a binary32 value to the nearest E4M3 code ([FP8-walkthrough] §4.2   */
/* step 4 and its RNE tip). Positive codes 0x00..0x7E are in increasing      */
/* order of magnitude, so the nearest code is one of the two codes that       */
/* bracket |v|; the midpoint of two E4M3 values is exact in double, so the    */
/* comparison below is exact.                                                 */
/* ------------------------------------------------------------------------- */
uint8_t oracle_e4m3_encode(float v)
{
    table_init();
    const unsigned sign = signbit(v) ? 0x80u : 0u;
    const double a = fabs((double)v);
    unsigned code;
    if (!(a < ORACLE_E4M3_MAX)) {
        code = 0x7Eu;                               /* saturate to 448 */
    } else {
        /* largest lo in [0, 0x7D] with table[lo] <= a (binary search) */
        unsigned lo = 0, hi = 0x7Eu;                /* invariant: table[lo] <= a < table[hi] */
        while (hi - lo > 1) {
            const unsigned mid = (lo + hi) / 2;
            if (g_table[mid] <= a)
                lo = mid;
            else
                hi = mid;
        }
        const double midpoint = 0.5 * (g_table[lo] + g_table[hi]);
        if (a < midpoint)
            code = lo;
        else if (a > midpoint)
            code = hi;
        else
            code = (lo & 1u) ? hi : lo;             /* tie: even mantissa */
    }
    return (uint8_t)(sign | code);
}

/* Encode an array (used by the pin tests). */
void oracle_e4m3_encode_array(const float *v, int64_t n, uint8_t *out)
{
    table_init();
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_e4m3_encode(v[i]);
}

/* Smallest power of two >= s (s > 0, finite), clamped to >= 2^-127, the
 * smallest UE8M0 value ([DeepGEMM-lib] §3.1 packed UE8M0 scales). */
float oracle_pow2_ceil(float s)
{
    int e;
    const float m = frexpf(s, &e);                  /* s = m * 2^e, m in [0.5, 1) */
    float p = (m == 0.5f) ? s : ldexpf(1.0f, e);
    const float lo = ldexpf(1.0f, -127);
    if (p < lo)
        p = lo;
    return p;
}

/* ------------------------------------------------------------------------- */
/* Block quantizer ([FP8-walkthrough] §4.2 steps 1-5, §3.1, §5.4).            */
/*   x: float [rows][ld_x] row-major; q: uint8 [rows][ld_q]; scales: float    */
/*   [ceil(rows/128)][ceil(cols/128)] row-major. mode 0 = FP32 scales,        */
/*   mode 1 = power-of-two (UE8M0) scales. Inputs must be finite.             */
/* Returns 0 on success, -1 if an input is not finite.                        */
/* ------------------------------------------------------------------------- */
int oracle_quantize(const float *x, int64_t rows, int64_t cols, int64_t ld_x,
                    int mode, uint8_t *q, int64_t ld_q, float *scales)
{
    table_init();
    const int64_t nbr = (rows + ORACLE_BLOCK - 1) / ORACLE_BLOCK;
    const int64_t nbc = (cols + ORACLE_BLOCK - 1) / ORACLE_BLOCK;
    int bad = 0;
#pragma omp parallel for schedule(dynamic) reduction(| : bad)
    for (int64_t b = 0; b < nbr * nbc; ++b) {
        const int64_t bi = b / nbc, bj = b % nbc;
        const int64_t r0 = bi * ORACLE_BLOCK, c0 = bj * ORACLE_BLOCK;
        const int64_t r1 = (r0 + ORACLE_BLOCK < rows) ? r0 + ORACLE_BLOCK : rows;
        const int64_t c1 = (c0 + ORACLE_BLOCK < cols) ? c0 + ORACLE_BLOCK : cols;
        /* step 2: max |x| over the block's valid elements */
        float amax = 0.0f;
        for (int64_t r = r0; r < r1; ++r)
            for (int64_t c = c0; c < c1; ++c) {
                const float ax = fabsf(x[r * ld_x + c]);
                if (!isfinite(ax))
                    bad = 1;
                if (ax > amax)
                    amax = ax;
            }
        /* step 3: scale = max_abs / 448, in FP32 */
        float s = amax / 448.0f;
        if (s == 0.0f)
            s = 1.0f;                               /* all-zero block */
        if (mode == 1)
            s = oracle_pow2_ceil(s);
        scales[bi * nbc + bj] = s;                  /* step 5: own array */
        /* step 4: divide by the scale, round to the nearest E4M3 value */
        for (int64_t r = r0; r < r1; ++r)
            for (int64_t c = c0; c < c1; ++c) {
                const float v = x[r * ld_x + c] / s;
                q[r * ld_q + c] = oracle_e4m3_encode(v);
            }
    }
    return bad ? -1 : 0;
}

/* ------------------------------------------------------------------------- */
/* Row-wise 1x128 quantizer: the same steps with blocks of one row and 128    */
/* columns ([FP8-walkthrough] §2.3: the block granularity is a trade-off;     */
/* [DeepGEMM-lib] §3.1: per-token activation scales beside 128x128 weight    */
/* scales).                                                                  */
/*   scales: float [rows][ceil(cols/128)] row-major. mode as above.           */
/* Returns 0 on success, -1 if an input is not finite.                        */
/* ------------------------------------------------------------------------- */
int oracle_quantize_1x128(const float *x, int64_t rows, int64_t cols, int64_t ld_x,
                          int mode, uint8_t *q, int64_t ld_q, float *scales)
{
    table_init();
    const int64_t nbc = (cols + ORACLE_BLOCK - 1) / ORACLE_BLOCK;
    int bad = 0;
#pragma omp parallel for schedule(static) reduction(| : bad)
    for (int64_t r = 0; r < rows; ++r) {
        const float *xrow = x + r * ld_x;
        for (int64_t bj = 0; bj < nbc; ++bj) {
            const int64_t c0 = bj * ORACLE_BLOCK;
            const int64_t c1 = (c0 + ORACLE_BLOCK < cols) ? c0 + ORACLE_BLOCK : cols;
            float amax = 0.0f;
            for (int64_t c = c0; c < c1; ++c) {
                const float ax = fabsf(xrow[c]);
                if (!isfinite(ax))
                    bad = 1;
                if (ax > amax)
                    amax = ax;
            }
            float s = amax / 448.0f;
            if (s == 0.0f)
                s = 1.0f;
            if (mode == 1)
                s = oracle_pow2_ceil(s);
            scales[r * nbc + bj] = s;
            for (int64_t c = c0; c < c1; ++c)
                q[r * ld_q + c] = oracle_e4m3_encode(xrow[c] / s);
        }
    }
    return bad ? -1 : 0;
}

/* ------------------------------------------------------------------------- */
/* Block-scaled NT GEMM in double ([FP8-walkthrough] §2.2, §4.3;             */
/* [DeepGEMM-lib] §3.1 NT layout, §4.1).                                      */
/*   A codes qa [M][ld_a] (K contiguous), scales sa [ceil(M/128)][K/128];     */
/*   B codes qb [N][ld_b] (K contiguous), scales sb [ceil(N/128)][K/128].     */
/*   For each requested row i = rows[r] (0 <= r < nrows) and every column j:  */
/*     C[r][j] = sum_kb sa[i/128,kb] * sb[j/128,kb] *                         */
/*               sum_{k in kb} dec(qa[i,k]) * dec(qb[j,k])                     */
/*     E[r][j] = sum_kb sa * sb * sum_{k in kb} |dec(qa[i,k]) * dec(qb[j,k])| */
/*   E (may be NULL) is the magnitude sum used by the parity tolerance.       */
/*   K must be a multiple of 128.                                             */
/* ------------------------------------------------------------------------- */
static void gemm_row(const uint8_t *arow, const float *sa_row,
                     const uint8_t *qb, int64_t ld_b, const float *sb,
                     int64_t N, int64_t K, double *crow, double *erow)
{
    const int64_t nkb = K / ORACLE_BLOCK;
    for (int64_t j = 0; j < N; ++j) {
        const uint8_t *brow = qb + j * ld_b;
        const float *sb_row = sb + (j / ORACLE_BLOCK) * nkb;
        double acc = 0.0, mag = 0.0;
        for (int64_t kb = 0; kb < nkb; ++kb) {
            double p = 0.0, pabs = 0.0;
            for (int64_t k = kb * ORACLE_BLOCK; k < (kb + 1) * ORACLE_BLOCK; ++k) {
                const double t = g_table[arow[k]] * g_table[brow[k]];
                p += t;
                pabs += fabs(t);
            }
            const double scale = (double)sa_row[kb] * (double)sb_row[kb];
            acc += scale * p;
            mag += fabs(scale) * pabs;
        }
        crow[j] = acc;
        if (erow)
            erow[j] = mag;
    }
}

void oracle_gemm_nt_rows(const uint8_t *qa, int64_t ld_a, const float *sa,
                         const uint8_t *qb, int64_t ld_b, const float *sb,
                         int64_t M, int64_t N, int64_t K,
                         const int64_t *rows, int64_t nrows,
                         double *C, double *E)
{
    table_init();
    (void)M;
    const int64_t nkb = K / ORACLE_BLOCK;
#pragma omp parallel for schedule(dynamic)
    for (int64_t r = 0; r < nrows; ++r) {
        const int64_t i = rows[r];
        gemm_row(qa + i * ld_a, sa + (i / ORACLE_BLOCK) * nkb, qb, ld_b, sb, N, K,
                 C + r * N, E ? E + r * N : NULL);
    }
}

/* Same with one A scale per row and K block: sa [M][K/128]. */
void oracle_gemm_nt_rows_a1x128(const uint8_t *qa, int64_t ld_a, const float *sa,
                                const uint8_t *qb, int64_t ld_b, const float *sb,
                                int64_t M, int64_t N, int64_t K,
                                const int64_t *rows, int64_t nrows,
                                double *C, double *E)
{
    table_init();
    (void)M;
    const int64_t nkb = K / ORACLE_BLOCK;
#pragma omp parallel for schedule(dynamic)
    for (int64_t r = 0; r < nrows; ++r) {
        const int64_t i = rows[r];
        gemm_row(qa + i * ld_a, sa + i * nkb, qb, ld_b, sb, N, K,
                 C + r * N, E ? E + r * N : NULL);
    }
}

/* ------------------------------------------------------------------------- */
/* M-grouped contiguous GEMM ([DeepGEMM-lib] §2.3, §3.2, §3.3).               */
/*   A [M_tot][ld_a] with scales sa [M_tot/128][K/128]; B [G][N][K] packed    */
/*   (row stride K) with scales sb [G][ceil(N/128)][K/128]; m_indices[i] is   */
/*   the expert of row i, or -1 for a padding row, whose output is zero.      */
/*   Computes the requested rows like oracle_gemm_nt_rows, with B and sb of   */
/*   expert m_indices[i]. Returns -1 if an index is >= G.                     */
/* ------------------------------------------------------------------------- */
static int grouped_rows(const uint8_t *qa, int64_t ld_a, const float *sa, int64_t sa_rows_per_scale,
                        const uint8_t *qb, const float *sb, int64_t G,
                        const int32_t *m_indices, int64_t N, int64_t K,
                        const int64_t *rows, int64_t nrows, double *C, double *E);

int oracle_grouped_gemm_rows(const uint8_t *qa, int64_t ld_a, const float *sa,
                             const uint8_t *qb, const float *sb, int64_t G,
                             const int32_t *m_indices, int64_t M_tot,
                             int64_t N, int64_t K,
                             const int64_t *rows, int64_t nrows,
                             double *C, double *E)
{
    (void)M_tot;
    return grouped_rows(qa, ld_a, sa, ORACLE_BLOCK, qb, sb, G, m_indices, N, K, rows, nrows, C, E);
}

/* Same with one A scale per row and K block: sa [M_tot][K/128]. */
int oracle_grouped_gemm_rows_a1x128(const uint8_t *qa, int64_t ld_a, const float *sa,
                                    const uint8_t *qb, const float *sb, int64_t G,
                                    const int32_t *m_indices, int64_t M_tot,
                                    int64_t N, int64_t K,
                                    const int64_t *rows, int64_t nrows,
                                    double *C, double *E)
{
    (void)M_tot;
    return grouped_rows(qa, ld_a, sa, 1, qb, sb, G, m_indices, N, K, rows, nrows, C, E);
}

/* Rows of the grouped GEMM; A scale row of output row i is i / sa_rows_per_scale. */
static int grouped_rows(const uint8_t *qa, int64_t ld_a, const float *sa, int64_t sa_rows_per_scale,
                        const uint8_t *qb, const float *sb, int64_t G,
                        const int32_t *m_indices, int64_t N, int64_t K,
                        const int64_t *rows, int64_t nrows, double *C, double *E)
{
    table_init();
    const int64_t nkb = K / ORACLE_BLOCK;
    const int64_t nbn = (N + ORACLE_BLOCK - 1) / ORACLE_BLOCK;
    int bad = 0;
#pragma omp parallel for schedule(dynamic) reduction(| : bad)
    for (int64_t r = 0; r < nrows; ++r) {
        const int64_t i = rows[r];
        const int32_t g = m_indices[i];
        double *crow = C + r * N;
        double *erow = E ? E + r * N : NULL;
        if (g < 0 || g >= G) {
            if (g >= G)
                bad = 1;
            for (int64_t j = 0; j < N; ++j) {
                crow[j] = 0.0;
                if (erow)
                    erow[j] = 0.0;
            }
            continue;
        }
        gemm_row(qa + i * ld_a, sa + (i / sa_rows_per_scale) * nkb,
                 qb + (int64_t)g * N * K, K, sb + (int64_t)g * nbn * nkb, N, K,
                 crow, erow);
    }
    return bad ? -1 : 0;
}

/* Number of OpenMP threads the oracle runs on. */
int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0)
        omp_set_num_threads(n);
#else
    (void)n;
#endif
}
