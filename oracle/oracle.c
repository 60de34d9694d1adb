/*
 * CPU oracle for the DeepGEMM-style FP8 GEMM with fine-grained scaling.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, obviously correct
 * definition that the CUDA path is checked against.  Only the test suite, the
 * smoke check and the CPU-baseline leg of the benchmark may load it.  It
 * shares no code, header, table or constant with the CUDA library.
 *
 * Sources (page title, then section):
 *   [P2] "DeepGEMM：一款支持FP8通用矩阵乘法(GEMM)的开源库"
 *        功能特色/细粒度缩放功能, 技术细节/两级累加技术, 功能特色/支持多种数据排列方式
 *   [P4] the 2kiu.com DeepGEMM tutorial, sections 2.2 低精度计算带来的新挑战,
 *        3.3 聚焦FP8, 4.4 精度控制与数值稳定性
 *   [P3] "DeepGEMM：面向大模型的高效矩阵计算加速方案", 四.2 (the per-expert loop
 *        that a grouped GEMM replaces)
 *   [P4] sections 1 and 2.2 (BF16 as the other low-precision format) and 7
 *        (MX / micro-scaling formats as the next step); the MX functions
 *        restate the OCP Microscaling Formats (MX) v1.0 specification (32-value
 *        blocks sharing an E8M0 power-of-two scale), which the pages point to
 *        but do not define
 *
 * Readings where the pages are silent:
 *   - E4M3 for both operands, bias 7, max 448, NaN at 0x7F/0xFF, no infinities.
 *   - scale s = max(amax, 1e-4) / 448 in fp32 (IEEE division); q = RNE-saturating
 *     E4M3 encode of fp32(x / s).
 *   - per 128-wide K block, the exact block sum p (in double) is rounded once
 *     to fp32 and promoted with acc = fmaf(p, sfa*sfb, acc), K blocks ascending.
 *   - D = bf16 round-to-nearest-even of acc.
 *   - BF16 GEMM: the exact sum of products, rounded to fp32, then to bf16.
 *   - MX: scale exponent floor(log2 amax) - 8 clamped to [-127, 127] (-127 for
 *     an all-zero block), elements E4M3 RNE saturating at 448; the GEMM is the
 *     exact sum of scaled 32-block sums, rounded to fp32, then to bf16.
 *
 * Parity pins: every function here is pinned by the CPU tests (closed forms,
 * library conversions, brute force and invariants); none is "parity unpinned".
 *
 * Build: gcc -O2 -ffp-contract=off -fopenmp -shared -fPIC (no fast-math, no
 * implicit FMA contraction: the only FMA is the explicit fmaf below).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_QBLOCK 128 /* 1x128 activation groups, 128x128 weight blocks */

/* ---------------------------------------------------------------- E4M3 --- */

/* Closed-form E4M3 decode: sign s, exponent e (4 bits, bias 7), mantissa m
 * (3 bits).  e==15 && m==7 is NaN; e==0 is subnormal (m * 2^-9). */
double oracle_e4m3_decode(uint8_t c)
{
    int s = (c >> 7) & 1;
    int e = (c >> 3) & 15;
    int m = c & 7;
    double mag;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        mag = ldexp((double)m, -9);
    else
        mag = ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -mag : mag;
}

/* The 256 decoded E4M3 values, filled from the closed form above when the
 * library is loaded (a lookup of that formula, not a second definition). */
static double g_dec[256];

__attribute__((constructor)) static void fill_decode_table(void)
{
    int c;
    for (c = 0; c < 256; ++c)
        g_dec[c] = oracle_e4m3_decode((uint8_t)c);
}

/* Brute-force RNE encode with saturation: the nearest of the 127 finite
 * magnitudes (codes 0x00..0x7E); on an exact tie the code with an even
 * mantissa (code LSB 0) wins; |x| >= 448 (and +-inf) saturates to 448; NaN
 * maps to 0x7F with the input's sign.  The sign bit is copied from x, so a
 * tiny negative value encodes as 0x80 (-0).  This is the definition; the
 * quantisers use oracle_e4m3_encode below, which the tests pin to it. */
uint8_t oracle_e4m3_encode_bruteforce(float x)
{
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double ax = fabs((double)x);
    int best = 0;
    double best_d = INFINITY;
    int c;
    if (isnan(x))
        return (uint8_t)(sign | 0x7F);
    if (ax >= 448.0)
        return (uint8_t)(sign | 0x7E);
    for (c = 0; c <= 0x7E; ++c) {
        double d = fabs(ax - oracle_e4m3_decode((uint8_t)c));
        if (d < best_d || (d == best_d && (c & 1) == 0)) {
            best_d = d;
            best = c;
        }
    }
    return (uint8_t)(sign | best);
}

/* The same encode, found faster: the finite magnitudes grow strictly with the
 * code, so |x| lies between two neighbouring codes lo < hi (bisection); the
 * nearer one wins and an exact tie goes to the even code.  Both distances are
 * exact in double (neighbours are within a factor of two of |x|, or zero). */
uint8_t oracle_e4m3_encode(float x)
{
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double ax = fabs((double)x);
    int lo = 0, hi = 0x7E, pick;
    double d_lo, d_hi;
    if (isnan(x))
        return (uint8_t)(sign | 0x7F);
    if (ax >= 448.0)
        return (uint8_t)(sign | 0x7E);
    /* invariant: g_dec[lo] <= ax < g_dec[hi] */
    while (hi - lo > 1) {
        int mid = (lo + hi) / 2;
        if (g_dec[mid] <= ax)
            lo = mid;
        else
            hi = mid;
    }
    d_lo = ax - g_dec[lo];
    d_hi = g_dec[hi] - ax;
    if (d_lo < d_hi)
        pick = lo;
    else if (d_hi < d_lo)
        pick = hi;
    else
        pick = (lo & 1) == 0 ? lo : hi;
    return (uint8_t)(sign | pick);
}

/* ---------------------------------------------------------------- BF16 --- */

/* fp32 -> bf16 bits, round to nearest even (NaN -> quiet NaN). */
uint16_t oracle_bf16_rne(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0)
        return (uint16_t)((u >> 16) | 0x0040u);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

float oracle_bf16_to_f32(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* ----------------------------------------------------------- quantisers --- */

/* Scale of one group from its amax: s = max(amax, 1e-4) / 448 (fp32). */
static float group_scale(float amax)
{
    float a = amax > 1e-4f ? amax : 1e-4f;
    return a / 448.0f;
}

/* Activation quantiser, one scale per row per 128-wide K group
 * ([P2] 细粒度缩放功能; [P4] 4.4: scales from data statistics, saturation of
 * out-of-range values).
 *   x   fp32 [M][K] row-major
 *   q   E4M3 [M][K] row-major
 *   sfa fp32 [K/128][ldsfa], M-major: sfa[kb*ldsfa + m] */
void oracle_quant_act_1x128(const float *x, int M, int K, uint8_t *q, float *sfa, int ldsfa)
{
    int KB = K / ORACLE_QBLOCK;
    int m;
#pragma omp parallel for schedule(static)
    for (m = 0; m < M; ++m) {
        int kb, k;
        for (kb = 0; kb < KB; ++kb) {
            const float *xg = x + (size_t)m * K + (size_t)kb * ORACLE_QBLOCK;
            uint8_t *qg = q + (size_t)m * K + (size_t)kb * ORACLE_QBLOCK;
            float amax = 0.0f, s;
            for (k = 0; k < ORACLE_QBLOCK; ++k)
                if (fabsf(xg[k]) > amax)
                    amax = fabsf(xg[k]);
            s = group_scale(amax);
            for (k = 0; k < ORACLE_QBLOCK; ++k)
                qg[k] = oracle_e4m3_encode(xg[k] / s);
            sfa[(size_t)kb * ldsfa + m] = s;
        }
    }
}

/* The same quantiser for bf16 activations: each value is widened exactly to
 * fp32 first. */
void oracle_quant_act_1x128_bf16(const uint16_t *x, int M, int K, uint8_t *q, float *sfa, int ldsfa)
{
    int KB = K / ORACLE_QBLOCK;
    int m;
#pragma omp parallel for schedule(static)
    for (m = 0; m < M; ++m) {
        int kb, k;
        for (kb = 0; kb < KB; ++kb) {
            const uint16_t *xg = x + (size_t)m * K + (size_t)kb * ORACLE_QBLOCK;
            uint8_t *qg = q + (size_t)m * K + (size_t)kb * ORACLE_QBLOCK;
            float amax = 0.0f, s;
            for (k = 0; k < ORACLE_QBLOCK; ++k) {
                float v = fabsf(oracle_bf16_to_f32(xg[k]));
                if (v > amax)
                    amax = v;
            }
            s = group_scale(amax);
            for (k = 0; k < ORACLE_QBLOCK; ++k)
                qg[k] = oracle_e4m3_encode(oracle_bf16_to_f32(xg[k]) / s);
            sfa[(size_t)kb * ldsfa + m] = s;
        }
    }
}

/* Weight quantiser, one scale per 128x128 block (the last N block may be
 * partial).
 *   w   fp32 [N][K] row-major
 *   q   E4M3 [N][K]
 *   sfb fp32 [ceil(N/128)][K/128]: sfb[nb*(K/128) + kb] */
void oracle_quant_weight_128x128(const float *w, int N, int K, uint8_t *q, float *sfb)
{
    int KB = K / ORACLE_QBLOCK;
    int NB = (N + ORACLE_QBLOCK - 1) / ORACLE_QBLOCK;
    int nb;
#pragma omp parallel for schedule(static)
    for (nb = 0; nb < NB; ++nb) {
        int kb, n, k;
        int n0 = nb * ORACLE_QBLOCK;
        int n1 = n0 + ORACLE_QBLOCK < N ? n0 + ORACLE_QBLOCK : N;
        for (kb = 0; kb < KB; ++kb) {
            int k0 = kb * ORACLE_QBLOCK;
            float amax = 0.0f, s;
            for (n = n0; n < n1; ++n)
                for (k = k0; k < k0 + ORACLE_QBLOCK; ++k)
                    if (fabsf(w[(size_t)n * K + k]) > amax)
                        amax = fabsf(w[(size_t)n * K + k]);
            s = group_scale(amax);
            for (n = n0; n < n1; ++n)
                for (k = k0; k < k0 + ORACLE_QBLOCK; ++k)
                    q[(size_t)n * K + k] = oracle_e4m3_encode(w[(size_t)n * K + k] / s);
            sfb[(size_t)nb * KB + kb] = s;
        }
    }
}

/* --------------------------------------------------------------- GEMM ---- */

/* One output row of D = A * B^T with two-level accumulation ([P2] 两级累加技术):
 * for each 128-wide K block, the block's exact sum of E4M3 products (exact in
 * double: every product is a multiple of 2^-18 and |p| < 2^25) is rounded once
 * to fp32 and promoted as acc = fmaf(p, sfa[m,kb] * sfb[n/128,kb], acc), K
 * blocks ascending; then D = bf16_rne(acc).
 *   a_row   E4M3 [K] (row m of A)
 *   sfa_row sfa of row m, element kb at sfa_row[kb * sfa_stride]
 *   b       E4M3 [N][K]
 *   sfb     fp32 [ceil(N/128)][K/128]
 *   d_row   bf16 bits [N] */
static void gemm_row(const uint8_t *a_row, const float *sfa_row, size_t sfa_stride,
                     const uint8_t *b, const float *sfb, int N, int K, uint16_t *d_row,
                     float *acc_out)
{
    int KB = K / ORACLE_QBLOCK;
    int n, kb, k;
    for (n = 0; n < N; ++n) {
        const uint8_t *b_row = b + (size_t)n * K;
        float acc = 0.0f;
        for (kb = 0; kb < KB; ++kb) {
            double p = 0.0;
            float scale;
            for (k = kb * ORACLE_QBLOCK; k < (kb + 1) * ORACLE_QBLOCK; ++k)
                p += g_dec[a_row[k]] * g_dec[b_row[k]];
            scale = sfa_row[(size_t)kb * sfa_stride] * sfb[(size_t)(n / ORACLE_QBLOCK) * KB + kb];
            acc = fmaf((float)p, scale, acc);
        }
        if (acc_out)
            acc_out[n] = acc;
        d_row[n] = oracle_bf16_rne(acc);
    }
}

/* Dense NT GEMM ([P2] 支持多种数据排列方式: the normal layout).
 *   a    E4M3 [M][K], sfa [K/128][ldsfa] (sfa[kb*ldsfa + m])
 *   b    E4M3 [N][K], sfb [ceil(N/128)][K/128]
 *   d    bf16 [M][N]
 *   acc  optional fp32 [M][N] copy of the promoted accumulator (may be NULL)
 *   rows optional list of n_rows row indices to compute (NULL = all M rows);
 *        rows not listed are left untouched. */
void oracle_gemm_nt(const uint8_t *a, const float *sfa, int ldsfa, const uint8_t *b,
                    const float *sfb, uint16_t *d, float *acc, int M, int N, int K,
                    const int32_t *rows, int n_rows)
{
    int count = rows ? n_rows : M;
    int i;
#pragma omp parallel for schedule(dynamic, 1)
    for (i = 0; i < count; ++i) {
        int m = rows ? rows[i] : i;
        gemm_row(a + (size_t)m * K, sfa + m, (size_t)ldsfa, b, sfb, N, K, d + (size_t)m * N,
                 acc ? acc + (size_t)m * N : NULL);
    }
}

/* MoE contiguous layout ([P2] 支持多种数据排列方式 / 应用场景-混合专家模型):
 * the experts' rows are concatenated; row m belongs to expert m_indices[m],
 * and a row whose index is negative is padding and is left untouched.  This is
 * the per-expert loop of [P3] 四.2 written per row.
 *   a [sum_M][K], sfa [K/128][ldsfa], b [G][N][K], sfb [G][ceil(N/128)][K/128],
 *   d [sum_M][N]. */
void oracle_grouped_contiguous(const uint8_t *a, const float *sfa, int ldsfa, const uint8_t *b,
                               const float *sfb, uint16_t *d, const int32_t *m_indices,
                               int sum_M, int N, int K, int G, const int32_t *rows, int n_rows)
{
    int KB = K / ORACLE_QBLOCK;
    int NB = (N + ORACLE_QBLOCK - 1) / ORACLE_QBLOCK;
    int count = rows ? n_rows : sum_M;
    int i;
#pragma omp parallel for schedule(dynamic, 1)
    for (i = 0; i < count; ++i) {
        int m = rows ? rows[i] : i;
        int g = m_indices[m];
        if (g < 0 || g >= G)
            continue;
        gemm_row(a + (size_t)m * K, sfa + m, (size_t)ldsfa, b + (size_t)g * N * K,
                 sfb + (size_t)g * NB * KB, N, K, d + (size_t)m * N, NULL);
    }
}

/* MoE masked layout ([P2] 支持多种数据排列方式): expert g owns a fixed buffer of
 * max_m rows of which the first masked_m[g] are valid (values above max_m are
 * read as max_m); the other rows of d are left untouched.
 *   a [G][max_m][K], sfa [G][K/128][ldsfa], b [G][N][K],
 *   sfb [G][ceil(N/128)][K/128], d [G][max_m][N]. */
void oracle_grouped_masked(const uint8_t *a, const float *sfa, int ldsfa, const uint8_t *b,
                           const float *sfb, uint16_t *d, const int32_t *masked_m, int G,
                           int max_m, int N, int K)
{
    int KB = K / ORACLE_QBLOCK;
    int NB = (N + ORACLE_QBLOCK - 1) / ORACLE_QBLOCK;
    int gm;
#pragma omp parallel for schedule(dynamic, 1)
    for (gm = 0; gm < G * max_m; ++gm) {
        int g = gm / max_m, m = gm % max_m;
        int valid = masked_m[g] < 0 ? 0 : (masked_m[g] > max_m ? max_m : masked_m[g]);
        if (m >= valid)
            continue;
        gemm_row(a + ((size_t)g * max_m + m) * K, sfa + (size_t)g * KB * ldsfa + m,
                 (size_t)ldsfa, b + (size_t)g * N * K, sfb + (size_t)g * NB * KB, N, K,
                 d + ((size_t)g * max_m + m) * N, NULL);
    }
}

/* ------------------------------------------------------------ BF16 GEMM --- */

/* Dense NT GEMM on bf16 operands, no scales (the second low-precision format
 * the pages name beside FP8: 2kiu.com tutorial 1 and 2.2):
 *   D[m][n] = bf16_rne(fp32(sum_k a[m][k] * b[n][k])).
 * The sum is taken in double, which is exact while the products (16
 * significant bits each) span fewer than 53 - 16 - log2(K) binades, as in
 * every pinned case; it is rounded once to fp32 (the accumulator type), then
 * to bf16.
 *   a bf16 bits [M][K], b bf16 bits [N][K], d bf16 bits [M][N]
 *   rows optional list of n_rows rows to compute (NULL = all); others untouched. */
void oracle_gemm_bf16_nt(const uint16_t *a, const uint16_t *b, uint16_t *d, int M, int N, int K,
                         const int32_t *rows, int n_rows)
{
    int count = rows ? n_rows : M;
    int i;
#pragma omp parallel for schedule(dynamic, 1)
    for (i = 0; i < count; ++i) {
        int m = rows ? rows[i] : i;
        const uint16_t *a_row = a + (size_t)m * K;
        int n, k;
        for (n = 0; n < N; ++n) {
            const uint16_t *b_row = b + (size_t)n * K;
            double sum = 0.0;
            for (k = 0; k < K; ++k)
                sum += (double)oracle_bf16_to_f32(a_row[k]) * (double)oracle_bf16_to_f32(b_row[k]);
            d[(size_t)m * N + n] = oracle_bf16_rne((float)sum);
        }
    }
}

/* ------------------------------------------------------ MX (microscaling) --- */
/* The MX formats the pages point to as the next step after per-group FP8
 * scaling (2kiu.com tutorial 7: MX / micro-scaling formats with finer scale
 * granularity), as the OCP Microscaling Formats (MX) specification v1.0
 * defines them: blocks of 32 consecutive elements share one scale of type
 * E8M0, a bare power of two. */

#define ORACLE_MX_BLOCK 32
#define ORACLE_E4M3_EMAX 8 /* exponent of the largest E4M3 power of two (256) */

/* E8M0 scale code c: 2^(c - 127); 0xFF is NaN. */
double oracle_ue8m0_decode(uint8_t c)
{
    if (c == 0xFF)
        return NAN;
    return ldexp(1.0, (int)c - 127);
}

/* MX quantiser of R rows of K values (the specification's conversion of a
 * vector of scalars to MX, with E4M3 elements):
 *   per row and 32-wide block along K: amax = max |x|;
 *   e = floor(log2(amax)) - 8, clamped to [-127, 127] (an all-zero block
 *   takes e = -127); scale code e + 127;
 *   q = E4M3 RNE of x / 2^e, saturating at 448 (the block's largest element
 *   lands in [256, 448]).
 *   x fp32 [R][K]; q out E4M3 [R][K]; sx out E8M0 [R][K/32] (sx[r*(K/32)+kb]).
 * x / 2^e is exact whenever it is a normal fp32 number; smaller quotients
 * encode to +-0 whatever their low bits. */
void oracle_quant_mx_1x32(const float *x, int R, int K, uint8_t *q, uint8_t *sx)
{
    int KB = K / ORACLE_MX_BLOCK;
    int r;
#pragma omp parallel for schedule(static)
    for (r = 0; r < R; ++r) {
        int kb, k;
        for (kb = 0; kb < KB; ++kb) {
            const float *xb = x + (size_t)r * K + (size_t)kb * ORACLE_MX_BLOCK;
            uint8_t *qb = q + (size_t)r * K + (size_t)kb * ORACLE_MX_BLOCK;
            double amax = 0.0;
            int e;
            for (k = 0; k < ORACLE_MX_BLOCK; ++k)
                if (fabs((double)xb[k]) > amax)
                    amax = fabs((double)xb[k]);
            if (amax == 0.0) {
                e = -127;
            } else {
                int ex;
                frexp(amax, &ex); /* amax = f * 2^ex, f in [0.5, 1): floor(log2 amax) = ex - 1 */
                e = ex - 1 - ORACLE_E4M3_EMAX;
                if (e < -127)
                    e = -127;
                if (e > 127)
                    e = 127;
            }
            sx[(size_t)r * KB + kb] = (uint8_t)(e + 127);
            for (k = 0; k < ORACLE_MX_BLOCK; ++k)
                qb[k] = oracle_e4m3_encode((float)ldexp((double)xb[k], -e));
        }
    }
}

/* MX GEMM, dense NT:
 *   D[m][n] = bf16_rne(fp32(sum_kb 2^(sa[m][kb]-127) * 2^(sb[n][kb]-127)
 *                                 * sum_{k in block kb} dec(a[m][k]) * dec(b[n][k]))),
 * kb over the 32-wide K blocks.  Every block sum is a multiple of 2^-18 below
 * 2^23 and the scales are powers of two, so the double sum is exact while the
 * scaled block sums span fewer than ~30 binades (every pinned case); it is
 * rounded once to fp32, then to bf16.
 *   a E4M3 [M][K], sa E8M0 [M][K/32], b E4M3 [N][K], sb E8M0 [N][K/32],
 *   d bf16 bits [M][N]; rows as in oracle_gemm_bf16_nt. */
void oracle_gemm_mx_nt(const uint8_t *a, const uint8_t *sa, const uint8_t *b, const uint8_t *sb,
                       uint16_t *d, int M, int N, int K, const int32_t *rows, int n_rows)
{
    int KB = K / ORACLE_MX_BLOCK;
    int count = rows ? n_rows : M;
    int i;
#pragma omp parallel for schedule(dynamic, 1)
    for (i = 0; i < count; ++i) {
        int m = rows ? rows[i] : i;
        int n, kb, k;
        for (n = 0; n < N; ++n) {
            double sum = 0.0;
            for (kb = 0; kb < KB; ++kb) {
                double p = 0.0;
                for (k = kb * ORACLE_MX_BLOCK; k < (kb + 1) * ORACLE_MX_BLOCK; ++k)
                    p += g_dec[a[(size_t)m * K + k]] * g_dec[b[(size_t)n * K + k]];
                sum += p * oracle_ue8m0_decode(sa[(size_t)m * KB + kb]) * oracle_ue8m0_decode(sb[(size_t)n * KB + kb]);
            }
            d[(size_t)m * N + n] = oracle_bf16_rne((float)sum);
        }
    }
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
