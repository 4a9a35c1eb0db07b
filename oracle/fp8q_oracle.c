/*
 * fp8q_oracle.c -- CPU oracle for fine-grained FP8 quantization and the
 * block-scaled FP8 GEMM.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the
 * cpu_baseline / reference legs of bench.py may load this file's library.
 * The CUDA path shares no code, header, table or constant generator with it.
 *
 * It is written to be read against the method, not to be fast: plain loops,
 * one group at a time, fp64 where the method is exact and fl32 (IEEE single,
 * round-to-nearest-even, no FMA contraction: build with -ffp-contract=off)
 * where the method rounds to FP32.
 *
 * Sources (DeepSeek-V3 FP8 training, as retold by five scraped web pages):
 *  - "Deepseek Ai News Expert Interview" (page 2), the E4M3/E5M2 passage:
 *    E4M3 (4-bit exponent, 3-bit mantissa) is used on all tensors; grouping
 *    elements lets a group share exponent bits against FP8's narrow range.
 *  - dssusan.co.kr page (page 3), the Figure 7 (a) passage: activations are
 *    grouped and scaled per 1x128 tile (one token, 128 channels); weights per
 *    128x128 block (128 input x 128 output channels).
 *  - "Eliminate Deepseek Ai News For Good" (page 5), the MMA-precision
 *    passage: tensor-core partial sums are copied to FP32 registers on CUDA
 *    cores when the accumulation interval is reached and accumulated there in
 *    full FP32.
 *  - inprokorea.com page (page 4), the accumulation-interval passage: 128
 *    elements (4 WGMMAs) is the interval.
 *  - "Is aI Hitting a Wall?" (page 1), the dequantization passage: the
 *    dequantization cost is absorbed into that promotion step, i.e. the
 *    scales are applied when a 128-K partial is promoted.
 * What the pages leave open is taken in its plainest reading:
 *  - E4M3 is OCP E4M3FN: bias 7, no infinities, S.1111.111 = NaN, max 448,
 *    subnormals m * 2^-9.  Rounding is round-to-nearest-even, saturating to
 *    +-448 (satfinite).  The sign of zero is kept.
 *  - scale of a group: a = max(amax, 2^-100); s = fl32(a / 448) is stored
 *    (dequantize: x ~ decode(q) * s); inv = fl32(448 / a); q = E4M3(fl32(x*inv)).
 *  - the 128x1 copy groups 128 consecutive tokens of one channel of the
 *    ORIGINAL input and is stored transposed.
 *  - promotion: acc = fl32(acc + fl32(fl32(P_kb) * fl32(sA * sB))), kb in
 *    ascending order ("pages order"); the exact form sums the same terms in
 *    fp64.
 * Parity of everything here is pinned by mathematics (exhaustive codec
 * checks, closed forms, library cross-checks, brute force), not by any
 * number the pages print: the pages print no worked example.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define GROUP 128

/* ------------------------------------------------------------------ */
/* E4M3 codec                                                          */
/* ------------------------------------------------------------------ */

/* decode one E4M3FN code to its exact value (exact in fp32 and fp64) */
float oracle_e4m3_decode(uint8_t c)
{
    int sign = c >> 7;
    int e = (c >> 3) & 0xF;
    int m = c & 0x7;
    double v;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);              /* subnormal: m/8 * 2^-6 */
    else
        v = ldexp((double)(8 + m), e - 10);    /* (1 + m/8) * 2^(e-7)   */
    return (float)(sign ? -v : v);
}

/* encode one finite fp32 value: round to nearest even on the E4M3 grid,
   then saturate to 448 */
uint8_t oracle_e4m3_encode(float v)
{
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    double a = fabs((double)v);
    double quantum, r;
    int ex;
    if (isnan(v))
        return (uint8_t)(sign | 0x7F);
    if (a == 0.0)
        return sign;
    /* grid spacing at |v|: 2^-9 below the smallest normal 2^-6, else
       2^(e-3) where 2^e <= a < 2^(e+1) */
    if (a < ldexp(1.0, -6)) {
        quantum = ldexp(1.0, -9);
    } else {
        (void)frexp(a, &ex);                    /* a = f * 2^ex, f in [0.5,1) */
        quantum = ldexp(1.0, (ex - 1) - 3);
    }
    r = nearbyint(a / quantum) * quantum;       /* default mode: ties to even */
    if (r > 448.0)
        r = 448.0;                              /* satfinite */
    if (r < ldexp(1.0, -6))                     /* subnormal (or 2^-6 = code 8) */
        return (uint8_t)(sign | (uint8_t)(r / ldexp(1.0, -9)));
    (void)frexp(r, &ex);
    {
        int e = ex - 1;                                        /* r in [2^e, 2^(e+1)) */
        int m = (int)((r / ldexp(1.0, e) - 1.0) * 8.0);        /* 0..7, exact */
        return (uint8_t)(sign | ((e + 7) << 3) | m);
    }
}

/* decode table built once from oracle_e4m3_decode (the GEMM below reads
   two codes per multiply-add) */
static double g_decode[256];

__attribute__((constructor)) static void build_decode_table(void)
{
    for (int c = 0; c < 256; ++c)
        g_decode[c] = (double)oracle_e4m3_decode((uint8_t)c);
}

void oracle_e4m3_encode_array(const float *v, int64_t n, uint8_t *out)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_e4m3_encode(v[i]);
}

void oracle_e4m3_decode_array(const uint8_t *c, int64_t n, float *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_e4m3_decode(c[i]);
}

/* ------------------------------------------------------------------ */
/* Group scale and element cast                                        */
/* ------------------------------------------------------------------ */

/* amax -> (s, inv); both IEEE single divisions, round to nearest even */
void oracle_group_scale(float amax, float *s, float *inv)
{
    float a = amax > 0x1p-100f ? amax : 0x1p-100f;
    *s = a / 448.0f;
    *inv = 448.0f / a;
}

/* input element: dtype 0 = BF16 (given as its 16 bits), 1 = FP32 */
static float load_x(const void *x, int dtype, int64_t i)
{
    if (dtype == 0) {
        uint32_t bits = (uint32_t)((const uint16_t *)x)[i] << 16;
        float f;
        memcpy(&f, &bits, 4);
        return f;
    }
    return ((const float *)x)[i];
}

static uint8_t cast_one(float x, float inv)
{
    volatile float prod = x * inv;              /* fl32(x * inv) */
    return oracle_e4m3_encode(prod);
}

/* ------------------------------------------------------------------ */
/* Quantizers                                                          */
/* ------------------------------------------------------------------ */

/* 1x128 activation groups (one token, 128 consecutive channels).
   x[M][K] row-major; q_row[M][K]; s_row[K/128][M] (K-block-major). */
void oracle_quantize_act_rows(const void *x, int dtype, int64_t M, int64_t K,
                              uint8_t *q_row, float *s_row)
{
    int64_t KB = K / GROUP;
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t kb = 0; kb < KB; ++kb) {
            float amax = 0.0f, s, inv;
            for (int64_t j = 0; j < GROUP; ++j) {
                float v = fabsf(load_x(x, dtype, m * K + kb * GROUP + j));
                if (v > amax)
                    amax = v;
            }
            oracle_group_scale(amax, &s, &inv);
            s_row[kb * M + m] = s;
            for (int64_t j = 0; j < GROUP; ++j) {
                int64_t i = m * K + kb * GROUP + j;
                q_row[i] = cast_one(load_x(x, dtype, i), inv);
            }
        }
    }
}

/* Optionally gathered rows: output row r quantizes input row src[r].
   q_row[R][K]; s_row[K/128][R].  Used for quantize-before-dispatch. */
void oracle_quantize_act_rows_gather(const void *x, int dtype, int64_t K,
                                     const int64_t *src, int64_t R,
                                     uint8_t *q_row, float *s_row)
{
    int64_t KB = K / GROUP;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < R; ++r) {
        int64_t m = src[r];
        for (int64_t kb = 0; kb < KB; ++kb) {
            float amax = 0.0f, s, inv;
            for (int64_t j = 0; j < GROUP; ++j) {
                float v = fabsf(load_x(x, dtype, m * K + kb * GROUP + j));
                if (v > amax)
                    amax = v;
            }
            oracle_group_scale(amax, &s, &inv);
            s_row[kb * R + r] = s;
            for (int64_t j = 0; j < GROUP; ++j)
                q_row[r * K + kb * GROUP + j] =
                    cast_one(load_x(x, dtype, m * K + kb * GROUP + j), inv);
        }
    }
}

/* 128x1 groups (128 consecutive tokens of one channel), from the original X,
   stored transposed: q_colT[K][M] (token index contiguous), s_col[M/128][K]. */
void oracle_quantize_act_cols(const void *x, int dtype, int64_t M, int64_t K,
                              uint8_t *q_colT, float *s_col)
{
    int64_t MB = M / GROUP;
#pragma omp parallel for schedule(static)
    for (int64_t k = 0; k < K; ++k) {
        for (int64_t mb = 0; mb < MB; ++mb) {
            float amax = 0.0f, s, inv;
            for (int64_t j = 0; j < GROUP; ++j) {
                float v = fabsf(load_x(x, dtype, (mb * GROUP + j) * K + k));
                if (v > amax)
                    amax = v;
            }
            oracle_group_scale(amax, &s, &inv);
            s_col[mb * K + k] = s;
            for (int64_t j = 0; j < GROUP; ++j) {
                int64_t m = mb * GROUP + j;
                q_colT[k * M + m] = cast_one(load_x(x, dtype, m * K + k), inv);
            }
        }
    }
}

/* 128x128 weight blocks.  w[N][K] row-major (PyTorch Linear layout: N
   output channels, K input channels); q[N][K]; s[N/128][K/128]. */
void oracle_quantize_weight(const void *w, int dtype, int64_t N, int64_t K,
                            uint8_t *q, float *s_blk)
{
    int64_t NB = N / GROUP, KB = K / GROUP;
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t nb = 0; nb < NB; ++nb) {
        for (int64_t kb = 0; kb < KB; ++kb) {
            float amax = 0.0f, s, inv;
            for (int64_t i = 0; i < GROUP; ++i)
                for (int64_t j = 0; j < GROUP; ++j) {
                    float v = fabsf(load_x(w, dtype, (nb * GROUP + i) * K + kb * GROUP + j));
                    if (v > amax)
                        amax = v;
                }
            oracle_group_scale(amax, &s, &inv);
            s_blk[nb * KB + kb] = s;
            for (int64_t i = 0; i < GROUP; ++i)
                for (int64_t j = 0; j < GROUP; ++j) {
                    int64_t e = (nb * GROUP + i) * K + kb * GROUP + j;
                    q[e] = cast_one(load_x(w, dtype, e), inv);
                }
        }
    }
}

/* ------------------------------------------------------------------ */
/* Block-scaled GEMM                                                   */
/* ------------------------------------------------------------------ */

/* Scale of the B operand for K-block kb and output column n.
   sb_gran 128: sB[N/128][K/128] (128x128 weight blocks)
   sb_gran 1:   sB[K/128][N]     (128x1 groups along K, used by Wgrad) */
static float scale_b(const float *sB, int sb_gran, int64_t N, int64_t KB,
                     int64_t kb, int64_t n)
{
    if (sb_gran == 1)
        return sB[kb * N + n];
    return sB[(n / GROUP) * KB + kb];
}

/* One output element C[m][n] of
 *   C = sum_kb  sA[kb][m] * sB(kb, n) * P_kb[m][n],
 *   P_kb[m][n] = sum_{k in block kb} decode(Aq[m][k]) * decode(Bq[n][k]).
 * Aq is [rowsA][K] with row stride K, sA is [K/128][lds_a] K-block-major,
 * Bq is [N][K].  Writes
 *   exact:   the fp64 sum (each P_kb is exact in fp64: 128 products of two
 *            4-bit significands stay far inside 53 bits),
 *   absref:  sum_k |a_dq * b_dq| (the tolerance's reference magnitude),
 *   pages:   the fl32 promotion order, kb ascending.  */
static void gemm_one(const uint8_t *Aq, const float *sA, int64_t lds_a,
                     const uint8_t *Bq, const float *sB, int64_t N, int64_t K,
                     int sb_gran, int64_t m, int64_t n,
                     double *exact, double *absref, float *pages)
{
    int64_t KB = K / GROUP;
    double ex = 0.0, ab = 0.0;
    float acc = 0.0f;
    for (int64_t kb = 0; kb < KB; ++kb) {
        double p = 0.0, pabs = 0.0;
        float sa = sA[kb * lds_a + m];
        float sb = scale_b(sB, sb_gran, N, KB, kb, n);
        for (int64_t j = 0; j < GROUP; ++j) {
            int64_t k = kb * GROUP + j;
            double prod = g_decode[Aq[m * K + k]] * g_decode[Bq[n * K + k]];
            p += prod;
            pabs += fabs(prod);
        }
        ex += ((double)sa * (double)sb) * p;
        ab += fabs((double)sa * (double)sb) * pabs;
        {
            volatile float pf = (float)p;            /* fl32(P_kb)        */
            volatile float s = sa * sb;              /* fl32(sA * sB)     */
            volatile float t = pf * s;               /* fl32(P * s)       */
            acc = acc + t;                           /* fl32(acc + ...)   */
        }
    }
    *exact = ex;
    *absref = ab;
    *pages = acc;
}

/* Dense GEMM at listed points (m_idx[i], n_idx[i]).  M is the number of
   rows of Aq and the row stride of sA.  Any output pointer may be NULL. */
void oracle_gemm_points(const uint8_t *Aq, const float *sA, const uint8_t *Bq,
                        const float *sB, int64_t M, int64_t N, int64_t K,
                        int sb_gran, const int64_t *m_idx, const int64_t *n_idx,
                        int64_t npts, double *c_exact, double *c_absref,
                        float *c_pages)
{
#pragma omp parallel for schedule(dynamic, 64)
    for (int64_t i = 0; i < npts; ++i) {
        double ex, ab;
        float pg;
        gemm_one(Aq, sA, M, Bq, sB, N, K, sb_gran, m_idx[i], n_idx[i], &ex, &ab, &pg);
        if (c_exact)
            c_exact[i] = ex;
        if (c_absref)
            c_absref[i] = ab;
        if (c_pages)
            c_pages[i] = pg;
    }
}

/* Full dense GEMM, C[M][N] row-major. */
void oracle_gemm(const uint8_t *Aq, const float *sA, const uint8_t *Bq,
                 const float *sB, int64_t M, int64_t N, int64_t K, int sb_gran,
                 double *c_exact, double *c_absref, float *c_pages)
{
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) {
            double ex, ab;
            float pg;
            gemm_one(Aq, sA, M, Bq, sB, N, K, sb_gran, m, n, &ex, &ab, &pg);
            if (c_exact)
                c_exact[m * N + n] = ex;
            if (c_absref)
                c_absref[m * N + n] = ab;
            if (c_pages)
                c_pages[m * N + n] = pg;
        }
}

/* MoE grouped GEMM at listed points.  Rows [off[e], off[e+1]) of Aq, sA and
   C belong to expert e, whose weight is Bq[e] ([N][K]) with scales
   sB[e] ([N/128][K/128]).  Each expert's result is the dense GEMM of its
   row slice; sA is [K/128][total_rows]. */
void oracle_grouped_gemm_points(const uint8_t *Aq, const float *sA,
                                const uint8_t *Bq, const float *sB,
                                const int64_t *row_offsets, int64_t E,
                                int64_t total_rows, int64_t N, int64_t K,
                                const int64_t *m_idx, const int64_t *n_idx,
                                int64_t npts, double *c_exact,
                                double *c_absref, float *c_pages)
{
    int64_t per_b = N * K, per_sb = (N / GROUP) * (K / GROUP);
#pragma omp parallel for schedule(dynamic, 64)
    for (int64_t i = 0; i < npts; ++i) {
        int64_t m = m_idx[i], e = 0;
        double ex = 0.0, ab = 0.0;
        float pg = 0.0f;
        while (e < E && !(row_offsets[e] <= m && m < row_offsets[e + 1]))
            ++e;
        if (e < E)
            gemm_one(Aq, sA, total_rows, Bq + e * per_b, sB + e * per_sb, N, K,
                     128, m, n_idx[i], &ex, &ab, &pg);
        if (c_exact)
            c_exact[i] = ex;
        if (c_absref)
            c_absref[i] = ab;
        if (c_pages)
            c_pages[i] = pg;
    }
}

/* ------------------------------------------------------------------ */
/* MX variant: 1x32 groups with power-of-two (E8M0) scales             */
/* ------------------------------------------------------------------ */
/*
 * Source: "Deepseek Ai News Expert Interview" (page 2), the DualPipe /
 * microscaling paragraph: the fine-grained strategy follows the microscaling
 * (MX) formats of Rouhani et al. (2023), and Blackwell tensor cores support
 * those formats with smaller groups.  The pages give no MX algorithm, so this
 * is the conversion the MX formats themselves define, in its plainest form:
 *  - a group is 32 consecutive elements along K of one row;
 *  - its shared exponent is floor(log2(amax)) minus 8, the exponent of the
 *    largest normal E4M3 binade (448 = 1.75 * 2^8), clamped to E8M0's
 *    [-127, 127]; a group whose amax is 0 takes -127;
 *  - the scale is X = 2^shared_exp, stored as the E8M0 byte shared_exp + 127;
 *  - each element is E4M3(fl32(x / X)) with the RNE satfinite cast above.
 *    x / X reaches up to 511.x, so the group's largest elements can
 *    saturate to 448.
 * Dequantization: x ~ decode(q) * 2^(byte - 127).  Dividing by a power of two
 * is exact in fl32 except below FP32's subnormal range, where the E4M3 cast
 * gives zero anyway.
 */
#define MX_GROUP 32
#define E4M3_EMAX 8

int oracle_mx_shared_exp(float amax)
{
    int e, se;
    if (!(amax > 0.0f))
        return -127;
    (void)frexpf(amax, &e);            /* amax = f * 2^e, f in [0.5, 1) */
    se = (e - 1) - E4M3_EMAX;          /* floor(log2(amax)) - 8 */
    if (se < -127)
        se = -127;
    if (se > 127)
        se = 127;
    return se;
}

/* x[M][K] row-major -> q[M][K] codes, e8[M][K/32] E8M0 scale bytes
   (plain row-major here; the GPU's tiled layout is a permutation of it). */
void oracle_mx_quantize_rows(const void *x, int dtype, int64_t M, int64_t K,
                             uint8_t *q, uint8_t *e8)
{
    int64_t G = K / MX_GROUP;
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t g = 0; g < G; ++g) {
            float amax = 0.0f;
            for (int64_t j = 0; j < MX_GROUP; ++j) {
                float v = fabsf(load_x(x, dtype, m * K + g * MX_GROUP + j));
                if (v > amax)
                    amax = v;
            }
            int se = oracle_mx_shared_exp(amax);
            float X = ldexpf(1.0f, se);
            e8[m * G + g] = (uint8_t)(se + 127);
            for (int64_t j = 0; j < MX_GROUP; ++j) {
                int64_t i = m * K + g * MX_GROUP + j;
                volatile float v = load_x(x, dtype, i) / X;   /* fl32(x / X) */
                q[i] = oracle_e4m3_encode(v);
            }
        }
    }
}

/* One output of the MX GEMM,
 *   C[m][n] = sum_g 2^(ea[m][g] - 127) * 2^(eb[n][g] - 127) * P_g,
 *   P_g = sum_{k in group g} decode(Aq[m][k]) * decode(Bq[n][k]).
 * Each P_g is exact in fp64 (32 products of 4-bit significands); the groups
 * are summed in fp64.  absref = sum_k |a_dq * b_dq|. */
static void mx_gemm_one(const uint8_t *Aq, const uint8_t *ea, const uint8_t *Bq,
                        const uint8_t *eb, int64_t K, int64_t m, int64_t n,
                        double *exact, double *absref)
{
    int64_t G = K / MX_GROUP;
    double ex = 0.0, ab = 0.0;
    for (int64_t g = 0; g < G; ++g) {
        double p = 0.0, pabs = 0.0;
        for (int64_t j = 0; j < MX_GROUP; ++j) {
            int64_t k = g * MX_GROUP + j;
            double prod = g_decode[Aq[m * K + k]] * g_decode[Bq[n * K + k]];
            p += prod;
            pabs += fabs(prod);
        }
        double scale = ldexp(1.0, (int)ea[m * G + g] - 127 + (int)eb[n * G + g] - 127);
        ex += scale * p;
        ab += scale * pabs;
    }
    *exact = ex;
    *absref = ab;
}

/* MX GEMM at listed points (m_idx[i], n_idx[i]).  Aq[M][K], ea[M][K/32],
   Bq[N][K], eb[N][K/32]. */
void oracle_mx_gemm_points(const uint8_t *Aq, const uint8_t *ea, const uint8_t *Bq,
                           const uint8_t *eb, int64_t K, const int64_t *m_idx,
                           const int64_t *n_idx, int64_t npts, double *c_exact,
                           double *c_absref)
{
#pragma omp parallel for schedule(dynamic, 64)
    for (int64_t i = 0; i < npts; ++i) {
        double ex, ab;
        mx_gemm_one(Aq, ea, Bq, eb, K, m_idx[i], n_idx[i], &ex, &ab);
        if (c_exact)
            c_exact[i] = ex;
        if (c_absref)
            c_absref[i] = ab;
    }
}

/* Number of OpenMP threads the oracle runs on (1 without OpenMP). */
int oracle_num_threads(void)
{
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Set the number of OpenMP threads later oracle calls run on (host
 * scheduling only; the arithmetic and its order per output are unchanged). */
void oracle_set_num_threads(int n)
{
#ifdef _OPENMP
    extern void omp_set_num_threads(int);
    omp_set_num_threads(n > 0 ? n : 1);
#else
    (void)n;
#endif
}
