/*
 * fp8_oracle.c -- CPU oracle for fine-grained FP8 quantisation and the
 * block-scaled FP8 GEMM with per-128-K FP32 promotion.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file; only the tests, the package's smoke check and the bench's
 * CPU-baseline leg use it.  It shares no code, header, table or constant with
 * the CUDA library.  Every definition is written from the method as the
 * DeepSeek-V3 Technical Report states it (the source pages reproduce its text):
 *   - section 3.3.1 / 3.3.2: all GEMM operands (Fprop, Dgrad, Wgrad) use E4M3,
 *     an FP8 format with a 4-bit exponent and a 3-bit mantissa, and elements
 *     are quantised in small groups that each carry their own scale, so that
 *     the narrow dynamic range is shared per group;
 *   - section 3.3.2: the scales sit along the GEMM's inner (K) dimension, so
 *     dequantisation happens per K group;
 *   - section 3.3.2, Figure 7(b): the tensor-core partial sum of each K
 *     interval N_C is moved to FP32 registers, multiplied by the scales and
 *     added there in full FP32 precision.
 * The group sizes (1x128 for activations, 128x128 for weights), the scale
 * amax/448 and N_C = 128 are the method's constants; the pages lost them in
 * extraction, and the report's design is taken as stated.
 *
 * Floating point: IEEE binary32 / binary64 with round-to-nearest-even, no
 * contraction (built with -ffp-contract=off), no fast-math.  The GEMM result
 * is formed in binary64: each 128-wide K block of decoded E4M3 products is an
 * exact sum (every decoded value is an integer multiple of 2^-9 and at most
 * 448, so a block sum is an integer multiple of 2^-18 below 2^43), then the
 * block is promoted with its two FP32 scales and added in binary64.
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *   - s = fl32(amax / 448) and q = E4M3_RNE_sat(fl32(x / s)) (divide by the
 *     stored FP32 scale; dequantisation is q * s);
 *   - a group whose amax is 0 gets s = 1 and all-zero codes;
 *   - quotients at or above 448 in magnitude saturate to +-448;
 *   - the sign of a zero code follows the sign of the input (0x80 for -0 and
 *     for negative values that round to zero).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------- E4M3 --- */

/* Round a non-negative binary64 value to the nearest integer, ties to even. */
static double round_half_even(double v)
{
    double f = floor(v);
    double d = v - f; /* exact: v is far below 2^52 wherever this is used */
    if (d > 0.5) return f + 1.0;
    if (d < 0.5) return f;
    return (fmod(f, 2.0) == 0.0) ? f : f + 1.0;
}

/*
 * E4M3 encoding of one binary32 value: exponent bias 7, 3 mantissa bits,
 * largest finite magnitude 1.75 * 2^8 = 448 (code 0x7E), code 0x7F/0xFF is
 * NaN, no infinities, subnormals m * 2^-9 for m = 1..7.  Rounding is to the
 * nearest representable value, ties to the even mantissa; magnitudes at or
 * above 448 saturate to 448.
 */
uint8_t fo_e4m3_encode(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    uint8_t sign = (uint8_t)((u >> 31) << 7);
    if (isnan(f)) return (uint8_t)(sign | 0x7F);
    double a = fabs((double)f);
    if (a >= 448.0) return (uint8_t)(sign | 0x7E);
    if (a < 0.015625) {
        /* below the smallest normal 2^-6: the grid is m * 2^-9, m = 0..8;
         * m = 8 is exactly 2^-6, whose code (exponent field 1, mantissa 0)
         * is the integer 8 as well. */
        double m = round_half_even(a * 512.0);
        return (uint8_t)(sign | (uint8_t)m);
    }
    int ex;
    double fr = frexp(a, &ex); /* a = fr * 2^ex, fr in [0.5, 1) */
    int e = ex - 1;            /* a = (2 fr) * 2^e, 2 fr in [1, 2) */
    double m = round_half_even((2.0 * fr - 1.0) * 8.0);
    if (m == 8.0) {            /* mantissa carried into the exponent */
        m = 0.0;
        e += 1;
    }
    int E = e + 7; /* 1..15; a < 448 keeps (E, m) at or below (15, 6) */
    return (uint8_t)(sign | (uint8_t)((E << 3) | (int)m));
}

/* Value of an E4M3 code, from the format definition. */
double fo_e4m3_decode(uint8_t c)
{
    int s = c >> 7, E = (c >> 3) & 0xF, m = c & 7;
    double v;
    if (E == 15 && m == 7) return NAN;
    if (E == 0)
        v = (double)m * ldexp(1.0, -9);
    else
        v = (1.0 + (double)m / 8.0) * ldexp(1.0, E - 7);
    return s ? -v : v;
}

void fo_e4m3_encode_array(const float* x, int64_t n, uint8_t* out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = fo_e4m3_encode(x[i]);
}

void fo_e4m3_decode_array(const uint8_t* c, int64_t n, double* out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = fo_e4m3_decode(c[i]);
}

/* ---------------------------------------------------------------- E5M6 --- */

/*
 * E5M6: a 12-bit floating-point element with a sign bit, a 5-bit exponent
 * and a 6-bit mantissa -- the customised format the report adopts for one
 * class of activations (section 3.3.1, next to E4M3 for the GEMM operands).
 * The pages give the field widths only; the rest is read as an IEEE-style
 * format, like the 5-bit-exponent FP16 and E5M2: bias 15, exponent field 31
 * reserved (mantissa 0 = infinity, else NaN), so the largest finite value is
 * (1 + 63/64) * 2^15 = 65024 (code 0x7BF), the smallest normal 2^-14 and the
 * subnormals m * 2^-20 for m = 1..63.  Encoding rounds to nearest, ties to
 * the even mantissa, and saturates: magnitudes at or above 65024 (and
 * infinities) give +-65024, as the E4M3 encoder saturates at 448.  Codes are
 * 12-bit values in a uint16 (sign in bit 11).
 */
uint16_t fo_e5m6_encode(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    uint16_t sign = (uint16_t)((u >> 31) << 11);
    if (isnan(f)) return (uint16_t)(sign | 0x7FF);
    double a = fabs((double)f);
    if (a >= 65024.0) return (uint16_t)(sign | 0x7BF);
    if (a < 0x1p-14) {
        /* the subnormal grid m * 2^-20, m = 0..64; m = 64 is 2^-14, whose
         * code (exponent field 1, mantissa 0) is the integer 64 as well */
        double m = round_half_even(a * 1048576.0);
        return (uint16_t)(sign | (uint16_t)m);
    }
    int ex;
    double fr = frexp(a, &ex); /* a = fr * 2^ex, fr in [0.5, 1) */
    int e = ex - 1;            /* a = (2 fr) * 2^e, e in [-14, 15] */
    double m = round_half_even((2.0 * fr - 1.0) * 64.0);
    if (m == 64.0) {           /* mantissa carried into the exponent */
        m = 0.0;
        e += 1;
    }
    /* a < 65024 keeps (e, m) at or below (15, 63): only a >= 65280 would
     * round up to 2^16 */
    return (uint16_t)(sign | (uint16_t)(((e + 15) << 6) | (int)m));
}

/* Value of an E5M6 code (low 12 bits), from the format definition. */
double fo_e5m6_decode(uint16_t c)
{
    int s = (c >> 11) & 1, E = (c >> 6) & 0x1F, m = c & 0x3F;
    double v;
    if (E == 31) v = (m == 0) ? INFINITY : NAN;
    else if (E == 0) v = (double)m * ldexp(1.0, -20);
    else v = (1.0 + (double)m / 64.0) * ldexp(1.0, E - 15);
    return s ? -v : v;
}

void fo_e5m6_encode_array(const float* x, int64_t n, uint16_t* out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = fo_e5m6_encode(x[i]);
}

void fo_e5m6_decode_array(const uint16_t* c, int64_t n, double* out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = fo_e5m6_decode(c[i]);
}

/* ---------------------------------------------------------------- BF16 --- */

/* A bfloat16 is the upper half of a binary32, so widening is exact. */
static float bf16_value(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Nearest bfloat16 (8 significant bits) to a binary32, ties to even: the 16
 * discarded bits are compared against the halfway pattern 0x8000. */
uint16_t fo_f32_to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if (isnan(f)) return (uint16_t)((u >> 16) | 0x0040);
    uint32_t hi = u >> 16, lo = u & 0xFFFFu;
    if (lo > 0x8000u || (lo == 0x8000u && (hi & 1u))) hi += 1u;
    return (uint16_t)hi;
}

void fo_round_f32(const double* c, int64_t n, float* out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = (float)c[i];
}

void fo_round_bf16(const double* c, int64_t n, uint16_t* out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = fo_f32_to_bf16((float)c[i]);
}

/* ------------------------------------------------------------ quantise --- */

/* Scale of one group: s = fl32(amax / 448); an all-zero group gets s = 1. */
float fo_group_scale(float amax)
{
    if (amax == 0.0f) return 1.0f;
    return amax / 448.0f;
}

/*
 * 1x128 activation quantisation.  x: bfloat16 [M][K] with row stride ldx.
 * Each row is split along K into groups of 128; each group gets its own
 * scale.  xq: codes [M][K] with row stride ldq.  sx: scales [K/128][M]
 * (group index major, row index contiguous).
 */
void fo_quant_act_1x128(const uint16_t* x, int64_t M, int64_t K, int64_t ldx,
                        uint8_t* xq, int64_t ldq, float* sx)
{
    int64_t KB = K / 128;
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t kb = 0; kb < KB; ++kb) {
            const uint16_t* g = x + m * ldx + kb * 128;
            float amax = 0.0f;
            for (int j = 0; j < 128; ++j) {
                float v = fabsf(bf16_value(g[j]));
                if (v > amax) amax = v;
            }
            float s = fo_group_scale(amax);
            sx[kb * M + m] = s;
            for (int j = 0; j < 128; ++j)
                xq[m * ldq + kb * 128 + j] = fo_e4m3_encode(bf16_value(g[j]) / s);
        }
    }
}

/* Scale of one E5M6 group: s = fl32(amax / 65024), the format's largest
 * finite value taking the place of E4M3's 448; an all-zero group gets s = 1. */
float fo_group_scale_e5m6(float amax)
{
    if (amax == 0.0f) { return 1.0f; }
    return amax / 65024.0f;
}

/*
 * 1x128 activation quantisation to E5M6 (the same fine-grained grouping as
 * fo_quant_act_1x128, section 3.3.2, with the E5M6 element format).
 * x: bfloat16 [M][K], row stride ldx.  q: 12-bit codes [M][K] (one uint16
 * each), row stride ldq.  sx: scales [K/128][M].
 */
void fo_quant_act_1x128_e5m6(const uint16_t* x, int64_t M, int64_t K, int64_t ldx,
                             uint16_t* q, int64_t ldq, float* sx)
{
    int64_t KB = K / 128;
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t kb = 0; kb < KB; ++kb) {
            const uint16_t* grp = x + m * ldx + kb * 128;
            float amax = 0.0f;
            for (int j = 0; j < 128; ++j) {
                float mag = fabsf(bf16_value(grp[j]));
                if (mag > amax) amax = mag;
            }
            float s = fo_group_scale_e5m6(amax);
            sx[m + kb * M] = s;
            for (int j = 0; j < 128; ++j)
                q[m * ldq + kb * 128 + j] = fo_e5m6_encode(bf16_value(grp[j]) / s);
        }
    }
}

/* ------------------------------------------------ power-of-two scales --- */

/*
 * Power-of-two group scales, the variant that Blackwell's block-scaled MMA
 * (MXFP8: one UE8M0 exponent per 32 elements along K) can apply inside the
 * tensor core.  The report's scale is amax / 448; here the scale is the
 * smallest power of two s = 2^e with amax / s <= 448, so that x / s is exact
 * and every code is the E4M3 rounding of an exactly scaled value.  e is kept
 * in the UE8M0 range [-127, 127] (a group whose amax would need a smaller
 * exponent keeps e = -127; its codes are then smaller than 448); an all-zero
 * group gets e = 0.  Written from the definition: the exponent is found by
 * stepping e upward until 448 * 2^e reaches amax.
 */
int fo_pow2_exponent(float amax)
{
    if (amax == 0.0f) return 0;
    int e = -127;
    while (e < 127 && (double)amax > 448.0 * ldexp(1.0, e)) ++e;
    return e;
}

/*
 * 1x128 activation quantisation with power-of-two scales.  x: bfloat16
 * [M][K], row stride ldx.  xq: codes [M][K], row stride ldq.  se8: UE8M0
 * exponent bytes e + 127, [K/128][M].
 */
void fo_quant_act_1x128_pow2(const uint16_t* x, int64_t M, int64_t K, int64_t ldx,
                             uint8_t* xq, int64_t ldq, uint8_t* se8)
{
    int64_t KB = K / 128;
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t kb = 0; kb < KB; ++kb) {
            const uint16_t* src = x + m * ldx + kb * 128;
            float amax = 0.0f;
            for (int j = 0; j < 128; ++j) {
                float av = fabsf(bf16_value(src[j]));
                if (av > amax) amax = av;
            }
            int e = fo_pow2_exponent(amax);
            se8[kb * M + m] = (uint8_t)(e + 127);
            for (int j = 0; j < 128; ++j) /* x / 2^e: exact in binary64 */
                xq[m * ldq + kb * 128 + j] = fo_e4m3_encode((float)ldexp((double)bf16_value(src[j]), -e));
        }
    }
}

/*
 * 128x128 weight quantisation with power-of-two scales.  w: bfloat16 [K][N]
 * (K = inner dimension), row stride ldw.  wq: codes [N][K].  se8: UE8M0 bytes
 * [K/128][N], one per row n of wq and K block (the 128 rows of a block share
 * their block's exponent), the per-row layout a block-scaled MMA reads.
 */
void fo_quant_weight_128x128_pow2(const uint16_t* w, int64_t K, int64_t N, int64_t ldw,
                                  uint8_t* wq, uint8_t* se8)
{
    int64_t KB = K / 128, NB = N / 128;
    for (int64_t nb = 0; nb < NB; ++nb) {
        for (int64_t kb = 0; kb < KB; ++kb) {
            float amax = 0.0f;
            for (int i = 0; i < 128; ++i)
                for (int j = 0; j < 128; ++j) {
                    float av = fabsf(bf16_value(w[(kb * 128 + i) * ldw + nb * 128 + j]));
                    if (av > amax) amax = av;
                }
            int e = fo_pow2_exponent(amax);
            for (int j = 0; j < 128; ++j) se8[kb * N + nb * 128 + j] = (uint8_t)(e + 127);
            for (int i = 0; i < 128; ++i)
                for (int j = 0; j < 128; ++j) {
                    int64_t k = kb * 128 + i, n = nb * 128 + j;
                    wq[n * K + k] = fo_e4m3_encode((float)ldexp((double)bf16_value(w[k * ldw + n]), -e));
                }
        }
    }
}

/*
 * 128x1 activation quantisation for the weight-gradient GEMM, whose inner
 * dimension is the token dimension M.  x: bfloat16 [M][K], row stride ldx,
 * M a multiple of 128.  Each column k is split along M into groups of 128
 * tokens.  xqT: codes [K][M] (transposed).  sxT: scales [M/128][K].
 */
void fo_quant_act_128x1(const uint16_t* x, int64_t M, int64_t K, int64_t ldx,
                        uint8_t* xqT, float* sxT)
{
    int64_t MB = M / 128;
    for (int64_t mb = 0; mb < MB; ++mb) {
        for (int64_t k = 0; k < K; ++k) {
            float amax = 0.0f;
            for (int i = 0; i < 128; ++i) {
                float v = fabsf(bf16_value(x[(mb * 128 + i) * ldx + k]));
                if (v > amax) amax = v;
            }
            float s = fo_group_scale(amax);
            sxT[mb * K + k] = s;
            for (int i = 0; i < 128; ++i)
                xqT[k * M + mb * 128 + i] =
                    fo_e4m3_encode(bf16_value(x[(mb * 128 + i) * ldx + k]) / s);
        }
    }
}

/*
 * 128x128 weight quantisation.  w: bfloat16 [K][N] (K = GEMM inner
 * dimension), row stride ldw.  One scale per 128x128 block.
 * wq:  codes [N][K] (each output feature's K values contiguous), may be NULL.
 * wqT: codes [K][N] (the input's own orientation), may be NULL.
 * sw:  scales [N/128][K/128].
 */
void fo_quant_weight_128x128(const uint16_t* w, int64_t K, int64_t N, int64_t ldw,
                             uint8_t* wq, uint8_t* wqT, float* sw)
{
    int64_t KB = K / 128, NB = N / 128;
    for (int64_t nb = 0; nb < NB; ++nb) {
        for (int64_t kb = 0; kb < KB; ++kb) {
            float amax = 0.0f;
            for (int i = 0; i < 128; ++i)
                for (int j = 0; j < 128; ++j) {
                    float v = fabsf(bf16_value(w[(kb * 128 + i) * ldw + nb * 128 + j]));
                    if (v > amax) amax = v;
                }
            float s = fo_group_scale(amax);
            sw[nb * KB + kb] = s;
            for (int i = 0; i < 128; ++i)
                for (int j = 0; j < 128; ++j) {
                    int64_t k = kb * 128 + i, n = nb * 128 + j;
                    uint8_t q = fo_e4m3_encode(bf16_value(w[k * ldw + n]) / s);
                    if (wq) wq[n * K + k] = q;
                    if (wqT) wqT[k * N + n] = q;
                }
        }
    }
}

/* --------------------------------------------------------------- GEMM ---- */

/* B-scale layouts (mirrors the meaning, not the code, of the library's). */
enum { FO_BSCALE_BLOCK128 = 0,   /* sb[N/128][K/128]: one scale per 128x128 block */
       FO_BSCALE_ROW1x128 = 1,   /* sb[K/128][N] with row stride ldsb: per (n, K block) */
       FO_BSCALE_BLOCK128_T = 2  /* sb[K/128][N/128]: the block grid stored transposed */ };

typedef struct {
    const uint8_t* aq; int64_t lda;      /* A codes [M][K] */
    const float* sa; int64_t ldsa;       /* sa[kb * ldsa + m] */
    const uint8_t* bq; int64_t ldb;      /* B codes [N][K] */
    const float* sb; int64_t ldsb; int bmode;
    int64_t M, N, K;
    const int64_t* rows; int64_t nrows;  /* rows of C to form */
    double* out;                          /* [nrows][N] */
    const double* dec;                    /* 256-entry decode table */
    int tid, nthreads;
} gemm_job;

static double b_scale(const gemm_job* j, int64_t n, int64_t kb)
{
    int64_t KB = j->K / 128, NB = j->N / 128;
    switch (j->bmode) {
    case FO_BSCALE_BLOCK128: return (double)j->sb[(n / 128) * KB + kb];
    case FO_BSCALE_ROW1x128: return (double)j->sb[kb * j->ldsb + n];
    default: return (double)j->sb[kb * NB + n / 128];
    }
}

/*
 * C[m][n] = sum over K blocks kb of  sa[m,kb] * sb[n,kb] * P_kb[m][n],
 * P_kb[m][n] = sum_{k in block kb} dec(aq[m][k]) * dec(bq[n][k]),
 * with P_kb exact and everything in binary64.
 */
static void* gemm_worker(void* arg)
{
    const gemm_job* j = (const gemm_job*)arg;
    int64_t KB = j->K / 128;
    for (int64_t i = j->tid; i < j->nrows; i += j->nthreads) {
        int64_t m = j->rows[i];
        const uint8_t* a = j->aq + m * j->lda;
        for (int64_t n = 0; n < j->N; ++n) {
            const uint8_t* b = j->bq + n * j->ldb;
            double acc = 0.0;
            for (int64_t kb = 0; kb < KB; ++kb) {
                double p = 0.0;
                for (int64_t k = kb * 128; k < kb * 128 + 128; ++k)
                    p += j->dec[a[k]] * j->dec[b[k]];
                acc += (double)j->sa[kb * j->ldsa + m] * b_scale(j, n, kb) * p;
            }
            j->out[i * j->N + n] = acc;
        }
    }
    return NULL;
}

void fo_gemm_blockscaled_rows(const uint8_t* aq, int64_t lda, const float* sa, int64_t ldsa,
                              const uint8_t* bq, int64_t ldb, const float* sb, int64_t ldsb,
                              int bmode, int64_t M, int64_t N, int64_t K,
                              const int64_t* rows, int64_t nrows, double* out, int nthreads)
{
    double dec[256];
    for (int c = 0; c < 256; ++c) dec[c] = fo_e4m3_decode((uint8_t)c);
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    gemm_job jobs[256];
    pthread_t th[256];
    for (int t = 0; t < nthreads; ++t) {
        gemm_job j = {aq, lda, sa, ldsa, bq, ldb, sb, ldsb, bmode, M, N, K,
                      rows, nrows, out, dec, t, nthreads};
        jobs[t] = j;
    }
    for (int t = 1; t < nthreads; ++t) pthread_create(&th[t], NULL, gemm_worker, &jobs[t]);
    gemm_worker(&jobs[0]);
    for (int t = 1; t < nthreads; ++t) pthread_join(th[t], NULL);
}
