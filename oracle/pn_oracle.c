/*
 * pn_oracle.c -- plain, slow CPU oracle for the PN weight formats pn3t / pn4t.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product path links, loads or calls
 * this file: only the tests, the smoke check and the CPU-baseline leg of the
 * benchmark use it. It shares no code, header, table or constant with the CUDA
 * library; every constant below is written out again from the format's
 * description.
 *
 * Source: tensorless docs, "Why a P100-native weight format" (the PN format
 * explanation page), sections "Every block is 34 bytes", "One lane, one word",
 * "Codes never straddle the two halves of a word", "Exact decode in fp32" and
 * "Zero is a code, and the scale has a sign".
 *
 * Readings taken where the page leaves a step open (each is listed in the
 * design notes of the repository):
 *   R1  block = fp16 scale d in bytes 0..1 (little-endian), then the eight
 *       32-bit code words w[0..7] in bytes 2..33 (little-endian).
 *   R2  weight k of a block (0 <= k < weights_per_block) is code c = k % cpw of
 *       word j = k / cpw; code c sits in half (c & 1) of the word (0 = bits
 *       0..15, 1 = bits 16..31) at bit offset bits * (c >> 1) inside that half.
 *       pn3t leaves bits 15 and 31 unused: written as 0, ignored on decode.
 *   R3  zero point z = 4 for pn3t (n - z in [-4, 3]) and z = 8 for pn4t
 *       (n - z in [-8, 7]).
 *   R4  quantiser: round-to-nearest with a signed block scale chosen so that
 *       the largest-magnitude weight (first index on ties) lands on step -z:
 *       d = fp16_rne(a / -z) (fp32 divide), codes n = clamp(rint(v / d), -z,
 *       z - 1) + z with an fp32 divide and round-half-to-even.  A block whose
 *       scale is 0 or underflows to a signed zero in fp16 is stored as the zero
 *       block (d = +0, every code = z).  A scale that overflows fp16 is
 *       saturated to +-65504.  Inputs must be finite.
 *   R5  GEMV y[m][r] = sum_k w[r][k] * x[m][k]: products and the sum in fp64,
 *       sequential in k, rounded to fp32 once.
 *   R12 GPTQ-style quantiser (tensorless docs, "How Qwen3.8-27B-PN3 uses it",
 *       says only "GPTQ-style"): the published GPTQ procedure (Frantar et al.,
 *       "GPTQ: Accurate Post-Training Quantization for Generative
 *       Pre-trained Transformers", ICLR 2023, Algorithm 1) with PN blocks as
 *       its groups.  H = 2 X^T X + lambda I over calibration inputs X [n][K],
 *       lambda = damp * mean(diag(2 X^T X)); U = the upper Cholesky factor of
 *       H^-1 (H^-1 = U^T U).  Columns k = 0 .. K-1 in order; when k starts a
 *       block, each row's scale comes from the block's current weights
 *       (rounded to fp32) by rule R4; column k is quantised by R4 with that
 *       scale, and the error (w - decoded) / U[k][k] is subtracted, times
 *       U[k][j], from every later column j.  All of it in fp64.
 *
 * Build: cc -O2 -std=c11 -fno-fast-math -ffp-contract=off -shared -fPIC.
 * -ffp-contract=off keeps every multiply and add a separately rounded IEEE
 * operation.  (The oracle tests also compile edited copies of this file,
 * each with one planted mistake, to show that the pins catch such mistakes.)
 */
#include <math.h>
#include <stdlib.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

#define ORACLE_PN3T 124
#define ORACLE_PN4T 125
#define ORACLE_BLOCK_BYTES 34

enum { ORACLE_OK = 0, ORACLE_EINVAL = 1 };

typedef struct {
    int per_block;  /* weights per block           */
    int per_word;   /* codes per 32-bit word (cpw) */
    int bits;       /* bits per code               */
    int zero;       /* zero point z                */
} oracle_fmt;

static int oracle_format(int type, oracle_fmt* f)
{
    if (type == ORACLE_PN3T) {        /* 80 weights, 10 three-bit codes/word */
        f->per_block = 80; f->per_word = 10; f->bits = 3; f->zero = 4;
        return 1;
    }
    if (type == ORACLE_PN4T) {        /* 64 weights, 8 four-bit codes/word */
        f->per_block = 64; f->per_word = 8; f->bits = 4; f->zero = 8;
        return 1;
    }
    return 0;
}

/* ---------------------------------------------------------------- fp16 ---- */

static uint32_t f32_bits(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }

/* IEEE binary16 -> fp32, exact (every binary16 value is a binary32 value). */
float oracle_half_to_float(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 0x1F;
    int mant = h & 0x3FF;
    double v;
    if (expo == 0)
        v = ldexp((double)mant, -24);                 /* zero / subnormal */
    else if (expo == 31)
        v = mant ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + mant), expo - 25);  /* normal */
    return (float)(sign ? -v : v);
}

/* fp32 -> IEEE binary16, round to nearest, ties to even. */
uint16_t oracle_float_to_half(float f)
{
    uint32_t x = f32_bits(f);
    uint16_t sign = (uint16_t)((x >> 16) & 0x8000u);
    uint32_t ax = x & 0x7FFFFFFFu;
    if (ax > 0x7F800000u) return (uint16_t)(sign | 0x7E00u);  /* NaN */
    if (ax >= 0x477FF000u) return (uint16_t)(sign | 0x7C00u); /* >= 65520: Inf */
    if (ax >= 0x38800000u) {                                  /* normal half */
        uint32_t expo = (ax >> 23) - 127 + 15;
        uint32_t mant = ax & 0x7FFFFFu;
        uint32_t r = (expo << 10) | (mant >> 13);
        uint32_t rem = mant & 0x1FFFu;
        if (rem > 0x1000u || (rem == 0x1000u && (r & 1u))) r++;
        return (uint16_t)(sign | r);
    }
    if (ax <= 0x33000000u) return sign;                       /* <= 2^-25 -> 0 */
    {                                                         /* subnormal half */
        uint32_t expo = ax >> 23;                             /* 102 .. 112 */
        uint32_t mant = (ax & 0x7FFFFFu) | 0x800000u;
        uint32_t shift = 126 - expo;                          /* 14 .. 24 */
        uint32_t m = mant >> shift;
        uint32_t rem = mant & ((1u << shift) - 1u);
        uint32_t halfway = 1u << (shift - 1);
        if (rem > halfway || (rem == halfway && (m & 1u))) m++;
        return (uint16_t)(sign | m);
    }
}

/* --------------------------------------------------------------- sizes ---- */

size_t oracle_row_bytes(int type, int64_t K)
{
    oracle_fmt f;
    if (!oracle_format(type, &f) || K <= 0 || K % f.per_block) return 0;
    return (size_t)(K / f.per_block) * ORACLE_BLOCK_BYTES;
}

/* ------------------------------------------------------- block helpers ---- */

static uint32_t load_u32_le(const uint8_t* p)
{
    return (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16) | ((uint32_t)p[3] << 24);
}

static void store_u32_le(uint8_t* p, uint32_t v)
{
    p[0] = (uint8_t)v; p[1] = (uint8_t)(v >> 8); p[2] = (uint8_t)(v >> 16); p[3] = (uint8_t)(v >> 24);
}

/* Bit position of weight k's code inside its word (reading R2). */
static int code_shift(const oracle_fmt* f, int k)
{
    int c = k % f->per_word;
    return 16 * (c & 1) + f->bits * (c >> 1);
}

static int code_word(const oracle_fmt* f, int k) { return k / f->per_word; }

/* Decode one 34-byte block into per_block fp32 weights: w = d * (n - z). */
static void decode_block(const oracle_fmt* f, const uint8_t* blk, float* out)
{
    uint16_t dbits = (uint16_t)(blk[0] | (blk[1] << 8));
    float d = oracle_half_to_float(dbits);
    uint32_t mask = (1u << f->bits) - 1u;
    for (int k = 0; k < f->per_block; ++k) {
        uint32_t word = load_u32_le(blk + 2 + 4 * code_word(f, k));
        int n = (int)((word >> code_shift(f, k)) & mask);
        out[k] = d * (float)(n - f->zero);    /* one IEEE fp32 multiply, exact */
    }
}

/* Quantise one block of per_block fp32 weights (reading R4). */
static void encode_block(const oracle_fmt* f, const float* v, uint8_t* blk)
{
    int z = f->zero;
    int jmax = 0;
    float amax = fabsf(v[0]);
    for (int j = 1; j < f->per_block; ++j) {
        if (fabsf(v[j]) > amax) { amax = fabsf(v[j]); jmax = j; }
    }
    float a = v[jmax];
    uint16_t dbits = 0;
    uint32_t words[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    int codes[80];

    int zero_block = (a == 0.0f);
    if (!zero_block) {
        float d32 = a / (float)(-z);          /* largest weight lands on step -z */
        dbits = oracle_float_to_half(d32);
        if ((dbits & 0x7FFFu) == 0) {
            zero_block = 1;                   /* underflow: the zero block */
        } else if ((dbits & 0x7FFFu) == 0x7C00u) {
            dbits = (uint16_t)((dbits & 0x8000u) | 0x7BFFu);   /* saturate to +-65504 */
        }
    }
    if (zero_block) {
        dbits = 0;
        for (int k = 0; k < f->per_block; ++k) codes[k] = z;
    } else {
        float d = oracle_half_to_float(dbits);
        for (int k = 0; k < f->per_block; ++k) {
            float q = rintf(v[k] / d);        /* fp32 divide, round half to even */
            if (q < (float)(-z)) q = (float)(-z);
            if (q > (float)(z - 1)) q = (float)(z - 1);
            codes[k] = (int)q + z;
        }
    }
    for (int k = 0; k < f->per_block; ++k)
        words[code_word(f, k)] |= (uint32_t)codes[k] << code_shift(f, k);

    blk[0] = (uint8_t)(dbits & 0xFF);
    blk[1] = (uint8_t)(dbits >> 8);
    for (int j = 0; j < 8; ++j) store_u32_le(blk + 2 + 4 * j, words[j]);
}

/* ------------------------------------------------------------ exported ---- */

/* Pack fp32 weights w[N][K] (row-major) into PN rows out[N][row_bytes]. */
int oracle_pack(int type, const float* w, int64_t N, int64_t K, uint8_t* out)
{
    oracle_fmt f;
    if (!oracle_format(type, &f) || N < 0 || K <= 0 || K % f.per_block || !w || !out)
        return ORACLE_EINVAL;
    int64_t nb = K / f.per_block;
    for (int64_t r = 0; r < N; ++r)
        for (int64_t b = 0; b < nb; ++b)
            encode_block(&f, w + r * K + b * f.per_block,
                         out + (r * nb + b) * ORACLE_BLOCK_BYTES);
    return ORACLE_OK;
}

/* Decode PN rows W[N][row_bytes] into fp32 weights w[N][K]. */
int oracle_unpack(int type, const uint8_t* W, int64_t N, int64_t K, float* w)
{
    oracle_fmt f;
    if (!oracle_format(type, &f) || N < 0 || K <= 0 || K % f.per_block || !W || !w)
        return ORACLE_EINVAL;
    int64_t nb = K / f.per_block;
    for (int64_t r = 0; r < N; ++r)
        for (int64_t b = 0; b < nb; ++b)
            decode_block(&f, W + (r * nb + b) * ORACLE_BLOCK_BYTES,
                         w + r * K + b * f.per_block);
    return ORACLE_OK;
}

/*
 * y[m][r] = sum_k w[r][k] * x[m][k] for 0 <= m < M, 0 <= r < N (reading R5).
 * x holds fp16 bit patterns [M][K]; y is fp32 [M][N].  If abs_sum is not NULL
 * it receives sum_k |w[r][k] * x[m][k]| in fp64 [M][N] (the scale of the
 * rounding-error bound).
 */
int oracle_gemv(int type, const uint8_t* W, int64_t N, int64_t K,
                const uint16_t* x, int M, float* y, double* abs_sum)
{
    oracle_fmt f;
    if (!oracle_format(type, &f) || N < 0 || K <= 0 || K % f.per_block || M < 1 || !W || !x || !y)
        return ORACLE_EINVAL;
    int64_t nb = K / f.per_block;
    float wblk[80];
    for (int m = 0; m < M; ++m) {
        const uint16_t* xm = x + (int64_t)m * K;
        for (int64_t r = 0; r < N; ++r) {
            double acc = 0.0, acc_abs = 0.0;
            for (int64_t b = 0; b < nb; ++b) {
                decode_block(&f, W + (r * nb + b) * ORACLE_BLOCK_BYTES, wblk);
                for (int k = 0; k < f.per_block; ++k) {
                    double xv = (double)oracle_half_to_float(xm[b * f.per_block + k]);
                    double p = (double)wblk[k] * xv;
                    acc += p;
                    acc_abs += fabs(p);
                }
            }
            y[(int64_t)m * N + r] = (float)acc;
            if (abs_sum) abs_sum[(int64_t)m * N + r] = acc_abs;
        }
    }
    return ORACLE_OK;
}

/* ---------------------------------------------------- Hadamard rotation --- */

/*
 * Runtime rotation of the activations that reach the PN weights (tensorless
 * docs, "Why a P100-native weight format", section "How Qwen3.8-27B-PN3 uses
 * it": the model applies a Hadamard rotation to those activations and the
 * engine performs it at run time).  The page gives neither the size nor the
 * normalisation of the rotation.  Reading R10: every run of B consecutive
 * activations of a row (B = 2^m, 2 <= B <= 4096, B dividing K) is multiplied
 * by the orthonormal Sylvester Hadamard matrix H_B / sqrt(B), where
 * H_1 = [1] and H_2n = [[H_n, H_n], [H_n, -H_n]].
 *
 * The arithmetic is fixed so that results are reproducible bit for bit: each
 * fp16 input is widened to fp32; the fast Walsh-Hadamard butterflies run in
 * stages h = 1, 2, 4, ..., B/2, in that order, each stage replacing the pair
 * (v[i], v[i+h]) for every i with (i & h) == 0 by (v[i] + v[i+h],
 * v[i] - v[i+h]) in fp32; each result is multiplied once, in fp32, by
 * s = 2^(-m/2) (m even) or s = 2^(-(m+1)/2) * fp32(sqrt(2)) (m odd, the
 * constant rounded to nearest), and rounded to fp16 (nearest, ties to even).
 *
 * x, out: fp16 bit patterns [M][K] (out may equal x).  out32, if not NULL,
 * receives the fp32 values before the final rounding.
 */
int oracle_hadamard(const uint16_t* x, int M, int64_t K, int B, uint16_t* out, float* out32)
{
    if (!x || !out || M < 1 || K <= 0 || B < 2 || B > 4096 || (B & (B - 1)) || K % B) return ORACLE_EINVAL;
    int m = 0;
    while ((1 << m) < B) ++m;
    const float sqrt2 = 1.41421356237309504880f;          /* fp32 nearest to sqrt(2) */
    float s = ldexpf(1.0f, -(m / 2));
    if (m % 2) s = ldexpf(sqrt2, -(m + 1) / 2);
    float v[4096];
    for (int row = 0; row < M; ++row) {
        for (int64_t base = 0; base < K; base += B) {
            const int64_t off = (int64_t)row * K + base;
            for (int i = 0; i < B; ++i) v[i] = oracle_half_to_float(x[off + i]);
            for (int h = 1; h < B; h *= 2) {
                for (int i = 0; i < B; ++i) {
                    if (i & h) continue;
                    const float a = v[i], b = v[i + h];
                    v[i] = a + b;
                    v[i + h] = a - b;
                }
            }
            for (int i = 0; i < B; ++i) {
                const float r = v[i] * s;
                if (out32) out32[off + i] = r;
                out[off + i] = oracle_float_to_half(r);
            }
        }
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------ prefill, large M --- */

/*
 * Prefill reconstruction (tensorless docs, "What the fork adds": the engine
 * dequantizes the weights for prefill and runs a chunked GEMM; v100-skinny
 * README, "How QPN works": above the skinny band the weights are rebuilt
 * transiently from the packed codes and never kept).  The pages give no
 * precision for the rebuilt weights.  Reading R11: each weight is the exact
 * fp32 product d * (n - z) of the decode, rounded once to fp16 (nearest, ties
 * to even; a product beyond the fp16 range becomes +-inf).
 *
 * W: PN rows [N][row_bytes]; w16: fp16 bit patterns [N][K].
 */
int oracle_unpack_f16(int type, const uint8_t* W, int64_t N, int64_t K, uint16_t* w16)
{
    oracle_fmt f;
    if (!oracle_format(type, &f) || N < 0 || K <= 0 || K % f.per_block || (N > 0 && (!W || !w16)))
        return ORACLE_EINVAL;
    int64_t nb = K / f.per_block;
    float wblk[80];
    for (int64_t r = 0; r < N; ++r)
        for (int64_t b = 0; b < nb; ++b) {
            decode_block(&f, W + (r * nb + b) * ORACLE_BLOCK_BYTES, wblk);
            for (int k = 0; k < f.per_block; ++k)
                w16[r * K + b * f.per_block + k] = oracle_float_to_half(wblk[k]);
        }
    return ORACLE_OK;
}

/*
 * The GEMM of the rebuilt weights: y[m][n] = sum_k w16[n][k] * x[m][k] for
 * m < M, n < N, every product and sum in fp64 and rounded to fp32 once at the
 * end; abs_sum (if not NULL) receives sum_k |w16[n][k] * x[m][k]| in fp64.
 * w16 [N][K] and x [M][K] are fp16 bit patterns; y and abs_sum are [M][N].
 */
int oracle_gemm_f16(const uint16_t* w16, int64_t N, int64_t K, const uint16_t* x, int M,
                    float* y, double* abs_sum)
{
    if (N < 0 || K <= 0 || M < 1 || (N > 0 && (!w16 || !x || !y))) return ORACLE_EINVAL;
    for (int m = 0; m < M; ++m) {
        const uint16_t* xrow = x + (int64_t)m * K;
        for (int64_t n = 0; n < N; ++n) {
            const uint16_t* wrow = w16 + n * K;
            double sum = 0.0, sum_abs = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double p = (double)oracle_half_to_float(wrow[k]) * (double)oracle_half_to_float(xrow[k]);
                sum += p;
                sum_abs += fabs(p);
            }
            y[(int64_t)m * N + n] = (float)sum;
            if (abs_sum) abs_sum[(int64_t)m * N + n] = sum_abs;
        }
    }
    return ORACLE_OK;
}

/* ---------------------------------------------------------------- GPTQ ---- */

/* Cholesky factor of the symmetric positive definite n x n matrix a (fp64,
 * row-major): a = c c^T with c lower triangular, written over c.  Returns 0 if
 * a pivot is not positive. */
static int cholesky_lower(const double* a, double* c, int64_t n)
{
    for (int64_t i = 0; i < n * n; ++i) c[i] = 0.0;
    for (int64_t j = 0; j < n; ++j) {
        double s = a[j * n + j];
        for (int64_t k = 0; k < j; ++k) s -= c[j * n + k] * c[j * n + k];
        if (!(s > 0.0)) return 0;
        double cjj = sqrt(s);
        c[j * n + j] = cjj;
        for (int64_t i = j + 1; i < n; ++i) {
            double t = a[i * n + j];
            for (int64_t k = 0; k < j; ++k) t -= c[i * n + k] * c[j * n + k];
            c[i * n + j] = t / cjj;
        }
    }
    return 1;
}

/* Inverse of the symmetric positive definite matrix a from its Cholesky
 * factor c (a = c c^T): a^-1 = c^-T c^-1, column by column by forward and back
 * substitution. */
static void spd_inverse(const double* c, double* inv, double* tmp, int64_t n)
{
    for (int64_t col = 0; col < n; ++col) {
        for (int64_t i = 0; i < n; ++i) {            /* c y = e_col */
            double s = (i == col) ? 1.0 : 0.0;
            for (int64_t k = 0; k < i; ++k) s -= c[i * n + k] * tmp[k];
            tmp[i] = s / c[i * n + i];
        }
        for (int64_t i = n - 1; i >= 0; --i) {       /* c^T x = y */
            double s = tmp[i];
            for (int64_t k = i + 1; k < n; ++k) s -= c[k * n + i] * inv[k * n + col];
            inv[i * n + col] = s / c[i * n + i];
        }
    }
}

/* Scale bits of one block from its current weights (rule R4), and whether it
 * is the zero block. */
static uint16_t block_scale(const oracle_fmt* f, const float* v, int* zero_block)
{
    int jmax = 0;
    float amax = fabsf(v[0]);
    for (int j = 1; j < f->per_block; ++j)
        if (fabsf(v[j]) > amax) { amax = fabsf(v[j]); jmax = j; }
    float a = v[jmax];
    *zero_block = (a == 0.0f);
    if (*zero_block) return 0;
    uint16_t dbits = oracle_float_to_half(a / (float)(-f->zero));
    if ((dbits & 0x7FFFu) == 0) { *zero_block = 1; return 0; }
    if ((dbits & 0x7FFFu) == 0x7C00u) dbits = (uint16_t)((dbits & 0x8000u) | 0x7BFFu);
    return dbits;
}

/* GPTQ-style quantisation (reading R12) of fp32 weights w[N][K] with
 * calibration inputs X[n][K] (fp32) and dampening `damp` (> 0) into PN rows
 * out[N][row_bytes]. */
int oracle_gptq(int type, const float* w, int64_t N, int64_t K, const float* X, int64_t n, double damp,
                uint8_t* out)
{
    oracle_fmt f;
    if (!oracle_format(type, &f) || N < 0 || K <= 0 || K % f.per_block || !w || !out || !X || n < 1 ||
        !(damp > 0.0))
        return ORACLE_EINVAL;
    const int64_t nb = K / f.per_block, z = f.zero;
    double* H = (double*)malloc(sizeof(double) * K * K);
    double* C = (double*)malloc(sizeof(double) * K * K);
    double* Hi = (double*)malloc(sizeof(double) * K * K);
    double* tmp = (double*)malloc(sizeof(double) * K);
    double* W = (double*)malloc(sizeof(double) * N * K);
    float* cur = (float*)malloc(sizeof(float) * f.per_block);
    uint16_t* dbits = (uint16_t*)malloc(sizeof(uint16_t) * (N > 0 ? N : 1));
    int* zero_blk = (int*)malloc(sizeof(int) * (N > 0 ? N : 1));
    int* codes = (int*)malloc(sizeof(int) * (N * K > 0 ? N * K : 1));
    int rc = ORACLE_OK;
    if (!H || !C || !Hi || !tmp || !W || !cur || !dbits || !zero_blk || !codes) { rc = ORACLE_EINVAL; goto done; }
    /* H = 2 X^T X, then dampened */
    for (int64_t i = 0; i < K; ++i)
        for (int64_t j = 0; j < K; ++j) {
            double s = 0.0;
            for (int64_t t = 0; t < n; ++t) s += (double)X[t * K + i] * (double)X[t * K + j];
            H[i * K + j] = 2.0 * s;
        }
    double mean_diag = 0.0;
    for (int64_t i = 0; i < K; ++i) mean_diag += H[i * K + i];
    mean_diag /= (double)K;
    for (int64_t i = 0; i < K; ++i) H[i * K + i] += damp * mean_diag;
    /* U: upper Cholesky factor of H^-1 (H^-1 = U^T U, U = the transpose of
     * the lower factor of H^-1) */
    if (!cholesky_lower(H, C, K)) { rc = ORACLE_EINVAL; goto done; }
    spd_inverse(C, Hi, tmp, K);
    if (!cholesky_lower(Hi, C, K)) { rc = ORACLE_EINVAL; goto done; }   /* C lower; U[k][j] = C[j][k] */
    for (int64_t i = 0; i < N * K; ++i) W[i] = (double)w[i];
    for (int64_t k = 0; k < K; ++k) {
        const int64_t b = k / f.per_block, kk = k % f.per_block;
        if (kk == 0)
            for (int64_t r = 0; r < N; ++r) {
                for (int j = 0; j < f.per_block; ++j) cur[j] = (float)W[r * K + b * f.per_block + j];
                dbits[r] = block_scale(&f, cur, &zero_blk[r]);
            }
        const double ukk = C[k * K + k];
        for (int64_t r = 0; r < N; ++r) {
            int code = (int)z;
            float wq = 0.0f;
            if (!zero_blk[r]) {
                float d = oracle_half_to_float(dbits[r]);
                float q = rintf((float)W[r * K + k] / d);
                if (q < (float)(-z)) q = (float)(-z);
                if (q > (float)(z - 1)) q = (float)(z - 1);
                code = (int)q + (int)z;
                wq = d * q;
            }
            codes[r * K + k] = code;
            const double err = (W[r * K + k] - (double)wq) / ukk;
            for (int64_t j = k + 1; j < K; ++j) W[r * K + j] -= err * C[j * K + k];
        }
        if (kk == f.per_block - 1)                     /* the block is complete: write it */
            for (int64_t r = 0; r < N; ++r) {
                uint8_t* blk = out + (r * nb + b) * ORACLE_BLOCK_BYTES;
                uint32_t words[8] = {0, 0, 0, 0, 0, 0, 0, 0};
                for (int j = 0; j < f.per_block; ++j)
                    words[code_word(&f, j)] |= (uint32_t)codes[r * K + b * f.per_block + j] << code_shift(&f, j);
                blk[0] = (uint8_t)(dbits[r] & 0xFF);
                blk[1] = (uint8_t)(dbits[r] >> 8);
                for (int j = 0; j < 8; ++j) store_u32_le(blk + 2 + 4 * j, words[j]);
            }
    }
done:
    free(H); free(C); free(Hi); free(tmp); free(W); free(cur); free(dbits); free(zero_blk); free(codes);
    return rc;
}
