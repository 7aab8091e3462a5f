/*
 * NF4 oracle: a plain, slow CPU statement of what the NF4 weight-only linear layer computes.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or load this file or the
 * library built from it: only the tests, the smoke check of __graft_entry__ and the cpu_baseline /
 * reference leg of bench.py use it.  It shares no code, table or constant generator with the CUDA
 * library, and it never reads anything the CUDA library produced except the outputs it is asked
 * to judge.
 *
 * Sources followed (page titles and the part of each page):
 *   - deep-fold README (wertick01/deep-fold, README.ru.md), format paragraph: a group of 64 weights
 *     holds 4-bit NF4 codes and one FP16 scale; the codes and scales are the whole payload, about
 *     3.76x smaller than BF16 for aligned matrices.
 *   - deep-fold README, method paragraph: NF4 is the data type introduced with QLoRA.  The 16 table
 *     values are the ones published with QLoRA (Dettmers et al., 2023, appendix).
 *   - deep-fold README, execution-path table: the linear kernels dequantize only the current tile
 *     and never write a dense weight matrix back; decode is an N=1 GEMV, prefill a GEMM of up to 32
 *     positions.
 *   - deep-fold README, overview paragraph: embeddings (PackedEmbed) reconstruct only the rows that
 *     are requested.
 *   The rest is the library's own pinned reading of what the pages leave open: absmax scale per
 *   group (fp32 max, stored as fp16 round-to-nearest-even), code = argmin_i |fp32(w/s) - T[i]| in
 *   fp32 with ties to the lower index, two codes per byte with the low nibble first, dequantized
 *   value bf16(fp32(T[c] * float(scale))), fp32-or-better accumulation and a bf16 output.
 *
 * Every function is written for a reader who checks it against those definitions by eye: plain
 * loops, IEEE single precision where the definition says fp32, double precision for the linear.
 * Build with -ffp-contract=off (no fused multiply-add may change a rounding) and without
 * -ffast-math.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define NF4_GROUP 64

/* The NormalFloat-4 table published with QLoRA (Dettmers et al., 2023), index 0..15.  Each literal
   is an exact binary32 number; the published literals, not a re-derivation, are the definition. */
static const float NF4_TABLE[16] = {
    -1.0f,
    -0.6961928009986877f,
    -0.5250730514526367f,
    -0.39491748809814453f,
    -0.28444138169288635f,
    -0.18477343022823334f,
    -0.09105003625154495f,
    0.0f,
    0.07958029955625534f,
    0.16093020141124725f,
    0.24611230194568634f,
    0.33791524171829224f,
    0.44070982933044434f,
    0.5626170039176941f,
    0.7229568362236023f,
    1.0f,
};

void oracle_nf4_table(float out[16]) {
    for (int i = 0; i < 16; i++) out[i] = NF4_TABLE[i];
}

/* ------------------------------------------------------------------------------------------------
 * Rounding of binary32 to binary16 and to bfloat16, round to nearest, ties to even.
 * ---------------------------------------------------------------------------------------------- */

/* binary32 -> binary16 bits.  A finite f is S * 2^(E-23) with a 24-bit significand S.  At the
   magnitude of f the binary16 quantum is 2^(max(E,-14) - 10); the bits of S below that quantum are
   dropped with round-to-nearest-even, and the result is re-encoded (a carry out of the 11-bit
   significand moves to the next binade; beyond 65504 the result is infinity). */
uint16_t oracle_f32_to_f16(float f) {
    uint32_t x;
    memcpy(&x, &f, 4);
    uint16_t sign = (uint16_t)((x >> 16) & 0x8000u);
    uint32_t e = (x >> 23) & 0xFFu;
    uint32_t frac = x & 0x7FFFFFu;
    if (e == 0xFFu) return (uint16_t)(sign | (frac ? 0x7E00u : 0x7C00u)); /* NaN (quiet) or inf */
    if (e == 0u) return sign; /* zero or binary32 subnormal: below 2^-126, rounds to a signed zero */
    int32_t E = (int32_t)e - 127;
    uint32_t S = 0x800000u | frac;
    int32_t qexp = (E > -14 ? E : -14) - 10; /* exponent of the binary16 quantum */
    int32_t shift = qexp - (E - 23);         /* number of low bits of S to drop (>= 13) */
    if (shift > 25) return sign;             /* |f| < a quarter quantum: rounds to zero */
    uint32_t r = S >> shift;
    uint32_t rem = S & ((1u << shift) - 1u);
    uint32_t half = 1u << (shift - 1);
    if (rem > half || (rem == half && (r & 1u))) r += 1u;
    if (E < -14) return (uint16_t)(sign | r); /* subnormal; r == 1024 encodes the smallest normal */
    if (r == 0x800u) {                          /* significand overflowed: next binade */
        r = 0x400u;
        E += 1;
    }
    if (E > 15) return (uint16_t)(sign | 0x7C00u);
    return (uint16_t)(sign | ((uint32_t)(E + 15) << 10) | (r - 0x400u));
}

/* binary16 bits -> binary32 (exact). */
float oracle_f16_to_f32(uint16_t h) {
    uint32_t e = (h >> 10) & 0x1Fu, m = h & 0x3FFu;
    float mag;
    if (e == 0u)
        mag = ldexpf((float)m, -24); /* subnormal: m * 2^-24 */
    else if (e == 31u)
        mag = m ? NAN : INFINITY;
    else
        mag = ldexpf((float)(0x400u | m), (int)e - 25); /* (1024 + m) * 2^(e - 15 - 10) */
    return (h & 0x8000u) ? -mag : mag;
}

/* binary32 -> bfloat16 bits.  bfloat16 keeps the binary32 sign and exponent and the top 7 fraction
   bits.  For finite values the 31 magnitude bits, read as an integer, grow with the magnitude and
   the 16 dropped bits are one uniform quantum inside each binade, so rounding that integer to a
   multiple of 2^16 with ties to even rounds the value to nearest-even; a carry into the exponent
   field is the correct next binade (and gives infinity past the largest finite value). */
uint16_t oracle_f32_to_bf16(float f) {
    uint32_t x;
    memcpy(&x, &f, 4);
    if ((x & 0x7F800000u) == 0x7F800000u) /* inf stays inf; NaN stays a (quiet) NaN */
        return (uint16_t)((x >> 16) | ((x & 0x7FFFFFu) ? 0x40u : 0u));
    uint32_t upper = x >> 16, lower = x & 0xFFFFu;
    if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u))) upper += 1u;
    return (uint16_t)upper;
}

/* bfloat16 bits -> binary32 (exact). */
float oracle_bf16_to_f32(uint16_t b) {
    uint32_t x = (uint32_t)b << 16;
    float f;
    memcpy(&f, &x, 4);
    return f;
}

void oracle_f32_to_f16_array(const float* in, int64_t n, uint16_t* out) {
    for (int64_t i = 0; i < n; i++) out[i] = oracle_f32_to_f16(in[i]);
}

void oracle_f32_to_bf16_array(const float* in, int64_t n, uint16_t* out) {
    for (int64_t i = 0; i < n; i++) out[i] = oracle_f32_to_bf16(in[i]);
}

/* ------------------------------------------------------------------------------------------------
 * Quantize and dequantize.
 * ---------------------------------------------------------------------------------------------- */

/* Nearest NF4 code of a normalised weight r: the first index i (scanning 0..15) at which the fp32
   distance |r - T[i]| is smallest.  The strict comparison sends ties to the lower index. */
int oracle_nf4_code(float r) {
    int best = 0;
    float best_d = fabsf(r - NF4_TABLE[0]);
    for (int i = 1; i < 16; i++) {
        float d = fabsf(r - NF4_TABLE[i]);
        if (d < best_d) {
            best_d = d;
            best = i;
        }
    }
    return best;
}

void oracle_nf4_code_array(const float* r, int64_t n, uint8_t* out) {
    for (int64_t i = 0; i < n; i++) out[i] = (uint8_t)oracle_nf4_code(r[i]);
}

/* One group of 64 weights: s = max |w| in fp32; the stored scale is fp16(s); each weight is divided
   by the fp32 s (not by the stored fp16 scale) and mapped to its nearest code.  An all-zero group
   (s = 0) gets code 7, the code whose table value is 0.  Codes 2j and 2j+1 share byte j, the even
   one in the low nibble. */
static void quantize_group(const float* w, uint8_t* codes, uint16_t* scale) {
    float s = 0.0f;
    for (int k = 0; k < NF4_GROUP; k++) {
        float a = fabsf(w[k]);
        if (a > s) s = a;
    }
    *scale = oracle_f32_to_f16(s);
    for (int j = 0; j < NF4_GROUP / 2; j++) {
        int lo = 7, hi = 7;
        if (s != 0.0f) {
            float r_lo = w[2 * j] / s;
            float r_hi = w[2 * j + 1] / s;
            lo = oracle_nf4_code(r_lo);
            hi = oracle_nf4_code(r_hi);
        }
        codes[j] = (uint8_t)(lo | (hi << 4));
    }
}

/* w: fp32 [N, K] row-major.  codes: u8 [N, K/2].  scales: fp16 bits [N, K/64].  The group runs along
   K inside one row.  Returns 0, or -1 when K is not a positive multiple of 64 or N < 0. */
int oracle_quantize(const float* w, int64_t N, int64_t K, uint8_t* codes, uint16_t* scales) {
    if (N < 0 || K <= 0 || K % NF4_GROUP != 0) return -1;
    int64_t G = K / NF4_GROUP;
    for (int64_t n = 0; n < N; n++)
        for (int64_t g = 0; g < G; g++)
            quantize_group(w + n * K + g * NF4_GROUP, codes + n * (K / 2) + g * (NF4_GROUP / 2),
                           scales + n * G + g);
    return 0;
}

/* Code of weight (n, k) in the packed layout. */
static int code_at(const uint8_t* codes, int64_t K, int64_t n, int64_t k) {
    uint8_t byte = codes[n * (K / 2) + k / 2];
    return (k % 2 == 0) ? (byte & 0x0F) : (byte >> 4);
}

/* Dequantized weight: bf16 round-to-nearest-even of the fp32 product T[c] * float(scale). */
static uint16_t dequant_value(int c, uint16_t scale) {
    float p = NF4_TABLE[c] * oracle_f16_to_f32(scale);
    return oracle_f32_to_bf16(p);
}

/* w_hat: bf16 bits [N, K]. */
int oracle_dequant(const uint8_t* codes, const uint16_t* scales, int64_t N, int64_t K, uint16_t* w_hat) {
    if (N < 0 || K <= 0 || K % NF4_GROUP != 0) return -1;
    int64_t G = K / NF4_GROUP;
    for (int64_t n = 0; n < N; n++)
        for (int64_t k = 0; k < K; k++)
            w_hat[n * K + k] = dequant_value(code_at(codes, K, n, k), scales[n * G + k / NF4_GROUP]);
    return 0;
}

/* Packed embedding rows (deep-fold README, overview paragraph: embeddings reconstruct only the
 * requested rows): out[i][k] = the dequantized weight (ids[i], k) of a V x K table; an id outside
 * [0, V) gives a row of zeros (the library's reading; the pages do not say).  Returns the number of
 * such ids. */
int64_t oracle_embed(const int32_t* ids, int64_t n_ids, const uint8_t* codes, const uint16_t* scales, int64_t V,
                     int64_t K, uint16_t* out) {
    if (n_ids < 0 || V < 0 || K <= 0 || K % NF4_GROUP != 0) return -1;
    int64_t G = K / NF4_GROUP, bad = 0;
    for (int64_t i = 0; i < n_ids; i++) {
        int64_t id = ids[i];
        for (int64_t k = 0; k < K; k++) {
            if (id < 0 || id >= V)
                out[i * K + k] = 0;
            else
                out[i * K + k] = dequant_value(code_at(codes, K, id, k), scales[id * G + k / NF4_GROUP]);
        }
        if (id < 0 || id >= V) bad++;
    }
    return bad;
}

/* ------------------------------------------------------------------------------------------------
 * Linear: y64[m, n] = sum_k x[m, k] * w_hat[n, k] in double precision, and the magnitude sum
 * sum_k |x[m, k] * w_hat[n, k]| that the acceptance bound is scaled by.  A bf16 x bf16 product
 * needs 16 significand bits, so every product is exact in double; only the running sums round.
 * ---------------------------------------------------------------------------------------------- */

typedef struct {
    const uint16_t* x;
    const uint8_t* codes;
    const uint16_t* scales;
    int64_t M, N, K;
    int64_t n0, n1;
    double* y64;
    double* abs_sum;
    int status;
} linear_job;

static void* linear_rows(void* arg) {
    linear_job* j = (linear_job*)arg;
    int64_t K = j->K, G = K / NF4_GROUP;
    double* wrow = (double*)malloc((size_t)K * sizeof(double));
    double* xrow = (double*)malloc((size_t)K * sizeof(double));
    if (!wrow || !xrow) {
        free(wrow);
        free(xrow);
        j->status = -2;
        return NULL;
    }
    for (int64_t n = j->n0; n < j->n1; n++) {
        for (int64_t k = 0; k < K; k++)
            wrow[k] = (double)oracle_bf16_to_f32(
                dequant_value(code_at(j->codes, K, n, k), j->scales[n * G + k / NF4_GROUP]));
        for (int64_t m = 0; m < j->M; m++) {
            for (int64_t k = 0; k < K; k++) xrow[k] = (double)oracle_bf16_to_f32(j->x[m * K + k]);
            double acc = 0.0, mag = 0.0;
            for (int64_t k = 0; k < K; k++) {
                double p = xrow[k] * wrow[k];
                acc += p;
                mag += fabs(p);
            }
            j->y64[m * j->N + n] = acc;
            j->abs_sum[m * j->N + n] = mag;
        }
    }
    free(wrow);
    free(xrow);
    j->status = 0;
    return NULL;
}

/* x: bf16 bits [M, K]; codes/scales as above; y64, abs_sum: double [M, N].  Rows n are split into
   contiguous ranges over `nthreads` threads; each output is computed by exactly one thread, in the
   same order, so the result does not depend on the thread count. */
int oracle_linear(const uint16_t* x, const uint8_t* codes, const uint16_t* scales, int64_t M, int64_t N,
                  int64_t K, double* y64, double* abs_sum, int nthreads) {
    if (M < 0 || N < 0 || K <= 0 || K % NF4_GROUP != 0) return -1;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if ((int64_t)nthreads > N) nthreads = (int)(N > 0 ? N : 1);
    linear_job jobs[256];
    pthread_t tids[256];
    int started[256];
    for (int t = 0; t < nthreads; t++) {
        jobs[t] = (linear_job){x, codes, scales, M, N, K, N * t / nthreads, N * (t + 1) / nthreads,
                               y64, abs_sum, -3};
        started[t] = (t > 0) && pthread_create(&tids[t], NULL, linear_rows, &jobs[t]) == 0;
    }
    linear_rows(&jobs[0]);
    for (int t = 1; t < nthreads; t++) {
        if (started[t])
            pthread_join(tids[t], NULL);
        else
            linear_rows(&jobs[t]); /* thread creation failed: do the range here */
    }
    for (int t = 0; t < nthreads; t++)
        if (jobs[t].status != 0) return jobs[t].status;
    return 0;
}

/* The same two sums for a list of (m, n) entries only, for matrices too large to evaluate whole. */
int oracle_linear_entries(const uint16_t* x, const uint8_t* codes, const uint16_t* scales, int64_t M,
                          int64_t N, int64_t K, const int64_t* m_idx, const int64_t* n_idx, int64_t count,
                          double* y64, double* abs_sum) {
    if (M < 0 || N < 0 || K <= 0 || K % NF4_GROUP != 0) return -1;
    int64_t G = K / NF4_GROUP;
    for (int64_t i = 0; i < count; i++) {
        int64_t m = m_idx[i], n = n_idx[i];
        if (m < 0 || m >= M || n < 0 || n >= N) return -1;
        double acc = 0.0, mag = 0.0;
        for (int64_t k = 0; k < K; k++) {
            double xv = (double)oracle_bf16_to_f32(x[m * K + k]);
            double wv = (double)oracle_bf16_to_f32(
                dequant_value(code_at(codes, K, n, k), scales[n * G + k / NF4_GROUP]));
            double p = xv * wv;
            acc += p;
            mag += fabs(p);
        }
        y64[i] = acc;
        abs_sum[i] = mag;
    }
    return 0;
}
