/*
 * CPU oracle for small-M block-quantized GEMV (Q4_0 / Q6_K weights against
 * Q8_1 activations) and the greedy top-1 reduction.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library's product path may call,
 * link or load this file; only the tests, the smoke check and the bench's CPU
 * baseline leg do.  It shares no code, header, table or helper with the CUDA
 * library: the block formats are decoded here from their definitions, written
 * out again independently.
 *
 * What it computes, and where the pages use it (the pages name the three
 * block formats but do not define them; the definitions below are the
 * llama.cpp-family ones the pages' kernels consume):
 *   - Q8_1 activation blocks: "Qwen3.6 27B B70 follow-up: Q8 activation
 *     cache", section "Q8_1 activation cache prototype" (the activation is
 *     quantized once to Q8_1 and reused by sibling Q4_0 matmuls).  Per block of
 *     32: d = max|x| / 127, q = round(x / d), s = d * sum(q); stored as fp16 d,
 *     fp16 s, int8 q[32] (36 bytes).
 *   - Q4_0 weights: blocks of 32, fp16 scale d, 4-bit q, value d * (q - 8);
 *     "Qwen3.6 27B Q4_0 DFlash/SYCL closure", section "What materially worked"
 *     item 2 (direct Q4_0 MMVQ for rows 1-17).
 *   - Q6_K weights: superblocks of 256, fp16 d, 16 int8 subscales (one per 16
 *     values), 6-bit q, value d * sc * (q - 32); "Q6_K M=6 fused DFlash top-1
 *     production record", sections "Why this was slow" and "Exactness and
 *     safety contracts" ([5120, 248320] Q6_K output weight) and "Memory and
 *     startup" (16 subscales and one fp16 scale per 256 values).
 *   - Q8_0, Q4_K and Q5_K weights (named among the further K-quant formats
 *     of "Qwen3.6 27B Q4_0 DFlash/SYCL closure" and of the DFlash KV-cache
 *     page): Q8_0 = blocks of 32, fp16 d, int8 q, value d * q; Q4_K =
 *     superblocks of 256, fp16 d and dmin, eight 6-bit scales and eight
 *     6-bit mins (one per 32 values), 4-bit q, value d * sc * q - dmin * m;
 *     Q5_K = the same with 5-bit q.
 *   - Top-1 with the lowest-token-ID finite-tie rule: same page, "Exactness and
 *     safety contracts", item 3.
 *   - RMSNorm fused with the Q8_1 quantizer ("Qwen3.6 27B Q4_0 DFlash/SYCL
 *     closure", Closed or negative paths): the plain definition in fp64,
 *     then the quantizer on the fp32 rounding of the normalized row.
 *
 * The dot products are the plain definition of the result: every Q8_1 block
 * dot is an exact integer sum, scaled by the two fp16 scales in fp64 and
 * summed in fp64.  The fp16 <-> binary conversions are written from the IEEE
 * 754 binary16 definition (round to nearest, ties to even).
 *
 * Readings where the pages are silent (the pages name the formats but do not
 * define their bytes):
 *   - Q8_1 block = {fp16 d, fp16 s, int8 q[32]}; q uses the fp32 d before its
 *     fp16 rounding; round() is half away from zero; an all-zero block has
 *     d = s = 0 and q = 0.
 *   - Q4_0 block = {fp16 d, uint8 qs[16]}; value i < 16 is the low nibble of
 *     qs[i], value i + 16 is the high nibble of qs[i].
 *   - Q6_K superblock = {uint8 ql[128], uint8 qh[64], int8 sc[16], fp16 d}
 *     with plain sequential packing: the low 4 bits of value i are nibble
 *     (i & 1) of ql[i >> 1], its high 2 bits are bits 2*(i & 3) of qh[i >> 2];
 *     subscale index i >> 4.
 *   - Q4_K superblock = {fp16 d, fp16 dmin, uint8 scales[12], uint8 qs[128]}
 *     as in llama.cpp: sub-block j < 4 has scale scales[j] & 63 and min
 *     scales[j + 4] & 63; j >= 4 has scale (scales[j + 4] & 15) | (scales[j - 4]
 *     >> 6) << 4 and min (scales[j + 4] >> 4) | (scales[j] >> 6) << 4.  Values
 *     64 c .. 64 c + 31 are the low nibbles of qs[32 c .. 32 c + 31] and values
 *     64 c + 32 .. 64 c + 63 their high nibbles; value i is in sub-block i / 32.
 *   - Q5_K superblock = {fp16 d, fp16 dmin, uint8 scales[12], uint8 qh[32],
 *     uint8 qs[128]} as in llama.cpp: scales, mins and the low 4 bits as Q4_K;
 *     the fifth bit of value i is bit (i / 32) of qh[i % 32].
 *
 * Build: cc -O2 -std=c11 -ffp-contract=off -fPIC -shared -pthread (no fast-math).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ */
/* binary16 from its IEEE 754 definition                                */
/* ------------------------------------------------------------------ */

/* float -> binary16 bits, round to nearest, ties to even. */
uint16_t oracle_f32_to_f16(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    uint16_t sign = (uint16_t)((u >> 31) << 15);
    if (isnan(f)) return (uint16_t)(sign | 0x7E00u);
    if (isinf(f)) return (uint16_t)(sign | 0x7C00u);
    double a = fabs((double)f);
    if (a < ldexp(1.0, -14)) {
        /* subnormal range: a whole number of 2^-24 units; 1024 units is the
         * smallest normal number, whose encoding is the same integer. */
        double units = rint(ldexp(a, 24));
        return (uint16_t)(sign | (uint16_t)units);
    }
    int e;
    frexp(a, &e);               /* a in [2^(e-1), 2^e) */
    int E = e - 1;              /* unbiased exponent    */
    double sig = rint(ldexp(a, 10 - E));   /* 11-bit significand in [1024, 2048] */
    if (sig == 2048.0) { sig = 1024.0; E += 1; }
    if (E > 15) return (uint16_t)(sign | 0x7C00u);
    return (uint16_t)(sign | (uint16_t)((E + 15) << 10) | (uint16_t)(sig - 1024.0));
}

/* binary16 bits -> double (exact). */
double oracle_f16_to_f64(uint16_t h)
{
    int s = (h >> 15) & 1;
    int E = (h >> 10) & 0x1F;
    int mant = h & 0x3FF;
    double v;
    if (E == 0)
        v = ldexp((double)mant, -24);
    else if (E == 31)
        v = mant ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + mant), E - 25);
    return s ? -v : v;
}

static uint16_t rd16(const uint8_t* p) { return (uint16_t)(p[0] | (p[1] << 8)); }
static void wr16(uint8_t* p, uint16_t v) { p[0] = (uint8_t)(v & 0xFF); p[1] = (uint8_t)(v >> 8); }

/* ------------------------------------------------------------------ */
/* Q8_1 activation quantization                                          */
/* ------------------------------------------------------------------ */

#define Q8_0_BYTES 34
#define Q4_K_BYTES 144
#define Q5_K_BYTES 176
#define Q8_1_BYTES 36
#define Q4_0_BYTES 18
#define Q6_K_BYTES 210

/* x: fp32 [M][ldx]; out: M * (K/32) blocks of 36 bytes, row-major [m][b]. */
void oracle_quantize_q8_1(const float* x, int64_t ldx, int M, int K, uint8_t* out)
{
    int nb = K / 32;
    for (int m = 0; m < M; ++m) {
        for (int b = 0; b < nb; ++b) {
            const float* xb = x + (int64_t)m * ldx + 32 * b;
            float amax = 0.0f;
            for (int i = 0; i < 32; ++i) {
                float a = fabsf(xb[i]);
                if (a > amax) amax = a;
            }
            float d = amax / 127.0f;
            int8_t q[32];
            int S = 0;
            for (int i = 0; i < 32; ++i) {
                int v = 0;
                if (amax != 0.0f) {
                    v = (int)roundf(xb[i] / d);
                    if (v > 127) v = 127;
                    if (v < -127) v = -127;
                }
                q[i] = (int8_t)v;
                S += v;
            }
            uint8_t* o = out + ((int64_t)m * nb + b) * Q8_1_BYTES;
            wr16(o, oracle_f32_to_f16(d));
            wr16(o + 2, oracle_f32_to_f16(d * (float)S));
            memcpy(o + 4, q, 32);
        }
    }
}

/* RMSNorm fused with the Q8_1 quantizer ("Qwen3.6 27B Q4_0 DFlash/SYCL
 * closure", Closed or negative paths: the down-to-next-RMSNorm/Q8
 * boundary; the pages name the fusion, not its arithmetic).  The plain
 * definition, per row, in fp64: S = sum_k x_k^2 (in increasing k),
 * r = 1 / sqrt(S / K + eps), xh_k = (x_k r) gamma_k; then xh rounded to
 * fp32 and quantized by oracle_quantize_q8_1 (the quantizer's fp32
 * definition decides the codes).  xh_out (may be NULL) receives the fp64
 * xh, [M][K], for the checks that need the exact value. */
void oracle_rmsnorm_quantize_q8_1(const float* x, int64_t ldx, const float* gamma, float eps, int M, int K,
                                  uint8_t* out, double* xh_out)
{
    float* xh = (float*)malloc(sizeof(float) * (size_t)K);
    if (!xh) return;
    for (int m = 0; m < M; ++m) {
        const float* xr = x + (int64_t)m * ldx;
        double S = 0.0;
        for (int k = 0; k < K; ++k) S += (double)xr[k] * (double)xr[k];
        const double r = 1.0 / sqrt(S / (double)K + (double)eps);
        for (int k = 0; k < K; ++k) {
            const double v = ((double)xr[k] * r) * (double)gamma[k];
            if (xh_out) xh_out[(int64_t)m * K + k] = v;
            xh[k] = (float)v;
        }
        oracle_quantize_q8_1(xh, K, 1, K, out + (int64_t)m * (K / 32) * Q8_1_BYTES);
    }
    free(xh);
}

/* ------------------------------------------------------------------ */
/* Weight decoding from the canonical block bytes                        */
/* ------------------------------------------------------------------ */

/* 4-bit code of value i (0..31) of a canonical Q4_0 block. */
static int q4_0_code(const uint8_t* blk, int i)
{
    const uint8_t* qs = blk + 2;
    return i < 16 ? (qs[i] & 0x0F) : (qs[i - 16] >> 4);
}

/* 6-bit code of value i (0..255) of a canonical Q6_K superblock. */
static int q6_k_code(const uint8_t* sb, int i)
{
    const uint8_t* ql = sb;
    const uint8_t* qh = sb + 128;
    int lo = (ql[i >> 1] >> (4 * (i & 1))) & 0x0F;
    int hi = (qh[i >> 2] >> (2 * (i & 3))) & 0x03;
    return lo | (hi << 4);
}

static int q6_k_subscale(const uint8_t* sb, int j) { return (int)(int8_t)sb[192 + j]; }
static uint16_t q6_k_d(const uint8_t* sb) { return rd16(sb + 208); }

/* Dequantized weights, fp64: the brute-force side of the pins. */
void oracle_dequant_q4_0(const uint8_t* w, int N, int K, double* out)
{
    int nb = K / 32;
    for (int n = 0; n < N; ++n)
        for (int b = 0; b < nb; ++b) {
            const uint8_t* blk = w + ((int64_t)n * nb + b) * Q4_0_BYTES;
            double d = oracle_f16_to_f64(rd16(blk));
            for (int i = 0; i < 32; ++i)
                out[(int64_t)n * K + 32 * b + i] = d * (double)(q4_0_code(blk, i) - 8);
        }
}

void oracle_dequant_q6_k(const uint8_t* w, int N, int K, double* out)
{
    int ns = K / 256;
    for (int n = 0; n < N; ++n)
        for (int s = 0; s < ns; ++s) {
            const uint8_t* sb = w + ((int64_t)n * ns + s) * Q6_K_BYTES;
            double d = oracle_f16_to_f64(q6_k_d(sb));
            for (int i = 0; i < 256; ++i)
                out[(int64_t)n * K + 256 * s + i] =
                    d * (double)q6_k_subscale(sb, i >> 4) * (double)(q6_k_code(sb, i) - 32);
        }
}

/* Q8_0 ("further K-quant formats"; the llama.cpp-family block): 32 weights,
 * fp16 d then int8 q[32], value d * q. */
void oracle_dequant_q8_0(const uint8_t* w, int N, int K, double* out)
{
    int nb = K / 32;
    for (int n = 0; n < N; ++n)
        for (int b = 0; b < nb; ++b) {
            const uint8_t* blk = w + ((int64_t)n * nb + b) * Q8_0_BYTES;
            double d = oracle_f16_to_f64(rd16(blk));
            for (int i = 0; i < 32; ++i) out[(int64_t)n * K + 32 * b + i] = d * (double)(int8_t)blk[2 + i];
        }
}

/* Q4_K and Q5_K: the scale and min of sub-block j (0..7) of a superblock. */
static void q4_k_scale_min(const uint8_t* sb, int j, int* sc, int* m)
{
    const uint8_t* s = sb + 4;
    if (j < 4) {
        *sc = s[j] & 63;
        *m = s[j + 4] & 63;
    } else {
        *sc = (s[j + 4] & 15) | ((s[j - 4] >> 6) << 4);
        *m = (s[j + 4] >> 4) | ((s[j] >> 6) << 4);
    }
}

/* Q4_K: the 4-bit code of value i (0..255) of a superblock. */
static int q4_k_code(const uint8_t* sb, int i)
{
    const uint8_t* qs = sb + 16;
    int c = i / 64, r = i % 64;
    return r < 32 ? (qs[32 * c + r] & 15) : (qs[32 * c + r - 32] >> 4);
}

/* Q5_K: the 5-bit code of value i (0..255): the Q4_K nibble of the code
 * bytes (after the 32 qh bytes) plus 16 times bit i / 32 of qh[i % 32]. */
static int q5_k_code(const uint8_t* sb, int i)
{
    const uint8_t* qh = sb + 16;
    const uint8_t* qs = sb + 48;
    int c = i / 64, r = i % 64;
    int lo = r < 32 ? (qs[32 * c + r] & 15) : (qs[32 * c + r - 32] >> 4);
    return lo + 16 * ((qh[i % 32] >> (i / 32)) & 1);
}

void oracle_dequant_q5_k(const uint8_t* w, int N, int K, double* out)
{
    int ns = K / 256;
    for (int n = 0; n < N; ++n)
        for (int s = 0; s < ns; ++s) {
            const uint8_t* sb = w + ((int64_t)n * ns + s) * Q5_K_BYTES;
            double d = oracle_f16_to_f64(rd16(sb)), dmin = oracle_f16_to_f64(rd16(sb + 2));
            for (int i = 0; i < 256; ++i) {
                int sc, m;
                q4_k_scale_min(sb, i / 32, &sc, &m);
                out[(int64_t)n * K + 256 * s + i] = d * (double)sc * (double)q5_k_code(sb, i) - dmin * (double)m;
            }
        }
}

void oracle_dequant_q4_k(const uint8_t* w, int N, int K, double* out)
{
    int ns = K / 256;
    for (int n = 0; n < N; ++n)
        for (int s = 0; s < ns; ++s) {
            const uint8_t* sb = w + ((int64_t)n * ns + s) * Q4_K_BYTES;
            double d = oracle_f16_to_f64(rd16(sb)), dmin = oracle_f16_to_f64(rd16(sb + 2));
            for (int i = 0; i < 256; ++i) {
                int sc, m;
                q4_k_scale_min(sb, i / 32, &sc, &m);
                out[(int64_t)n * K + 256 * s + i] = d * (double)sc * (double)q4_k_code(sb, i) - dmin * (double)m;
            }
        }
}

void oracle_dequant_q8_1(const uint8_t* xq, int M, int K, double* out)
{
    int nb = K / 32;
    for (int m = 0; m < M; ++m)
        for (int b = 0; b < nb; ++b) {
            const uint8_t* blk = xq + ((int64_t)m * nb + b) * Q8_1_BYTES;
            double d = oracle_f16_to_f64(rd16(blk));
            for (int i = 0; i < 32; ++i)
                out[(int64_t)m * K + 32 * b + i] = d * (double)(int8_t)blk[4 + i];
        }
}

/* ------------------------------------------------------------------ */
/* Exact integer block dots                                              */
/* ------------------------------------------------------------------ */

/* I = sum_i (q_w(i) - 8) * q_a(i) over one 32-value block. */
static int32_t block_dot_q4_0(const uint8_t* wblk, const uint8_t* ablk)
{
    int32_t I = 0;
    for (int i = 0; i < 32; ++i)
        I += (q4_0_code(wblk, i) - 8) * (int32_t)(int8_t)ablk[4 + i];
    return I;
}

/* I = sum_i q_w(i) * q_a(i) over one 32-value Q8_0 block. */
static int32_t block_dot_q8_0(const uint8_t* wblk, const uint8_t* ablk)
{
    int32_t I = 0;
    for (int i = 0; i < 32; ++i) I += (int32_t)(int8_t)wblk[2 + i] * (int32_t)(int8_t)ablk[4 + i];
    return I;
}

/* J = sum over the two 16-value subblocks j of block bb of superblock sb:
 *     sc_j * sum_i (q(i) - 32) * q_a(i). */
static int32_t block_dot_q6_k(const uint8_t* sb, int bb, const uint8_t* ablk)
{
    int32_t J = 0;
    for (int h = 0; h < 2; ++h) {
        int j = 2 * bb + h;
        int32_t g = 0;
        for (int t = 0; t < 16; ++t) {
            int i = 16 * j + t;
            g += (q6_k_code(sb, i) - 32) * (int32_t)(int8_t)ablk[4 + 16 * h + t];
        }
        J += q6_k_subscale(sb, j) * g;
    }
    return J;
}

/* Q4_K, block bb (sub-block bb) of superblock sb: I = sum_i q(i) * q_a(i)
 * and A = sum_i q_a(i), the two exact integers of
 * sum_i (d sc q(i) - dmin m) * d_a q_a(i) = d sc d_a I - dmin m d_a A. */
static void block_dot_q4_k(const uint8_t* sb, int bb, const uint8_t* ablk, int32_t* I, int32_t* A, int five)
{
    int32_t i1 = 0, a1 = 0;
    for (int t = 0; t < 32; ++t) {
        int32_t qa = (int32_t)(int8_t)ablk[4 + t];
        i1 += (five ? q5_k_code(sb, 32 * bb + t) : q4_k_code(sb, 32 * bb + t)) * qa;
        a1 += qa;
    }
    *I = i1;
    *A = a1;
}

/* I[m][n][b] for every block: the integer dots before any scaling. */
void oracle_block_dots_q4_0(const uint8_t* w, const uint8_t* xq, int M, int K, int N, int32_t* I)
{
    int nb = K / 32;
    for (int m = 0; m < M; ++m)
        for (int n = 0; n < N; ++n)
            for (int b = 0; b < nb; ++b)
                I[((int64_t)m * N + n) * nb + b] =
                    block_dot_q4_0(w + ((int64_t)n * nb + b) * Q4_0_BYTES,
                                   xq + ((int64_t)m * nb + b) * Q8_1_BYTES);
}

void oracle_block_dots_q6_k(const uint8_t* w, const uint8_t* xq, int M, int K, int N, int32_t* I)
{
    int nb = K / 32, ns = K / 256;
    for (int m = 0; m < M; ++m)
        for (int n = 0; n < N; ++n)
            for (int b = 0; b < nb; ++b)
                I[((int64_t)m * N + n) * nb + b] =
                    block_dot_q6_k(w + ((int64_t)n * ns + b / 8) * Q6_K_BYTES, b % 8,
                                   xq + ((int64_t)m * nb + b) * Q8_1_BYTES);
}

/* ------------------------------------------------------------------ */
/* y[m][n] = sum_b d_w * d_a * I_b  (fp64), and S[m][n] = sum_b |term|   */
/* ------------------------------------------------------------------ */

typedef struct {
    int fmt; /* 0 = Q4_0, 1 = Q6_K, 2 = Q8_0, 3 = Q4_K, 4 = Q5_K */
    const uint8_t* w;
    const uint8_t* xq;
    int M, K, N;
    int n0, n1;
    double* y;
    double* S;
} gemv_job;

static void gemv_rows(const gemv_job* j)
{
    int nb = j->K / 32, ns = j->K / 256;
    for (int n = j->n0; n < j->n1; ++n) {
        for (int m = 0; m < j->M; ++m) {
            double acc = 0.0, sabs = 0.0;
            for (int b = 0; b < nb; ++b) {
                const uint8_t* ablk = j->xq + ((int64_t)m * nb + b) * Q8_1_BYTES;
                double da = oracle_f16_to_f64(rd16(ablk));
                double dw;
                int32_t I;
                if (j->fmt == 3 || j->fmt == 4) {
                    /* two terms: d sc d_a I and - dmin m d_a A */
                    const uint8_t* sb =
                        j->w + ((int64_t)n * ns + b / 8) * (j->fmt == 3 ? Q4_K_BYTES : Q5_K_BYTES);
                    int sc, mn;
                    int32_t A;
                    q4_k_scale_min(sb, b % 8, &sc, &mn);
                    block_dot_q4_k(sb, b % 8, ablk, &I, &A, j->fmt == 4);
                    double t1 = oracle_f16_to_f64(rd16(sb)) * (double)sc * da * (double)I;
                    double t2 = -oracle_f16_to_f64(rd16(sb + 2)) * (double)mn * da * (double)A;
                    acc += t1 + t2;
                    sabs += fabs(t1) + fabs(t2);
                    continue;
                }
                if (j->fmt == 0) {
                    const uint8_t* wblk = j->w + ((int64_t)n * nb + b) * Q4_0_BYTES;
                    dw = oracle_f16_to_f64(rd16(wblk));
                    I = block_dot_q4_0(wblk, ablk);
                } else if (j->fmt == 1) {
                    const uint8_t* sb = j->w + ((int64_t)n * ns + b / 8) * Q6_K_BYTES;
                    dw = oracle_f16_to_f64(q6_k_d(sb));
                    I = block_dot_q6_k(sb, b % 8, ablk);
                } else {
                    const uint8_t* wblk = j->w + ((int64_t)n * nb + b) * Q8_0_BYTES;
                    dw = oracle_f16_to_f64(rd16(wblk));
                    I = block_dot_q8_0(wblk, ablk);
                }
                double t = dw * da * (double)I;
                acc += t;
                sabs += fabs(t);
            }
            j->y[(int64_t)m * j->N + n] = acc;
            if (j->S) j->S[(int64_t)m * j->N + n] = sabs;
        }
    }
}

static void* gemv_thread(void* p)
{
    gemv_rows((const gemv_job*)p);
    return NULL;
}

static void gemv_run(int fmt, const uint8_t* w, const uint8_t* xq, int M, int K, int N,
                     double* y, double* S, int nthreads)
{
    if (nthreads < 1) nthreads = 1;
    if (nthreads > N) nthreads = N > 0 ? N : 1;
    gemv_job* jobs = (gemv_job*)calloc((size_t)nthreads, sizeof(gemv_job));
    pthread_t* th = (pthread_t*)calloc((size_t)nthreads, sizeof(pthread_t));
    for (int t = 0; t < nthreads; ++t) {
        gemv_job j = {fmt, w, xq, M, K, N,
                      (int)((int64_t)N * t / nthreads), (int)((int64_t)N * (t + 1) / nthreads), y, S};
        jobs[t] = j;
    }
    for (int t = 1; t < nthreads; ++t) pthread_create(&th[t], NULL, gemv_thread, &jobs[t]);
    gemv_rows(&jobs[0]);
    for (int t = 1; t < nthreads; ++t) pthread_join(th[t], NULL);
    free(jobs);
    free(th);
}

/* w: canonical Q8_0 [N][K/32] x 34 B; otherwise as oracle_qgemv_q4_0. */
void oracle_qgemv_q8_0(const uint8_t* w, const uint8_t* xq, int M, int K, int N,
                       double* y, double* S, int nthreads)
{
    gemv_run(2, w, xq, M, K, N, y, S, nthreads);
}

/* w: canonical Q4_K [N][K/256] x 144 B; S sums both terms' magnitudes. */
void oracle_qgemv_q4_k(const uint8_t* w, const uint8_t* xq, int M, int K, int N,
                       double* y, double* S, int nthreads)
{
    gemv_run(3, w, xq, M, K, N, y, S, nthreads);
}

/* w: canonical Q5_K [N][K/256] x 176 B; as oracle_qgemv_q4_k. */
void oracle_qgemv_q5_k(const uint8_t* w, const uint8_t* xq, int M, int K, int N,
                       double* y, double* S, int nthreads)
{
    gemv_run(4, w, xq, M, K, N, y, S, nthreads);
}

/* w: canonical Q4_0 [N][K/32] x 18 B; xq: Q8_1 [M][K/32] x 36 B;
 * y, S: fp64 [M][N] (S may be NULL). */
void oracle_qgemv_q4_0(const uint8_t* w, const uint8_t* xq, int M, int K, int N,
                       double* y, double* S, int nthreads)
{
    gemv_run(0, w, xq, M, K, N, y, S, nthreads);
}

/* w: canonical Q6_K [N][K/256] x 210 B. */
void oracle_qgemv_q6_k(const uint8_t* w, const uint8_t* xq, int M, int K, int N,
                       double* y, double* S, int nthreads)
{
    gemv_run(1, w, xq, M, K, N, y, S, nthreads);
}

/* ------------------------------------------------------------------ */
/* Greedy top-1 with the lowest-token-ID finite-tie rule                 */
/* ------------------------------------------------------------------ */

/* ids[m] = the lowest n attaining the maximum of y[m][0..N); -0 equals +0;
 * NaN never wins; a row that is all NaN gives 0.  +Inf is an ordinary value. */
void oracle_top1_f64(const double* y, int64_t ldy, int M, int N, int32_t* ids)
{
    for (int m = 0; m < M; ++m) {
        const double* r = y + (int64_t)m * ldy;
        int best = -1;
        for (int n = 0; n < N; ++n) {
            if (isnan(r[n])) continue;
            if (best < 0 || r[n] > r[best]) best = n;
        }
        ids[m] = best < 0 ? 0 : best;
    }
}

void oracle_top1_f32(const float* y, int64_t ldy, int M, int N, int32_t* ids)
{
    for (int m = 0; m < M; ++m) {
        const float* r = y + (int64_t)m * ldy;
        int best = -1;
        for (int n = 0; n < N; ++n) {
            if (isnan(r[n])) continue;
            if (best < 0 || r[n] > r[best]) best = n;
        }
        ids[m] = best < 0 ? 0 : best;
    }
}
