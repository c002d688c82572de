/*
 * ORACLE -- test infrastructure only.
 *
 * A plain, slow, obviously-correct CPU statement of what the quantized decode GEMV computes.  Only the
 * test suite, the smoke check and the benchmark's CPU-baseline leg load it; the CUDA library never
 * calls, links or includes anything from here, and this file includes nothing from the library.
 *
 * What it follows:
 *   - vllm.cpp PR #1936 ("raise Qwen3.5-4B Q4_K_M gfx1100 decode"), the SGLang/vLLM study section: the
 *     activation row is quantized ONCE to q8_1-style int8 blocks, then every output row streams its
 *     K-quant super-blocks, dequantizes them and reduces the dot product.  The integer block dots are
 *     exact under any association (same page, the dp4a / amd_mixed_dot section), so the result is a
 *     closed-form quantity: y[i,n] = sum_k w[n,k] * xhat[i,k].  This file computes exactly that in
 *     fp64 with one sequential loop, from weights and activations decoded element by element.
 *   - The same page, QuantizeQ8KK / warp-coop section: amax of the block, scale amax/127, nearest-int,
 *     clamp to 127.  The q8_1 block is specified step by step below because it is an encoding whose
 *     bytes must match bit for bit.
 *   - MetaInfer-cpp README, W8A16 section: int8 weights with a scale, 16-bit activations, fp32
 *     accumulation.  Here the result is formed in fp64 from the decoded values (the reference value).
 *
 * Block formats (no page gives bit packing; these are this project's own, stated from the block
 * semantics of the synthetic workloads).  All multi-byte fields little-endian, fp16 = IEEE binary16.
 *   q8_1 (36 B / 32 values): d fp16 @0, s fp16 @2, qs[32] int8 @4.  xhat = d * q.
 *   Q4_K (144 B / 256): d fp16 @0, dmin fp16 @2, 12 bytes @4 holding a 96-bit little-endian bit string
 *        whose field f occupies bits 6f..6f+5 (f < 8: sc[f], f >= 8: mn[f-8]), qs[128] @16 where byte
 *        32g+t holds element 64g+t (low nibble) and element 64g+32+t (high nibble).
 *        w[e] = d * sc[e/32] * q[e] - dmin * mn[e/32].
 *   Q6_K (210 B / 256): ql[128] @0 where byte 64h+t holds the low 4 bits of element 128h+t (low nibble)
 *        and of element 128h+64+t (high nibble); qh[64] @128 where byte 32h+t holds bits 4..5 of element
 *        128h+32k+t in its bits 2k..2k+1; sc[16] int8 @192; d fp16 @208.  w[e] = d * sc[e/16] * (q[e]-32).
 *   Q8_0 (34 B / 32): d fp16 @0, qs[32] int8 @2.  w = d * q.
 *   Q5_K (176 B / 256): the Q4_K header (d, dmin, 96-bit scale string) @0; qh[32] @16 where bit j of byte t
 *        is bit 4 of element 32j+t; qs[128] @48 packed as Q4_K's qs.  q[e] in 0..31,
 *        w[e] = d * sc[e/32] * q[e] - dmin * mn[e/32].  (vllm.cpp PR #1936 decodes Q5_K in the same
 *        integer-dot loops as Q4_K/Q6_K, the amd_mixed_dot section.)
 *   A matrix is row-major: row n is K/256 (or K/32) consecutive blocks, rows contiguous, no padding.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORACLE_Q4_K = 1, ORACLE_Q6_K = 2, ORACLE_Q8_0 = 3, ORACLE_Q5_K = 5 };

/* ------------------------------------------------------------------------------------------------ */
/* Scalar encodings                                                                                   */

/* IEEE binary16 -> value (exact in fp64). */
double oracle_fp16_to_f64(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 31;
    int f = h & 1023;
    double v;
    if (e == 0) v = ldexp((double)f, -24);
    else if (e == 31) v = f ? NAN : INFINITY;
    else v = ldexp((double)(1024 + f), e - 25);
    return sign ? -v : v;
}

/* bfloat16 -> value (exact in fp64). */
double oracle_bf16_to_f64(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* fp32 -> IEEE binary16, round to nearest, ties to even; overflow -> inf, NaN -> quiet NaN. */
uint16_t oracle_f32_to_fp16(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
    uint32_t a = u & 0x7FFFFFFFu;
    if (a >= 0x7F800000u) return (uint16_t)(sign | (a > 0x7F800000u ? 0x7E00u : 0x7C00u));
    if (a >= 0x477FF000u) return (uint16_t)(sign | 0x7C00u); /* >= 65520 rounds to inf */
    int e32 = (int)(a >> 23) - 127;
    uint32_t mant = a & 0x7FFFFFu;
    if (e32 >= -14) { /* normal binary16 */
        uint32_t h = ((uint32_t)(e32 + 15) << 10) | (mant >> 13);
        uint32_t rem = mant & 0x1FFFu;
        if (rem > 0x1000u || (rem == 0x1000u && (h & 1u))) h += 1u;
        return (uint16_t)(sign | h);
    }
    /* subnormal binary16 (unit 2^-24) or zero */
    uint32_t sig = (a >> 23) ? (0x800000u | mant) : mant;
    int s = -(e32 + 1); /* value = sig * 2^(e32-23) = (sig >> s) units of 2^-24 */
    if ((a >> 23) == 0 || s > 24) return sign;
    uint32_t h = sig >> s;
    uint32_t rem = sig & ((1u << s) - 1u);
    uint32_t half = 1u << (s - 1);
    if (rem > half || (rem == half && (h & 1u))) h += 1u;
    return (uint16_t)(sign | h);
}

static uint16_t rd_u16(const uint8_t* p) { return (uint16_t)(p[0] | (p[1] << 8)); }

/* ------------------------------------------------------------------------------------------------ */
/* Activation quantizer: fp32 [m, K] -> q8_1 blocks.                                                  */
/* Per 32-value block:                                                                                */
/*   amax = max |x|                        (fp32, exact)                                              */
/*   d32  = amax / 127                     (one IEEE fp32 division, nearest-even)                     */
/*   d    = binary16(d32)                  (nearest-even)                                             */
/*   q    = clamp(roundf(x / d32), -127, 127)  (IEEE fp32 division, ties away from zero);             */
/*          q = 0 for every value when d32 == 0                                                       */
/*   s    = binary16(float(d) * sum(q))    (the fp32 product is exact: 11-bit times 13-bit)           */

void oracle_quantize_act(const float* x, int m, int K, uint8_t* xq) {
    int nb = K / 32;
    for (int i = 0; i < m; ++i) {
        for (int b = 0; b < nb; ++b) {
            const float* xb = x + (size_t)i * K + (size_t)b * 32;
            uint8_t* out = xq + ((size_t)i * nb + b) * 36;
            float amax = 0.0f;
            for (int j = 0; j < 32; ++j) {
                float a = fabsf(xb[j]);
                if (a > amax) amax = a;
            }
            float d32 = amax / 127.0f;
            uint16_t dh = oracle_f32_to_fp16(d32);
            int sum = 0;
            for (int j = 0; j < 32; ++j) {
                int q = 0;
                if (d32 != 0.0f) {
                    float r = roundf(xb[j] / d32);
                    if (r > 127.0f) r = 127.0f;
                    if (r < -127.0f) r = -127.0f;
                    q = (r == r) ? (int)r : 0;
                }
                out[4 + j] = (uint8_t)(int8_t)q;
                sum += q;
            }
            float dfl = (float)oracle_fp16_to_f64(dh);
            float sp = dfl * (float)sum;
            uint16_t sh = oracle_f32_to_fp16(sp);
            out[0] = (uint8_t)(dh & 0xFF); out[1] = (uint8_t)(dh >> 8);
            out[2] = (uint8_t)(sh & 0xFF); out[3] = (uint8_t)(sh >> 8);
        }
    }
}

/* q8_1 blocks -> xhat [m, K] = fp16(d) * q. */
void oracle_dequant_q8_1(const uint8_t* xq, int m, int K, double* xhat) {
    int nb = K / 32;
    for (int i = 0; i < m; ++i)
        for (int b = 0; b < nb; ++b) {
            const uint8_t* blk = xq + ((size_t)i * nb + b) * 36;
            double d = oracle_fp16_to_f64(rd_u16(blk));
            for (int j = 0; j < 32; ++j) xhat[(size_t)i * K + (size_t)b * 32 + j] = d * (double)(int8_t)blk[4 + j];
        }
}

/* ------------------------------------------------------------------------------------------------ */
/* Weight decoders: one row (K values) from its blocks.                                              */

static int bit_at(const uint8_t* p, int t) { return (p[t >> 3] >> (t & 7)) & 1; }

/* The 16 six-bit fields of the 96-bit scale string at b + 4 (Q4_K and Q5_K): sc[0..7], then mn[0..7]. */
static void kquant_fields(const uint8_t* b, int field[16]) {
    for (int f = 0; f < 16; ++f) {
        int v = 0;
        for (int k = 0; k < 6; ++k) v |= bit_at(b + 4, 6 * f + k) << k;
        field[f] = v;
    }
}

/* Low 4 bits of element e from a Q4_K-style qs[128] array. */
static int low_nibble_code(const uint8_t* qs, int e) {
    int g = e / 64, r = e % 64;
    return (r < 32) ? (qs[32 * g + r] & 0x0F) : (qs[32 * g + r - 32] >> 4);
}

/* w[e] = d * sc[e/32] * q[e] - dmin * mn[e/32] (Q4_K and Q5_K). */
static double kquant_weight(double d, double dmin, const int field[16], int q, int e) {
    int j = e / 32;
    return d * (double)field[j] * (double)q - dmin * (double)field[8 + j];
}

static void dequant_q4k_block(const uint8_t* b, double* w) {
    double d = oracle_fp16_to_f64(rd_u16(b));
    double dmin = oracle_fp16_to_f64(rd_u16(b + 2));
    int field[16];
    kquant_fields(b, field);
    for (int e = 0; e < 256; ++e) w[e] = kquant_weight(d, dmin, field, low_nibble_code(b + 16, e), e);
}

static void dequant_q5k_block(const uint8_t* b, double* w) {
    double d = oracle_fp16_to_f64(rd_u16(b));
    double dmin = oracle_fp16_to_f64(rd_u16(b + 2));
    int field[16];
    kquant_fields(b, field);
    const uint8_t* qh = b + 16;
    const uint8_t* qs = b + 48;
    for (int e = 0; e < 256; ++e) {
        int hi = (qh[e % 32] >> (e / 32)) & 1;
        int q = low_nibble_code(qs, e) + 16 * hi;
        w[e] = kquant_weight(d, dmin, field, q, e);
    }
}

static void dequant_q6k_block(const uint8_t* b, double* w) {
    const uint8_t* ql = b;
    const uint8_t* qh = b + 128;
    const int8_t* sc = (const int8_t*)(b + 192);
    double d = oracle_fp16_to_f64(rd_u16(b + 208));
    for (int e = 0; e < 256; ++e) {
        int h = e / 128, r = e % 128;
        int lo = (r < 64) ? (ql[64 * h + r] & 0x0F) : (ql[64 * h + r - 64] >> 4);
        int k = r / 32, t = r % 32;
        int hi = (qh[32 * h + t] >> (2 * k)) & 3;
        int q = lo | (hi << 4);
        w[e] = d * (double)sc[e / 16] * (double)(q - 32);
    }
}

static void dequant_q80_block(const uint8_t* b, double* w) {
    double d = oracle_fp16_to_f64(rd_u16(b));
    for (int j = 0; j < 32; ++j) w[j] = d * (double)(int8_t)b[2 + j];
}

static int fmt_block(int fmt, int* bytes, int* elems) {
    switch (fmt) {
    case ORACLE_Q4_K: *bytes = 144; *elems = 256; return 0;
    case ORACLE_Q5_K: *bytes = 176; *elems = 256; return 0;
    case ORACLE_Q6_K: *bytes = 210; *elems = 256; return 0;
    case ORACLE_Q8_0: *bytes = 34; *elems = 32; return 0;
    }
    return -1;
}

int64_t oracle_row_bytes(int fmt, int K) {
    int bb, be;
    if (fmt_block(fmt, &bb, &be) || K % be) return -1;
    return (int64_t)(K / be) * bb;
}

/* Dequantize row n of an [N, K] matrix into w[K].  Returns 0, or -1 on a bad format / K. */
int oracle_dequant_row(int fmt, const uint8_t* W, int K, int64_t n, double* w) {
    int bb, be;
    if (fmt_block(fmt, &bb, &be) || K % be) return -1;
    int nb = K / be;
    const uint8_t* row = W + (size_t)n * (size_t)nb * (size_t)bb;
    for (int b = 0; b < nb; ++b) {
        const uint8_t* blk = row + (size_t)b * bb;
        double* wb = w + (size_t)b * be;
        if (fmt == ORACLE_Q4_K) dequant_q4k_block(blk, wb);
        else if (fmt == ORACLE_Q5_K) dequant_q5k_block(blk, wb);
        else if (fmt == ORACLE_Q6_K) dequant_q6k_block(blk, wb);
        else dequant_q80_block(blk, wb);
    }
    return 0;
}

/* ------------------------------------------------------------------------------------------------ */
/* GEMV: y[i, r] = sum_k w[rows[r], k] * xhat[i, k], fp64, one sequential loop over k.              */
/* y is [m, nrows] row-major.  rows == NULL means all N rows in order (nrows = N).                    */

int oracle_gemv_rows(int fmt, const uint8_t* W, const uint8_t* xq, int m, int N, int K,
                     const int64_t* rows, int64_t nrows, double* y) {
    if (oracle_row_bytes(fmt, K) < 0 || K % 32 || m < 1) return -1;
    double* xhat = (double*)malloc(sizeof(double) * (size_t)m * K);
    double* w = (double*)malloc(sizeof(double) * (size_t)K);
    if (!xhat || !w) { free(xhat); free(w); return -2; }
    oracle_dequant_q8_1(xq, m, K, xhat);
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t n = rows ? rows[r] : r;
        if (n < 0 || n >= N) { free(xhat); free(w); return -1; }
        oracle_dequant_row(fmt, W, K, n, w);
        for (int i = 0; i < m; ++i) {
            const double* xi = xhat + (size_t)i * K;
            double acc = 0.0;
            for (int k = 0; k < K; ++k) acc += w[k] * xi[k];
            y[(size_t)i * nrows + r] = acc;
        }
    }
    free(xhat);
    free(w);
    return 0;
}

int oracle_gemv(int fmt, const uint8_t* W, const uint8_t* xq, int m, int N, int K, double* y) {
    return oracle_gemv_rows(fmt, W, xq, m, N, K, NULL, N, y);
}

/* W8A16: y[i, r] = sum_k (d_blk * q[n, k]) * bf16(x[i, k]), fp64, sequential over k. */
int oracle_w8a16_rows(const uint8_t* W, const uint16_t* x, int m, int N, int K,
                      const int64_t* rows, int64_t nrows, double* y) {
    if (K % 32 || m < 1) return -1;
    double* xv = (double*)malloc(sizeof(double) * (size_t)m * K);
    double* w = (double*)malloc(sizeof(double) * (size_t)K);
    if (!xv || !w) { free(xv); free(w); return -2; }
    for (size_t t = 0; t < (size_t)m * K; ++t) xv[t] = oracle_bf16_to_f64(x[t]);
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t n = rows ? rows[r] : r;
        if (n < 0 || n >= N) { free(xv); free(w); return -1; }
        oracle_dequant_row(ORACLE_Q8_0, W, K, n, w);
        for (int i = 0; i < m; ++i) {
            const double* xi = xv + (size_t)i * K;
            double acc = 0.0;
            for (int k = 0; k < K; ++k) acc += w[k] * xi[k];
            y[(size_t)i * nrows + r] = acc;
        }
    }
    free(xv);
    free(w);
    return 0;
}

int oracle_w8a16(const uint8_t* W, const uint16_t* x, int m, int N, int K, double* y) {
    return oracle_w8a16_rows(W, x, m, N, K, NULL, N, y);
}

/* Per-output-channel INT8 W8A16 (MetaInfer-cpp README, the Qwen3-14B TP4 W8A16 decode section: signed
 * INT8 weights, an fp32 scale per output channel, bf16 activations, fp32 accumulation):
 *   y[i, r] = scale[n] * sum_k q[n, k] * bf16(x[i, k]),  n = rows[r],
 * formed in fp64 (the products are exact; one sequential sum, then one multiply by the scale). */
int oracle_w8c_rows(const int8_t* W, const float* scale, const uint16_t* x, int m, int N, int K,
                    const int64_t* rows, int64_t nrows, double* y) {
    if (K % 32 || m < 1) return -1;
    double* xv = (double*)malloc(sizeof(double) * (size_t)m * K);
    if (!xv) return -2;
    for (size_t t = 0; t < (size_t)m * K; ++t) xv[t] = oracle_bf16_to_f64(x[t]);
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t n = rows ? rows[r] : r;
        if (n < 0 || n >= N) { free(xv); return -1; }
        const int8_t* wn = W + (size_t)n * K;
        for (int i = 0; i < m; ++i) {
            const double* xi = xv + (size_t)i * K;
            double acc = 0.0;
            for (int k = 0; k < K; ++k) acc += (double)wn[k] * xi[k];
            y[(size_t)i * nrows + r] = (double)scale[n] * acc;
        }
    }
    free(xv);
    return 0;
}
