/*
 * Seeded synthetic-input generator shared by the tests, the benchmark and the smoke check.
 *
 * It draws random numbers and writes them into the storage layout of each block format; it holds none of
 * the quantize/dequantize/dot arithmetic of the GEMV method.  Every value is a pure function of
 * (seed, counter), so any range of a tensor can be regenerated independently and in parallel.
 *
 * Random source: SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom number generators",
 * OOPSLA 2014), used in its counter form: output(seed, c) = mix64(seed + (c + 1) * GOLDEN).
 *
 * Value recipes (the synthetic workloads of the decode sweeps):
 *   - fp16 scales: uniform in [lo, hi] drawn in fp64, then rounded to binary16 (round-to-nearest-even).
 *   - N(0,1) activations: Box-Muller on two fp64 uniforms, rounded to fp32 (or fp32 -> bf16, RNE).
 *   - Q5_K-style block (176 B): as Q4_K, plus 32 random bytes of high code bits (codes uniform 0..31).
 *   - Q4_K-style block (144 B): d, dmin fp16 uniform scales; 12 scale bytes and 128 code bytes uniformly
 *     random (so every 6-bit scale/min field is uniform 0..63 and every 4-bit code uniform 0..15).
 *   - Q6_K-style block (210 B): 192 random bytes of low/high code bits (codes uniform 0..63), 16 int8
 *     sub-scales uniform in -64..63, fp16 d.
 *   - Q8_0-style block (34 B): fp16 d, 32 int8 codes uniform in -127..127.
 * Field offsets follow the block layouts declared in include/qgemv.h.
 */
#include <stdint.h>
#include <string.h>
#include <math.h>
#include <pthread.h>
#include <unistd.h>

#define GOLDEN 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

uint64_t qgen_u64(uint64_t seed, uint64_t counter) { return mix64(seed + (counter + 1) * GOLDEN); }

/* Derive an independent stream seed from a parent seed and a tag. */
uint64_t qgen_derive(uint64_t parent, uint64_t tag) { return mix64(parent ^ mix64(tag + GOLDEN)); }

static inline double unit_f64(uint64_t u) { return (double)(u >> 11) * (1.0 / 9007199254740992.0); }

static inline uint16_t to_fp16_bits(double v) {
    _Float16 h = (_Float16)v; /* one IEEE rounding, nearest-even */
    uint16_t b;
    memcpy(&b, &h, 2);
    return b;
}

static inline uint16_t f32_to_bf16_bits(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return (uint16_t)((u >> 16) | 0x40u);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

static inline uint16_t fp16_uniform(uint64_t seed, uint64_t c, double lo, double hi) {
    return to_fp16_bits(lo + (hi - lo) * unit_f64(qgen_u64(seed, c)));
}

static inline void normal_pair(uint64_t seed, uint64_t pair, double* z0, double* z1) {
    double u1 = 1.0 - unit_f64(qgen_u64(seed, 2 * pair)); /* (0, 1] */
    double u2 = unit_f64(qgen_u64(seed, 2 * pair + 1));
    double r = sqrt(-2.0 * log(u1));
    double a = 6.283185307179586476925286766559 * u2;
    *z0 = r * cos(a);
    *z1 = r * sin(a);
}

static inline void put_u16(uint8_t* p, uint16_t v) { p[0] = (uint8_t)(v & 0xFF); p[1] = (uint8_t)(v >> 8); }

static inline void put_u64_bytes(uint8_t* p, uint64_t v, int n) {
    for (int i = 0; i < n; ++i) p[i] = (uint8_t)(v >> (8 * i));
}

/* ---------------------------------------------------------------------------------------------------- */
/* Per-item generators: item index -> bytes.  Each consumes a fixed counter window per item.            */

typedef struct {
    int kind;
    void* dst;
    uint64_t seed;
    double lo, hi;
    int64_t begin, end; /* item range */
} job_t;

enum { K_Q4K = 1, K_Q6K = 2, K_Q80 = 3, K_NORMAL_F32 = 4, K_NORMAL_BF16 = 5, K_BYTES = 6, K_FP16U = 7, K_Q5K = 8 };

static void gen_q4k_block(uint8_t* b, uint64_t seed, int64_t i, double lo, double hi) {
    uint64_t c0 = (uint64_t)i * 20u;
    put_u16(b + 0, fp16_uniform(seed, c0 + 0, lo, hi));
    put_u16(b + 2, fp16_uniform(seed, c0 + 1, lo, hi));
    uint8_t rnd[144];
    for (int w = 0; w < 18; ++w) put_u64_bytes(rnd + 8 * w, qgen_u64(seed, c0 + 2 + w), 8);
    memcpy(b + 4, rnd, 12);        /* scales: 16 six-bit fields */
    memcpy(b + 16, rnd + 16, 128); /* 256 four-bit codes */
}

static void gen_q5k_block(uint8_t* b, uint64_t seed, int64_t i, double lo, double hi) {
    uint64_t c0 = (uint64_t)i * 24u;
    put_u16(b + 0, fp16_uniform(seed, c0 + 0, lo, hi));
    put_u16(b + 2, fp16_uniform(seed, c0 + 1, lo, hi));
    uint8_t rnd[176];
    for (int w = 0; w < 22; ++w) put_u64_bytes(rnd + 8 * w, qgen_u64(seed, c0 + 2 + w), 8);
    memcpy(b + 4, rnd, 12);        /* scales: 16 six-bit fields */
    memcpy(b + 16, rnd + 16, 160); /* 256 high bits (32 B), then 256 four-bit codes (128 B) */
}

static void gen_q6k_block(uint8_t* b, uint64_t seed, int64_t i, double lo, double hi) {
    uint64_t c0 = (uint64_t)i * 27u;
    uint8_t rnd[208];
    for (int w = 0; w < 26; ++w) put_u64_bytes(rnd + 8 * w, qgen_u64(seed, c0 + 1 + w), 8);
    memcpy(b, rnd, 192); /* low nibbles (128 B) + high 2-bit pairs (64 B) */
    for (int j = 0; j < 16; ++j) {
        int v = (int)(rnd[192 + j] & 0x7F) - 64; /* uniform -64..63 */
        b[192 + j] = (uint8_t)(int8_t)v;
    }
    put_u16(b + 208, fp16_uniform(seed, c0, lo, hi));
}

static void gen_q80_block(uint8_t* b, uint64_t seed, int64_t i, double lo, double hi) {
    uint64_t c0 = (uint64_t)i * 33u;
    put_u16(b, fp16_uniform(seed, c0, lo, hi));
    for (int j = 0; j < 32; ++j) {
        uint64_t u = qgen_u64(seed, c0 + 1 + j) >> 32;
        int v = (int)((u * 255u) >> 32) - 127; /* uniform -127..127 */
        b[2 + j] = (uint8_t)(int8_t)v;
    }
}

static void run_range(job_t* j) {
    for (int64_t i = j->begin; i < j->end; ++i) {
        switch (j->kind) {
        case K_Q4K: gen_q4k_block((uint8_t*)j->dst + 144 * i, j->seed, i, j->lo, j->hi); break;
        case K_Q5K: gen_q5k_block((uint8_t*)j->dst + 176 * i, j->seed, i, j->lo, j->hi); break;
        case K_Q6K: gen_q6k_block((uint8_t*)j->dst + 210 * i, j->seed, i, j->lo, j->hi); break;
        case K_Q80: gen_q80_block((uint8_t*)j->dst + 34 * i, j->seed, i, j->lo, j->hi); break;
        case K_NORMAL_F32:
        case K_NORMAL_BF16: { /* item = one Box-Muller pair */
            double z0, z1;
            normal_pair(j->seed, (uint64_t)i, &z0, &z1);
            float f0 = (float)z0, f1 = (float)z1;
            if (j->kind == K_NORMAL_F32) {
                float* d = (float*)j->dst;
                d[2 * i] = f0;
                d[2 * i + 1] = f1;
            } else {
                uint16_t* d = (uint16_t*)j->dst;
                d[2 * i] = f32_to_bf16_bits(f0);
                d[2 * i + 1] = f32_to_bf16_bits(f1);
            }
            break;
        }
        case K_BYTES: put_u64_bytes((uint8_t*)j->dst + 8 * i, qgen_u64(j->seed, (uint64_t)i), 8); break;
        case K_FP16U: ((uint16_t*)j->dst)[i] = fp16_uniform(j->seed, (uint64_t)i, j->lo, j->hi); break;
        }
    }
}

static void* thread_main(void* p) {
    run_range((job_t*)p);
    return 0;
}

static void run_parallel(int kind, void* dst, uint64_t seed, double lo, double hi, int64_t items) {
    long ncpu = sysconf(_SC_NPROCESSORS_ONLN);
    int nt = (int)(ncpu < 1 ? 1 : (ncpu > 32 ? 32 : ncpu));
    if (items < 65536) nt = 1;
    job_t jobs[32];
    pthread_t th[32];
    int64_t per = (items + nt - 1) / nt;
    int started = 0;
    for (int t = 0; t < nt; ++t) {
        jobs[t].kind = kind; jobs[t].dst = dst; jobs[t].seed = seed; jobs[t].lo = lo; jobs[t].hi = hi;
        jobs[t].begin = per * t < items ? per * t : items;
        jobs[t].end = per * (t + 1) < items ? per * (t + 1) : items;
        if (t == 0) continue;
        if (pthread_create(&th[t], 0, thread_main, &jobs[t]) == 0) started |= (1 << t);
        else run_range(&jobs[t]);
    }
    run_range(&jobs[0]);
    for (int t = 1; t < nt; ++t)
        if (started & (1 << t)) pthread_join(th[t], 0);
}

/* ---------------------------------------------------------------------------------------------------- */
/* Exported fills.  Sizes are in items of the named kind.                                                */

void qgen_q4k(uint8_t* dst, int64_t nblocks, uint64_t seed, double lo, double hi) { run_parallel(K_Q4K, dst, seed, lo, hi, nblocks); }
void qgen_q5k(uint8_t* dst, int64_t nblocks, uint64_t seed, double lo, double hi) { run_parallel(K_Q5K, dst, seed, lo, hi, nblocks); }
void qgen_q6k(uint8_t* dst, int64_t nblocks, uint64_t seed, double lo, double hi) { run_parallel(K_Q6K, dst, seed, lo, hi, nblocks); }
void qgen_q80(uint8_t* dst, int64_t nblocks, uint64_t seed, double lo, double hi) { run_parallel(K_Q80, dst, seed, lo, hi, nblocks); }

/* n must be even (pairs). */
void qgen_normal_f32(float* dst, int64_t n, uint64_t seed) { run_parallel(K_NORMAL_F32, dst, seed, 0, 0, n / 2); }
void qgen_normal_bf16(uint16_t* dst, int64_t n, uint64_t seed) { run_parallel(K_NORMAL_BF16, dst, seed, 0, 0, n / 2); }

/* n must be a multiple of 8. */
void qgen_bytes(uint8_t* dst, int64_t n, uint64_t seed) { run_parallel(K_BYTES, dst, seed, 0, 0, n / 8); }

void qgen_fp16_uniform(uint16_t* dst, int64_t n, uint64_t seed, double lo, double hi) { run_parallel(K_FP16U, dst, seed, lo, hi, n); }

/* Per-channel INT8 weights: n int8 values uniform in -127..127 (the symmetric quantizer's range). */
void qgen_int8_sym(int8_t* dst, int64_t n, uint64_t seed) {
    for (int64_t i = 0; i < n; ++i) {
        uint64_t u = qgen_u64(seed, (uint64_t)i) >> 32;
        dst[i] = (int8_t)((int)((u * 255u) >> 32) - 127);
    }
}

/* n fp32 values uniform in [lo, hi] (drawn in fp64, rounded to fp32). */
void qgen_f32_uniform(float* dst, int64_t n, uint64_t seed, double lo, double hi) {
    for (int64_t i = 0; i < n; ++i) dst[i] = (float)(lo + (hi - lo) * unit_f64(qgen_u64(seed, (uint64_t)i)));
}
