/*
 * Seeded synthetic-input generator for the DSA decode/prefill workloads.
 *
 * This module produces random numbers and lays them out; it contains none of
 * the indexer or attention arithmetic.  Both the CPU oracle's tests and the
 * CUDA path's tests/benchmark draw their inputs from here, so that the two
 * sides see bit-identical data.
 *
 * Random source: SplitMix64 (Steele, Lea, Flood, "Fast splittable pseudorandom
 * number generators", OOPSLA 2014).  The i-th output of a SplitMix64 stream
 * with state `key` is mix64(key + (i + 1) * GOLDEN); we use it as a
 * counter-based generator, so any element can be produced independently and
 * the result does not depend on thread count or machine.
 *
 * Normal variates use the classical "sum of twelve uniforms minus six"
 * (Irwin-Hall n = 12: mean 0, variance 1, support [-6, 6]).  Every step is
 * exact integer arithmetic followed by one exact division by 2^16, so x86 and
 * Arm hosts produce identical bits (no libm calls).
 *
 * FP8 E4M3 encoding follows the OCP 8-bit floating point specification
 * (OFP8, E4M3 variant: bias 7, no infinities, S.1111.111 is NaN, maximum
 * finite 448), rounding to nearest-even with saturation to +-448.
 */
#include <stdint.h>
#include <string.h>
#include <math.h>
#include <stdlib.h>

#define GOLDEN 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

/* i-th output (i >= 0) of the SplitMix64 stream whose initial state is key. */
uint64_t dsa_gen_draw(uint64_t key, uint64_t i) { return mix64(key + (i + 1) * GOLDEN); }

/* Independent stream for (seed, tensor id). */
uint64_t dsa_gen_stream_key(uint64_t seed, uint64_t tensor_id) {
    return mix64(mix64(seed ^ 0x6A09E667F3BCC909ULL) + tensor_id * GOLDEN);
}

static inline uint16_t f32_to_bf16_rne(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7F800000u) == 0x7F800000u) return (uint16_t)((u >> 16) | ((u & 0xFFFFu) ? 0x40u : 0u));
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

/* Irwin-Hall(12) - 6 from three 64-bit draws (twelve 16-bit uniforms). Exact in float. */
static inline float ih12(uint64_t key, uint64_t c) {
    int64_t s = 0;
    for (int k = 0; k < 3; ++k) {
        uint64_t d = dsa_gen_draw(key, 3 * c + (uint64_t)k);
        s += (int64_t)(d & 0xFFFF) + (int64_t)((d >> 16) & 0xFFFF) + (int64_t)((d >> 32) & 0xFFFF) +
             (int64_t)(d >> 48);
    }
    /* sum_k (u_k + 0.5) / 65536 - 6 = (s + 6 - 6 * 65536) / 65536, exact. */
    return (float)((double)(s + 6 - 6 * 65536) / 65536.0);
}

/* out[i] = bf16(scale * N(0,1)) for counters offset .. offset+n-1.  scale must be a power of two
 * (or 1) for the product to stay exact before rounding. */
void dsa_gen_normal_bf16(uint64_t key, uint64_t offset, int64_t n, float scale, uint16_t* out) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = f32_to_bf16_rne(scale * ih12(key, offset + (uint64_t)i));
}

/* out[i] = lo + (hi - lo) * u, u = 24-bit uniform in [0, 1). */
void dsa_gen_uniform_f32(uint64_t key, uint64_t offset, int64_t n, float lo, float hi, float* out) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        float u = (float)(dsa_gen_draw(key, offset + (uint64_t)i) >> 40) * (1.0f / 16777216.0f);
        out[i] = lo + (hi - lo) * u;
    }
}

/* Uniform integers in [lo, hi] (inclusive). */
void dsa_gen_uniform_int(uint64_t key, uint64_t offset, int64_t n, int64_t lo, int64_t hi, int64_t* out) {
    uint64_t span = (uint64_t)(hi - lo) + 1;
    for (int64_t i = 0; i < n; ++i) out[i] = lo + (int64_t)(dsa_gen_draw(key, offset + (uint64_t)i) % span);
}

/* Fisher-Yates permutation of 0..n-1 (Durstenfeld order, j drawn in [0, i]). */
void dsa_gen_permutation(uint64_t key, int32_t n, int32_t* out) {
    for (int32_t i = 0; i < n; ++i) out[i] = i;
    for (int32_t i = n - 1; i > 0; --i) {
        int32_t j = (int32_t)(dsa_gen_draw(key, (uint64_t)i) % (uint64_t)(i + 1));
        int32_t t = out[i];
        out[i] = out[j];
        out[j] = t;
    }
}

/* m distinct values from 0..n-1 (partial Fisher-Yates), in draw order.  Returns 0 on success. */
int dsa_gen_sample_without_replacement(uint64_t key, int32_t n, int32_t m, int32_t* out) {
    if (m < 0 || m > n) return -1;
    int32_t* a = (int32_t*)malloc(sizeof(int32_t) * (size_t)(n > 0 ? n : 1));
    if (!a) return -2;
    for (int32_t i = 0; i < n; ++i) a[i] = i;
    for (int32_t i = 0; i < m; ++i) {
        int32_t j = i + (int32_t)(dsa_gen_draw(key, (uint64_t)i) % (uint64_t)(n - i));
        int32_t t = a[i];
        a[i] = a[j];
        a[j] = t;
        out[i] = a[i];
    }
    free(a);
    return 0;
}

/*
 * Fill a paged cache [num_pages, page_size, width] (bf16 bits) with N(0,1) * scale rows.
 * Logical row (b, s) draws counters starting at ((b * row_stride_b) + s) * width, so its content
 * does not depend on which physical page holds it.  Slots of a page past the sequence end stay
 * untouched (the caller zero-initialises the cache).
 */
void dsa_gen_paged_normal_bf16(uint64_t key, int32_t batch, const int32_t* seq_lens, const int32_t* page_table,
                               int32_t max_pages, int32_t page_size, int32_t width, int64_t row_stride_b,
                               float scale, uint16_t* cache) {
    for (int32_t b = 0; b < batch; ++b) {
        int32_t L = seq_lens[b];
#pragma omp parallel for schedule(static)
        for (int32_t s = 0; s < L; ++s) {
            int64_t phys = (int64_t)page_table[(int64_t)b * max_pages + s / page_size] * page_size + s % page_size;
            uint64_t c0 = (uint64_t)(((int64_t)b * row_stride_b + s) * (int64_t)width);
            uint16_t* dst = cache + phys * width;
            for (int32_t d = 0; d < width; ++d) dst[d] = f32_to_bf16_rne(scale * ih12(key, c0 + (uint64_t)d));
        }
    }
}

/* OCP E4M3 encode, round-to-nearest-even, saturating to +-448.  NaN input gives 0x7F. */
uint8_t dsa_gen_e4m3_encode(float v) {
    if (v != v) return 0x7F;
    uint8_t sign = (v < 0.0f || (v == 0.0f && signbit(v))) ? 0x80 : 0x00;
    double a = fabs((double)v);
    if (a >= 448.0) return (uint8_t)(sign | 0x7E);
    if (a < 0.015625) { /* below 2^-6: subnormal grid, quantum 2^-9 */
        double n = nearbyint(a * 512.0);
        return (uint8_t)(sign | (uint8_t)n); /* n == 8 is the smallest normal, code 0x08 */
    }
    int e;
    frexp(a, &e); /* a = f * 2^e, f in [0.5, 1) -> a in [2^(e-1), 2^e) */
    int ex = e - 1;  /* a in [2^ex, 2^(ex+1)) */
    double n = nearbyint(ldexp(a, 3 - ex)); /* in [8, 16] */
    if (n >= 16.0) { n = 8.0; ex += 1; }
    int field = ex + 7;
    uint8_t code = (uint8_t)((field << 3) | ((int)n - 8));
    if (field > 15 || code == 0x7F) code = 0x7E;
    return (uint8_t)(sign | code);
}

/*
 * Per-row dynamic quantisation to E4M3: scale = absmax(row) / 448 (1 when the row is all zero),
 * code = e4m3(x / scale).  x is bf16 bits, [rows, cols].  This prepares FP8 inputs; it is not part
 * of the scoring arithmetic.
 */
void dsa_gen_quantize_e4m3_rows(const uint16_t* x, int64_t rows, int32_t cols, uint8_t* codes, float* scales) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        const uint16_t* xr = x + r * cols;
        float amax = 0.0f;
        for (int32_t c = 0; c < cols; ++c) {
            uint32_t u = (uint32_t)xr[c] << 16;
            float f;
            memcpy(&f, &u, 4);
            float af = fabsf(f);
            if (af > amax) amax = af;
        }
        float scale = amax > 0.0f ? amax / 448.0f : 1.0f;
        scales[r] = scale;
        for (int32_t c = 0; c < cols; ++c) {
            uint32_t u = (uint32_t)xr[c] << 16;
            float f;
            memcpy(&f, &u, 4);
            codes[r * cols + c] = dsa_gen_e4m3_encode(f / scale);
        }
    }
}

/* Element-wise E4M3 encoding of n floats (see dsa_gen_e4m3_encode). */
void dsa_gen_e4m3_encode_array(const float* x, int64_t n, uint8_t* out) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = dsa_gen_e4m3_encode(x[i]);
}
