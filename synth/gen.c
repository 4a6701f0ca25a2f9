/*
 * Seeded synthetic inputs for the int8 weight-only Qwen3 decoder.
 *
 * This file is input preparation, shared by the CUDA path's tests/bench and
 * by the CPU oracle's tests.  It holds no model arithmetic: only random draws
 * and the offline per-output-channel int8 quantiser that turns bf16 weights
 * into the (int8, fp32 scale) pairs the library's init() consumes.
 *
 * Quantisation reading ("Model-agnostic LLM inference", section "The quantized
 * load cache": int8 weights plus one scale per row, about one byte per
 * parameter): symmetric, scale = amax(row)/127 in fp32, code =
 * clamp(rint(w/scale), -127, 127) with round-half-to-even; an all-zero row
 * gets scale 1 and codes 0.
 *
 * Random numbers: splitmix64 (Steele, Lea, Flood 2014, "Fast splittable
 * pseudorandom number generators") used as a counter-based generator:
 * draw(key, c) = mix64(key + (c + 1) * 0x9E3779B97F4A7C15).
 * Normals: Box-Muller in double from two draws per pair of elements.
 *
 * Build: gcc -O2 -fPIC -shared -fopenmp -ffp-contract=off gen.c -lm
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define SM_GAMMA 0x9E3779B97F4A7C15ULL
#define KEY_GAMMA 0xD1B54A32D192ED03ULL

static inline uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

static inline uint64_t draw(uint64_t key, uint64_t c) { return mix64(key + (c + 1) * SM_GAMMA); }

/* Key of stream number `index` under `seed` (tensor index, prompt index, ...). */
uint64_t synth_key(uint64_t seed, uint64_t index) { return mix64(seed + (index + 1) * KEY_GAMMA); }

/* Raw 64-bit draws, counters [start, start + n). */
void synth_draws(uint64_t key, uint64_t start, int64_t n, uint64_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = draw(key, start + (uint64_t)i);
}

static inline uint16_t f32_to_bf16_rne(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    uint32_t bias = 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)((u + bias) >> 16);
}

static inline float bf16_to_f32(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* Standard normal number `i` of stream `key`: elements 2j and 2j+1 share the
 * Box-Muller pair built from draws 2j (radius) and 2j+1 (angle). */
static inline double normal_at(uint64_t key, int64_t i) {
    int64_t j = i >> 1;
    uint64_t a = draw(key, 2 * (uint64_t)j);
    uint64_t b = draw(key, 2 * (uint64_t)j + 1);
    double u1 = ((double)(a >> 11) + 1.0) * 0x1.0p-53; /* (0, 1] */
    double u2 = (double)(b >> 11) * 0x1.0p-53;         /* [0, 1) */
    double r = sqrt(-2.0 * log(u1));
    double t = 6.283185307179586476925286766559 * u2;
    return (i & 1) ? r * sin(t) : r * cos(t);
}

/* n bf16 values bf16(float(sigma * N(0,1))) (RNE at both narrowings). */
void synth_normal_bf16(uint64_t key, int64_t n, double sigma, uint16_t* out) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = f32_to_bf16_rne((float)(sigma * normal_at(key, i)));
}

/* n fp32 values float(mean + sigma * N(0,1)). */
void synth_normal_f32(uint64_t key, int64_t n, double mean, double sigma, float* out) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = (float)(mean + sigma * normal_at(key, i));
}

/* Per-row symmetric int8 quantisation of a bf16 matrix [rows, cols]. */
void synth_quantize_rows_bf16(const uint16_t* w, int64_t rows, int64_t cols, int8_t* q, float* scale) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        const uint16_t* wr = w + r * cols;
        float amax = 0.0f;
        for (int64_t c = 0; c < cols; ++c) {
            float v = fabsf(bf16_to_f32(wr[c]));
            if (v > amax) amax = v;
        }
        float s = (amax > 0.0f) ? amax / 127.0f : 1.0f;
        scale[r] = s;
        for (int64_t c = 0; c < cols; ++c) {
            float v = rintf(bf16_to_f32(wr[c]) / s);
            if (v > 127.0f) v = 127.0f;
            if (v < -127.0f) v = -127.0f;
            q[r * cols + c] = (int8_t)v;
        }
    }
}

/* Same quantiser on fp32 input (used by tests that plant exact values). */
void synth_quantize_rows_f32(const float* w, int64_t rows, int64_t cols, int8_t* q, float* scale) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        const float* wr = w + r * cols;
        float amax = 0.0f;
        for (int64_t c = 0; c < cols; ++c) {
            float v = fabsf(wr[c]);
            if (v > amax) amax = v;
        }
        float s = (amax > 0.0f) ? amax / 127.0f : 1.0f;
        scale[r] = s;
        for (int64_t c = 0; c < cols; ++c) {
            float v = rintf(wr[c] / s);
            if (v > 127.0f) v = 127.0f;
            if (v < -127.0f) v = -127.0f;
            q[r * cols + c] = (int8_t)v;
        }
    }
}

/* Draw an N(0, sigma) bf16 matrix from stream `key` and quantise it row by
 * row, without materialising the bf16 matrix (row-chunked). */
void synth_matrix_i8(uint64_t key, int64_t rows, int64_t cols, double sigma, int8_t* q, float* scale) {
#pragma omp parallel
    {
        /* one row of bf16 values per thread, on the stack for cols <= 16384 */
        uint16_t buf[16384];
#pragma omp for schedule(static)
        for (int64_t r = 0; r < rows; ++r) {
            int64_t base = r * cols;
            float amax = 0.0f;
            for (int64_t c = 0; c < cols; ++c) {
                buf[c] = f32_to_bf16_rne((float)(sigma * normal_at(key, base + c)));
                float v = fabsf(bf16_to_f32(buf[c]));
                if (v > amax) amax = v;
            }
            float s = (amax > 0.0f) ? amax / 127.0f : 1.0f;
            scale[r] = s;
            for (int64_t c = 0; c < cols; ++c) {
                float v = rintf(bf16_to_f32(buf[c]) / s);
                if (v > 127.0f) v = 127.0f;
                if (v < -127.0f) v = -127.0f;
                q[base + c] = (int8_t)v;
            }
        }
    }
}

/* n token ids uniform on [0, vocab) (draw mod vocab). */
void synth_ids(uint64_t key, int64_t n, int32_t vocab, int32_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = (int32_t)(draw(key, (uint64_t)i) % (uint64_t)vocab);
}

/* n lengths uniform on [lo, hi] inclusive (lo + draw mod (hi - lo + 1)). */
void synth_lengths(uint64_t key, int64_t n, int32_t lo, int32_t hi, int32_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = lo + (int32_t)(draw(key, (uint64_t)i) % (uint64_t)(hi - lo + 1));
}
