/*
 * Seeded synthetic inputs shared by the CUDA path's tests and bench and by the
 * CPU oracle.  Nothing here computes any part of the cross-entropy method: this
 * file only turns (seed, stream, index) into numbers.
 *
 * Generator: SplitMix64 (G. L. Steele, D. Lea, C. H. Flood, "Fast splittable
 * pseudorandom number generators", OOPSLA 2014), used counter-style: the i-th
 * draw of a stream is the SplitMix64 finaliser applied to key + (i+1)*gamma,
 * which is exactly the (i+1)-th output of a SplitMix64 generator whose state
 * starts at key.  Every element therefore depends only on its own index, so any
 * slice can be produced independently (and in parallel) with the same bytes.
 *
 * Normals: Box-Muller (G. E. P. Box, M. E. Muller, 1958) with the host libm;
 * draw pair k = (u1, u2) gives element 2k = r*cos(2*pi*u2) and 2k+1 = r*sin(...),
 * r = sqrt(-2 ln(1-u1)).  Values are rounded once to float, then to bfloat16
 * by round-to-nearest-even where bf16 output is asked for.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define GAMMA 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

/* Key of stream `stream` under `seed`. */
uint64_t wl_stream_key(uint64_t seed, uint64_t stream) {
    return mix64(seed + GAMMA) ^ mix64(stream * 0xD1B54A32D192ED03ULL + 0x8CB92BA72F3D8DD7ULL);
}

static inline uint64_t draw(uint64_t key, uint64_t i) { return mix64(key + (i + 1) * GAMMA); }

/* 53-bit uniform in [0, 1). */
static inline double unit(uint64_t z) { return (double)(z >> 11) * (1.0 / 9007199254740992.0); }

static inline uint16_t f32_to_bf16_rne(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

/* Raw 64-bit draws i in [i0, i0+n). */
void wl_u64(uint64_t key, uint64_t i0, int64_t n, uint64_t* out) {
    for (int64_t k = 0; k < n; ++k) out[k] = draw(key, i0 + (uint64_t)k);
}

/* Uniform doubles in [0,1) for draws i in [i0, i0+n). */
void wl_uniform(uint64_t key, uint64_t i0, int64_t n, double* out) {
    for (int64_t k = 0; k < n; ++k) out[k] = unit(draw(key, i0 + (uint64_t)k));
}

/* Standard normal element e (Box-Muller pair e/2, cos or sin by parity). */
static inline double normal_at(uint64_t key, uint64_t e) {
    uint64_t pair = e >> 1;
    double u1 = unit(draw(key, 2 * pair));
    double u2 = unit(draw(key, 2 * pair + 1));
    double r = sqrt(-2.0 * log(1.0 - u1));
    double a = 6.283185307179586 * u2;
    return (e & 1) ? r * sin(a) : r * cos(a);
}

/*
 * Element e in [e0, e0+n): mean + sigma * normal, except that when spike_p > 0
 * the element is replaced, with probability spike_p, by a value uniform in
 * [spike_lo, spike_hi) (decided by a second stream `spike_key`).
 * dtype 0 = float32 output, 1 = bfloat16 output (uint16 bits).
 */
void wl_normal(uint64_t key, uint64_t e0, int64_t n, double mean, double sigma,
               uint64_t spike_key, double spike_p, double spike_lo, double spike_hi,
               int dtype, void* out) {
    for (int64_t k = 0; k < n; ++k) {
        uint64_t e = e0 + (uint64_t)k;
        double v = mean + sigma * normal_at(key, e);
        if (spike_p > 0.0) {
            if (unit(draw(spike_key, 2 * e)) < spike_p)
                v = spike_lo + (spike_hi - spike_lo) * unit(draw(spike_key, 2 * e + 1));
        }
        float f = (float)v;
        if (dtype == 0) ((float*)out)[k] = f;
        else ((uint16_t*)out)[k] = f32_to_bf16_rne(f);
    }
}

/*
 * Same as wl_normal, for a row-major matrix with row stride ld >= cols:
 * element (r, c) takes index r*cols + c of the stream, so the values do not
 * depend on ld.  Fills rows [r0, r1).  Padding columns are left untouched.
 */
void wl_normal_matrix(uint64_t key, int64_t r0, int64_t r1, int64_t cols, int64_t ld,
                      double mean, double sigma, uint64_t spike_key, double spike_p,
                      double spike_lo, double spike_hi, int dtype, void* out) {
    size_t es = dtype == 0 ? 4 : 2;
    for (int64_t r = r0; r < r1; ++r) {
        char* row = (char*)out + (size_t)(r - r0) * (size_t)ld * es;
        wl_normal(key, (uint64_t)r * (uint64_t)cols, cols, mean, sigma, spike_key, spike_p,
                  spike_lo, spike_hi, dtype, row);
    }
}
