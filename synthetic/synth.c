/*
 * Seeded, counter-based synthetic inputs for the batch-1 decode engine and its
 * oracle.  This file draws random numbers only; it holds none of the decoder's
 * arithmetic.  Every element is a pure function of (seed, tensor_id, index), so
 * any slice can be regenerated alone and the result does not depend on the
 * thread count.
 *
 * Definition (stated so that another implementation can reproduce it):
 *   key(seed, tid, j)   = seed XOR (tid << 40) XOR j                (uint64)
 *   splitmix64(z):        z += 0x9E3779B97F4A7C15;
 *                         z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9;
 *                         z = (z ^ (z >> 27)) * 0x94D049BB133111EB;
 *                         return z ^ (z >> 31)
 *   unit(x)             = ((x >> 11) + 1) * 2^-53                   in (0, 1]
 *   normal(seed,tid,i)  = sqrt(-2 ln u1) * cos(2 pi u2),  u1 = unit(splitmix64(key(.., 2i))),
 *                                                          u2 = unit(splitmix64(key(.., 2i+1)))
 *   All in IEEE double; the fp16 outputs are the double value times `std`,
 *   rounded to nearest-even fp16 by the compiler's _Float16 conversion.
 *
 * Built with -ffp-contract=off so that no fused multiply-add changes a result
 * between the x86 and Arm builds.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define SYNTH_PI 3.14159265358979323846

static inline uint64_t splitmix64(uint64_t z) {
    z += 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

static inline uint64_t synth_key(uint64_t seed, uint64_t tid, uint64_t j) {
    return seed ^ (tid << 40) ^ j;
}

static inline double synth_unit(uint64_t x) {
    return (double)((x >> 11) + 1) * (1.0 / 9007199254740992.0);
}

static inline double synth_normal(uint64_t seed, uint64_t tid, uint64_t i) {
    double u1 = synth_unit(splitmix64(synth_key(seed, tid, 2 * i)));
    double u2 = synth_unit(splitmix64(synth_key(seed, tid, 2 * i + 1)));
    return sqrt(-2.0 * log(u1)) * cos(2.0 * SYNTH_PI * u2);
}

static inline uint16_t f16_bits(double v) {
    _Float16 h = (_Float16)v;
    uint16_t b;
    memcpy(&b, &h, 2);
    return b;
}

/* out[i] = fp16(std * normal(seed, tid, i)), i in [0, n). */
void synth_normal_f16(uint64_t seed, uint64_t tid, double std_dev, int64_t n, uint16_t* out) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = f16_bits(std_dev * synth_normal(seed, tid, (uint64_t)i));
}

/* out[i] = fp32(std * normal(seed, tid, i)). */
void synth_normal_f32(uint64_t seed, uint64_t tid, double std_dev, int64_t n, float* out) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = (float)(std_dev * synth_normal(seed, tid, (uint64_t)i));
}

/* out[i] = splitmix64(key(seed, tid, i)) mod m  (token ids uniform in [0, m)). */
void synth_uniform_int(uint64_t seed, uint64_t tid, int64_t n, int64_t m, int32_t* out) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = (int32_t)(splitmix64(synth_key(seed, tid, (uint64_t)i)) % (uint64_t)m);
}

/*
 * Activations with rare outliers: out[i] = fp16(normal(seed, tid, i)) except
 * that, with probability p_out (decided by a third hash stream), the element
 * is replaced by +mag or -mag (sign from the lowest bit of that hash, a bit
 * that the selector draw does not use).
 */
void synth_outlier_f16(uint64_t seed, uint64_t tid, double p_out, double mag, int64_t n, uint16_t* out) {
    const uint64_t tid_sel = tid ^ 0x5A5A5Aull;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        uint64_t h = splitmix64(synth_key(seed, tid_sel, (uint64_t)i));
        double u = synth_unit(h);
        double v = (u <= p_out) ? ((h & 1u) ? -mag : mag) : synth_normal(seed, tid, (uint64_t)i);
        out[i] = f16_bits(v);
    }
}
