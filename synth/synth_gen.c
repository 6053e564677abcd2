/* Seeded bf16 normal samples: the C twin of synth/__init__.py.
 *
 * Same definition as the Python module (counter-based SplitMix64 words,
 * Box-Muller pairs, float64 -> float32 -> bfloat16 round-to-nearest-even),
 * written as a loop over element pairs so that the large workloads are
 * generated in well under a second.  No attention arithmetic lives here.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define GAMMA 0x9E3779B97F4A7C15ULL

static uint64_t mix64(uint64_t z) {
    z ^= z >> 30;
    z *= 0xBF58476D1CE4E5B9ULL;
    z ^= z >> 27;
    z *= 0x94D049BB133111EBULL;
    z ^= z >> 31;
    return z;
}

static uint16_t f32_to_bf16(float x) {
    uint32_t b;
    memcpy(&b, &x, 4);
    uint32_t rounding = ((b >> 16) & 1u) + 0x7FFFu;
    return (uint16_t)((b + rounding) >> 16);
}

/* n samples of N(0, sigma^2) from stream `stream` under `seed` into out[]. */
void synth_normal_bf16(uint64_t seed, int stream, int64_t n, double sigma, uint16_t *out) {
    const uint64_t base = mix64(seed * 4u + (uint64_t)stream + 1u);
    const int64_t npairs = (n + 1) / 2;
    const double two_pi = 2.0 * 3.14159265358979323846;
#pragma omp parallel for schedule(static)
    for (int64_t p = 0; p < npairs; ++p) {
        uint64_t w1 = mix64(base + (uint64_t)(2 * p + 1) * GAMMA);
        uint64_t w2 = mix64(base + (uint64_t)(2 * p + 2) * GAMMA);
        double u1 = ((double)(w1 >> 11) + 1.0) * 0x1p-53;
        double u2 = ((double)(w2 >> 11) + 1.0) * 0x1p-53;
        double r = sqrt(-2.0 * log(u1));
        double th = two_pi * u2;
        double z0 = r * cos(th) * sigma;
        double z1 = r * sin(th) * sigma;
        out[2 * p] = f32_to_bf16((float)z0);
        if (2 * p + 1 < n) out[2 * p + 1] = f32_to_bf16((float)z1);
    }
}
