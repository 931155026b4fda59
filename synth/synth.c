/* Seeded synthetic client updates for the FedAvg aggregation tests and bench:
 * host side.  Input creation only -- no aggregation arithmetic lives here.
 *
 * Definition (shared, bit for bit, with synth_dev.cu):
 *   draw(key, c)  = c-th output of SplitMix64 seeded with key
 *                   (Steele, Lea & Flood, OOPSLA 2014)
 *   client key    = draw(seed, client)
 *   normal value  : element i takes draws 3i..3i+2 of the client key; the
 *                   twelve 16-bit fields u_j give the Irwin-Hall(12) sum
 *                   s = sum(u_j) - 393210, z = s * 2^-16  (mean 0, var ~1)
 *   Student-t(3)  : element i takes draws 12i..12i+11 -> four sums s0..s3,
 *                   t = (s0*2^-16) / sqrt(((s1^2+s2^2+s3^2)*2^-32) / 3)
 *   value         = sigma * z  (or sigma * t), one IEEE double multiply
 *   stored fp32   = value rounded to float (round to nearest)
 *   stored bf16   = upper 16 bits of that float (truncation toward zero)
 * Every operation is either integer or a single correctly rounded IEEE
 * double operation, so host and device agree exactly.  Build without
 * floating-point contraction (-ffp-contract=off).
 */
#include <stdint.h>
#include <string.h>
#include <math.h>

#define SM64_GAMMA 0x9E3779B97F4A7C15ULL

static inline uint64_t sm64_mix(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

static inline uint64_t sm64_draw(uint64_t key, uint64_t c) {
    return sm64_mix(key + (c + 1) * SM64_GAMMA);
}

static inline int64_t ih12(uint64_t key, uint64_t c0) {
    int64_t s = 0;
    for (int d = 0; d < 3; ++d) {
        uint64_t r = sm64_draw(key, c0 + (uint64_t)d);
        s += (int64_t)(r & 0xFFFF) + (int64_t)((r >> 16) & 0xFFFF) +
             (int64_t)((r >> 32) & 0xFFFF) + (int64_t)(r >> 48);
    }
    return s - 393210;
}

uint64_t synth_client_key(uint64_t seed, uint64_t client) {
    return sm64_draw(seed, client);
}

double synth_value(uint64_t key, int dist, double sigma, uint64_t i) {
    if (dist == 0) {
        double z = (double)ih12(key, 3 * i) * 0x1p-16;
        return sigma * z;
    }
    int64_t s0 = ih12(key, 12 * i);
    int64_t s1 = ih12(key, 12 * i + 3);
    int64_t s2 = ih12(key, 12 * i + 6);
    int64_t s3 = ih12(key, 12 * i + 9);
    int64_t vi = s1 * s1 + s2 * s2 + s3 * s3;
    if (vi == 0) vi = 1;
    double v = (double)vi * 0x1p-32;
    double q = v / 3.0;
    double r = sqrt(q);
    double t = ((double)s0 * 0x1p-16) / r;
    return sigma * t;
}

/* Fill out[0..n) with elements first..first+n-1 of (seed, client).
 * dtype 0 = fp32 (float*), 1 = bf16 (uint16_t*). */
void synth_fill(uint64_t seed, uint64_t client, int dist, double sigma, int dtype,
                uint64_t first, uint64_t n, void* out) {
    uint64_t key = synth_client_key(seed, client);
    if (dtype == 0) {
        float* o = (float*)out;
        for (uint64_t j = 0; j < n; ++j) o[j] = (float)synth_value(key, dist, sigma, first + j);
    } else {
        uint16_t* o = (uint16_t*)out;
        for (uint64_t j = 0; j < n; ++j) {
            float f = (float)synth_value(key, dist, sigma, first + j);
            uint32_t u;
            memcpy(&u, &f, 4);
            o[j] = (uint16_t)(u >> 16);
        }
    }
}

/* Gather: out[j] = element idx[j] of (seed, client). */
void synth_gather(uint64_t seed, uint64_t client, int dist, double sigma, int dtype,
                  const uint64_t* idx, uint64_t n, void* out) {
    uint64_t key = synth_client_key(seed, client);
    for (uint64_t j = 0; j < n; ++j) {
        float f = (float)synth_value(key, dist, sigma, idx[j]);
        if (dtype == 0) {
            ((float*)out)[j] = f;
        } else {
            uint32_t u;
            memcpy(&u, &f, 4);
            ((uint16_t*)out)[j] = (uint16_t)(u >> 16);
        }
    }
}
