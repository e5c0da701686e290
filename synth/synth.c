/*
 * synth.c -- seeded, counter-based synthetic input generator.
 *
 * This module produces the input tensors (hidden states, router logits,
 * expert weights, bias) that both the CPU oracle and the CUDA path consume.
 * It holds none of the MoE layer's arithmetic: only random numbers and the
 * fp32 -> bf16 storage rounding of the generated values.
 *
 * Generator definition (each element depends only on (seed, tensor_id, i),
 * so any slice of a tensor reproduces the same bytes as the whole tensor):
 *
 *   mix(z)      = the splitmix64 finaliser (Steele, Lea, Flood 2014):
 *                 z ^= z>>30; z *= 0xbf58476d1ce4e5b9;
 *                 z ^= z>>27; z *= 0x94d049bb133111eb; z ^= z>>31
 *   key         = mix(mix(seed + G) ^ mix(tensor_id + 2G)),  G = 0x9e3779b97f4a7c15
 *   word(c)     = mix(key + (c+1)*G)
 *   uniform(c)  = ((word(c) >> 11) + 1) * 2^-53            in (0, 1]
 *   pair q      : u1 = uniform(2q), u2 = uniform(2q+1),
 *                 r = sqrt(-2 ln u1), theta = 2 pi u2       (Box-Muller)
 *   normal(i)   = r cos(theta) for even i, r sin(theta) for odd i, q = i/2
 *
 * Values are formed in double, scaled (mean + std*normal), rounded to fp32
 * (round to nearest even), and for bf16 tensors rounded again fp32 -> bf16
 * (round to nearest even on the upper 16 bits).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define G64 0x9e3779b97f4a7c15ULL

static uint64_t mix64(uint64_t z) {
    z ^= z >> 30;
    z *= 0xbf58476d1ce4e5b9ULL;
    z ^= z >> 27;
    z *= 0x94d049bb133111ebULL;
    z ^= z >> 31;
    return z;
}

static uint64_t stream_key(uint64_t seed, uint64_t tensor_id) {
    return mix64(mix64(seed + G64) ^ mix64(tensor_id + 2 * G64));
}

static double uniform01(uint64_t key, uint64_t c) {
    uint64_t w = mix64(key + (c + 1) * G64);
    return (double)((w >> 11) + 1) * (1.0 / 9007199254740992.0);
}

/* the standard normal deviate number i of the stream */
static double normal_at(uint64_t key, uint64_t i) {
    uint64_t q = i >> 1;
    double u1 = uniform01(key, 2 * q);
    double u2 = uniform01(key, 2 * q + 1);
    double r = sqrt(-2.0 * log(u1));
    double th = 6.283185307179586476925286766559 * u2;
    return (i & 1) ? r * sin(th) : r * cos(th);
}

static uint16_t f32_to_bf16_rne(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu)) return 0x7fc0; /* NaN */
    u += 0x7fffu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

/* out[j] = fp32(mean + std * normal(start + j)), j in [0, n) */
void synth_normal_f32(uint64_t seed, uint64_t tensor_id, uint64_t start, int64_t n,
                      double mean, double std, float* out) {
    uint64_t key = stream_key(seed, tensor_id);
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < n; ++j) out[j] = (float)(mean + std * normal_at(key, start + (uint64_t)j));
}

/* out[j] = bf16(fp32(std * normal(start + j))), j in [0, n) */
void synth_normal_bf16(uint64_t seed, uint64_t tensor_id, uint64_t start, int64_t n,
                       double std, uint16_t* out) {
    uint64_t key = stream_key(seed, tensor_id);
    /* pairs share (u1, u2): walk them two at a time for speed, same values */
#pragma omp parallel for schedule(static)
    for (int64_t jj = 0; jj < (n + 1) / 2; ++jj) {
        int64_t j0 = 2 * jj;
        uint64_t i0 = start + (uint64_t)j0;
        if ((i0 & 1) == 0 && j0 + 1 < n) {
            uint64_t q = i0 >> 1;
            double u1 = uniform01(key, 2 * q);
            double u2 = uniform01(key, 2 * q + 1);
            double r = sqrt(-2.0 * log(u1));
            double th = 6.283185307179586476925286766559 * u2;
            out[j0] = f32_to_bf16_rne((float)(std * (r * cos(th))));
            out[j0 + 1] = f32_to_bf16_rne((float)(std * (r * sin(th))));
        } else {
            for (int64_t j = j0; j < j0 + 2 && j < n; ++j)
                out[j] = f32_to_bf16_rne((float)(std * normal_at(key, start + (uint64_t)j)));
        }
    }
}

/* uniform integers in [0, m): out[j] = floor(uniform(start + j) * m) clamped to m-1 */
void synth_uniform_int(uint64_t seed, uint64_t tensor_id, uint64_t start, int64_t n,
                       int64_t m, int32_t* out) {
    uint64_t key = stream_key(seed, tensor_id);
    for (int64_t j = 0; j < n; ++j) {
        int64_t v = (int64_t)(uniform01(key, start + (uint64_t)j) * (double)m);
        out[j] = (int32_t)(v >= m ? m - 1 : v);
    }
}

/* fp32 -> bf16 round-to-nearest-even of an existing buffer (input preparation) */
void synth_f32_to_bf16(const float* in, int64_t n, uint16_t* out) {
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < n; ++j) out[j] = f32_to_bf16_rne(in[j]);
}
