/*
 * Seeded, counter-based synthetic input generator.
 *
 * This file is shared input plumbing: it serves both the CPU oracle and the
 * GPU path with the same bytes, and it holds none of the decoding method's
 * arithmetic (no norm, no GEMV, no attention, no rounding of activations).
 *
 * Definition (version independent, the same on x86_64 and aarch64):
 *   mix(z)            SplitMix64 output function (Steele, Lea, Flood 2014):
 *                       z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9
 *                       z = (z ^ (z >> 27)) * 0x94D049BB133111EB
 *                       z =  z ^ (z >> 31)
 *   key(seed, tid)    mix(seed * 0x9E3779B97F4A7C15 + tid + 1)
 *   r(seed, tid, c)   mix(key + (c + 1) * 0x9E3779B97F4A7C15)
 *                     (the SplitMix64 sequence started at state `key`,
 *                      indexed by counter c, so any element is computable
 *                      on its own)
 *   u(c)              ((r(c) >> 11) + 1) * 2^-53, in (0, 1]
 *   normal pair j     Box-Muller on u(2j), u(2j+1) in double precision:
 *                       n[2j]   = sqrt(-2 ln u(2j)) * cos(2 pi u(2j+1))
 *                       n[2j+1] = sqrt(-2 ln u(2j)) * sin(2 pi u(2j+1))
 *   bf16 value        sigma * n  -> nearest float -> bfloat16 by
 *                     round-to-nearest-even on the upper 16 bits
 *   gain value        1 + sigma * n -> nearest float -> bfloat16 (same rounding)
 *   token id          r(c) mod n_vocab
 *
 * Every element depends only on (seed, tid, element index), so a tensor can
 * be generated in pieces, by any number of threads, in any order.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define GOLDEN 0x9E3779B97F4A7C15ULL

static inline uint64_t sm_mix(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

static inline uint64_t sm_key(uint64_t seed, uint64_t tid) {
    return sm_mix(seed * GOLDEN + tid + 1ULL);
}

/* Plain SplitMix64 stream: state s, n outputs (state += GOLDEN; out = mix). */
void synth_splitmix64_stream(uint64_t state, uint64_t *out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) {
        state += GOLDEN;
        out[i] = sm_mix(state);
    }
}

uint64_t synth_raw(uint64_t seed, uint64_t tid, uint64_t c) {
    return sm_mix(sm_key(seed, tid) + (c + 1ULL) * GOLDEN);
}

static inline double sm_unit(uint64_t r) {
    return (double)((r >> 11) + 1ULL) * (1.0 / 9007199254740992.0);
}

static inline uint16_t f32_to_bf16_bits(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7F800000u) == 0x7F800000u) { /* inf / nan: keep, quiet nan */
        return (uint16_t)((u >> 16) | ((u & 0xFFFFu) ? 0x40u : 0u));
    }
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

static inline double sm_normal(uint64_t key, int64_t i) {
    int64_t j = i >> 1;
    double u1 = sm_unit(sm_mix(key + (uint64_t)(2 * j + 1) * GOLDEN));
    double u2 = sm_unit(sm_mix(key + (uint64_t)(2 * j + 2) * GOLDEN));
    double rad = sqrt(-2.0 * log(u1));
    double ang = 6.283185307179586476925286766559 * u2;
    return (i & 1) ? rad * sin(ang) : rad * cos(ang);
}

/* Normal(0, sigma) values as float, elements [i0, i0 + n) of tensor (seed, tid). */
void synth_normal_f32(uint64_t seed, uint64_t tid, int64_t i0, int64_t n, double sigma,
                      float *out) {
    uint64_t key = sm_key(seed, tid);
#pragma omp parallel for schedule(static)
    for (int64_t k = 0; k < n; ++k) out[k] = (float)(sigma * sm_normal(key, i0 + k));
}

/* Normal(0, sigma) values as bfloat16 bits, elements [i0, i0 + n). */
void synth_normal_bf16(uint64_t seed, uint64_t tid, int64_t i0, int64_t n, double sigma,
                       uint16_t *out) {
    uint64_t key = sm_key(seed, tid);
#pragma omp parallel for schedule(static)
    for (int64_t k = 0; k < n; ++k)
        out[k] = f32_to_bf16_bits((float)(sigma * sm_normal(key, i0 + k)));
}

/*
 * KV-cache prefill: fills positions [0, n_pos) of a cache laid out as
 * [n_heads][max_pos][head_dim] bf16; element (h, p, j) takes the value of
 * element index (h * n_pos + p) * head_dim + j of tensor (seed, tid).
 * Positions >= n_pos are left untouched.
 */
void synth_kv_prefill_bf16(uint64_t seed, uint64_t tid, int n_heads, int max_pos, int n_pos,
                           int head_dim, double sigma, uint16_t *cache) {
    uint64_t key = sm_key(seed, tid);
#pragma omp parallel for collapse(2) schedule(static)
    for (int h = 0; h < n_heads; ++h)
        for (int p = 0; p < n_pos; ++p) {
            int64_t src = ((int64_t)h * n_pos + p) * head_dim;
            uint16_t *dst = cache + ((int64_t)h * max_pos + p) * head_dim;
            for (int j = 0; j < head_dim; ++j)
                dst[j] = f32_to_bf16_bits((float)(sigma * sm_normal(key, src + j)));
        }
}

/* Uniform token ids in [0, n_vocab): element c of tensor (seed, tid). */
void synth_tokens(uint64_t seed, uint64_t tid, int64_t n, int64_t n_vocab, int32_t *out) {
    for (int64_t c = 0; c < n; ++c) out[c] = (int32_t)(synth_raw(seed, tid, (uint64_t)c) % (uint64_t)n_vocab);
}

/* Norm gains 1 + sigma * n as bfloat16 bits, n the standard normal element c of
 * tensor (seed, tid): the seeded non-unit gains of the parity tests. */
void synth_gain_bf16(uint64_t seed, uint64_t tid, int64_t n, double sigma, uint16_t *out) {
    uint64_t key = sm_key(seed, tid);
    for (int64_t k = 0; k < n; ++k) out[k] = f32_to_bf16_bits((float)(1.0 + sigma * sm_normal(key, k)));
}

/* Fill with a constant bfloat16 bit pattern (used for norm gains = 1.0). */
void synth_fill_bf16(uint16_t *out, int64_t n, uint16_t bits) {
    for (int64_t k = 0; k < n; ++k) out[k] = bits;
}
