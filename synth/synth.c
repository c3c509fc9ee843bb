/*
 * synth.c — seeded synthetic inputs for the decode-step workloads.
 *
 * This module produces the weights, the prefilled KV cache and the token
 * stream that both the CUDA path and the CPU oracle consume.  It holds none
 * of the decode step's arithmetic: it only draws numbers.  Every value is a
 * pure function of (seed, tensor name, element index), so any slice of any
 * tensor can be regenerated independently and in parallel, and the result
 * does not depend on the thread count.
 *
 * Generator: the splitmix64 sequence (Steele, Lea, Flood, "Fast splittable
 * pseudorandom number generators", OOPSLA 2014).  A tensor's stream starts at
 * state mix(seed * K1 + fnv1a64(name)); element draw j is mix(state + (j+1)*G)
 * with G the 64-bit golden-ratio increment, i.e. the j-th output of a
 * splitmix64 generator seeded with that state.
 *
 * Normals: Box-Muller (Box & Muller 1958) on two draws per element, in double.
 * int8: multiply-shift of the top 32 bits onto 255 values, then -127.
 * bf16: round-to-nearest-even of the float32 value.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

#define GOLDEN 0x9E3779B97F4A7C15ull

static inline uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

uint64_t synth_name_hash(const char *name) {
    uint64_t h = 0xcbf29ce484222325ull; /* FNV-1a 64 */
    for (const unsigned char *p = (const unsigned char *)name; *p; ++p) {
        h ^= (uint64_t)*p;
        h *= 0x100000001b3ull;
    }
    return h;
}

static inline uint64_t stream_state(uint64_t seed, const char *name) {
    return mix64(seed * 0xD1B54A32D192ED03ull + synth_name_hash(name));
}

static inline uint64_t draw(uint64_t state, uint64_t j) {
    return mix64(state + (j + 1) * GOLDEN);
}

/* uniform in (0, 1] from the top 53 bits */
static inline double unit_open0(uint64_t r) {
    return ((double)(r >> 11) + 1.0) * (1.0 / 9007199254740992.0);
}

/* uniform in [0, 1) from the top 53 bits */
static inline double unit_closed0(uint64_t r) {
    return (double)(r >> 11) * (1.0 / 9007199254740992.0);
}

static inline uint16_t f32_to_bf16_rne(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7f800000u) == 0x7f800000u) /* inf / nan: keep, quiet nan */
        return (uint16_t)((u >> 16) | ((u & 0xffffu) ? 0x40u : 0u));
    u += 0x7fffu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

static inline double normal_at(uint64_t state, uint64_t i) {
    double u1 = unit_open0(draw(state, 2 * i));
    double u2 = unit_closed0(draw(state, 2 * i + 1));
    return sqrt(-2.0 * log(u1)) * cos(6.283185307179586476925 * u2);
}

/* out[i] = bf16(mean + std * N_i) for i in [0, n); element i is the (offset+i)-th of the stream */
void synth_normal_bf16(uint64_t seed, const char *name, double mean, double std,
                       uint64_t offset, uint16_t *out, int64_t n) {
    uint64_t st = stream_state(seed, name);
#pragma omp parallel for schedule(static, 65536)
    for (int64_t i = 0; i < n; ++i)
        out[i] = f32_to_bf16_rne((float)(mean + std * normal_at(st, offset + (uint64_t)i)));
}

/* out[i] = mean + std * N_i as float32 */
void synth_normal_f32(uint64_t seed, const char *name, double mean, double std,
                      uint64_t offset, float *out, int64_t n) {
    uint64_t st = stream_state(seed, name);
#pragma omp parallel for schedule(static, 65536)
    for (int64_t i = 0; i < n; ++i)
        out[i] = (float)(mean + std * normal_at(st, offset + (uint64_t)i));
}

/* out[i] uniform integer in [-127, 127] */
void synth_uniform_i8(uint64_t seed, const char *name, uint64_t offset, int8_t *out, int64_t n) {
    uint64_t st = stream_state(seed, name);
#pragma omp parallel for schedule(static, 65536)
    for (int64_t i = 0; i < n; ++i) {
        uint64_t r = draw(st, offset + (uint64_t)i) >> 32;
        out[i] = (int8_t)((int)((r * 255u) >> 32) - 127);
    }
}

/* n 4-bit codes, each uniform in [1, 15] (the values -7..7 around the zero
 * point 8), packed two per byte: code 2j in the low nibble of out[j], code
 * 2j + 1 in the high nibble (n even) */
void synth_uniform_u4(uint64_t seed, const char *name, uint64_t offset, uint8_t *out, int64_t n) {
    uint64_t st = stream_state(seed, name);
#pragma omp parallel for schedule(static, 65536)
    for (int64_t j = 0; j < n / 2; ++j) {
        uint8_t c[2];
        for (int h = 0; h < 2; ++h) {
            uint64_t r = draw(st, offset + (uint64_t)(2 * j + h)) >> 32;
            c[h] = (uint8_t)(1 + ((r * 15u) >> 32));
        }
        out[j] = (uint8_t)(c[0] | (c[1] << 4));
    }
}

/* out[i] = base * (1 + jitter * U_i), U_i uniform in [0, 1) */
void synth_scales_f32(uint64_t seed, const char *name, double base, double jitter,
                      float *out, int64_t n) {
    uint64_t st = stream_state(seed, name);
    for (int64_t i = 0; i < n; ++i)
        out[i] = (float)(base * (1.0 + jitter * unit_closed0(draw(st, (uint64_t)i))));
}

/* raw draws, exposed for the generator's own statistical checks */
void synth_raw_u64(uint64_t seed, const char *name, uint64_t offset, uint64_t *out, int64_t n) {
    uint64_t st = stream_state(seed, name);
    for (int64_t i = 0; i < n; ++i) out[i] = draw(st, offset + (uint64_t)i);
}

/*
 * Prefilled KV cache, layout [L][Bmax][nkv][Smax][d] bf16 for K and for V.
 * Positions [0, ctx) of every (layer, batch row, kv head) hold N(0,1) draws;
 * positions >= ctx are zero.  Row (l, b, g) draws from stream
 * "kv.{K|V}" at offset ((l*Bmax + b)*nkv + g) * Smax * d, so for a fixed
 * cache shape the value at (l, b, g, pos, i) does not depend on ctx.
 */
void synth_kv_cache(uint64_t seed, int L, int Bmax, int nkv, int Smax, int d, int ctx,
                    uint16_t *kc, uint16_t *vc) {
    uint64_t sk = stream_state(seed, "kv.K");
    uint64_t sv = stream_state(seed, "kv.V");
    int64_t rows = (int64_t)L * Bmax * nkv;
    int64_t rowlen = (int64_t)Smax * d;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < rows; ++r) {
        uint64_t base = (uint64_t)(r * rowlen);
        for (int64_t e = 0; e < rowlen; ++e) {
            int64_t pos = e / d;
            uint16_t kv = 0, vv = 0;
            if (pos < ctx) {
                kv = f32_to_bf16_rne((float)normal_at(sk, base + (uint64_t)e));
                vv = f32_to_bf16_rne((float)normal_at(sv, base + (uint64_t)e));
            }
            kc[r * rowlen + e] = kv;
            vc[r * rowlen + e] = vv;
        }
    }
}

/* the plain splitmix64 sequence from a given state (known-answer checks) */
void synth_splitmix64_seq(uint64_t state, int64_t n, uint64_t *out) {
    for (int64_t i = 0; i < n; ++i) out[i] = draw(state, (uint64_t)i);
}
