/*
 * Seeded synthetic inputs: model weights, prompt ids, sampling uniforms, KV prefixes.
 *
 * This file holds no arithmetic of the decode step. It only draws the numbers
 * that both the CUDA engine and the CPU oracle then consume byte for byte.
 *
 * Generator: counter-based splitmix64 (Steele, Lea & Flood, "Fast splittable
 * pseudorandom number generators", OOPSLA 2014; finaliser constants of
 * Vigna's public-domain splitmix64.c). Stream value i of key k is
 * mix(k + (i + 1) * GOLDEN). Normal deviates use the Box-Muller transform
 * (Box & Muller 1958): values 2n and 2n+1 of the stream give the pair
 * (r cos 2πu2, r sin 2πu2), r = sqrt(-2 ln u1).
 *
 * Storage rounding: fp32 draw -> round-to-nearest-even to fp16 / bf16, or
 * per-output-row scaled e4m3 (OCP FP8 E4M3 "fn": bias 7, no infinities,
 * S.1111.111 = NaN, largest finite 448), saturating at 448.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#include <stddef.h>

#define GOLDEN 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

uint64_t synth_key(uint64_t seed, uint64_t tensor_id) { return mix64(seed ^ mix64(tensor_id + GOLDEN)); }

static inline uint64_t stream(uint64_t key, uint64_t i) { return mix64(key + (i + 1) * GOLDEN); }

/* Element i of the standard-normal stream of key. */
static inline double normal_at(uint64_t key, uint64_t i) {
  uint64_t n = i >> 1;
  double u1 = ((double)(stream(key, 2 * n) >> 11) + 1.0) * 0x1.0p-53; /* (0, 1] */
  double u2 = (double)(stream(key, 2 * n + 1) >> 11) * 0x1.0p-53;    /* [0, 1) */
  double r = sqrt(-2.0 * log(u1));
  double a = 6.283185307179586476925286766559 * u2;
  return (i & 1) ? r * sin(a) : r * cos(a);
}

static inline float draw(uint64_t key, uint64_t i, float stdv) { return (float)((double)stdv * normal_at(key, i)); }

/* fp32 -> IEEE binary16, round to nearest even (generator-side storage rounding). */
static inline uint16_t to_f16(float f) {
  uint32_t x; memcpy(&x, &f, 4);
  uint32_t sign = (x >> 16) & 0x8000u;
  uint32_t ax = x & 0x7FFFFFFFu;
  if (ax > 0x7F800000u) return (uint16_t)(sign | 0x7E00u);        /* NaN */
  if (ax >= 0x477FF000u) return (uint16_t)(sign | 0x7C00u);       /* rounds to >= 65520 -> inf */
  if (ax < 0x38800000u) {                                         /* below 2^-14: subnormal half */
    /* value = ax as float; half subnormal unit = 2^-24 */
    float a; memcpy(&a, &ax, 4);
    double q = (double)a * 16777216.0; /* exact: a * 2^24 */
    double r = nearbyint(q);           /* ties-to-even under the default rounding mode */
    return (uint16_t)(sign | (uint32_t)r);
  }
  uint32_t e = (ax >> 23) - 112u;   /* rebias 127 -> 15 */
  uint32_t m = ax & 0x7FFFFFu;
  uint32_t h = (e << 10) | (m >> 13);
  uint32_t rem = m & 0x1FFFu;
  if (rem > 0x1000u || (rem == 0x1000u && (h & 1u))) h += 1u;     /* carry may bump the exponent: correct */
  return (uint16_t)(sign | h);
}

static inline uint16_t to_bf16(float f) {
  uint32_t x; memcpy(&x, &f, 4);
  if ((x & 0x7FFFFFFFu) > 0x7F800000u) return (uint16_t)((x >> 16) | 0x40u);
  uint32_t lsb = (x >> 16) & 1u;
  return (uint16_t)((x + 0x7FFFu + lsb) >> 16);
}

/* e4m3fn encode with round-to-nearest-even and saturation to +-448. */
static inline uint8_t to_e4m3(float f) {
  uint8_t sign = (f < 0.0f || (f == 0.0f && signbit(f))) ? 0x80 : 0x00;
  double a = fabs((double)f);
  if (isnan(f)) return 0x7F;
  if (a >= 448.0) return (uint8_t)(sign | 0x7E);
  if (a < 0x1.0p-6) {                                  /* subnormal range, unit 2^-9 */
    double q = nearbyint(a * 512.0);                   /* 0..8; 8 is the smallest normal's code */
    return (uint8_t)(sign | (uint8_t)q);
  }
  int e; double fr = frexp(a, &e);                     /* a = fr * 2^e, fr in [0.5, 1) */
  e -= 1;                                              /* a = (2 fr) * 2^e, 2 fr in [1, 2) */
  double m = nearbyint((2.0 * fr - 1.0) * 8.0);        /* 0..8 */
  if (m >= 8.0) { m = 0.0; e += 1; }
  int code = ((e + 7) << 3) | (int)m;
  if (code > 0x7E) code = 0x7E;
  return (uint8_t)(sign | code);
}

void synth_normal_f32(uint64_t seed, uint64_t tensor_id, float stdv, float* out, size_t n) {
  uint64_t key = synth_key(seed, tensor_id);
#pragma omp parallel for schedule(static)
  for (long long i = 0; i < (long long)n; ++i) out[i] = draw(key, (uint64_t)i, stdv);
}

void synth_normal_f16(uint64_t seed, uint64_t tensor_id, float stdv, uint16_t* out, size_t n) {
  uint64_t key = synth_key(seed, tensor_id);
#pragma omp parallel for schedule(static)
  for (long long i = 0; i < (long long)n; ++i) out[i] = to_f16(draw(key, (uint64_t)i, stdv));
}

void synth_normal_bf16(uint64_t seed, uint64_t tensor_id, float stdv, uint16_t* out, size_t n) {
  uint64_t key = synth_key(seed, tensor_id);
#pragma omp parallel for schedule(static)
  for (long long i = 0; i < (long long)n; ++i) out[i] = to_bf16(draw(key, (uint64_t)i, stdv));
}

/* Row-scaled e4m3: for each of `rows` rows of `cols` fp32 draws w,
 * s = max|w| / 448 and q = e4m3(w / s) (the division in fp32). A row of zeros gets s = 1. */
void synth_normal_e4m3_rows(uint64_t seed, uint64_t tensor_id, float stdv, size_t rows, size_t cols,
                            uint8_t* q, float* scales) {
  uint64_t key = synth_key(seed, tensor_id);
#pragma omp parallel for schedule(static)
  for (long long r = 0; r < (long long)rows; ++r) {
    float amax = 0.0f;
    for (size_t c = 0; c < cols; ++c) {
      float w = draw(key, (uint64_t)r * cols + c, stdv);
      float aw = fabsf(w);
      if (aw > amax) amax = aw;
    }
    float s = amax > 0.0f ? amax / 448.0f : 1.0f;
    scales[r] = s;
    for (size_t c = 0; c < cols; ++c) {
      float w = draw(key, (uint64_t)r * cols + c, stdv);
      q[(size_t)r * cols + c] = to_e4m3(w / s);
    }
  }
}

void synth_f32_to_f16(const float* in, uint16_t* out, size_t n) {
  for (size_t i = 0; i < n; ++i) out[i] = to_f16(in[i]);
}
void synth_f32_to_bf16(const float* in, uint16_t* out, size_t n) {
  for (size_t i = 0; i < n; ++i) out[i] = to_bf16(in[i]);
}
void synth_f32_to_e4m3(const float* in, uint8_t* out, size_t n) {
  for (size_t i = 0; i < n; ++i) out[i] = to_e4m3(in[i]);
}

/* Uniform token ids in [0, vocab): id_i = floor(hi32(stream_i) * vocab / 2^32). */
void synth_tokens(uint64_t seed, uint64_t stream_id, uint32_t vocab, int32_t* out, size_t n) {
  uint64_t key = synth_key(seed, stream_id);
  for (size_t i = 0; i < n; ++i) out[i] = (int32_t)(((stream(key, i) >> 32) * (uint64_t)vocab) >> 32);
}

/* Sampling uniforms in [0, 1) with 24 random bits: u_n = (mix(seed ^ n) >> 40) * 2^-24. */
void synth_uniforms(uint64_t seed, uint64_t first, float* out, size_t n) {
  for (size_t i = 0; i < n; ++i) out[i] = (float)((double)(mix64(seed ^ (first + i)) >> 40) * 0x1.0p-24);
}
