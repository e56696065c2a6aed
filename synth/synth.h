/*
 * synth.h - seeded, counter-based synthetic input generator.
 *
 * This module produces every synthetic input of the decode-step workloads:
 * weights, pre-filled KV-cache contents, prompt tokens, start tokens and
 * per-slot start positions.  It holds none of the decode step's arithmetic.
 * The same inline functions compile for the host (C, the CPU oracle and its
 * tests) and for the GPU (CUDA fill kernels), so a value is a pure function
 * of (seed, tensor kind, layer, sub-index, element index) and is bitwise
 * identical on both sides.
 *
 * Definition (each step is exact integer arithmetic or one IEEE rounding):
 *  - word n of a stream with key K is the SplitMix64 output function applied
 *    to K + (n+1)*0x9E3779B97F4A7C15 (Steele, Lea & Flood, "Fast splittable
 *    pseudorandom number generators", OOPSLA 2014; constants as in Vigna's
 *    public-domain splitmix64.c);
 *  - the key of a logical tensor mixes the run seed with (kind, layer, sub);
 *  - an approximately standard-normal value for element i is the Irwin-Hall
 *    sum of twelve 16-bit uniforms taken from words 3i, 3i+1, 3i+2:
 *    n = S - 393210 (an exact integer, |n| <= 393210), z = n / 65536;
 *    z has mean 0 and standard deviation sqrt(1 - 2^-32);
 *  - a value with standard deviation sigma is the fp32 product
 *    (float(n) * 2^-16) * sigma (one round-to-nearest-even rounding);
 *  - bf16 storage rounds that fp32 value to nearest-even on its bit pattern.
 * No transcendental function is involved, so host and device agree bit for
 * bit without depending on either side's math library.
 */
#ifndef SYNTH_H
#define SYNTH_H

#include <stdint.h>
#include <string.h>

#if defined(__CUDACC__)
#define SYNTH_FN static __host__ __device__ __forceinline__
#else
#define SYNTH_FN static inline
#endif

#define SYNTH_GAMMA 0x9E3779B97F4A7C15ULL

/* storage types of generated values */
enum { SYNTH_F32 = 0, SYNTH_BF16 = 1 };

/* logical tensor kinds (part of a stream key) */
enum {
  SYNTH_TOK_EMBD = 1,
  SYNTH_ATTN_NORM = 2,
  SYNTH_WQ = 3,
  SYNTH_WK = 4,
  SYNTH_WV = 5,
  SYNTH_WO = 6,
  SYNTH_FFN_NORM = 7,
  SYNTH_WGATE = 8,
  SYNTH_WUP = 9,
  SYNTH_WDOWN = 10,
  SYNTH_WROUTER = 11,
  SYNTH_OUT_NORM = 12,
  SYNTH_OUTPUT = 13,
  SYNTH_KCACHE = 14,
  SYNTH_VCACHE = 15,
  SYNTH_TOKENS = 16,
  SYNTH_POSITIONS = 17
};

/* SplitMix64 output function */
SYNTH_FN uint64_t synth_mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

/* word n (n >= 0) of the SplitMix64 sequence whose state starts at key */
SYNTH_FN uint64_t synth_word(uint64_t key, uint64_t n) {
  return synth_mix64(key + (n + 1ULL) * SYNTH_GAMMA);
}

/* stream key of one logical tensor: kind < 2^16, sub < 2^24, layer < 2^24 */
SYNTH_FN uint64_t synth_key(uint64_t seed, uint32_t kind, uint32_t layer, uint32_t sub) {
  uint64_t k = synth_mix64(seed + SYNTH_GAMMA);
  uint64_t tag = ((uint64_t)(kind & 0xFFFFu) << 48) | ((uint64_t)(sub & 0xFFFFFFu) << 24) |
                 (uint64_t)(layer & 0xFFFFFFu);
  return synth_mix64(k ^ synth_mix64(tag + 0x632BE59BD9B4E019ULL));
}

/* Irwin-Hall(12) integer: sum of twelve 16-bit uniforms minus their mean */
SYNTH_FN int32_t synth_ih12(uint64_t key, uint64_t idx) {
  uint32_t s = 0;
  for (int r = 0; r < 3; ++r) {
    uint64_t w = synth_word(key, 3ULL * idx + (uint64_t)r);
    s += (uint32_t)(w & 0xFFFFu) + (uint32_t)((w >> 16) & 0xFFFFu) +
         (uint32_t)((w >> 32) & 0xFFFFu) + (uint32_t)(w >> 48);
  }
  return (int32_t)s - 393210;
}

/* approximately N(0, sigma^2) as an fp32 value */
SYNTH_FN float synth_normal_f32(uint64_t key, uint64_t idx, float sigma) {
  float z = (float)synth_ih12(key, idx) * (1.0f / 65536.0f);
  return z * sigma;
}

/* fp32 -> bf16 bit pattern, round to nearest even (inputs are finite) */
SYNTH_FN uint16_t synth_f32_to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

SYNTH_FN float synth_bf16_to_f32(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* the generated value after rounding to its storage type, as fp32 */
SYNTH_FN float synth_value(uint64_t key, uint64_t idx, float sigma, int dtype) {
  float v = synth_normal_f32(key, idx, sigma);
  return dtype == SYNTH_BF16 ? synth_bf16_to_f32(synth_f32_to_bf16(v)) : v;
}

/* uniform integer in [lo, lo + n) for element idx (multiply-shift on 32 high bits) */
SYNTH_FN int64_t synth_uniform_int(uint64_t key, uint64_t idx, int64_t lo, uint32_t n) {
  uint64_t hi = synth_word(key, idx) >> 32;
  return lo + (int64_t)((hi * (uint64_t)n) >> 32);
}

#endif /* SYNTH_H */
