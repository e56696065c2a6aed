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

#include <math.h>
#include <stdint.h>
#include <string.h>

#if defined(__CUDACC__)
#define SYNTH_FN static __host__ __device__ __forceinline__
#else
#define SYNTH_FN static inline
#endif

#define SYNTH_GAMMA 0x9E3779B97F4A7C15ULL

/* storage types of generated values (SYNTH_Q8, SYNTH_Q4: weight matrices
   only, in blocks of 32 along a row; see synth_q8_block, synth_q4_block) */
enum { SYNTH_F32 = 0, SYNTH_BF16 = 1, SYNTH_Q8 = 2, SYNTH_Q4 = 3 };

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

/* fp32 -> IEEE binary16 bit pattern, round to nearest even, for finite
   non-negative inputs below 65520 (normal and subnormal results) */
SYNTH_FN uint16_t synth_f32_to_f16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  const int e = (int)(u >> 23) - 127 + 15;    /* biased binary16 exponent */
  const uint32_t m = (u & 0x7FFFFFu) | (e > -64 ? 0x800000u : 0u);
  if ((u & 0x7FFFFFFFu) == 0u) return 0;
  if (e >= 1) {                                /* normal: drop 13 mantissa bits */
    uint32_t h = ((uint32_t)e << 10) | ((u & 0x7FFFFFu) >> 13);
    const uint32_t rem = u & 0x1FFFu;
    if (rem > 0x1000u || (rem == 0x1000u && (h & 1u))) ++h;
    return (uint16_t)h;
  }
  const int sh = 14 - e;                       /* subnormal: value = m * 2^(e - 15 - 23 + 1) */
  if (sh > 24) return 0;
  uint32_t h = m >> sh;
  const uint32_t rem = m & ((1u << sh) - 1u), half = 1u << (sh - 1);
  if (rem > half || (rem == half && (h & 1u))) ++h;
  return (uint16_t)h;
}

/* IEEE binary16 bit pattern (finite, non-negative) -> fp32, exact */
SYNTH_FN float synth_f16_to_f32(uint16_t h) {
  const uint32_t e = (h >> 10) & 0x1Fu, m = h & 0x3FFu;
  uint32_t u;
  if (e == 0) {
    if (m == 0) return 0.0f;
    return (float)m * (1.0f / 16777216.0f);   /* m * 2^-24, exact */
  }
  u = ((e - 15u + 127u) << 23) | (m << 13);
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* Q8 weights, in blocks of 32 consecutive elements of a row (element indices
   idx0 .. idx0 + 31, idx0 a multiple of 32): w_i are the generated fp32
   values; the block's scale is d = fp16(max_i |w_i| / 127) (one fp32
   division, one rounding to fp16, nearest even); q_i = w_i / float(d)
   rounded to the nearest integer (ties to even, rintf) and clamped to
   [-127, 127], or 0 when d is 0.  The element's weight is float(d) * q_i,
   exact in fp32. */
#define SYNTH_Q8_BLOCK 32
SYNTH_FN void synth_q8_block(uint64_t key, uint64_t idx0, float sigma, int8_t *q, uint16_t *d_out) {
  float w[SYNTH_Q8_BLOCK];
  float amax = 0.0f;
  for (int i = 0; i < SYNTH_Q8_BLOCK; ++i) {
    w[i] = synth_normal_f32(key, idx0 + (uint64_t)i, sigma);
    const float a = w[i] < 0.0f ? -w[i] : w[i];
    if (a > amax) amax = a;
  }
  const uint16_t d = synth_f32_to_f16(amax / 127.0f);
  const float df = synth_f16_to_f32(d);
  for (int i = 0; i < SYNTH_Q8_BLOCK; ++i) {
    float r = df > 0.0f ? rintf(w[i] / df) : 0.0f;
    if (r > 127.0f) r = 127.0f;
    if (r < -127.0f) r = -127.0f;
    q[i] = (int8_t)r;
  }
  *d_out = d;
}

/* bytes of one Q8 row of `cols` weights: the int8 values, then one fp16
   scale per 32 (the layout of the decode-step library's Q8 matrices) */
SYNTH_FN int64_t synth_q8_row_bytes(int64_t cols) { return cols + cols / 16; }

/* Q4 weights, in blocks of 32 consecutive elements of a row (element indices
   idx0 .. idx0 + 31, idx0 a multiple of 32): w_i are the generated fp32
   values; the block's scale is d = fp16(max_i |w_i| / 7) (one fp32 division,
   one rounding to fp16, nearest even); the 4-bit code of element i is
   u_i = clamp(rint(w_i / float(d)), -8, 7) + 8 in [0, 15] (ties to even; all
   8 when d is 0).  The element's weight is float(d) * (u_i - 8), exact in
   fp32 (the GGUF Q4_0 block: 32 codes and one fp16 scale). */
#define SYNTH_Q4_BLOCK 32
SYNTH_FN void synth_q4_block(uint64_t key, uint64_t idx0, float sigma, uint8_t *u, uint16_t *d_out) {
  float w[SYNTH_Q4_BLOCK];
  float amax = 0.0f;
  for (int i = 0; i < SYNTH_Q4_BLOCK; ++i) {
    w[i] = synth_normal_f32(key, idx0 + (uint64_t)i, sigma);
    const float a = w[i] < 0.0f ? -w[i] : w[i];
    if (a > amax) amax = a;
  }
  const uint16_t d = synth_f32_to_f16(amax / 7.0f);
  const float df = synth_f16_to_f32(d);
  for (int i = 0; i < SYNTH_Q4_BLOCK; ++i) {
    float r = df > 0.0f ? rintf(w[i] / df) : 0.0f;
    if (r > 7.0f) r = 7.0f;
    if (r < -8.0f) r = -8.0f;
    u[i] = (uint8_t)((int)r + 8);
  }
  *d_out = d;
}

/* bytes of one Q4 row of `cols` weights: the 4-bit codes, two per byte
   (byte j holds element 2j in its low and element 2j + 1 in its high
   nibble), then one fp16 scale per 32 (the layout of the decode-step
   library's Q4 matrices) */
SYNTH_FN int64_t synth_q4_row_bytes(int64_t cols) { return cols / 2 + cols / 16; }

/* uniform integer in [lo, lo + n) for element idx (multiply-shift on 32 high bits) */
SYNTH_FN int64_t synth_uniform_int(uint64_t key, uint64_t idx, int64_t lo, uint32_t n) {
  uint64_t hi = synth_word(key, idx) >> 32;
  return lo + (int64_t)((hi * (uint64_t)n) >> 32);
}

#endif /* SYNTH_H */
