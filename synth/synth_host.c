/*
 * synth_host.c - host entry points of the synthetic input generator.
 * Each function writes generated values for a contiguous range of a logical
 * tensor's elements (row-major logical index), rounded to the storage type.
 */
#include "synth.h"

uint64_t synth_host_key(uint64_t seed, uint32_t kind, uint32_t layer, uint32_t sub) {
  return synth_key(seed, kind, layer, sub);
}

/* out[i] = value of element idx0 + i, rounded to dtype, widened to fp32 */
void synth_host_fill_f32(float *out, uint64_t key, uint64_t idx0, int64_t n, float sigma,
                         int dtype) {
  for (int64_t i = 0; i < n; ++i) out[i] = synth_value(key, idx0 + (uint64_t)i, sigma, dtype);
}

/* out[i] = bf16 bit pattern of element idx0 + i */
void synth_host_fill_bf16(uint16_t *out, uint64_t key, uint64_t idx0, int64_t n, float sigma) {
  for (int64_t i = 0; i < n; ++i)
    out[i] = synth_f32_to_bf16(synth_normal_f32(key, idx0 + (uint64_t)i, sigma));
}

/* out[i] = Irwin-Hall(12) integer of element idx0 + i */
void synth_host_fill_ih12(int32_t *out, uint64_t key, uint64_t idx0, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = synth_ih12(key, idx0 + (uint64_t)i);
}

/* out[i] = uniform integer in [lo, lo + range) for element idx0 + i */
void synth_host_fill_uniform_int(int64_t *out, uint64_t key, uint64_t idx0, int64_t n, int64_t lo,
                                 uint32_t range) {
  for (int64_t i = 0; i < n; ++i) out[i] = synth_uniform_int(key, idx0 + (uint64_t)i, lo, range);
}

/* raw SplitMix64 words (for checks against the published sequence) */
void synth_host_words(uint64_t *out, uint64_t key, uint64_t n0, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = synth_word(key, n0 + (uint64_t)i);
}

uint16_t synth_host_f32_to_bf16(float f) { return synth_f32_to_bf16(f); }
