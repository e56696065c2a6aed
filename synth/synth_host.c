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

/* Q8 rows [row0, row0 + nrows) of a [.][cols] matrix (cols a multiple of 32):
   the library's row layout (cols int8 values, then cols / 32 fp16 scales)
   into out_rows (nrows * synth_q8_row_bytes(cols) bytes), and, if out_f32 is
   given, the weights float(d) * q as fp32 */
void synth_host_fill_q8_rows(uint8_t *out_rows, float *out_f32, uint64_t key, int64_t row0,
                             int64_t nrows, int64_t cols, float sigma) {
  const int64_t rb = synth_q8_row_bytes(cols), nb = cols / SYNTH_Q8_BLOCK;
  for (int64_t r = 0; r < nrows; ++r)
    for (int64_t b = 0; b < nb; ++b) {
      int8_t q[SYNTH_Q8_BLOCK];
      uint16_t d;
      synth_q8_block(key, (uint64_t)((row0 + r) * cols + b * SYNTH_Q8_BLOCK), sigma, q, &d);
      if (out_rows) {
        uint8_t *row = out_rows + r * rb;
        for (int j = 0; j < SYNTH_Q8_BLOCK; ++j) row[b * SYNTH_Q8_BLOCK + j] = (uint8_t)q[j];
        memcpy(row + cols + 2 * b, &d, 2);
      }
      if (out_f32) {
        const float df = synth_f16_to_f32(d);
        for (int j = 0; j < SYNTH_Q8_BLOCK; ++j) out_f32[r * cols + b * SYNTH_Q8_BLOCK + j] = df * (float)q[j];
      }
    }
}

/* Q4 rows [row0, row0 + nrows) of a [.][cols] matrix (cols a multiple of 32):
   the library's row layout (cols / 2 bytes of 4-bit codes, two per byte,
   then cols / 32 fp16 scales) into out_rows (nrows * synth_q4_row_bytes(cols)
   bytes), and, if out_f32 is given, the weights float(d) * (u - 8) as fp32 */
void synth_host_fill_q4_rows(uint8_t *out_rows, float *out_f32, uint64_t key, int64_t row0,
                             int64_t nrows, int64_t cols, float sigma) {
  const int64_t rb = synth_q4_row_bytes(cols), nb = cols / SYNTH_Q4_BLOCK;
  for (int64_t r = 0; r < nrows; ++r)
    for (int64_t b = 0; b < nb; ++b) {
      uint8_t u[SYNTH_Q4_BLOCK];
      uint16_t d;
      synth_q4_block(key, (uint64_t)((row0 + r) * cols + b * SYNTH_Q4_BLOCK), sigma, u, &d);
      if (out_rows) {
        uint8_t *row = out_rows + r * rb;
        for (int j = 0; j < SYNTH_Q4_BLOCK; j += 2)
          row[(b * SYNTH_Q4_BLOCK + j) / 2] = (uint8_t)(u[j] | (u[j + 1] << 4));
        memcpy(row + cols / 2 + 2 * b, &d, 2);
      }
      if (out_f32) {
        const float df = synth_f16_to_f32(d);
        for (int j = 0; j < SYNTH_Q4_BLOCK; ++j)
          out_f32[r * cols + b * SYNTH_Q4_BLOCK + j] = df * (float)((int)u[j] - 8);
      }
    }
}

uint16_t synth_host_f32_to_f16(float f) { return synth_f32_to_f16(f); }
float synth_host_f16_to_f32(uint16_t h) { return synth_f16_to_f32(h); }
