/*
 * synth_cuda.cu - device fill kernels of the synthetic input generator.
 *
 * They write generated values straight into the decode-step library's device
 * layouts, so multi-GB weight sets never cross the host link.  Every value
 * equals the host generator's value for the same logical element.
 * C ABI; all sizes in elements; return 0 or the CUDA error code.
 */
#include <cuda_runtime.h>
#include <stdint.h>

#include "synth.h"

namespace {

__device__ __forceinline__ void store_value(void *dst, int dtype, int64_t off, float v) {
  if (dtype == SYNTH_BF16)
    static_cast<uint16_t *>(dst)[off] = synth_f32_to_bf16(v);
  else
    static_cast<float *>(dst)[off] = v;
}

/* logical row r of a [rows][cols] tensor goes to device row dst_row0 + r*dst_row_step */
__global__ void fill_matrix_kernel(void *dst, int dtype, int64_t dst_row0, int64_t dst_row_step,
                                   int64_t rows, int64_t cols, uint64_t key, float sigma) {
  const int64_t n = rows * cols;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / cols, c = i - r * cols;
    const float v = synth_normal_f32(key, (uint64_t)i, sigma);
    store_value(dst, dtype, (dst_row0 + r * dst_row_step) * cols + c, v);
  }
}

/* Q8: one thread per 32-element block; logical row r goes to device row
   dst_row0 + r*dst_row_step of synth_q8_row_bytes(cols) bytes */
__global__ void fill_q8_kernel(uint8_t *dst, int64_t dst_row0, int64_t dst_row_step, int64_t rows,
                               int64_t cols, uint64_t key, float sigma) {
  const int64_t nb = cols / SYNTH_Q8_BLOCK, n = rows * nb;
  const int64_t rb = synth_q8_row_bytes(cols);
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / nb, b = i - r * nb;
    int8_t q[SYNTH_Q8_BLOCK];
    uint16_t d;
    synth_q8_block(key, (uint64_t)(r * cols + b * SYNTH_Q8_BLOCK), sigma, q, &d);
    uint8_t *row = dst + (dst_row0 + r * dst_row_step) * rb;
    for (int j = 0; j < SYNTH_Q8_BLOCK; ++j) row[b * SYNTH_Q8_BLOCK + j] = (uint8_t)q[j];
    reinterpret_cast<uint16_t *>(row + cols)[b] = d;
  }
}

/* Q4: one thread per 32-element block; logical row r goes to device row
   dst_row0 + r*dst_row_step of synth_q4_row_bytes(cols) bytes */
__global__ void fill_q4_kernel(uint8_t *dst, int64_t dst_row0, int64_t dst_row_step, int64_t rows,
                               int64_t cols, uint64_t key, float sigma) {
  const int64_t nb = cols / SYNTH_Q4_BLOCK, n = rows * nb;
  const int64_t rb = synth_q4_row_bytes(cols);
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / nb, b = i - r * nb;
    uint8_t u[SYNTH_Q4_BLOCK];
    uint16_t d;
    synth_q4_block(key, (uint64_t)(r * cols + b * SYNTH_Q4_BLOCK), sigma, u, &d);
    uint8_t *row = dst + (dst_row0 + r * dst_row_step) * rb;
    for (int j = 0; j < SYNTH_Q4_BLOCK; j += 2)
      row[(b * SYNTH_Q4_BLOCK + j) / 2] = (uint8_t)(u[j] | (u[j + 1] << 4));
    reinterpret_cast<uint16_t *>(row + cols / 2)[b] = d;
  }
}

__global__ void fill_const_kernel(void *dst, int dtype, int64_t n, float value) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x)
    store_value(dst, dtype, i, value);
}

/* KV block [n_kv][cap][hd]; logical element (position j, head g, dim d) has index
   (j*n_kv + g)*hd + d and lives in slot j % cap */
__global__ void fill_kv_kernel(void *dst, int dtype, int n_kv, int64_t cap, int hd, int64_t j_lo,
                               int64_t j_hi, uint64_t key, float sigma) {
  const int64_t per_pos = (int64_t)n_kv * hd;
  const int64_t n = (j_hi - j_lo) * per_pos;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t j = j_lo + i / per_pos;
    const int64_t rem = i - (j - j_lo) * per_pos;
    const int64_t g = rem / hd, d = rem - g * hd;
    const uint64_t idx = (uint64_t)((j * n_kv + g) * hd + d);
    const float v = synth_normal_f32(key, idx, sigma);
    store_value(dst, dtype, (g * cap + (j % cap)) * hd + d, v);
  }
}

__global__ void fill_uniform_int_kernel(int32_t *dst, int64_t n, uint64_t key, uint64_t idx0,
                                        int64_t lo, uint32_t range) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x)
    dst[i] = (int32_t)synth_uniform_int(key, idx0 + (uint64_t)i, lo, range);
}

int grid_for(int64_t n) {
  int64_t g = (n + 255) / 256;
  if (g > 65536) g = 65536;
  if (g < 1) g = 1;
  return (int)g;
}

}  // namespace

extern "C" {

uint64_t synth_dev_key(uint64_t seed, uint32_t kind, uint32_t layer, uint32_t sub) {
  return synth_key(seed, kind, layer, sub);
}

int synth_dev_fill_matrix(void *dst, int dtype, int64_t dst_row0, int64_t dst_row_step,
                          int64_t rows, int64_t cols, uint64_t key, float sigma,
                          cudaStream_t stream) {
  if (rows <= 0 || cols <= 0) return 0;
  if (dtype == SYNTH_Q8) {
    if (cols % SYNTH_Q8_BLOCK) return (int)cudaErrorInvalidValue;
    fill_q8_kernel<<<grid_for(rows * (cols / SYNTH_Q8_BLOCK)), 256, 0, stream>>>(
        static_cast<uint8_t *>(dst), dst_row0, dst_row_step, rows, cols, key, sigma);
    return (int)cudaGetLastError();
  }
  if (dtype == SYNTH_Q4) {
    if (cols % SYNTH_Q4_BLOCK) return (int)cudaErrorInvalidValue;
    fill_q4_kernel<<<grid_for(rows * (cols / SYNTH_Q4_BLOCK)), 256, 0, stream>>>(
        static_cast<uint8_t *>(dst), dst_row0, dst_row_step, rows, cols, key, sigma);
    return (int)cudaGetLastError();
  }
  fill_matrix_kernel<<<grid_for(rows * cols), 256, 0, stream>>>(dst, dtype, dst_row0, dst_row_step,
                                                                rows, cols, key, sigma);
  return (int)cudaGetLastError();
}

int synth_dev_fill_const(void *dst, int dtype, int64_t n, float value, cudaStream_t stream) {
  if (n <= 0) return 0;
  fill_const_kernel<<<grid_for(n), 256, 0, stream>>>(dst, dtype, n, value);
  return (int)cudaGetLastError();
}

int synth_dev_fill_kv(void *dst, int dtype, int n_kv, int64_t cap, int hd, int64_t j_lo,
                      int64_t j_hi, uint64_t key, float sigma, cudaStream_t stream) {
  if (j_hi <= j_lo) return 0;
  if (cap <= 0 || j_hi - j_lo > cap) return (int)cudaErrorInvalidValue;
  fill_kv_kernel<<<grid_for((j_hi - j_lo) * n_kv * hd), 256, 0, stream>>>(dst, dtype, n_kv, cap, hd,
                                                                          j_lo, j_hi, key, sigma);
  return (int)cudaGetLastError();
}

int synth_dev_fill_uniform_int(int32_t *dst, int64_t n, uint64_t key, uint64_t idx0, int64_t lo,
                               uint32_t range, cudaStream_t stream) {
  if (n <= 0) return 0;
  fill_uniform_int_kernel<<<grid_for(n), 256, 0, stream>>>(dst, n, key, idx0, lo, range);
  return (int)cudaGetLastError();
}

}  // extern "C"
