// pnb_noalloc.cu - split-KV decode attention for callers that cannot allocate.
//
// Some callers must not allocate GPU memory at all: code that runs inside an
// allocator-free region (a real-time or safety-certified loop that forbids
// cudaMalloc after start-up), a framework that owns every byte of device
// memory through its own pool and rejects foreign allocations, or a plugin
// loaded into a host process that only hands over input and output buffers.
// pnb_attention_decode_static serves them: the scratch that the attention
// kernel needs between its split CTAs (per-split max / sum / partial output,
// per-KV-head arrival counters and the kernel's I/O word) lives in one
// file-scope device array that every GPU holds from library load until exit.
#include <cuda_runtime.h>

#include <cmath>
#include <mutex>

#include "pnb.h"
#include "pnb_kernels.cuh"

using namespace pnb;

namespace {

// The static scratch: [I/O word: 256 B][counters: kMaxCounters x 4 B][partials].
constexpr size_t kScratchBytes = PNB_STATIC_SCRATCH_BYTES;
constexpr size_t kIoBytes = 256;
constexpr int kMaxCounters = 1024;
constexpr size_t kCountersBytes = kMaxCounters * 4;
constexpr size_t kPartialBytes = kScratchBytes - kIoBytes - kCountersBytes;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

// Device address of g_scratch per device, found once with that device current.
unsigned char *g_addr[kMaxDevices] = {};
std::mutex g_addr_mu;

int scratch_address(unsigned char **out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PNB_E_CUDA;
  std::lock_guard<std::mutex> lock(g_addr_mu);
  if (!g_addr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) return PNB_E_CUDA;
    g_addr[dev] = static_cast<unsigned char *>(p);
  }
  *out = g_addr[dev];
  return PNB_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" int pnb_attention_decode_static(const float *q_dev, const void *k_dev, const void *v_dev,
                                           int32_t dtype, int32_t n_head, int32_t n_kv_head,
                                           int32_t head_dim, int32_t cap, int32_t window,
                                           int32_t pos, float *out_dev, int32_t *err_dev,
                                           pnb_stream stream) {
  if (!q_dev || !k_dev || !v_dev || !out_dev) return PNB_E_NULL;
  if (!aligned16(q_dev) || !aligned16(k_dev) || !aligned16(v_dev) || !aligned16(out_dev) ||
      (reinterpret_cast<uintptr_t>(err_dev) & 3u))
    return PNB_E_ALIGN;
  if (dtype != PNB_F32 && dtype != PNB_BF16) return PNB_E_INVAL;
  if (head_dim != 32 && head_dim != 64 && head_dim != 128) return PNB_E_UNSUPPORTED;
  if (n_head <= 0 || n_kv_head <= 0 || n_head % n_kv_head || cap <= 0 || window < 0) return PNB_E_INVAL;
  if (pos < 0 || (window == 0 && pos >= cap) || (window > 0 && cap < window && pos >= cap))
    return PNB_E_INVAL;
  const int G = n_head / n_kv_head;
  const AttnGeom ag = attn_geom(dtype, head_dim, G);
  const int zgroups = G / ag.heads_per_cta;
  if (n_kv_head * zgroups > kMaxCounters) return PNB_E_TOO_LARGE;
  // split count: one wave of CTAs, limited by the cache length and by what the
  // static partial store holds
  int num_sms = 0, dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return PNB_E_CUDA;
  const size_t per_split = (size_t)n_head * (head_dim + 2) * 4;
  if (per_split > kPartialBytes) return PNB_E_TOO_LARGE;
  int n_split = num_sms / (n_kv_head * zgroups);
  n_split = n_split < 1 ? 1 : n_split;
  n_split = n_split < cap / 16 ? n_split : (cap / 16 > 1 ? cap / 16 : 1);
  const int fit = (int)(kPartialBytes / per_split);
  n_split = n_split < fit ? n_split : fit;

  unsigned char *base = nullptr;
  int rc = scratch_address(&base);
  if (rc != PNB_OK) return rc;
  if (prepare_attn_kernel(dtype, head_dim, ag) != cudaSuccess) return PNB_E_CUDA;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  StepIO *io = reinterpret_cast<StepIO *>(base);
  // the I/O word and the arrival counters start at zero on every call
  if (cudaMemsetAsync(base, 0, kIoBytes + kCountersBytes, st) != cudaSuccess) return PNB_E_CUDA;
  if (launch_set_pos(io, pos, st) != cudaSuccess) return PNB_E_CUDA;
  AttnArgs a{};
  a.q = q_dev;
  a.k_cache = k_dev;
  a.v_cache = v_dev;
  a.n_head = n_head;
  a.n_kv = n_kv_head;
  a.cap = cap;
  a.window = window;
  a.n_split = n_split;
  a.part = reinterpret_cast<float *>(base + kIoBytes + kCountersBytes);
  a.counter = reinterpret_cast<unsigned *>(base + kIoBytes);
  a.out = out_dev;
  a.qscale = (float)(1.4426950408889634 / std::sqrt((double)head_dim));
  a.stage_pos = ag.stage_pos;
  a.nstages = ag.nstages;
  a.io = io;
  if (launch_attn(dtype, head_dim, a, ag, st, false) != cudaSuccess) return PNB_E_CUDA;
  // the kernel's error bits leave the shared array before another call can
  // clear them (a device-to-device copy: no allocation)
  if (err_dev && cudaMemcpyAsync(err_dev, &io->error, sizeof(int32_t), cudaMemcpyDeviceToDevice,
                                 st) != cudaSuccess)
    return PNB_E_CUDA;
  return PNB_OK;
}
