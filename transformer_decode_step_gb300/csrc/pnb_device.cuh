// pnb_device.cuh - sm_103a building blocks of the decode-step kernels:
// mbarrier / bulk-copy (TMA) / programmatic-dependent-launch wrappers in
// inline PTX, bounded waits, bf16 unpacking and warp reductions.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace pnb {

// ------------------------------------------------------------------ limits
constexpr int kConsumerWarps = 8;                        // compute warps per CTA
constexpr int kThreads = (kConsumerWarps + 1) * 32;      // + one producer warp
constexpr int kConsumerThreads = kConsumerWarps * 32;
constexpr int kMaxSegments = 8;                          // matrices in one GEMV launch
constexpr unsigned long long kWaitLimitNs = 1000000000ull;  // bounded waits: 1 s

// device-side error bits (mirror of PNB_DEV_ERR_*)
constexpr int kErrToken = 1;
constexpr int kErrTimeout = 2;

// -------------------------------------------------------------- shared mem
__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

// make barrier initialisation visible to the async (bulk-copy) proxy
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Wait for the phase with the given parity to complete; gives up after about
// kWaitLimitNs (or 2^26 polls) and returns false.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 255u) == 0u) {
      if (global_ns() - t0 > kWaitLimitNs || it > (1u << 26)) return false;
    }
  }
}

// 1-D bulk copy global -> shared, completion counted on an mbarrier (TMA).
// dst, src and bytes must be multiples of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes,
                                         uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// -------------------------------------------- programmatic dependent launch
// wait until the preceding kernel in the stream has completed and its writes
// are visible (no-op when launched without the PDL attribute)
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// allow the next kernel in the stream to be scheduled
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// named barrier among the consumer warps only (id 1; id 0 is __syncthreads)
__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumerThreads) : "memory");
}

// ------------------------------------------------------------ arithmetic
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// two bf16 packed in a 32-bit word -> two floats (exact)
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Shared-memory layout of an fp32 activation vector read by 16-byte weight
// vectors: four padding floats after every 32 floats keep the 32-byte x
// chunks of eight consecutive lanes on distinct banks.
__device__ __forceinline__ int xpad(int i) { return i + ((i >> 5) << 2); }
__host__ __device__ constexpr int xpad_size(int n) { return n + ((n + 31) / 32) * 4; }

// storage of one element
template <typename T>
struct Elem;
template <>
struct Elem<float> {
  static constexpr int kBytes = 4;
  __device__ static float load(const float *p, int64_t i) { return p[i]; }
  __device__ static void store(float *p, int64_t i, float v) { p[i] = v; }
};
template <>
struct Elem<__nv_bfloat16> {
  static constexpr int kBytes = 2;
  __device__ static float load(const __nv_bfloat16 *p, int64_t i) { return __bfloat162float(p[i]); }
  __device__ static void store(__nv_bfloat16 *p, int64_t i, float v) {
    p[i] = __float2bfloat16_rn(v);
  }
};

// The state's device I/O block: next input token, position, error bits.
struct StepIO {
  int32_t token;
  int32_t pos;
  int32_t error;
  int32_t pad;
};

__device__ __forceinline__ void set_error(int32_t *err, int bits) { atomicOr(err, bits); }

}  // namespace pnb
