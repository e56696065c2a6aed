// pnb_device.cuh - sm_103a building blocks of the decode-step kernels:
// mbarrier / bulk-copy (TMA) / programmatic-dependent-launch wrappers in
// inline PTX, bounded waits, bf16 unpacking and warp reductions.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace pnb {

// ------------------------------------------------------------------ limits
// weight-streaming (GEMV) kernels: 16 compute warps + one producer warp
constexpr int kGemvWarps = 16;
constexpr int kGemvConsumers = kGemvWarps * 32;
constexpr int kGemvThreads = kGemvConsumers + 32;
// attention kernel: 8 compute warps + one producer warp
constexpr int kAttnWarps = 8;
constexpr int kAttnConsumers = kAttnWarps * 32;
constexpr int kAttnThreads = kAttnConsumers + 32;
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

// Same, backing off between polls: for the single producer thread, whose
// polling would otherwise take issue slots from the compute warps.
__device__ __forceinline__ bool mbar_wait_backoff(uint64_t *bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  for (uint32_t it = 1;; ++it) {
    __nanosleep(64);
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 255u) == 0u) {
      if (global_ns() - t0 > kWaitLimitNs || it > (1u << 24)) return false;
    }
  }
}

// Wait for the phase with the given parity to complete; gives up after about
// limit_ns (or 2^26 polls) and returns false.
__device__ __forceinline__ bool mbar_wait_for(uint64_t *bar, uint32_t parity,
                                              unsigned long long limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 255u) == 0u) {
      if (global_ns() - t0 > limit_ns || it > (1u << 26)) return false;
    }
  }
}

// The kernels' bounded wait: gives up after about kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity) {
  return mbar_wait_for(bar, parity, kWaitLimitNs);
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

// hint: bring [src, src + bytes) into L2 (no completion tracking)
__device__ __forceinline__ void bulk_prefetch_l2(const void *src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// -------------------------------------------- programmatic dependent launch
// wait until the preceding kernel in the stream has completed and its writes
// are visible (no-op when launched without the PDL attribute)
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// allow the next kernel in the stream to be scheduled
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// named barrier among the N consumer threads only (id 1; id 0 is __syncthreads)
template <int N>
__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(N) : "memory");
}

// d = a * b + c on packed pairs of fp32 (one instruction for two FMAs)
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  unsigned long long d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;"
      : "=l"(d)
      : "l"(*reinterpret_cast<unsigned long long *>(&a)),
        "l"(*reinterpret_cast<unsigned long long *>(&b)),
        "l"(*reinterpret_cast<unsigned long long *>(&c)));
  return *reinterpret_cast<float2 *>(&d);
}

// the two bf16 of a 32-bit word as an fp32 pair (low half first), exact
__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
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

// N consecutive elements at p (4-, 8- or 16-byte aligned as their size) as fp32
template <typename T, int N>
__device__ __forceinline__ void load_vals(const T *p, float (&f)[N]) {
  if constexpr (sizeof(T) == 2) {
    if constexpr (N == 8) {
      const uint4 u = *reinterpret_cast<const uint4 *>(p);
      f[0] = bf16lo(u.x); f[1] = bf16hi(u.x); f[2] = bf16lo(u.y); f[3] = bf16hi(u.y);
      f[4] = bf16lo(u.z); f[5] = bf16hi(u.z); f[6] = bf16lo(u.w); f[7] = bf16hi(u.w);
    } else if constexpr (N == 4) {
      const uint2 u = *reinterpret_cast<const uint2 *>(p);
      f[0] = bf16lo(u.x); f[1] = bf16hi(u.x); f[2] = bf16lo(u.y); f[3] = bf16hi(u.y);
    } else if constexpr (N == 2) {
      const uint32_t u = *reinterpret_cast<const uint32_t *>(p);
      f[0] = bf16lo(u); f[1] = bf16hi(u);
    } else {
      f[0] = __uint_as_float((uint32_t)(*reinterpret_cast<const uint16_t *>(p)) << 16);
    }
  } else {
    if constexpr (N == 4) {
      const float4 u = *reinterpret_cast<const float4 *>(p);
      f[0] = u.x; f[1] = u.y; f[2] = u.z; f[3] = u.w;
    } else if constexpr (N == 2) {
      const float2 u = *reinterpret_cast<const float2 *>(p);
      f[0] = u.x; f[1] = u.y;
    } else {
      f[0] = *p;
    }
  }
}

// fp32 -> storage type -> fp32 (round to nearest even for bf16)
template <typename T>
__device__ __forceinline__ float round_to(float v) {
  if constexpr (sizeof(T) == 2) return __bfloat162float(__float2bfloat16_rn(v));
  else return v;
}

// Tag type of Q8 weight rows: K int8 values, then K / 32 fp16 scales (one per
// block of 32 consecutive values); weight k = scale[k / 32] * value[k].
struct Q8 {};

// Tag type of Q4 weight rows: K / 2 bytes of 4-bit codes (byte j holds code
// 2j in its low and code 2j + 1 in its high nibble), then K / 32 fp16 scales;
// weight k = scale[k / 32] * (code[k] - 8).
struct Q4 {};

// KV-cache element type of a model with weights of type T (bf16 for Q8, Q4)
template <typename T>
struct KvOf {
  using type = T;
};
template <>
struct KvOf<Q8> {
  using type = __nv_bfloat16;
};
template <>
struct KvOf<Q4> {
  using type = __nv_bfloat16;
};

// The state's device I/O block: next input token, position, error bits.
struct StepIO {
  int32_t token;
  int32_t pos;
  int32_t error;
  uint32_t draws;  // sampler draws taken by this sequence (picks its uniform)
};

__device__ __forceinline__ void set_error(int32_t *err, int bits) { atomicOr(err, bits); }

}  // namespace pnb
