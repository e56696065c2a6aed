// pnb_pattn.cu - attention of a prefill chunk on CUDA cores.
//
// A prefill chunk is n <= 64 consecutive prompt tokens of one sequence, run as
// n virtual slots of a batched step that share the state's KV cache (the
// chunk's QKV kernel has already stored the chunk's own keys and values).
// Token j at position p_j attends to the positions [max(0, p_j - W + 1), p_j]
// (all of [0, p_j] without a window).  The batched decode attention would
// read the cached prefix once per token; here one CTA takes a block of query
// rows - (token, query head) pairs of one KV head - and walks the positions
// once in tiles of kPTile:
//   * the tile's keys and values go to shared memory (fp32, rows padded by
//     four words, so that rows start in different banks and stay 16-byte
//     aligned for vector loads);
//   * each row's scores (q . k scaled by log2(e) / sqrt(hd)) update a running
//     max and sum in the log2 domain, as the decode kernels do, and the
//     row's output is rescaled and accumulated in registers;
// and the outputs are written as the bf16 high / low rows of the output
// projection's operand, like the batched attention kernels.
#include <cuda_bf16.h>
#include <math.h>

#include "pnb_kernels.cuh"

namespace pnb {
namespace {

constexpr int kPThreads = 256;
constexpr int kPRows = 16;     // query rows per CTA (16 threads per row)
constexpr int kPTile = 64;     // positions per tile

template <int HD>
__global__ void __launch_bounds__(kPThreads) k_pattn(const PAttnArgs a) {
  extern __shared__ float psm[];
  constexpr int LD = HD + 4;                   // padded row of a K / V tile
  constexpr int CPT = HD / 16;                 // output columns per thread (contiguous)
  float *qs = psm;                             // [kPRows][HD]
  float *ks = qs + kPRows * HD;                // [kPTile][LD]
  float *vs = ks + kPTile * LD;                // [kPTile][LD]
  float *ps = vs + kPTile * LD;                // [kPRows][kPTile]
  const int tid = threadIdx.x;
  const int g = blockIdx.x;                    // KV head
  const int G = a.n_head / a.n_kv;
  const int rows = a.n * G;                    // (token, head in group) rows of this KV head
  const int r0 = blockIdx.y * kPRows;
  const int row = tid >> 4, sub = tid & 15;    // 16 threads per row
  const int rg = r0 + row;
  const bool live = rg < rows;
  const int j = live ? rg / G : 0, hh = live ? rg - (rg / G) * G : 0;
  pdl_wait();
  pdl_trigger();
  const int pj = live ? a.pos[j] : -1;
  const int lo_j = a.window > 0 ? max(0, pj - a.window + 1) : 0;
  // the block's position range: the union of its rows' ranges
  const int last_row = min(rows, r0 + kPRows) - 1;
  const int p_hi = a.pos[last_row / G];
  const int p_first = a.pos[r0 / G];
  const int p_lo = a.window > 0 ? max(0, p_first - a.window + 1) : 0;

  // queries, pre-scaled
  for (int i = tid; i < kPRows * HD; i += kPThreads) {
    const int r = i / HD, d = i - r * HD, rr = r0 + r;
    float v = 0.f;
    if (rr < rows) {
      const int jj = rr / G, h = g * G + (rr - jj * G);
      v = a.q[((size_t)jj * a.n_head + h) * HD + d] * a.qscale;
    }
    qs[i] = v;
  }
  float m = -INFINITY, l = 0.f;
  float o[CPT];
#pragma unroll
  for (int c = 0; c < CPT; ++c) o[c] = 0.f;
  const __nv_bfloat16 *kb = a.k + (size_t)g * a.cap * HD;
  const __nv_bfloat16 *vb = a.v + (size_t)g * a.cap * HD;

  for (int t0 = p_lo; t0 <= p_hi; t0 += kPTile) {
    __syncthreads();   // the previous tile is consumed (and qs written, first time)
    const int nt = min(kPTile, p_hi + 1 - t0);
    for (int i = tid; i < kPTile * (HD / 2); i += kPThreads) {
      const int p = i / (HD / 2), d2 = i - p * (HD / 2);
      float2 kv = make_float2(0.f, 0.f), vv = make_float2(0.f, 0.f);
      if (p < nt) {
        const size_t off = (size_t)((t0 + p) % a.cap) * HD + 2 * d2;
        kv = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(kb + off));
        vv = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(vb + off));
      }
      ks[p * LD + 2 * d2] = kv.x;
      ks[p * LD + 2 * d2 + 1] = kv.y;
      vs[p * LD + 2 * d2] = vv.x;
      vs[p * LD + 2 * d2 + 1] = vv.y;
    }
    __syncthreads();
    // scores of this row for positions sub, sub + 16, sub + 32, sub + 48
    float s[kPTile / 16];
    {
      // one q vector load serves the four positions
      const float4 *q4 = reinterpret_cast<const float4 *>(qs + row * HD);
      float acc[kPTile / 16];
#pragma unroll
      for (int c = 0; c < kPTile / 16; ++c) acc[c] = 0.f;
#pragma unroll 8
      for (int d4 = 0; d4 < HD / 4; ++d4) {
        const float4 qv = q4[d4];
#pragma unroll
        for (int c = 0; c < kPTile / 16; ++c) {
          const float4 kv = reinterpret_cast<const float4 *>(ks + (sub + 16 * c) * LD)[d4];
          acc[c] = fmaf(qv.x, kv.x, fmaf(qv.y, kv.y, fmaf(qv.z, kv.z, fmaf(qv.w, kv.w, acc[c]))));
        }
      }
#pragma unroll
      for (int c = 0; c < kPTile / 16; ++c) s[c] = acc[c];
    }
    float tmax = -INFINITY;
#pragma unroll
    for (int c = 0; c < kPTile / 16; ++c) {
      const int p = sub + 16 * c, pos = t0 + p;
      const bool ok = live && p < nt && pos >= lo_j && pos <= pj;
      s[c] = ok ? s[c] : -INFINITY;
      tmax = fmaxf(tmax, s[c]);
    }
    // the row's 16 threads are one half-warp
#pragma unroll
    for (int off = 8; off; off >>= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, off));
    const float mn = fmaxf(m, tmax);
    float tsum = 0.f;
#pragma unroll
    for (int c = 0; c < kPTile / 16; ++c) {
      const float e = s[c] == -INFINITY ? 0.f : exp2f(s[c] - mn);
      ps[row * kPTile + sub + 16 * c] = e;
      tsum += e;
    }
#pragma unroll
    for (int off = 8; off; off >>= 1) tsum += __shfl_xor_sync(0xffffffffu, tsum, off);
    const float f = m == -INFINITY ? 0.f : exp2f(m - mn);
    l = l * f + tsum;
    m = mn;
    __syncwarp();
    // output columns CPT * sub .. CPT * sub + CPT - 1 of this row
#pragma unroll
    for (int c = 0; c < CPT; ++c) o[c] *= f;
    const float *pr = ps + row * kPTile;
    for (int p = 0; p < nt; ++p) {
      const float w = pr[p];
      const float *vr = vs + p * LD + CPT * sub;
      if constexpr (CPT % 4 == 0) {
#pragma unroll
        for (int c = 0; c < CPT; c += 4) {
          const float4 vv = *reinterpret_cast<const float4 *>(vr + c);
          o[c] = fmaf(w, vv.x, o[c]);
          o[c + 1] = fmaf(w, vv.y, o[c + 1]);
          o[c + 2] = fmaf(w, vv.z, o[c + 2]);
          o[c + 3] = fmaf(w, vv.w, o[c + 3]);
        }
      } else {
#pragma unroll
        for (int c = 0; c < CPT; ++c) o[c] = fmaf(w, vr[c], o[c]);
      }
    }
  }
  if (!live) return;
  const float inv = l > 0.f ? 1.f / l : 0.f;
  const int h = g * G + hh;
#pragma unroll
  for (int c = 0; c < CPT; ++c) {
    const float v = o[c] * inv;
    const __nv_bfloat16 hi = __float2bfloat16_rn(v);
    const __nv_bfloat16 lo = __float2bfloat16_rn(v - __bfloat162float(hi));
    const size_t col = (size_t)h * HD + CPT * sub + c;
    a.xop[(size_t)j * a.xop_ld + col] = hi;
    a.xop[(size_t)(a.bp + j) * a.xop_ld + col] = lo;
  }
}

template <int HD>
constexpr int pattn_smem() {
  return (kPRows * HD + 2 * kPTile * (HD + 4) + kPRows * kPTile) * 4;
}

template <int HD>
cudaError_t launch_hd(const PAttnArgs &a, cudaStream_t st, bool pdl, bool prepare_only) {
  if (prepare_only)
    return cudaFuncSetAttribute(k_pattn<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                pattn_smem<HD>());
  const int rows = a.n * (a.n_head / a.n_kv);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)a.n_kv, (unsigned)((rows + kPRows - 1) / kPRows));
  cfg.blockDim = dim3(kPThreads);
  cfg.dynamicSmemBytes = pattn_smem<HD>();
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, k_pattn<HD>, a);
}

}  // namespace

cudaError_t launch_pattn(int head_dim, const PAttnArgs &a, cudaStream_t st, bool pdl) {
  switch (head_dim) {
    case 32: return launch_hd<32>(a, st, pdl, false);
    case 64: return launch_hd<64>(a, st, pdl, false);
    case 128: return launch_hd<128>(a, st, pdl, false);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t prepare_pattn_kernels() {
  cudaError_t e;
  if ((e = launch_hd<32>(PAttnArgs{}, nullptr, false, true)) != cudaSuccess) return e;
  if ((e = launch_hd<64>(PAttnArgs{}, nullptr, false, true)) != cudaSuccess) return e;
  return launch_hd<128>(PAttnArgs{}, nullptr, false, true);
}

}  // namespace pnb
