// pnb_batch.cu - kernels of the batched-slot decode step: B sequences, each
// with its own KV cache and position, advance one token together.
//
// Every projection is one tensor-core GEMM Y[b][r] = sum_k W[r][k] X[b][k]
// that streams each weight once for all B slots.  A CTA owns units of
// (128-row weight tile, K range).  Warp 0 streams 64-column chunks of the
// weight tile and of the slots' operand with tiled TMA loads (128-byte
// swizzle) into a ring; warp 1 issues tcgen05.mma (M = 128 rows, N = 2 x the
// padded slot count: each operand row is split into a bf16 high part and a
// bf16 low part, so the products keep about 16 bits of the fp32 activation)
// into one of two TMEM accumulators; warps 2-5 read the accumulator back with
// tcgen05.ld, add the high and low columns and apply the fused epilogue: RoPE
// and the per-slot KV store, the residual add, SwiGLU into the next operand,
// or the LM head with each slot's argmax.  K-split units leave partial tiles
// that the last arriving CTA sums in a fixed order.
#include <cuda.h>
#include <cuda_bf16.h>
#include <float.h>
#include <limits.h>
#include <math.h>

#include "pnb_kernels.cuh"
#include "pnb_tc.cuh"

namespace pnb {
namespace {

extern __shared__ __align__(1024) uint8_t b_smem[];

constexpr int kBThreads = 192;       // warp 0 TMA, warp 1 MMA, warps 2-5 epilogue
constexpr int kWTile = 128 * 128;    // bytes of a 128-row x 64-column bf16 weight tile
constexpr int kBExtra = 1024 + 512 + 2048;  // alignment, barriers, argmax scratch

__device__ __forceinline__ float silu_b(float z) { return z / (1.0f + expf(-z)); }

__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// Fixed point of the residual K-part sums: units of 2^-32, 64-bit integers.
// Scaling an fp32 value by 2^32 is exact, so each part converts to the
// nearest unit directly (no fp64: its rate on this part is a small fraction
// of fp32's).
constexpr float kFixScale = 4294967296.0f, kFixUnit = 1.0f / 4294967296.0f;
__device__ __forceinline__ void fix_add(long long *p, float v) {
  atomicAdd(reinterpret_cast<unsigned long long *>(p),
            static_cast<unsigned long long>(__float2ll_rn(v * kFixScale)));
}
// x plus its pending fixed-point sum (the sum rounded to fp32, then the add)
__device__ __forceinline__ float fix_fold(float x, long long a) {
  return x + __ll2float_rn(a) * kFixUnit;
}
__device__ __forceinline__ float4 fold4(float4 f, const long long *acc) {
  const longlong2 a0 = __ldcg(reinterpret_cast<const longlong2 *>(acc));
  const longlong2 a1 = __ldcg(reinterpret_cast<const longlong2 *>(acc) + 1);
  return make_float4(fix_fold(f.x, a0.x), fix_fold(f.y, a0.y), fix_fold(f.z, a1.x), fix_fold(f.w, a1.y));
}

__device__ __forceinline__ void am_merge(float &v, int &i, float ov, int oi) {
  if (ov > v || (ov == v && oi < i)) {
    v = ov;
    i = oi;
  }
}

// ------------------------------------------------------------------ norm
// One CTA per slot: RMSNorm(x_b) * w into the operand's rows b (bf16 of the
// value) and bp + b (bf16 of what the first rounding left).  On the first
// layer x_b is the embedding row of the slot's token, and the CTA also
// publishes the slot table, the slot's position and its RoPE angles.
template <bool FOLD>   // FOLD: fold the fixed-point K-part sums into x first
__global__ void __launch_bounds__(256) k_bnorm(const BNormArgs a) {
  __shared__ float red[8];
  __shared__ int tok_s, pos_s;
  const int b = blockIdx.x, tid = threadIdx.x;
  if (tid == 0) ktrace(a.tr, 0);
  // norm weights do not depend on earlier kernels
  constexpr int kPer = 16;   // elements per thread per pass (4 float4)
  pdl_wait();
  pdl_trigger();
  if (tid == 0) ktrace(a.tr, 1);
  const __nv_bfloat16 *row = nullptr;
  if (a.emb) {
    if (b == 0 && tid == 0) *a.err = 0;   // the batch's error word, per step
    if (tid == 0) {
      const BSlot s = a.slots[b];
      a.slots_dev[b] = s;
      int tok = a.tokens ? a.tokens[b] : s.io->token;
      if (tok < 0 || tok >= a.n_vocab) {
        set_error(&s.io->error, kErrToken);
        tok = 0;
      }
      int pos = s.io->pos;
      if (pos < 0 || pos >= a.n_ctx) {
        set_error(&s.io->error, kErrToken);
        pos = 0;
      }
      tok_s = tok;
      pos_s = pos;
      a.pos[b] = pos;
    }
    __syncthreads();
    row = static_cast<const __nv_bfloat16 *>(a.emb) + (size_t)tok_s * a.E;
    const int half = a.hd / 2;
    for (int i = tid; i < half; i += 256) {
      const double phi = (double)pos_s * a.inv_freq[i];
      const double k = rint(phi * 0.15915494309189535);
      double r = fma(-k, 6.283185307179586, phi);
      r = fma(-k, 2.4492935982947064e-16, r);
      float sn, cs;
      sincosf((float)r, &sn, &cs);
      a.rope[(size_t)b * half + i] = make_float2(cs, sn);
    }
  }
  // one pass when E <= 256 * kPer (all loads issued before use), else a loop
  const float *xr = a.x + (size_t)b * a.E;
  float v[kPer];
  float ss = 0.f;
  for (int base = 0; base < a.E; base += 256 * kPer) {
#pragma unroll
    for (int j = 0; j < kPer / 4; ++j) {
      const int i = base + (j * 256 + tid) * 4;
      float4 f = make_float4(0.f, 0.f, 0.f, 0.f);
      if (i < a.E) {
        if (row) {
          const uint2 u = *reinterpret_cast<const uint2 *>(row + i);
          f = make_float4(bf16lo(u.x), bf16hi(u.x), bf16lo(u.y), bf16hi(u.y));
        } else {
          f = __ldcg(reinterpret_cast<const float4 *>(xr + i));
          if constexpr (FOLD) f = fold4(f, a.acc + (size_t)b * a.E + i);
        }
      }
      v[4 * j] = f.x;
      v[4 * j + 1] = f.y;
      v[4 * j + 2] = f.z;
      v[4 * j + 3] = f.w;
    }
#pragma unroll
    for (int j = 0; j < kPer; ++j) ss = fmaf(v[j], v[j], ss);
  }
  ss = warp_sum(ss);
  if ((tid & 31) == 0) red[tid >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
  for (int w = 0; w < 8; ++w) tot += red[w];
  const float inv = 1.0f / sqrtf(tot / (float)a.E + a.eps);
  __nv_bfloat16 *hi = a.xop + (size_t)b * a.E, *lo = a.xop + (size_t)(a.bp + b) * a.E;
  for (int base = 0; base < a.E; base += 256 * kPer) {
    if (a.E > 256 * kPer) {   // reload this pass's values (long rows only)
#pragma unroll
      for (int j = 0; j < kPer / 4; ++j) {
        const int i = base + (j * 256 + tid) * 4;
        float4 f = make_float4(0.f, 0.f, 0.f, 0.f);
        if (i < a.E) {
          if (row) {
            const uint2 u = *reinterpret_cast<const uint2 *>(row + i);
            f = make_float4(bf16lo(u.x), bf16hi(u.x), bf16lo(u.y), bf16hi(u.y));
          } else {
            f = __ldcg(reinterpret_cast<const float4 *>(xr + i));
            if constexpr (FOLD) f = fold4(f, a.acc + (size_t)b * a.E + i);
          }
        }
        v[4 * j] = f.x;
        v[4 * j + 1] = f.y;
        v[4 * j + 2] = f.z;
        v[4 * j + 3] = f.w;
      }
    }
#pragma unroll
    for (int j = 0; j < kPer / 4; ++j) {
      const int i = base + (j * 256 + tid) * 4;
      if (i >= a.E) continue;
      const float4 w = *reinterpret_cast<const float4 *>(a.norm_w + i);
      if (row || FOLD) *reinterpret_cast<float4 *>(a.x_out + (size_t)b * a.E + i) =
          make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
      if constexpr (FOLD) {
        longlong2 *z = reinterpret_cast<longlong2 *>(a.acc + (size_t)b * a.E + i);
        z[0] = make_longlong2(0, 0);
        z[1] = make_longlong2(0, 0);
      }
      const float n[4] = {v[4 * j] * inv * w.x, v[4 * j + 1] * inv * w.y, v[4 * j + 2] * inv * w.z,
                          v[4 * j + 3] * inv * w.w};
      __nv_bfloat16 h[4], l[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        h[e] = __float2bfloat16_rn(n[e]);
        l[e] = __float2bfloat16_rn(n[e] - __bfloat162float(h[e]));
      }
      *reinterpret_cast<uint2 *>(hi + i) = *reinterpret_cast<const uint2 *>(h);
      *reinterpret_cast<uint2 *>(lo + i) = *reinterpret_cast<const uint2 *>(l);
    }
  }
  if (tid == 0) ktrace(a.tr, 5);
}

// ------------------------------------------------------------------ GEMM

struct Smem {
  uint8_t *ring;
  uint64_t *full, *empty, *accf, *acce;
  uint32_t *tslot;
  int *flag;
  float *amv;   // [4][64]
  int *ami;     // [4][64]
};

template <int BP>
__device__ __forceinline__ Smem carve(int ns) {
  constexpr int SB = kWTile + 2 * BP * 128;
  Smem m;
  const uint32_t base = smem_addr(b_smem);
  m.ring = b_smem + ((1024u - (base & 1023u)) & 1023u);
  m.full = reinterpret_cast<uint64_t *>(m.ring + (size_t)ns * SB);
  m.empty = m.full + ns;
  m.accf = m.empty + ns;
  m.acce = m.accf + 2;
  m.tslot = reinterpret_cast<uint32_t *>(m.acce + 2);
  m.flag = reinterpret_cast<int *>(m.tslot + 1);
  m.amv = reinterpret_cast<float *>(m.ring + (size_t)ns * SB + 512);
  m.ami = reinterpret_cast<int *>(m.amv + 4 * 64);
  return m;
}

// units of this CTA: u = blockIdx.x, +gridDim.x, ...; each is a (tile, k range)
struct UnitChunks {
  const BGemmArgs *a;
  int u, c, c1;
  __device__ __forceinline__ void range(int unit) {
    const int ks = unit % a->ksplit;
    c = (int)((int64_t)a->nchunks * ks / a->ksplit);
    c1 = (int)((int64_t)a->nchunks * (ks + 1) / a->ksplit);
  }
  __device__ __forceinline__ void start(const BGemmArgs *args) {
    a = args;
    u = blockIdx.x;
    if (u < a->units) range(u);
  }
  // advance to the next chunk; false at the end
  __device__ __forceinline__ bool valid() const { return u < a->units; }
  __device__ __forceinline__ void next() {
    if (++c >= c1) {
      u += gridDim.x;
      if (u < a->units) range(u);
    }
  }
};

// the epilogue of one 128-row tile: thread owns row `row` of tile `tile`;
// y[b] = (W x_b)[row] for b < B
// The epilogue of one 128-row tile: thread owns row `row` of tile `tile`;
// y[b] = (W x_b)[row] for b < B.  Slots go in chunks of 16 whose loads are all
// issued before any of the chunk's stores (stores and loads may alias, so the
// compiler would otherwise keep one round trip per slot).
constexpr int kEpiChunk = 16;

// Slots b0 .. b0 + C - 1 of the epilogue (all BP slots at once up to 64
// padded slots; 32 at a time above).  ARG: the LM head also keeps each slot's
// best row (else it writes logits only).
template <int C, int KIND, bool ARG = true>
__device__ __forceinline__ void epilogue(const BGemmArgs &a, int tile, int row, const float (&y)[C],
                                         int b0, float (&bv)[C], int (&bi)[C]) {
  const int grow = tile * 128 + row;
  const bool in = grow < a.rows;
  constexpr int CH = C < kEpiChunk ? C : kEpiChunk;
  if constexpr (KIND == kEpiResid) {
#pragma unroll
    for (int c0 = 0; c0 < C; c0 += CH) {
      float xv[CH];
#pragma unroll
      for (int j = 0; j < CH; ++j) {
        const int b = b0 + c0 + j;
        xv[j] = (in && b < a.B) ? __ldcg(a.x + (size_t)b * a.rows + grow) : 0.f;
      }
#pragma unroll
      for (int j = 0; j < CH; ++j) {
        const int b = b0 + c0 + j;
        if (in && b < a.B) a.x[(size_t)b * a.rows + grow] = xv[j] + y[c0 + j];
      }
    }
  } else if constexpr (KIND == kEpiResidGate) {
#pragma unroll
    for (int c0 = 0; c0 < C; c0 += CH) {
      float xv[CH], gs[CH];
#pragma unroll
      for (int j = 0; j < CH; ++j) {
        const int b = b0 + c0 + j;
        const bool live = in && b < a.B;
        gs[j] = live ? a.gate[(size_t)b * a.gate_ld] : 0.f;
        xv[j] = gs[j] != 0.f ? __ldcg(a.x + (size_t)b * a.rows + grow) : 0.f;
      }
#pragma unroll
      for (int j = 0; j < CH; ++j)
        if (gs[j] != 0.f) a.x[(size_t)(b0 + c0 + j) * a.rows + grow] = xv[j] + gs[j] * y[c0 + j];
    }
  } else if constexpr (KIND == kEpiQkv) {
    const int hd = a.hd, half = hd / 2;
    const int qrows = a.n_head * hd, krows = a.n_kv * hd;
    const bool even = (grow & 1) == 0;
    const bool rope = grow < qrows + krows;
    const bool is_q = grow < qrows, is_k = !is_q && rope;
    const int kx = grow - qrows - (is_k ? 0 : krows);
    const int gk = kx / hd, d = kx - gk * hd;
    const int pair = (grow % hd) >> 1;
    const float bias = (a.bias && in) ? a.bias[grow] : 0.f;
#pragma unroll
    for (int c0 = 0; c0 < C; c0 += CH) {
      float yv[CH], par[CH];
      float2 cs[CH];
      int slot[CH];
      uint8_t *base[CH];
#pragma unroll
      for (int j = 0; j < CH; ++j) {
        const int b = b0 + c0 + j;
        yv[j] = y[c0 + j] + bias;
        par[j] = __shfl_xor_sync(0xffffffffu, yv[j], 1);
        const bool live = in && b < a.B;
        cs[j] = (live && rope) ? a.rope[(size_t)b * half + pair] : make_float2(1.f, 0.f);
        slot[j] = (live && !is_q) ? a.pos[b] : 0;
        base[j] = (live && !is_q) ? a.slots[b].kv : nullptr;
      }
#pragma unroll
      for (int j = 0; j < CH; ++j) {
        const int b = b0 + c0 + j;
        if (!(in && b < a.B)) continue;
        float v = yv[j];
        if (rope) {
          const float v0 = even ? yv[j] : par[j], v1 = even ? par[j] : yv[j];
          v = even ? v0 * cs[j].x - v1 * cs[j].y : v0 * cs[j].y + v1 * cs[j].x;
        }
        if (is_q) {
          a.q[(size_t)b * qrows + grow] = v;
        } else {
          uint8_t *kvb = base[j] + a.kv_off + (is_k ? 0 : a.layer_kv_bytes);
          reinterpret_cast<__nv_bfloat16 *>(kvb)[((size_t)gk * a.cap + slot[j] % a.cap) * hd + d] =
              __float2bfloat16_rn(v);
        }
      }
    }
  } else if constexpr (KIND == kEpiGateUp) {
    const bool even = (grow & 1) == 0;
#pragma unroll
    for (int j = 0; j < C; ++j) {
      const int b = b0 + j;
      const float par = __shfl_xor_sync(0xffffffffu, y[j], 1);
      if (b < a.B && in && even) {
        const float h = silu_b(y[j]) * par;
        const __nv_bfloat16 hi = __float2bfloat16_rn(h);
        const __nv_bfloat16 lo = __float2bfloat16_rn(h - __bfloat162float(hi));
        const int i = grow >> 1;
        a.xop[(size_t)b * a.xop_ld + i] = hi;
        a.xop[(size_t)(a.bp + b) * a.xop_ld + i] = lo;
      }
    }
  } else {  // kEpiLm
    if (in) {
#pragma unroll
      for (int j = 0; j < C; ++j) {
        const int b = b0 + j;
        if (b < a.B) {
          if (a.logits) a.logits[(size_t)b * a.rows + grow] = y[j];
          if constexpr (ARG) am_merge(bv[j], bi[j], y[j], grow);
        }
      }
    }
  }
}

template <int BP, int KIND>
__global__ void __launch_bounds__(kBThreads, 1) k_bgemm(const __grid_constant__ CUtensorMap tw,
                                                        const __grid_constant__ CUtensorMap tx,
                                                        const BGemmArgs a) {
  // the epilogue kind, and whether residual K parts go into the fixed-point sum
  constexpr int EK = KIND == kEpiResidFix ? kEpiResid : (KIND == kEpiResidGateFix ? kEpiResidGate : KIND);
  constexpr bool FIX = KIND != EK;
  constexpr int N = 2 * BP;
  constexpr int XB = N * 128, SB = kWTile + XB;
  constexpr uint32_t ACOLS = N < 32 ? 32u : (uint32_t)N;
  constexpr uint32_t TCOLS = 2 * ACOLS;
  const int ns = a.nstages;
  const Smem m = carve<BP>(ns);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    ktrace(a.tr, 0);
    for (int s = 0; s < ns; ++s) {
      mbar_init(&m.full[s], 1);
      mbar_init(&m.empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&m.accf[i], 1);
      mbar_init(&m.acce[i], 4);
    }
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(m.tslot, TCOLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t taddr = *m.tslot;

  if (warp == 0) {
    if (lane == 0) {
      // weights do not depend on earlier kernels: the first ring's weight
      // tiles go out before griddepcontrol.wait, their operand tiles after it
      bool ok = true;
      UnitChunks it;
      it.start(&a);
      int n = 0;
      for (; it.valid() && n < ns; ++n, it.next()) {
        mbar_arrive_expect_tx(&m.full[n], SB);
        tma_load_2d(m.ring + (size_t)n * SB, &tw, it.c * 64, (it.u / a.ksplit) * 128, &m.full[n]);
      }
      pdl_wait();
      pdl_trigger();
      ktrace(a.tr, 7);
      UnitChunks jt;
      jt.start(&a);
      for (int i = 0; jt.valid(); ++i, jt.next()) {
        const int s = i % ns, r = i / ns;
        if (i >= n) {
          if (!mbar_wait(&m.empty[s], (r - 1) & 1)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&m.full[s], SB);
          tma_load_2d(m.ring + (size_t)s * SB, &tw, jt.c * 64, (jt.u / a.ksplit) * 128, &m.full[s]);
        }
        tma_load_2d(m.ring + (size_t)s * SB + kWTile, &tx, jt.c * 64, 0, &m.full[s]);
      }
      ktrace(a.tr, 6);
      if (!ok) set_error(a.err, kErrTimeout);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(128, N);
      bool ok = true;
      int i = 0, j = 0;
      for (int u = blockIdx.x; u < a.units && ok; u += gridDim.x, ++j) {
        const int acc = j & 1;
        if (j >= 2 && !mbar_wait(&m.acce[acc], ((j >> 1) - 1) & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = taddr + (uint32_t)acc * ACOLS;
        const int ks = u % a.ksplit;
        const int c0 = (int)((int64_t)a.nchunks * ks / a.ksplit);
        const int c1 = (int)((int64_t)a.nchunks * (ks + 1) / a.ksplit);
        for (int c = c0; c < c1; ++c, ++i) {
          const int s = i % ns, r = i / ns;
          if (!mbar_wait(&m.full[s], r & 1)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (i == 0) ktrace(a.tr, 1);
          const uint8_t *wt = m.ring + (size_t)s * SB, *xt = wt + kWTile;
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_bf16(d, desc_k_sw128(wt, k * 32), desc_k_sw128(xt, k * 32), idesc, c > c0 || k > 0);
          mma_commit(&m.empty[s]);
        }
        if (ok) mma_commit(&m.accf[acc]);
      }
      ktrace(a.tr, 2);
      if (!ok) set_error(a.err, kErrTimeout);
    }
    __syncwarp();
  } else {
    // epilogue warps 2-5: TMEM lane quarter (warp % 4), one tile row per thread;
    // positions, RoPE angles, the slot table and the residual come from
    // earlier kernels
    pdl_wait();
    const int q = warp & 3, row = 32 * q + lane;
    if constexpr (BP > 64) {
      // 128 padded slots: each accumulator row is read and applied 32 slots
      // at a time (a row's 128 values would not fit in registers); the LM
      // head writes logits only, and a per-slot argmax kernel follows
      float dv[32];
      int di[32];
      bool ok = true;
      int j = 0;
      for (int u = blockIdx.x; u < a.units; u += gridDim.x, ++j) {
        const int acc = j & 1;
        if (ok && !mbar_wait(&m.accf[acc], (j >> 1) & 1)) {
          ok = false;
          if (lane == 0) set_error(a.err, kErrTimeout);
        }
        if (j == 0 && row == 0) ktrace(a.tr, 3);
        const int tile = u / a.ksplit;
        const int grow = tile * 128 + row;
        const uint32_t t0 = taddr + ((uint32_t)(32 * q) << 16) + (uint32_t)acc * ACOLS;
        if (ok) tc_fence_after();
#pragma unroll 1
        for (int c0 = 0; c0 < BP; c0 += 32) {
          float y[32];
          if (ok) {
            float h[32], l[32];
            tmem_ld32(t0 + c0, h);
            tmem_ld32(t0 + BP + c0, l);
#pragma unroll
            for (int i = 0; i < 32; ++i) y[i] = h[i] + l[i];
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) y[i] = 0.f;
          }
          if (a.ksplit == 1) {
            epilogue<32, EK, false>(a, tile, row, y, c0, dv, di);
          } else if constexpr (EK == kEpiResid) {
            if (grow < a.rows) {
#pragma unroll
              for (int i = 0; i < 32; ++i)
                if (c0 + i < a.B) {
                  if constexpr (FIX) fix_add(a.acc + (size_t)(c0 + i) * a.rows + grow, y[i]);
                  else atomicAdd(a.x + (size_t)(c0 + i) * a.rows + grow, y[i]);
                }
            }
          } else if constexpr (EK == kEpiResidGate) {
            if (grow < a.rows) {
#pragma unroll
              for (int i = 0; i < 32; ++i)
                if (c0 + i < a.B) {
                  const float gs = a.gate[(size_t)(c0 + i) * a.gate_ld];
                  if (gs != 0.f) {
                    if constexpr (FIX) fix_add(a.acc + (size_t)(c0 + i) * a.rows + grow, gs * y[i]);
                    else atomicAdd(a.x + (size_t)(c0 + i) * a.rows + grow, gs * y[i]);
                  }
                }
            }
          } else {
            // a partial tile: k_bmerge (QKV, gate/up) or the tile's last CTA
            // (LM head) sums the K parts
            float *P = a.part + (size_t)u * a.B * 128;
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (c0 + i < a.B) P[(size_t)(c0 + i) * 128 + row] = y[i];
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&m.acce[acc]);
        if constexpr (EK == kEpiLm) {
          if (a.ksplit > 1) {
            __threadfence();
            epi_sync();
            if (row == 0) *m.flag = atomicAdd(&a.tile_cnt[tile], 1u) == (unsigned)a.ksplit - 1u;
            epi_sync();
            if (*m.flag) {
              __threadfence();
              const float *P0 = a.part + (size_t)tile * a.ksplit * a.B * 128;
#pragma unroll 1
              for (int c0 = 0; c0 < BP; c0 += 32) {
                float y[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) y[i] = 0.f;
                for (int k = 0; k < a.ksplit; ++k) {
#pragma unroll
                  for (int i = 0; i < 32; ++i)
                    if (c0 + i < a.B) y[i] += __ldcg(P0 + ((size_t)k * a.B + c0 + i) * 128 + row);
                }
                epilogue<32, kEpiLm, false>(a, tile, row, y, c0, dv, di);
              }
              if (row == 0) a.tile_cnt[tile] = 0u;
            }
            epi_sync();
          }
        }
      }
      if (row == 0) ktrace(a.tr, 4);
    } else {
      float bv[BP];
      int bi[BP];
  #pragma unroll
      for (int b = 0; b < BP; ++b) {
        bv[b] = -FLT_MAX;
        bi[b] = INT_MAX;
      }
      bool ok = true;
      int j = 0;
      for (int u = blockIdx.x; u < a.units; u += gridDim.x, ++j) {
        const int acc = j & 1;
        if (ok && !mbar_wait(&m.accf[acc], (j >> 1) & 1)) {
          ok = false;
          if (lane == 0) set_error(a.err, kErrTimeout);
        }
        if (j == 0 && row == 0) ktrace(a.tr, 3);
        float y[BP];
  #pragma unroll
        for (int b = 0; b < BP; ++b) y[b] = 0.f;
        if (ok) {
          tc_fence_after();
          const uint32_t t0 = taddr + ((uint32_t)(32 * q) << 16) + (uint32_t)acc * ACOLS;
          if constexpr (BP == 16) {
            float v[32];
            tmem_ld32(t0, v);
  #pragma unroll
            for (int b = 0; b < 16; ++b) y[b] = v[b] + v[16 + b];
          } else {
  #pragma unroll
            for (int cb = 0; cb < N / 32; ++cb) {
              float v[32];
              tmem_ld32(t0 + 32 * cb, v);
  #pragma unroll
              for (int i = 0; i < 32; ++i) {
                if (32 * cb < BP) y[32 * cb + i] = v[i];
                else y[32 * cb - BP + i] += v[i];
              }
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&m.acce[acc]);
        const int tile = u / a.ksplit;
        if (a.ksplit == 1) {
          epilogue<BP, EK>(a, tile, row, y, 0, bv, bi);
        } else if constexpr (EK == kEpiResid) {
          // a residual update is a sum: each K part adds its share with a
          // fire-and-forget reduction, in fp32 (order not fixed) or, for the
          // deterministic step, in 64-bit fixed point (the next norm folds it in)
          const int grow = tile * 128 + row;
          if (grow < a.rows) {
  #pragma unroll
            for (int b = 0; b < BP; ++b)
              if (b < a.B) {
                if constexpr (FIX) fix_add(a.acc + (size_t)b * a.rows + grow, y[b]);
                else atomicAdd(a.x + (size_t)b * a.rows + grow, y[b]);
              }
          }
        } else if constexpr (EK == kEpiResidGate) {
          const int grow = tile * 128 + row;
          if (grow < a.rows) {
  #pragma unroll
            for (int b = 0; b < BP; ++b)
              if (b < a.B) {
                const float gs = a.gate[(size_t)b * a.gate_ld];
                if (gs != 0.f) {
                  if constexpr (FIX) fix_add(a.acc + (size_t)b * a.rows + grow, gs * y[b]);
                  else atomicAdd(a.x + (size_t)b * a.rows + grow, gs * y[b]);
                }
              }
          }
        } else if constexpr (KIND == kEpiQkv || KIND == kEpiGateUp) {
          // partial tile only: k_bmerge sums the K parts and applies the epilogue
          float *P = a.part + (size_t)u * a.B * 128;
  #pragma unroll
          for (int b = 0; b < BP; ++b)
            if (b < a.B) P[(size_t)b * 128 + row] = y[b];
        } else {
          float *P = a.part + (size_t)u * a.B * 128;
  #pragma unroll
          for (int b = 0; b < BP; ++b)
            if (b < a.B) P[(size_t)b * 128 + row] = y[b];
          __threadfence();
          epi_sync();
          if (row == 0) *m.flag = atomicAdd(&a.tile_cnt[tile], 1u) == (unsigned)a.ksplit - 1u;
          epi_sync();
          if (*m.flag) {
            __threadfence();
            const float *P0 = a.part + (size_t)tile * a.ksplit * a.B * 128;
            // fixed order over the K parts; each part's loads are independent
  #pragma unroll
            for (int b = 0; b < BP; ++b) y[b] = 0.f;
            for (int k = 0; k < a.ksplit; ++k) {
              float t[BP];
  #pragma unroll
              for (int b = 0; b < BP; ++b)
                t[b] = b < a.B ? __ldcg(P0 + ((size_t)k * a.B + b) * 128 + row) : 0.f;
  #pragma unroll
              for (int b = 0; b < BP; ++b) y[b] += t[b];
            }
            epilogue<BP, EK>(a, tile, row, y, 0, bv, bi);
            if (row == 0) a.tile_cnt[tile] = 0u;
          }
          epi_sync();
        }
      }
      if (row == 0) ktrace(a.tr, 4);
      if constexpr (KIND == kEpiLm) {
        // each slot's best row of this CTA, then of the launch (last CTA)
  #pragma unroll
        for (int b = 0; b < BP; ++b) {
          float v = bv[b];
          int i = bi[b];
  #pragma unroll
          for (int o = 16; o > 0; o >>= 1)
            am_merge(v, i, __shfl_xor_sync(0xffffffffu, v, o), __shfl_xor_sync(0xffffffffu, i, o));
          if (lane == 0) {
            m.amv[(warp - 2) * 64 + b] = v;
            m.ami[(warp - 2) * 64 + b] = i;
          }
        }
        epi_sync();
        if (row < a.B) {
          float v = m.amv[row];
          int i = m.ami[row];
          for (int w = 1; w < 4; ++w) am_merge(v, i, m.amv[w * 64 + row], m.ami[w * 64 + row]);
          a.am_val[(size_t)row * gridDim.x + blockIdx.x] = v;
          a.am_idx[(size_t)row * gridDim.x + blockIdx.x] = i;
        }
        __threadfence();
        epi_sync();
        if (row == 0) *m.flag = atomicAdd(a.am_cnt, 1u) == gridDim.x - 1u;
        epi_sync();
        if (*m.flag) {
          __threadfence();
          if (row < a.B) {
            float v = -FLT_MAX;
            int i = INT_MAX;
            for (int c0 = 0; c0 < (int)gridDim.x; c0 += 16) {
              float cv[16];
              int ci[16];
  #pragma unroll
              for (int j = 0; j < 16; ++j) {
                const int c = c0 + j < (int)gridDim.x ? c0 + j : c0;
                cv[j] = __ldcg(a.am_val + (size_t)row * gridDim.x + c);
                ci[j] = __ldcg(a.am_idx + (size_t)row * gridDim.x + c);
              }
  #pragma unroll
              for (int j = 0; j < 16; ++j)
                if (c0 + j < (int)gridDim.x) am_merge(v, i, cv[j], ci[j]);
            }
            StepIO *io = a.slots[row].io;
            if (i < 0 || i >= a.rows) {
              set_error(&io->error, kErrToken);
              i = 0;
            }
            if (a.argmax_out) a.argmax_out[row] = i;
            io->token = i;
            io->pos = a.pos[row] + 1;
            const int e = *reinterpret_cast<volatile int32_t *>(a.err);
            if (e) set_error(&io->error, e);
          }
          if (row == 0) *a.am_cnt = 0u;
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) ktrace(a.tr, 5);
  if (warp == 1) tmem_dealloc(taddr, TCOLS);
}

// The K parts of a split QKV or gate/up GEMM, summed in a fixed order, and
// the fused epilogue: one thread per (row pair, slot).  Partial tiles are
// [tile * ksplit + k][slot][128 rows].
template <int KIND>
__global__ void __launch_bounds__(256) k_bmerge(const BGemmArgs a) {
  pdl_wait();
  pdl_trigger();
  const int npair = a.rows / 2;
  const int64_t idx = (int64_t)blockIdx.x * 256 + threadIdx.x;
  if (idx >= (int64_t)npair * a.B) return;
  const int b = (int)(idx / npair), pr = (int)(idx - (int64_t)b * npair);
  const int r = 2 * pr, tile = r >> 7, i = r & 127;
  float2 s = make_float2(0.f, 0.f);
  for (int k0 = 0; k0 < a.ksplit; k0 += 4) {
    float2 t[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int k = k0 + j < a.ksplit ? k0 + j : k0;
      t[j] = __ldcg(reinterpret_cast<const float2 *>(
          a.part + (((size_t)tile * a.ksplit + k) * a.B + b) * 128 + i));
    }
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (k0 + j < a.ksplit) {
        s.x += t[j].x;
        s.y += t[j].y;
      }
  }
  if constexpr (KIND == kEpiQkv) {
    const int hd = a.hd, qrows = a.n_head * hd, krows = a.n_kv * hd;
    float v0 = s.x, v1 = s.y;
    if (a.bias) {
      v0 += a.bias[r];
      v1 += a.bias[r + 1];
    }
    if (r < qrows + krows) {
      const float2 cs = a.rope[(size_t)b * (hd / 2) + ((r % hd) >> 1)];
      const float t0 = v0 * cs.x - v1 * cs.y, t1 = v0 * cs.y + v1 * cs.x;
      v0 = t0;
      v1 = t1;
    }
    if (r < qrows) {
      *reinterpret_cast<float2 *>(a.q + (size_t)b * qrows + r) = make_float2(v0, v1);
    } else {
      const bool is_k = r < qrows + krows;
      const int kx = r - qrows - (is_k ? 0 : krows);
      const int gk = kx / hd, d = kx - gk * hd;
      uint8_t *base = a.slots[b].kv + a.kv_off + (is_k ? 0 : a.layer_kv_bytes);
      __nv_bfloat16 *dst = reinterpret_cast<__nv_bfloat16 *>(base) +
                           ((size_t)gk * a.cap + a.pos[b] % a.cap) * hd + d;
      dst[0] = __float2bfloat16_rn(v0);
      dst[1] = __float2bfloat16_rn(v1);
    }
  } else {
    const float h = silu_b(s.x) * s.y;
    const __nv_bfloat16 hi = __float2bfloat16_rn(h);
    a.xop[(size_t)b * a.xop_ld + pr] = hi;
    a.xop[(size_t)(a.bp + b) * a.xop_ld + pr] = __float2bfloat16_rn(h - __bfloat162float(hi));
  }
}

template <int BP, int KIND>
cudaError_t launch_k(const void *tw, const void *tx, const BGemmArgs &a, int grid, int smem,
                     cudaStream_t st, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kBThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, k_bgemm<BP, KIND>, *static_cast<const CUtensorMap *>(tw),
                            *static_cast<const CUtensorMap *>(tx), a);
}

template <int BP>
cudaError_t launch_bp(const void *tw, const void *tx, const BGemmArgs &a, int grid, int smem,
                      cudaStream_t st, bool pdl) {
  switch (a.kind) {
    case kEpiQkv: return launch_k<BP, kEpiQkv>(tw, tx, a, grid, smem, st, pdl);
    case kEpiResid: return launch_k<BP, kEpiResid>(tw, tx, a, grid, smem, st, pdl);
    case kEpiGateUp: return launch_k<BP, kEpiGateUp>(tw, tx, a, grid, smem, st, pdl);
    case kEpiLm: return launch_k<BP, kEpiLm>(tw, tx, a, grid, smem, st, pdl);
    case kEpiResidGate: return launch_k<BP, kEpiResidGate>(tw, tx, a, grid, smem, st, pdl);
    case kEpiResidFix: return launch_k<BP, kEpiResidFix>(tw, tx, a, grid, smem, st, pdl);
    case kEpiResidGateFix: return launch_k<BP, kEpiResidGateFix>(tw, tx, a, grid, smem, st, pdl);
    default: return cudaErrorInvalidValue;
  }
}

template <int BP>
cudaError_t prepare_bp(int smem) {
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(k_bgemm<BP, kEpiQkv>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                smem)) != cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(k_bgemm<BP, kEpiResid>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                smem)) != cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(k_bgemm<BP, kEpiGateUp>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                smem)) != cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(k_bgemm<BP, kEpiResidFix>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                smem)) != cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(k_bgemm<BP, kEpiResidGateFix>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) != cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(k_bgemm<BP, kEpiResidGate>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) != cudaSuccess)
    return e;
  return cudaFuncSetAttribute(k_bgemm<BP, kEpiLm>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
}

}  // namespace

int bgemm_smem(int bp, int nstages) { return nstages * (kWTile + 2 * bp * 128) + kBExtra; }

cudaError_t launch_bgemm(const void *tmap_w, const void *tmap_x, const BGemmArgs &a, int grid,
                         int smem, cudaStream_t st, bool pdl) {
  switch (a.bp) {
    case 16: return launch_bp<16>(tmap_w, tmap_x, a, grid, smem, st, pdl);
    case 32: return launch_bp<32>(tmap_w, tmap_x, a, grid, smem, st, pdl);
    case 64: return launch_bp<64>(tmap_w, tmap_x, a, grid, smem, st, pdl);
    case 128: return launch_bp<128>(tmap_w, tmap_x, a, grid, smem, st, pdl);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_bmerge(const BGemmArgs &a, cudaStream_t st, bool pdl) {
  const int64_t n = (int64_t)(a.rows / 2) * a.B;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((n + 255) / 256));
  cfg.blockDim = dim3(256);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  if (a.kind == kEpiQkv) return cudaLaunchKernelEx(&cfg, k_bmerge<kEpiQkv>, a);
  if (a.kind == kEpiGateUp) return cudaLaunchKernelEx(&cfg, k_bmerge<kEpiGateUp>, a);
  return cudaErrorInvalidValue;
}

namespace {
// one CTA per slot; per slot the arithmetic of the single-sequence router
__global__ void __launch_bounds__(256, 1) k_brouter(const BRouterArgs a) {
  extern __shared__ float rsm[];
  float *xs = rsm;
  float *red = xs + a.E;
  float *r = red + 32;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, b = blockIdx.x;
  pdl_wait();
  pdl_trigger();
  const float *x = a.x + (size_t)b * a.E;
  for (int i = tid; i < a.E; i += 256) xs[i] = x[i];
  float ss = 0.f;
  for (int i = tid; i < a.E; i += 256) ss = fmaf(xs[i], xs[i], ss);
  ss = warp_sum(ss);
  if (lane == 0) red[warp] = ss;
  __syncthreads();
  float tot = 0.f;
  for (int k = 0; k < 8; ++k) tot += red[k];
  const float inv = 1.0f / sqrtf(tot / (float)a.E + a.eps);
  for (int i = tid; i < a.E; i += 256) xs[i] = xs[i] * inv * a.norm_w[i];
  __syncthreads();
  for (int e = warp; e < a.n_expert; e += 8) {
    const __nv_bfloat16 *row = a.w + (int64_t)e * a.E;
    float acc = 0.f;
    for (int i = lane; i < a.E; i += 32) acc = fmaf(__bfloat162float(row[i]), xs[i], acc);
    acc = warp_sum(acc);
    if (lane == 0) r[e] = acc;
  }
  __syncthreads();
  if (tid == 0) {
    int idx[kMaxSegments];
    float mx = -FLT_MAX;
    for (int i = 0; i < a.k; ++i) {
      int best = -1;
      for (int e = 0; e < a.n_expert; ++e) {
        bool taken = false;
        for (int j = 0; j < i; ++j) taken |= (idx[j] == e);
        if (!taken && (best < 0 || r[e] > r[best])) best = e;
      }
      idx[i] = best;
      mx = fmaxf(mx, r[best]);
    }
    float z = 0.f;
    for (int i = 0; i < a.k; ++i) z += expf(r[idx[i]] - mx);
    float *g = a.gates + (size_t)b * a.n_expert;
    for (int e = 0; e < a.n_expert; ++e) g[e] = 0.f;
    for (int i = 0; i < a.k; ++i) g[idx[i]] = expf(r[idx[i]] - mx) / z;
  }
}
}  // namespace

cudaError_t launch_brouter(const BRouterArgs &a, int B, cudaStream_t st, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)B);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = (size_t)(a.E + 32 + a.n_expert) * 4;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, k_brouter, a);
}

cudaError_t prepare_bgemm_kernels(int smem_bytes) {
  cudaError_t e;
  if ((e = prepare_bp<16>(smem_bytes)) != cudaSuccess) return e;
  if ((e = prepare_bp<32>(smem_bytes)) != cudaSuccess) return e;
  if ((e = prepare_bp<64>(smem_bytes)) != cudaSuccess) return e;
  return prepare_bp<128>(smem_bytes);
}

namespace {
// Greedy pick of each slot after an LM head that wrote logits only (128
// padded slots): one CTA per slot, lowest id on ties; then the slot's next
// token and position, and the batch's error bits, as the LM head's own merge
// does at up to 64 slots.
__global__ void __launch_bounds__(256) k_bargmax(const BArgmaxArgs a) {
  __shared__ float sv[8];
  __shared__ int si[8];
  const int b = blockIdx.x, tid = threadIdx.x;
  pdl_wait();
  pdl_trigger();
  const float *lg = a.logits + (size_t)b * a.V;
  float v = -FLT_MAX;
  int i = INT_MAX;
  for (int r = tid; r < a.V; r += 256) am_merge(v, i, __ldcg(lg + r), r);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
    am_merge(v, i, __shfl_xor_sync(0xffffffffu, v, o), __shfl_xor_sync(0xffffffffu, i, o));
  if ((tid & 31) == 0) {
    sv[tid >> 5] = v;
    si[tid >> 5] = i;
  }
  __syncthreads();
  if (tid == 0) {
    for (int w = 1; w < 8; ++w) am_merge(v, i, sv[w], si[w]);
    StepIO *io = a.slots[b].io;
    if (i < 0 || i >= a.V) {
      set_error(&io->error, kErrToken);
      i = 0;
    }
    if (a.argmax_out) a.argmax_out[b] = i;
    io->token = i;
    io->pos = a.pos[b] + 1;
    const int e = *reinterpret_cast<volatile int32_t *>(a.err);
    if (e) set_error(&io->error, e);
  }
}
}  // namespace

cudaError_t launch_bargmax(const BArgmaxArgs &a, cudaStream_t st, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.B);
  cfg.blockDim = dim3(256);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, k_bargmax, a);
}

cudaError_t launch_bnorm(const BNormArgs &a, cudaStream_t st, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.B);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  if (a.acc && !a.emb) return cudaLaunchKernelEx(&cfg, k_bnorm<true>, a);
  return cudaLaunchKernelEx(&cfg, k_bnorm<false>, a);
}

}  // namespace pnb
