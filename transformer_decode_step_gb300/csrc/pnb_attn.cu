// pnb_attn.cu - split-KV flash-decode attention for one query token (GQA,
// optional sliding window, ring KV cache).
//
// Grid (n_split, n_kv, zgroups).  A CTA takes one KV head g, a block of
// `heads_per_cta` of the query heads that share it, and one contiguous chunk
// of the attended positions [lo, pos].  Warp 8 streams the chunk's K and V
// rows through a shared-memory ring with 1-D bulk copies; rows of positions
// before `pos` are issued before griddepcontrol.wait (earlier steps wrote
// them), the current position only after it.  Eight consumer warps score four
// positions at a time (eight lanes per position), keep a running max / sum /
// weighted V per head in the log2 domain, and merge across warps.  Each CTA
// writes (max, sum, unnormalised output) for its chunk; the last CTA of a KV
// head (atomic arrival counter, no waiting) merges all chunks.
#include <cuda_bf16.h>
#include <math.h>

#include "pnb_kernels.cuh"

namespace pnb {
namespace {

extern __shared__ __align__(128) uint8_t a_smem[];

struct AttnSmem {
  int ring, mo, mm, ml, flag, bars, total;
};

__host__ __device__ inline AttnSmem attn_smem(int stage_pos, int nstages, int hd, int gb, int es) {
  AttnSmem L;
  L.ring = 0;
  L.mo = align_up(nstages * 2 * stage_pos * hd * es, 16);
  L.mm = L.mo + kAttnWarps * gb * hd * 4;
  L.ml = L.mm + kAttnWarps * gb * 4;
  L.flag = L.ml + kAttnWarps * gb * 4;
  L.bars = align_up(L.flag + 16, 16);
  L.total = L.bars + 2 * nstages * 8;
  return L;
}

template <typename T, int HD, int GB>
__global__ void __launch_bounds__(kAttnThreads, 1) k_attn(const AttnArgs a) {
  constexpr int ES = (int)sizeof(T);
  constexpr int DPL = HD / 8;                             // dims per lane when scoring
  constexpr int UNIT = (DPL * ES < 16) ? DPL * ES : 16;   // bytes per shared-memory load
  constexpr int EPU = UNIT / ES;
  constexpr int C = DPL / EPU;                            // loads per lane per key row
  constexpr int VPL = HD / 32;                            // dims per lane when accumulating V
  constexpr int ROTDIV = 8 / C;                           // lanes sharing a load order
  const int SP = a.stage_pos, NS = a.nstages;
  const int G = a.n_head / a.n_kv;
  const int zgroups = G / GB;
  const int split = blockIdx.x, g = blockIdx.y;
  const int b = blockIdx.z / zgroups, z = blockIdx.z - b * zgroups;   // slot (0 for one sequence)
  const int h0 = g * G + z * GB;
  const bool batched = a.slots != nullptr;
  const BSlot bs = batched ? a.slots[b] : BSlot{nullptr, a.io};
  int32_t *err = &bs.io->error;
  const float *qb = a.q + (size_t)b * a.n_head * HD;
  float *part = a.part + (size_t)b * a.n_head * a.n_split * (HD + 2);
  unsigned *counter = a.counter + (size_t)b * a.n_kv * zgroups;
  const void *k_cache = batched ? static_cast<const void *>(bs.kv + a.kv_off) : a.k_cache;
  const void *v_cache = batched ? static_cast<const void *>(bs.kv + a.kv_off + a.layer_kv_bytes)
                                : a.v_cache;

  // positions of this CTA (pos was written by an earlier step: readable before the wait)
  const int pos = batched ? a.pos[b] : a.io->pos;
  // the first position whose K / V the preceding kernel wrote: this one, or
  // a prefill chunk's first (its tokens share the cache); stages reaching it
  // are loaded after the dependency wait
  const int p_new = batched && a.shared_cache ? a.pos[0] : pos;
  const int lo = a.window > 0 ? max(0, pos - a.window + 1) : 0;
  const int n = pos - lo + 1;
  const int chunk = (n + a.n_split - 1) / a.n_split;
  const int c0 = lo + split * chunk;
  const int npos = max(0, min(pos + 1, c0 + chunk) - c0);
  const int nst = (npos + SP - 1) / SP;

  const AttnSmem L = attn_smem(SP, NS, HD, GB, ES);
  T *ring = reinterpret_cast<T *>(a_smem + L.ring);
  float *mo = reinterpret_cast<float *>(a_smem + L.mo);
  float *mm = reinterpret_cast<float *>(a_smem + L.mm);
  float *ml = reinterpret_cast<float *>(a_smem + L.ml);
  int *flag = reinterpret_cast<int *>(a_smem + L.flag);
  uint64_t *full = reinterpret_cast<uint64_t *>(a_smem + L.bars);
  uint64_t *empty = full + NS;
  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kAttnWarps);
    }
    fence_barrier_init();
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
  if (tid == 0) ktrace(a.tr, 0);

  if (warp == kAttnWarps) {
    if (lane == 0) {
      const T *kb = static_cast<const T *>(k_cache) + (int64_t)g * a.cap * HD;
      const T *vb = static_cast<const T *>(v_cache) + (int64_t)g * a.cap * HD;
      bool waited = false, ok = true;
      int st = 0;
      for (; st < nst; ++st) {
        const int a0 = c0 + st * SP, np = min(SP, npos - st * SP);
        const int slot = st % NS, round = st / NS;
        if (!waited && (a0 + np > p_new || st == NS)) {
          ktrace(a.tr, 6);
          pdl_wait();
          pdl_trigger();
          ktrace(a.tr, 7);
          waited = true;
        }
        if (round > 0 && !mbar_wait(&empty[slot], (round - 1) & 1)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&full[slot], 2u * np * HD * ES);
        T *ks = ring + (size_t)slot * 2 * SP * HD, *vs = ks + SP * HD;
        const int s0 = a0 % a.cap, n1 = min(np, a.cap - s0);
        bulk_g2s(ks, kb + (int64_t)s0 * HD, n1 * HD * ES, &full[slot]);
        bulk_g2s(vs, vb + (int64_t)s0 * HD, n1 * HD * ES, &full[slot]);
        if (n1 < np) {
          bulk_g2s(ks + n1 * HD, kb, (np - n1) * HD * ES, &full[slot]);
          bulk_g2s(vs + n1 * HD, vb, (np - n1) * HD * ES, &full[slot]);
        }
      }
      if (!waited) {
        pdl_wait();
        pdl_trigger();
      }
      if (!ok) set_error(err, kErrTimeout);
      for (int j = st > NS ? st - NS : 0; j < st; ++j)
        if (!mbar_wait(&full[j % NS], (j / NS) & 1)) set_error(err, kErrTimeout);
    }
    return;
  }

  // ------------------------------------------------------------ consumers
  pdl_wait();
  if (tid == 0) ktrace(a.tr, 1);
  const int sub = lane & 7, t = lane >> 3;
  const int rot = sub / ROTDIV;
  float qr[GB][C][EPU];
#pragma unroll
  for (int gh = 0; gh < GB; ++gh)
#pragma unroll
    for (int c = 0; c < C; ++c) {
      const int u = (c + rot) % C;
#pragma unroll
      for (int e = 0; e < EPU; ++e)
        qr[gh][c][e] = qb[(int64_t)(h0 + gh) * HD + sub * DPL + u * EPU + e] * a.qscale;
    }
  if (tid == 0) ktrace(a.tr, 2);
  float m[GB], l[GB], o[GB][VPL];
#pragma unroll
  for (int gh = 0; gh < GB; ++gh) {
    m[gh] = -INFINITY;
    l[gh] = 0.f;
#pragma unroll
    for (int d = 0; d < VPL; ++d) o[gh][d] = 0.f;
  }
  const int PPW = SP / kAttnWarps;
  bool ok = true;
  for (int st = 0; st < nst; ++st) {
    const int slot = st % NS, round = st / NS;
    if (ok && !mbar_wait(&full[slot], round & 1)) {
      ok = false;
      if (lane == 0) set_error(err, kErrTimeout);
    }
    if (st == 0 && tid == 0) ktrace(a.tr, 3);
    if (!ok) continue;
    const T *ks = ring + (size_t)slot * 2 * SP * HD, *vs = ks + SP * HD;
    const int np = min(SP, npos - st * SP);
    for (int it = 0; it < PPW; it += 4) {
      const int pbase = warp * PPW + it;
      if (pbase >= np) break;
      const int pi = pbase + t;
      const bool valid = pi < np;
      float s[GB];
#pragma unroll
      for (int gh = 0; gh < GB; ++gh) s[gh] = 0.f;
      if (valid) {
        const T *kr = ks + pi * HD + sub * DPL;
        float kf[C][EPU];
#pragma unroll
        for (int c = 0; c < C; ++c) load_vals<T, EPU>(kr + ((c + rot) % C) * EPU, kf[c]);
#pragma unroll
        for (int gh = 0; gh < GB; ++gh) {
          float acc = 0.f;
#pragma unroll
          for (int c = 0; c < C; ++c)
#pragma unroll
            for (int e = 0; e < EPU; ++e) acc = fmaf(qr[gh][c][e], kf[c][e], acc);
          s[gh] = acc;
        }
      }
#pragma unroll
      for (int gh = 0; gh < GB; ++gh) {
        s[gh] += __shfl_xor_sync(0xffffffffu, s[gh], 4);
        s[gh] += __shfl_xor_sync(0xffffffffu, s[gh], 2);
        s[gh] += __shfl_xor_sync(0xffffffffu, s[gh], 1);
        if (!valid) s[gh] = -INFINITY;
      }
      float sc[4][GB];
#pragma unroll
      for (int tt = 0; tt < 4; ++tt)
#pragma unroll
        for (int gh = 0; gh < GB; ++gh) sc[tt][gh] = __shfl_sync(0xffffffffu, s[gh], tt * 8);
      float vv[4][VPL];
#pragma unroll
      for (int tt = 0; tt < 4; ++tt) {
        if (pbase + tt < np) {
          load_vals<T, VPL>(vs + (pbase + tt) * HD + lane * VPL, vv[tt]);
        } else {
#pragma unroll
          for (int d = 0; d < VPL; ++d) vv[tt][d] = 0.f;
        }
      }
#pragma unroll
      for (int gh = 0; gh < GB; ++gh) {
        float mx = m[gh];
#pragma unroll
        for (int tt = 0; tt < 4; ++tt) mx = fmaxf(mx, sc[tt][gh]);
        if (mx == -INFINITY) continue;
        const float alpha = exp2f(m[gh] - mx);
        l[gh] *= alpha;
#pragma unroll
        for (int d = 0; d < VPL; ++d) o[gh][d] *= alpha;
#pragma unroll
        for (int tt = 0; tt < 4; ++tt) {
          if (pbase + tt < np) {
            const float p = exp2f(sc[tt][gh] - mx);
            l[gh] += p;
#pragma unroll
            for (int d = 0; d < VPL; ++d) o[gh][d] = fmaf(p, vv[tt][d], o[gh][d]);
          }
        }
        m[gh] = mx;
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[slot]);
  }

  if (tid == 0) ktrace(a.tr, 4);
  // merge the eight warps of this CTA
#pragma unroll
  for (int gh = 0; gh < GB; ++gh) {
    if (lane == 0) {
      mm[warp * GB + gh] = m[gh];
      ml[warp * GB + gh] = l[gh];
    }
#pragma unroll
    for (int d = 0; d < VPL; ++d) mo[(warp * GB + gh) * HD + lane * VPL + d] = o[gh][d];
  }
  consumer_sync<kAttnConsumers>();
  for (int idx = tid; idx < GB * HD; idx += kAttnConsumers) {
    const int gh = idx / HD, d = idx - gh * HD;
    float M = -INFINITY;
    for (int w = 0; w < kAttnWarps; ++w) M = fmaxf(M, mm[w * GB + gh]);
    float Ls = 0.f, Os = 0.f;
    if (M != -INFINITY) {
      for (int w = 0; w < kAttnWarps; ++w) {
        const float f = exp2f(mm[w * GB + gh] - M);
        Ls = fmaf(ml[w * GB + gh], f, Ls);
        Os = fmaf(mo[(w * GB + gh) * HD + d], f, Os);
      }
    }
    float *P = part + ((int64_t)(h0 + gh) * a.n_split + split) * (HD + 2);
    if (d == 0) {
      P[0] = M;
      P[1] = Ls;
    }
    P[2 + d] = Os;
  }
  __threadfence();
  consumer_sync<kAttnConsumers>();
  if (tid == 0) {
    const unsigned prev = atomicAdd(&counter[g * zgroups + z], 1u);
    *flag = (prev == (unsigned)a.n_split - 1u);
  }
  consumer_sync<kAttnConsumers>();
  if (*flag) {
    __threadfence();
    // one pass over the splits, eight splits' loads in flight at a time
    const int ns = a.n_split;
    for (int idx = tid; idx < GB * HD; idx += kAttnConsumers) {
      const int gh = idx / HD, d = idx - gh * HD;
      const float *P0 = part + (int64_t)(h0 + gh) * ns * (HD + 2);
      float M = -INFINITY, Ls = 0.f, Os = 0.f;
      for (int s0 = 0; s0 < ns; s0 += 8) {
        float pm[8], pl[8], po[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float *P = P0 + (int64_t)(s0 + j < ns ? s0 + j : 0) * (HD + 2);
          pm[j] = __ldcg(P);
          pl[j] = __ldcg(P + 1);
          po[j] = __ldcg(P + 2 + d);
        }
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (s0 + j >= ns) pm[j] = -INFINITY;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (pm[j] == -INFINITY) continue;
          const float Mn = fmaxf(M, pm[j]);
          const float f0 = exp2f(M - Mn), f1 = exp2f(pm[j] - Mn);
          Ls = Ls * f0 + pl[j] * f1;
          Os = Os * f0 + po[j] * f1;
          M = Mn;
        }
      }
      const float o = Os / Ls;
      if (a.xop) {
        // bf16 hi / lo parts of the next GEMM's operand
        const __nv_bfloat16 hi = __float2bfloat16_rn(o);
        const __nv_bfloat16 lo = __float2bfloat16_rn(o - __bfloat162float(hi));
        const size_t col = (size_t)(h0 + gh) * HD + d;
        a.xop[(size_t)b * a.xop_ld + col] = hi;
        a.xop[(size_t)(a.bp + b) * a.xop_ld + col] = lo;
      } else {
        a.out[(int64_t)(h0 + gh) * HD + d] = o;
      }
    }
    if (tid == 0) counter[g * zgroups + z] = 0u;
  }
  if (tid == 0) ktrace(a.tr, 5);
}

template <typename T, int HD, int GB>
cudaError_t launch_one(const AttnArgs &a, const AttnGeom &ag, cudaStream_t st, bool pdl,
                       bool prepare_only) {
  auto kern = k_attn<T, HD, GB>;
  if (prepare_only) {
    if (ag.smem <= 48 * 1024) return cudaSuccess;
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, ag.smem);
  }
  const int G = a.n_head / a.n_kv;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.n_split, a.n_kv, (G / GB) * (a.slots ? a.nb : 1));
  cfg.blockDim = dim3(kAttnThreads);
  cfg.dynamicSmemBytes = ag.smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

template <typename T, int HD>
cudaError_t launch_hd(const AttnArgs &a, const AttnGeom &ag, cudaStream_t st, bool pdl,
                      bool prep) {
  switch (ag.heads_per_cta) {
    case 1: return launch_one<T, HD, 1>(a, ag, st, pdl, prep);
    case 2: return launch_one<T, HD, 2>(a, ag, st, pdl, prep);
    case 4: return launch_one<T, HD, 4>(a, ag, st, pdl, prep);
    case 8:
      if constexpr (HD <= 64) return launch_one<T, HD, 8>(a, ag, st, pdl, prep);
      return cudaErrorInvalidValue;
    default: return cudaErrorInvalidValue;
  }
}

template <typename T>
cudaError_t launch_t(int hd, const AttnArgs &a, const AttnGeom &ag, cudaStream_t st, bool pdl,
                     bool prep) {
  switch (hd) {
    case 32: return launch_hd<T, 32>(a, ag, st, pdl, prep);
    case 64: return launch_hd<T, 64>(a, ag, st, pdl, prep);
    case 128: return launch_hd<T, 128>(a, ag, st, pdl, prep);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

AttnGeom attn_geom(int dtype, int head_dim, int group) {
  AttnGeom ag;
  const int es = dtype ? 2 : 4;
  int gb = 1;
  while (gb * 2 <= 8 && group % (gb * 2) == 0 && gb * 2 * head_dim <= 512) gb *= 2;
  ag.heads_per_cta = gb;
  int sp = 8192 / (head_dim * es);
  sp = sp < 32 ? 32 : sp - sp % 32;
  ag.stage_pos = sp;
  int ns = (96 * 1024) / (2 * sp * head_dim * es);
  ag.nstages = ns < 2 ? 2 : (ns > 8 ? 8 : ns);
  ag.smem = attn_smem(sp, ag.nstages, head_dim, gb, es).total;
  return ag;
}

cudaError_t launch_attn(int dtype, int head_dim, const AttnArgs &a, const AttnGeom &ag,
                        cudaStream_t st, bool pdl) {
  return dtype ? launch_t<__nv_bfloat16>(head_dim, a, ag, st, pdl, false)
               : launch_t<float>(head_dim, a, ag, st, pdl, false);
}

cudaError_t prepare_attn_kernel(int dtype, int head_dim, const AttnGeom &ag) {
  AttnArgs a{};
  return dtype ? launch_t<__nv_bfloat16>(head_dim, a, ag, nullptr, false, true)
               : launch_t<float>(head_dim, a, ag, nullptr, false, true);
}

}  // namespace pnb
