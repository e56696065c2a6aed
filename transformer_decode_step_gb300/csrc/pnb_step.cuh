// pnb_step.cuh - the whole single-sequence decode step as one persistent kernel.
//
// One cooperative launch per step, one CTA per SM (all CTAs co-resident).
// Warp 16 of every CTA is the producer: one thread walks the step's phases in
// order (per layer: QKV, attention, output projection, gate/up, down; then the
// LM head) and streams this CTA's share of each phase's weight rows and KV
// positions through one shared-memory ring with 1-D bulk copies.  Only two
// things make it wait besides ring space: the KV entry of the current
// position (written in the same layer's QKV phase; it waits for that phase's
// grid barrier) and, for MoE, the experts the router picked.  So the weight
// stream runs across phase boundaries and HBM stays busy while the compute
// warps synchronise.
//
// Warp 17 walks the same sequence a few items ahead of the producer and only
// issues L2 prefetches for it, so DRAM keeps streaming while the compute
// warps cross a phase boundary and the ring refills from L2.
//
// Warps 0-15 compute each phase from the ring, write its outputs, and meet the
// other CTAs at a grid barrier (generation counter; every wait is bounded and a
// timeout sets an abort flag that releases all other waiters).  The attention
// phase gives every CTA one contiguous range of the flattened (KV head,
// position) space; each CTA writes one partial (max, sum, unnormalised output)
// per KV head it touches, and the last CTA to finish a head merges its
// partials (arrival counter, no waiting).
#pragma once

#include "pnb_gemv_dev.cuh"

namespace pnb {

struct StepLayer {
  const void *wqkv, *wo, *w_gate_up, *w_down, *w_router;
  const void *const *tab_gate_up;  // MoE: this layer's expert tables (device)
  const void *const *tab_down;
  const float *attn_norm, *ffn_norm;
  void *kc, *vc;                   // this layer's [n_kv][cap][hd] caches
};

struct StepArgs {
  int E, H, Hkv, hd, F, V, L, X, k, cap, window;
  float eps, qscale;
  Geom g_qkv, g_o, g_gu, g_dn, g_lm;
  int nslots, slot_bytes, sp;      // ring slots, slot bytes, positions per attention slot
  int union_floats;                // shared scratch shared by GEMV partials and attention merge
  const void *tok_embd, *output;
  const float *out_norm;
  const double *inv_freq;
  const StepLayer *layers;
  float *x, *q, *o, *h, *attn_part, *lm_val;
  int32_t *lm_idx;
  unsigned *attn_cnt, *lm_cnt, *bar_count, *bar_gen;
  float *ss_part;            // [2][gridDim.x] per-CTA sums of squares of the rows of x it wrote
  int32_t *abort_flag;
  float *logits;
  int32_t *argmax_out;
  StepIO *io;
  unsigned long long *trace;  // optional [gridDim.x][phases][4] timestamps (ns)
};

// trace slots: 0 = compute warps done with the phase, 1 = past its grid
// barrier, 2 = producer done issuing the phase, 3 = time warp 0 spent waiting
// for ring data during the phase
__device__ __forceinline__ void trace_mark(const StepArgs &a, int phase, int what) {
  if (a.trace && what != 2) {
    const int nph = 5 * a.L + 1;
    a.trace[((size_t)blockIdx.x * nph + phase) * 6 + what] = global_ns();
  }
}
__device__ __forceinline__ void trace_add_wait(const StepArgs &a, int phase, unsigned long long ns) {
  if (a.trace && threadIdx.x == 0) {
    const int nph = 5 * a.L + 1;
    a.trace[((size_t)blockIdx.x * nph + phase) * 6 + 3] += ns;
  }
}

// shared scalars of one CTA
constexpr int kStepWarps = kGemvWarps + 2;          // compute + producer + prefetcher
constexpr int kStepThreads = kStepWarps * 32;
constexpr int kPrefetchAhead = 12;                   // items the prefetcher runs ahead

struct StepShared {
  volatile unsigned issued;  // items the producer has issued into the ring
  unsigned gen0;         // grid-barrier generation at kernel start
  int pos, token;
  volatile int route;    // MoE: layer + 1 once eidx / gate hold that layer's choice
  int flag;
  int32_t eidx[kMaxSegments];
  float gate[kMaxSegments];
  float rlog[64];
};

struct StepSmem {
  int ring, uni, qs, red, sh, bars, total;
};

constexpr int kMaxQStage = 8 * 128;   // query heads of one KV head x head_dim, fp32

__host__ __device__ inline StepSmem step_smem(int nslots, int slot_bytes, int union_floats) {
  StepSmem L;
  L.ring = 0;
  L.uni = align_up(nslots * slot_bytes, 128);
  L.qs = align_up(L.uni + union_floats * 4, 16);
  L.red = align_up(L.qs + kMaxQStage * 4, 16);
  L.sh = align_up(L.red + 64 * 4, 16);
  L.bars = align_up(L.sh + (int)sizeof(StepShared), 16);
  L.total = L.bars + 2 * nslots * 8;
  return L;
}

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned *p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_u32(unsigned *p, unsigned v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ int ld_volatile_i32(const int32_t *p) {
  return *reinterpret_cast<const volatile int32_t *>(p);
}

// Wait until at least n grid barriers of this launch have completed.
// Bounded; gives up (and raises the abort flag) on timeout or abort.
__device__ __forceinline__ bool wait_barriers(const StepArgs &a, unsigned gen0, unsigned n) {
  const unsigned long long t0 = global_ns();
  for (uint32_t it = 0;; ++it) {
    if (ld_acquire_u32(a.bar_gen) - gen0 >= n) return true;
    __nanosleep(32);
    if ((it & 255u) == 255u) {
      if (ld_volatile_i32(a.abort_flag)) return false;
      if (global_ns() - t0 > kWaitLimitNs || it > (1u << 26)) {
        atomicExch(a.abort_flag, 1);
        set_error(&a.io->error, kErrTimeout);
        return false;
      }
    }
  }
}

// ------------------------------------------------------------- ring (producer)

struct RingP {
  uint8_t *base;
  uint64_t *full, *empty;
  int nslots, slot_bytes;
  uint32_t i;   // items issued
  RingPos rp;   // slot of item i and its use parity
  bool ok;
  int32_t *err;
  volatile unsigned *issued;  // published issue count (producer) / followed (prefetcher)
  bool prefetch;              // prefetch mode: L2 hints only, kPrefetchAhead items ahead
  // start an item of `bytes` total arriving in up to four copies
  __device__ __forceinline__ uint8_t *begin(uint32_t bytes) {
    if (prefetch) {
      if (!ok) return nullptr;
      const unsigned long long t0 = global_ns();
      for (uint32_t it = 0; (int)(i - *issued) >= kPrefetchAhead; ++it) {
        if ((it & 255u) == 255u && global_ns() - t0 > kWaitLimitNs) {
          ok = false;   // stop prefetching; the producer does not depend on it
          return nullptr;
        }
      }
      return base;   // any non-null marker
    }
    if (ok && i >= (uint32_t)nslots && !mbar_wait_backoff(&empty[rp.slot], rp.phase ^ 1u)) {
      ok = false;
      set_error(err, kErrTimeout);
    }
    if (!ok) return nullptr;
    mbar_arrive_expect_tx(&full[rp.slot], bytes);
    return base + rp.slot * (uint32_t)slot_bytes;
  }
  __device__ __forceinline__ void copy(void *dst, const void *src, uint32_t bytes) {
    if (prefetch)
      bulk_prefetch_l2(src, bytes);
    else
      bulk_g2s(dst, src, bytes, &full[rp.slot]);
  }
  __device__ __forceinline__ void end() {
    ++i;
    rp.advance();
    if (!prefetch) *issued = i;
  }
  __device__ void drain() {
    if (prefetch) return;
    const uint32_t last = i < (uint32_t)nslots ? i : (uint32_t)nslots;
    RingPos dp = rp;
    for (uint32_t j = 0; j < last; ++j) {
      if (dp.slot == 0) {
        dp.slot = dp.n;
        dp.phase ^= 1u;
      }
      --dp.slot;
      if (!mbar_wait(&full[dp.slot], dp.phase)) set_error(err, kErrTimeout);
    }
  }
};

// ------------------------------------------------------------- ring (consumer)

struct RingC {
  uint8_t *base;
  uint64_t *full, *empty;
  int nslots, slot_bytes;
  RingPos rp;
  bool ok;
  int32_t *err;
  unsigned long long waited_ns;   // thread 0, when tracing
  bool timing;
  unsigned long long dot_ns;      // thread 0: time inside GEMV slots (after the data arrived)
  unsigned long long t_start, t_end;  // thread 0: last GEMV consumption start / end
  __device__ __forceinline__ const uint8_t *wait(int lane) {
    const unsigned long long t0 = timing ? global_ns() : 0ull;
    if (ok && !mbar_wait(&full[rp.slot], rp.phase)) {
      ok = false;
      if (lane == 0) set_error(err, kErrTimeout);
    }
    if (timing) waited_ns += global_ns() - t0;
    return ok ? base + rp.slot * (uint32_t)slot_bytes : nullptr;
  }
  __device__ __forceinline__ void release(int lane) {
    __syncwarp();
    if (ok && lane == 0) mbar_arrive(&empty[rp.slot]);
    rp.advance();
  }
};

// Grid barrier among the compute warps of all CTAs (barrier number nbar,
// 1-based within this launch).  All 512 compute threads call it.
__device__ __forceinline__ void grid_barrier(const StepArgs &a, StepShared &sh, unsigned nbar,
                                             RingC &R) {
  gemv_sync();
  if (threadIdx.x == 0) {
    trace_mark(a, nbar - 1, 0);
    trace_add_wait(a, nbar - 1, R.waited_ns);
    if (a.trace) {
      unsigned long long *tr = a.trace + ((size_t)blockIdx.x * (5 * a.L + 1) + nbar - 1) * 6;
      tr[2] = R.dot_ns;
      tr[4] = R.t_start;
      tr[5] = R.t_end;
    }
    R.waited_ns = 0;
    R.dot_ns = 0;
    __threadfence();
    const unsigned prev = atomicAdd(a.bar_count, 1u);
    if (prev == gridDim.x - 1) {
      atomicExch(a.bar_count, 0u);
      __threadfence();
      st_release_u32(a.bar_gen, sh.gen0 + nbar);
    } else {
      wait_barriers(a, sh.gen0, nbar);
    }
    trace_mark(a, nbar - 1, 1);
  }
  gemv_sync();
}

// CTA c's share of rows [0, total) in units of `align` rows
__device__ __forceinline__ void row_range(int64_t total, int align, int64_t *r0, int64_t *r1) {
  const int64_t units = total / align;
  *r0 = units * blockIdx.x / gridDim.x * align;
  *r1 = units * (blockIdx.x + 1) / gridDim.x * align;
}

__device__ __forceinline__ void prod_gemv(RingP &R, const Geom &g, int nseg, const void *const *w,
                                          int64_t rows, bool summed, int align) {
  int64_t r0, r1;
  row_range(summed ? rows : rows * nseg, align, &r0, &r1);
  ItemIter it(r0, r1, rows, nseg, summed, g.rows_per_stage);
  Item item;
  while (it.next(item)) {
    const uint32_t bytes = (uint32_t)item.n * (uint32_t)g.row_bytes;
    uint8_t *dst = R.begin(bytes);
    if (dst) R.copy(dst, static_cast<const uint8_t *>(w[item.seg]) + item.row * g.row_bytes, bytes);
    R.end();
  }
}

template <typename T, int NV, typename Reload>
__device__ __forceinline__ void cons_gemv(RingC &R, const Geom &g, int nseg, int64_t rows, bool summed,
                                          int align, XSlice<T, NV> &xs, float *part, int warp,
                                          int lane, int64_t *r0o, Reload &&reload) {
  int64_t r0, r1;
  row_range(summed ? rows : rows * nseg, align, &r0, &r1);
  *r0o = r0;
  if (R.timing) R.t_start = global_ns();
  const int cw = g.cw, groups = kGemvWarps / cw;
  const int grp = warp / cw, cc = warp - grp * cw;
  const int vpr = g.vpr;
  ItemIter it(r0, r1, rows, nseg, summed, g.rows_per_stage);
  Item item;
  int cur = 0;
  while (it.next(item)) {
    if (summed && item.seg != cur) {
      reload(item.seg);
      cur = item.seg;
    }
    const uint8_t *stage = R.wait(lane);
    const unsigned long long td = R.timing ? global_ns() : 0ull;
    if (stage) {
      float *pp = part + ((summed ? item.seg : 0) * g.rows_cta_max + item.local) * cw;
      for (int r = grp; r < item.n; r += groups) {
        const float v = warp_sum(dot_row<T, NV>(stage + (size_t)r * g.row_bytes, xs, vpr, cc, cw, lane));
        if (lane == 0) pp[r * cw + cc] = v;
      }
    }
    R.release(lane);
    if (R.timing) R.dot_ns += global_ns() - td;
  }
  if (R.timing) R.t_end = global_ns();
}

// -------------------------------------------------------------- attention

// The CTA's slice of the flattened (kv head, position) space: positions
// [lo, pos] of every KV head, n = pos - lo + 1 per head, T = n_kv * n total.
struct AttnRange {
  int lo, n;
  int64_t T, f0, f1;   // this CTA's flattened range [f0, f1)
};

__device__ __forceinline__ AttnRange attn_range(const StepArgs &a, int pos) {
  AttnRange r;
  r.lo = a.window > 0 ? max(0, pos - a.window + 1) : 0;
  r.n = pos - r.lo + 1;
  r.T = (int64_t)a.Hkv * r.n;
  r.f0 = r.T * blockIdx.x / gridDim.x;
  r.f1 = r.T * (blockIdx.x + 1) / gridDim.x;
  return r;
}

// CTA owning flattened position f
__device__ __forceinline__ int attn_owner(int64_t f, int64_t T, int G) {
  return (int)(((f + 1) * G - 1) / T);
}

// whether CTA c's range is non-empty (all are when T >= G)
__device__ __forceinline__ bool attn_nonempty(int c, int64_t T, int G) {
  return T * c / G < T * (c + 1) / G;
}

template <typename T, int HD>
__device__ __forceinline__ void prod_attn(RingP &R, const StepArgs &a, const StepLayer &ly, int pos,
                                          unsigned gen0, unsigned qkv_barrier) {
  const AttnRange ar = attn_range(a, pos);
  constexpr int ES = (int)sizeof(T);
  bool waited = false;
  for (int64_t f = ar.f0; f < ar.f1;) {
    const int g = (int)(f / ar.n);
    const int64_t seg_end = min(ar.f1, (int64_t)(g + 1) * ar.n);
    const T *kb = static_cast<const T *>(ly.kc) + (int64_t)g * a.cap * HD;
    const T *vb = static_cast<const T *>(ly.vc) + (int64_t)g * a.cap * HD;
    for (int np = 0; f < seg_end; f += np) {
      const int p0 = ar.lo + (int)(f - (int64_t)g * ar.n);
      np = (int)min((int64_t)a.sp, seg_end - f);
      if (!waited && p0 + np > pos && !R.prefetch) {
        // this slot holds the current position, written by this layer's QKV phase
        if (!wait_barriers(a, gen0, qkv_barrier)) R.ok = false;
        asm volatile("fence.proxy.async.global;" ::: "memory");
        waited = true;
      }
      uint8_t *dst = R.begin(2u * np * HD * ES);
      if (dst) {
        T *ks = reinterpret_cast<T *>(dst), *vs = ks + a.sp * HD;
        const int s0 = p0 % a.cap, n1 = min(np, a.cap - s0);
        R.copy(ks, kb + (int64_t)s0 * HD, n1 * HD * ES);
        R.copy(vs, vb + (int64_t)s0 * HD, n1 * HD * ES);
        if (n1 < np) {
          R.copy(ks + n1 * HD, kb, (np - n1) * HD * ES);
          R.copy(vs + n1 * HD, vb, (np - n1) * HD * ES);
        }
      }
      R.end();
    }
  }
}

template <typename T, int N>
__device__ __forceinline__ void load_vals_s(const T *p, float (&f)[N]) {
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
    if constexpr (N == 8) {
      const float4 u = *reinterpret_cast<const float4 *>(p), w = *reinterpret_cast<const float4 *>(p + 4);
      f[0] = u.x; f[1] = u.y; f[2] = u.z; f[3] = u.w; f[4] = w.x; f[5] = w.y; f[6] = w.z; f[7] = w.w;
    } else if constexpr (N == 4) {
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

// One attention phase: for each KV head this CTA touches, the online softmax
// over its positions (16 lanes per position, 2 positions per warp step, G
// query heads at once), a merge of the 16 warps, the CTA's partial, and - for
// the last CTA of a head - the merge of every partial of that head into o.
template <typename T, int HD, int G>
__device__ __forceinline__ void cons_attn(RingC &R, const StepArgs &a, int pos, float *uni, float *qs,
                                          StepShared &sh, int warp, int lane, int tid) {
  constexpr int DPL = HD / 16;   // dims per lane when scoring
  constexpr int VPL = HD / 32;   // dims per lane when accumulating V
  const AttnRange ar = attn_range(a, pos);
  const int PPW = a.sp / kGemvWarps;    // positions per warp per slot (even)
  float *mo = uni;                       // [16][G][HD]
  float *mm = mo + kGemvWarps * G * HD;  // [16][G]
  float *ml = mm + kGemvWarps * G;       // [16][G]
  const int GC = gridDim.x;
  for (int64_t f = ar.f0; f < ar.f1;) {
    const int g = (int)(f / ar.n);
    const int64_t seg_end = min(ar.f1, (int64_t)(g + 1) * ar.n);
    const int half = lane >> 4, sub = lane & 15;
    // this KV head's query heads, pre-scaled, staged in shared memory
    for (int i = tid; i < G * HD; i += kGemvConsumers) qs[i] = __ldcg(a.q + (int64_t)g * G * HD + i) * a.qscale;
    gemv_sync();
    float m[G], l[G], o[G][VPL];
#pragma unroll
    for (int gh = 0; gh < G; ++gh) {
      m[gh] = -INFINITY;
      l[gh] = 0.f;
#pragma unroll
      for (int d = 0; d < VPL; ++d) o[gh][d] = 0.f;
    }
    for (int np = 0; f < seg_end; f += np) {
      np = (int)min((int64_t)a.sp, seg_end - f);
      const uint8_t *stage = R.wait(lane);
      if (stage) {
        const T *ks = reinterpret_cast<const T *>(stage), *vs = ks + a.sp * HD;
        for (int it = 0; it < PPW; it += 2) {
          const int pbase = warp * PPW + it;
          if (pbase >= np) break;
          const int pi = pbase + half;
          const bool valid = pi < np;
          float s[G];
#pragma unroll
          for (int gh = 0; gh < G; ++gh) s[gh] = 0.f;
          if (valid) {
            float kf[DPL];
            load_vals_s<T, DPL>(ks + pi * HD + sub * DPL, kf);
#pragma unroll
            for (int gh = 0; gh < G; ++gh) {
              float qv[DPL];
              load_vals_s<float, DPL>(qs + gh * HD + sub * DPL, qv);
              float acc = 0.f;
#pragma unroll
              for (int e = 0; e < DPL; ++e) acc = fmaf(qv[e], kf[e], acc);
              s[gh] = acc;
            }
          }
#pragma unroll
          for (int gh = 0; gh < G; ++gh) {
            s[gh] += __shfl_xor_sync(0xffffffffu, s[gh], 8);
            s[gh] += __shfl_xor_sync(0xffffffffu, s[gh], 4);
            s[gh] += __shfl_xor_sync(0xffffffffu, s[gh], 2);
            s[gh] += __shfl_xor_sync(0xffffffffu, s[gh], 1);
            if (!valid) s[gh] = -INFINITY;
          }
          float sc[2][G];
#pragma unroll
          for (int gh = 0; gh < G; ++gh) {
            sc[0][gh] = __shfl_sync(0xffffffffu, s[gh], 0);
            sc[1][gh] = __shfl_sync(0xffffffffu, s[gh], 16);
          }
          float vv[2][VPL];
#pragma unroll
          for (int tt = 0; tt < 2; ++tt) {
            if (pbase + tt < np) {
              load_vals_s<T, VPL>(vs + (pbase + tt) * HD + lane * VPL, vv[tt]);
            } else {
#pragma unroll
              for (int d = 0; d < VPL; ++d) vv[tt][d] = 0.f;
            }
          }
#pragma unroll
          for (int gh = 0; gh < G; ++gh) {
            const float mx = fmaxf(m[gh], fmaxf(sc[0][gh], sc[1][gh]));
            if (mx == -INFINITY) continue;
            const float alpha = exp2f(m[gh] - mx);
            l[gh] *= alpha;
#pragma unroll
            for (int d = 0; d < VPL; ++d) o[gh][d] *= alpha;
#pragma unroll
            for (int tt = 0; tt < 2; ++tt) {
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
      }
      R.release(lane);
    }

    // merge the 16 warps of this CTA into one partial for head group g
#pragma unroll
    for (int gh = 0; gh < G; ++gh) {
      if (lane == 0) {
        mm[warp * G + gh] = m[gh];
        ml[warp * G + gh] = l[gh];
      }
#pragma unroll
      for (int d = 0; d < VPL; ++d) mo[(warp * G + gh) * HD + lane * VPL + d] = o[gh][d];
    }
    gemv_sync();
    const int c_first = attn_owner((int64_t)g * ar.n, ar.T, GC);
    const int c_last = attn_owner((int64_t)(g + 1) * ar.n - 1, ar.T, GC);
    const int slot = blockIdx.x - c_first;
    for (int idx = tid; idx < G * HD; idx += kGemvConsumers) {
      const int gh = idx / HD, d = idx - gh * HD;
      float M = -INFINITY;
      for (int w = 0; w < kGemvWarps; ++w) M = fmaxf(M, mm[w * G + gh]);
      float Ls = 0.f, Os = 0.f;
      if (M != -INFINITY) {
        for (int w = 0; w < kGemvWarps; ++w) {
          const float fw = exp2f(mm[w * G + gh] - M);
          Ls = fmaf(ml[w * G + gh], fw, Ls);
          Os = fmaf(mo[(w * G + gh) * HD + d], fw, Os);
        }
      }
      float *P = a.attn_part + (((int64_t)g * GC + slot) * G + gh) * (HD + 2);
      if (d == 0) {
        P[0] = M;
        P[1] = Ls;
      }
      P[2 + d] = Os;
    }
    __threadfence();
    gemv_sync();
    if (tid == 0) {
      int nz = 0;
      for (int c = c_first; c <= c_last; ++c) nz += attn_nonempty(c, ar.T, GC);
      const unsigned prev = atomicAdd(&a.attn_cnt[g], 1u);
      sh.flag = prev == (unsigned)(nz - 1);
    }
    gemv_sync();
    if (sh.flag) {
      __threadfence();
      const int nc = c_last - c_first + 1;
      for (int idx = tid; idx < G * HD; idx += kGemvConsumers) {
        const int gh = idx / HD, d = idx - gh * HD;
        float M = -INFINITY, Ls = 0.f, Os = 0.f;
        for (int s0 = 0; s0 < nc; s0 += 8) {
          float pm[8], pl[8], po[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int sp = s0 + j < nc ? s0 + j : 0;
            const float *P = a.attn_part + (((int64_t)g * GC + sp) * G + gh) * (HD + 2);
            pm[j] = __ldcg(P);
            pl[j] = __ldcg(P + 1);
            po[j] = __ldcg(P + 2 + d);
          }
#pragma unroll
          for (int j = 0; j < 8; ++j)
            if (!(s0 + j < nc && attn_nonempty(c_first + s0 + j, ar.T, GC))) pm[j] = -INFINITY;
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
        a.o[(int64_t)(g * G + gh) * HD + d] = Os / Ls;
      }
      if (tid == 0) a.attn_cnt[g] = 0u;
    }
    gemv_sync();
  }
}

// ------------------------------------------------------------------ RMSNorm via partials

// After a phase that rewrote rows [r0, r1) of x: publish this CTA's sum of
// x^2 over those rows into ss_part[buf][blockIdx.x].  All compute threads.
__device__ __forceinline__ void publish_ss(const StepArgs &a, const float *xv, int64_t r0, int64_t r1,
                                           int buf, float *red, int tid) {
  float ss = 0.f;
  for (int64_t r = r0 + tid; r < r1; r += kGemvConsumers) ss = fmaf(xv[r - r0], xv[r - r0], ss);
  ss = warp_sum(ss);
  if ((tid & 31) == 0) red[32 + (tid >> 5)] = ss;
  gemv_sync();
  if (tid == 0) {
    float t = 0.f;
    for (int w = 0; w < kGemvWarps; ++w) t += red[32 + w];
    a.ss_part[buf * gridDim.x + blockIdx.x] = t;
  }
}

// Activation slice of RMSNorm(x) * w for the next phase: the lane's raw
// columns and the published partial sums are fetched together (one round
// trip), then scaled.  All compute threads; ends synced.
template <typename T, int NV>
__device__ __forceinline__ void norm_slice(const StepArgs &a, XSlice<T, NV> &xs, const float *w,
                                           const Geom &g, int buf, float *red, int warp, int lane) {
  load_slice(xs, a.x, 1.0f, w, g, warp, lane);
  if (warp == 0) {
    const int G = gridDim.x;
    float t = 0.f;
    for (int base = lane; base < G; base += 256) {
      float v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int i = base + 32 * j;
        v[j] = __ldcg(a.ss_part + buf * G + (i < G ? i : 0));
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) t += base + 32 * j < G ? v[j] : 0.f;
    }
    t = warp_sum(t);
    if (lane == 0) red[0] = t;
  }
  gemv_sync();
  const float inv = 1.0f / sqrtf(red[0] / (float)a.E + a.eps);
#pragma unroll
  for (int t = 0; t < NV; ++t)
#pragma unroll
    for (int e = 0; e < Vec<T>::N / 2; ++e) {
      xs.p[t][e].x *= inv;
      xs.p[t][e].y *= inv;
    }
  gemv_sync();
}

// ------------------------------------------------------------------ kernel

template <typename T, int HD, int G>
__global__ void __launch_bounds__(kStepThreads, 1) k_step(const StepArgs a) {
  constexpr int NV = 4;
  const StepSmem SL = step_smem(a.nslots, a.slot_bytes, a.union_floats);
  uint8_t *ring = g_smem + SL.ring;
  float *uni = reinterpret_cast<float *>(g_smem + SL.uni);
  float *qs = reinterpret_cast<float *>(g_smem + SL.qs);
  float *red = reinterpret_cast<float *>(g_smem + SL.red);
  StepShared &sh = *reinterpret_cast<StepShared *>(g_smem + SL.sh);
  uint64_t *full = reinterpret_cast<uint64_t *>(g_smem + SL.bars);
  uint64_t *empty = full + a.nslots;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
  if (tid == 0) {
    if (a.trace) a.trace[((size_t)blockIdx.x * (5 * a.L + 1) + 5 * a.L) * 6 + 1] = global_ns();
    for (int s = 0; s < a.nslots; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kGemvWarps);
    }
    fence_barrier_init();
    sh.gen0 = ld_acquire_u32(a.bar_gen);
    sh.pos = a.io->pos;
    sh.token = a.io->token;
    sh.route = 0;
    sh.issued = 0;
  }
  __syncthreads();
  const int pos = sh.pos;
  const bool moe = a.X > 0;
  const int kk = moe ? a.k : 1;
  const int qkv_rows = (a.H + 2 * a.Hkv) * a.hd;

  // ------------------------------------------------ producer (16) / prefetcher (17)
  if (warp >= kGemvWarps) {
    if (lane == 0) {
      RingP R{ring, full, empty, a.nslots, a.slot_bytes, 0u,
              RingPos{0u, 0u, (uint32_t)a.nslots}, true, &a.io->error, &sh.issued,
              warp == kGemvWarps + 1};
      unsigned nbar = 0;
      for (int l = 0; l < a.L; ++l) {
        const StepLayer &ly = a.layers[l];
        const void *w1[1];
        w1[0] = ly.wqkv;
        prod_gemv(R, a.g_qkv, 1, w1, qkv_rows, false, 2);
        trace_mark(a, nbar, 2);
        ++nbar;
        prod_attn<T, HD>(R, a, ly, pos, sh.gen0, nbar);
        trace_mark(a, nbar, 2);
        ++nbar;
        w1[0] = ly.wo;
        prod_gemv(R, a.g_o, 1, w1, a.E, false, 1);
        trace_mark(a, nbar, 2);
        ++nbar;
        const void *wg[kMaxSegments], *wd[kMaxSegments];
        if (moe) {
          // the compute warps publish this layer's routing in shared memory
          const unsigned long long t0 = global_ns();
          for (uint32_t it = 0; sh.route != l + 1; ++it) {
            if ((it & 255u) == 255u &&
                (global_ns() - t0 > kWaitLimitNs || ld_volatile_i32(a.abort_flag))) {
              R.ok = false;
              if (!R.prefetch) set_error(&a.io->error, kErrTimeout);
              break;
            }
          }
          __threadfence_block();
          for (int i = 0; i < kk; ++i) {
            const int e = (R.ok && sh.route == l + 1) ? sh.eidx[i] : 0;
            wg[i] = ly.tab_gate_up[e];
            wd[i] = ly.tab_down[e];
          }
        } else {
          wg[0] = ly.w_gate_up;
          wd[0] = ly.w_down;
        }
        prod_gemv(R, a.g_gu, kk, wg, 2 * (int64_t)a.F, false, 2);
        trace_mark(a, nbar, 2);
        ++nbar;
        prod_gemv(R, a.g_dn, kk, wd, a.E, true, 1);
        trace_mark(a, nbar, 2);
        ++nbar;
      }
      const void *w1[1] = {a.output};
      prod_gemv(R, a.g_lm, 1, w1, a.V, false, 1);
      trace_mark(a, nbar, 2);
      R.drain();
    }
    return;
  }

  // ------------------------------------------------------------ compute warps
  RingC R{ring, full, empty, a.nslots, a.slot_bytes, RingPos{0u, 0u, (uint32_t)a.nslots}, true,
          &a.io->error, 0ull, a.trace != nullptr && tid == 0, 0ull, 0ull, 0ull};
  XSlice<T, NV> xs;
  unsigned nbar = 0;
  int64_t r0;
  int tok = sh.token;
  if (tok < 0 || tok >= a.V) {
    if (tid == 0 && blockIdx.x == 0) set_error(&a.io->error, kErrToken);
    tok = 0;
  }
  const int slot = pos % a.cap;
  for (int l = 0; l < a.L; ++l) {
    const StepLayer &ly = a.layers[l];
    // ---- QKV: RMSNorm (of the embedding row in layer 0), Wqkv, RoPE, cache append
    if (l == 0) {
      const T *row = static_cast<const T *>(a.tok_embd) + (int64_t)tok * a.E;
      const float inv = rms_inv(row, a.E, a.eps, red, tid);
      if (blockIdx.x == 0)
        for (int i = tid * 2; i < a.E; i += kGemvConsumers * 2)
          *reinterpret_cast<float2 *>(a.x + i) = load2(row, i);
      load_slice(xs, row, inv, ly.attn_norm, a.g_qkv, warp, lane);
    } else {
      norm_slice(a, xs, ly.attn_norm, a.g_qkv, 1, red, warp, lane);
    }
    cons_gemv<T, NV>(R, a.g_qkv, 1, qkv_rows, false, 2, xs, uni, warp, lane, &r0, [](int) {});
    gemv_sync();
    {
      int64_t rr0, rr1;
      row_range(qkv_rows, 2, &rr0, &rr1);
      const int hd = a.hd, qrows = a.H * hd, krows = a.Hkv * hd;
      for (int64_t r = rr0 + 2 * tid; r < rr1; r += 2 * kGemvConsumers) {
        const int loc = (int)(r - rr0), rr = (int)r;
        float v0 = row_total(uni, loc, a.g_qkv.cw), v1 = row_total(uni, loc + 1, a.g_qkv.cw);
        if (rr < qrows + krows) {
          float sn, cs;
          rope_sincos(pos, a.inv_freq[(rr % hd) >> 1], &sn, &cs);
          const float t0 = v0 * cs - v1 * sn, t1 = v0 * sn + v1 * cs;
          v0 = t0;
          v1 = t1;
        }
        if (rr < qrows) {
          a.q[rr] = v0;
          a.q[rr + 1] = v1;
        } else {
          const bool is_k = rr < qrows + krows;
          const int k = rr - qrows - (is_k ? 0 : krows);
          const int gk = k / hd, d = k - gk * hd;
          T *dst = static_cast<T *>(is_k ? ly.kc : ly.vc) + ((int64_t)gk * a.cap + slot) * hd + d;
          Elem<T>::store(dst, 0, v0);
          Elem<T>::store(dst, 1, v1);
        }
      }
    }
    grid_barrier(a, sh, ++nbar, R);

    // ---- attention
    cons_attn<T, HD, G>(R, a, pos, uni, qs, sh, warp, lane, tid);
    grid_barrier(a, sh, ++nbar, R);

    // ---- output projection + residual
    load_slice(xs, a.o, 1.0f, nullptr, a.g_o, warp, lane);
    cons_gemv<T, NV>(R, a.g_o, 1, a.E, false, 1, xs, uni, warp, lane, &r0, [](int) {});
    gemv_sync();
    {
      int64_t rr0, rr1;
      row_range(a.E, 1, &rr0, &rr1);
      for (int64_t r = rr0 + tid; r < rr1; r += kGemvConsumers)
        a.x[r] = __ldcg(a.x + r) + row_total(uni, (int)(r - rr0), a.g_o.cw);
      gemv_sync();
      publish_ss(a, a.x + rr0, rr0, rr1, 0, red, tid);
    }
    grid_barrier(a, sh, ++nbar, R);

    // ---- FFN: RMSNorm, (router,) gate/up, SwiGLU
    norm_slice(a, xs, ly.ffn_norm, a.g_gu, 0, red, warp, lane);
    const float inv = 1.0f / sqrtf(red[0] / (float)a.E + a.eps);
    if (moe) {
      // every CTA routes for itself (same inputs, same arithmetic, same choice)
      for (int e = warp; e < a.X; e += kGemvWarps) {
        const T *wr = static_cast<const T *>(ly.w_router) + (int64_t)e * a.E;
        float acc = 0.f;
        for (int i = lane * 2; i < a.E; i += 64) {
          const float2 wv = load2(wr, i), xv = load2(a.x, i), nv = load2(ly.ffn_norm, i);
          acc = fmaf(wv.x, xv.x * inv * nv.x, acc);
          acc = fmaf(wv.y, xv.y * inv * nv.y, acc);
        }
        acc = warp_sum(acc);
        if (lane == 0) sh.rlog[e] = acc;
      }
      gemv_sync();
      if (tid == 0) {
        float mx = -FLT_MAX;
        for (int i = 0; i < kk; ++i) {
          int best = -1;
          for (int e = 0; e < a.X; ++e) {
            bool taken = false;
            for (int j = 0; j < i; ++j) taken |= (sh.eidx[j] == e);
            if (!taken && (best < 0 || sh.rlog[e] > sh.rlog[best])) best = e;
          }
          sh.eidx[i] = best;
          mx = fmaxf(mx, sh.rlog[best]);
        }
        float z = 0.f;
        for (int i = 0; i < kk; ++i) z += expf(sh.rlog[sh.eidx[i]] - mx);
        for (int i = 0; i < kk; ++i) sh.gate[i] = expf(sh.rlog[sh.eidx[i]] - mx) / z;
        __threadfence_block();
        sh.route = l + 1;
      }
      gemv_sync();
    }
    cons_gemv<T, NV>(R, a.g_gu, kk, 2 * (int64_t)a.F, false, 2, xs, uni, warp, lane, &r0, [](int) {});
    gemv_sync();
    {
      int64_t rr0, rr1;
      row_range(kk * 2 * (int64_t)a.F, 2, &rr0, &rr1);
      for (int64_t r = rr0 + 2 * tid; r < rr1; r += 2 * kGemvConsumers) {
        const int loc = (int)(r - rr0);
        const int seg = (int)(r / (2 * (int64_t)a.F));
        const int i = (int)((r - seg * 2 * (int64_t)a.F) >> 1);
        const float gte = row_total(uni, loc, a.g_gu.cw), up = row_total(uni, loc + 1, a.g_gu.cw);
        a.h[(int64_t)seg * a.F + i] = silu(gte) * up;
      }
    }
    grid_barrier(a, sh, ++nbar, R);

    // ---- down projection(s) + residual
    load_slice(xs, a.h, 1.0f, nullptr, a.g_dn, warp, lane);
    cons_gemv<T, NV>(R, a.g_dn, kk, a.E, true, 1, xs, uni, warp, lane, &r0, [&](int seg) {
      load_slice(xs, a.h + (int64_t)seg * a.F, 1.0f, nullptr, a.g_dn, warp, lane);
    });
    gemv_sync();
    {
      int64_t rr0, rr1;
      row_range(a.E, 1, &rr0, &rr1);
      for (int64_t r = rr0 + tid; r < rr1; r += kGemvConsumers) {
        float acc = 0.f;
        for (int s = 0; s < kk; ++s)
          acc = fmaf(moe ? sh.gate[s] : 1.0f,
                     row_total(uni + s * a.g_dn.rows_cta_max * a.g_dn.cw, (int)(r - rr0), a.g_dn.cw), acc);
        a.x[r] = __ldcg(a.x + r) + acc;
      }
      gemv_sync();
      publish_ss(a, a.x + rr0, rr0, rr1, 1, red, tid);
    }
    grid_barrier(a, sh, ++nbar, R);
  }

  // ---- final RMSNorm, LM head, greedy token, pos += 1
  {
    norm_slice(a, xs, a.out_norm, a.g_lm, 1, red, warp, lane);
    cons_gemv<T, NV>(R, a.g_lm, 1, a.V, false, 1, xs, uni, warp, lane, &r0, [](int) {});
    gemv_sync();
    int64_t rr0, rr1;
    row_range(a.V, 1, &rr0, &rr1);
    float best = -FLT_MAX;
    int bi = INT_MAX;
    for (int64_t r = rr0 + tid; r < rr1; r += kGemvConsumers) {
      const float v = row_total(uni, (int)(r - rr0), a.g_lm.cw);
      if (a.logits) a.logits[r] = v;
      argmax_merge(best, bi, v, (int)r);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
      argmax_merge(best, bi, __shfl_xor_sync(0xffffffffu, best, off), __shfl_xor_sync(0xffffffffu, bi, off));
    int *redi = reinterpret_cast<int *>(red + 32);
    if (lane == 0) {
      red[warp] = best;
      redi[warp] = bi;
    }
    gemv_sync();
    if (tid == 0) {
      trace_mark(a, 5 * a.L, 0);
      trace_add_wait(a, 5 * a.L, R.waited_ns);
      for (int w = 1; w < kGemvWarps; ++w) argmax_merge(best, bi, red[w], redi[w]);
      a.lm_val[blockIdx.x] = best;
      a.lm_idx[blockIdx.x] = bi;
      __threadfence();
      const unsigned prev = atomicAdd(a.lm_cnt, 1u);
      sh.flag = prev == gridDim.x - 1;
    }
    gemv_sync();
    if (sh.flag && warp == 0) {
      // the last CTA merges every CTA's candidate: one warp, loads in flight
      __threadfence();
      const int G = gridDim.x;
      float fv = -FLT_MAX;
      int fi = INT_MAX;
      for (int base = lane; base < G; base += 256) {
        float v[8];
        int ix[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int b = base + 32 * j < G ? base + 32 * j : 0;
          v[j] = __ldcg(a.lm_val + b);
          ix[j] = __ldcg(a.lm_idx + b);
        }
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (base + 32 * j < G) argmax_merge(fv, fi, v[j], ix[j]);
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1)
        argmax_merge(fv, fi, __shfl_xor_sync(0xffffffffu, fv, off), __shfl_xor_sync(0xffffffffu, fi, off));
      if (lane == 0) {
        if (fi < 0 || fi >= a.V) {
          set_error(&a.io->error, kErrToken);
          fi = 0;
        }
        if (a.argmax_out) *a.argmax_out = fi;
        a.io->token = fi;
        a.io->pos = pos + 1;
        *a.lm_cnt = 0u;
      }
    }
  }
}

}  // namespace pnb
