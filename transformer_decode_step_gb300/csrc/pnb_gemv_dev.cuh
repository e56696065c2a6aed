// pnb_gemv_dev.cuh - device building blocks of the weight-streaming kernels:
// ring item enumeration, the producer loops, register slices of the
// activation vector, RMSNorm factor, row dot products, RoPE angles.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <float.h>
#include <limits.h>
#include <math.h>

#include <type_traits>

#include "pnb_kernels.cuh"

namespace pnb {

extern __shared__ __align__(128) uint8_t g_smem[];

__device__ __forceinline__ void gemv_sync() { consumer_sync<kGemvConsumers>(); }

struct Item {
  int seg;       // segment (matrix) index
  int64_t row;   // first row inside the segment
  int n;         // rows in this ring slot
  int local;     // first row relative to the CTA's range
};

// Ring items of the CTA's rows [r0, r1): whole-row runs inside one segment, at
// most rows_per_stage rows each.  Summed mode walks the range once per segment.
// Incremental: one division when constructed, none per item.
struct ItemIter {
  int64_t r0, r1, rows, r, seg_base;
  int nseg, rps, seg;
  bool summed;
  __device__ __forceinline__ ItemIter(int64_t r0_, int64_t r1_, int64_t rows_, int nseg_,
                                      bool summed_, int rps_)
      : r0(r0_), r1(r1_), rows(rows_), r(r0_), nseg(nseg_), rps(rps_), seg(0), summed(summed_) {
    if (!summed && r0 < r1) seg = (int)(r0 / rows);
    seg_base = summed ? 0 : (int64_t)seg * rows;
  }
  __device__ __forceinline__ bool next(Item &it) {
    if (r0 >= r1) return false;
    if (summed) {
      if (r >= r1) {
        ++seg;
        r = r0;
      }
      if (seg >= nseg) return false;
      const int n = (int)((int64_t)rps < r1 - r ? (int64_t)rps : r1 - r);
      it.seg = seg;
      it.row = r;
      it.n = n;
      it.local = (int)(r - r0);
      r += n;
      return true;
    }
    if (r >= r1) return false;
    if (r >= seg_base + rows) {
      ++seg;
      seg_base += rows;
    }
    int64_t n64 = (int64_t)rps < r1 - r ? (int64_t)rps : r1 - r;
    if (seg_base + rows - r < n64) n64 = seg_base + rows - r;
    it.seg = seg;
    it.row = r - seg_base;
    it.n = (int)n64;
    it.local = (int)(r - r0);
    r += n64;
    return true;
  }
};

// Position in a ring of n slots: slot index and the parity of its current use.
struct RingPos {
  uint32_t slot, phase, n;
  __device__ __forceinline__ void advance() {
    if (++slot == n) {
      slot = 0;
      phase ^= 1u;
    }
  }
};

struct Ctx {
  uint8_t *ring;
  float *part, *red;
  float2 *rope;
  int *info, *items;
  uint64_t *full, *empty;
  int64_t r0, r1;
};

// Carve shared memory, compute the CTA's row range, initialise the ring barriers.
__device__ __forceinline__ Ctx gemv_setup(const Geom &g, int64_t total_rows) {
  const SmemLayout L = smem_layout(g);
  Ctx c;
  c.ring = g_smem + L.ring;
  c.part = reinterpret_cast<float *>(g_smem + L.part);
  c.red = reinterpret_cast<float *>(g_smem + L.red);
  c.info = reinterpret_cast<int *>(g_smem + L.info);
  c.items = reinterpret_cast<int *>(g_smem + L.items);
  c.rope = reinterpret_cast<float2 *>(g_smem + L.rope);
  c.full = reinterpret_cast<uint64_t *>(g_smem + L.bars);
  c.empty = c.full + g.nstages;
  const int64_t units = total_rows / g.row_align;
  c.r0 = units * blockIdx.x / gridDim.x * g.row_align;
  c.r1 = units * (blockIdx.x + 1) / gridDim.x * g.row_align;
  if (threadIdx.x == 0) {
    for (int s = 0; s < g.nstages; ++s) {
      mbar_init(&c.full[s], 1);
      mbar_init(&c.empty[s], kGemvWarps);
    }
    fence_barrier_init();
  }
  __syncthreads();
  return c;
}

// Before issuing copy i, wait until copy i - inflight has landed: a producer
// keeps only what saturates its share of HBM in flight, so that the
// activation loads of this and the neighbouring kernels do not queue behind a
// whole ring of weight requests.
__device__ __forceinline__ bool inflight_wait(const Geom &g, const Ctx &c, uint32_t i) {
  if (i < (uint32_t)g.inflight) return true;
  const uint32_t j = i - (uint32_t)g.inflight;
  return mbar_wait(&c.full[j % (uint32_t)g.nstages], (j / (uint32_t)g.nstages) & 1u);
}

// Producer: stream the CTA's rows.  With `prefetch`, the first ring's worth is
// issued before griddepcontrol.wait (weights do not depend on earlier kernels).
// Always ends by waiting (bounded) for its last copies to land.
__device__ __forceinline__ void produce(const Geom &g, const Segs &s, bool summed, bool prefetch, const Ctx &c,
                        int32_t *err, const KTrace &tr) {
  bool waited = false;
  if (!prefetch) {
    pdl_wait();
    pdl_trigger();
    waited = true;
  }
  const void *w[kMaxSegments];
  for (int i = 0; i < s.n; ++i) w[i] = s.table ? s.table[s.expert_idx[i]] : s.w[i];
  ItemIter it(c.r0, c.r1, s.rows, s.n, summed, g.rows_per_stage);
  Item item;
  uint32_t i = 0;
  RingPos rp{0u, 0u, (uint32_t)g.nstages};
  bool ok = true;
  while (it.next(item)) {
    if (!waited && i == (uint32_t)g.nstages) {
      ktrace(tr, 6);
      pdl_wait();
      pdl_trigger();
      ktrace(tr, 7);
      waited = true;
    }
    if (!inflight_wait(g, c, i) ||
        (i >= (uint32_t)g.nstages && !mbar_wait(&c.empty[rp.slot], rp.phase ^ 1u))) {
      ok = false;
      break;
    }
    const uint32_t bytes = (uint32_t)item.n * (uint32_t)g.row_bytes;
    mbar_arrive_expect_tx(&c.full[rp.slot], bytes);
    bulk_g2s(c.ring + rp.slot * (uint32_t)g.stage_bytes,
             static_cast<const uint8_t *>(w[item.seg]) + item.row * g.row_bytes, bytes,
             &c.full[rp.slot]);
    ++i;
    rp.advance();
  }
  if (!waited) {
    ktrace(tr, 6);
    pdl_wait();
    pdl_trigger();
    ktrace(tr, 7);
  }
  if (!ok) set_error(err, kErrTimeout);
  // wait for the copies still in flight: the last min(i, nstages) items
  const uint32_t last = i < (uint32_t)g.nstages ? i : (uint32_t)g.nstages;
  RingPos dp = rp;
  for (uint32_t j = 0; j < last; ++j) {
    if (dp.slot == 0) {
      dp.slot = dp.n;
      dp.phase ^= 1u;
    }
    --dp.slot;
    if (!mbar_wait(&c.full[dp.slot], dp.phase)) set_error(err, kErrTimeout);
  }
}

// ------------------------------------------------------- dynamic claiming
//
// Ring items (rows_per_stage rows of one segment) are numbered over all
// segments.  The first n_static_total items are split evenly over the CTAs
// and streamed first; the rest (when there are any) are claimed one at a time
// from the launch's work[0] counter (four claims in flight, issued while the
// static share streams), so CTAs that started late or stream slowly take
// fewer.  A CTA takes at most cap_items.  The slot info tells consumers the
// item's row count and CTA-local index; a row count of -1 ends the stream.  Once its claims
// have returned, each CTA counts itself in work[1]; the last one puts both
// counters back to zero for the next launch.

// (32-bit arithmetic: a segment has fewer than 2^31 rows; 64-bit divisions
// are emulated and cost the epilogues, which run on the kernel's tail)
__device__ __forceinline__ void item_rows(const Geom &g, int64_t rows, int item, int &seg,
                                          int64_t &row0, int &n) {
  const int rows32 = (int)rows, rps = g.rows_per_stage;
  const int ips = (rows32 + rps - 1) / rps;
  seg = item / ips;
  const int r0 = (item - seg * ips) * rps;
  row0 = r0;
  n = rps < rows32 - r0 ? rps : rows32 - r0;
}

__device__ __forceinline__ void finish_claims(unsigned *work) {
  __threadfence();
  const unsigned prev = atomicAdd(work + 1, 1u);
  if (prev == gridDim.x - 1) {
    __threadfence();
    atomicExch(work, 0u);
    atomicExch(work + 1, 0u);
  }
}

__device__ __forceinline__ void produce_dyn(const Geom &g, const Segs &s, bool prefetch, const Ctx &c,
                                            unsigned *work, int32_t *err, const KTrace &tr) {
  constexpr int D = 4;
  bool waited = false;
  if (!prefetch) {
    pdl_wait();
    pdl_trigger();
    waited = true;
  }
  const void *w[kMaxSegments];
  for (int i = 0; i < s.n; ++i) w[i] = s.table ? s.table[s.expert_idx[i]] : s.w[i];
  const int cap = g.cap_items;
  // static share: a balanced split of the static items; the rest are claimed
  const unsigned base = g.n_static_total;                           // first claimed item
  const unsigned pool = (unsigned)g.n_items - base;                 // claimable items
  const int s0 = (int)((int64_t)base * blockIdx.x / gridDim.x);
  const int n_own = (int)((int64_t)base * (blockIdx.x + 1) / gridDim.x) - s0;
  int k = 0;                 // items taken
  uint32_t i = 0;            // copies issued
  RingPos rp{0u, 0u, (uint32_t)g.nstages};
  bool ok = true;
  // one item: wait for room, publish the slot info, issue the copy
  auto issue = [&](int item) {
    if (!waited && i == (uint32_t)g.nstages) {
      ktrace(tr, 6);
      pdl_wait();
      pdl_trigger();
      ktrace(tr, 7);
      waited = true;
    }
    if (!inflight_wait(g, c, i) ||
        (i >= (uint32_t)g.nstages && !mbar_wait(&c.empty[rp.slot], rp.phase ^ 1u))) {
      ok = false;
      return;
    }
    int seg, n;
    int64_t row0;
    item_rows(g, s.rows, item, seg, row0, n);
    c.info[2 * rp.slot] = n;
    c.info[2 * rp.slot + 1] = k;
    c.items[k] = item;
    ++k;
    const uint32_t bytes = (uint32_t)n * (uint32_t)g.row_bytes;
    mbar_arrive_expect_tx(&c.full[rp.slot], bytes);
    bulk_g2s(c.ring + rp.slot * (uint32_t)g.stage_bytes,
             static_cast<const uint8_t *>(w[seg]) + row0 * g.row_bytes, bytes, &c.full[rp.slot]);
    ++i;
    rp.advance();
  };
  // claims for the shared tail go out first; their results are needed only
  // once the static share has been issued.  pending counts claims whose
  // items would still fit under the cap.
  unsigned q[D];
  int pending = 0;
#pragma unroll
  for (int d = 0; d < D; ++d) {
    if (pool > 0 && n_own + pending < cap) {
      q[d] = atomicAdd(work, 1u);
      ++pending;
    } else {
      q[d] = pool;
    }
  }
  for (int j = 0; j < n_own && ok; ++j) issue(s0 + j);
  bool more = ok && pool > 0;
  while (more) {
#pragma unroll
    for (int d = 0; d < D; ++d) {
      if (!more) continue;
      if (q[d] >= pool || !ok) {   // claims return in order: every later one fails too
        more = false;
        continue;
      }
      issue((int)(base + q[d]));
      --pending;
      if (ok && k + pending + 1 <= cap) {
        q[d] = atomicAdd(work, 1u);
        ++pending;
      } else {
        q[d] = pool;
      }
    }
  }
  if (!waited) {
    ktrace(tr, 6);
    pdl_wait();
    pdl_trigger();
    ktrace(tr, 7);
  }
  // end of stream, as soon as the last item is out: the end slot's previous
  // copy has landed once the consumers have released it
  if (ok && i >= (uint32_t)g.nstages && !mbar_wait(&c.empty[rp.slot], rp.phase ^ 1u)) ok = false;
  if (ok) {
    c.items[cap] = k;
    c.info[2 * rp.slot] = -1;
    mbar_arrive(&c.full[rp.slot]);
  }
  // wait for the other copies still in flight (the CTA must not end before
  // they land, should its consumers give up early)
  const uint32_t last = i < (uint32_t)g.nstages - 1u ? i : (uint32_t)g.nstages - 1u;
  RingPos dp = rp;
  for (uint32_t j = 0; j < last; ++j) {
    if (dp.slot == 0) {
      dp.slot = dp.n;
      dp.phase ^= 1u;
    }
    --dp.slot;
    if (!mbar_wait(&c.full[dp.slot], dp.phase)) ok = false;
  }
  if (!ok) set_error(err, kErrTimeout);
  // every claim has returned (the comparison waits for the values): count this
  // CTA out of the launch's claiming
  unsigned all = 0xffffffffu;
#pragma unroll
  for (int d = 0; d < D; ++d) all &= q[d];
  if (all == 0xfffffffeu) set_error(err, kErrTimeout);
  if (pool > 0) finish_claims(work);
}

// ------------------------------------------------------- activation slices

// elements per 16-byte weight vector
template <typename T>
struct Vec;
template <>
struct Vec<__nv_bfloat16> {
  static constexpr int N = 8;
};
template <>
struct Vec<float> {
  static constexpr int N = 4;
};
template <>
struct Vec<Q8> {
  static constexpr int N = 8;   // 8-byte vectors of int8 values (the row's fp16 scales follow)
};
template <>
struct Vec<Q4> {
  static constexpr int N = 8;   // 4-byte vectors of 4-bit codes (the row's fp16 scales follow)
};

// A lane's slice of the activation vector: for t < NV, the Vec<T>::N columns
// of 16-byte vector v(t) = c*32 + lane + t*32*cw (c = the warp's column slot),
// as fp32 pairs.
template <typename T, int NV>
struct XSlice {
  float2 p[NV][Vec<T>::N / 2];
};

__device__ __forceinline__ float2 load2(const float *src, int col) {
  return __ldcg(reinterpret_cast<const float2 *>(src + col));
}
__device__ __forceinline__ float2 load2(const __nv_bfloat16 *src, int col) {
  return bf16x2_to_float2(*reinterpret_cast<const uint32_t *>(src + col));
}

// One Q8 row (the embedding row of a token): values at p, scales at p + K.
struct Q8Row {
  const uint8_t *p;
  int K;
};

__device__ __forceinline__ float2 load2(const Q8Row *src, int col) {
  const int8_t *v = reinterpret_cast<const int8_t *>(src->p);
  const float d = __half2float(reinterpret_cast<const __half *>(src->p + src->K)[col / 32]);
  return make_float2(d * (float)v[col], d * (float)v[col + 1]);
}

// One Q4 row (the embedding row of a token): codes at p, scales at p + K / 2.
struct Q4Row {
  const uint8_t *p;
  int K;
};

__device__ __forceinline__ float2 load2(const Q4Row *src, int col) {
  const uint32_t b = src->p[col >> 1];   // col even: codes col (low nibble) and col + 1
  const float d = __half2float(reinterpret_cast<const __half *>(src->p + src->K / 2)[col / 32]);
  return make_float2(d * (float)((int)(b & 15u) - 8), d * (float)((int)(b >> 4) - 8));
}

// The N consecutive source columns [col, col + N) of one weight vector as fp32
// pairs.  An fp32 source comes in 16-byte loads: the lanes of a warp sit one
// vector (4 or 8 columns) apart, so 8-byte loads would fetch every sector of
// the vector from L2 two or four times over.  col is a multiple of N, and the
// vectors are 16-byte aligned.
template <int N, typename S>
__device__ __forceinline__ void load_cols(const S *src, int col, float2 (&o)[N / 2]) {
#pragma unroll
  for (int e = 0; e < N / 2; ++e) o[e] = load2(src, col + 2 * e);
}
template <int N>
__device__ __forceinline__ void load_cols(const float *src, int col, float2 (&o)[N / 2]) {
  static_assert(N % 4 == 0, "whole 16-byte vectors");
#pragma unroll
  for (int j = 0; j < N / 4; ++j) {
    const float4 v = __ldcg(reinterpret_cast<const float4 *>(src + col) + j);
    o[2 * j] = make_float2(v.x, v.y);
    o[2 * j + 1] = make_float2(v.z, v.w);
  }
}
template <int N>
__device__ __forceinline__ void load_cols(const __nv_bfloat16 *src, int col, float2 (&o)[N / 2]) {
  if constexpr (N == 8) {
    const uint4 u = *reinterpret_cast<const uint4 *>(src + col);
    o[0] = bf16x2_to_float2(u.x);
    o[1] = bf16x2_to_float2(u.y);
    o[2] = bf16x2_to_float2(u.z);
    o[3] = bf16x2_to_float2(u.w);
  } else {
#pragma unroll
    for (int e = 0; e < N / 2; ++e) o[e] = load2(src, col + 2 * e);
  }
}

// xs = src * scale * w (w optional), columns of this lane only.  Every load
// is issued (from an always-valid address) before any is used, so the lane
// pays one memory round trip, not one per vector.
template <typename T, int NV, typename S>
__device__ __forceinline__ void load_slice(XSlice<T, NV> &xs, const S *src, float scale,
                                           const float *w, const Geom &g, int warp, int lane) {
  constexpr int P = Vec<T>::N / 2;
  const int vpr = g.vpr, c = warp % g.cw;
  float2 xv[NV][P], wv[NV][P];
#pragma unroll
  for (int t = 0; t < NV; ++t) {
    const int v = c * 32 + lane + t * 32 * g.cw;
    const int vc = v < vpr ? v : 0;
    load_cols<Vec<T>::N>(src, vc * Vec<T>::N, xv[t]);
    if (w) {
      load_cols<Vec<T>::N>(w, vc * Vec<T>::N, wv[t]);
    } else {
#pragma unroll
      for (int e = 0; e < P; ++e) wv[t][e] = make_float2(1.f, 1.f);
    }
  }
#pragma unroll
  for (int t = 0; t < NV; ++t) {
    const bool valid = c * 32 + lane + t * 32 * g.cw < vpr;
#pragma unroll
    for (int e = 0; e < P; ++e)
      xs.p[t][e] = valid ? make_float2(xv[t][e].x * scale * wv[t][e].x, xv[t][e].y * scale * wv[t][e].y)
                         : make_float2(0.f, 0.f);
  }
}

// 1 / sqrt(mean(src^2) + eps) over E elements; all consumer threads, ends
// synced.  Loads go out eight at a time before they are used.
template <typename S>
__device__ __forceinline__ float rms_inv(const S *src, int E, float eps, float *red, int tid) {
  float ss = 0.f;
  for (int base = tid * 2; base < E; base += kGemvConsumers * 2 * 8) {
    float2 v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int i = base + j * kGemvConsumers * 2;
      v[j] = load2(src, i < E ? i : 0);
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (base + j * kGemvConsumers * 2 < E) {
        ss = fmaf(v[j].x, v[j].x, ss);
        ss = fmaf(v[j].y, v[j].y, ss);
      }
    }
  }
  ss = warp_sum(ss);
  if ((tid & 31) == 0) red[tid >> 5] = ss;
  gemv_sync();
  float tot = 0.f;
  for (int k = 0; k < kGemvWarps; ++k) tot += red[k];
  return 1.0f / sqrtf(tot / (float)E + eps);
}

// ---------------------------------------------------------------- dot products

template <int NV>
__device__ __forceinline__ float dot_row_q8(const uint8_t *row, const XSlice<Q8, NV> &xs, int vpr,
                                            int c, int cw, int lane);
template <int NV>
__device__ __forceinline__ float dot_row_q4(const uint8_t *row, const XSlice<Q4, NV> &xs, int vpr,
                                            int c, int cw, int lane);

template <typename T, int NV>
__device__ __forceinline__ float dot_row(const uint8_t *row, const XSlice<T, NV> &xs, int vpr,
                                         int c, int cw, int lane) {
  if constexpr (std::is_same<T, Q8>::value) {
    return dot_row_q8<NV>(row, xs, vpr, c, cw, lane);
  } else if constexpr (std::is_same<T, Q4>::value) {
    return dot_row_q4<NV>(row, xs, vpr, c, cw, lane);
  } else {
  constexpr int P = Vec<T>::N / 2;
  uint4 wv[NV];
#pragma unroll
  for (int t = 0; t < NV; ++t) {
    const int v = c * 32 + lane + t * 32 * cw;
    wv[t] = *reinterpret_cast<const uint4 *>(row + 16 * (v < vpr ? v : 0));
  }
  float2 acc[P];
#pragma unroll
  for (int e = 0; e < P; ++e) acc[e] = make_float2(0.f, 0.f);
#pragma unroll
  for (int t = 0; t < NV; ++t) {
    if (c * 32 + lane + t * 32 * cw < vpr) {
      const uint4 w = wv[t];
      if constexpr (P == 4) {
        acc[0] = ffma2(bf16x2_to_float2(w.x), xs.p[t][0], acc[0]);
        acc[1] = ffma2(bf16x2_to_float2(w.y), xs.p[t][1], acc[1]);
        acc[2] = ffma2(bf16x2_to_float2(w.z), xs.p[t][2], acc[2]);
        acc[3] = ffma2(bf16x2_to_float2(w.w), xs.p[t][3], acc[3]);
      } else {
        acc[0] = ffma2(make_float2(__uint_as_float(w.x), __uint_as_float(w.y)), xs.p[t][0], acc[0]);
        acc[1] = ffma2(make_float2(__uint_as_float(w.z), __uint_as_float(w.w)), xs.p[t][1], acc[1]);
      }
    }
  }
  float s = 0.f;
#pragma unroll
  for (int e = 0; e < P; ++e) s += acc[e].x + acc[e].y;
  return s;
  }
}

// Q8 rows: each 8-byte vector is 8 int8 values of one quarter of a block of
// 32, scaled once by the block's fp16 scale (stored after the row's K
// values).  A byte permute makes the float 2^23 + (q + 128) of each value
// (the value biased to unsigned, in the low mantissa bits) and one packed FMA
// removes 2^23 + 128 exactly, so each q is exact before it is multiplied.
template <int NV>
__device__ __forceinline__ float dot_row_q8(const uint8_t *row, const XSlice<Q8, NV> &xs, int vpr,
                                            int c, int cw, int lane) {
  uint2 wv[NV];
  float dv[NV];
#pragma unroll
  for (int t = 0; t < NV; ++t) {
    const int v = c * 32 + lane + t * 32 * cw;
    const int vc = v < vpr ? v : 0;
    wv[t] = *reinterpret_cast<const uint2 *>(row + 8 * vc);
    dv[t] = __half2float(reinterpret_cast<const __half *>(row + 8 * vpr)[vc >> 2]);
  }
  const float2 off = make_float2(-8388736.0f, -8388736.0f), one = make_float2(1.f, 1.f);
  float s = 0.f;
#pragma unroll
  for (int t = 0; t < NV; ++t) {
    if (c * 32 + lane + t * 32 * cw < vpr) {
      const uint32_t w2[2] = {wv[t].x ^ 0x80808080u, wv[t].y ^ 0x80808080u};
      float2 acc = make_float2(0.f, 0.f);
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const float2 q0 = ffma2(make_float2(__uint_as_float(__byte_perm(w2[k], 0x4B000000u, 0x7440)),
                                            __uint_as_float(__byte_perm(w2[k], 0x4B000000u, 0x7441))),
                                one, off);
        const float2 q1 = ffma2(make_float2(__uint_as_float(__byte_perm(w2[k], 0x4B000000u, 0x7442)),
                                            __uint_as_float(__byte_perm(w2[k], 0x4B000000u, 0x7443))),
                                one, off);
        acc = ffma2(q0, xs.p[t][2 * k], acc);
        acc = ffma2(q1, xs.p[t][2 * k + 1], acc);
      }
      s = fmaf(acc.x + acc.y, dv[t], s);
    }
  }
  return s;
}

// Q4 rows: each 4-byte vector is 8 codes of one quarter of a block of 32.
// The low and the high nibbles are masked into two words of four bytes, a
// byte permute makes the float 2^23 + u of each code (the code in the low
// mantissa bits) and one packed FMA removes 2^23 + 8 exactly, so each u - 8
// is exact before it multiplies the fp32 activation pair it belongs to; each
// vector is scaled once by its block's fp16 scale.
template <int NV>
__device__ __forceinline__ float dot_row_q4(const uint8_t *row, const XSlice<Q4, NV> &xs, int vpr,
                                            int c, int cw, int lane) {
  uint32_t wv[NV];
  float dv[NV];
#pragma unroll
  for (int t = 0; t < NV; ++t) {
    const int v = c * 32 + lane + t * 32 * cw;
    const int vc = v < vpr ? v : 0;
    wv[t] = *reinterpret_cast<const uint32_t *>(row + 4 * vc);
    dv[t] = __half2float(reinterpret_cast<const __half *>(row + 4 * vpr)[vc >> 2]);
  }
  const float2 off = make_float2(-8388616.0f, -8388616.0f), one = make_float2(1.f, 1.f);
  float s = 0.f;
#pragma unroll
  for (int t = 0; t < NV; ++t) {
    if (c * 32 + lane + t * 32 * cw < vpr) {
      const uint32_t lo = wv[t] & 0x0F0F0F0Fu, hi = (wv[t] >> 4) & 0x0F0F0F0Fu;
      float2 acc = make_float2(0.f, 0.f);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 q = ffma2(make_float2(__uint_as_float(__byte_perm(lo, 0x4B000000u, 0x7440u + k)),
                                           __uint_as_float(__byte_perm(hi, 0x4B000000u, 0x7440u + k))),
                               one, off);
        acc = ffma2(q, xs.p[t][k], acc);
      }
      s = fmaf(acc.x + acc.y, dv[t], s);
    }
  }
  return s;
}

// Warp partials of four rows at once: the lane's products p[i] of rows i are
// summed over the warp with six shuffles (two halving exchanges, then three
// steps over the remaining eight lanes); lanes 8i .. 8i + 7 end with row i.
__device__ __forceinline__ float warp_sum4(float p0, float p1, float p2, float p3, int lane) {
  const bool hi = lane & 16, mid = lane & 8;
  const float a0 = (hi ? p2 : p0) + __shfl_xor_sync(0xffffffffu, hi ? p0 : p2, 16);
  const float a1 = (hi ? p3 : p1) + __shfl_xor_sync(0xffffffffu, hi ? p1 : p3, 16);
  float v = (mid ? a1 : a0) + __shfl_xor_sync(0xffffffffu, mid ? a0 : a1, 8);
  v += __shfl_xor_sync(0xffffffffu, v, 4);
  v += __shfl_xor_sync(0xffffffffu, v, 2);
  v += __shfl_xor_sync(0xffffffffu, v, 1);
  return v;
}

// How a warp shares the staged rows: kGemvWarps / cw row groups of cw warps;
// this warp is column slot cc of row group grp (computed once per kernel).
struct RowSplit {
  int cw, groups, grp, cc, vpr;
  __device__ __forceinline__ RowSplit(int cw_, int vpr_, int warp)
      : cw(cw_), groups(kGemvWarps / cw_), grp(warp / cw_), cc(warp % cw_), vpr(vpr_) {}
};

// Partial sums of the n staged rows at `stage` into part[(base + r) * cw + cc];
// with one row group (cw == 16) and rows short enough that a ring slot holds
// several, the rows go four at a time through warp_sum4.
template <typename T, int NV>
__device__ __forceinline__ void dot_item(const uint8_t *stage, int n, int row_bytes, const XSlice<T, NV> &xs,
                                         float *part, int base, const RowSplit &sp, int lane) {
  const int groups = sp.groups, cc = sp.cc, cw = sp.cw, vpr = sp.vpr;
  int r = sp.grp;
  if constexpr (NV <= 2) {   // rows of at most 16 KB: ring slots hold four or more
   if (groups == 1) {
    for (; r + 4 <= n; r += 4) {
      const uint8_t *rw = stage + (size_t)r * row_bytes;
      const float v = warp_sum4(dot_row<T, NV>(rw, xs, vpr, cc, cw, lane),
                                dot_row<T, NV>(rw + row_bytes, xs, vpr, cc, cw, lane),
                                dot_row<T, NV>(rw + 2 * row_bytes, xs, vpr, cc, cw, lane),
                                dot_row<T, NV>(rw + 3 * row_bytes, xs, vpr, cc, cw, lane), lane);
      if ((lane & 7) == 0) part[(base + r + (lane >> 3)) * cw + cc] = v;
    }
   }
  }
  for (; r < n; r += groups) {
    const float v = warp_sum(dot_row<T, NV>(stage + (size_t)r * row_bytes, xs, vpr, cc, cw, lane));
    if (lane == 0) part[(base + r) * cw + cc] = v;
  }
}

// Consumer loop over the CTA's ring items.  `reload(seg)` refreshes the
// lane's activation slice when a summed launch moves to the next segment.  A
// wait that expires sets the error bit and the warp stops consuming.
template <typename T, int NV, typename Reload>
__device__ __forceinline__ void consume(const Geom &g, const Segs &s, bool summed, const Ctx &c,
                        XSlice<T, NV> &xs, int warp, int lane, int32_t *err, const KTrace &tr,
                        Reload &&reload) {
  const int cw = g.cw;
  const RowSplit sp(cw, g.vpr, warp);
  ItemIter it(c.r0, c.r1, s.rows, s.n, summed, g.rows_per_stage);
  Item item;
  RingPos rp{0u, 0u, (uint32_t)g.nstages};
  int cur = 0;
  bool ok = true;
  while (it.next(item)) {
    if (summed && item.seg != cur) {
      reload(item.seg);
      cur = item.seg;
    }
    const uint32_t slot = rp.slot;
    if (ok && !mbar_wait(&c.full[slot], rp.phase)) {
      ok = false;
      if (lane == 0) set_error(err, kErrTimeout);
    }
    if (tr.p && warp == 0 && lane == 0 && item.local == 0 && item.seg == 0) ktrace(tr, 3);
    if (ok) {
      const uint8_t *stage = c.ring + slot * (uint32_t)g.stage_bytes;
      float *part = c.part + ((summed ? item.seg : 0) * g.rows_cta_max + item.local) * cw;
      dot_item<T, NV>(stage, item.n, g.row_bytes, xs, part, 0, sp, lane);
      __syncwarp();
      if (lane == 0) mbar_arrive(&c.empty[slot]);
    }
    rp.advance();
  }
}

// Consumer loop of a dynamically claimed stream: the rows of the CTA's k-th
// item leave their partial sums in part[(k * rows_per_stage + r) * cw + warp
// column].  Ends at the end-of-stream slot (or a wait that expires).
template <typename T, int NV>
__device__ __forceinline__ void consume_dyn(const Geom &g, const Ctx &c, const XSlice<T, NV> &xs,
                                            int warp, int lane, int32_t *err, const KTrace &tr) {
  const int cw = g.cw;
  const RowSplit sp(cw, g.vpr, warp);
  RingPos rp{0u, 0u, (uint32_t)g.nstages};
  bool first = true;
  for (;;) {
    const uint32_t slot = rp.slot;
    if (!mbar_wait(&c.full[slot], rp.phase)) {
      if (lane == 0) set_error(err, kErrTimeout);
      return;
    }
    if (first && warp == 0 && lane == 0) ktrace(tr, 3);
    first = false;
    const int2 inf = *reinterpret_cast<const int2 *>(c.info + 2 * slot);
    const int n = inf.x, kk = inf.y;
    if (n < 0) return;
    const uint8_t *stage = c.ring + slot * (uint32_t)g.stage_bytes;
    float *part = c.part + (size_t)kk * g.rows_per_stage * cw;
    dot_item<T, NV>(stage, n, g.row_bytes, xs, part, 0, sp, lane);
    __syncwarp();
    if (lane == 0) mbar_arrive(&c.empty[slot]);
    rp.advance();
  }
}

// Rows the CTA took, for the fused epilogues: f(k, r, seg, row) for row r of
// its k-th item (row = the row inside segment seg), spread over the consumer
// threads; with `pairs`, only even r (the pair's first row).
template <typename F>
__device__ __forceinline__ void for_claimed_rows(const Geom &g, const Ctx &c, int64_t rows, bool pairs,
                                                 int tid, F &&f) {
  const int k = c.items[g.cap_items];
  const int rps = g.rows_per_stage, step = pairs ? 2 : 1;
  const int per = rps / step;
  for (int idx = tid; idx < k * per; idx += kGemvConsumers) {
    const int j = idx / per, r = (idx - j * per) * step;
    int seg, n;
    int64_t row0;
    item_rows(g, rows, c.items[j], seg, row0, n);
    if (r < n) f(j, r, seg, row0 + r);
  }
}

// The cw per-warp partial sums of one row (16-byte aligned), added in a fixed
// pairwise order from 16-byte loads: the epilogues run on the kernel's tail,
// where a serial chain of cw dependent shared-memory loads and adds cost
// about 3% of a decode step.
__device__ __forceinline__ float sum_partials(const float *p, int cw) {
  const float4 *q = reinterpret_cast<const float4 *>(p);
  auto s4 = [](float4 v) { return (v.x + v.y) + (v.z + v.w); };
  if (cw == 16) return (s4(q[0]) + s4(q[1])) + (s4(q[2]) + s4(q[3]));
  if (cw == 8) return s4(q[0]) + s4(q[1]);
  if (cw == 4) return s4(q[0]);
  float v = 0.f;
  for (int w = 0; w < cw; ++w) v += p[w];
  return v;
}

__device__ __forceinline__ float item_row_total(const Geom &g, const Ctx &c, int k, int r) {
  return sum_partials(c.part + ((size_t)k * g.rows_per_stage + r) * g.cw, g.cw);
}

// The multiplier slice of an RMSNorm weight (1 without one): weights do not
// depend on earlier kernels, so this is loaded before griddepcontrol.wait
// (the wait holds until such loads return; with one lane per column the
// slice is a few hundred bytes per warp).
template <typename T, int NV>
__device__ __forceinline__ void load_weight_slice(XSlice<T, NV> &ws, const float *w, const Geom &g,
                                                  int warp, int lane) {
  constexpr int P = Vec<T>::N / 2;
  const int vpr = g.vpr, c = warp % g.cw;
#pragma unroll
  for (int t = 0; t < NV; ++t) {
    const int v = c * 32 + lane + t * 32 * g.cw;
    const int vc = v < vpr ? v : 0;
    if (w) {
      load_cols<Vec<T>::N>(w, vc * Vec<T>::N, ws.p[t]);
    } else {
#pragma unroll
      for (int e = 0; e < P; ++e) ws.p[t][e] = make_float2(1.f, 1.f);
    }
  }
}

// xs = RMSNorm(src) * (multiplier already in xs), columns of this lane only,
// with one round trip to memory: the sum of squares comes from the slices of
// the first cw warps, which together hold every element once (every row group
// holds the same columns, so all threads get the same fixed-order total).
template <typename T, int NV, typename S>
__device__ __forceinline__ void norm_slice(XSlice<T, NV> &xs, const S *src, int E, float eps,
                                           const Geom &g, float *red, int warp, int lane) {
  constexpr int P = Vec<T>::N / 2;
  const int vpr = g.vpr, c = warp % g.cw;
  float2 xv[NV][P];
#pragma unroll
  for (int t = 0; t < NV; ++t) {
    const int v = c * 32 + lane + t * 32 * g.cw;
    const int vc = v < vpr ? v : 0;
    load_cols<Vec<T>::N>(src, vc * Vec<T>::N, xv[t]);
  }
  float ss = 0.f;
#pragma unroll
  for (int t = 0; t < NV; ++t) {
    const bool valid = c * 32 + lane + t * 32 * g.cw < vpr;
#pragma unroll
    for (int e = 0; e < P; ++e) {
      if (!valid) xv[t][e] = make_float2(0.f, 0.f);
      ss = fmaf(xv[t][e].x, xv[t][e].x, ss);
      ss = fmaf(xv[t][e].y, xv[t][e].y, ss);
    }
  }
  ss = warp_sum(ss);
  if (lane == 0) red[warp] = ss;
  gemv_sync();
  float tot = 0.f;
  for (int w = 0; w < g.cw; ++w) tot += red[w];
  const float inv = 1.0f / sqrtf(tot / (float)E + eps);
#pragma unroll
  for (int t = 0; t < NV; ++t)
#pragma unroll
    for (int e = 0; e < P; ++e)
      xs.p[t][e] = make_float2(xv[t][e].x * inv * xs.p[t][e].x, xv[t][e].y * inv * xs.p[t][e].y);
}

__device__ __forceinline__ float row_total(const float *part, int local, int cw) {
  return sum_partials(part + local * cw, cw);
}

// sin / cos of pos * inv_freq: the angle is formed and reduced to [-pi, pi]
// in fp64 (two-term Cody-Waite reduction by 2*pi), then evaluated in fp32.
__device__ __forceinline__ void rope_sincos(int pos, double inv_freq, float *s, float *c) {
  const double phi = (double)pos * inv_freq;
  const double k = rint(phi * 0.15915494309189535);  // 1 / (2 pi)
  double r = fma(-k, 6.283185307179586, phi);          // 2 pi, high part
  r = fma(-k, 2.4492935982947064e-16, r);              // 2 pi, low part
  sincosf((float)r, s, c);
}

__device__ __forceinline__ float silu(float z) { return z / (1.0f + expf(-z)); }

__device__ __forceinline__ void argmax_merge(float &v, int &i, float ov, int oi) {
  if (ov > v || (ov == v && oi < i)) {
    v = ov;
    i = oi;
  }
}


}  // namespace pnb
