// pnb_gemv.cu - weight-streaming kernels of the decode step.
//
// One structure serves every projection of the step: a CTA owns a contiguous
// range of output rows; warp 8 (one elected thread) streams those rows, whole,
// through a ring of shared-memory slots with 1-D bulk copies; warps 0-7 wait
// for the previous kernel (griddepcontrol.wait), build the fp32 activation
// vector in shared memory (RMSNorm fused where the step has one), multiply the
// staged rows by it and run the fused epilogue.  Partial sums are combined in
// a fixed order, so results are bitwise reproducible run to run.
#include <cuda_bf16.h>
#include <float.h>
#include <limits.h>
#include <math.h>

#include "pnb_kernels.cuh"

namespace pnb {
namespace {

extern __shared__ __align__(128) uint8_t g_smem[];

struct Item {
  int seg;       // segment (matrix) index
  int64_t row;   // first row inside the segment
  int n;         // rows in this ring slot
  int local;     // first row relative to the CTA's range
};

// Ring items of the CTA's rows [r0, r1): whole-row runs inside one segment, at
// most rows_per_stage rows each.  Summed mode walks the range once per segment.
struct ItemIter {
  int64_t r0, r1, rows, r;
  int nseg, rps, seg;
  bool summed;
  __device__ ItemIter(int64_t r0_, int64_t r1_, int64_t rows_, int nseg_, bool summed_, int rps_)
      : r0(r0_), r1(r1_), rows(rows_), r(r0_), nseg(nseg_), rps(rps_), seg(0), summed(summed_) {}
  __device__ bool next(Item &it) {
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
    const int s = (int)(r / rows);
    const int64_t sr = r - (int64_t)s * rows;
    int64_t n64 = (int64_t)rps < r1 - r ? (int64_t)rps : r1 - r;
    if (rows - sr < n64) n64 = rows - sr;
    const int n = (int)n64;
    it.seg = s;
    it.row = sr;
    it.n = n;
    it.local = (int)(r - r0);
    r += n;
    return true;
  }
};

struct Ctx {
  uint8_t *ring;
  float *xs, *part, *red;
  uint64_t *full, *empty;
  int64_t r0, r1;
};

// Carve shared memory, compute the CTA's row range, initialise the ring barriers.
__device__ Ctx gemv_setup(const Geom &g, int64_t total_rows) {
  const SmemLayout L = smem_layout(g);
  Ctx c;
  c.ring = g_smem + L.ring;
  c.xs = reinterpret_cast<float *>(g_smem + L.xs);
  c.part = reinterpret_cast<float *>(g_smem + L.part);
  c.red = reinterpret_cast<float *>(g_smem + L.red);
  c.full = reinterpret_cast<uint64_t *>(g_smem + L.bars);
  c.empty = c.full + g.nstages;
  const int64_t units = total_rows / g.row_align;
  c.r0 = units * blockIdx.x / gridDim.x * g.row_align;
  c.r1 = units * (blockIdx.x + 1) / gridDim.x * g.row_align;
  if (threadIdx.x == 0) {
    for (int s = 0; s < g.nstages; ++s) {
      mbar_init(&c.full[s], 1);
      mbar_init(&c.empty[s], kConsumerWarps);
    }
    fence_barrier_init();
  }
  __syncthreads();
  return c;
}

// Producer: stream the CTA's rows.  With `prefetch`, the first ring's worth is
// issued before griddepcontrol.wait (weights do not depend on earlier kernels).
// Always ends by waiting (bounded) for its last copies to land.
__device__ void produce(const Geom &g, const Segs &s, bool summed, bool prefetch, const Ctx &c,
                        int32_t *err) {
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
  bool ok = true;
  while (it.next(item)) {
    const uint32_t slot = i % g.nstages, round = i / g.nstages;
    if (!waited && i == (uint32_t)g.nstages) {
      pdl_wait();
      pdl_trigger();
      waited = true;
    }
    if (round > 0 && !mbar_wait(&c.empty[slot], (round - 1) & 1)) {
      ok = false;
      break;
    }
    const uint32_t bytes = (uint32_t)item.n * (uint32_t)g.row_bytes;
    mbar_arrive_expect_tx(&c.full[slot], bytes);
    bulk_g2s(c.ring + (size_t)slot * g.stage_bytes,
             static_cast<const uint8_t *>(w[item.seg]) + item.row * g.row_bytes, bytes,
             &c.full[slot]);
    ++i;
  }
  if (!waited) {
    pdl_wait();
    pdl_trigger();
  }
  if (!ok) set_error(err, kErrTimeout);
  const uint32_t first = i > (uint32_t)g.nstages ? i - g.nstages : 0;
  for (uint32_t j = first; j < i; ++j)
    if (!mbar_wait(&c.full[j % g.nstages], (j / g.nstages) & 1)) set_error(err, kErrTimeout);
}

// ---------------------------------------------------------------- dot products

// acc over 16-byte weight vectors [v0, v1) of one staged row; lane-strided
template <typename T>
__device__ __forceinline__ float dot_range(const uint8_t *row, int v0, int v1, const float *xs,
                                           int lane);

template <>
__device__ __forceinline__ float dot_range<__nv_bfloat16>(const uint8_t *row, int v0, int v1,
                                                          const float *xs, int lane) {
  float a0 = 0.f, a1 = 0.f;
  int v = v0 + lane;
  for (; v + 32 < v1; v += 64) {
    const uint4 w0 = *reinterpret_cast<const uint4 *>(row + 16 * v);
    const uint4 w1 = *reinterpret_cast<const uint4 *>(row + 16 * (v + 32));
    const float *p0 = xs + xpad(8 * v);
    const float *p1 = xs + xpad(8 * (v + 32));
    const float4 x0 = *reinterpret_cast<const float4 *>(p0);
    const float4 x1 = *reinterpret_cast<const float4 *>(p0 + 4);
    const float4 y0 = *reinterpret_cast<const float4 *>(p1);
    const float4 y1 = *reinterpret_cast<const float4 *>(p1 + 4);
    a0 = fmaf(bf16lo(w0.x), x0.x, a0);
    a0 = fmaf(bf16hi(w0.x), x0.y, a0);
    a0 = fmaf(bf16lo(w0.y), x0.z, a0);
    a0 = fmaf(bf16hi(w0.y), x0.w, a0);
    a0 = fmaf(bf16lo(w0.z), x1.x, a0);
    a0 = fmaf(bf16hi(w0.z), x1.y, a0);
    a0 = fmaf(bf16lo(w0.w), x1.z, a0);
    a0 = fmaf(bf16hi(w0.w), x1.w, a0);
    a1 = fmaf(bf16lo(w1.x), y0.x, a1);
    a1 = fmaf(bf16hi(w1.x), y0.y, a1);
    a1 = fmaf(bf16lo(w1.y), y0.z, a1);
    a1 = fmaf(bf16hi(w1.y), y0.w, a1);
    a1 = fmaf(bf16lo(w1.z), y1.x, a1);
    a1 = fmaf(bf16hi(w1.z), y1.y, a1);
    a1 = fmaf(bf16lo(w1.w), y1.z, a1);
    a1 = fmaf(bf16hi(w1.w), y1.w, a1);
  }
  if (v < v1) {
    const uint4 w0 = *reinterpret_cast<const uint4 *>(row + 16 * v);
    const float *p0 = xs + xpad(8 * v);
    const float4 x0 = *reinterpret_cast<const float4 *>(p0);
    const float4 x1 = *reinterpret_cast<const float4 *>(p0 + 4);
    a0 = fmaf(bf16lo(w0.x), x0.x, a0);
    a0 = fmaf(bf16hi(w0.x), x0.y, a0);
    a0 = fmaf(bf16lo(w0.y), x0.z, a0);
    a0 = fmaf(bf16hi(w0.y), x0.w, a0);
    a0 = fmaf(bf16lo(w0.z), x1.x, a0);
    a0 = fmaf(bf16hi(w0.z), x1.y, a0);
    a0 = fmaf(bf16lo(w0.w), x1.z, a0);
    a0 = fmaf(bf16hi(w0.w), x1.w, a0);
  }
  return a0 + a1;
}

template <>
__device__ __forceinline__ float dot_range<float>(const uint8_t *row, int v0, int v1,
                                                  const float *xs, int lane) {
  float a0 = 0.f, a1 = 0.f;
  int v = v0 + lane;
  for (; v + 32 < v1; v += 64) {
    const float4 w0 = *reinterpret_cast<const float4 *>(row + 16 * v);
    const float4 w1 = *reinterpret_cast<const float4 *>(row + 16 * (v + 32));
    const float4 x0 = *reinterpret_cast<const float4 *>(xs + xpad(4 * v));
    const float4 y0 = *reinterpret_cast<const float4 *>(xs + xpad(4 * (v + 32)));
    a0 = fmaf(w0.x, x0.x, a0);
    a0 = fmaf(w0.y, x0.y, a0);
    a0 = fmaf(w0.z, x0.z, a0);
    a0 = fmaf(w0.w, x0.w, a0);
    a1 = fmaf(w1.x, y0.x, a1);
    a1 = fmaf(w1.y, y0.y, a1);
    a1 = fmaf(w1.z, y0.z, a1);
    a1 = fmaf(w1.w, y0.w, a1);
  }
  if (v < v1) {
    const float4 w0 = *reinterpret_cast<const float4 *>(row + 16 * v);
    const float4 x0 = *reinterpret_cast<const float4 *>(xs + xpad(4 * v));
    a0 = fmaf(w0.x, x0.x, a0);
    a0 = fmaf(w0.y, x0.y, a0);
    a0 = fmaf(w0.z, x0.z, a0);
    a0 = fmaf(w0.w, x0.w, a0);
  }
  return a0 + a1;
}

// One ring slot: nrows staged rows -> partial sums part[r * wpr + slice].
template <typename T>
__device__ __forceinline__ void dot_slot(const uint8_t *stage, int nrows, const Geom &g,
                                         const float *xs, float *part, int warp, int lane) {
  const int vpr = g.row_bytes / 16;
  if (g.rows_per_stage >= kConsumerWarps) {
    for (int r = warp; r < nrows; r += kConsumerWarps) {
      const float acc = warp_sum(dot_range<T>(stage + (size_t)r * g.row_bytes, 0, vpr, xs, lane));
      if (lane == 0) part[r * g.wpr] = acc;
    }
  } else {
    const int r = warp / g.wpr, ws = warp - r * g.wpr;
    if (r < nrows) {
      const int v0 = min(vpr, ws * g.chunk), v1 = min(vpr, v0 + g.chunk);
      const float acc = warp_sum(dot_range<T>(stage + (size_t)r * g.row_bytes, v0, v1, xs, lane));
      if (lane == 0) part[r * g.wpr + ws] = acc;
    }
  }
}

// Consumer loop over the CTA's ring items; `reload(seg)` refreshes xs when a
// summed launch moves to the next segment.  A wait that expires sets the
// error bit and the warp stops consuming, but keeps joining the barriers.
template <typename T, typename Reload>
__device__ void consume(const Geom &g, const Segs &s, bool summed, const Ctx &c, int warp, int lane,
                        int32_t *err, Reload &&reload) {
  ItemIter it(c.r0, c.r1, s.rows, s.n, summed, g.rows_per_stage);
  Item item;
  uint32_t i = 0;
  int cur = 0;
  bool ok = true;
  while (it.next(item)) {
    if (summed && item.seg != cur) {
      consumer_sync();
      reload(item.seg);
      consumer_sync();
      cur = item.seg;
    }
    const uint32_t slot = i % g.nstages, round = i / g.nstages;
    if (ok && !mbar_wait(&c.full[slot], round & 1)) {
      ok = false;
      if (lane == 0) set_error(err, kErrTimeout);
    }
    if (ok) {
      dot_slot<T>(c.ring + (size_t)slot * g.stage_bytes, item.n, g, c.xs,
                  c.part + ((summed ? item.seg : 0) * g.rows_cta_max + item.local) * g.wpr, warp,
                  lane);
      __syncwarp();
      if (lane == 0) mbar_arrive(&c.empty[slot]);
    }
    ++i;
  }
}

__device__ __forceinline__ float row_total(const float *part, int local, int wpr) {
  float v = 0.f;
  for (int w = 0; w < wpr; ++w) v += part[local * wpr + w];
  return v;
}

// ------------------------------------------------------- activation vectors

template <typename T>
__device__ __forceinline__ float4 load4(const T *p, int i);
template <>
__device__ __forceinline__ float4 load4<float>(const float *p, int i) {
  return *reinterpret_cast<const float4 *>(p + i);
}
template <>
__device__ __forceinline__ float4 load4<__nv_bfloat16>(const __nv_bfloat16 *p, int i) {
  const uint2 u = *reinterpret_cast<const uint2 *>(p + i);
  return make_float4(bf16lo(u.x), bf16hi(u.x), bf16lo(u.y), bf16hi(u.y));
}

// xs = RMSNorm(src) * w (padded layout); src is the fp32 residual or, when
// emb_row is set, a row of the embedding table (also copied to x_out).
// Called by the 256 consumer threads; ends with a consumer barrier.
template <typename T>
__device__ void load_rmsnorm(float *xs, float *red, const float *x, const T *emb_row,
                             const float *w, int E, float eps, float *x_out, int tid) {
  float ss = 0.f;
  for (int i = tid * 4; i < E; i += kConsumerThreads * 4) {
    const float4 v = emb_row ? load4<T>(emb_row, i) : load4<float>(x, i);
    ss = fmaf(v.x, v.x, ss);
    ss = fmaf(v.y, v.y, ss);
    ss = fmaf(v.z, v.z, ss);
    ss = fmaf(v.w, v.w, ss);
  }
  ss = warp_sum(ss);
  if ((tid & 31) == 0) red[tid >> 5] = ss;
  consumer_sync();
  float tot = 0.f;
  for (int k = 0; k < kConsumerWarps; ++k) tot += red[k];
  const float inv = 1.0f / sqrtf(tot / (float)E + eps);
  for (int i = tid * 4; i < E; i += kConsumerThreads * 4) {
    const float4 v = emb_row ? load4<T>(emb_row, i) : load4<float>(x, i);
    const float4 wn = *reinterpret_cast<const float4 *>(w + i);
    float4 o;
    o.x = v.x * inv * wn.x;
    o.y = v.y * inv * wn.y;
    o.z = v.z * inv * wn.z;
    o.w = v.w * inv * wn.w;
    *reinterpret_cast<float4 *>(xs + xpad(i)) = o;
    if (x_out) *reinterpret_cast<float4 *>(x_out + i) = v;
  }
  consumer_sync();
}

__device__ void load_plain(float *xs, const float *v, int K, int tid) {
  for (int i = tid * 4; i < K; i += kConsumerThreads * 4)
    *reinterpret_cast<float4 *>(xs + xpad(i)) = *reinterpret_cast<const float4 *>(v + i);
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

// ------------------------------------------------------------------ kernels

template <typename T>
__global__ void __launch_bounds__(kThreads, 1) k_qkv(const QkvArgs a) {
  const Ctx c = gemv_setup(a.g, a.s.rows * a.s.n);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
  if (warp == kConsumerWarps) {
    if (lane == 0) produce(a.g, a.s, false, true, c, &a.io->error);
    return;
  }
  pdl_wait();
  const T *emb_row = nullptr;
  if (a.emb) {
    int tok = a.io->token;
    if (tok < 0 || tok >= a.n_vocab) {
      if (tid == 0 && blockIdx.x == 0) set_error(&a.io->error, kErrToken);
      tok = 0;
    }
    emb_row = static_cast<const T *>(a.emb) + (int64_t)tok * a.g.K;
  }
  load_rmsnorm<T>(c.xs, c.red, a.x, emb_row, a.norm_w, a.g.K, a.eps,
                  (a.emb && blockIdx.x == 0) ? a.x_out : nullptr, tid);
  consume<T>(a.g, a.s, false, c, warp, lane, &a.io->error, [](int) {});
  consumer_sync();

  const int pos = a.io->pos;
  const int slot = pos % a.cap;
  const int hd = a.head_dim;
  const int qrows = a.n_head * hd, krows = a.n_kv * hd;
  for (int64_t r = c.r0 + 2 * tid; r < c.r1; r += 2 * kConsumerThreads) {
    const int loc = (int)(r - c.r0), rr = (int)r;
    float v0 = row_total(c.part, loc, a.g.wpr), v1 = row_total(c.part, loc + 1, a.g.wpr);
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
      T *dst = static_cast<T *>(is_k ? a.k_cache : a.v_cache) + ((int64_t)gk * a.cap + slot) * hd + d;
      Elem<T>::store(dst, 0, v0);
      Elem<T>::store(dst, 1, v1);
    }
  }
}

template <typename T>
__global__ void __launch_bounds__(kThreads, 1) k_resid(const ResidArgs a) {
  const Ctx c = gemv_setup(a.g, a.s.rows * a.s.n);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
  if (warp == kConsumerWarps) {
    if (lane == 0) produce(a.g, a.s, false, true, c, &a.io->error);
    return;
  }
  pdl_wait();
  load_plain(c.xs, a.vec, a.g.K, tid);
  consumer_sync();
  consume<T>(a.g, a.s, false, c, warp, lane, &a.io->error, [](int) {});
  consumer_sync();
  for (int64_t r = c.r0 + tid; r < c.r1; r += kConsumerThreads)
    a.x[r] += row_total(c.part, (int)(r - c.r0), a.g.wpr);
}

template <typename T>
__global__ void __launch_bounds__(kThreads, 1) k_gateup(const GateUpArgs a) {
  const Ctx c = gemv_setup(a.g, a.s.rows * a.s.n);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
  if (warp == kConsumerWarps) {
    if (lane == 0) produce(a.g, a.s, false, a.s.table == nullptr, c, &a.io->error);
    return;
  }
  pdl_wait();
  load_rmsnorm<T>(c.xs, c.red, a.x, nullptr, a.norm_w, a.g.K, a.eps, nullptr, tid);
  consume<T>(a.g, a.s, false, c, warp, lane, &a.io->error, [](int) {});
  consumer_sync();
  for (int64_t r = c.r0 + 2 * tid; r < c.r1; r += 2 * kConsumerThreads) {
    const int loc = (int)(r - c.r0);
    const int seg = (int)(r / a.s.rows);
    const int i = (int)((r - seg * a.s.rows) >> 1);
    const float gte = row_total(c.part, loc, a.g.wpr), up = row_total(c.part, loc + 1, a.g.wpr);
    a.h[(int64_t)seg * a.n_ff + i] = silu(gte) * up;
  }
}

template <typename T>
__global__ void __launch_bounds__(kThreads, 1) k_down_moe(const DownMoeArgs a) {
  const Ctx c = gemv_setup(a.g, a.s.rows);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
  if (warp == kConsumerWarps) {
    if (lane == 0) produce(a.g, a.s, true, false, c, &a.io->error);
    return;
  }
  pdl_wait();
  load_plain(c.xs, a.h, a.g.K, tid);
  consumer_sync();
  consume<T>(a.g, a.s, true, c, warp, lane, &a.io->error,
             [&](int seg) { load_plain(c.xs, a.h + (int64_t)seg * a.n_ff, a.g.K, tid); });
  consumer_sync();
  for (int64_t r = c.r0 + tid; r < c.r1; r += kConsumerThreads) {
    float acc = 0.f;
    for (int s = 0; s < a.s.n; ++s)
      acc = fmaf(a.gate[s], row_total(c.part + s * a.g.rows_cta_max * a.g.wpr, (int)(r - c.r0), a.g.wpr),
                 acc);
    a.x[r] += acc;
  }
}

__device__ __forceinline__ void argmax_merge(float &v, int &i, float ov, int oi) {
  if (ov > v || (ov == v && oi < i)) {
    v = ov;
    i = oi;
  }
}

template <typename T>
__global__ void __launch_bounds__(kThreads, 1) k_lmhead(const LmArgs a) {
  const Ctx c = gemv_setup(a.g, a.s.rows);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
  if (warp == kConsumerWarps) {
    if (lane == 0) produce(a.g, a.s, false, true, c, &a.io->error);
    return;
  }
  pdl_wait();
  load_rmsnorm<T>(c.xs, c.red, a.x, nullptr, a.norm_w, a.g.K, a.eps, nullptr, tid);
  consume<T>(a.g, a.s, false, c, warp, lane, &a.io->error, [](int) {});
  consumer_sync();
  float best = -FLT_MAX;
  int bi = INT_MAX;
  for (int64_t r = c.r0 + tid; r < c.r1; r += kConsumerThreads) {
    const float v = row_total(c.part, (int)(r - c.r0), a.g.wpr);
    if (a.logits) a.logits[r] = v;
    argmax_merge(best, bi, v, (int)r);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
    argmax_merge(best, bi, __shfl_xor_sync(0xffffffffu, best, o), __shfl_xor_sync(0xffffffffu, bi, o));
  int *redi = reinterpret_cast<int *>(c.red + 32);
  if (lane == 0) {
    c.red[warp] = best;
    redi[warp] = bi;
  }
  consumer_sync();
  if (tid == 0) {
    for (int w = 1; w < kConsumerWarps; ++w) argmax_merge(best, bi, c.red[w], redi[w]);
    a.part_val[blockIdx.x] = best;
    a.part_idx[blockIdx.x] = bi;
    __threadfence();
    const unsigned prev = atomicAdd(a.counter, 1u);
    if (prev == gridDim.x - 1) {
      __threadfence();
      float fv = -FLT_MAX;
      int fi = INT_MAX;
      for (unsigned b = 0; b < gridDim.x; ++b) argmax_merge(fv, fi, __ldcg(a.part_val + b), __ldcg(a.part_idx + b));
      if (fi < 0 || fi >= a.s.rows) {
        set_error(&a.io->error, kErrToken);
        fi = 0;
      }
      if (a.argmax_out) *a.argmax_out = fi;
      a.io->token = fi;
      a.io->pos = a.io->pos + 1;
      *a.counter = 0u;
    }
  }
}

// Router: one CTA.  r = Wr RMSNorm(x); the k largest (lower index on ties);
// gate = softmax over the chosen logits.
template <typename T>
__global__ void __launch_bounds__(kConsumerThreads, 1) k_router(const RouterArgs a) {
  float *xs = reinterpret_cast<float *>(g_smem);
  float *red = xs + xpad_size(a.E);
  float *r = red + 64;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  pdl_wait();
  pdl_trigger();
  load_rmsnorm<T>(xs, red, a.x, nullptr, a.norm_w, a.E, a.eps, nullptr, tid);
  constexpr int EPV = 16 / (int)sizeof(T);
  for (int e = warp; e < a.n_expert; e += kConsumerWarps) {
    const uint8_t *row = static_cast<const uint8_t *>(a.w) + (int64_t)e * a.E * sizeof(T);
    float acc = 0.f;
    for (int v = lane; v < a.E / EPV; v += 32) acc += dot_range<T>(row, v, v + 1, xs, 0);
    acc = warp_sum(acc);
    if (lane == 0) r[e] = acc;
  }
  consumer_sync();
  if (tid == 0) {
    int idx[64];
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
    for (int i = 0; i < a.k; ++i) {
      a.idx[i] = idx[i];
      a.gate[i] = expf(r[idx[i]] - mx) / z;
    }
  }
}

__global__ void k_set_token(StepIO *io, int32_t token) { io->token = token; }
__global__ void k_set_pos(StepIO *io, int32_t pos) { io->pos = pos; }

template <typename Kern, typename Args>
cudaError_t launch(Kern kernel, const Args &a, dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                   bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, a);
}

template <typename Kern>
cudaError_t ensure_smem(Kern kernel, int bytes) {
  if (bytes <= 48 * 1024) return cudaSuccess;
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

template <typename Kern, typename Args>
cudaError_t launch_gemv(Kern kernel, const Args &a, int grid, cudaStream_t st, bool pdl) {
  return launch(kernel, a, dim3(grid), dim3(kThreads), smem_layout(a.g).total, st, pdl);
}

template <typename T>
cudaError_t prepare_t(int bytes) {
  cudaError_t e;
  if ((e = ensure_smem(k_qkv<T>, bytes)) != cudaSuccess) return e;
  if ((e = ensure_smem(k_resid<T>, bytes)) != cudaSuccess) return e;
  if ((e = ensure_smem(k_gateup<T>, bytes)) != cudaSuccess) return e;
  if ((e = ensure_smem(k_down_moe<T>, bytes)) != cudaSuccess) return e;
  if ((e = ensure_smem(k_lmhead<T>, bytes)) != cudaSuccess) return e;
  return ensure_smem(k_router<T>, bytes);
}

}  // namespace

cudaError_t launch_qkv(int dtype, const QkvArgs &a, int grid, cudaStream_t st, bool pdl) {
  return dtype ? launch_gemv(k_qkv<__nv_bfloat16>, a, grid, st, pdl)
               : launch_gemv(k_qkv<float>, a, grid, st, pdl);
}
cudaError_t launch_resid(int dtype, const ResidArgs &a, int grid, cudaStream_t st, bool pdl) {
  return dtype ? launch_gemv(k_resid<__nv_bfloat16>, a, grid, st, pdl)
               : launch_gemv(k_resid<float>, a, grid, st, pdl);
}
cudaError_t launch_gateup(int dtype, const GateUpArgs &a, int grid, cudaStream_t st, bool pdl) {
  return dtype ? launch_gemv(k_gateup<__nv_bfloat16>, a, grid, st, pdl)
               : launch_gemv(k_gateup<float>, a, grid, st, pdl);
}
cudaError_t launch_down_moe(int dtype, const DownMoeArgs &a, int grid, cudaStream_t st, bool pdl) {
  return dtype ? launch_gemv(k_down_moe<__nv_bfloat16>, a, grid, st, pdl)
               : launch_gemv(k_down_moe<float>, a, grid, st, pdl);
}
cudaError_t launch_lmhead(int dtype, const LmArgs &a, int grid, cudaStream_t st, bool pdl) {
  return dtype ? launch_gemv(k_lmhead<__nv_bfloat16>, a, grid, st, pdl)
               : launch_gemv(k_lmhead<float>, a, grid, st, pdl);
}
cudaError_t launch_router(int dtype, const RouterArgs &a, cudaStream_t st, bool pdl) {
  const int smem = (xpad_size(a.E) + 64 + a.n_expert) * 4;
  if (dtype) return launch(k_router<__nv_bfloat16>, a, dim3(1), dim3(kConsumerThreads), smem, st, pdl);
  return launch(k_router<float>, a, dim3(1), dim3(kConsumerThreads), smem, st, pdl);
}
cudaError_t prepare_gemv_kernels(int dtype, int smem_bytes) {
  return dtype ? prepare_t<__nv_bfloat16>(smem_bytes) : prepare_t<float>(smem_bytes);
}
cudaError_t launch_set_token(StepIO *io, int32_t token, cudaStream_t st) {
  k_set_token<<<1, 1, 0, st>>>(io, token);
  return cudaGetLastError();
}
cudaError_t launch_set_pos(StepIO *io, int32_t pos, cudaStream_t st) {
  k_set_pos<<<1, 1, 0, st>>>(io, pos);
  return cudaGetLastError();
}

}  // namespace pnb
