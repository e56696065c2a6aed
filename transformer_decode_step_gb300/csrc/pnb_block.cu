// pnb_block.cu - the attention half of a decoder layer as one kernel.
//
// The step of "Engine Architecture" (per layer: RMSNorm, q / k / v
// projections, RoPE, KV append, causal attention over the window, output
// projection into the residual) has three global dependencies when each
// phase is its own kernel: the attention needs the whole head's q / k / v,
// and the output projection needs every head's attention output.  Here one
// thread-block cluster of C CTAs owns one query head, so both dependencies
// stay inside the cluster and travel through distributed shared memory
// instead of L2:
//
//   warp 16 (one thread) streams, through one shared-memory ring, the CTA's
//     share of (a) the head's rows of Wq and its KV head's rows of Wk, Wv
//     (1-D bulk copies), (b) the cached K / V positions of the window
//     (1-D bulk copies, split at the ring's wrap), and (c) the rows of the
//     head's column block of Wo (2-D tensor copies);
//   warps 0-15 compute the normed row dot products of (a) and send them to
//     every CTA of the cluster (st.async, counted on the receiver's
//     mbarrier); every CTA then holds the head's q, k, v, applies RoPE, and
//     the owner of the KV head appends k, v to the cache.  They score and
//     accumulate (b) with an online softmax (eight lanes per position, log2
//     domain), fold in the current position (from shared memory), merge
//     their sixteen warps and send the CTA's (max, sum, weighted V) to every
//     CTA; all merge the C partials in the same order, and multiply the rows
//     of (c) by the result.
//
// Each head's output-projection value of a residual row is rounded to a
// 64-bit fixed-point word (units of 2^-32) and added into the state's
// accumulator with an integer atomic: the sum does not depend on the order in
// which the heads arrive, so steps stay bitwise reproducible.  The next
// RMSNorm reads x + accumulator and the down-projection kernel folds the
// accumulator into x and clears it.
#include <cuda.h>
#include <cuda_bf16.h>
#include <float.h>
#include <math.h>

#include "pnb_gemv_dev.cuh"
#include "pnb_tc.cuh"

namespace pnb {
namespace {

// ---------------------------------------------------------- cluster helpers
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire;" ::: "memory");
}
// address of the same shared-memory object in the cluster's CTA `rank`
__device__ __forceinline__ uint32_t peer_addr(const void *local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr(local)), "r"(rank));
  return r;
}
// store into a cluster CTA's shared memory; the bytes complete on that CTA's mbarrier
__device__ __forceinline__ void st_async_v4(uint32_t addr, float4 v, uint32_t bar) {
  asm volatile(
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
          addr),
      "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void st_async_v2(uint32_t addr, float2 v, uint32_t bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.f32 [%0], {%1, %2}, [%3];" ::"r"(
                   addr),
               "f"(v.x), "f"(v.y), "r"(bar)
               : "memory");
}
// fire-and-forget 64-bit integer add in global memory (no value returned)
__device__ __forceinline__ void red_add_u64(unsigned long long *addr, unsigned long long v) {
  asm volatile("red.relaxed.gpu.global.add.u64 [%0], %1;" ::"l"(addr), "l"(v) : "memory");
}

// bounded wait for a phase whose bytes come from the cluster's CTAs
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t *bar, uint32_t parity) {
  const unsigned long long t0 = global_ns();
  for (uint32_t it = 0;; ++it) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    if (ok) return true;
    if ((it & 255u) == 255u && (global_ns() - t0 > kWaitLimitNs || it > (1u << 26))) return false;
  }
}

// Ring items of the three streams, in the order both sides walk them.
// Rows r of the head's virtual [q; k; v] block (hd rows each): one item never
// crosses from one block to the next (they are separate rows of Wqkv).
template <int HD>
__device__ __forceinline__ int qkv_item_rows(int r, int r1, int rps) {
  const int blk_end = (r / HD + 1) * HD;
  return min(rps, min(r1 - r, blk_end - r));
}
// cached positions from p: stops at the ring's wrap
__device__ __forceinline__ int kv_item_pos(int p, int p1, int kv_item, int cap) {
  return min(kv_item, min(p1 - p, cap - p % cap));
}

struct BlockRange {
  int r0, r1;   // rows of the head's [q; k; v]
  int p0, p1;   // cached positions
  int e0, e1;   // rows of Wo (residual rows)
};

template <typename T, int HD>
__device__ __forceinline__ void produce_block(const BlockArgs &a, const CUtensorMap *wo_map,
                                              const BlockRange &R, int h, int g, int pos, uint8_t *ring,
                                              uint64_t *full, uint64_t *empty, int32_t *err) {
  constexpr int ES = (int)sizeof(T);
  const BlockGeom &b = a.b;
  const uint32_t NS = (uint32_t)b.nstages, SB = (uint32_t)b.stage_bytes;
  uint32_t i = 0;
  RingPos rp{0u, 0u, NS};
  bool waited = false, ok = true;
  // room for copy i (the first ring's worth goes out before griddepcontrol.wait:
  // weights and the cache's earlier positions do not depend on earlier kernels;
  // a copy with `dep` set reads what the previous kernel wrote)
  auto room = [&](bool dep) -> bool {
    if (!waited && (i == NS || dep)) {
      ktrace(a.tr, 6);
      pdl_wait();
      pdl_trigger();
      waited = true;
    }
    return i < NS || mbar_wait(&empty[rp.slot], rp.phase ^ 1u);
  };
  const uint8_t *wq = static_cast<const uint8_t *>(a.wqkv);
  const size_t rb = (size_t)b.g.row_bytes;
  for (int r = R.r0; r < R.r1 && ok;) {
    const int n = qkv_item_rows<HD>(r, R.r1, b.g.rows_per_stage);
    const int blk = r / HD, rin = r - blk * HD;
    const int64_t src = blk == 0 ? (int64_t)h * HD + rin
                                 : (int64_t)(a.H + (blk - 1) * a.Hkv + g) * HD + rin;
    if (!room(false)) {
      ok = false;
      break;
    }
    const uint32_t bytes = (uint32_t)n * (uint32_t)rb;
    mbar_arrive_expect_tx(&full[rp.slot], bytes);
    bulk_g2s(ring + rp.slot * SB, wq + src * rb, bytes, &full[rp.slot]);
    ++i;
    rp.advance();
    r += n;
  }
  const size_t head_bytes = (size_t)a.cap * HD * ES;
  const uint8_t *kb = static_cast<const uint8_t *>(a.k_cache) + (size_t)g * head_bytes;
  const uint8_t *vb = static_cast<const uint8_t *>(a.v_cache) + (size_t)g * head_bytes;
  for (int p = R.p0; p < R.p1 && ok;) {
    const int n = kv_item_pos(p, R.p1, b.kv_item, a.cap);
    if (!room(p + n > pos)) {   // the current position: written by the QKV kernel
      ok = false;
      break;
    }
    const uint32_t bytes = (uint32_t)(n * HD * ES);
    const size_t off = (size_t)(p % a.cap) * HD * ES;
    uint8_t *dst = ring + rp.slot * SB;
    mbar_arrive_expect_tx(&full[rp.slot], 2u * bytes);
    bulk_g2s(dst, kb + off, bytes, &full[rp.slot]);
    bulk_g2s(dst + (size_t)b.kv_item * HD * ES, vb + off, bytes, &full[rp.slot]);
    ++i;
    rp.advance();
    p += n;
  }
  for (int r = R.e0; r < R.e1 && ok; r += b.o_item) {
    if (!room(false)) {
      ok = false;
      break;
    }
    mbar_arrive_expect_tx(&full[rp.slot], (uint32_t)(b.o_item * HD * ES));
    tma_load_2d(ring + rp.slot * SB, wo_map, h * HD, r, &full[rp.slot]);
    ++i;
    rp.advance();
  }
  if (!waited) {
    ktrace(a.tr, 6);
    pdl_wait();
    pdl_trigger();
  }
  if (!ok) set_error(err, kErrTimeout);
  // the copies still in flight land before the CTA may end
  const uint32_t last = i < NS ? i : NS;
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

template <typename T, int NV, int HD>
__global__ void __launch_bounds__(kGemvThreads, 1)
    k_attn_block(const __grid_constant__ CUtensorMap wo_map, const BlockArgs a) {
  constexpr int ES = (int)sizeof(T);
  const BlockGeom &b = a.b;
  const int C = b.C, NS = b.nstages;
  const uint32_t rank = cluster_rank();
  const int h = blockIdx.x / C, g = h / (a.H / a.Hkv);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
  int32_t *err = &a.io->error;

  const BlockSmem L = block_smem(b, HD);
  uint8_t *sm = g_smem + ((1024u - (smem_addr(g_smem) & 1023u)) & 1023u);
  uint8_t *ring = sm + L.ring;
  float *part = reinterpret_cast<float *>(sm + L.part);
  float *qkv = reinterpret_cast<float *>(sm + L.qkv);
  float *wst = reinterpret_cast<float *>(sm + L.wst);
  float *apart = reinterpret_cast<float *>(sm + L.apart);
  float *ofin = reinterpret_cast<float *>(sm + L.ofin);
  float2 *rope = reinterpret_cast<float2 *>(sm + L.rope);
  float *red = reinterpret_cast<float *>(sm + L.red);
  uint64_t *full = reinterpret_cast<uint64_t *>(sm + L.bars);
  uint64_t *empty = full + NS;
  uint64_t *xq = empty + NS;   // the head's q / k / v rows have arrived
  uint64_t *xa = xq + 1;       // the cluster's softmax partials have arrived
  if (tid == 0) {
    ktrace(a.tr, 0);
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kGemvWarps);
    }
    mbar_init(xq, 1);
    mbar_init(xa, 1);
    fence_barrier_init();
    // bytes the cluster's CTAs store here: every row of [q; k; v], and one
    // (weighted V, max, sum) per CTA
    if (!a.q_in) mbar_arrive_expect_tx(xq, 3u * HD * 4u);
    mbar_arrive_expect_tx(xa, (uint32_t)C * (HD * 4u + 8u));
  }
  __syncthreads();
  cluster_arrive();   // barriers initialised (waited on before the first remote store)

  // this CTA's share of the three streams.  pos was written by an earlier step
  // (the first layer's launch waits for all earlier work): readable before the wait.
  const bool own_qkv = a.q_in == nullptr;
  const int pos = a.io->pos;
  const int lo = a.window > 0 ? max(0, pos - a.window + 1) : 0;
  // cached positions: with its own q / k / v the current one comes from the
  // exchange, else the QKV kernel has stored it
  const int npos = pos - lo + (own_qkv ? 0 : 1);
  const int E = b.g.K;
  BlockRange R;
  R.r0 = own_qkv ? b.rows_cta * (int)rank : 0;
  R.r1 = own_qkv ? R.r0 + b.rows_cta : 0;
  R.p0 = lo + (int)((int64_t)npos * rank / C);
  R.p1 = lo + (int)((int64_t)npos * (rank + 1) / C);
  R.e0 = E / C * (int)rank;
  R.e1 = R.e0 + E / C;

  if (warp == kGemvWarps) {
    if (lane == 0) produce_block<T, HD>(a, &wo_map, R, h, g, pos, ring, full, empty, err);
    __syncwarp();
    cluster_wait();
    cluster_arrive();   // no CTA ends while a peer may still store into it
    cluster_wait();
    return;
  }

  // ------------------------------------------------- (a) q / k / v rows
  const int cw = b.g.cw;
  const RowSplit sp(cw, b.g.vpr, warp);
  const uint32_t SB = (uint32_t)b.stage_bytes;
  RingPos rp{0u, 0u, (uint32_t)NS};
  bool ok = true;
  auto take = [&](uint32_t slot) -> bool {
    if (ok && !mbar_wait(&full[slot], rp.phase)) {
      ok = false;
      if (lane == 0) set_error(err, kErrTimeout);
    }
    return ok;
  };
  auto release = [&](uint32_t slot) {
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[slot]);
  };
  if (own_qkv) {
    XSlice<T, NV> xs;
    load_weight_slice(xs, a.norm_w, b.g, warp, lane);
    pdl_wait();
    if (tid == 0) ktrace(a.tr, 1);
    const double inv_freq = tid < HD / 2 ? a.inv_freq[tid] : 0.0;
    if (a.emb) {
      int tok = a.io->token;
      if (tok < 0 || tok >= a.n_vocab) {
        if (tid == 0 && blockIdx.x == 0) set_error(err, kErrToken);
        tok = 0;
      }
      const T *row = static_cast<const T *>(a.emb) + (int64_t)tok * E;
      if (blockIdx.x == 0)
        for (int i = tid * 2; i < E; i += kGemvConsumers * 2)
          *reinterpret_cast<float2 *>(a.x_out + i) = load2(row, i);
      norm_slice(xs, row, E, a.eps, b.g, red, warp, lane);
    } else {
      norm_slice(xs, a.x, E, a.eps, b.g, red, warp, lane);
    }
    if (tid == 0) ktrace(a.tr, 2);
    if (tid < HD / 2) {
      float sn, cs;
      rope_sincos(pos, inv_freq, &sn, &cs);
      rope[tid] = make_float2(cs, sn);
    }

    for (int r = R.r0; r < R.r1;) {
      const int n = qkv_item_rows<HD>(r, R.r1, b.g.rows_per_stage);
      const uint32_t slot = rp.slot;
      const bool first = r == R.r0;
      if (take(slot)) {
        if (first && tid == 0) ktrace(a.tr, 3);
        dot_item<T, NV>(ring + slot * SB, n, b.g.row_bytes, xs, part, r - R.r0, sp, lane);
        release(slot);
      }
      rp.advance();
      r += n;
    }
    gemv_sync();

    // exchange 1: every CTA of the cluster gets this CTA's rows
    cluster_wait();
    if (tid < b.rows_cta / 4) {
      float4 v;
      v.x = row_total(part, 4 * tid + 0, cw);
      v.y = row_total(part, 4 * tid + 1, cw);
      v.z = row_total(part, 4 * tid + 2, cw);
      v.w = row_total(part, 4 * tid + 3, cw);
      float *dst = qkv + R.r0 + 4 * tid;
      for (int p = 0; p < C; ++p) st_async_v4(peer_addr(dst, p), v, peer_addr(xq, p));
    }
    if (!mbar_wait_cluster(xq, 0) && lane == 0) set_error(err, kErrTimeout);
    if (tid == 0) ktrace(a.tr, 4);

    // RoPE on q and k (adjacent pairs), then k and v in the cache's precision
    if (tid < HD) {
      const int j = tid % (HD / 2);
      float *v = qkv + (tid < HD / 2 ? 0 : HD) + 2 * j;
      const float2 cs = rope[j];
      const float v0 = v[0], v1 = v[1];
      v[0] = v0 * cs.x - v1 * cs.y;
      v[1] = v0 * cs.y + v1 * cs.x;
    }
    gemv_sync();
    if (tid < HD) {
      const float kr = round_to<T>(qkv[HD + tid]), vr = round_to<T>(qkv[2 * HD + tid]);
      if (rank == 0 && h % (a.H / a.Hkv) == 0) {   // the KV head's first query head appends
        const size_t at = ((size_t)g * a.cap + pos % a.cap) * HD + tid;
        Elem<T>::store(static_cast<T *>(a.k_cache), at, kr);
        Elem<T>::store(static_cast<T *>(a.v_cache), at, vr);
      }
      qkv[HD + tid] = kr;
      qkv[2 * HD + tid] = vr;
      if (rank == 0 && a.q_out) a.q_out[(size_t)h * HD + tid] = qkv[tid];
    }
    gemv_sync();

  } else {
    // the QKV kernel has rotated the queries and stored the current K / V
    pdl_wait();
    if (tid == 0) ktrace(a.tr, 1);
    if (tid < HD) qkv[tid] = a.q_in[(size_t)h * HD + tid];
    gemv_sync();
    cluster_wait();
  }

  // ------------------------------------------------- (b) attention
  constexpr int DPL = HD / 8;                             // dims per lane when scoring
  constexpr int UNIT = (DPL * ES < 16) ? DPL * ES : 16;   // bytes per shared-memory load
  constexpr int EPU = UNIT / ES;
  constexpr int NCH = DPL / EPU;                          // loads per lane per key row
  constexpr int VPL = HD / 32;                            // dims per lane when accumulating V
  constexpr int ROTDIV = 8 / NCH;                         // lanes sharing a load order
  const int sub = lane & 7, t = lane >> 3;
  const int rot = sub / ROTDIV;
  float qr[NCH][EPU];
#pragma unroll
  for (int c = 0; c < NCH; ++c) {
    const int u = (c + rot) % NCH;
#pragma unroll
    for (int e = 0; e < EPU; ++e) qr[c][e] = qkv[sub * DPL + u * EPU + e] * a.qscale;
  }
  float m = -INFINITY, l = 0.f, o[VPL];
#pragma unroll
  for (int d = 0; d < VPL; ++d) o[d] = 0.f;
  // up to four scored positions (scores sc, V rows vv) into the warp's state
  auto accumulate = [&](const float (&sc)[4], const float (&vv)[4][VPL], int nv) {
    float mx = m;
#pragma unroll
    for (int tt = 0; tt < 4; ++tt)
      if (tt < nv) mx = fmaxf(mx, sc[tt]);
    if (mx == -INFINITY) return;
    const float alpha = exp2f(m - mx);
    l *= alpha;
#pragma unroll
    for (int d = 0; d < VPL; ++d) o[d] *= alpha;
#pragma unroll
    for (int tt = 0; tt < 4; ++tt) {
      if (tt < nv) {
        const float p = exp2f(sc[tt] - mx);
        l += p;
#pragma unroll
        for (int d = 0; d < VPL; ++d) o[d] = fmaf(p, vv[tt][d], o[d]);
      }
    }
    m = mx;
  };
  const size_t vofs = (size_t)b.kv_item * HD * ES;
  for (int p = R.p0; p < R.p1;) {
    const int n = kv_item_pos(p, R.p1, b.kv_item, a.cap);
    const uint32_t slot = rp.slot;
    if (take(slot)) {
      const T *ks = reinterpret_cast<const T *>(ring + slot * SB);
      const T *vs = reinterpret_cast<const T *>(ring + slot * SB + vofs);
      for (int pb = warp * 4; pb < n; pb += kGemvWarps * 4) {   // warp-uniform
        const int pi = pb + t;
        const bool valid = pi < n;
        float s = 0.f;
        if (valid) {
          const T *kr = ks + pi * HD + sub * DPL;
          float kf[NCH][EPU];
#pragma unroll
          for (int c = 0; c < NCH; ++c) load_vals<T, EPU>(kr + ((c + rot) % NCH) * EPU, kf[c]);
#pragma unroll
          for (int c = 0; c < NCH; ++c)
#pragma unroll
            for (int e = 0; e < EPU; ++e) s = fmaf(qr[c][e], kf[c][e], s);
        }
        s += __shfl_xor_sync(0xffffffffu, s, 4);
        s += __shfl_xor_sync(0xffffffffu, s, 2);
        s += __shfl_xor_sync(0xffffffffu, s, 1);
        float sc[4], vv[4][VPL];
#pragma unroll
        for (int tt = 0; tt < 4; ++tt) sc[tt] = __shfl_sync(0xffffffffu, s, tt * 8);
        const int nv = min(4, n - pb);
#pragma unroll
        for (int tt = 0; tt < 4; ++tt) {
          if (tt < nv) {
            load_vals<T, VPL>(vs + (pb + tt) * HD + lane * VPL, vv[tt]);
          } else {
#pragma unroll
            for (int d = 0; d < VPL; ++d) vv[tt][d] = 0.f;
          }
        }
        accumulate(sc, vv, nv);
      }
      release(slot);
    }
    rp.advance();
    p += n;
  }
  // the current position (rounded k, v from the exchange) on the last CTA
  if (own_qkv && rank == (uint32_t)C - 1 && warp == 0) {
    float s = 0.f;
#pragma unroll
    for (int d = 0; d < VPL; ++d) s = fmaf(qkv[lane * VPL + d] * a.qscale, qkv[HD + lane * VPL + d], s);
    s = warp_sum(s);
    float sc[4] = {s, -INFINITY, -INFINITY, -INFINITY}, vv[4][VPL];
#pragma unroll
    for (int tt = 0; tt < 4; ++tt)
#pragma unroll
      for (int d = 0; d < VPL; ++d) vv[tt][d] = tt == 0 ? qkv[2 * HD + lane * VPL + d] : 0.f;
    accumulate(sc, vv, 1);
  }
  // merge the sixteen warps
  float *ws = wst + warp * (HD + 4);
  if (lane == 0) {
    ws[HD] = m;
    ws[HD + 1] = l;
  }
#pragma unroll
  for (int d = 0; d < VPL; ++d) ws[lane * VPL + d] = o[d];
  gemv_sync();
  // exchange 2: the CTA's (weighted V, max, sum) to every CTA of the cluster
  if (tid < HD / 4) {
    float M = -INFINITY;
    for (int w = 0; w < kGemvWarps; ++w) M = fmaxf(M, wst[w * (HD + 4) + HD]);
    float Ls = 0.f;
    float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
    if (M != -INFINITY) {
      for (int w = 0; w < kGemvWarps; ++w) {
        const float *wr = wst + w * (HD + 4);
        const float f = exp2f(wr[HD] - M);
        Ls = fmaf(wr[HD + 1], f, Ls);
        O.x = fmaf(wr[4 * tid + 0], f, O.x);
        O.y = fmaf(wr[4 * tid + 1], f, O.y);
        O.z = fmaf(wr[4 * tid + 2], f, O.z);
        O.w = fmaf(wr[4 * tid + 3], f, O.w);
      }
    }
    float *dst = apart + rank * (HD + 4);
    for (int p = 0; p < C; ++p) {
      const uint32_t bar = peer_addr(xa, p);
      st_async_v4(peer_addr(dst + 4 * tid, p), O, bar);
      if (tid == 0) st_async_v2(peer_addr(dst + HD, p), make_float2(M, Ls), bar);
    }
  }
  if (!mbar_wait_cluster(xa, 0) && lane == 0) set_error(err, kErrTimeout);
  if (tid == 0) ktrace(a.tr, 5);
  if (tid < HD) {
    float M = -INFINITY;
    for (int c = 0; c < C; ++c) M = fmaxf(M, apart[c * (HD + 4) + HD]);
    float Ls = 0.f, Os = 0.f;
    for (int c = 0; c < C; ++c) {
      const float *pc = apart + c * (HD + 4);
      if (pc[HD] == -INFINITY) continue;
      const float f = exp2f(pc[HD] - M);
      Ls = fmaf(pc[HD + 1], f, Ls);
      Os = fmaf(pc[tid], f, Os);
    }
    ofin[tid] = Os / Ls;
    if (rank == 0 && a.o_out) a.o_out[(size_t)h * HD + tid] = ofin[tid];
  }
  gemv_sync();

  // ------------------------------------------------- (c) output projection
  constexpr int VN = 16 / ES;    // elements per 16-byte vector
  constexpr int LR = HD / VN;    // lanes per Wo row
  constexpr int RW = 32 / LR;    // rows per warp pass
  const int vl = lane % LR, rl = lane / LR;
  float ov[VN];
#pragma unroll
  for (int j = 0; j < VN; ++j) ov[j] = ofin[vl * VN + j];
  unsigned long long *acc = reinterpret_cast<unsigned long long *>(a.acc);
  for (int r = R.e0; r < R.e1; r += b.o_item) {
    const uint32_t slot = rp.slot;
    if (take(slot)) {
      const T *tile = reinterpret_cast<const T *>(ring + slot * SB);
      for (int base = warp * RW; base < b.o_item; base += kGemvWarps * RW) {   // warp-uniform
        const int row = base + rl;
        float w[VN];
        load_vals<T, VN>(tile + (size_t)row * HD + vl * VN, w);
        float y = 0.f;
#pragma unroll
        for (int j = 0; j < VN; ++j) y = fmaf(w[j], ov[j], y);
#pragma unroll
        for (int off = LR / 2; off > 0; off >>= 1) y += __shfl_xor_sync(0xffffffffu, y, off);
        if (vl == 0) {
          if (!(fabsf(y) < kFixLimit)) {
            set_error(err, kErrRange);
            y = y > 0.f ? kFixLimit : (y < 0.f ? -kFixLimit : 0.f);
          }
          red_add_u64(acc + r + row, (unsigned long long)__float2ll_rn(y * kFixScale));
        }
      }
      release(slot);
    }
    rp.advance();
  }
  cluster_arrive();
  cluster_wait();
  if (tid == 0) ktrace(a.tr, 7);
}

template <typename T, int NV, int HD>
cudaError_t launch_t(const void *wo_map, const BlockArgs &a, cudaStream_t st, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.H * a.b.C);
  cfg.blockDim = dim3(kGemvThreads);
  cfg.dynamicSmemBytes = a.b.smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = a.b.C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, k_attn_block<T, NV, HD>, *static_cast<const CUtensorMap *>(wo_map), a);
}

template <typename T, int NV, int HD>
int max_clusters_t(const BlockGeom &b, int n_clusters) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(n_clusters * b.C);
  cfg.blockDim = dim3(kGemvThreads);
  cfg.dynamicSmemBytes = b.smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = b.C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, k_attn_block<T, NV, HD>, &cfg) != cudaSuccess) return 0;
  return n;
}

template <typename T, int HD>
cudaError_t prepare_hd(int bytes) {
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(k_attn_block<T, 1, HD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                bytes)) != cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(k_attn_block<T, 2, HD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                bytes)) != cudaSuccess)
    return e;
  return cudaFuncSetAttribute(k_attn_block<T, 4, HD>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

template <typename T>
cudaError_t prepare_t(int bytes) {
  cudaError_t e;
  if ((e = prepare_hd<T, 32>(bytes)) != cudaSuccess) return e;
  if ((e = prepare_hd<T, 64>(bytes)) != cudaSuccess) return e;
  return prepare_hd<T, 128>(bytes);
}

// one instantiation per (vectors per lane, head_dim)
template <typename T>
cudaError_t launch_dtype(int hd, const void *wo_map, const BlockArgs &a, cudaStream_t st, bool pdl) {
  switch (a.b.g.nv * 1000 + hd) {
    case 1032: return launch_t<T, 1, 32>(wo_map, a, st, pdl);
    case 1064: return launch_t<T, 1, 64>(wo_map, a, st, pdl);
    case 1128: return launch_t<T, 1, 128>(wo_map, a, st, pdl);
    case 2032: return launch_t<T, 2, 32>(wo_map, a, st, pdl);
    case 2064: return launch_t<T, 2, 64>(wo_map, a, st, pdl);
    case 2128: return launch_t<T, 2, 128>(wo_map, a, st, pdl);
    case 4032: return launch_t<T, 4, 32>(wo_map, a, st, pdl);
    case 4064: return launch_t<T, 4, 64>(wo_map, a, st, pdl);
    case 4128: return launch_t<T, 4, 128>(wo_map, a, st, pdl);
    default: return cudaErrorInvalidValue;
  }
}

template <typename T>
int clusters_dtype(int hd, const BlockGeom &b, int n) {
  switch (b.g.nv * 1000 + hd) {
    case 1032: return max_clusters_t<T, 1, 32>(b, n);
    case 1064: return max_clusters_t<T, 1, 64>(b, n);
    case 1128: return max_clusters_t<T, 1, 128>(b, n);
    case 2032: return max_clusters_t<T, 2, 32>(b, n);
    case 2064: return max_clusters_t<T, 2, 64>(b, n);
    case 2128: return max_clusters_t<T, 2, 128>(b, n);
    case 4032: return max_clusters_t<T, 4, 32>(b, n);
    case 4064: return max_clusters_t<T, 4, 64>(b, n);
    case 4128: return max_clusters_t<T, 4, 128>(b, n);
    default: return 0;
  }
}

}  // namespace

cudaError_t launch_attn_block(int dtype, int head_dim, const void *wo_map, const BlockArgs &a,
                              cudaStream_t st, bool pdl) {
  return dtype ? launch_dtype<__nv_bfloat16>(head_dim, wo_map, a, st, pdl)
               : launch_dtype<float>(head_dim, wo_map, a, st, pdl);
}

cudaError_t prepare_attn_block_kernels(int dtype, int smem_bytes) {
  return dtype ? prepare_t<__nv_bfloat16>(smem_bytes) : prepare_t<float>(smem_bytes);
}

int attn_block_max_clusters(int dtype, int head_dim, const BlockGeom &b, int n_clusters) {
  return dtype ? clusters_dtype<__nv_bfloat16>(head_dim, b, n_clusters)
               : clusters_dtype<float>(head_dim, b, n_clusters);
}

}  // namespace pnb
