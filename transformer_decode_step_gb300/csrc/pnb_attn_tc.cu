// pnb_attn_tc.cu - decode attention on tcgen05 tensor cores (bf16 KV cache).
//
// One CTA takes one KV head g of one sequence (slot) and a range of
// 128-position tiles of its attended positions [lo, pos]; the G query heads
// that share g are computed together.
//   warp 0   streams the K and V tiles of each 128 positions with tiled TMA
//            loads (128-byte swizzle) from the state's tensor maps into a ring;
//   warp 1   issues S = K Q^T (M = 128 positions, N = 16: rows h and 8 + h of
//            Q hold the bf16 high and low parts of query head h, scaled by
//            log2(e) / sqrt(hd)) and O = P V (M = 128 rows of P, N = hd, V as
//            an MN-major operand), accumulators in TMEM;
//   warps 2-5 own one position each: they read S back (tcgen05.ld), keep the
//            running max and sum per head (online softmax in the log2
//            domain), write P = exp2(s - max) as bf16 high / low parts into
//            rows h and 8 + h of a swizzled shared tile, and warp 4 (TMEM
//            lanes 0-31, the rows of P that carry heads) folds each tile's O
//            into its registers with the rescale factor.
// The splits of a KV head's position range form one thread-block cluster:
// each CTA sends its (max, sum, O) partial of query head h to cluster CTA
// h mod n_split through distributed shared memory (st.async completing on the
// receiver's mbarrier), and the receiving CTAs merge by log-sum-exp in split
// order and write the output.
#include <cuda.h>
#include <algorithm>
#include <cuda_bf16.h>
#include <limits.h>
#include <math.h>

#include "pnb_kernels.cuh"
#include "pnb_tc.cuh"

namespace pnb {
namespace {

extern __shared__ __align__(1024) uint8_t t_smem[];

constexpr int kTThreads = 192;
constexpr int kTile = 128;          // positions per tile
constexpr int kBox = 128 * 128;     // bytes of one 128-row x 64-column bf16 box

// byte offset of (row, byte column) in a [rows][128 B] tile with 128-byte swizzle
__device__ __forceinline__ uint32_t sw128(int row, int col_bytes) {
  return (uint32_t)row * 128u + ((((uint32_t)col_bytes >> 4) ^ ((uint32_t)row & 7u)) << 4) +
         ((uint32_t)col_bytes & 15u);
}

__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void epi_sync_t() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

__device__ __forceinline__ void cl_arrive() { asm volatile("barrier.cluster.arrive.release;" ::: "memory"); }
__device__ __forceinline__ void cl_wait() { asm volatile("barrier.cluster.wait.acquire;" ::: "memory"); }
// address of the same shared-memory object in the cluster's CTA `rank`
__device__ __forceinline__ uint32_t cl_peer(const void *local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr(local)), "r"(rank));
  return r;
}
// stores into a cluster CTA's shared memory; the bytes complete on its mbarrier
__device__ __forceinline__ void cl_st_f32(uint32_t addr, float v, uint32_t bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.f32 [%0], %1, [%2];" ::"r"(addr),
               "f"(v), "r"(bar)
               : "memory");
}
__device__ __forceinline__ void cl_st_v2(uint32_t addr, float2 v, uint32_t bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.f32 [%0], {%1, %2}, [%3];" ::"r"(
                   addr),
               "f"(v.x), "f"(v.y), "r"(bar)
               : "memory");
}
__device__ __forceinline__ void cl_st_v4(uint32_t addr, float4 v, uint32_t bar) {
  asm volatile(
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
          addr),
      "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "r"(bar)
      : "memory");
}
// bounded wait for bytes stored by the cluster's CTAs
__device__ __forceinline__ bool cl_mbar_wait(uint64_t *bar, uint32_t parity) {
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

// The split partials a CTA merges: query heads h with h % n_split == rank,
// [local head][split][hd + 4] floats (O, then max and sum).
constexpr int kMaxSplit = 8;   // portable cluster size (16-CTA clusters measured slower)
__host__ __device__ constexpr int merge_floats(int hd) { return 16 * (hd + 4); }

// descriptor of an MN-major operand tile with 128-byte swizzle: 64-element
// atoms along N lbo bytes apart, groups of 8 K-rows 1024 bytes apart
__device__ __forceinline__ uint64_t desc_mn_sw128(const void *tile, uint32_t lbo) {
  const uint32_t addr = smem_addr(tile);
  uint64_t d = 0;
  d |= (uint64_t)((addr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)(1024u >> 4) << 32;
  d |= (uint64_t)1u << 46;
  d |= (uint64_t)2u << 61;
  return d;
}

// head_dim 128 computes O^T = V^T P^T (M = 128 dims, V as an MN-major A
// operand, P a 16-row K-major B operand, O^T in 16 TMEM columns: one dim per
// softmax thread); head_dim 64 computes O = P V (M = 128 rows of P, of which
// rows h and 8 + h carry head h, V an MN-major B operand, O in 64 columns
// read by the warp on TMEM lanes 0-31).
template <int HD>
struct TL {
  static constexpr bool VT = HD == 128;
  static constexpr int KT = HD / 64 * kBox;             // K tile bytes (HD / 64 boxes)
  static constexpr int STAGE = 2 * KT;                  // K and V
  static constexpr int PCH = VT ? 2048 : kBox;          // P bytes per 64-position chunk
  static constexpr int PT = 2 * PCH;                    // P tile: 128 positions
  static constexpr int QT = HD / 64 * 2048;             // Q tile: 16 rows x HD
  static constexpr uint32_t TCOLS = VT ? 64u : 256u;    // TMEM columns
  static constexpr uint32_t OCOL = VT ? 32u : 128u;     // O's first column
};

struct TBars {
  uint64_t *full, *empty;
  uint64_t *s_full, *s_empty, *p_full, *p_empty, *o_full, *o_empty, *q_ready, *merge_full;
};

template <int HD, int G>
__global__ void __launch_bounds__(kTThreads, 1) k_attn_tc(const AttnTcArgs a) {
  constexpr int KT = TL<HD>::KT, STAGE = TL<HD>::STAGE, PT = TL<HD>::PT, QT = TL<HD>::QT;
  constexpr bool VT = TL<HD>::VT;
  constexpr int PCH = TL<HD>::PCH;
  constexpr uint32_t TCOLS = TL<HD>::TCOLS;
  const int NS = a.nstages;
  const bool batched = a.slots != nullptr;
  const int split = blockIdx.x, g = blockIdx.y;
  const int b = batched && a.use_order ? (int)a.order[blockIdx.z] : (int)blockIdx.z;
  // column h: query head h0 + h % GH of virtual slot b * T + h / GH (T = 1:
  // the CTA's slot, every column one of its query heads)
  const int T = batched && a.tok_group > 1 ? a.tok_group : 1;
  const int GH = G / T;
  const int h0 = g * GH;
  auto col_slot = [&](int h) { return b * T + h / GH; };
  auto col_head = [&](int h) { return h0 + h % GH; };
  const BSlot bs = batched ? a.slots[b * T] : BSlot{nullptr, a.io, a.maps};
  int32_t *err = &bs.io->error;
  const CUtensorMap *maps = static_cast<const CUtensorMap *>(bs.maps) + 2 * a.layer;
  const CUtensorMap *kmap = maps, *vmap = maps + 1;
  const int ns = a.n_split;         // splits = CTAs of this KV head's cluster
  const bool clustered = ns > 1;
  // query heads this CTA merges: h = split + j * ns < G
  const int nloc = split < G ? (G - 1 - split) / ns + 1 : 0;

  // positions: [lo_h, pos_h] per column (a dead column, past the last slot,
  // attends to nothing); the CTA's tiles cover the union [lo, pos], 128
  // aligned positions each, split evenly
  int posc[G], loc[G];
  int pos = -1, lo = INT_MAX;
#pragma unroll
  for (int h = 0; h < G; ++h) {
    const bool live = !batched || col_slot(h) < a.nb;
    posc[h] = live ? (batched ? a.pos[col_slot(h)] : a.io->pos) : -1;
    loc[h] = live ? (a.window > 0 ? max(0, posc[h] - a.window + 1) : 0) : INT_MAX;
    pos = max(pos, posc[h]);
    lo = min(lo, loc[h]);
  }
  const int t_first = lo / kTile, t_last = pos / kTile;
  const int nt_all = t_last - t_first + 1;
  const int tb = t_first + (int)((int64_t)nt_all * split / ns);
  const int ntiles = t_first + (int)((int64_t)nt_all * (split + 1) / ns) - tb;

  // shared memory
  const uint32_t base = smem_addr(t_smem);
  uint8_t *sm = t_smem + ((1024u - (base & 1023u)) & 1023u);
  uint8_t *ring = sm;
  uint8_t *P = ring + (size_t)NS * STAGE;
  uint8_t *Q = P + 2 * PT;
  TBars bar;
  bar.full = reinterpret_cast<uint64_t *>(Q + QT);
  bar.empty = bar.full + NS;
  bar.s_full = bar.empty + NS;
  bar.s_empty = bar.s_full + 1;
  bar.p_full = bar.s_empty + 1;
  bar.p_empty = bar.p_full + 2;
  bar.o_full = bar.p_empty + 2;
  bar.o_empty = bar.o_full + 1;
  bar.q_ready = bar.o_empty + 1;
  bar.merge_full = bar.q_ready + 1;
  uint32_t *tslot = reinterpret_cast<uint32_t *>(bar.merge_full + 1);
  float *red = reinterpret_cast<float *>(tslot + 4);   // [2][4][8] maxima, then [4][8] sums
  float *recv = reinterpret_cast<float *>(Q + QT + 1024);   // merge_floats(HD)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    ktrace(a.tr, 0);
    for (int s = 0; s < NS; ++s) {
      mbar_init(&bar.full[s], 1);
      mbar_init(&bar.empty[s], 1);
    }
    mbar_init(bar.s_full, 1);
    mbar_init(bar.s_empty, 4);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar.p_full[i], 4);
      mbar_init(&bar.p_empty[i], 1);
    }
    mbar_init(bar.o_full, 1);
    mbar_init(bar.o_empty, 1);
    mbar_init(bar.q_ready, 4);
    mbar_init(bar.merge_full, 1);
    fence_barrier_init();
    // bytes the cluster's CTAs will store here: (O, max, sum) per split and head
    if (clustered && nloc > 0) mbar_arrive_expect_tx(bar.merge_full, (uint32_t)(nloc * ns * (HD * 4 + 8)));
  }
  if (warp == 1) {
    tmem_alloc(tslot, TCOLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (clustered) cl_arrive();   // the merge barrier is armed before any peer stores into it
  bool cl_waited = false;
  const uint32_t taddr = *tslot;
  const uint32_t t_s = taddr, t_o = taddr + TL<HD>::OCOL;

  if (warp == 0) {
    if (lane == 0) {
      // tiles before the first new position were written by earlier steps;
      // a tile holding a new position (pos, or from a prefill chunk's first
      // token on) waits for the kernel that wrote this step's K / V
      const int p_new = batched && a.shared_cache ? a.pos[0] : pos;
      bool waited = false, ok = true;
      for (int i = 0; i < ntiles; ++i) {
        const int T = tb + i, s = i % NS, r = i / NS;
        if (!waited && ((T + 1) * kTile > p_new || i == NS)) {
          ktrace(a.tr, 6);
          pdl_wait();
          pdl_trigger();
          ktrace(a.tr, 7);
          waited = true;
        }
        if (i >= NS && !mbar_wait(&bar.empty[s], (r - 1) & 1)) {
          ok = false;
          break;
        }
        const int y = g * a.cap + (T * kTile) % a.cap;
        uint8_t *kt = ring + (size_t)s * STAGE, *vt = kt + KT;
        mbar_arrive_expect_tx(&bar.full[s], STAGE);
#pragma unroll
        for (int c = 0; c < HD / 64; ++c) {
          tma_load_2d(kt + c * kBox, kmap, c * 64, y, &bar.full[s]);
          tma_load_2d(vt + c * kBox, vmap, c * 64, y, &bar.full[s]);
        }
      }
      if (!waited) {
        ktrace(a.tr, 6);
        pdl_wait();
        pdl_trigger();
        ktrace(a.tr, 7);
      }
      if (!ok) set_error(err, kErrTimeout);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(128, 16);
      // V MN-major: as A of O^T = V^T P^T (head_dim 128) or as B of O = P V
      constexpr uint32_t idesc_o = VT ? (idesc_bf16_f32(128, 16) | (1u << 15))
                                      : (idesc_bf16_f32(128, HD) | (1u << 16));
      bool ok = mbar_wait(bar.q_ready, 0);
      auto issue_s = [&](int t) {
        const uint8_t *kt = ring + (size_t)(t % NS) * STAGE;
#pragma unroll
        for (int c = 0; c < HD / 64; ++c)
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_bf16(t_s, desc_k_sw128(kt + c * kBox, k * 32), desc_k_sw128(Q + c * 2048, k * 32), idesc_s,
                     c > 0 || k > 0);
        mma_commit(bar.s_full);
      };
      if (ok && ntiles > 0) {
        ok = mbar_wait(&bar.full[0], 0);
        if (ok) {
          tc_fence_after();
          issue_s(0);
        }
      }
      for (int t = 0; t < ntiles && ok; ++t) {
        if (t + 1 < ntiles) {
          ok = mbar_wait(&bar.full[(t + 1) % NS], ((t + 1) / NS) & 1) && mbar_wait(bar.s_empty, t & 1);
          if (!ok) break;
          tc_fence_after();
          issue_s(t + 1);
        }
        ok = mbar_wait(&bar.p_full[t & 1], (t >> 1) & 1);
        if (!ok) break;
        tc_fence_after();
        const uint8_t *pt = P + (size_t)(t & 1) * PT;
        const uint8_t *vt = ring + (size_t)(t % NS) * STAGE + KT;
        // O accumulates in TMEM over the CTA's tiles (rescaled in place when the
        // softmax warps raise their reference max)
#pragma unroll
        for (int pc = 0; pc < kTile / 16; ++pc) {
          const uint64_t dp = desc_k_sw128(pt + (pc >> 2) * PCH, (pc & 3) * 32);
          const uint64_t dv = desc_mn_sw128(vt + pc * 2048, kBox);
          if constexpr (VT) mma_bf16(t_o, dv, dp, idesc_o, t > 0 || pc > 0);
          else mma_bf16(t_o, dp, dv, idesc_o, t > 0 || pc > 0);
        }
        mma_commit(bar.o_full);
        mma_commit(&bar.p_empty[t & 1]);
        mma_commit(&bar.empty[t % NS]);
      }
      if (!ok) set_error(err, kErrTimeout);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------ softmax warps 2-5
    const int q = warp & 3, tid = threadIdx.x - 64;   // position 32 q + lane of each tile
    // Q operand: rows h / 8 + h = high / low bf16 of q_h * qscale, zero rows elsewhere
    for (int i = tid * 16; i < QT; i += 128 * 16) *reinterpret_cast<uint4 *>(Q + i) = make_uint4(0, 0, 0, 0);
    pdl_wait();   // q comes from the QKV kernel
    epi_sync_t();
    for (int i = tid; i < G * HD; i += 128) {
      const int h = i / HD, d = i - h * HD;
      const float v = (col_slot(h) < (batched ? a.nb : 1))
                          ? a.q[((size_t)col_slot(h) * a.n_head + col_head(h)) * HD + d] * a.qscale
                          : 0.f;
      const __nv_bfloat16 hi = __float2bfloat16_rn(v);
      const __nv_bfloat16 lo = __float2bfloat16_rn(v - __bfloat162float(hi));
      uint8_t *tile = Q + (d >> 6) * 2048;
      *reinterpret_cast<__nv_bfloat16 *>(tile + sw128(h, (d & 63) * 2)) = hi;
      *reinterpret_cast<__nv_bfloat16 *>(tile + sw128(8 + h, (d & 63) * 2)) = lo;
    }
    fence_async_smem();
    epi_sync_t();
    if (lane == 0) mbar_arrive(bar.q_ready);
    if (tid == 0) ktrace(a.tr, 1);
    // P tiles: only rows h and 8 + h are ever written; the rest must be zero
    // (first used by the first P V product, after this CTA's first softmax)
    for (int i = tid * 16; i < 2 * PT; i += 128 * 16) *reinterpret_cast<uint4 *>(P + i) = make_uint4(0, 0, 0, 0);
    fence_async_smem();
    epi_sync_t();

    // Online softmax with a reference max per head that only moves when a
    // tile's max exceeds it by more than 2^8: P = exp2(s - ref) stays below
    // 256, sums stay per thread, and O (in TMEM) is rescaled only on a move.
    constexpr float kTau = 8.f;
    float m[G], l[G];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      m[h] = -INFINITY;
      l[h] = 0.f;
    }
    bool ok = true;
    for (int t = 0; t < ntiles; ++t) {
      if (ok && !mbar_wait(bar.s_full, t & 1)) {
        ok = false;
        if (lane == 0) set_error(err, kErrTimeout);
      }
      float v[32];
      if (ok) {
        tc_fence_after();
        tmem_ld32(t_s + ((uint32_t)(32 * q) << 16), v);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = 0.f;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar.s_empty);
      const int p = (tb + t) * kTile + 32 * q + lane;
      bool valid[G];
      float sc[G];
      float *rm = red + (t & 1) * 32;
#pragma unroll
      for (int h = 0; h < G; ++h) {
        valid[h] = p >= loc[h] && p <= posc[h];
        sc[h] = valid[h] ? v[h] + v[8 + h] : -INFINITY;
        const float mx = warp_max(sc[h]);
        if (lane == 0) rm[q * 8 + h] = mx;
      }
      epi_sync_t();
      bool move = false;
      float scale[G];
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float mt = fmaxf(fmaxf(rm[h], rm[8 + h]), fmaxf(rm[16 + h], rm[24 + h]));
        scale[h] = 1.f;
        if (mt > m[h] + kTau) {
          scale[h] = m[h] == -INFINITY ? 0.f : exp2f(m[h] - mt);
          m[h] = mt;
          l[h] *= scale[h];
          move = true;
        }
      }
      if (t > 0 && (VT || q == 0)) {
        // the previous tile's P V product is done: o_full is consumed phase by
        // phase (before this tile's P is published, so at most one phase is
        // ever pending and the parity wait cannot alias); then rescale O if
        // the reference max moved
        if (ok && !mbar_wait(bar.o_full, (t - 1) & 1)) {
          ok = false;
          if (lane == 0) set_error(err, kErrTimeout);
        }
        if (VT && ok && move) {
          // O^T: this thread's lane is a dim; column h / 8 + h is head h
          tc_fence_after();
          float w[32];
          tmem_ld32(t_o + ((uint32_t)(32 * q) << 16), w);
#pragma unroll
          for (int h = 0; h < G; ++h) {
            w[h] *= scale[h];
            w[8 + h] *= scale[h];
          }
          tmem_st32(t_o + ((uint32_t)(32 * q) << 16), w);
          tc_fence_before();
        } else if (!VT && ok && move) {
          tc_fence_after();
          float al = 1.f;
#pragma unroll
          for (int h = 0; h < G; ++h)
            if ((lane & 7) == h) al = scale[h];
#pragma unroll
          for (int c = 0; c < HD / 32; ++c) {
            float w[32];
            tmem_ld32(t_o + 32 * c, w);
#pragma unroll
            for (int i = 0; i < 32; ++i) w[i] *= al;
            tmem_st32(t_o + 32 * c, w);
          }
          tc_fence_before();
        }
      }
      float pp[G];
#pragma unroll
      for (int h = 0; h < G; ++h) {
        pp[h] = (valid[h] && m[h] != -INFINITY) ? exp2f(sc[h] - m[h]) : 0.f;
        l[h] += pp[h];
      }
      // P of this tile into buffer t & 1, once the P V product of tile t - 2 is done
      if (t >= 2 && ok && !mbar_wait(&bar.p_empty[t & 1], ((t >> 1) - 1) & 1)) {
        ok = false;
        if (lane == 0) set_error(err, kErrTimeout);
      }
      uint8_t *pt = P + (size_t)(t & 1) * PT + ((32 * q + lane) >> 6) * PCH;
      const int cb = ((32 * q + lane) & 63) * 2;
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const __nv_bfloat16 hi = __float2bfloat16_rn(pp[h]);
        const __nv_bfloat16 lo2 = __float2bfloat16_rn(pp[h] - __bfloat162float(hi));
        *reinterpret_cast<__nv_bfloat16 *>(pt + sw128(h, cb)) = hi;
        *reinterpret_cast<__nv_bfloat16 *>(pt + sw128(8 + h, cb)) = lo2;
      }
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar.p_full[t & 1]);
    }
    if (threadIdx.x == 128) ktrace(a.tr, 3);
    // row sums over the CTA's positions (fixed order: lanes, then warps)
    float *rs = red + 64;
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float sw = warp_sum(l[h]);
      if (lane == 0) rs[q * 8 + h] = sw;
    }
    epi_sync_t();
#pragma unroll
    for (int h = 0; h < G; ++h) l[h] = rs[h] + rs[8 + h] + rs[16 + h] + rs[24 + h];
    if constexpr (VT) {
      // O^T: thread = dim d, columns h / 8 + h = high / low parts of head h
      float oh[G];
#pragma unroll
      for (int h = 0; h < G; ++h) oh[h] = 0.f;
      if (ntiles > 0) {
        if (ok && !mbar_wait(bar.o_full, (ntiles - 1) & 1)) {
          ok = false;
          if (lane == 0) set_error(err, kErrTimeout);
        }
        if (ok) {
          tc_fence_after();
          float w[32];
          tmem_ld32(t_o + ((uint32_t)(32 * q) << 16), w);
#pragma unroll
          for (int h = 0; h < G; ++h) oh[h] = w[h] + w[8 + h];
        }
      }
      const int d = 32 * q + lane;
      if (!clustered) {
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const size_t col = (size_t)col_head(h) * HD + d;
          const float x = l[h] > 0.f ? oh[h] / l[h] : 0.f;
          if (a.xop) {
            const int r = col_slot(h);
            if (r < a.nb) {
              const __nv_bfloat16 hi = __float2bfloat16_rn(x);
              a.xop[(size_t)r * a.xop_ld + col] = hi;
              a.xop[(size_t)(a.bp + r) * a.xop_ld + col] = __float2bfloat16_rn(x - __bfloat162float(hi));
            }
          } else {
            a.out[col] = x;
          }
        }
      } else {
        cl_wait();
        cl_waited = true;
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const uint32_t rr = (uint32_t)(h % ns);
          float *dst = recv + ((h / ns) * ns + split) * (HD + 4);
          const uint32_t mb = cl_peer(bar.merge_full, rr);
          cl_st_f32(cl_peer(dst + d, rr), oh[h], mb);
          if (d == 0) cl_st_v2(cl_peer(dst + HD, rr), make_float2(m[h], l[h]), mb);
        }
      }
    } else {
      float o[HD];   // warp 4 (TMEM lanes 0-31): row lane of O
  #pragma unroll
      for (int d = 0; d < HD; ++d) o[d] = 0.f;
      if (q == 0 && ntiles > 0) {
        if (ok && !mbar_wait(bar.o_full, (ntiles - 1) & 1)) {
          ok = false;
          if (lane == 0) set_error(err, kErrTimeout);
        }
        if (ok) {
          tc_fence_after();
  #pragma unroll
          for (int c = 0; c < HD / 32; ++c) {
            float w[32];
            tmem_ld32(t_o + 32 * c, w);
  #pragma unroll
            for (int i = 0; i < 32; ++i) o[32 * c + i] = w[i];
          }
        }
      }
      // (max, sum, O) per head: lane h adds its low-part row 8 + h; with one split
      // this is the output, else a partial for the merge
      if (clustered) {
        cl_wait();
        cl_waited = true;
      }
      if (q == 0) {
  #pragma unroll
        for (int d = 0; d < HD; ++d) o[d] += __shfl_down_sync(0xffffffffu, o[d], 8);
        if (lane < G) {
          float mh = 0.f, lh = 0.f;
  #pragma unroll
          for (int h = 0; h < G; ++h)
            if (lane == h) {
              mh = m[h];
              lh = l[h];
            }
          if (a.n_split == 1) {
            const float inv = lh > 0.f ? 1.f / lh : 0.f;
            const size_t row = (size_t)col_head(lane) * HD;
            if (a.xop) {
              const int r = col_slot(lane);
              if (r < a.nb) {
  #pragma unroll
                for (int d = 0; d < HD; ++d) {
                  const float x = o[d] * inv;
                  const __nv_bfloat16 hi = __float2bfloat16_rn(x);
                  a.xop[(size_t)r * a.xop_ld + row + d] = hi;
                  a.xop[(size_t)(a.bp + r) * a.xop_ld + row + d] = __float2bfloat16_rn(x - __bfloat162float(hi));
                }
              }
            } else {
  #pragma unroll
              for (int d = 0; d < HD; d += 4)
                *reinterpret_cast<float4 *>(a.out + row + d) =
                    make_float4(o[d] * inv, o[d + 1] * inv, o[d + 2] * inv, o[d + 3] * inv);
            }
          } else {
            const uint32_t rr = (uint32_t)(lane % ns);
            float *dst = recv + ((lane / ns) * ns + split) * (HD + 4);
            const uint32_t mb = cl_peer(bar.merge_full, rr);
  #pragma unroll
            for (int d = 0; d < HD; d += 4)
              cl_st_v4(cl_peer(dst + d, rr), make_float4(o[d], o[d + 1], o[d + 2], o[d + 3]), mb);
            cl_st_v2(cl_peer(dst + HD, rr), make_float2(mh, lh), mb);
          }
        }
      }
    }
    if (threadIdx.x == 128) ktrace(a.tr, 4);
    if (clustered && nloc > 0) {
      // merge this CTA's query heads over the splits, in split order
      if (!cl_mbar_wait(bar.merge_full, 0) && lane == 0) set_error(err, kErrTimeout);
      for (int idx = tid; idx < nloc * HD; idx += 128) {
        const int j = idx / HD, d = idx - j * HD;
        const float *R = recv + (size_t)j * ns * (HD + 4);
        float M = -INFINITY;
        for (int s2 = 0; s2 < ns; ++s2) M = fmaxf(M, R[s2 * (HD + 4) + HD]);
        float Ls = 0.f, Os = 0.f;
        for (int s2 = 0; s2 < ns; ++s2) {
          const float *Rs = R + s2 * (HD + 4);
          if (Rs[HD] == -INFINITY) continue;
          const float f = exp2f(Rs[HD] - M);
          Ls = fmaf(Rs[HD + 1], f, Ls);
          Os = fmaf(Rs[d], f, Os);
        }
        const float x = Ls > 0.f ? Os / Ls : 0.f;
        const int hc = split + j * ns;
        const size_t col = (size_t)col_head(hc) * HD + d;
        if (a.xop) {
          const int r = col_slot(hc);
          if (r < a.nb) {
            const __nv_bfloat16 hi = __float2bfloat16_rn(x);
            a.xop[(size_t)r * a.xop_ld + col] = hi;
            a.xop[(size_t)(a.bp + r) * a.xop_ld + col] = __float2bfloat16_rn(x - __bfloat162float(hi));
          }
        } else {
          a.out[col] = x;
        }
      }
    }
  }
  tc_fence_before();
  if (clustered) {   // no CTA ends while a peer may still store into it
    if (!cl_waited) cl_wait();
    cl_arrive();
    cl_wait();
  }
  __syncthreads();
  if (threadIdx.x == 0) ktrace(a.tr, 5);
  if (warp == 1) tmem_dealloc(taddr, TCOLS);
}

// ------------------------------------------------------------------ persistent
// Batched slots with one CTA's worth of work per (slot, KV head) item and more
// items than SMs (head_dim 128, no splits): one CTA per SM walks a list of
// items, and its TMA ring runs on across them, so the next item's first tiles
// are in flight while the current one finishes (a grid of short CTAs pays each
// CTA's start and drain instead).  Items are ranked longest first (slot order,
// then KV head).  With a claim counter the producer takes the next ranked
// item with one atomic add when it reaches the last tile of the current one
// (list scheduling in rank order: a CTA whose SM streams faster takes more;
// the ring ahead of the consumers hides the round trip); without
// one, CTA c takes its k-th item at k * grid + c for even k and
// k * grid + grid - 1 - c for odd k.  The producer publishes each item through
// a small queue in shared memory that the MMA and softmax warps read in order.
// Q (shared memory) and O (TMEM) are double-buffered by item parity; the roles
// and the per-tile protocol are those of k_attn_tc.
struct TpItem {
  int j;       // ranked item, or -1 past the CTA's last
  int b, g;    // slot and KV head
  int pos, lo; // attended positions [lo, pos]
  int tb, nt;  // first tile and tile count
};

__device__ __forceinline__ TpItem tp_item(const AttnTcArgs &a, int j) {
  TpItem it;
  it.j = j >= 0 && j < a.nb * a.n_kv ? j : -1;
  if (it.j < 0) {
    it.b = it.g = it.pos = it.lo = it.tb = it.nt = 0;
    return it;
  }
  const int z = j / a.n_kv;
  it.g = j - z * a.n_kv;
  it.b = a.use_order ? (int)a.order[z] : z;
  it.pos = a.pos[it.b];
  it.lo = a.window > 0 ? max(0, it.pos - a.window + 1) : 0;
  it.tb = it.lo / kTile;
  it.nt = it.pos / kTile - it.tb + 1;
  return it;
}

constexpr int kTpHd = 128;
constexpr int kTpQueue = 8;         // item queue entries (the producer runs at most a ring ahead)
constexpr uint32_t kTpCols = 128;   // S at column 0, O of even / odd items at 32 / 64

__host__ __device__ constexpr int tp_smem(int nstages) {
  return 1024 + nstages * TL<kTpHd>::STAGE + 2 * TL<kTpHd>::PT + 2 * TL<kTpHd>::QT + 1024;
}

template <int G>
__global__ void __launch_bounds__(kTThreads, 1) k_attn_tp(const AttnTcArgs a) {
  constexpr int HD = kTpHd;
  constexpr int KT = TL<HD>::KT, STAGE = TL<HD>::STAGE, PT = TL<HD>::PT, QT = TL<HD>::QT;
  constexpr int PCH = TL<HD>::PCH;
  const int NS = a.nstages;

  const uint32_t base = smem_addr(t_smem);
  uint8_t *sm = t_smem + ((1024u - (base & 1023u)) & 1023u);
  uint8_t *ring = sm;
  uint8_t *P = ring + (size_t)NS * STAGE;
  uint8_t *Qb = P + 2 * PT;   // two Q tiles
  uint64_t *full = reinterpret_cast<uint64_t *>(Qb + 2 * QT);
  uint64_t *empty = full + NS;
  uint64_t *s_full = empty + NS, *s_empty = s_full + 1;
  uint64_t *p_full = s_empty + 1, *p_empty = p_full + 2;
  uint64_t *o_full = p_empty + 2, *q_ready = o_full + 1, *o_free = q_ready + 2;
  uint64_t *it_full = o_free + 2, *it_empty = it_full + kTpQueue;
  uint32_t *tslot = reinterpret_cast<uint32_t *>(it_empty + kTpQueue);
  float *red = reinterpret_cast<float *>(tslot + 4);   // [2][4][8] maxima, then [4][8] sums
  int *itq = reinterpret_cast<int *>(red + 96);        // [kTpQueue] ranked items (-1: no more)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    ktrace(a.tr, 0);
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(s_full, 1);
    mbar_init(s_empty, 4);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&p_full[i], 4);
      mbar_init(&p_empty[i], 1);
      mbar_init(&q_ready[i], 4);
      mbar_init(&o_free[i], 4);
    }
    for (int i = 0; i < kTpQueue; ++i) {
      mbar_init(&it_full[i], 1);
      mbar_init(&it_empty[i], 5);   // the MMA thread and the four softmax warps
    }
    mbar_init(o_full, 1);
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tslot, kTpCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t taddr = *tslot;
  const uint32_t t_s = taddr;
  auto t_o = [&](int k) { return taddr + 32u + 32u * (uint32_t)(k & 1); };

  if (warp == 0) {
    if (lane == 0) {
      const int items = a.nb * a.n_kv, grid = (int)gridDim.x, c = (int)blockIdx.x;
      auto claim = [&](int k) -> int {
        if (a.tp_claim) {
          const unsigned v = atomicAdd(a.tp_claim, 1u);
          return v < (unsigned)items ? (int)v : -1;
        }
        const int j = k * grid + ((k & 1) ? grid - 1 - c : c);
        return j < items ? j : -1;
      };
      // queue entry k: item k of this CTA (-1: no more)
      auto publish = [&](int k, int j) -> bool {
        const int e = k % kTpQueue;
        if (k >= kTpQueue && !mbar_wait(&it_empty[e], ((k / kTpQueue) - 1) & 1)) return false;
        itq[e] = j;
        mbar_arrive(&it_full[e]);
        return true;
      };
      // a tile holding an item's own position waits for the kernel that wrote
      // this step's K / V; earlier tiles were written by earlier steps
      bool waited = false, ok = true;
      int i = 0;
      int j = claim(0);
      ok = publish(0, j);
      for (int k = 0; ok && j >= 0; ++k) {
        // the next item is claimed at this one's last tile (earlier claims
        // would let the first CTAs to start take two items each) and
        // published once that tile is issued
        int jn = -1;
        bool claimed = false;
        const TpItem it = tp_item(a, j);
        int32_t *err = &a.slots[it.b].io->error;
        const CUtensorMap *maps = static_cast<const CUtensorMap *>(a.slots[it.b].maps) + 2 * a.layer;
        for (int t = 0; t < it.nt; ++t, ++i) {
          const int T = it.tb + t, s = i % NS, r = i / NS;
          if (t == it.nt - 1) {
            jn = claim(k + 1);
            claimed = true;
          }
          if (!waited && ((T + 1) * kTile > it.pos || i == NS)) {
            ktrace(a.tr, 6);
            pdl_wait();
            pdl_trigger();
            ktrace(a.tr, 7);
            waited = true;
          }
          if (i >= NS && !mbar_wait(&empty[s], (r - 1) & 1)) {
            set_error(err, kErrTimeout);
            ok = false;
            break;
          }
          const int y = it.g * a.cap + (T * kTile) % a.cap;
          uint8_t *kt = ring + (size_t)s * STAGE, *vt = kt + KT;
          mbar_arrive_expect_tx(&full[s], STAGE);
#pragma unroll
          for (int cc = 0; cc < HD / 64; ++cc) {
            tma_load_2d(kt + cc * kBox, maps, cc * 64, y, &full[s]);
            tma_load_2d(vt + cc * kBox, maps + 1, cc * 64, y, &full[s]);
          }
        }
        if (ok && !claimed) jn = claim(k + 1);
        if (ok && !publish(k + 1, jn)) {
          set_error(err, kErrTimeout);
          ok = false;
        }
        j = jn;
      }
      if (!waited) {
        pdl_wait();
        pdl_trigger();
      }
      if (a.tp_claim) {
        // every CTA is past its last claim once all have counted themselves
        // done: the last one resets the counters for the next launch
        __threadfence();
        if (atomicAdd(a.tp_claim + 1, 1u) == (unsigned)grid - 1u) {
          atomicExch(a.tp_claim, 0u);
          atomicExch(a.tp_claim + 1, 0u);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(128, 16);
      constexpr uint32_t idesc_o = idesc_bf16_f32(128, 16) | (1u << 15);   // V^T MN-major as A
      bool ok = true;
      int kq = 0;   // queue entries read
      auto next_item = [&]() -> TpItem {
        const int e = kq % kTpQueue;
        if (!mbar_wait(&it_full[e], (kq / kTpQueue) & 1)) {
          ok = false;
          return tp_item(a, -1);
        }
        const int jj = itq[e];
        mbar_arrive(&it_empty[e]);
        ++kq;
        return tp_item(a, jj);
      };
      // S of ring tile i for item kk
      auto issue_s = [&](int i, int kk) {
        const uint8_t *kt = ring + (size_t)(i % NS) * STAGE;
        const uint8_t *Q = Qb + (size_t)(kk & 1) * QT;
#pragma unroll
        for (int cc = 0; cc < HD / 64; ++cc)
#pragma unroll
          for (int kc = 0; kc < 4; ++kc)
            mma_bf16(t_s, desc_k_sw128(kt + cc * kBox, kc * 32), desc_k_sw128(Q + cc * 2048, kc * 32),
                     idesc_s, cc > 0 || kc > 0);
        mma_commit(s_full);
      };
      TpItem cur = next_item();
      int32_t *merr = cur.j >= 0 ? &a.slots[cur.b].io->error : nullptr;
      if (cur.j >= 0) {
        ok = mbar_wait(&q_ready[0], 0) && mbar_wait(&full[0], 0);
        if (ok) {
          tc_fence_after();
          issue_s(0, 0);
        }
      }
      // the CTA's tiles in order: item k, its tile t, ring index i.  Within an
      // item, S of tile i + 1 goes out before P V of tile i; at an item's end,
      // P V first (the next item's Q is staged after the softmax warps have
      // published this item's last P)
      int k = 0, t = 0;
      for (int i = 0; cur.j >= 0 && ok; ++i) {
        int nk = k, ntt = t + 1;
        TpItem nxt = cur;
        if (ntt == cur.nt) {
          nk = k + 1;
          ntt = 0;
          nxt = next_item();
          if (!ok) break;
        }
        const bool boundary = nk != k;
        if (!boundary) {
          ok = mbar_wait(&full[(i + 1) % NS], ((i + 1) / NS) & 1) && mbar_wait(s_empty, i & 1);
          if (!ok) break;
          tc_fence_after();
          issue_s(i + 1, nk);
        }
        ok = mbar_wait(&p_full[i & 1], (i >> 1) & 1);
        // O buffer k & 1 was read out after item k - 2
        if (ok && t == 0 && k >= 2) ok = mbar_wait(&o_free[k & 1], ((k >> 1) - 1) & 1);
        if (!ok) break;
        tc_fence_after();
        const uint8_t *pt = P + (size_t)(i & 1) * PT;
        const uint8_t *vt = ring + (size_t)(i % NS) * STAGE + KT;
#pragma unroll
        for (int pc = 0; pc < kTile / 16; ++pc) {
          const uint64_t dp = desc_k_sw128(pt + (pc >> 2) * PCH, (pc & 3) * 32);
          const uint64_t dv = desc_mn_sw128(vt + pc * 2048, kBox);
          mma_bf16(t_o(k), dv, dp, idesc_o, t > 0 || pc > 0);
        }
        mma_commit(o_full);
        mma_commit(&p_empty[i & 1]);
        mma_commit(&empty[i % NS]);
        if (boundary && nxt.j >= 0) {
          ok = mbar_wait(&full[(i + 1) % NS], ((i + 1) / NS) & 1) && mbar_wait(s_empty, i & 1) &&
               mbar_wait(&q_ready[nk & 1], (nk >> 1) & 1);
          if (!ok) break;
          tc_fence_after();
          issue_s(i + 1, nk);
        }
        k = nk;
        t = ntt;
        cur = nxt;
        if (cur.j >= 0) merr = &a.slots[cur.b].io->error;
      }
      if (!ok && merr) set_error(merr, kErrTimeout);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------ softmax warps 2-5
    const int q = warp & 3, tid = threadIdx.x - 64;   // position 32 q + lane of each tile
    bool ok = true;
    int kq = 0;   // queue entries read
    auto next_item = [&]() -> TpItem {
      const int e = kq % kTpQueue;
      int jj = -1;
      if (ok && mbar_wait(&it_full[e], (kq / kTpQueue) & 1)) jj = itq[e];
      else ok = false;
      __syncwarp();
      if (lane == 0) mbar_arrive(&it_empty[e]);
      ++kq;
      return tp_item(a, jj);
    };
    auto stage_q = [&](const TpItem &it, int kk) {
      uint8_t *Q = Qb + (size_t)(kk & 1) * QT;
      for (int i = tid; i < G * HD; i += 128) {
        const int h = i / HD, d = i - h * HD;
        const float v = a.q[((size_t)it.b * a.n_head + it.g * G + h) * HD + d] * a.qscale;
        const __nv_bfloat16 hi = __float2bfloat16_rn(v);
        const __nv_bfloat16 lo = __float2bfloat16_rn(v - __bfloat162float(hi));
        uint8_t *tile = Q + (d >> 6) * 2048;
        *reinterpret_cast<__nv_bfloat16 *>(tile + sw128(h, (d & 63) * 2)) = hi;
        *reinterpret_cast<__nv_bfloat16 *>(tile + sw128(8 + h, (d & 63) * 2)) = lo;
      }
      fence_async_smem();
      epi_sync_t();
      if (lane == 0) mbar_arrive(&q_ready[kk & 1]);
    };
    // Q and P: only rows h and 8 + h are ever written; the rest must be zero
    for (int i = tid * 16; i < 2 * QT; i += 128 * 16) *reinterpret_cast<uint4 *>(Qb + i) = make_uint4(0, 0, 0, 0);
    for (int i = tid * 16; i < 2 * PT; i += 128 * 16) *reinterpret_cast<uint4 *>(P + i) = make_uint4(0, 0, 0, 0);
    pdl_wait();   // q comes from the QKV kernel
    epi_sync_t();
    TpItem cur = next_item();
    if (cur.j >= 0) stage_q(cur, 0);
    if (tid == 0) ktrace(a.tr, 1);

    constexpr float kTau = 8.f;
    int i = 0;
    for (int k = 0; cur.j >= 0; ++k) {
      int32_t *err = &a.slots[cur.b].io->error;
      float m[G], l[G];
#pragma unroll
      for (int h = 0; h < G; ++h) {
        m[h] = -INFINITY;
        l[h] = 0.f;
      }
      for (int t = 0; t < cur.nt; ++t, ++i) {
        if (ok && !mbar_wait(s_full, i & 1)) {
          ok = false;
          if (lane == 0) set_error(err, kErrTimeout);
        }
        float v[32];
        if (ok) {
          tc_fence_after();
          tmem_ld32(t_s + ((uint32_t)(32 * q) << 16), v);
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = 0.f;
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(s_empty);
        const int p = (cur.tb + t) * kTile + 32 * q + lane;
        const bool valid = p >= cur.lo && p <= cur.pos;
        float sc[G];
        float *rm = red + (i & 1) * 32;
#pragma unroll
        for (int h = 0; h < G; ++h) {
          sc[h] = valid ? v[h] + v[8 + h] : -INFINITY;
          const float mx = warp_max(sc[h]);
          if (lane == 0) rm[q * 8 + h] = mx;
        }
        epi_sync_t();
        bool move = false;
        float scale[G];
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float mt = fmaxf(fmaxf(rm[h], rm[8 + h]), fmaxf(rm[16 + h], rm[24 + h]));
          scale[h] = 1.f;
          if (mt > m[h] + kTau) {
            scale[h] = m[h] == -INFINITY ? 0.f : exp2f(m[h] - mt);
            m[h] = mt;
            l[h] *= scale[h];
            move = true;
          }
        }
        if (t > 0) {
          // the previous tile's P V product is done; rescale O if the reference max moved
          if (ok && !mbar_wait(o_full, (i - 1) & 1)) {
            ok = false;
            if (lane == 0) set_error(err, kErrTimeout);
          }
          if (ok && move) {
            tc_fence_after();
            float w[32];
            tmem_ld32(t_o(k) + ((uint32_t)(32 * q) << 16), w);
#pragma unroll
            for (int h = 0; h < G; ++h) {
              w[h] *= scale[h];
              w[8 + h] *= scale[h];
            }
            tmem_st32(t_o(k) + ((uint32_t)(32 * q) << 16), w);
            tc_fence_before();
          }
        }
        float pp[G];
#pragma unroll
        for (int h = 0; h < G; ++h) {
          pp[h] = (valid && m[h] != -INFINITY) ? exp2f(sc[h] - m[h]) : 0.f;
          l[h] += pp[h];
        }
        // P into buffer i & 1, once the P V product of tile i - 2 is done
        if (i >= 2 && ok && !mbar_wait(&p_empty[i & 1], ((i >> 1) - 1) & 1)) {
          ok = false;
          if (lane == 0) set_error(err, kErrTimeout);
        }
        uint8_t *pt = P + (size_t)(i & 1) * PT + ((32 * q + lane) >> 6) * PCH;
        const int cb = ((32 * q + lane) & 63) * 2;
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const __nv_bfloat16 hi = __float2bfloat16_rn(pp[h]);
          const __nv_bfloat16 lo2 = __float2bfloat16_rn(pp[h] - __bfloat162float(hi));
          *reinterpret_cast<__nv_bfloat16 *>(pt + sw128(h, cb)) = hi;
          *reinterpret_cast<__nv_bfloat16 *>(pt + sw128(8 + h, cb)) = lo2;
        }
        fence_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[i & 1]);
      }
      // the next item and its Q (into the buffer of item k - 1, whose S
      // products this warp group has consumed)
      const TpItem nxt = next_item();
      if (nxt.j >= 0) stage_q(nxt, k + 1);
      // row sums over the item's positions (fixed order: lanes, then warps)
      float *rs = red + 64;
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float sw = warp_sum(l[h]);
        if (lane == 0) rs[q * 8 + h] = sw;
      }
      epi_sync_t();
#pragma unroll
      for (int h = 0; h < G; ++h) l[h] = rs[h] + rs[8 + h] + rs[16 + h] + rs[24 + h];
      // O^T of the item: thread = dim d, columns h / 8 + h = high / low parts of head h
      float oh[G];
#pragma unroll
      for (int h = 0; h < G; ++h) oh[h] = 0.f;
      if (ok && !mbar_wait(o_full, (i - 1) & 1)) {
        ok = false;
        if (lane == 0) set_error(err, kErrTimeout);
      }
      if (ok) {
        tc_fence_after();
        float w[32];
        tmem_ld32(t_o(k) + ((uint32_t)(32 * q) << 16), w);
#pragma unroll
        for (int h = 0; h < G; ++h) oh[h] = w[h] + w[8 + h];
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&o_free[k & 1]);
      const int d = 32 * q + lane;
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const size_t col = (size_t)(cur.g * G + h) * HD + d;
        const float x = l[h] > 0.f ? oh[h] / l[h] : 0.f;
        const __nv_bfloat16 hi = __float2bfloat16_rn(x);
        a.xop[(size_t)cur.b * a.xop_ld + col] = hi;
        a.xop[(size_t)(a.bp + cur.b) * a.xop_ld + col] = __float2bfloat16_rn(x - __bfloat162float(hi));
      }
      cur = nxt;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) ktrace(a.tr, 5);
  if (warp == 1) tmem_dealloc(taddr, kTpCols);
}

template <int HD, int G>
cudaError_t launch_g(const AttnTcArgs &a, cudaStream_t st, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  const int T = a.slots && a.tok_group > 1 ? a.tok_group : 1;
  cfg.gridDim = dim3(a.n_split, a.n_kv, a.slots ? (a.nb + T - 1) / T : 1);
  cfg.blockDim = dim3(kTThreads);
  cfg.dynamicSmemBytes = attn_tc_smem(HD, a.nstages);
  cfg.stream = st;
  if (a.n_split < 1 || a.n_split > kMaxSplit) return cudaErrorInvalidValue;
  cudaLaunchAttribute attr[2];
  int na = 0;
  attr[na].id = cudaLaunchAttributeClusterDimension;   // the splits of one KV head
  attr[na].val.clusterDim.x = a.n_split;
  attr[na].val.clusterDim.y = 1;
  attr[na].val.clusterDim.z = 1;
  ++na;
  if (pdl) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, k_attn_tc<HD, G>, a);
}

template <int G>
cudaError_t launch_tp(const AttnTcArgs &a, cudaStream_t st, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(std::min(a.nb * a.n_kv, a.persist));
  cfg.blockDim = dim3(kTThreads);
  cfg.dynamicSmemBytes = tp_smem(a.nstages);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  int na = 0;
  if (pdl) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, k_attn_tp<G>, a);
}

template <int HD>
cudaError_t launch_hd_tc(int G, const AttnTcArgs &a, cudaStream_t st, bool pdl) {
  switch (G) {
    case 1: return launch_g<HD, 1>(a, st, pdl);
    case 2: return launch_g<HD, 2>(a, st, pdl);
    case 4: return launch_g<HD, 4>(a, st, pdl);
    case 8: return launch_g<HD, 8>(a, st, pdl);
    default: return cudaErrorInvalidValue;
  }
}

template <int HD>
cudaError_t prepare_hd_tc() {
  const int smem = attn_tc_smem(HD, attn_tc_stages(HD));
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(k_attn_tc<HD, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) != cudaSuccess) return e;
  if ((e = cudaFuncSetAttribute(k_attn_tc<HD, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) != cudaSuccess) return e;
  if ((e = cudaFuncSetAttribute(k_attn_tc<HD, 4>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) != cudaSuccess) return e;
  return cudaFuncSetAttribute(k_attn_tc<HD, 8>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
}

}  // namespace

int attn_tc_stages(int head_dim) { return 3; }

int attn_tc_max_split() { return kMaxSplit; }

int attn_tc_smem(int head_dim, int nstages) {
  const int stage = 2 * (head_dim / 64) * kBox;
  const int p_tiles = head_dim == 128 ? 2 * 2 * 2048 : 2 * 2 * kBox;
  return 1024 + nstages * stage + p_tiles + (head_dim / 64) * 2048 + 1024 + merge_floats(head_dim) * 4;
}

cudaError_t launch_attn_tc(int head_dim, int group, const AttnTcArgs &a, cudaStream_t st, bool pdl) {
  if (a.persist > 0) {
    if (head_dim != kTpHd || !a.slots || a.n_split != 1 || a.tok_group > 1 || a.shared_cache || !a.xop)
      return cudaErrorInvalidValue;
    switch (group) {
      case 1: return launch_tp<1>(a, st, pdl);
      case 2: return launch_tp<2>(a, st, pdl);
      case 4: return launch_tp<4>(a, st, pdl);
      case 8: return launch_tp<8>(a, st, pdl);
      default: return cudaErrorInvalidValue;
    }
  }
  if (head_dim == 128) return launch_hd_tc<128>(group, a, st, pdl);
  if (head_dim == 64) return launch_hd_tc<64>(group, a, st, pdl);
  return cudaErrorInvalidValue;
}

cudaError_t prepare_attn_tc_kernels() {
  cudaError_t e = prepare_hd_tc<128>();
  if (e != cudaSuccess) return e;
  const int tps = tp_smem(attn_tc_stages(kTpHd));
  if ((e = cudaFuncSetAttribute(k_attn_tp<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, tps)) != cudaSuccess) return e;
  if ((e = cudaFuncSetAttribute(k_attn_tp<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, tps)) != cudaSuccess) return e;
  if ((e = cudaFuncSetAttribute(k_attn_tp<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, tps)) != cudaSuccess) return e;
  if ((e = cudaFuncSetAttribute(k_attn_tp<8>, cudaFuncAttributeMaxDynamicSharedMemorySize, tps)) != cudaSuccess) return e;
  return prepare_hd_tc<64>();
}

}  // namespace pnb
