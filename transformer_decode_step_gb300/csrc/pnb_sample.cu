// pnb_sample.cu - the decode loop's token sampler ("Engine Architecture",
// section "Sampling"):
//   (1) z = logit / temperature (temperature <= 0: greedy argmax);
//   (2) repetition penalty on each distinct token of the recent window
//       (z / penalty when z > 0, z * penalty otherwise);
//   (3) top-k, (4) top-p ("until the cumulative probability exceeds p"),
//   (5) softmax, (6) multinomial draw with u from the state's draw counter.
// The draw order is z descending, token id ascending on ties.  Nothing is
// sorted: each of top-k, top-p and the draw is a radix descent over the
// 32-bit order key of z (four 8-bit levels, a 256-bin histogram each) that
// finds the element at which a running total - a count for top-k, softmax
// mass for top-p and the draw - first exceeds a threshold.  Masses are
// exp(z - z_max) in 64-bit fixed point (units of 2^-40), so every sum is an
// exact integer and the result does not depend on the order of atomics.
//
// One sequence is one thread-block cluster of kSampCluster CTAs; CTA r owns
// a contiguous range of token ids.  Each level, every CTA builds the
// histogram of its range and stores it into every CTA's shared memory
// (distributed shared memory); after one cluster barrier each CTA sums the
// copies, so all CTAs take the same decisions.  (The receive buffers
// alternate between two copies: a CTA rewrites a copy only after the next
// barrier, which every peer reaches after its reads of that copy.)  Over all
// tokens a CTA counts into kPrivCopies histograms (the top byte of the key
// has few distinct values, so one histogram would serialise on a handful of
// addresses).  When the tokens up to the first level's chosen bin number at
// most kListMax in the whole cluster, each CTA moves its own into a
// shared-memory list and every later level and descent runs on the lists;
// when they number at most kSoloMax, CTA 0 gathers them and finishes alone.
// z is written back over the logits (the pages' sampler also changes them in
// place).
#include "pnb_kernels.cuh"

#include <climits>

namespace pnb {
namespace {

constexpr int kSampThreads = 1024;
constexpr int kSampWarps = kSampThreads / 32;
constexpr int kSampCluster = 8;
constexpr int kListMax = 4096;     // list entries per CTA (and in the whole cluster)
constexpr int kSoloMax = 1024;     // lists this short are finished by CTA 0 alone
constexpr int kTailMax = 256;      // top-k sets this small are sorted and scanned directly
constexpr int kPrivCopies = 8;     // histograms per CTA over all tokens (warp w uses w % 8)
constexpr int kPrivStride = 257;   // a copy's row, padded so copies start in different banks
constexpr float kMassUnit = 1099511627776.0f;  // 2^40

// A bin's 64-bit total is counted as three 32-bit words of 14-bit chunks
// (total = w0 + w1 * 2^14 + w2 * 2^28), so every add is a native,
// non-returning 32-bit shared-memory atomic and no word can overflow: a mass
// is at most 2^40; one private copy takes at most n_vocab / 64 < 2^16 values
// (n_vocab < 2^22), the list histogram at most kListMax.
struct SampSmem {
  // every CTA's histogram as pushed into this CTA: [copy][from rank][bin] =
  // {total, count << 32 | lowest id}
  ulonglong2 xin[2][kSampCluster][256];
  unsigned long long mine_tot[256], mine_cf[256];  // this CTA's histogram, to push
  unsigned long long xs[2];         // published scalar (cluster_gather)
  unsigned long long tot[256];      // the cluster's merged totals
  int first[256];
  unsigned cnt[256];
  int lfirst[256];                  // this CTA's lowest id per bin
  unsigned h0[256], h1[256], h2[256];
  unsigned long long gath[kSampCluster];
  unsigned long long wsum[kSampWarps];
  unsigned long long before, t, total;
  int bin, found;
  unsigned nlist, nle;
  float zmax;
  float lz[kListMax];
  int lid[kListMax];
  unsigned p0[kPrivCopies * kPrivStride], p1[kPrivCopies * kPrivStride];
  unsigned p2[kPrivCopies * kPrivStride], pcnt[kPrivCopies * kPrivStride];
  // followed by the recent-token bitmap, (n_vocab + 31) / 32 words
};

// ------------------------------------------------------------- cluster
__device__ __forceinline__ void cl_sync() {
  asm volatile("barrier.cluster.arrive.release;" ::: "memory");
  asm volatile("barrier.cluster.wait.acquire;" ::: "memory");
}
__device__ __forceinline__ uint32_t cl_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cl_peer(const void *local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr(local)), "r"(rank));
  return r;
}
__device__ __forceinline__ unsigned long long cl_ld_u64(uint32_t a) {
  unsigned long long v;
  asm volatile("ld.shared::cluster.u64 %0, [%1];" : "=l"(v) : "r"(a) : "memory");
  return v;
}
__device__ __forceinline__ void cl_st_u32(uint32_t a, unsigned v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(a), "r"(v) : "memory");
}
__device__ __forceinline__ void cl_st_v2u64(uint32_t a, unsigned long long x, unsigned long long y) {
  asm volatile("st.shared::cluster.v2.u64 [%0], {%1, %2};" ::"r"(a), "l"(x), "l"(y) : "memory");
}

// merge rounds: round k publishes into copy k & 1.  solo: the candidates are
// in CTA 0's list and CTA 0 finishes alone (no more cluster barriers); idle:
// this CTA is not CTA 0 and has nothing left but the final barrier.
struct Cl {
  uint32_t rank;
  int round;
  bool solo, idle;
};

// every CTA contributes v; afterwards sm.gath[r] holds CTA r's value in every CTA
__device__ void cluster_gather(SampSmem &sm, Cl &cl, unsigned long long v) {
  const int b = cl.round++ & 1;
  if (threadIdx.x == 0) sm.xs[b] = v;
  cl_sync();
  if (threadIdx.x < kSampCluster) sm.gath[threadIdx.x] = cl_ld_u64(cl_peer(&sm.xs[b], threadIdx.x));
  __syncthreads();
}

// ------------------------------------------------------------- keys
// order key: ascending key = descending z; -0 is keyed as +0
__device__ __forceinline__ uint32_t order_key(float z) {
  uint32_t b = __float_as_uint(z);
  if (b == 0x80000000u) b = 0;
  return (b & 0x80000000u) ? b : (~b & 0x7FFFFFFFu);
}

__device__ __forceinline__ float key_value(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? k : (~k & 0x7FFFFFFFu));
}

__device__ __forceinline__ unsigned long long mass_of(float z, float zmax) {
  return __float2ull_rn(expf(z - zmax) * kMassUnit);
}

// SplitMix64 (Steele, Lea & Flood, OOPSLA 2014): word n of the sequence
// seeded with `seed`; the top 24 bits give u in [0, 1)
__device__ __forceinline__ double draw_uniform(unsigned long long seed, unsigned long long n) {
  unsigned long long z = seed + (n + 1ull) * 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  z ^= z >> 31;
  return (double)(z >> 40) * (1.0 / 16777216.0);
}

// a prefix of the draw order: (key < k) or (key == k and id <= id)
struct Cut {
  uint32_t key;
  int id;
};
__device__ __forceinline__ Cut all_cut() { return Cut{0xFFFFFFFFu, INT_MAX}; }

__device__ __forceinline__ bool in_cut(const Cut &c, uint32_t k, int id) {
  return k < c.key || (k == c.key && id <= c.id);
}

// the elements a CTA walks: its token range [lo, hi) of z in global memory
// (index = id), or its shared-memory list [0, hi) (ids within its range, any
// order)
struct Src {
  const float *z;
  const int *id;  // nullptr: tokens, index = id
  int lo, hi;
  __device__ __forceinline__ float zv(int i) const { return z[i]; }
  __device__ __forceinline__ int idv(int i) const { return id ? id[i] : i; }
};

// the threshold of a descent: t, or floor(frac * the total of the elements
// walked), known once the first level's histogram is complete
struct Thresh {
  unsigned long long t;
  double frac;
  bool use_frac;
};

// result of a descent: the key of the element where the running total first
// exceeds t, the total before that key's group, the group's total and its
// lowest id; t as used and the total of all elements walked
struct Hit {
  uint32_t key;
  unsigned long long before, group, t, total;
  int first;
};

__device__ __forceinline__ void add_chunks(unsigned *w0, unsigned *w1, unsigned *w2,
                                           unsigned long long v) {
  atomicAdd(w0, (unsigned)(v & 0x3FFFu));
  atomicAdd(w1, (unsigned)((v >> 14) & 0x3FFFu));
  atomicAdd(w2, (unsigned)(v >> 28));
}

__device__ __forceinline__ unsigned long long chunks(unsigned w0, unsigned w1, unsigned w2) {
  return (unsigned long long)w0 + ((unsigned long long)w1 << 14) + ((unsigned long long)w2 << 28);
}

// warp 0: the first of the 256 merged bins at which before + running sum
// exceeds the threshold (on the first level of a fractional threshold, t is
// fixed here from the merged total); with counts, also the number of
// elements in the bins up to the chosen one
__device__ __forceinline__ void pick_bin(SampSmem &sm, unsigned long long before,
                                         unsigned long long t, const Thresh &th, bool first_level,
                                         bool with_counts) {
  const int lane = threadIdx.x;
  unsigned long long v[8], own = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    v[j] = sm.tot[8 * lane + j];
    own += v[j];
  }
  unsigned long long incl = own;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long y = __shfl_up_sync(~0u, incl, o);
    if (lane >= o) incl += y;
  }
  if (first_level) {
    const unsigned long long total = __shfl_sync(~0u, incl, 31);
    if (th.use_frac) {
      t = (unsigned long long)floor((double)total * th.frac);
      if (t >= total && total) t = total - 1;
    }
    if (lane == 0) sm.total = total;
  }
  if (lane == 0) sm.t = t;
  unsigned long long run = before + incl - own;
  const bool mine = run <= t && t < run + own;
  if (mine) {
    int j = 0;
    while (j < 7 && run + v[j] <= t) run += v[j++];
    sm.bin = 8 * lane + j;
    sm.before = run;
  }
  // unreachable when the threshold is below the total; keep the last
  // non-empty bin so the descent still ends on an element
  const unsigned any = __ballot_sync(~0u, mine);
  if (!any) {
    const unsigned ne = __ballot_sync(~0u, own != 0);
    if (ne && lane == 31 - __clz(ne)) {
      int j = 7;
      while (j > 0 && v[j] == 0) --j;
      unsigned long long r = before + incl - own;
      for (int q = 0; q < j; ++q) r += v[q];
      sm.bin = 8 * lane + j;
      sm.before = r;
    } else if (!ne && lane == 0) {
      sm.bin = 255;
      sm.before = before;
    }
  }
  if (with_counts) {
    __syncwarp();
    const int b = sm.bin;
    unsigned c = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) c += 8 * lane + j <= b ? sm.cnt[8 * lane + j] : 0u;
    for (int o = 16; o; o >>= 1) c += __shfl_xor_sync(~0u, c, o);
    if (lane == 0) sm.nle = c;
  }
}

// this CTA's list: the tokens of its range inside cuts c, c1 and c2 (any
// order); returns their number, of which the first kListMax are stored
__device__ unsigned compact(SampSmem &sm, const float *z, int lo, int hi, const Cut &c,
                            const Cut &c1, const Cut &c2) {
  const int tid = threadIdx.x, lane = tid & 31;
  if (tid == 0) sm.nlist = 0;
  __syncthreads();
  for (int i0 = lo; i0 < hi; i0 += kSampThreads) {
    const int i = i0 + tid;
    const float v = i < hi ? z[i] : 0.0f;
    const uint32_t k = order_key(v);
    const bool in = i < hi && in_cut(c, k, i) && in_cut(c1, k, i) && in_cut(c2, k, i);
    const unsigned bal = __ballot_sync(~0u, in);
    if (!bal) continue;
    const int leader = __ffs(bal) - 1;
    unsigned base = 0;
    if (lane == leader) base = atomicAdd(&sm.nlist, (unsigned)__popc(bal));
    base = __shfl_sync(~0u, base, leader);
    if (in) {
      const unsigned slot = base + __popc(bal & ((1u << lane) - 1u));
      if (slot < (unsigned)kListMax) {
        sm.lz[slot] = v;
        sm.lid[slot] = i;
      }
    }
  }
  __syncthreads();
  return sm.nlist;
}

// this CTA's list entries inside cuts c, c1 and c2, moved to the front of the
// list (through the private-histogram words as scratch); at most kTailMax of
// them, which the caller knows from merged counts
__device__ unsigned filter_list(SampSmem &sm, int n, const Cut &c, const Cut &c1, const Cut &c2) {
  float *tz = reinterpret_cast<float *>(sm.p0);
  int *tid_ = reinterpret_cast<int *>(sm.p1);
  if (threadIdx.x == 0) sm.nlist = 0;
  __syncthreads();
  for (int i = threadIdx.x; i < n; i += kSampThreads) {
    const float v = sm.lz[i];
    const uint32_t k = order_key(v);
    const int id = sm.lid[i];
    if (in_cut(c, k, id) && in_cut(c1, k, id) && in_cut(c2, k, id)) {
      const unsigned slot = atomicAdd(&sm.nlist, 1u);
      if (slot < (unsigned)kTailMax) {
        tz[slot] = v;
        tid_[slot] = id;
      }
    }
  }
  __syncthreads();
  const unsigned m = min(sm.nlist, (unsigned)kTailMax);
  for (unsigned i = threadIdx.x; i < m; i += kSampThreads) {
    sm.lz[i] = tz[i];
    sm.lid[i] = tid_[i];
  }
  __syncthreads();
  return m;
}

// the cluster's tokens of the ranges inside cuts c, c1 and c2 - at most
// kListMax of them, which the caller knows from merged counts - into lists:
// each CTA compacts its range into its own list; when they number at most
// kSoloMax in all, each CTA stores its entries into CTA 0 after those of the
// CTAs before it, and from there CTA 0 goes on alone (one CTA's histogram
// over a short list costs less than a cluster barrier per level)
__device__ void to_list(SampSmem &sm, Cl &cl, Src &src, const Cut &c, const Cut &c1,
                        const Cut &c2) {
  const unsigned n = src.id ? filter_list(sm, src.hi, c, c1, c2)
                            : min(compact(sm, src.z, src.lo, src.hi, c, c1, c2), (unsigned)kListMax);
  cluster_gather(sm, cl, n);
  unsigned off = 0, total = 0;
  for (int r = 0; r < kSampCluster; ++r) {
    if (r == (int)cl.rank) off = total;
    total += (unsigned)sm.gath[r];
  }
  if (total > (unsigned)kSoloMax) {
    src = Src{sm.lz, sm.lid, 0, (int)n};
    return;
  }
  if (cl.rank != 0)
    for (unsigned j = threadIdx.x; j < n; j += kSampThreads) {
      cl_st_u32(cl_peer(&sm.lz[off + j], 0), __float_as_uint(sm.lz[j]));
      cl_st_u32(cl_peer(&sm.lid[off + j], 0), (unsigned)sm.lid[j]);
    }
  cl_sync();  // CTA 0's list is complete
  cl.solo = true;
  cl.idle = cl.rank != 0;
  src = Src{sm.lz, sm.lid, 0, cl.idle ? 0 : (int)total};
}

// cluster-wide radix descent over the elements inside c1 and c2, in the draw
// order, weighting each by 1 (kMass false) or by its fixed-point mass.  When
// the first level runs over tokens and the elements up to its chosen bin fit
// the lists, they move there and src becomes the list (the caller's later
// descents, which only need those elements, use it too).
template <bool kMass>
__device__ Hit descend(SampSmem &sm, Cl &cl, Src &src, const Cut &c1, const Cut &c2,
                       const Thresh &th) {
  const int tid = threadIdx.x, copy = (tid >> 5) % kPrivCopies;
  uint32_t prefix = 0, mask = 0;
  unsigned long long before = 0, t = th.t;
  const float zmax = sm.zmax;
  Hit h;
  h.total = 0;
  for (int level = 0; level < 4; ++level) {
    const int shift = 24 - 8 * level;
    const bool priv = src.id == nullptr;
    const bool counts = priv && level == 0;
    const int b = cl.round & 1;  // the publish copy of this level's merge
    if (priv) {
      for (int j = tid; j < kPrivCopies * kPrivStride; j += kSampThreads) {
        sm.p0[j] = 0;
        if (kMass) {
          sm.p1[j] = 0;
          sm.p2[j] = 0;
          if (counts) sm.pcnt[j] = 0;
        }
      }
    } else if (tid < 256) {
      sm.h0[tid] = 0;
      sm.h1[tid] = 0;
      sm.h2[tid] = 0;
    }
    if (tid < 256) sm.lfirst[tid] = INT_MAX;
    __syncthreads();
    for (int i = src.lo + tid; i < src.hi; i += kSampThreads) {
      const float z = src.zv(i);
      const uint32_t k = order_key(z);
      if ((k & mask) != prefix) continue;
      const int id = src.idv(i);
      if (!in_cut(c1, k, id) || !in_cut(c2, k, id)) continue;
      const int bin = (k >> shift) & 255;
      if (priv) {
        const int r = copy * kPrivStride + bin;
        if (kMass) {
          add_chunks(&sm.p0[r], &sm.p1[r], &sm.p2[r], mass_of(z, zmax));
          if (counts) atomicAdd(&sm.pcnt[r], 1u);
        } else {
          atomicAdd(&sm.p0[r], 1u);
        }
      } else if (kMass) {
        add_chunks(&sm.h0[bin], &sm.h1[bin], &sm.h2[bin], mass_of(z, zmax));
      } else {
        atomicAdd(&sm.h0[bin], 1u);
      }
      if (level == 3) atomicMin(&sm.lfirst[bin], id);
    }
    __syncthreads();
    if (tid < 256) {
      unsigned long long acc = 0;
      unsigned c = 0;
      if (priv) {
        for (int w = 0; w < kPrivCopies; ++w) {
          const int r = w * kPrivStride + tid;
          acc += kMass ? chunks(sm.p0[r], sm.p1[r], sm.p2[r]) : (unsigned long long)sm.p0[r];
          if (kMass && counts) c += sm.pcnt[r];
        }
      } else {
        acc = kMass ? chunks(sm.h0[tid], sm.h1[tid], sm.h2[tid]) : (unsigned long long)sm.h0[tid];
      }
      sm.mine_tot[tid] = acc;
      sm.mine_cf[tid] = ((unsigned long long)(kMass ? c : (unsigned)acc) << 32) |
                        (unsigned)sm.lfirst[tid];
    }
    __syncthreads();
    if (cl.solo) {
      if (tid < 256) {
        sm.tot[tid] = sm.mine_tot[tid];
        sm.cnt[tid] = (unsigned)(sm.mine_cf[tid] >> 32);
        sm.first[tid] = (int)(unsigned)sm.mine_cf[tid];
      }
    } else {
      // merge the cluster's histograms: push ours into every CTA (stores do
      // not wait), one barrier, then sum the copies locally
      for (int j = tid; j < kSampCluster * 256; j += kSampThreads) {
        const int r = j >> 8, bn = j & 255;
        cl_st_v2u64(cl_peer(&sm.xin[b][cl.rank][bn], r), sm.mine_tot[bn], sm.mine_cf[bn]);
      }
      ++cl.round;
      cl_sync();
    }
    if (!cl.solo && tid < 256) {
      unsigned long long s = 0;
      unsigned c = 0;
      int f = INT_MAX;
#pragma unroll
      for (int r = 0; r < kSampCluster; ++r) {
        const ulonglong2 e = sm.xin[b][r][tid];
        s += e.x;
        c += (unsigned)(e.y >> 32);
        f = min(f, (int)(unsigned)e.y);
      }
      sm.tot[tid] = s;
      sm.cnt[tid] = c;
      sm.first[tid] = f;
    }
    __syncthreads();
    if (tid < 32) pick_bin(sm, before, t, th, level == 0, counts);
    __syncthreads();
    const int bin = sm.bin;
    before = sm.before;
    t = sm.t;
    if (level == 0) h.total = sm.total;
    prefix |= (uint32_t)bin << shift;
    mask |= 0xFFu << shift;
    if (level == 3) {
      h.group = sm.tot[bin];
      h.first = sm.first[bin];
    }
    if (counts && sm.nle <= (unsigned)kListMax) {
      // the rest of this descent and the caller's next ones run on CTA 0's list
      const Cut up_to_bin{((uint32_t)bin << 24) | 0xFFFFFFu, INT_MAX};
      to_list(sm, cl, src, up_to_bin, c1, c2);
      if (cl.idle) return h;
    }
    __syncthreads();  // sm.bin etc. are rewritten next level
  }
  h.key = prefix;
  h.before = before;
  h.t = t;
  return h;
}

// id of the m-th element (1-based, id order) in the cluster inside c1 and c2
// whose key is `key`.  CTA ranges are in id order, so the CTAs' member counts
// say which CTA holds it; that CTA finds it in its range (tokens: per-warp
// contiguous id ranges counted, then walked by the warp that holds it; list:
// the member whose rank among the list's member ids is right).
__device__ int nth_id(SampSmem &sm, Cl &cl, const Src &src, const Cut &c1, const Cut &c2,
                      uint32_t key, unsigned long long m) {
  const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
  auto member = [&](int i) {
    const uint32_t k = order_key(src.zv(i));
    const int id = src.idv(i);
    return k == key && in_cut(c1, k, id) && in_cut(c2, k, id);
  };
  const int n = src.hi - src.lo;
  const int per = (n + kSampWarps - 1) / kSampWarps;
  const int wlo = src.lo + min(n, w * per), whi = src.lo + min(n, (w + 1) * per);
  unsigned long long cnt = 0;
  for (int base = wlo; base < whi; base += 32) {
    const int i = base + lane;
    cnt += __popc(__ballot_sync(~0u, i < whi && member(i)));
  }
  if (lane == 0) sm.wsum[w] = cnt;
  if (tid == 0) sm.found = INT_MAX;
  __syncthreads();
  unsigned long long local = 0, woff = 0;
  for (int j = 0; j < kSampWarps; ++j) {
    if (j == w) woff = local;
    local += sm.wsum[j];
  }
  unsigned long long off = 0;
  if (!cl.solo) {
    cluster_gather(sm, cl, local);
    for (uint32_t r = 0; r < cl.rank; ++r) off += sm.gath[r];
  }
  if (off < m && m <= off + local) {
    const unsigned long long ml = m - off;
    if (src.id) {
      for (int i = src.lo + tid; i < src.hi; i += kSampThreads) {
        if (!member(i)) continue;
        const int id = src.idv(i);
        unsigned long long r = 1;
        for (int j = src.lo; j < src.hi; ++j) r += (src.idv(j) < id && member(j)) ? 1u : 0u;
        if (r == ml) sm.found = id;
      }
    } else if (woff < ml && ml <= woff + cnt) {
      unsigned long long run = woff;
      for (int base = wlo; base < whi; base += 32) {
        const int i = base + lane;
        const unsigned bal = __ballot_sync(~0u, i < whi && member(i));
        const int c = __popc(bal);
        if (run + c >= ml) {
          unsigned bb = bal;
          for (unsigned long long r = run + 1; r < ml; ++r) bb &= bb - 1;
          if (lane == __ffs(bb) - 1) sm.found = i;
          break;
        }
        run += c;
      }
    }
  }
  __syncthreads();
  if (cl.solo) return sm.found;
  cluster_gather(sm, cl, (unsigned long long)(unsigned)sm.found);
  int id = INT_MAX;
  for (int r = 0; r < kSampCluster; ++r) id = min(id, (int)(unsigned)sm.gath[r]);
  return id;
}

// the `rank`-th element of a descent's group (1-based): its lowest id when
// rank is 1, every id (cut at INT_MAX) when it is the whole group
__device__ __forceinline__ int group_cut(SampSmem &sm, Cl &cl, const Src &src, const Cut &c1,
                                         const Cut &c2, const Hit &h, unsigned long long rank,
                                         unsigned long long members) {
  if (rank >= members) return INT_MAX;
  if (rank == 1) return h.first;
  return nth_id(sm, cl, src, c1, c2, h.key, rank);
}

// CTA 0 alone, with exactly the top-k candidates (n <= kTailMax) in its
// list: order them (each entry's rank is the number of entries before it in
// the draw order), take the running fixed-point masses in that order, then
// top-p and the draw are each the first position whose running mass exceeds
// its threshold - the same integers the radix descents compare
__device__ int sort_tail(SampSmem &sm, int n, bool top_p, float p, double u) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  float *sz = reinterpret_cast<float *>(sm.h0);
  int *sid = reinterpret_cast<int *>(sm.h1);
  if (tid < n) {
    const float zi = sm.lz[tid];
    const uint32_t ki = order_key(zi);
    const int idi = sm.lid[tid];
    int rank = 0;
    for (int j = 0; j < n; ++j) {
      const uint32_t kj = order_key(sm.lz[j]);
      rank += (kj < ki || (kj == ki && sm.lid[j] < idi)) ? 1 : 0;
    }
    sz[rank] = zi;
    sid[rank] = idi;
  }
  __syncthreads();
  // inclusive running masses over positions 0 .. kTailMax - 1 (8 warps)
  unsigned long long m = tid < n ? mass_of(sz[tid], sm.zmax) : 0ull;
  if (tid < kTailMax) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long y = __shfl_up_sync(~0u, m, o);
      if (lane >= o) m += y;
    }
    if (lane == 31) sm.wsum[warp] = m;
  }
  __syncthreads();
  if (tid < kTailMax) {
    for (int w = 0; w < warp; ++w) m += sm.wsum[w];
    sm.tot[tid] = m;
  }
  if (tid == 0) sm.found = -1;
  __syncthreads();
  unsigned long long total = sm.tot[n - 1];
  int nk = n;
  if (top_p) {
    unsigned long long t = (unsigned long long)floor((double)total * (double)fmaxf(p, 0.0f));
    if (t >= total) t = total - 1;
    if (tid < n && sm.tot[tid] > t && (tid == 0 || sm.tot[tid - 1] <= t)) sm.found = tid;
    __syncthreads();
    nk = sm.found + 1;
    total = sm.tot[nk - 1];
    __syncthreads();
    if (tid == 0) sm.found = -1;
    __syncthreads();
  }
  unsigned long long t = (unsigned long long)floor((double)total * u);
  if (t >= total) t = total - 1;
  if (tid < nk && sm.tot[tid] > t && (tid == 0 || sm.tot[tid - 1] <= t)) sm.found = tid;
  __syncthreads();
  return sid[max(sm.found, 0)];
}

__global__ void __cluster_dims__(kSampCluster, 1, 1) __launch_bounds__(kSampThreads, 1)
    k_sample(const __grid_constant__ SampleArgs a) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  SampSmem &sm = *reinterpret_cast<SampSmem *>(smem_raw);
  uint32_t *recent_bits = reinterpret_cast<uint32_t *>(smem_raw + sizeof(SampSmem));
  Cl cl{cl_rank(), 0, false, false};
  const SampleSlot &sl = a.slot[blockIdx.x / kSampCluster];
  const int V = a.n_vocab;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per = (V + kSampCluster - 1) / kSampCluster;
  const int lo = min(V, (int)cl.rank * per), hi = min(V, lo + per);
  float *z = sl.logits;
  int token;

  if (!(sl.temperature > 0.0f)) {
    // greedy: the smallest (order key, id) - the largest logit, lowest id on ties
    unsigned long long best = ~0ull;
    for (int i = lo + tid; i < hi; i += kSampThreads)
      best = min(best, ((unsigned long long)order_key(z[i]) << 32) | (unsigned)i);
    for (int o = 16; o; o >>= 1) best = min(best, __shfl_xor_sync(~0u, best, o));
    if (lane == 0) sm.wsum[warp] = best;
    __syncthreads();
    if (tid == 0)
      for (int w = 1; w < kSampWarps; ++w) best = min(best, sm.wsum[w]);
    cluster_gather(sm, cl, best);
    best = ~0ull;
    for (int r = 0; r < kSampCluster; ++r) best = min(best, sm.gath[r]);
    token = best == ~0ull ? 0 : (int)(unsigned)best;
  } else {
    // (1) + (2): z = logit / T, then the penalty on the recent tokens
    const bool penal = sl.n_recent > 0 && sl.repeat_penalty != 1.0f && lo < hi;
    if (penal) {
      for (int i = (lo >> 5) + tid; i <= ((hi - 1) >> 5); i += kSampThreads) recent_bits[i] = 0;
      __syncthreads();
      for (int j = tid; j < sl.n_recent; j += kSampThreads) {
        const int t = sl.recent[j];
        if (t >= lo && t < hi) atomicOr(&recent_bits[t >> 5], 1u << (t & 31));
      }
      __syncthreads();
    }
    float zm = -INFINITY;
    for (int i = lo + tid; i < hi; i += kSampThreads) {
      float v = z[i] / sl.temperature;
      if (penal && (recent_bits[i >> 5] >> (i & 31) & 1u))
        v = v > 0.0f ? v / sl.repeat_penalty : v * sl.repeat_penalty;
      z[i] = v;
      zm = fmaxf(zm, v);
    }
    for (int o = 16; o; o >>= 1) zm = fmaxf(zm, __shfl_xor_sync(~0u, zm, o));
    if (lane == 0) sm.wsum[warp] = __float_as_uint(zm);
    __syncthreads();
    if (tid == 0)
      for (int w = 1; w < kSampWarps; ++w) zm = fmaxf(zm, __uint_as_float((unsigned)sm.wsum[w]));
    cluster_gather(sm, cl, __float_as_uint(zm));
    zm = -INFINITY;
    for (int r = 0; r < kSampCluster; ++r) zm = fmaxf(zm, __uint_as_float((unsigned)sm.gath[r]));
    if (tid == 0) sm.zmax = zm;
    __syncthreads();

    Src src{z, nullptr, lo, hi};
    token = 0;
    do {
      // (3) top-k: the k-th element of the draw order by count
      Cut ck = all_cut();
      const int k = (sl.top_k <= 0 || sl.top_k >= V) ? V : sl.top_k;
      if (k < V) {
        const Hit h = descend<false>(sm, cl, src, all_cut(), all_cut(),
                                     Thresh{(unsigned long long)(k - 1), 0.0, false});
        if (cl.idle) break;
        ck = Cut{h.key, group_cut(sm, cl, src, all_cut(), all_cut(), h, k - h.before, h.group)};
        if (k <= kTailMax) {
          // exactly the k candidates into CTA 0, which sorts them
          int n;
          if (cl.solo) {
            n = (int)filter_list(sm, src.hi, ck, all_cut(), all_cut());
          } else {
            to_list(sm, cl, src, ck, all_cut(), all_cut());
            if (cl.idle) break;
            n = min(src.hi, kTailMax);
          }
          token = sort_tail(sm, max(n, 1), sl.top_p < 1.0f, sl.top_p,
                            draw_uniform(sl.seed, sl.io->draws));
          break;
        }
        if (src.id == nullptr && k <= kListMax) {
          to_list(sm, cl, src, ck, all_cut(), all_cut());  // exactly the k candidates
          if (cl.idle) break;
        }
      }
      // (4) top-p: up to the element at which the cumulative mass exceeds
      // p * the candidates' total
      Cut cp = all_cut();
      unsigned long long kept = 0;
      const bool top_p = sl.top_p < 1.0f;
      if (top_p) {
        const Hit h = descend<true>(sm, cl, src, ck, all_cut(),
                                    Thresh{0, (double)fmaxf(sl.top_p, 0.0f), true});
        if (cl.idle) break;
        const unsigned long long w = max(mass_of(key_value(h.key), sm.zmax), 1ull);
        const unsigned long long rank = (h.t - h.before) / w + 1, members = h.group / w;
        cp = Cut{h.key, group_cut(sm, cl, src, ck, all_cut(), h, rank, members)};
        kept = h.before + rank * w;
      }
      // (5) + (6): the draw, u times the kept mass
      const double u = draw_uniform(sl.seed, sl.io->draws);
      Thresh th{0, u, true};
      if (top_p) {
        const unsigned long long t = (unsigned long long)floor((double)kept * u);
        th = Thresh{t >= kept ? kept - 1 : t, 0.0, false};
      }
      const Hit h = descend<true>(sm, cl, src, ck, cp, th);
      if (cl.idle) break;
      const unsigned long long w = max(mass_of(key_value(h.key), sm.zmax), 1ull);
      const unsigned long long rank = (h.t - h.before) / w + 1;
      token = rank == 1 ? h.first : nth_id(sm, cl, src, ck, cp, h.key, rank);
      if (token == INT_MAX) token = h.first;
    } while (false);
  }
  // no CTA leaves while a peer may still read its shared memory, and every
  // CTA has read the draw counter before it advances
  cl_sync();
  if (cl.rank == 0 && tid == 0) {
    sl.io->token = token;
    sl.io->draws += 1u;
    if (sl.out) *sl.out = token;
  }
}

__global__ void k_set_draws(StepIO *io, uint32_t draws) { io->draws = draws; }

}  // namespace

cudaError_t launch_set_draws(StepIO *io, uint32_t draws, cudaStream_t st) {
  k_set_draws<<<1, 1, 0, st>>>(io, draws);
  return cudaGetLastError();
}

size_t sample_smem_bytes(int n_vocab) {
  return sizeof(SampSmem) + (size_t)((n_vocab + 31) / 32) * 4;
}

cudaError_t prepare_sample_kernel(int n_vocab) {
  return cudaFuncSetAttribute(k_sample, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)sample_smem_bytes(n_vocab));
}

cudaError_t launch_sample(const SampleArgs &a, int n_slots, cudaStream_t st) {
  k_sample<<<n_slots * kSampCluster, kSampThreads, sample_smem_bytes(a.n_vocab), st>>>(a);
  return cudaGetLastError();
}

}  // namespace pnb
