// pnb_sample.cu - the decode loop's token sampler ("Engine Architecture",
// section "Sampling"), one 1024-thread CTA per sequence:
//   (1) z = logit / temperature (temperature <= 0: greedy argmax);
//   (2) repetition penalty on each distinct token of the recent window
//       (z / penalty when z > 0, z * penalty otherwise);
//   (3) top-k, (4) top-p ("until the cumulative probability exceeds p"),
//   (5) softmax, (6) multinomial draw with u from the state's draw counter.
// The draw order is z descending, token id ascending on ties.  Nothing is
// sorted: each of top-k, top-p and the draw is a radix descent over the
// 32-bit order key of z (four 8-bit levels, a 256-bin shared-memory histogram
// each) that finds the element at which a running total - a count for top-k,
// softmax mass for top-p and the draw - first exceeds a threshold.  Masses
// are exp(z - z_max) in 64-bit fixed point (units of 2^-40), so every sum is
// an exact integer and the result does not depend on the order of atomics.
// z is written back over the logits (the pages' sampler also changes them in
// place); once top-k leaves at most kListMax candidates, they move to shared
// memory in id order and the remaining descents run there.
#include "pnb_kernels.cuh"

#include <climits>

namespace pnb {
namespace {

constexpr int kSampThreads = 1024;
constexpr int kSampWarps = kSampThreads / 32;
constexpr int kListMax = 4096;
constexpr float kMassUnit = 1099511627776.0f;  // 2^40

struct SampSmem {
  unsigned hist_lo[256], hist_hi[256];  // a 64-bit total per bin as two words
  int first[256];
  unsigned long long wcnt[kSampWarps];
  float wz[kSampWarps];
  int wid[kSampWarps];
  unsigned long long before;
  int bin;
  int found;
  float zmax;
  float lz[kListMax];
  int lid[kListMax];
  // followed by the recent-token bitmap, (n_vocab + 31) / 32 words
};

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

// the elements the descents walk: every token (z in global memory, index =
// id) or the shared-memory candidate list (in id order)
struct Src {
  const float *z;
  const int *id;  // nullptr: index is the id
  int n;
  __device__ __forceinline__ float zv(int i) const { return z[i]; }
  __device__ __forceinline__ int idv(int i) const { return id ? id[i] : i; }
};

// result of a descent: the key of the element where the running total first
// exceeds the threshold, the total before that key's group, the group's total
// and its lowest id
struct Hit {
  uint32_t key;
  unsigned long long before, group;
  int first;
};

// 64-bit add into a bin held as two 32-bit words: 32-bit shared-memory
// atomics are native, and the add that wraps the low word carries into the
// high one (atomicAdd returns the word before the add, so each wrap is seen
// exactly once and the pair ends exact whatever the order)
__device__ __forceinline__ void bin_add(SampSmem &sm, int bin, unsigned long long v) {
  const unsigned lo = (unsigned)v, hi = (unsigned)(v >> 32);
  const unsigned old = atomicAdd(&sm.hist_lo[bin], lo);
  const unsigned carry = old + lo < old ? 1u : 0u;
  if (hi + carry) atomicAdd(&sm.hist_hi[bin], hi + carry);
}

__device__ __forceinline__ unsigned long long bin_total(const SampSmem &sm, int bin) {
  return ((unsigned long long)sm.hist_hi[bin] << 32) | sm.hist_lo[bin];
}

// warp 0: the first of 256 bins at which before + running sum exceeds t
__device__ __forceinline__ void pick_bin(SampSmem &sm, unsigned long long before,
                                         unsigned long long t) {
  const int lane = threadIdx.x;
  unsigned long long v[8], own = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    v[j] = bin_total(sm, 8 * lane + j);
    own += v[j];
  }
  unsigned long long incl = own;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long y = __shfl_up_sync(~0u, incl, o);
    if (lane >= o) incl += y;
  }
  unsigned long long run = before + incl - own;
  const bool mine = run <= t && t < run + own;
  if (mine) {
    int j = 0;
    while (j < 7 && run + v[j] <= t) run += v[j++];
    sm.bin = 8 * lane + j;
    sm.before = run;
  }
  // unreachable when the caller's threshold is below the total; keep the
  // last non-empty bin so the descent still ends on an element
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
}

// block-wide radix descent over src's elements inside c1 and c2, in the draw
// order, weighting each by 1 (kMass false) or by its fixed-point mass
template <bool kMass>
__device__ Hit descend(SampSmem &sm, const Src &src, const Cut &c1, const Cut &c2,
                       unsigned long long t) {
  uint32_t prefix = 0, mask = 0;
  unsigned long long before = 0;
  const float zmax = sm.zmax;
  Hit h;
  for (int level = 0; level < 4; ++level) {
    const int shift = 24 - 8 * level;
    if (threadIdx.x < 256) {
      sm.hist_lo[threadIdx.x] = 0;
      sm.hist_hi[threadIdx.x] = 0;
      sm.first[threadIdx.x] = INT_MAX;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < src.n; i += kSampThreads) {
      const float z = src.zv(i);
      const uint32_t k = order_key(z);
      if ((k & mask) != prefix) continue;
      const int id = src.idv(i);
      if (!in_cut(c1, k, id) || !in_cut(c2, k, id)) continue;
      const int bin = (k >> shift) & 255;
      if (kMass)
        bin_add(sm, bin, mass_of(z, zmax));
      else
        atomicAdd(&sm.hist_lo[bin], 1u);
      if (level == 3) atomicMin(&sm.first[bin], id);
    }
    __syncthreads();
    if (threadIdx.x < 32) pick_bin(sm, before, t);
    __syncthreads();
    const int b = sm.bin;
    before = sm.before;
    prefix |= (uint32_t)b << shift;
    mask |= 0xFFu << shift;
    if (level == 3) {
      h.group = bin_total(sm, b);
      h.first = sm.first[b];
    }
    __syncthreads();  // hist is cleared next level
  }
  h.key = prefix;
  h.before = before;
  return h;
}

// id of the m-th element (1-based, id order) of src inside c1 and c2 whose key
// is `key`: each warp counts a contiguous range, then the warp holding the
// m-th walks its range again
__device__ int nth_id(SampSmem &sm, const Src &src, const Cut &c1, const Cut &c2, uint32_t key,
                      unsigned long long m) {
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int per = (src.n + kSampWarps - 1) / kSampWarps;
  const int lo = min(src.n, w * per), hi = min(src.n, lo + per);
  auto hit = [&](int i) {
    if (i >= hi) return false;
    const uint32_t k = order_key(src.zv(i));
    const int id = src.idv(i);
    return k == key && in_cut(c1, k, id) && in_cut(c2, k, id);
  };
  unsigned long long cnt = 0;
  for (int base = lo; base < hi; base += 32) cnt += __popc(__ballot_sync(~0u, hit(base + lane)));
  if (lane == 0) sm.wcnt[w] = cnt;
  if (threadIdx.x == 0) sm.found = INT_MAX;
  __syncthreads();
  unsigned long long off = 0;
  for (int j = 0; j < w; ++j) off += sm.wcnt[j];
  if (off < m && m <= off + cnt) {
    unsigned long long run = off;
    for (int base = lo; base < hi; base += 32) {
      const unsigned bal = __ballot_sync(~0u, hit(base + lane));
      const int c = __popc(bal);
      if (run + c >= m) {
        unsigned b = bal;
        for (unsigned long long r = run + 1; r < m; ++r) b &= b - 1;
        if (lane == __ffs(b) - 1) sm.found = src.idv(base + lane);
        break;
      }
      run += c;
    }
  }
  __syncthreads();
  return sm.found;
}

// the `rank`-th element of a descent's group (1-based): its lowest id when
// rank is 1, every id (cut at INT_MAX) when it is the whole group
__device__ __forceinline__ int group_cut(SampSmem &sm, const Src &src, const Cut &c1,
                                         const Cut &c2, const Hit &h, unsigned long long rank,
                                         unsigned long long members) {
  if (rank >= members) return INT_MAX;
  if (rank == 1) return h.first;
  return nth_id(sm, src, c1, c2, h.key, rank);
}

__global__ void __launch_bounds__(kSampThreads, 1) k_sample(const __grid_constant__ SampleArgs a) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  SampSmem &sm = *reinterpret_cast<SampSmem *>(smem_raw);
  uint32_t *recent_bits = reinterpret_cast<uint32_t *>(smem_raw + sizeof(SampSmem));
  const SampleSlot &sl = a.slot[blockIdx.x];
  const int V = a.n_vocab;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  float *z = sl.logits;
  int token;

  if (!(sl.temperature > 0.0f)) {
    // greedy: argmax of the logits, lowest id on ties
    float best = -INFINITY;
    int bid = INT_MAX;
    for (int i = tid; i < V; i += kSampThreads) {
      const float v = z[i];
      if (v > best || (v == best && i < bid)) {
        best = v;
        bid = i;
      }
    }
    for (int o = 16; o; o >>= 1) {
      const float ov = __shfl_xor_sync(~0u, best, o);
      const int oi = __shfl_xor_sync(~0u, bid, o);
      if (ov > best || (ov == best && oi < bid)) {
        best = ov;
        bid = oi;
      }
    }
    if (lane == 0) {
      sm.wz[warp] = best;
      sm.wid[warp] = bid;
    }
    __syncthreads();
    if (tid == 0) {
      for (int w = 1; w < kSampWarps; ++w)
        if (sm.wz[w] > best || (sm.wz[w] == best && sm.wid[w] < bid)) {
          best = sm.wz[w];
          bid = sm.wid[w];
        }
      sm.found = bid == INT_MAX ? 0 : bid;
    }
    __syncthreads();
    token = sm.found;
  } else {
    // (1) + (2): z = logit / T, then the penalty on the recent tokens
    const int words = (V + 31) >> 5;
    const bool penal = sl.n_recent > 0 && sl.repeat_penalty != 1.0f;
    if (penal) {
      for (int i = tid; i < words; i += kSampThreads) recent_bits[i] = 0;
      __syncthreads();
      for (int j = tid; j < sl.n_recent; j += kSampThreads) {
        const int t = sl.recent[j];
        if (t >= 0 && t < V) atomicOr(&recent_bits[t >> 5], 1u << (t & 31));
      }
      __syncthreads();
    }
    float zm = -INFINITY;
    for (int i = tid; i < V; i += kSampThreads) {
      float v = z[i] / sl.temperature;
      if (penal && (recent_bits[i >> 5] >> (i & 31) & 1u))
        v = v > 0.0f ? v / sl.repeat_penalty : v * sl.repeat_penalty;
      z[i] = v;
      zm = fmaxf(zm, v);
    }
    for (int o = 16; o; o >>= 1) zm = fmaxf(zm, __shfl_xor_sync(~0u, zm, o));
    if (lane == 0) sm.wz[warp] = zm;
    __syncthreads();
    if (tid == 0) {
      for (int w = 1; w < kSampWarps; ++w) zm = fmaxf(zm, sm.wz[w]);
      sm.zmax = zm;
    }
    __syncthreads();

    // (3) top-k: the k-th element of the draw order by count
    Src src{z, nullptr, V};
    Cut ck = all_cut();
    const int k = (sl.top_k <= 0 || sl.top_k >= V) ? V : sl.top_k;
    if (k < V) {
      const Hit h = descend<false>(sm, src, all_cut(), all_cut(), (unsigned long long)(k - 1));
      ck = Cut{h.key, group_cut(sm, src, all_cut(), all_cut(), h, k - h.before, h.group)};
    }
    // the candidates move to shared memory, in id order, when they fit (the
    // count is checked again before any slot is written)
    if (k <= kListMax) {
      const int per = (V + kSampWarps - 1) / kSampWarps;
      const int lo = min(V, warp * per), hi = min(V, lo + per);
      unsigned cnt = 0;
      for (int base = lo; base < hi; base += 32) {
        const int i = base + lane;
        cnt += __popc(__ballot_sync(~0u, i < hi && in_cut(ck, order_key(z[i]), i)));
      }
      if (lane == 0) sm.wcnt[warp] = cnt;
      __syncthreads();
      unsigned off = 0, total = 0;
      for (int j = 0; j < kSampWarps; ++j) {
        if (j == warp) off = total;
        total += (unsigned)sm.wcnt[j];
      }
      for (int base = lo; base < hi && total <= (unsigned)kListMax; base += 32) {
        const int i = base + lane;
        const float v = i < hi ? z[i] : 0.0f;
        const bool in = i < hi && in_cut(ck, order_key(v), i);
        const unsigned bal = __ballot_sync(~0u, in);
        if (in) {
          const unsigned slot = off + __popc(bal & ((1u << lane) - 1u));
          sm.lz[slot] = v;
          sm.lid[slot] = i;
        }
        off += __popc(bal);
      }
      __syncthreads();
      if (total <= (unsigned)kListMax) {
        src = Src{sm.lz, sm.lid, (int)total};
        ck = all_cut();
      }
    }
    // (4) top-p: up to the element whose cumulative mass exceeds p * total
    Cut cp = all_cut();
    unsigned long long kept;
    // the candidates' total mass
    {
      unsigned long long part = 0;
      const float zmax = sm.zmax;
      for (int i = tid; i < src.n; i += kSampThreads) {
        const float v = src.zv(i);
        if (in_cut(ck, order_key(v), src.idv(i))) part += mass_of(v, zmax);
      }
      for (int o = 16; o; o >>= 1) part += __shfl_xor_sync(~0u, part, o);
      __syncthreads();
      if (lane == 0) sm.wcnt[warp] = part;
      __syncthreads();
      kept = 0;
      for (int w = 0; w < kSampWarps; ++w) kept += sm.wcnt[w];
      __syncthreads();
    }
    if (sl.top_p < 1.0f) {
      const double tp = floor((double)kept * (double)fmaxf(sl.top_p, 0.0f));
      const unsigned long long t = (unsigned long long)tp;
      const Hit h = descend<true>(sm, src, ck, all_cut(), t);
      const unsigned long long w = max(mass_of(key_value(h.key), sm.zmax), 1ull);
      const unsigned long long rank = (t - h.before) / w + 1, members = h.group / w;
      cp = Cut{h.key, group_cut(sm, src, ck, all_cut(), h, rank, members)};
      kept = h.before + rank * w;
    }
    // (5) + (6): the draw, in the kept mass
    const double u = draw_uniform(sl.seed, sl.io->draws);
    unsigned long long t = (unsigned long long)floor((double)kept * u);
    if (t >= kept) t = kept - 1;
    const Hit h = descend<true>(sm, src, ck, cp, t);
    const unsigned long long w = max(mass_of(key_value(h.key), sm.zmax), 1ull);
    const unsigned long long rank = (t - h.before) / w + 1;
    token = rank == 1 ? h.first : nth_id(sm, src, ck, cp, h.key, rank);
    if (token == INT_MAX) token = h.first;
  }
  __syncthreads();
  if (tid == 0) {
    sl.io->token = token;
    sl.io->draws += 1u;
    if (sl.out) *sl.out = token;
  }
}

}  // namespace

namespace {
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
  k_sample<<<n_slots, kSampThreads, sample_smem_bytes(a.n_vocab), st>>>(a);
  return cudaGetLastError();
}

}  // namespace pnb
