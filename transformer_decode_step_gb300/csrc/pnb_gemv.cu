// pnb_gemv.cu - weight-streaming kernels of the decode step.
//
// One structure serves every projection of the step.  A CTA owns a contiguous
// range of output rows.  Warp 16 (one elected thread) streams those rows,
// whole, through a ring of shared-memory slots with 1-D bulk copies.  Warps
// 0-15 wait for the previous kernel (griddepcontrol.wait), build their slice
// of the fp32 activation vector in registers (RMSNorm fused where the step has
// one), then take `16 / cw` staged rows at a time, `cw` warps per row, each
// lane covering fixed 16-byte column vectors of the row.  Per-row partial sums
// are combined in a fixed order, so results are bitwise reproducible.
#include <cuda_bf16.h>
#include <float.h>
#include <limits.h>
#include <math.h>

#include "pnb_gemv_dev.cuh"

namespace pnb {
namespace {

// ------------------------------------------------------------------ kernels

#define GEMV_ROLES(ARGS, SUMMED, PREFETCH, ROWS)                                   \
  const Ctx c = gemv_setup(ARGS.g, ROWS);                                          \
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x; \
  if (tid == 0) ktrace(ARGS.tr, 0);                                                \
  if (warp == kGemvWarps) {                                                        \
    if (lane == 0) produce(ARGS.g, ARGS.s, SUMMED, PREFETCH, c, &ARGS.io->error, ARGS.tr); \
    return;                                                                        \
  }

// dynamically claimed row chunks (every launch but the summed MoE down projection)
#define GEMV_ROLES_DYN(ARGS, PREFETCH)                                             \
  const Ctx c = gemv_setup(ARGS.g, 0);                                             \
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x; \
  if (tid == 0) ktrace(ARGS.tr, 0);                                                \
  if (warp == kGemvWarps) {                                                        \
    if (lane == 0) produce_dyn(ARGS.g, ARGS.s, PREFETCH, c, ARGS.work, &ARGS.io->error, ARGS.tr); \
    return;                                                                        \
  }

template <typename T, int NV>
__global__ void __launch_bounds__(kGemvThreads, 1) k_qkv(const QkvArgs a) {
  GEMV_ROLES_DYN(a, true)
  XSlice<T, NV> xs;
  load_weight_slice(xs, a.norm_w, a.g, warp, lane);
  const int hd = a.head_dim;
  // The position was written by the previous step's last kernel (or before
  // the step), which has completed when any layer's QKV kernel starts: the
  // RoPE angles are tabulated before the dependency wait.
  const int pos = a.io->pos;
  if (tid < hd / 2) {
    float sn, cs;
    rope_sincos(pos, a.inv_freq[tid], &sn, &cs);
    c.rope[tid] = make_float2(cs, sn);
  }
  pdl_wait();
  if (tid == 0) ktrace(a.tr, 1);
  if (a.emb) {
    int tok = a.io->token;
    if (tok < 0 || tok >= a.n_vocab) {
      if (tid == 0 && blockIdx.x == 0) set_error(&a.io->error, kErrToken);
      tok = 0;
    }
    auto embed = [&](const auto *row) {
      if (blockIdx.x == 0)
        for (int i = tid * 2; i < a.g.K; i += kGemvConsumers * 2)
          *reinterpret_cast<float2 *>(a.x_out + i) = load2(row, i);
      norm_slice(xs, row, a.g.K, a.eps, a.g, c.red, warp, lane);
    };
    if constexpr (std::is_same<T, Q8>::value) {
      const Q8Row row{static_cast<const uint8_t *>(a.emb) + (int64_t)tok * a.g.row_bytes, a.g.K};
      embed(&row);
    } else if constexpr (std::is_same<T, Q4>::value) {
      const Q4Row row{static_cast<const uint8_t *>(a.emb) + (int64_t)tok * a.g.row_bytes, a.g.K};
      embed(&row);
    } else {
      embed(static_cast<const T *>(a.emb) + (int64_t)tok * a.g.K);
    }
  } else {
    norm_slice(xs, a.x, a.g.K, a.eps, a.g, c.red, warp, lane);
  }
  if (tid == 0) ktrace(a.tr, 2);
  consume_dyn<T, NV>(a.g, c, xs, warp, lane, &a.io->error, a.tr);
  gemv_sync();
  if (tid == 0) ktrace(a.tr, 4);

  const int slot = pos % a.cap;
  const int qrows = a.n_head * hd, krows = a.n_kv * hd;
  for_claimed_rows(a.g, c, a.s.rows, true, tid, [&](int k, int r, int, int64_t row) {
    const int rr = (int)row;
    float v0 = item_row_total(a.g, c, k, r), v1 = item_row_total(a.g, c, k, r + 1);
    if (a.bias) {
      v0 += a.bias[rr];
      v1 += a.bias[rr + 1];
    }
    if (rr < qrows + krows) {
      const float2 cs = c.rope[(rr % hd) >> 1];
      const float t0 = v0 * cs.x - v1 * cs.y, t1 = v0 * cs.y + v1 * cs.x;
      v0 = t0;
      v1 = t1;
    }
    if (rr < qrows) {
      a.q[rr] = v0;
      a.q[rr + 1] = v1;
    } else {
      const bool is_k = rr < qrows + krows;
      const int kx = rr - qrows - (is_k ? 0 : krows);
      const int gk = kx / hd, d = kx - gk * hd;
      using C = typename KvOf<T>::type;
      C *dst = static_cast<C *>(is_k ? a.k_cache : a.v_cache) + ((int64_t)gk * a.cap + slot) * hd + d;
      Elem<C>::store(dst, 0, v0);
      Elem<C>::store(dst, 1, v1);
    }
  });
  if (tid == 0) ktrace(a.tr, 5);
}

template <typename T, int NV>
__global__ void __launch_bounds__(kGemvThreads, 1) k_resid(const ResidArgs a) {
  GEMV_ROLES_DYN(a, true)
  // The residual rows this thread adds to in the epilogue, loaded before the
  // dependency wait: x was last written two (down projection) or three
  // (output projection) kernels back, and those have completed when this
  // kernel's CTAs start.  Rows follow the static split of the items (the
  // rows of the CTA's k-th item are the epilogue's indices k * rps + r).
  int64_t xrow = -1;
  float xpre = 0.f;
  if (a.g.n_static_total == a.g.n_items) {
    const int rps = a.g.rows_per_stage;
    const int s0 = (int)((int64_t)a.g.n_items * blockIdx.x / gridDim.x);
    const int n_own = (int)((int64_t)a.g.n_items * (blockIdx.x + 1) / gridDim.x) - s0;
    if (tid < n_own * rps) {
      int seg, n;
      int64_t row0;
      item_rows(a.g, a.s.rows, s0 + tid / rps, seg, row0, n);
      if (tid % rps < n) {
        xrow = row0 + tid % rps;
        xpre = __ldcg(a.x + xrow);
      }
    }
  }
  pdl_wait();
  if (tid == 0) ktrace(a.tr, 1);
  XSlice<T, NV> xs;
  load_slice(xs, a.vec, 1.0f, nullptr, a.g, warp, lane);
  if (tid == 0) ktrace(a.tr, 2);
  consume_dyn<T, NV>(a.g, c, xs, warp, lane, &a.io->error, a.tr);
  gemv_sync();
  if (tid == 0) ktrace(a.tr, 4);
  for_claimed_rows(a.g, c, a.s.rows, false, tid, [&](int k, int r, int, int64_t row) {
    a.x[row] = (row == xrow ? xpre : a.x[row]) + item_row_total(a.g, c, k, r);
  });
  if (tid == 0) ktrace(a.tr, 5);
}

template <typename T, int NV>
__global__ void __launch_bounds__(kGemvThreads, 1) k_gateup(const GateUpArgs a) {
  GEMV_ROLES_DYN(a, a.s.table == nullptr)
  XSlice<T, NV> xs;
  load_weight_slice(xs, a.norm_w, a.g, warp, lane);
  pdl_wait();
  if (tid == 0) ktrace(a.tr, 1);
  norm_slice(xs, a.x, a.g.K, a.eps, a.g, c.red, warp, lane);
  if (tid == 0) ktrace(a.tr, 2);
  consume_dyn<T, NV>(a.g, c, xs, warp, lane, &a.io->error, a.tr);
  gemv_sync();
  if (tid == 0) ktrace(a.tr, 4);
  for_claimed_rows(a.g, c, a.s.rows, true, tid, [&](int k, int r, int seg, int64_t row) {
    const float gte = item_row_total(a.g, c, k, r), up = item_row_total(a.g, c, k, r + 1);
    a.h[(int64_t)seg * a.n_ff + (row >> 1)] = silu(gte) * up;
  });
  if (tid == 0) ktrace(a.tr, 5);
}

template <typename T, int NV>
__global__ void __launch_bounds__(kGemvThreads, 1) k_down_moe(const DownMoeArgs a) {
  GEMV_ROLES(a, true, false, a.s.rows)
  pdl_wait();
  if (tid == 0) ktrace(a.tr, 1);
  XSlice<T, NV> xs;
  load_slice(xs, a.h, 1.0f, nullptr, a.g, warp, lane);
  if (tid == 0) ktrace(a.tr, 2);
  consume<T, NV>(a.g, a.s, true, c, xs, warp, lane, &a.io->error, a.tr, [&](int seg) {
    load_slice(xs, a.h + (int64_t)seg * a.n_ff, 1.0f, nullptr, a.g, warp, lane);
  });
  gemv_sync();
  if (tid == 0) ktrace(a.tr, 4);
  for (int64_t r = c.r0 + tid; r < c.r1; r += kGemvConsumers) {
    float acc = 0.f;
    for (int s = 0; s < a.s.n; ++s)
      acc = fmaf(a.gate[s], row_total(c.part + s * a.g.rows_cta_max * a.g.cw, (int)(r - c.r0), a.g.cw),
                 acc);
    a.x[r] += acc;
  }
  if (tid == 0) ktrace(a.tr, 5);
}

template <typename T, int NV>
__global__ void __launch_bounds__(kGemvThreads, 1) k_lmhead(const LmArgs a) {
  GEMV_ROLES_DYN(a, true)
  XSlice<T, NV> xs;
  load_weight_slice(xs, a.norm_w, a.g, warp, lane);
  pdl_wait();
  if (tid == 0) ktrace(a.tr, 1);
  norm_slice(xs, a.x, a.g.K, a.eps, a.g, c.red, warp, lane);
  if (tid == 0) ktrace(a.tr, 2);
  consume_dyn<T, NV>(a.g, c, xs, warp, lane, &a.io->error, a.tr);
  gemv_sync();
  if (tid == 0) ktrace(a.tr, 4);
  float best = -FLT_MAX;
  int bi = INT_MAX;
  for_claimed_rows(a.g, c, a.s.rows, false, tid, [&](int k, int r, int, int64_t row) {
    const float v = item_row_total(a.g, c, k, r);
    if (a.logits) a.logits[row] = v;
    argmax_merge(best, bi, v, (int)row);
  });
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
    argmax_merge(best, bi, __shfl_xor_sync(0xffffffffu, best, o), __shfl_xor_sync(0xffffffffu, bi, o));
  int *redi = reinterpret_cast<int *>(c.red + 32);
  if (lane == 0) {
    c.red[warp] = best;
    redi[warp] = bi;
  }
  gemv_sync();
  int *last = redi + 16;
  if (tid == 0) {
    for (int w = 1; w < kGemvWarps; ++w) argmax_merge(best, bi, c.red[w], redi[w]);
    a.part_val[blockIdx.x] = best;
    a.part_idx[blockIdx.x] = bi;
    __threadfence();
    const unsigned prev = atomicAdd(a.counter, 1u);
    *last = prev == gridDim.x - 1;
  }
  gemv_sync();
  if (*last && warp == 0) {
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
        v[j] = __ldcg(a.part_val + b);
        ix[j] = __ldcg(a.part_idx + b);
      }
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (base + 32 * j < G) argmax_merge(fv, fi, v[j], ix[j]);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
      argmax_merge(fv, fi, __shfl_xor_sync(0xffffffffu, fv, off), __shfl_xor_sync(0xffffffffu, fi, off));
    if (lane == 0) {
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
  if (tid == 0) ktrace(a.tr, 5);
}

// Router: one CTA of 256 threads.  r = Wr RMSNorm(x); the k largest (lower
// index on ties); gate = softmax over the chosen logits.
template <typename T>
__global__ void __launch_bounds__(256, 1) k_router(const RouterArgs a) {
  float *xs = reinterpret_cast<float *>(g_smem);
  float *red = xs + a.E;
  float *r = red + 32;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  pdl_wait();
  pdl_trigger();
  for (int i = tid; i < a.E; i += 256) xs[i] = a.x[i];
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
    float acc = 0.f;
    if constexpr (std::is_same<T, Q8>::value || std::is_same<T, Q4>::value) {
      // a quantized router row (values, then the blocks' fp16 scales), in pairs
      using Row = typename std::conditional<std::is_same<T, Q8>::value, Q8Row, Q4Row>::type;
      const int64_t rb = std::is_same<T, Q8>::value ? a.E + a.E / 16 : a.E / 2 + a.E / 16;
      const Row row{static_cast<const uint8_t *>(a.w) + (int64_t)e * rb, a.E};
      for (int i = 2 * lane; i < a.E; i += 64) {
        const float2 w = load2(&row, i);
        acc = fmaf(w.x, xs[i], acc);
        acc = fmaf(w.y, xs[i + 1], acc);
      }
    } else {
      const T *row = static_cast<const T *>(a.w) + (int64_t)e * a.E;
      for (int i = lane; i < a.E; i += 32) acc = fmaf(Elem<T>::load(row, i), xs[i], acc);
    }
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
    for (int i = 0; i < a.k; ++i) {
      a.idx[i] = idx[i];
      a.gate[i] = expf(r[idx[i]] - mx) / z;
    }
  }
}

// Prefill chunks: n virtual slots at the state's next n positions; then the
// state takes the last slot's token and position and every slot's error bits.
__global__ void k_prefill_begin(StepIO *pio, const StepIO *state, int n) {
  const int b = threadIdx.x;
  if (b < n) pio[b] = StepIO{0, state->pos + b, 0, 0};
}
__global__ void k_prefill_end(StepIO *state, const StepIO *pio, int n) {
  if (threadIdx.x != 0) return;
  int32_t e = 0;
  for (int b = 0; b < n; ++b) e |= pio[b].error;
  state->token = pio[n - 1].token;
  state->pos = pio[n - 1].pos;
  if (e) set_error(&state->error, e);
}

// A bounded wait that runs out, the way any of the kernels' waits would: one
// thread copies `bytes` of src into shared memory with a bulk copy, then waits
// with a limit of limit_ns on an mbarrier that nothing arrives on.  When the
// wait gives up it sets the timeout bit in the state's error word, waits (with
// the normal limit) for its copy to land, and returns: the kernel ends with no
// copy in flight and the context stays usable.
__global__ void k_wait_probe(const uint8_t *src, uint32_t bytes, unsigned long long limit_ns,
                             StepIO *io) {
  __shared__ __align__(128) uint8_t buf[kWaitProbeBytes];
  __shared__ uint64_t full, never;
  if (threadIdx.x != 0) return;
  mbar_init(&full, 1);
  mbar_init(&never, 1);
  fence_barrier_init();
  mbar_arrive_expect_tx(&full, bytes);
  bulk_g2s(buf, src, bytes, &full);
  if (!mbar_wait_for(&never, 0u, limit_ns)) set_error(&io->error, kErrTimeout);
  if (!mbar_wait(&full, 0u)) set_error(&io->error, kErrTimeout);
}

__global__ void k_set_token(StepIO *io, int32_t token) { io->token = token; }
__global__ void k_copy_token(StepIO *io, const int32_t *token) { io->token = *token; }
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

// dispatch on the lane's vector count
#define GEMV_LAUNCH(KERNEL, T, ARGS, GRID, ST, PDL)                                                  \
  switch (ARGS.g.nv) {                                                                               \
    case 1: return launch(KERNEL<T, 1>, ARGS, dim3(GRID), dim3(kGemvThreads), smem_layout(ARGS.g).total, ST, PDL); \
    case 2: return launch(KERNEL<T, 2>, ARGS, dim3(GRID), dim3(kGemvThreads), smem_layout(ARGS.g).total, ST, PDL); \
    case 4: return launch(KERNEL<T, 4>, ARGS, dim3(GRID), dim3(kGemvThreads), smem_layout(ARGS.g).total, ST, PDL); \
    default: return cudaErrorInvalidValue;                                                          \
  }

template <typename T, int NV>
cudaError_t prepare_nv(int bytes) {
  cudaError_t e;
  if ((e = ensure_smem(k_qkv<T, NV>, bytes)) != cudaSuccess) return e;
  if ((e = ensure_smem(k_resid<T, NV>, bytes)) != cudaSuccess) return e;
  if ((e = ensure_smem(k_gateup<T, NV>, bytes)) != cudaSuccess) return e;
  if ((e = ensure_smem(k_down_moe<T, NV>, bytes)) != cudaSuccess) return e;
  return ensure_smem(k_lmhead<T, NV>, bytes);
}

template <typename T>
cudaError_t prepare_t(int bytes) {
  cudaError_t e;
  if ((e = prepare_nv<T, 1>(bytes)) != cudaSuccess) return e;
  if ((e = prepare_nv<T, 2>(bytes)) != cudaSuccess) return e;
  if ((e = prepare_nv<T, 4>(bytes)) != cudaSuccess) return e;
  return ensure_smem(k_router<T>, bytes);
}

}  // namespace

// weight storage type: 0 fp32, 1 bf16, 2 Q8, 3 Q4
#define GEMV_DTYPES(KERNEL, ARGS, GRID, ST, PDL)                       \
  if (dtype == 3) { GEMV_LAUNCH(KERNEL, Q4, ARGS, GRID, ST, PDL) }      \
  if (dtype == 2) { GEMV_LAUNCH(KERNEL, Q8, ARGS, GRID, ST, PDL) }      \
  if (dtype == 1) { GEMV_LAUNCH(KERNEL, __nv_bfloat16, ARGS, GRID, ST, PDL) } \
  GEMV_LAUNCH(KERNEL, float, ARGS, GRID, ST, PDL)

cudaError_t launch_qkv(int dtype, const QkvArgs &a, int grid, cudaStream_t st, bool pdl) {
  GEMV_DTYPES(k_qkv, a, grid, st, pdl)
}
cudaError_t launch_resid(int dtype, const ResidArgs &a, int grid, cudaStream_t st, bool pdl) {
  GEMV_DTYPES(k_resid, a, grid, st, pdl)
}
cudaError_t launch_gateup(int dtype, const GateUpArgs &a, int grid, cudaStream_t st, bool pdl) {
  GEMV_DTYPES(k_gateup, a, grid, st, pdl)
}
cudaError_t launch_down_moe(int dtype, const DownMoeArgs &a, int grid, cudaStream_t st, bool pdl) {
  GEMV_DTYPES(k_down_moe, a, grid, st, pdl)
}
cudaError_t launch_lmhead(int dtype, const LmArgs &a, int grid, cudaStream_t st, bool pdl) {
  GEMV_DTYPES(k_lmhead, a, grid, st, pdl)
}
cudaError_t launch_router(int dtype, const RouterArgs &a, cudaStream_t st, bool pdl) {
  const int smem = (a.E + 32 + a.n_expert) * 4;
  if (dtype == 3) return launch(k_router<Q4>, a, dim3(1), dim3(256), smem, st, pdl);
  if (dtype == 2) return launch(k_router<Q8>, a, dim3(1), dim3(256), smem, st, pdl);
  if (dtype == 1) return launch(k_router<__nv_bfloat16>, a, dim3(1), dim3(256), smem, st, pdl);
  return launch(k_router<float>, a, dim3(1), dim3(256), smem, st, pdl);
}
cudaError_t prepare_gemv_kernels(int dtype, int smem_bytes) {
  if (dtype == 3) return prepare_t<Q4>(smem_bytes);
  if (dtype == 2) return prepare_t<Q8>(smem_bytes);
  return dtype ? prepare_t<__nv_bfloat16>(smem_bytes) : prepare_t<float>(smem_bytes);
}
cudaError_t launch_set_token(StepIO *io, int32_t token, cudaStream_t st) {
  k_set_token<<<1, 1, 0, st>>>(io, token);
  return cudaGetLastError();
}
cudaError_t launch_copy_token(StepIO *io, const int32_t *token, cudaStream_t st) {
  k_copy_token<<<1, 1, 0, st>>>(io, token);
  return cudaGetLastError();
}
cudaError_t launch_prefill_begin(StepIO *pio, const StepIO *state, int n, cudaStream_t st) {
  k_prefill_begin<<<1, 128, 0, st>>>(pio, state, n);
  return cudaGetLastError();
}
cudaError_t launch_prefill_end(StepIO *state, const StepIO *pio, int n, cudaStream_t st) {
  k_prefill_end<<<1, 32, 0, st>>>(state, pio, n);
  return cudaGetLastError();
}
cudaError_t launch_wait_probe(const void *src, uint32_t bytes, unsigned long long limit_ns, StepIO *io,
                              cudaStream_t st) {
  k_wait_probe<<<1, 32, 0, st>>>(static_cast<const uint8_t *>(src), bytes, limit_ns, io);
  return cudaGetLastError();
}
cudaError_t launch_set_pos(StepIO *io, int32_t pos, cudaStream_t st) {
  k_set_pos<<<1, 1, 0, st>>>(io, pos);
  return cudaGetLastError();
}

}  // namespace pnb
