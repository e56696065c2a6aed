// pnb_api.cu - the C ABI (include/pnb.h): validation, geometry planning,
// workspace, the per-step launch sequence and its CUDA-graph capture.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <new>
#include <vector>

#include "pnb.h"
#include "pnb_kernels.cuh"

using namespace pnb;

namespace {

// bytes of whole rows per GEMV ring slot; rows longer than 16 KB (the down
// projections) go two to a slot where two fit in 64 KB: with one row per slot
// the per-slot consumer work (a barrier wait, the cross-lane reductions) was
// spread over too few bytes, and Llama-7B's down projection took 19.1 us per
// layer against 17.4 us with two
constexpr int kStageTarget = 36 * 1024;
constexpr int kLongRowBytes = 16 * 1024;
constexpr int kLongRowStage = 64 * 1024;
constexpr int kRingBudget = 192 * 1024;   // bytes of GEMV ring per CTA
constexpr int kMaxSmem = 227 * 1024;
// prefill chunks whose positions stay below this run their attention as one
// chunk kernel (CUDA cores, each tile of the prefix read once per 16 query
// rows); past it the per-token tensor-core attention is faster
constexpr int kChunkAttnMaxPos = 256;
constexpr int kMaxBatch = 64;
// prefill chunk: up to 128 virtual slots (the pages' default chunk length)
constexpr int kMaxChunk = 128;
#ifndef PNB_INFLIGHT_KB
#define PNB_INFLIGHT_KB 192
#endif
constexpr int kInflightBytes = PNB_INFLIGHT_KB * 1024;  // weight copies in flight per CTA
#ifndef PNB_STATIC_PCT
#define PNB_STATIC_PCT 100
#endif
constexpr int kStaticPct = PNB_STATIC_PCT;  // share of a launch's items split statically

int ceil_div(int64_t a, int64_t b) { return (int)((a + b - 1) / b); }

// rows_total: rows over all segments; nseg: segments concatenated in it (0 when
// the launch sums its segments into the same rows: static row ranges).
// wt: weight storage type (PNB_F32, PNB_BF16, PNB_Q8_0 or PNB_Q4_0)
Geom plan_gemv(int K, int wt, int64_t rows_total, int row_align, int nsum, int grid, int nseg) {
  Geom g{};
  g.K = K;
  const bool q = wt == PNB_Q8_0 || wt == PNB_Q4_0;
  g.es = q ? 1 : (wt == PNB_BF16 ? 2 : 4);
  // Q8: the values, then fp16 scales; Q4: the codes, two per byte, then the scales
  g.row_bytes = wt == PNB_Q8_0 ? K + K / 16 : (wt == PNB_Q4_0 ? K / 2 + K / 16 : K * g.es);
  g.vpr = q ? K / 8 : g.row_bytes / 16;   // Q8: 8-byte, Q4: 4-byte vectors of 8 values
  int rps = 1;
  const int target = g.row_bytes > kLongRowBytes ? kLongRowStage : kStageTarget;
  while (rps * 2 <= 64 && rps * 2 * g.row_bytes <= target) rps *= 2;
  rps = std::max(rps, row_align);   // row pairs never straddle two ring items
  g.rows_per_stage = rps;
  g.stage_bytes = rps * g.row_bytes;
  // warps per row: as many as the row has 32-lane column groups (up to all
  // sixteen), so that each activation element is loaded by one lane of the
  // CTA only: the load after griddepcontrol.wait shares the SM's ingress with
  // the weight ring, and its latency grows with its volume
  const int vpr = g.vpr;
  int cw = 1;
  while (cw < kGemvWarps && (cw * 2 * 32 <= vpr || kGemvWarps / cw > rps)) cw *= 2;
  g.cw = cw;
  const int nv = ceil_div(vpr, 32 * cw);
  g.nv = nv <= 1 ? 1 : (nv <= 2 ? 2 : (nv <= 4 ? 4 : 8));  // 8 = unsupported
  g.row_align = row_align;
  const int64_t units = rows_total / row_align;
  g.rows_cta_max = ceil_div(units, grid) * row_align;
  g.nsum = nsum;
  if (nseg > 0) {
    const int64_t per_seg = rows_total / nseg;
    g.n_items = nseg * ceil_div(per_seg, rps);
    g.n_static_total = kStaticPct >= 100 ? g.n_items
                        : (int)((int64_t)g.n_items * kStaticPct / (100 * (int64_t)grid)) * grid;
    const int64_t pool = g.n_items - g.n_static_total;
    g.cap_items = ceil_div(g.n_static_total, grid) + (pool > 0 ? ceil_div(2 * pool, grid) + 4 : 0);
  }
  g.nstages = 2;
  const int fixed = smem_layout(g).total - 2 * g.stage_bytes - 2 * 16;  // everything but the ring
  const int ring = std::min(kRingBudget, kMaxSmem - fixed - 1024);
  g.nstages = std::min(12, std::max(2, ring / g.stage_bytes));
  g.inflight = std::max(1, std::min(g.nstages, ceil_div(kInflightBytes, g.stage_bytes)));
  return g;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t align256(size_t v) { return (v + 255) / 256 * 256; }

}  // namespace

struct pnb_model {
  pnb_config cfg;
  int device = 0, num_sms = 0, grid = 0;
  int hd = 0, n_sets = 0, qkv_rows = 0, cap = 0;
  int kv_es = 0;                         // KV-cache element bytes (bf16 for bf16, Q8 and Q4 weights)
  int kv_dt = 0;                         // KV-cache element type (PNB_F32 or PNB_BF16)
  const void *tok_embd = nullptr;
  const float *out_norm = nullptr;
  const void *output = nullptr;
  std::vector<const float *> attn_norm, ffn_norm;
  std::vector<const void *> wqkv, wo, w_router, w_gate_up, w_down;
  std::vector<const float *> bqkv;       // per layer q / k / v bias, empty when the model has none
  double *inv_freq = nullptr;            // device [hd/2]
  const void **tab_gate_up = nullptr;    // device [n_layer][expert_count]
  const void **tab_down = nullptr;
  Geom g_qkv{}, g_o{}, g_gateup{}, g_down{}, g_lm{};
  AttnGeom ag{};
  int n_split = 1, zgroups = 1;
  bool graphs = true;
  // tensor-core attention (bf16 KV, head_dim 64 / 128, <= 8 query heads per KV head)
  bool attn_tc_ok = false, attn_tc = false;
  int n_split_tc = 1;
  bool sample_ok = false;                // the sampler kernel fits this vocabulary
  int mode_gen = 0;                      // bumped when a launch mode changes (graphs re-captured)
  bool det_batch = false;                // batched residual K parts in fixed point
  cudaStream_t cap_stream = nullptr;     // stream used for graph capture
  struct BatchCtx *batch = nullptr;      // batched-slot step (made on first use)
};

// One tensor-core GEMM of the batched step: its split and grid.
struct BPlan {
  int rows = 0, K = 0, tiles = 0, ksplit = 1, units = 0, grid = 0;
};

// Device workspace, tensor maps, plans and the captured graph of the
// batched-slot step of one model.
struct BatchCtx {
  uint8_t *ws = nullptr;
  float *xb = nullptr, *qb = nullptr, *apart = nullptr, *gpart = nullptr, *am_val = nullptr;
  unsigned *acnt = nullptr, *tile_cnt = nullptr, *am_cnt = nullptr;
  int32_t *am_idx = nullptr, *pos = nullptr, *err = nullptr;
  StepIO *pio = nullptr;                 // prefill: the I/O words of a chunk's virtual slots
  float *gates = nullptr;                // MoE: [slot][expert] router weights (0 = not chosen)
  long long *acc = nullptr;              // [slot][n_embd] residual K-part sums, fixed point 2^-32
  unsigned *tp_cnt = nullptr;            // persistent attention: [claim, done], zero between launches
  __nv_bfloat16 *xop_e = nullptr, *xop_o = nullptr, *xop_f = nullptr;
  float2 *rope = nullptr;
  BSlot *slots = nullptr;
  std::vector<CUtensorMap> w_qkv, w_o, w_gu, w_dn;
  CUtensorMap w_lm;
  CUtensorMap x_e[4], x_o[4], x_f[4];   // per padded slot count 16, 32, 64, 128
  BPlan p_qkv, p_o, p_gu, p_dn, p_lm;
  int nstages[4] = {0, 0, 0, 0}, smem[4] = {0, 0, 0, 0};
  float *lgs = nullptr;                  // 128-slot LM head: logits when the caller wants none
  // captured step and what it was captured for
  cudaGraphExec_t exec = nullptr;
  int g_B = 0, g_gen = -1;
  std::vector<pnb_state *> g_states;
  const int32_t *g_tokens = nullptr;
  float *g_logits = nullptr;
  int32_t *g_argmax = nullptr;
};

struct pnb_state {
  pnb_model *m = nullptr;
  uint8_t *kv = nullptr;
  size_t kv_bytes = 0;
  int32_t pos = 0;                       // host mirror of the device position
  uint8_t *ws = nullptr;                 // device workspace
  StepIO *io = nullptr;
  float *x = nullptr, *q = nullptr, *attn = nullptr, *h = nullptr, *part = nullptr;
  float *gate = nullptr, *lm_val = nullptr;
  int32_t *idx = nullptr, *lm_idx = nullptr;
  unsigned *attn_cnt = nullptr, *lm_cnt = nullptr;
  size_t counters_off = 0, counters_bytes = 0;
  unsigned *work = nullptr;              // [launch][claim, done] item counters
  unsigned long long *ktrace = nullptr;  // optional per-CTA timestamps of the step's kernels
  void *maps = nullptr;                  // device [layer][K|V] tensor maps over kv (tensor-core attention)
  int g_gen = -1;                        // model mode generation the graph was captured in
  cudaGraphExec_t exec = nullptr;
  float *g_logits = nullptr;
  int32_t *g_argmax = nullptr;
  // begin / poll seam: the state's own stream, the event of its last begun
  // work, whether it is outstanding and the logits buffer it writes
  cudaStream_t astream = nullptr;
  cudaEvent_t aevent = nullptr;
  bool pending = false;
  float *a_logits = nullptr;
};

namespace {

int check_device(const pnb_model *m) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return PNB_E_CUDA;
  return dev == m->device ? PNB_OK : PNB_E_WRONG_DEVICE;
}

int validate_config(const pnb_config *c) {
  if (c->n_vocab <= 0 || c->n_embd <= 0 || c->n_head <= 0 || c->n_kv_head <= 0 ||
      c->n_layer <= 0 || c->n_ff <= 0 || c->n_ctx <= 0)
    return PNB_E_INVAL;
  if (c->n_embd % c->n_head || c->n_head % c->n_kv_head) return PNB_E_INVAL;
  if (c->rope_neox != 0 && c->rope_neox != 1) return PNB_E_INVAL;
  const int hd = c->n_embd / c->n_head;
  if (hd % 2) return PNB_E_INVAL;
  if (hd != 32 && hd != 64 && hd != 128) return PNB_E_UNSUPPORTED;
  if (c->n_embd % 8 || c->n_ff % 8) return PNB_E_INVAL;
  if (c->sliding_window < 0 || !(c->rope_theta > 0.0) || !(c->rms_norm_eps >= 0.0)) return PNB_E_INVAL;
  if (c->dtype != PNB_F32 && c->dtype != PNB_BF16 && c->dtype != PNB_Q8_0 && c->dtype != PNB_Q4_0)
    return PNB_E_INVAL;
  // Q8 / Q4 rows (the values, then K / 32 fp16 scales) are whole 16-byte vectors
  if ((c->dtype == PNB_Q8_0 || c->dtype == PNB_Q4_0) && (c->n_embd % 256 || c->n_ff % 256))
    return PNB_E_UNSUPPORTED;
  if (c->expert_count < 0 || c->expert_count > 64) return PNB_E_INVAL;
  if (c->expert_count > 0 &&
      (c->expert_used <= 0 || c->expert_used > c->expert_count || c->expert_used > kMaxSegments))
    return PNB_E_INVAL;
  return PNB_OK;
}

void plan(pnb_model *m) {
  const pnb_config &c = m->cfg;
  const int E = c.n_embd, F = c.n_ff, wt = c.dtype, grid = m->grid;
  const int k = c.expert_count > 0 ? c.expert_used : 1;
  m->g_qkv = plan_gemv(E, wt, m->qkv_rows, 2, 1, grid, 1);
  m->g_o = plan_gemv(c.n_head * m->hd, wt, E, 1, 1, grid, 1);
  m->g_gateup = plan_gemv(E, wt, (int64_t)k * 2 * F, 2, 1, grid, k);
  m->g_down = plan_gemv(F, wt, E, 1, k, grid, c.expert_count > 0 ? 0 : 1);
  m->g_lm = plan_gemv(E, wt, c.n_vocab, 1, 1, grid, 1);
  const int G = c.n_head / c.n_kv_head;
  m->ag = attn_geom(m->kv_dt, m->hd, G);
  m->zgroups = G / m->ag.heads_per_cta;
  // one wave: at most one CTA per SM (the attention CTA's registers allow one)
  const int want = std::max(1, m->num_sms / (c.n_kv_head * m->zgroups));
  m->n_split = std::max(1, std::min(want, std::max(1, m->cap / 16)));
  // tensor-core attention: 128-position tiles; a ring cache must hold whole tiles
  m->attn_tc_ok = m->kv_dt == PNB_BF16 && (m->hd == 64 || m->hd == 128) &&
                  (G == 1 || G == 2 || G == 4 || G == 8) &&
                  (c.sliding_window == 0 || m->cap % 128 == 0);
  // the splits of a KV head form one thread-block cluster (merged in shared memory)
  m->n_split_tc = std::max(1, std::min({attn_tc_max_split(), m->num_sms / c.n_kv_head, ceil_div(m->cap, 128)}));
}

int max_smem(const pnb_model *m) {
  int s = std::max({smem_layout(m->g_qkv).total, smem_layout(m->g_o).total,
                    smem_layout(m->g_gateup).total, smem_layout(m->g_down).total,
                    smem_layout(m->g_lm).total, m->ag.smem});
  return s;
}

// every streaming GEMV fits the kernels' register slices (at most 4 vectors per lane)
bool geoms_supported(const pnb_model *m) {
  for (const Geom *g : {&m->g_qkv, &m->g_o, &m->g_gateup, &m->g_down, &m->g_lm})
    if (g->nv > 4) return false;
  return true;
}

// Enqueue one kernel of the single-sequence step.
cudaError_t enqueue_kernel(pnb_model *m, pnb_state *s, int kind, int l, cudaStream_t st, bool pdl,
                           float *logits, int32_t *argmax) {
  const pnb_config &c = m->cfg;
  const int E = c.n_embd, H = c.n_head, Hkv = c.n_kv_head, hd = m->hd, F = c.n_ff;
  const size_t layer_kv = (size_t)Hkv * m->cap * hd * m->kv_es;
  uint8_t *kc = s->kv + (size_t)(2 * l) * layer_kv, *vc = kc + layer_kv;
  const float eps = (float)c.rms_norm_eps;
  const bool moe = c.expert_count > 0;
  const int k = moe ? c.expert_used : 1;
  const KTrace tr{s->ktrace, kind == PNB_KERNEL_LM_HEAD ? 6 * c.n_layer : 6 * l + kind};
  unsigned *work = s->work + 2 * tr.phase;
  switch (kind) {
    case PNB_KERNEL_QKV: {
      QkvArgs qa{};
      qa.g = m->g_qkv;
      qa.s.n = 1;
      qa.s.rows = m->qkv_rows;
      qa.s.w[0] = m->wqkv[l];
      qa.x = s->x;
      qa.emb = l == 0 ? m->tok_embd : nullptr;
      qa.x_out = s->x;
      qa.n_vocab = c.n_vocab;
      qa.norm_w = m->attn_norm[l];
      qa.eps = eps;
      qa.n_head = H;
      qa.n_kv = Hkv;
      qa.head_dim = hd;
      qa.inv_freq = m->inv_freq;
      qa.bias = m->bqkv.empty() ? nullptr : m->bqkv[l];
      qa.q = s->q;
      qa.k_cache = kc;
      qa.v_cache = vc;
      qa.cap = m->cap;
      qa.window = c.sliding_window;
      qa.io = s->io;
      qa.tr = tr;
      qa.work = work;
      return launch_qkv(c.dtype, qa, m->grid, st, pdl);
    }
    case PNB_KERNEL_ATTN: {
      if (m->attn_tc) {
        AttnTcArgs ta{};
        ta.q = s->q;
        ta.maps = s->maps;
        ta.layer = l;
        ta.n_head = H;
        ta.n_kv = Hkv;
        ta.cap = m->cap;
        ta.window = c.sliding_window;
        ta.n_split = m->n_split_tc;
        ta.qscale = (float)(1.4426950408889634 / std::sqrt((double)hd));
        ta.out = s->attn;
        ta.io = s->io;
        ta.nstages = attn_tc_stages(hd);
        ta.tr = tr;
        return launch_attn_tc(hd, H / Hkv, ta, st, pdl);
      }
      AttnArgs aa{};
      aa.q = s->q;
      aa.k_cache = kc;
      aa.v_cache = vc;
      aa.n_head = H;
      aa.n_kv = Hkv;
      aa.cap = m->cap;
      aa.window = c.sliding_window;
      aa.n_split = m->n_split;
      aa.part = s->part;
      aa.counter = s->attn_cnt;
      aa.out = s->attn;
      aa.qscale = (float)(1.4426950408889634 / std::sqrt((double)hd));
      aa.stage_pos = m->ag.stage_pos;
      aa.nstages = m->ag.nstages;
      aa.io = s->io;
      aa.tr = tr;
      return launch_attn(m->kv_dt, hd, aa, m->ag, st, pdl);
    }
    case PNB_KERNEL_OPROJ: {
      ResidArgs oa{};
      oa.g = m->g_o;
      oa.s.n = 1;
      oa.s.rows = E;
      oa.s.w[0] = m->wo[l];
      oa.vec = s->attn;
      oa.x = s->x;
      oa.io = s->io;
      oa.tr = tr;
      oa.work = work;
      return launch_resid(c.dtype, oa, m->grid, st, pdl);
    }
    case PNB_KERNEL_ROUTER: {
      if (!moe) return cudaErrorInvalidValue;
      RouterArgs ra{};
      ra.w = m->w_router[l];
      ra.n_expert = c.expert_count;
      ra.k = k;
      ra.E = E;
      ra.x = s->x;
      ra.norm_w = m->ffn_norm[l];
      ra.eps = eps;
      ra.idx = s->idx;
      ra.gate = s->gate;
      ra.io = s->io;
      ra.tr = tr;
      return launch_router(c.dtype, ra, st, pdl);
    }
    case PNB_KERNEL_GATE_UP: {
      GateUpArgs ga{};
      ga.g = m->g_gateup;
      ga.s.rows = 2 * (int64_t)F;
      ga.x = s->x;
      ga.norm_w = m->ffn_norm[l];
      ga.eps = eps;
      ga.h = s->h;
      ga.n_ff = F;
      ga.io = s->io;
      ga.tr = tr;
      ga.work = work;
      ga.s.n = k;
      if (moe) {
        ga.s.table = m->tab_gate_up + (size_t)l * c.expert_count;
        ga.s.expert_idx = s->idx;
      } else {
        ga.s.w[0] = m->w_gate_up[l];
      }
      return launch_gateup(c.dtype, ga, m->grid, st, pdl);
    }
    case PNB_KERNEL_DOWN: {
      if (!moe) {
        ResidArgs da{};
        da.g = m->g_down;
        da.s.n = 1;
        da.s.rows = E;
        da.s.w[0] = m->w_down[l];
        da.vec = s->h;
        da.x = s->x;
        da.io = s->io;
        da.tr = tr;
        da.work = work;
        return launch_resid(c.dtype, da, m->grid, st, pdl);
      }
      DownMoeArgs da{};
      da.g = m->g_down;
      da.s.n = k;
      da.s.rows = E;
      da.s.table = m->tab_down + (size_t)l * c.expert_count;
      da.s.expert_idx = s->idx;
      da.h = s->h;
      da.n_ff = F;
      da.gate = s->gate;
      da.x = s->x;
      da.io = s->io;
      da.tr = tr;
      return launch_down_moe(c.dtype, da, m->grid, st, pdl);
    }
    case PNB_KERNEL_LM_HEAD: {
      LmArgs la{};
      la.g = m->g_lm;
      la.s.n = 1;
      la.s.rows = c.n_vocab;
      la.s.w[0] = m->output;
      la.x = s->x;
      la.norm_w = m->out_norm;
      la.eps = eps;
      la.logits = logits;
      la.argmax_out = argmax;
      la.part_val = s->lm_val;
      la.part_idx = s->lm_idx;
      la.counter = s->lm_cnt;
      la.io = s->io;
      la.tr = tr;
      la.work = work;
      return launch_lmhead(c.dtype, la, m->grid, st, pdl);
    }
    default:
      return cudaErrorInvalidValue;
  }
}

// Enqueue one single-sequence step (everything after the token write): one
// kernel per phase; the first waits for all earlier stream work, every later
// one is launched with programmatic stream serialization.
cudaError_t enqueue_step(pnb_model *m, pnb_state *s, cudaStream_t st, float *logits,
                         int32_t *argmax) {
  const bool moe = m->cfg.expert_count > 0;
  cudaError_t e;
  for (int l = 0; l < m->cfg.n_layer; ++l) {
    if ((e = enqueue_kernel(m, s, PNB_KERNEL_QKV, l, st, l > 0, nullptr, nullptr)) != cudaSuccess)
      return e;
    if ((e = enqueue_kernel(m, s, PNB_KERNEL_ATTN, l, st, true, nullptr, nullptr)) != cudaSuccess)
      return e;
    if ((e = enqueue_kernel(m, s, PNB_KERNEL_OPROJ, l, st, true, nullptr, nullptr)) != cudaSuccess)
      return e;
    if (moe && (e = enqueue_kernel(m, s, PNB_KERNEL_ROUTER, l, st, true, nullptr, nullptr)) !=
                   cudaSuccess)
      return e;
    if ((e = enqueue_kernel(m, s, PNB_KERNEL_GATE_UP, l, st, true, nullptr, nullptr)) != cudaSuccess)
      return e;
    if ((e = enqueue_kernel(m, s, PNB_KERNEL_DOWN, l, st, true, nullptr, nullptr)) != cudaSuccess)
      return e;
  }
  return enqueue_kernel(m, s, PNB_KERNEL_LM_HEAD, 0, st, true, logits, argmax);
}


// ------------------------------------------------------------ batched step

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    cudaDriverEntryPointQueryResult q;
    void *p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// 2-D bf16 tensor map over [rows][K] (K contiguous), boxes of 64 columns x box_rows
// rows, 128-byte swizzle (the layout the tcgen05 descriptors expect)
bool encode_map(CUtensorMap *map, const void *base, int64_t rows, int K, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  const cuuint32_t es[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Split of a GEMM over K so that (tiles x ksplit) units fill whole waves of
// the SMs: the smallest split reaching 88% wave efficiency, else the best.
BPlan plan_bgemm(int64_t rows, int K, int num_sms) {
  BPlan p;
  p.rows = (int)rows;
  p.K = K;
  p.tiles = ceil_div(rows, 128);
  const int nchunks = K / 64;
  double best = -1.0;
  for (int ks = 1; ks <= std::min(16, nchunks); ++ks) {
    const int64_t U = (int64_t)p.tiles * ks;
    const int64_t waves = (U + num_sms - 1) / num_sms;
    const double eff = (double)U / (double)(waves * num_sms);
    if (eff > best + 1e-9) {
      best = eff;
      p.ksplit = ks;
    }
    if (eff >= 0.88) {
      p.ksplit = ks;
      break;
    }
  }
  p.units = p.tiles * p.ksplit;
  p.grid = std::min(p.units, num_sms);
  return p;
}

int bp_index(int bp) { return bp == 16 ? 0 : (bp == 32 ? 1 : (bp == 64 ? 2 : 3)); }

int attn_split_b(const pnb_model *m, int B) {
  if (m->attn_tc) {
    // one wave of CTAs split evenly; when one CTA per (slot, KV head) would
    // leave part of the wave idle, two per slot (the long slots' CTAs start
    // first, so the second partial wave fills in behind them)
    const int per = m->cfg.n_kv_head * B;
    int split = m->num_sms / per;
    if (split == 1 && per < m->num_sms) split = 2;
    return std::max(1, std::min({attn_tc_max_split(), split, ceil_div(m->cap, 128)}));
  }
  const int per = m->cfg.n_kv_head * m->zgroups * B;
  return std::max(1, std::min(m->num_sms / std::max(1, per), std::max(1, m->cap / 16)));
}

int attn_split_b_max(const pnb_model *m, int B) {
  const int tc = std::max(1, std::min({attn_tc_max_split(), m->num_sms / (m->cfg.n_kv_head * B),
                                       ceil_div(m->cap, 128)}));
  const int per = m->cfg.n_kv_head * m->zgroups * B;
  const int cc = std::max(1, std::min(m->num_sms / std::max(1, per), std::max(1, m->cap / 16)));
  return std::max(tc, cc);
}

void batch_free(BatchCtx *b) {
  if (!b) return;
  if (b->exec) cudaGraphExecDestroy(b->exec);
  cudaFree(b->ws);
  delete b;
}

// Batched-slot workspace, tensor maps and plans (bf16 dense models; outside
// any stream capture).
int batch_setup(pnb_model *m) {
  if (m->batch) return PNB_OK;
  const pnb_config &c = m->cfg;
  const int E = c.n_embd, F = c.n_ff, Hd = c.n_head * m->hd, L = c.n_layer;
  const int MB = kMaxChunk, BPmax = 128;
  BatchCtx *b = new (std::nothrow) BatchCtx();
  if (!b) return PNB_E_NOMEM;
  b->p_qkv = plan_bgemm(m->qkv_rows, E, m->num_sms);
  b->p_o = plan_bgemm(E, Hd, m->num_sms);
  b->p_gu = plan_bgemm(2 * (int64_t)F, E, m->num_sms);
  b->p_dn = plan_bgemm(E, F, m->num_sms);
  b->p_lm = plan_bgemm(c.n_vocab, E, m->num_sms);
  int64_t gpart = 0, tiles = 0;
  for (const BPlan *p : {&b->p_qkv, &b->p_o, &b->p_gu, &b->p_dn, &b->p_lm}) {
    if (p->ksplit > 1) gpart = std::max(gpart, (int64_t)p->units * MB * 128);
    tiles = std::max(tiles, (int64_t)p->tiles);
  }
  int64_t apart = 0;
  for (int B = 1; B <= MB; ++B)
    apart = std::max(apart, (int64_t)B * attn_split_b_max(m, B) * c.n_head * (m->hd + 2));
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off += align256(bytes);
    return o;
  };
  const size_t o_xb = take((size_t)MB * E * 4), o_qb = take((size_t)MB * Hd * 4);
  const size_t o_ap = take((size_t)apart * 4), o_ac = take((size_t)MB * c.n_kv_head * m->zgroups * 4);
  const size_t o_xe = take((size_t)2 * BPmax * E * 2), o_xo = take((size_t)2 * BPmax * Hd * 2);
  const size_t o_xf = take((size_t)2 * BPmax * F * 2);
  const size_t o_rope = take((size_t)MB * (m->hd / 2) * 8), o_pos = take((size_t)MB * 4);
  const size_t o_slots = take((size_t)MB * sizeof(BSlot));
  const size_t o_gp = take((size_t)std::max<int64_t>(gpart, 1) * 4), o_tc = take((size_t)tiles * 4);
  const size_t o_amv = take((size_t)MB * m->num_sms * 4), o_ami = take((size_t)MB * m->num_sms * 4);
  const size_t o_amc = take(4), o_err = take(4), o_pio = take((size_t)MB * sizeof(StepIO));
  const size_t o_gates = take((size_t)MB * std::max(1, c.expert_count) * 4);
  const size_t o_acc = take((size_t)MB * E * 8);
  const size_t o_lgs = take((size_t)MB * c.n_vocab * 4);
  const size_t o_tpc = take(2 * sizeof(unsigned));
  if (cudaMalloc(&b->ws, off) != cudaSuccess) {
    delete b;
    return PNB_E_NOMEM;
  }
  if (cudaMemset(b->ws, 0, off) != cudaSuccess) {
    batch_free(b);
    return PNB_E_CUDA;
  }
  b->xb = reinterpret_cast<float *>(b->ws + o_xb);
  b->qb = reinterpret_cast<float *>(b->ws + o_qb);
  b->apart = reinterpret_cast<float *>(b->ws + o_ap);
  b->acnt = reinterpret_cast<unsigned *>(b->ws + o_ac);
  b->xop_e = reinterpret_cast<__nv_bfloat16 *>(b->ws + o_xe);
  b->xop_o = reinterpret_cast<__nv_bfloat16 *>(b->ws + o_xo);
  b->xop_f = reinterpret_cast<__nv_bfloat16 *>(b->ws + o_xf);
  b->rope = reinterpret_cast<float2 *>(b->ws + o_rope);
  b->pos = reinterpret_cast<int32_t *>(b->ws + o_pos);
  b->slots = reinterpret_cast<BSlot *>(b->ws + o_slots);
  b->gpart = reinterpret_cast<float *>(b->ws + o_gp);
  b->tile_cnt = reinterpret_cast<unsigned *>(b->ws + o_tc);
  b->am_val = reinterpret_cast<float *>(b->ws + o_amv);
  b->am_idx = reinterpret_cast<int32_t *>(b->ws + o_ami);
  b->am_cnt = reinterpret_cast<unsigned *>(b->ws + o_amc);
  b->err = reinterpret_cast<int32_t *>(b->ws + o_err);
  b->pio = reinterpret_cast<StepIO *>(b->ws + o_pio);
  b->gates = reinterpret_cast<float *>(b->ws + o_gates);
  b->acc = reinterpret_cast<long long *>(b->ws + o_acc);
  b->lgs = reinterpret_cast<float *>(b->ws + o_lgs);
  b->tp_cnt = reinterpret_cast<unsigned *>(b->ws + o_tpc);
  bool ok = true;
  b->w_qkv.resize(L);
  b->w_o.resize(L);
  const int S = m->n_sets;                // experts (1 when dense): maps per layer and expert
  b->w_gu.resize((size_t)L * S);
  b->w_dn.resize((size_t)L * S);
  for (int l = 0; l < L && ok; ++l) {
    ok = encode_map(&b->w_qkv[l], m->wqkv[l], m->qkv_rows, E, 128) &&
         encode_map(&b->w_o[l], m->wo[l], E, Hd, 128);
    for (int e = 0; ok && e < S; ++e)
      ok = encode_map(&b->w_gu[(size_t)l * S + e], m->w_gate_up[(size_t)l * S + e], 2 * (int64_t)F,
                      E, 128) &&
           encode_map(&b->w_dn[(size_t)l * S + e], m->w_down[(size_t)l * S + e], E, F, 128);
  }
  ok = ok && encode_map(&b->w_lm, m->output, c.n_vocab, E, 128);
  for (int i = 0; i < 4 && ok; ++i) {
    const int bp = 16 << i;
    ok = encode_map(&b->x_e[i], b->xop_e, 2 * bp, E, 2 * bp) &&
         encode_map(&b->x_o[i], b->xop_o, 2 * bp, Hd, 2 * bp) &&
         encode_map(&b->x_f[i], b->xop_f, 2 * bp, F, 2 * bp);
    const int fixed = bgemm_smem(bp, 0);
    b->nstages[i] = std::min(8, (kMaxSmem - fixed) / (128 * 128 + 2 * bp * 128));
    b->smem[i] = bgemm_smem(bp, b->nstages[i]);
  }
  if (!ok) {
    batch_free(b);
    return PNB_E_UNSUPPORTED;
  }
  if (prepare_bgemm_kernels(kMaxSmem) != cudaSuccess || prepare_pattn_kernels() != cudaSuccess) {
    batch_free(b);
    return PNB_E_CUDA;
  }
  m->batch = b;
  return PNB_OK;
}

BGemmArgs bgemm_args(const pnb_model *m, const BatchCtx *b, const BPlan &p, int kind, int B, int bp) {
  BGemmArgs g{};
  g.rows = p.rows;
  g.K = p.K;
  g.nchunks = p.K / 64;
  g.tiles = p.tiles;
  g.ksplit = p.ksplit;
  g.units = p.units;
  g.B = B;
  g.bp = bp;
  g.kind = kind;
  g.nstages = b->nstages[bp_index(bp)];
  g.part = b->gpart;
  g.tile_cnt = b->tile_cnt;
  g.rope = b->rope;
  g.slots = b->slots;
  g.pos = b->pos;
  g.n_head = m->cfg.n_head;
  g.n_kv = m->cfg.n_kv_head;
  g.hd = m->hd;
  g.cap = m->cap;
  g.err = b->err;
  g.acc = b->acc;
  if (m->det_batch && kind == kEpiResid) g.kind = kEpiResidFix;
  if (m->det_batch && kind == kEpiResidGate) g.kind = kEpiResidGateFix;
  return g;
}

// Enqueue one batched step: per layer the attention norm, QKV GEMM (RoPE, KV
// store), attention, o-proj GEMM (residual), FFN norm, gate/up GEMM (SwiGLU),
// down GEMM (residual); then the final norm and the LM-head GEMM (argmax,
// position advance).  The first kernel waits for all earlier stream work;
// every later one uses programmatic stream serialization.
// chunk: the slots are one sequence's consecutive tokens sharing its cache
// (a prefill chunk).  kChunkKernel: the attention runs as one CUDA-core chunk
// kernel; kChunkGroups: on the tensor cores, consecutive tokens sharing each
// pass over the cached positions (token groups); kChunkSlots: the per-slot
// attention kernel, each token a slot.
enum { kSlots = 0, kChunkKernel = 1, kChunkGroups = 2, kChunkSlots = 3 };
cudaError_t enqueue_batch(pnb_model *m, const BSlot *slots, int B, const int32_t *tokens,
                          unsigned long long *trace, cudaStream_t st, float *logits, int32_t *argmax,
                          int chunk = kSlots, const uint8_t *order = nullptr) {
  const bool shared_kv = chunk == kChunkKernel;
  BatchCtx *b = m->batch;
  const pnb_config &c = m->cfg;
  const int E = c.n_embd, Hd = c.n_head * m->hd, F = c.n_ff;
  const int bp = B <= 16 ? 16 : (B <= 32 ? 32 : (B <= 64 ? 64 : 128)), bi = bp_index(bp);
  const int smem = b->smem[bi];
  const size_t layer_kv = (size_t)c.n_kv_head * m->cap * m->hd * m->kv_es;
  const float eps = (float)c.rms_norm_eps;
  cudaError_t e;
  BNormArgs na{};
  na.x = b->xb;
  na.x_out = b->xb;
  na.n_vocab = c.n_vocab;
  na.E = E;
  na.B = B;
  na.bp = bp;
  na.eps = eps;
  na.xop = b->xop_e;
  na.slots_dev = b->slots;
  na.pos = b->pos;
  na.rope = b->rope;
  na.inv_freq = m->inv_freq;
  na.hd = m->hd;
  na.n_ctx = c.n_ctx;
  na.err = b->err;
  for (int i = 0; i < B; ++i) na.slots[i] = slots[i];
  for (int l = 0; l < c.n_layer; ++l) {
    na.emb = l == 0 ? m->tok_embd : nullptr;
    na.tokens = l == 0 ? tokens : nullptr;
    na.acc = l == 0 || !m->det_batch ? nullptr : b->acc;
    na.norm_w = m->attn_norm[l];
    na.tr = KTrace{trace, 7 * l};
    if ((e = launch_bnorm(na, st, l > 0)) != cudaSuccess) return e;
    BGemmArgs g = bgemm_args(m, b, b->p_qkv, kEpiQkv, B, bp);
    g.tr = KTrace{trace, 7 * l + 1};
    g.bias = m->bqkv.empty() ? nullptr : m->bqkv[l];
    g.q = b->qb;
    g.kv_off = (size_t)(2 * l) * layer_kv;
    g.layer_kv_bytes = layer_kv;
    if ((e = launch_bgemm(&b->w_qkv[l], &b->x_e[bi], g, b->p_qkv.grid, smem, st, true)) != cudaSuccess)
      return e;
    if (g.ksplit > 1 && (e = launch_bmerge(g, st, true)) != cudaSuccess) return e;
    if (shared_kv) {
      PAttnArgs pa{};
      pa.q = b->qb;
      pa.k = reinterpret_cast<const __nv_bfloat16 *>(slots[0].kv + (size_t)(2 * l) * layer_kv);
      pa.v = reinterpret_cast<const __nv_bfloat16 *>(slots[0].kv + (size_t)(2 * l + 1) * layer_kv);
      pa.pos = b->pos;
      pa.n = B;
      pa.n_head = c.n_head;
      pa.n_kv = c.n_kv_head;
      pa.cap = m->cap;
      pa.window = c.sliding_window;
      pa.qscale = (float)(1.4426950408889634 / std::sqrt((double)m->hd));
      pa.xop = b->xop_o;
      pa.xop_ld = Hd;
      pa.bp = bp;
      if ((e = launch_pattn(m->hd, pa, st, true)) != cudaSuccess) return e;
    } else if (m->attn_tc) {
      AttnTcArgs ta{};
      ta.q = b->qb;
      ta.layer = l;
      ta.n_head = c.n_head;
      ta.n_kv = c.n_kv_head;
      ta.cap = m->cap;
      ta.window = c.sliding_window;
      ta.n_split = attn_split_b(m, B);
      ta.qscale = (float)(1.4426950408889634 / std::sqrt((double)m->hd));
      ta.xop = b->xop_o;
      ta.xop_ld = Hd;
      ta.bp = bp;
      ta.nb = B;
      ta.slots = b->slots;
      ta.pos = b->pos;
      ta.nstages = attn_tc_stages(m->hd);
      ta.tr = KTrace{trace, 7 * l + 2};
      ta.shared_cache = chunk != kSlots;
      if (chunk == kSlots && order) {
        ta.use_order = 1;
        for (int i = 0; i < B; ++i) ta.order[i] = order[i];
      }
      // more (slot, KV head) items than SMs, one split each: one persistent
      // CTA per SM walks its items with the ring running on between them
      if (chunk == kSlots && ta.n_split == 1 && m->hd == 128 && B * c.n_kv_head > m->num_sms) {
        ta.persist = m->num_sms;
        ta.tp_claim = b->tp_cnt;
      }
      int cols = c.n_head / c.n_kv_head;
      if (chunk == kChunkGroups) {
        // a chunk's tokens share the cache: T consecutive tokens per CTA
        // column block (all 8 columns of the MMA) read the cached positions
        // once for all of them instead of once each
        ta.tok_group = std::max(1, 8 / cols);
        cols *= ta.tok_group;
        const int groups = (B + ta.tok_group - 1) / ta.tok_group;
        ta.n_split = std::max(1, std::min({attn_tc_max_split(), m->num_sms / (c.n_kv_head * groups),
                                           ceil_div(m->cap, 128)}));
      }
      if ((e = launch_attn_tc(m->hd, cols, ta, st, true)) != cudaSuccess) return e;
    } else {
    AttnArgs aa{};
    aa.q = b->qb;
    aa.n_head = c.n_head;
    aa.n_kv = c.n_kv_head;
    aa.cap = m->cap;
    aa.window = c.sliding_window;
    aa.n_split = attn_split_b(m, B);
    aa.part = b->apart;
    aa.counter = b->acnt;
    aa.qscale = (float)(1.4426950408889634 / std::sqrt((double)m->hd));
    aa.stage_pos = m->ag.stage_pos;
    aa.nstages = m->ag.nstages;
    aa.slots = b->slots;
    aa.pos = b->pos;
    aa.kv_off = (size_t)(2 * l) * layer_kv;
    aa.layer_kv_bytes = layer_kv;
    aa.xop = b->xop_o;
    aa.xop_ld = Hd;
    aa.bp = bp;
    aa.nb = B;
    aa.shared_cache = chunk != kSlots;
    aa.tr = KTrace{trace, 7 * l + 2};
    if ((e = launch_attn(m->kv_dt, m->hd, aa, m->ag, st, true)) != cudaSuccess) return e;
    }
    g = bgemm_args(m, b, b->p_o, kEpiResid, B, bp);
    g.tr = KTrace{trace, 7 * l + 3};
    g.x = b->xb;
    if ((e = launch_bgemm(&b->w_o[l], &b->x_o[bi], g, b->p_o.grid, smem, st, true)) != cudaSuccess)
      return e;
    na.emb = nullptr;
    na.tokens = nullptr;
    na.acc = m->det_batch ? b->acc : nullptr;
    na.norm_w = m->ffn_norm[l];
    na.tr = KTrace{trace, 7 * l + 4};
    if ((e = launch_bnorm(na, st, true)) != cudaSuccess) return e;
    // dense: one SwiGLU FFN.  MoE: the router gives every slot its experts'
    // weights; then each expert's FFN runs over all slots (the weights are
    // streamed once either way, and at these slot counts that is the cost)
    // and its down projection adds weight * output to the slots that chose it
    const int S = m->n_sets;
    if (c.expert_count > 0) {
      BRouterArgs ra{};
      ra.w = static_cast<const __nv_bfloat16 *>(m->w_router[l]);
      ra.n_expert = c.expert_count;
      ra.k = c.expert_used;
      ra.E = E;
      ra.x = b->xb;
      ra.norm_w = m->ffn_norm[l];
      ra.eps = (float)c.rms_norm_eps;
      ra.gates = b->gates;
      ra.tr = KTrace{trace, 7 * l + 4};
      if ((e = launch_brouter(ra, B, st, true)) != cudaSuccess) return e;
    }
    for (int ex = 0; ex < S; ++ex) {
      g = bgemm_args(m, b, b->p_gu, kEpiGateUp, B, bp);
      g.tr = KTrace{trace, 7 * l + 5};
      g.xop = b->xop_f;
      g.xop_ld = F;
      if ((e = launch_bgemm(&b->w_gu[(size_t)l * S + ex], &b->x_e[bi], g, b->p_gu.grid, smem, st,
                            true)) != cudaSuccess)
        return e;
      if (g.ksplit > 1 && (e = launch_bmerge(g, st, true)) != cudaSuccess) return e;
      g = bgemm_args(m, b, b->p_dn, c.expert_count > 0 ? kEpiResidGate : kEpiResid, B, bp);
      g.tr = KTrace{trace, 7 * l + 6};
      g.x = b->xb;
      if (c.expert_count > 0) {
        g.gate = b->gates + ex;
        g.gate_ld = c.expert_count;
      }
      if ((e = launch_bgemm(&b->w_dn[(size_t)l * S + ex], &b->x_f[bi], g, b->p_dn.grid, smem, st,
                            true)) != cudaSuccess)
        return e;
    }
  }
  na.emb = nullptr;
  na.tokens = nullptr;
  na.acc = m->det_batch ? b->acc : nullptr;
  na.norm_w = m->out_norm;
  na.tr = KTrace{trace, 7 * c.n_layer};
  if ((e = launch_bnorm(na, st, true)) != cudaSuccess) return e;
  BGemmArgs g = bgemm_args(m, b, b->p_lm, kEpiLm, B, bp);
  g.tr = KTrace{trace, 7 * c.n_layer + 1};
  g.logits = logits;
  g.argmax_out = argmax;
  g.am_val = b->am_val;
  g.am_idx = b->am_idx;
  g.am_cnt = b->am_cnt;
  if (bp <= 64) return launch_bgemm(&b->w_lm, &b->x_e[bi], g, b->p_lm.grid, smem, st, true);
  // 128 slots: the LM head writes logits only; the greedy pick follows
  if (!logits) g.logits = b->lgs;
  if ((e = launch_bgemm(&b->w_lm, &b->x_e[bi], g, b->p_lm.grid, smem, st, true)) != cudaSuccess) return e;
  BArgmaxArgs ma{};
  ma.logits = g.logits;
  ma.V = c.n_vocab;
  ma.B = B;
  ma.slots = b->slots;
  ma.pos = b->pos;
  ma.argmax_out = argmax;
  ma.err = b->err;
  return launch_bargmax(ma, st, true);
}

}  // namespace

extern "C" {

const char *pnb_strerror(int code) {
  switch (code) {
    case PNB_OK: return "ok";
    case PNB_E_INVAL: return "invalid configuration or argument";
    case PNB_E_NULL: return "required pointer is NULL";
    case PNB_E_ALIGN: return "device pointer not 16-byte aligned";
    case PNB_E_CTX_FULL: return "position reached n_ctx";
    case PNB_E_UNSUPPORTED: return "unsupported by this build";
    case PNB_E_CUDA: return "CUDA runtime error";
    case PNB_E_TOKEN: return "token id out of range";
    case PNB_E_DEVICE: return "device-side check failed";
    case PNB_E_NOMEM: return "allocation failed";
    case PNB_E_WRONG_DEVICE: return "current device differs from the model's device";
    case PNB_E_TOO_LARGE: return "exceeds the static scratch of the allocation-free entry point";
    case PNB_E_BUSY: return "a begun step of this state has not been polled to completion";
    default: return "unknown error";
  }
}

int pnb_model_create(const pnb_config *cfg, const pnb_weights *w, pnb_model **out) {
  if (!cfg || !w || !out) return PNB_E_NULL;
  *out = nullptr;
  int rc = validate_config(cfg);
  if (rc != PNB_OK) return rc;
  const pnb_config &c = *cfg;
  const bool moe = c.expert_count > 0;
  const int n_sets = moe ? c.expert_count : 1;
  if (!w->tok_embd || !w->out_norm || !w->output || !w->attn_norm || !w->wqkv || !w->wo ||
      !w->ffn_norm || !w->w_gate_up || !w->w_down || (moe && !w->w_router))
    return PNB_E_NULL;
  if (!aligned16(w->tok_embd) || !aligned16(w->out_norm) || !aligned16(w->output)) return PNB_E_ALIGN;
  for (int l = 0; l < c.n_layer; ++l) {
    const void *ps[] = {w->attn_norm[l], w->wqkv[l], w->wo[l], w->ffn_norm[l],
                        moe ? w->w_router[l] : w->wo[l]};
    for (const void *p : ps) {
      if (!p) return PNB_E_NULL;
      if (!aligned16(p)) return PNB_E_ALIGN;
    }
    for (int e = 0; e < n_sets; ++e) {
      const void *gu = w->w_gate_up[l * n_sets + e], *dn = w->w_down[l * n_sets + e];
      if (!gu || !dn) return PNB_E_NULL;
      if (!aligned16(gu) || !aligned16(dn)) return PNB_E_ALIGN;
    }
    if (w->bqkv) {
      if (!w->bqkv[l]) return PNB_E_NULL;
      if (!aligned16(w->bqkv[l])) return PNB_E_ALIGN;
    }
  }
  pnb_model *m = new (std::nothrow) pnb_model();
  if (!m) return PNB_E_NOMEM;
  try {
    m->cfg = c;
    m->hd = c.n_embd / c.n_head;
    m->n_sets = n_sets;
    m->qkv_rows = (c.n_head + 2 * c.n_kv_head) * m->hd;
    m->kv_dt = c.dtype == PNB_F32 ? PNB_F32 : PNB_BF16;
    m->kv_es = m->kv_dt == PNB_BF16 ? 2 : 4;
    m->cap = c.sliding_window > 0 ? std::min(c.sliding_window, c.n_ctx) : c.n_ctx;
    m->tok_embd = w->tok_embd;
    m->out_norm = w->out_norm;
    m->output = w->output;
    m->attn_norm.assign(w->attn_norm, w->attn_norm + c.n_layer);
    m->ffn_norm.assign(w->ffn_norm, w->ffn_norm + c.n_layer);
    m->wqkv.assign(w->wqkv, w->wqkv + c.n_layer);
    if (w->bqkv) m->bqkv.assign(w->bqkv, w->bqkv + c.n_layer);
    m->wo.assign(w->wo, w->wo + c.n_layer);
    if (moe) m->w_router.assign(w->w_router, w->w_router + c.n_layer);
    m->w_gate_up.assign(w->w_gate_up, w->w_gate_up + (size_t)c.n_layer * n_sets);
    m->w_down.assign(w->w_down, w->w_down + (size_t)c.n_layer * n_sets);
  } catch (...) {
    delete m;
    return PNB_E_NOMEM;
  }
  if (cudaGetDevice(&m->device) != cudaSuccess ||
      cudaDeviceGetAttribute(&m->num_sms, cudaDevAttrMultiProcessorCount, m->device) != cudaSuccess) {
    delete m;
    return PNB_E_CUDA;
  }
  m->grid = m->num_sms;
  plan(m);
  if (max_smem(m) > kMaxSmem || !geoms_supported(m)) {
    delete m;
    return PNB_E_UNSUPPORTED;
  }
  // RoPE frequencies rope_theta^(-2i/hd), fp64
  std::vector<double> f(m->hd / 2);
  for (int i = 0; i < m->hd / 2; ++i) f[i] = std::pow(c.rope_theta, -2.0 * i / m->hd);
  bool ok = cudaMalloc(&m->inv_freq, f.size() * sizeof(double)) == cudaSuccess &&
            cudaMemcpy(m->inv_freq, f.data(), f.size() * sizeof(double), cudaMemcpyHostToDevice) ==
                cudaSuccess;
  if (ok && moe) {
    const size_t n = (size_t)c.n_layer * c.expert_count;
    ok = cudaMalloc(&m->tab_gate_up, n * sizeof(void *)) == cudaSuccess &&
         cudaMalloc(&m->tab_down, n * sizeof(void *)) == cudaSuccess &&
         cudaMemcpy(m->tab_gate_up, m->w_gate_up.data(), n * sizeof(void *), cudaMemcpyHostToDevice) ==
             cudaSuccess &&
         cudaMemcpy(m->tab_down, m->w_down.data(), n * sizeof(void *), cudaMemcpyHostToDevice) ==
             cudaSuccess;
  }
  if (ok) ok = cudaStreamCreateWithFlags(&m->cap_stream, cudaStreamNonBlocking) == cudaSuccess;
  if (ok) ok = prepare_gemv_kernels(c.dtype, kMaxSmem) == cudaSuccess &&
               prepare_attn_kernel(m->kv_dt, m->hd, m->ag) == cudaSuccess;
  // the sampler: its fixed-point mass counters need n_vocab < 2^22, its
  // recent-token bitmap one bit per token in shared memory
  if (ok && c.n_vocab < (1 << 22) && sample_smem_bytes(c.n_vocab) <= (size_t)kMaxSmem)
    m->sample_ok = prepare_sample_kernel(c.n_vocab) == cudaSuccess;
  // tensor-core attention where the shape allows it (bf16 KV, whole tiles)
  if (ok) {
    if (m->attn_tc_ok) m->attn_tc_ok = encode_fn() != nullptr && prepare_attn_tc_kernels() == cudaSuccess;
    m->attn_tc = m->attn_tc_ok;
    cudaGetLastError();   // a declined option leaves no sticky launch error behind
  }
  if (!ok) {
    pnb_model_free(m);
    return PNB_E_CUDA;
  }
  *out = m;
  return PNB_OK;
}

void pnb_model_free(pnb_model *m) {
  if (!m) return;
  cudaFree(m->inv_freq);
  cudaFree(m->tab_gate_up);
  cudaFree(m->tab_down);
  if (m->cap_stream) cudaStreamDestroy(m->cap_stream);
  batch_free(m->batch);
  delete m;
}

size_t pnb_state_kv_bytes(const pnb_model *m) {
  if (!m) return 0;
  return (size_t)m->cfg.n_layer * 2 * m->cfg.n_kv_head * m->cap * m->hd * m->kv_es;
}

int pnb_state_new(pnb_model *m, void *kv_dev, size_t kv_bytes, pnb_state **out) {
  if (!m || !kv_dev || !out) return PNB_E_NULL;
  *out = nullptr;
  if (!aligned16(kv_dev)) return PNB_E_ALIGN;
  if (kv_bytes < pnb_state_kv_bytes(m)) return PNB_E_INVAL;
  int rc = check_device(m);
  if (rc != PNB_OK) return rc;
  const pnb_config &c = m->cfg;
  const int k = c.expert_count > 0 ? c.expert_used : 1;
  pnb_state *s = new (std::nothrow) pnb_state();
  if (!s) return PNB_E_NOMEM;
  s->m = m;
  s->kv = static_cast<uint8_t *>(kv_dev);
  s->kv_bytes = kv_bytes;
  // workspace carve
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off += align256(bytes);
    return o;
  };
  const size_t o_io = take(sizeof(StepIO));
  const size_t o_x = take((size_t)c.n_embd * 4);
  const size_t o_q = take((size_t)c.n_head * m->hd * 4);
  const size_t o_attn = take((size_t)c.n_head * m->hd * 4);
  const size_t o_h = take((size_t)k * c.n_ff * 4);
  const size_t o_part = take((size_t)c.n_head * std::max(m->n_split, m->n_split_tc) * (m->hd + 2) * 4);
  const size_t o_gate = take((size_t)k * 4);
  const size_t o_idx = take((size_t)k * 4);
  const size_t o_lmv = take((size_t)m->grid * 4);
  const size_t o_lmi = take((size_t)m->grid * 4);
  const size_t n_cnt = (size_t)(c.n_kv_head * m->zgroups + 1) + 2 * (6 * c.n_layer + 1);
  const size_t o_cnt = take(n_cnt * 4);
  const size_t o_maps = m->attn_tc_ok ? take((size_t)2 * c.n_layer * sizeof(CUtensorMap)) : 0;
  if (cudaMalloc(&s->ws, off) != cudaSuccess) {
    delete s;
    return PNB_E_NOMEM;
  }
  s->io = reinterpret_cast<StepIO *>(s->ws + o_io);
  s->x = reinterpret_cast<float *>(s->ws + o_x);
  s->q = reinterpret_cast<float *>(s->ws + o_q);
  s->attn = reinterpret_cast<float *>(s->ws + o_attn);
  s->h = reinterpret_cast<float *>(s->ws + o_h);
  s->part = reinterpret_cast<float *>(s->ws + o_part);
  s->gate = reinterpret_cast<float *>(s->ws + o_gate);
  s->idx = reinterpret_cast<int32_t *>(s->ws + o_idx);
  s->lm_val = reinterpret_cast<float *>(s->ws + o_lmv);
  s->lm_idx = reinterpret_cast<int32_t *>(s->ws + o_lmi);
  s->attn_cnt = reinterpret_cast<unsigned *>(s->ws + o_cnt);
  s->lm_cnt = s->attn_cnt + c.n_kv_head * m->zgroups;
  s->work = s->lm_cnt + 1;
  s->counters_off = o_cnt;
  s->counters_bytes = n_cnt * 4;
  std::vector<CUtensorMap> maps;
  if (m->attn_tc_ok) {
    // [layer][K|V] maps over this state's cache: rows = n_kv_head * cap positions, hd columns
    s->maps = s->ws + o_maps;
    maps.resize((size_t)2 * c.n_layer);
    const size_t layer_kv_b = (size_t)c.n_kv_head * m->cap * m->hd * m->kv_es;
    for (int l = 0; l < c.n_layer; ++l)
      for (int kind = 0; kind < 2; ++kind)
        if (!encode_map(&maps[2 * l + kind], s->kv + (size_t)(2 * l + kind) * layer_kv_b,
                        (int64_t)c.n_kv_head * m->cap, m->hd, 128)) {
          cudaFree(s->ws);
          delete s;
          return PNB_E_CUDA;
        }
  }
  if (cudaMemset(s->ws, 0, off) != cudaSuccess ||
      (s->maps && cudaMemcpy(s->maps, maps.data(), maps.size() * sizeof(CUtensorMap),
                             cudaMemcpyHostToDevice) != cudaSuccess)) {
    cudaFree(s->ws);
    delete s;
    return PNB_E_CUDA;
  }
  *out = s;
  return PNB_OK;
}

void pnb_state_free(pnb_state *s) {
  if (!s) return;
  if (s->exec) cudaGraphExecDestroy(s->exec);
  if (s->astream) cudaStreamSynchronize(s->astream);
  if (s->aevent) cudaEventDestroy(s->aevent);
  if (s->astream) cudaStreamDestroy(s->astream);
  cudaFree(s->ws);
  delete s;
}

int pnb_state_reset(pnb_state *s, pnb_stream stream) {
  if (!s) return PNB_E_NULL;
  int rc = check_device(s->m);
  if (rc != PNB_OK) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(s->kv, 0, pnb_state_kv_bytes(s->m), st) != cudaSuccess ||
      cudaMemsetAsync(s->io, 0, sizeof(StepIO), st) != cudaSuccess ||
      cudaMemsetAsync(s->ws + s->counters_off, 0, s->counters_bytes, st) != cudaSuccess)
    return PNB_E_CUDA;
  s->pos = 0;
  return PNB_OK;
}

int pnb_state_set_pos(pnb_state *s, int32_t pos, pnb_stream stream) {
  if (!s) return PNB_E_NULL;
  if (pos < 0 || pos >= s->m->cfg.n_ctx) return PNB_E_INVAL;
  int rc = check_device(s->m);
  if (rc != PNB_OK) return rc;
  if (launch_set_pos(s->io, pos, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return PNB_E_CUDA;
  s->pos = pos;
  return PNB_OK;
}

int pnb_state_get_pos(const pnb_state *s, int32_t *pos) {
  if (!s || !pos) return PNB_E_NULL;
  *pos = s->pos;
  return PNB_OK;
}

int pnb_state_check(pnb_state *s, int32_t *device_error) {
  if (!s) return PNB_E_NULL;
  int rc = check_device(s->m);
  if (rc != PNB_OK) return rc;
  StepIO io;
  if (cudaDeviceSynchronize() != cudaSuccess ||
      cudaMemcpy(&io, s->io, sizeof(io), cudaMemcpyDeviceToHost) != cudaSuccess)
    return PNB_E_CUDA;
  if (device_error) *device_error = io.error;
  return io.error ? PNB_E_DEVICE : PNB_OK;
}

int pnb_forward(pnb_model *m, pnb_state *s, int32_t token, pnb_stream stream, float *logits_dev,
                int32_t *argmax_dev) {
  if (!m || !s) return PNB_E_NULL;
  if (s->m != m) return PNB_E_INVAL;
  if (token != PNB_TOKEN_PREV && (token < 0 || token >= m->cfg.n_vocab)) return PNB_E_TOKEN;
  if ((logits_dev && !aligned16(logits_dev)) || (argmax_dev && (reinterpret_cast<uintptr_t>(argmax_dev) & 3u)))
    return PNB_E_ALIGN;
  if (s->pos >= m->cfg.n_ctx) return PNB_E_CTX_FULL;
  int rc = check_device(m);
  if (rc != PNB_OK) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (token != PNB_TOKEN_PREV && launch_set_token(s->io, token, st) != cudaSuccess) return PNB_E_CUDA;
  if (!m->graphs) {
    if (enqueue_step(m, s, st, logits_dev, argmax_dev) != cudaSuccess) return PNB_E_CUDA;
  } else {
    if (!s->exec || s->g_logits != logits_dev || s->g_argmax != argmax_dev || s->g_gen != m->mode_gen) {
      if (s->exec) {
        cudaGraphExecDestroy(s->exec);
        s->exec = nullptr;
      }
      cudaGraph_t graph = nullptr;
      if (cudaStreamBeginCapture(m->cap_stream, cudaStreamCaptureModeThreadLocal) != cudaSuccess)
        return PNB_E_CUDA;
      cudaError_t le = enqueue_step(m, s, m->cap_stream, logits_dev, argmax_dev);
      cudaError_t ce = cudaStreamEndCapture(m->cap_stream, &graph);
      if (le != cudaSuccess || ce != cudaSuccess) {
        if (graph) cudaGraphDestroy(graph);
        return PNB_E_CUDA;
      }
      cudaError_t ie = cudaGraphInstantiate(&s->exec, graph, 0);
      cudaGraphDestroy(graph);
      if (ie != cudaSuccess) {
        s->exec = nullptr;
        return PNB_E_CUDA;
      }
      s->g_logits = logits_dev;
      s->g_argmax = argmax_dev;
      s->g_gen = m->mode_gen;
    }
    if (cudaGraphLaunch(s->exec, st) != cudaSuccess) return PNB_E_CUDA;
  }
  s->pos += 1;
  return PNB_OK;
}

int pnb_forward_batch(pnb_model *m, pnb_state *const *states, int32_t B, const int32_t *tokens_dev,
                      pnb_stream stream, float *logits_dev, int32_t *argmax_dev) {
  if (!m || !states) return PNB_E_NULL;
  if (B < 1 || B > kMaxBatch) return PNB_E_INVAL;
  const pnb_config &c = m->cfg;
  if (c.dtype != PNB_BF16) return PNB_E_UNSUPPORTED;
  if (c.n_embd % 64 || (c.n_head * m->hd) % 64 || c.n_ff % 64) return PNB_E_UNSUPPORTED;
  for (int i = 0; i < B; ++i) {
    if (!states[i]) return PNB_E_NULL;
    if (states[i]->m != m) return PNB_E_INVAL;
    for (int j = 0; j < i; ++j)
      if (states[j] == states[i]) return PNB_E_INVAL;
  }
  if ((logits_dev && !aligned16(logits_dev)) ||
      (argmax_dev && (reinterpret_cast<uintptr_t>(argmax_dev) & 3u)) ||
      (tokens_dev && (reinterpret_cast<uintptr_t>(tokens_dev) & 3u)))
    return PNB_E_ALIGN;
  for (int i = 0; i < B; ++i)
    if (states[i]->pos >= c.n_ctx) return PNB_E_CTX_FULL;
  int rc = check_device(m);
  if (rc != PNB_OK) return rc;
  if (B == 1) {
    // one slot: the single-sequence step (weight-streaming GEMVs) is the faster
    // way through a batch of one; the slot's token is copied on the device
    cudaStream_t st1 = reinterpret_cast<cudaStream_t>(stream);
    if (tokens_dev && launch_copy_token(states[0]->io, tokens_dev, st1) != cudaSuccess) return PNB_E_CUDA;
    return pnb_forward(m, states[0], PNB_TOKEN_PREV, stream, logits_dev, argmax_dev);
  }
  if ((rc = batch_setup(m)) != PNB_OK) return rc;
  BatchCtx *b = m->batch;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  BSlot slots[kMaxBatch];
  for (int i = 0; i < B; ++i) slots[i] = BSlot{states[i]->kv, states[i]->io, states[i]->maps};
  // the attention's slot order: longest attended range first (ties: lower
  // slot), from the positions at capture; all slots advance together, so the
  // ranking holds while the graph is replayed
  uint8_t order[kMaxBatch];
  {
    int len[kMaxBatch];
    for (int i = 0; i < B; ++i) {
      const int64_t n = states[i]->pos + 1;
      len[i] = (int)(c.sliding_window > 0 ? std::min<int64_t>(n, c.sliding_window) : n);
      order[i] = (uint8_t)i;
    }
    std::stable_sort(order, order + B, [&](uint8_t x, uint8_t y) { return len[x] > len[y]; });
  }
  unsigned long long *trace = states[0]->ktrace;   // optional, the first slot's buffer
  if (!m->graphs) {
    if (enqueue_batch(m, slots, B, tokens_dev, trace, st, logits_dev, argmax_dev, kSlots, order) !=
        cudaSuccess)
      return PNB_E_CUDA;
  } else {
    const bool same = b->exec && b->g_B == B && b->g_gen == m->mode_gen && b->g_tokens == tokens_dev &&
                      b->g_logits == logits_dev &&
                      b->g_argmax == argmax_dev &&
                      std::equal(states, states + B, b->g_states.begin(), b->g_states.end());
    if (!same) {
      if (b->exec) {
        cudaGraphExecDestroy(b->exec);
        b->exec = nullptr;
      }
      cudaGraph_t graph = nullptr;
      if (cudaStreamBeginCapture(m->cap_stream, cudaStreamCaptureModeThreadLocal) != cudaSuccess)
        return PNB_E_CUDA;
      cudaError_t le = enqueue_batch(m, slots, B, tokens_dev, trace, m->cap_stream, logits_dev, argmax_dev,
                                     kSlots, order);
      cudaError_t ce = cudaStreamEndCapture(m->cap_stream, &graph);
      if (le != cudaSuccess || ce != cudaSuccess) {
        if (graph) cudaGraphDestroy(graph);
        return PNB_E_CUDA;
      }
      cudaError_t ie = cudaGraphInstantiate(&b->exec, graph, 0);
      cudaGraphDestroy(graph);
      if (ie != cudaSuccess) {
        b->exec = nullptr;
        return PNB_E_CUDA;
      }
      b->g_B = B;
      b->g_gen = m->mode_gen;
      b->g_states.assign(states, states + B);
      b->g_tokens = tokens_dev;
      b->g_logits = logits_dev;
      b->g_argmax = argmax_dev;
    }
    if (cudaGraphLaunch(b->exec, st) != cudaSuccess) return PNB_E_CUDA;
  }
  for (int i = 0; i < B; ++i) states[i]->pos += 1;
  return PNB_OK;
}

int pnb_sample_batch(pnb_model *m, pnb_state *const *states, int32_t B, float *logits_dev,
                     const pnb_sampling_params *params, const int32_t *const *recent_dev,
                     const int32_t *n_recent, pnb_stream stream, int32_t *tokens_dev) {
  if (!m || !states || !logits_dev || !params) return PNB_E_NULL;
  if (B < 1 || B > kSampleMaxSlots) return PNB_E_INVAL;
  if (!aligned16(logits_dev) || (tokens_dev && (reinterpret_cast<uintptr_t>(tokens_dev) & 3u)))
    return PNB_E_ALIGN;
  const int V = m->cfg.n_vocab;
  SampleArgs a;
  a.n_vocab = V;
  for (int b = 0; b < B; ++b) {
    pnb_state *s = states[b];
    const pnb_sampling_params &p = params[b];
    if (!s) return PNB_E_NULL;
    if (s->m != m) return PNB_E_INVAL;
    for (int j = 0; j < b; ++j)
      if (states[j] == s) return PNB_E_INVAL;
    const int32_t nr = n_recent ? n_recent[b] : 0;
    const int32_t *rec = recent_dev ? recent_dev[b] : nullptr;
    if (nr < 0) return PNB_E_INVAL;
    if (nr > 0 && !rec) return PNB_E_NULL;
    if (rec && (reinterpret_cast<uintptr_t>(rec) & 3u)) return PNB_E_ALIGN;
    if (std::isnan(p.temperature) || std::isinf(p.temperature) || !(p.repeat_penalty > 0.0f) ||
        std::isinf(p.repeat_penalty) || std::isnan(p.top_p))
      return PNB_E_INVAL;
    a.slot[b] = SampleSlot{logits_dev + (size_t)b * V, rec, nr, p.top_k, p.temperature,
                           p.repeat_penalty, p.top_p, (unsigned long long)p.seed, s->io,
                           tokens_dev ? tokens_dev + b : nullptr};
  }
  if (!m->sample_ok) return PNB_E_UNSUPPORTED;
  int rc = check_device(m);
  if (rc != PNB_OK) return rc;
  return launch_sample(a, B, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? PNB_OK
                                                                                    : PNB_E_CUDA;
}

int pnb_sample(pnb_model *m, pnb_state *s, float *logits_dev, const pnb_sampling_params *params,
               const int32_t *recent_dev, int32_t n_recent, pnb_stream stream, int32_t *token_dev) {
  return pnb_sample_batch(m, &s, 1, logits_dev, params, &recent_dev, &n_recent, stream, token_dev);
}

int pnb_state_set_draw(pnb_state *s, uint32_t draw, pnb_stream stream) {
  if (!s) return PNB_E_NULL;
  int rc = check_device(s->m);
  if (rc != PNB_OK) return rc;
  return launch_set_draws(s->io, draw, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? PNB_OK
             : PNB_E_CUDA;
}

namespace {
int async_setup(pnb_state *s) {
  if (!s->astream && cudaStreamCreateWithFlags(&s->astream, cudaStreamNonBlocking) != cudaSuccess) {
    s->astream = nullptr;
    return PNB_E_CUDA;
  }
  if (!s->aevent && cudaEventCreateWithFlags(&s->aevent, cudaEventDisableTiming) != cudaSuccess) {
    s->aevent = nullptr;
    return PNB_E_CUDA;
  }
  return PNB_OK;
}
}  // namespace

int pnb_state_stream(pnb_state *s, pnb_stream *out) {
  if (!s || !out) return PNB_E_NULL;
  int rc = check_device(s->m);
  if (rc == PNB_OK) rc = async_setup(s);
  if (rc != PNB_OK) return rc;
  *out = reinterpret_cast<pnb_stream>(s->astream);
  return PNB_OK;
}

int pnb_forward_begin(pnb_model *m, pnb_state *s, int32_t token, float *logits_dev,
                      int32_t *argmax_dev) {
  if (!m || !s) return PNB_E_NULL;
  if (s->m != m) return PNB_E_INVAL;
  if (s->pending) return PNB_E_BUSY;
  int rc = check_device(m);
  if (rc == PNB_OK) rc = async_setup(s);
  if (rc != PNB_OK) return rc;
  rc = pnb_forward(m, s, token, reinterpret_cast<pnb_stream>(s->astream), logits_dev, argmax_dev);
  if (rc != PNB_OK) return rc;
  if (cudaEventRecord(s->aevent, s->astream) != cudaSuccess) return PNB_E_CUDA;
  s->pending = true;
  s->a_logits = logits_dev;
  return PNB_OK;
}

int pnb_sample_begin(pnb_model *m, pnb_state *s, float *logits_dev,
                     const pnb_sampling_params *params, const int32_t *recent_dev,
                     int32_t n_recent, int32_t *token_dev) {
  if (!m || !s) return PNB_E_NULL;
  if (s->m != m) return PNB_E_INVAL;
  int rc = check_device(m);
  if (rc == PNB_OK) rc = async_setup(s);
  if (rc != PNB_OK) return rc;
  rc = pnb_sample(m, s, logits_dev, params, recent_dev, n_recent,
                  reinterpret_cast<pnb_stream>(s->astream), token_dev);
  if (rc != PNB_OK) return rc;
  if (cudaEventRecord(s->aevent, s->astream) != cudaSuccess) return PNB_E_CUDA;
  if (!s->pending) s->a_logits = logits_dev;
  s->pending = true;
  return PNB_OK;
}

int pnb_forward_poll(pnb_model *m, pnb_state *s, float **logits_out) {
  if (!m || !s) return PNB_E_NULL;
  if (s->m != m || !s->pending) return PNB_E_INVAL;
  const cudaError_t q = cudaEventQuery(s->aevent);
  if (q == cudaErrorNotReady) return 1;
  s->pending = false;
  if (q != cudaSuccess) return PNB_E_CUDA;
  StepIO io;
  if (cudaMemcpyAsync(&io, s->io, sizeof(io), cudaMemcpyDeviceToHost, s->astream) != cudaSuccess ||
      cudaStreamSynchronize(s->astream) != cudaSuccess)
    return PNB_E_CUDA;
  if (io.error) return PNB_E_DEVICE;
  if (logits_out) *logits_out = s->a_logits;
  return PNB_OK;
}

int pnb_prefill(pnb_model *m, pnb_state *s, const int32_t *tokens_dev, int32_t T, pnb_stream stream,
                float *logits_dev, int32_t *argmax_dev) {
  if (!m || !s || !tokens_dev) return PNB_E_NULL;
  if (s->m != m || T < 1) return PNB_E_INVAL;
  if ((logits_dev && !aligned16(logits_dev)) ||
      (argmax_dev && (reinterpret_cast<uintptr_t>(argmax_dev) & 3u)) ||
      (reinterpret_cast<uintptr_t>(tokens_dev) & 3u))
    return PNB_E_ALIGN;
  const pnb_config &c = m->cfg;
  if ((int64_t)s->pos + T > c.n_ctx) return PNB_E_CTX_FULL;
  int rc = check_device(m);
  if (rc != PNB_OK) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const bool batched = c.dtype == PNB_BF16 && c.n_embd % 64 == 0 &&
                       (c.n_head * m->hd) % 64 == 0 && c.n_ff % 64 == 0;
  if (batched && (rc = batch_setup(m)) != PNB_OK) return rc;
  const bool ring = c.sliding_window > 0 && m->cap < c.n_ctx;
  const size_t V = (size_t)c.n_vocab;
  for (int i = 0; i < T;) {
    int n = std::min(kMaxChunk, T - i);
    // a ring cache must not wrap inside a chunk: a later chunk position would
    // overwrite a slot inside an earlier chunk token's window
    if (ring) n = s->pos >= m->cap ? 1 : std::min(n, m->cap - s->pos);
    float *lg = logits_dev ? logits_dev + (size_t)i * V : nullptr;
    int32_t *am = argmax_dev ? argmax_dev + i : nullptr;
    if (n == 1 || !batched) {
      // one token: the single-sequence step (launched directly, not as a graph)
      n = 1;
      if (launch_copy_token(s->io, tokens_dev + i, st) != cudaSuccess ||
          enqueue_step(m, s, st, lg, am) != cudaSuccess)
        return PNB_E_CUDA;
    } else {
      BatchCtx *b = m->batch;
      BSlot slots[kMaxChunk];
      for (int j = 0; j < n; ++j) slots[j] = BSlot{s->kv, &b->pio[j], s->maps};
      if (launch_prefill_begin(b->pio, s->io, n, st) != cudaSuccess ||
          enqueue_batch(m, slots, n, tokens_dev + i, nullptr, st, lg, am,
                        s->pos + n <= kChunkAttnMaxPos ? kChunkKernel
                                                       : (m->attn_tc ? kChunkGroups : kChunkSlots)) !=
              cudaSuccess ||
          launch_prefill_end(s->io, b->pio, n, st) != cudaSuccess)
        return PNB_E_CUDA;
    }
    s->pos += n;
    i += n;
  }
  return PNB_OK;
}

int pnb_model_set_tensor_attention(pnb_model *m, int enable) {
  if (!m) return PNB_E_NULL;
  if (enable && !m->attn_tc_ok) return PNB_E_UNSUPPORTED;
  ++m->mode_gen;
  m->attn_tc = enable != 0;
  return PNB_OK;
}

int pnb_model_is_tensor_attention(const pnb_model *m) { return m && m->attn_tc ? 1 : 0; }

int pnb_model_set_graphs(pnb_model *m, int enable) {
  if (!m) return PNB_E_NULL;
  ++m->mode_gen;
  m->graphs = enable != 0;
  return PNB_OK;
}

int pnb_model_set_deterministic_batch(pnb_model *m, int enable) {
  if (!m) return PNB_E_NULL;
  ++m->mode_gen;
  m->det_batch = enable != 0;
  return PNB_OK;
}

int pnb_step_kernel_count(const pnb_model *m, int32_t B) {
  if (!m) return PNB_E_NULL;
  if (B == 1) return pnb_step_kernel_count(m, 0) + 1;   // token copy + the single-sequence step
  if (B > 1) {
    // batched: norm, QKV (+ merge of its K parts), attention, o, norm, gate/up
    // (+ merge), down per layer; final norm and LM head
    // (MoE: the router, then gate/up (+ merge) and down per expert)
    const int qmerge = plan_bgemm(m->qkv_rows, m->cfg.n_embd, m->num_sms).ksplit > 1;
    const int fmerge = plan_bgemm(2 * (int64_t)m->cfg.n_ff, m->cfg.n_embd, m->num_sms).ksplit > 1;
    const int ffn = m->n_sets * (2 + fmerge) + (m->cfg.expert_count > 0 ? 1 : 0);
    return m->cfg.n_layer * (5 + qmerge + ffn) + 2;
  }
  const int per_layer = 3 + (m->cfg.expert_count > 0 ? 3 : 2);
  return m->cfg.n_layer * per_layer + 1;
}

int pnb_step_kernel(pnb_model *m, pnb_state *s, int32_t kind, int32_t layer, pnb_stream stream) {
  if (!m || !s) return PNB_E_NULL;
  if (s->m != m) return PNB_E_INVAL;
  if (kind < PNB_KERNEL_QKV || kind > PNB_KERNEL_LM_HEAD) return PNB_E_INVAL;
  if (kind == PNB_KERNEL_ROUTER && m->cfg.expert_count == 0) return PNB_E_INVAL;
  if (layer < 0 || layer >= m->cfg.n_layer) return PNB_E_INVAL;
  int rc = check_device(m);
  if (rc != PNB_OK) return rc;
  if (enqueue_kernel(m, s, kind, layer, reinterpret_cast<cudaStream_t>(stream), false, nullptr,
                     nullptr) != cudaSuccess)
    return PNB_E_CUDA;
  return PNB_OK;
}

int pnb_state_set_trace(pnb_state *s, uint64_t *trace_dev, size_t bytes) {
  if (!s) return PNB_E_NULL;
  if (trace_dev) {
    const int L = s->m->cfg.n_layer;
    const size_t need = (size_t)(7 * L + 2) * kTraceCtas * 8 * 8;
    if (bytes < need) return PNB_E_INVAL;
    if (reinterpret_cast<uintptr_t>(trace_dev) & 7u) return PNB_E_ALIGN;
  }
  s->ktrace = reinterpret_cast<unsigned long long *>(trace_dev);
  if (s->exec) {   // the captured graph holds the old argument
    cudaGraphExecDestroy(s->exec);
    s->exec = nullptr;
  }
  return PNB_OK;
}

int pnb_state_wait_probe(pnb_state *s, uint64_t limit_ns, pnb_stream stream) {
  if (!s) return PNB_E_NULL;
  if (limit_ns > 1000000000ull) return PNB_E_INVAL;
  int rc = check_device(s->m);
  if (rc != PNB_OK) return rc;
  // the copy reads the state's own residual buffer (n_embd fp32, a multiple of 32 bytes)
  const uint32_t bytes = (uint32_t)std::min<size_t>((size_t)s->m->cfg.n_embd * 4, kWaitProbeBytes);
  if (launch_wait_probe(s->x, bytes, limit_ns, s->io, reinterpret_cast<cudaStream_t>(stream)) !=
      cudaSuccess)
    return PNB_E_CUDA;
  return PNB_OK;
}

int pnb_state_activations(const pnb_state *s, pnb_activations *out) {
  if (!s || !out) return PNB_E_NULL;
  out->x = s->x;
  out->q = s->q;
  out->attn = s->attn;
  out->h = s->h;
  return PNB_OK;
}

}  // extern "C"
