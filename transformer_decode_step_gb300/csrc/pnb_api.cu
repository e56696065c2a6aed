// pnb_api.cu - the C ABI (include/pnb.h): validation, geometry planning,
// workspace, the per-step launch sequence and its CUDA-graph capture.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <new>
#include <vector>

#include "pnb.h"
#include "pnb_kernels.cuh"
#include "pnb_step.cuh"

using namespace pnb;

namespace {

constexpr int kStageTarget = 32 * 1024;   // bytes of whole rows per GEMV ring slot
constexpr int kRingBudget = 192 * 1024;   // bytes of GEMV ring per CTA
constexpr int kMaxSmem = 227 * 1024;
constexpr int kMaxBatch = 64;
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
Geom plan_gemv(int K, int es, int64_t rows_total, int row_align, int nsum, int grid, int nseg) {
  Geom g{};
  g.K = K;
  g.es = es;
  g.row_bytes = K * es;
  int rps = 1;
  while (rps * 2 <= 64 && rps * 2 * g.row_bytes <= kStageTarget) rps *= 2;
  rps = std::max(rps, row_align);   // row pairs never straddle two ring items
  g.rows_per_stage = rps;
  g.stage_bytes = rps * g.row_bytes;
  // warps per row: enough that a lane holds at most 4 column vectors, and no
  // more row groups than rows per ring slot
  const int vpr = g.row_bytes / 16;
  int cw = 1;
  while (cw < kGemvWarps && (cw * 32 * 4 < vpr || kGemvWarps / cw > rps)) cw *= 2;
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
  g.nstages = std::min(8, std::max(2, ring / g.stage_bytes));
  g.inflight = std::max(1, std::min(g.nstages, ceil_div(kInflightBytes, g.stage_bytes)));
  return g;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t align256(size_t v) { return (v + 255) / 256 * 256; }

}  // namespace

struct pnb_model {
  pnb_config cfg;
  int device = 0, num_sms = 0, grid = 0;
  int hd = 0, n_sets = 0, qkv_rows = 0, es = 0, cap = 0;
  const void *tok_embd = nullptr;
  const float *out_norm = nullptr;
  const void *output = nullptr;
  std::vector<const float *> attn_norm, ffn_norm;
  std::vector<const void *> wqkv, wo, w_router, w_gate_up, w_down;
  double *inv_freq = nullptr;            // device [hd/2]
  const void **tab_gate_up = nullptr;    // device [n_layer][expert_count]
  const void **tab_down = nullptr;
  Geom g_qkv{}, g_o{}, g_gateup{}, g_down{}, g_lm{};
  AttnGeom ag{};
  int n_split = 1, zgroups = 1;
  bool graphs = true;
  // persistent step kernel
  bool persistent = false;
  int st_nslots = 0, st_slot_bytes = 0, st_sp = 0, st_union = 0, st_smem = 0;
  cudaStream_t cap_stream = nullptr;     // stream used for graph capture
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
  unsigned *bar_count = nullptr, *bar_gen = nullptr;
  int32_t *abort_flag = nullptr;
  unsigned *work = nullptr;              // [launch][claim, done] item counters
  float *step_part = nullptr;            // attention partials of the persistent kernel
  float *ss_part = nullptr;              // per-CTA sums of squares [2][grid]
  StepLayer *layers = nullptr;           // device [n_layer]
  unsigned long long *trace = nullptr;   // optional phase timestamps (persistent kernel)
  unsigned long long *ktrace = nullptr;  // optional per-CTA timestamps (per-phase kernels)
  cudaGraphExec_t exec = nullptr;
  float *g_logits = nullptr;
  int32_t *g_argmax = nullptr;
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
  const int hd = c->n_embd / c->n_head;
  if (hd % 2) return PNB_E_INVAL;
  if (hd != 32 && hd != 64 && hd != 128) return PNB_E_UNSUPPORTED;
  if (c->n_embd % 8 || c->n_ff % 8) return PNB_E_INVAL;
  if (c->sliding_window < 0 || !(c->rope_theta > 0.0) || !(c->rms_norm_eps >= 0.0)) return PNB_E_INVAL;
  if (c->dtype != PNB_F32 && c->dtype != PNB_BF16) return PNB_E_INVAL;
  if (c->expert_count < 0 || c->expert_count > 64) return PNB_E_INVAL;
  if (c->expert_count > 0 &&
      (c->expert_used <= 0 || c->expert_used > c->expert_count || c->expert_used > kMaxSegments))
    return PNB_E_INVAL;
  return PNB_OK;
}

void plan(pnb_model *m) {
  const pnb_config &c = m->cfg;
  const int E = c.n_embd, F = c.n_ff, es = m->es, grid = m->grid;
  const int k = c.expert_count > 0 ? c.expert_used : 1;
  m->g_qkv = plan_gemv(E, es, m->qkv_rows, 2, 1, grid, 1);
  m->g_o = plan_gemv(c.n_head * m->hd, es, E, 1, 1, grid, 1);
  m->g_gateup = plan_gemv(E, es, (int64_t)k * 2 * F, 2, 1, grid, k);
  m->g_down = plan_gemv(F, es, E, 1, k, grid, c.expert_count > 0 ? 0 : 1);
  m->g_lm = plan_gemv(E, es, c.n_vocab, 1, 1, grid, 1);
  const int G = c.n_head / c.n_kv_head;
  m->ag = attn_geom(c.dtype, m->hd, G);
  m->zgroups = G / m->ag.heads_per_cta;
  // one wave: at most one CTA per SM (the attention CTA's registers allow one)
  const int want = std::max(1, m->num_sms / (c.n_kv_head * m->zgroups));
  m->n_split = std::max(1, std::min(want, std::max(1, m->cap / 16)));
}

bool geoms_supported(const pnb_model *m);

// Persistent-kernel geometry: one ring slot holds the largest GEMV stage or a
// 2 x sp x head_dim KV stage; the scratch union holds the largest per-CTA
// partial array or the attention merge area.
void plan_step(pnb_model *m) {
  const pnb_config &c = m->cfg;
  const int G = c.n_head / c.n_kv_head, hd = m->hd, es = m->es;
  m->persistent = false;
  if (!(hd == 32 || hd == 64 || hd == 128) || !(G == 1 || G == 2 || G == 4 || G == 8) ||
      G * hd > 512)
    return;
  int slot = 0, uni = 0;
  for (const Geom *g : {&m->g_qkv, &m->g_o, &m->g_gateup, &m->g_down, &m->g_lm}) {
    slot = std::max(slot, g->stage_bytes);
    uni = std::max(uni, g->rows_cta_max * g->cw * g->nsum);
  }
  slot = std::max(slot, 2 * 32 * hd * es);
  int sp = slot / (2 * hd * es);
  sp = std::min(256, sp - sp % 32);
  uni = std::max(uni, kGemvWarps * G * (hd + 2));
  const int fixed = step_smem(1, slot, uni).total - slot;
  int ns = std::min(kRingBudget / slot, (kMaxSmem - fixed - 1024) / slot);
  if (ns < 2) return;
  ns = std::min(ns, 8);
  m->st_nslots = ns;
  m->st_slot_bytes = slot;
  m->st_sp = sp;
  m->st_union = uni;
  m->st_smem = step_smem(ns, slot, uni).total;
  if (m->st_smem > kMaxSmem || !geoms_supported(m)) return;
  StepArgs dummy{};
  int bps = 0;
  cudaError_t e = (c.dtype ? step_bf16 : step_f32)(hd, G, dummy, m->grid, m->st_smem, nullptr, true, &bps);
  m->persistent = e == cudaSuccess && bps >= 1;
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
  const size_t layer_kv = (size_t)Hkv * m->cap * hd * m->es;
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
      return launch_attn(c.dtype, hd, aa, m->ag, st, pdl);
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

// The persistent kernel's arguments for state s.
StepArgs step_args(const pnb_model *m, const pnb_state *s, float *logits, int32_t *argmax) {
  const pnb_config &c = m->cfg;
  StepArgs a{};
  a.E = c.n_embd;
  a.H = c.n_head;
  a.Hkv = c.n_kv_head;
  a.hd = m->hd;
  a.F = c.n_ff;
  a.V = c.n_vocab;
  a.L = c.n_layer;
  a.X = c.expert_count;
  a.k = c.expert_count > 0 ? c.expert_used : 1;
  a.cap = m->cap;
  a.window = c.sliding_window;
  a.eps = (float)c.rms_norm_eps;
  a.qscale = (float)(1.4426950408889634 / std::sqrt((double)m->hd));
  a.g_qkv = m->g_qkv;
  a.g_o = m->g_o;
  a.g_gu = m->g_gateup;
  a.g_dn = m->g_down;
  a.g_lm = m->g_lm;
  a.nslots = m->st_nslots;
  a.slot_bytes = m->st_slot_bytes;
  a.sp = m->st_sp;
  a.union_floats = m->st_union;
  a.tok_embd = m->tok_embd;
  a.output = m->output;
  a.out_norm = m->out_norm;
  a.inv_freq = m->inv_freq;
  a.layers = s->layers;
  a.x = s->x;
  a.q = s->q;
  a.o = s->attn;
  a.h = s->h;
  a.attn_part = s->step_part;
  a.lm_val = s->lm_val;
  a.lm_idx = s->lm_idx;
  a.attn_cnt = s->attn_cnt;
  a.lm_cnt = s->lm_cnt;
  a.bar_count = s->bar_count;
  a.bar_gen = s->bar_gen;
  a.abort_flag = s->abort_flag;
  a.ss_part = s->ss_part;
  a.logits = logits;
  a.argmax_out = argmax;
  a.io = s->io;
  a.trace = s->trace;
  return a;
}

// Enqueue one single-sequence step (everything after the token write): the
// persistent kernel when the model supports it, else one kernel per phase
// (the first waits for all earlier stream work; every later one is launched
// with programmatic stream serialization).
cudaError_t enqueue_step(pnb_model *m, pnb_state *s, cudaStream_t st, float *logits,
                         int32_t *argmax) {
  if (m->persistent) {
    const StepArgs a = step_args(m, s, logits, argmax);
    const int G = m->cfg.n_head / m->cfg.n_kv_head;
    return (m->cfg.dtype ? step_bf16 : step_f32)(m->hd, G, a, m->grid, m->st_smem, st, false, nullptr);
  }
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
  }
  pnb_model *m = new (std::nothrow) pnb_model();
  if (!m) return PNB_E_NOMEM;
  try {
    m->cfg = c;
    m->hd = c.n_embd / c.n_head;
    m->n_sets = n_sets;
    m->qkv_rows = (c.n_head + 2 * c.n_kv_head) * m->hd;
    m->es = c.dtype == PNB_BF16 ? 2 : 4;
    m->cap = c.sliding_window > 0 ? std::min(c.sliding_window, c.n_ctx) : c.n_ctx;
    m->tok_embd = w->tok_embd;
    m->out_norm = w->out_norm;
    m->output = w->output;
    m->attn_norm.assign(w->attn_norm, w->attn_norm + c.n_layer);
    m->ffn_norm.assign(w->ffn_norm, w->ffn_norm + c.n_layer);
    m->wqkv.assign(w->wqkv, w->wqkv + c.n_layer);
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
               prepare_attn_kernel(c.dtype, m->hd, m->ag) == cudaSuccess;
  // one kernel per phase is the default: on the 7B-class shapes it is the
  // faster of the two; the persistent kernel is opt-in
  if (ok) {
    plan_step(m);
    m->persistent = false;
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
  delete m;
}

size_t pnb_state_kv_bytes(const pnb_model *m) {
  if (!m) return 0;
  return (size_t)m->cfg.n_layer * 2 * m->cfg.n_kv_head * m->cap * m->hd * m->es;
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
  const size_t o_part = take((size_t)c.n_head * m->n_split * (m->hd + 2) * 4);
  const size_t o_gate = take((size_t)k * 4);
  const size_t o_idx = take((size_t)k * 4);
  const size_t o_lmv = take((size_t)m->grid * 4);
  const size_t o_lmi = take((size_t)m->grid * 4);
  const size_t n_cnt = (size_t)(c.n_kv_head * m->zgroups + 1 + 3) + 2 * (6 * c.n_layer + 1);
  const size_t o_cnt = take(n_cnt * 4);
  const size_t o_spart = take((size_t)c.n_head * m->grid * (m->hd + 2) * 4);
  const size_t o_layers = take((size_t)c.n_layer * sizeof(StepLayer));
  const size_t o_ss = take((size_t)2 * m->grid * 4);
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
  s->bar_count = s->lm_cnt + 1;
  s->bar_gen = s->lm_cnt + 2;
  s->abort_flag = reinterpret_cast<int32_t *>(s->lm_cnt + 3);
  s->work = s->lm_cnt + 4;
  s->counters_off = o_cnt;
  s->counters_bytes = n_cnt * 4;
  s->step_part = reinterpret_cast<float *>(s->ws + o_spart);
  s->layers = reinterpret_cast<StepLayer *>(s->ws + o_layers);
  s->ss_part = reinterpret_cast<float *>(s->ws + o_ss);
  // per-layer table of the persistent kernel
  std::vector<StepLayer> lt(c.n_layer);
  const size_t layer_kv = (size_t)c.n_kv_head * m->cap * m->hd * m->es;
  for (int l = 0; l < c.n_layer; ++l) {
    StepLayer &L = lt[l];
    L.wqkv = m->wqkv[l];
    L.wo = m->wo[l];
    L.attn_norm = m->attn_norm[l];
    L.ffn_norm = m->ffn_norm[l];
    if (c.expert_count > 0) {
      L.w_router = m->w_router[l];
      L.tab_gate_up = m->tab_gate_up + (size_t)l * c.expert_count;
      L.tab_down = m->tab_down + (size_t)l * c.expert_count;
    } else {
      L.w_gate_up = m->w_gate_up[l];
      L.w_down = m->w_down[l];
    }
    L.kc = s->kv + (size_t)(2 * l) * layer_kv;
    L.vc = s->kv + (size_t)(2 * l + 1) * layer_kv;
  }
  if (cudaMemset(s->ws, 0, off) != cudaSuccess ||
      cudaMemcpy(s->layers, lt.data(), lt.size() * sizeof(StepLayer), cudaMemcpyHostToDevice) !=
          cudaSuccess) {
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
    if (!s->exec || s->g_logits != logits_dev || s->g_argmax != argmax_dev) {
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
    }
    if (cudaGraphLaunch(s->exec, st) != cudaSuccess) return PNB_E_CUDA;
  }
  s->pos += 1;
  return PNB_OK;
}

int pnb_forward_batch(pnb_model *m, pnb_state *const *states, int32_t B, const int32_t *tokens_dev,
                      pnb_stream stream, float *logits_dev, int32_t *argmax_dev) {
  (void)tokens_dev;
  (void)stream;
  (void)logits_dev;
  (void)argmax_dev;
  if (!m || !states) return PNB_E_NULL;
  if (B < 1 || B > kMaxBatch) return PNB_E_INVAL;
  if (m->cfg.expert_count > 0) return PNB_E_UNSUPPORTED;
  return PNB_E_UNSUPPORTED;
}

int pnb_model_set_persistent(pnb_model *m, int enable) {
  if (!m) return PNB_E_NULL;
  if (!enable) {
    m->persistent = false;
    return PNB_OK;
  }
  plan_step(m);
  return m->persistent ? PNB_OK : PNB_E_UNSUPPORTED;
}

int pnb_model_is_persistent(const pnb_model *m) { return m && m->persistent ? 1 : 0; }

int pnb_model_set_graphs(pnb_model *m, int enable) {
  if (!m) return PNB_E_NULL;
  m->graphs = enable != 0;
  return PNB_OK;
}

int pnb_step_kernel_count(const pnb_model *m, int32_t B) {
  if (!m) return PNB_E_NULL;
  (void)B;
  if (m->persistent) return 1;
  const int per_layer = m->cfg.expert_count > 0 ? 6 : 5;
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
    const size_t need = std::max((size_t)s->m->grid * (5 * L + 1) * 6 * 8,
                                 (size_t)(6 * L + 1) * kTraceCtas * 8 * 8);
    if (bytes < need) return PNB_E_INVAL;
    if (reinterpret_cast<uintptr_t>(trace_dev) & 7u) return PNB_E_ALIGN;
  }
  s->trace = reinterpret_cast<unsigned long long *>(trace_dev);
  s->ktrace = s->trace;
  if (s->exec) {   // the captured graph holds the old argument
    cudaGraphExecDestroy(s->exec);
    s->exec = nullptr;
  }
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
