/*
 * oracle.c - plain, slow CPU forward of the Llama-family transformer decode step.
 *
 * TEST INFRASTRUCTURE.  This file is the correctness reference for the GPU
 * library.  Only the test suite, the smoke check and the CPU-baseline leg of
 * the benchmark may load it.  It shares no code with the GPU path; the only
 * thing both sides use is the seeded input generator (synth/synth.h).
 *
 * What it computes follows the Pantheon engine pages:
 *  - the decode seam: one call takes one token and the state (KV cache, pos)
 *    and returns fp32 logits over the vocabulary, advancing pos by one
 *    ("Core Engine API", section "pn_model struct": forward is
 *    tm_tensor* (*)(pn_model*, uint32_t token, pn_state*));
 *  - one forward shared by Llama, Qwen2, Mistral and Mixtral, with the
 *    differences carried by config fields: n_kv_head (grouped-query heads),
 *    rope_theta, rms_norm_eps, sliding_window (0 = off) and expert_count > 0
 *    for the MoE FFN ("Engine Architecture", sections "Architecture
 *    Detection" and "Config Parsing");
 *  - the per-layer buffers of the arena budget (5*n_embd + 3*n_ff +
 *    2*n_kv_head*head_dim floats; MoE adds n_experts + 2*n_experts_used)
 *    name the intermediates computed below ("Core Engine API", section
 *    "Scratch (arena) estimation");
 *  - greedy sampling is argmax ("Engine Architecture", section "Sampling",
 *    temperature 0); the prompt is fed one token per forward
 *    ("Engine Architecture", section "Generation Loop").
 * The pages do not write out the layer math (the linked Llama forward page is
 * missing), so the layer is the standard pre-norm Llama decoder; each reading
 * the pages leave open is named at the function that makes it.
 *
 * Precision: the pages' engine keeps every buffer in fp32 ("Engine
 * Architecture", section "Weight Loading Modes": F32 tensors).  The oracle
 * does the same: every intermediate vector is stored as fp32, while every
 * reduction (dot product, sum of squares, softmax sum) is accumulated in fp64
 * and rounded once to fp32.  Weights and the KV cache hold their storage type
 * (fp32, or bf16 values widened exactly to fp32; Q8 weights are their
 * block's fp16 scale times the int8 value, the dequantization of a GGUF
 * Q8_0 block, and Q4 weights the scale times the 4-bit code less 8, that of
 * a GGUF Q4_0 block: "Engine Architecture", "Weight Loading Modes",
 * quantized mode, per-block dequantization inside the matvec - exact in
 * fp32).  New K/V
 * entries are rounded fp32 -> bf16 (nearest even) before they are stored when the cache
 * is bf16; the argmax is taken over the fp32 logits, lowest id on ties.
 */
#include <math.h>
#include <omp.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include "../synth/synth.h"

/* ------------------------------------------------------------------ types */

typedef struct {
  int32_t n_vocab, n_embd, n_head, n_kv_head, n_layer, n_ff, n_ctx;
  double rope_theta, rms_norm_eps;
  int32_t sliding_window; /* 0 = no window */
  int32_t expert_count;   /* 0 = dense FFN */
  int32_t expert_used;    /* top-k */
  int32_t dtype;          /* storage of weights: 0 fp32, 1 bf16, 2 Q8 (blocks of 32: int8
                             values times an fp16 scale), 3 Q4 (blocks of 32: 4-bit codes
                             less 8 times an fp16 scale); KV: fp32 for 0, bf16 otherwise */
  int32_t qkv_bias;       /* 1: bias vectors added to q, k, v (Qwen2) */
  int32_t rope_neox;      /* 1: RoPE pairs dimension i with i + hd/2 (Phi-3) */
} orc_config;

enum { ORC_EXPLICIT = 0, ORC_SYNTH = 1, ORC_CONST = 2 };

/* one logical tensor (row-major logical shape) */
typedef struct {
  int32_t mode;
  int32_t pad_;
  const float *data; /* ORC_EXPLICIT: storage values as fp32, row-major */
  uint64_t key;      /* ORC_SYNTH: generator stream key */
  float sigma;       /* ORC_SYNTH: standard deviation */
  float value;       /* ORC_CONST: every element */
} orc_tensor;

/* per-layer tensor slots; experts follow as (gate, up, down) triples, then
   the q, k and v bias vectors (fp32; used when qkv_bias is set) */
enum {
  ORC_L_ATTN_NORM = 0,
  ORC_L_WQ = 1,
  ORC_L_WK = 2,
  ORC_L_WV = 3,
  ORC_L_WO = 4,
  ORC_L_FFN_NORM = 5,
  ORC_L_WROUTER = 6,
  ORC_L_EXPERT0 = 7
};
/* global slots */
enum { ORC_G_TOK_EMBD = 0, ORC_G_OUT_NORM = 1, ORC_G_OUTPUT = 2 };

typedef struct {
  orc_config cfg;
  int32_t head_dim, n_ffn_sets; /* n_ffn_sets = max(1, expert_count) */
  orc_tensor glob[3];
  orc_tensor *layer; /* n_layer * (7 + 3*n_ffn_sets) */
} orc_model;

typedef struct {
  const orc_model *m;
  int64_t pos;
  float *k; /* [n_layer][n_ctx][n_kv_head][head_dim] */
  float *v;
  /* diagnostic, not arithmetic: over the MoE layers of the last forward, the
     smallest gap between the k-th chosen router logit and the best unchosen
     one, relative to the layer's largest |logit| (INFINITY for dense models) */
  double route_margin;
} orc_state;

/* ------------------------------------------------------------- helpers */

/* fp32 -> bf16 -> fp32, round to nearest even on the bit pattern */
float orc_round_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7F800000u) == 0x7F800000u) { /* inf / nan pass through */
    u &= 0xFFFF0000u;
    if (f != f) u |= 0x00400000u;
  } else {
    u += 0x7FFFu + ((u >> 16) & 1u);
    u &= 0xFFFF0000u;
  }
  float r;
  memcpy(&r, &u, 4);
  return r;
}

static int64_t layer_slots(const orc_model *m) { return 7 + 3 * (int64_t)m->n_ffn_sets + 3; }
static int bias_slot(const orc_model *m, int which) { return 7 + 3 * m->n_ffn_sets + which; }

static const orc_tensor *ltensor(const orc_model *m, int l, int slot) {
  return &m->layer[(int64_t)l * layer_slots(m) + slot];
}

/* row r of a [rows][cols] tensor, as fp32 storage values */
static void get_row(const orc_tensor *t, int64_t r, int64_t cols, int dtype, float *out) {
  if (t->mode == ORC_EXPLICIT) {
    memcpy(out, t->data + r * cols, (size_t)cols * sizeof(float));
  } else if (t->mode == ORC_SYNTH && dtype == SYNTH_Q8) {
    /* Q8 weights: per block of 32, the weight is the block's fp16 scale
       times the element's int8 value (GGUF Q8_0 dequantization) */
    const uint64_t base = (uint64_t)(r * cols);
    for (int64_t b = 0; b + SYNTH_Q8_BLOCK <= cols; b += SYNTH_Q8_BLOCK) {
      int8_t q[SYNTH_Q8_BLOCK];
      uint16_t d;
      synth_q8_block(t->key, base + (uint64_t)b, t->sigma, q, &d);
      const float df = synth_f16_to_f32(d);
      for (int j = 0; j < SYNTH_Q8_BLOCK; ++j) out[b + j] = df * (float)q[j];
    }
  } else if (t->mode == ORC_SYNTH && dtype == SYNTH_Q4) {
    /* Q4 weights: per block of 32, the weight is the block's fp16 scale
       times the element's 4-bit code less 8 (GGUF Q4_0 dequantization) */
    const uint64_t base = (uint64_t)(r * cols);
    for (int64_t b = 0; b + SYNTH_Q4_BLOCK <= cols; b += SYNTH_Q4_BLOCK) {
      uint8_t u[SYNTH_Q4_BLOCK];
      uint16_t d;
      synth_q4_block(t->key, base + (uint64_t)b, t->sigma, u, &d);
      const float df = synth_f16_to_f32(d);
      for (int j = 0; j < SYNTH_Q4_BLOCK; ++j) out[b + j] = df * (float)((int)u[j] - 8);
    }
  } else if (t->mode == ORC_SYNTH) {
    const uint64_t base = (uint64_t)(r * cols);
    for (int64_t c = 0; c < cols; ++c) out[c] = synth_value(t->key, base + (uint64_t)c, t->sigma, dtype);
  } else {
    for (int64_t c = 0; c < cols; ++c) out[c] = t->value;
  }
}

/* --------------------------------------------------- building blocks */

void orc_set_threads(int n) {
  if (n > 0) omp_set_num_threads(n);
}
int orc_max_threads(void) { return omp_get_max_threads(); }

/* y = W x for W [rows][cols]: fp64 dot product per row, rounded to fp32 */
void orc_matvec(const orc_tensor *w, int64_t rows, int64_t cols, int dtype, const float *x,
                float *y) {
#pragma omp parallel
  {
    float *row = (float *)malloc((size_t)cols * sizeof(float));
#pragma omp for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
      get_row(w, r, cols, dtype, row);
      double acc = 0.0;
      for (int64_t c = 0; c < cols; ++c) acc += (double)row[c] * (double)x[c];
      y[r] = (float)acc;
    }
    free(row);
  }
}

/* RMSNorm: out_i = x_i / sqrt(mean(x^2) + eps) * w_i.
   Reading: eps is added inside the square root and the weight multiplies after
   normalising (rms_norm_eps, default 1e-5: "Engine Architecture", "Config Parsing"). */
void orc_rmsnorm(const float *x, const float *w, int64_t n, double eps, float *out) {
  double ss = 0.0;
  for (int64_t i = 0; i < n; ++i) ss += (double)x[i] * (double)x[i];
  const double inv = 1.0 / sqrt(ss / (double)n + eps);
  for (int64_t i = 0; i < n; ++i) out[i] = (float)((double)x[i] * inv * (double)w[i]);
}

/* RoPE on one head vector of length hd at position pos, in place.
   Reading: the Llama path rotates adjacent pairs (2i, 2i+1); the NeoX-style
   half split belongs to the separate Phi-3 forward ("Engine Architecture",
   "Architecture Detection").  Pair i turns by pos * theta^(-2i/hd) with
   theta = rope_theta (default 10000, "Config Parsing"). */
void orc_rope(float *v, int hd, int64_t pos, double theta) {
  for (int i = 0; i < hd / 2; ++i) {
    const double freq = pow(theta, -2.0 * (double)i / (double)hd);
    const double phi = (double)pos * freq;
    const double c = cos(phi), s = sin(phi);
    const double a = v[2 * i], b = v[2 * i + 1];
    v[2 * i] = (float)(a * c - b * s);
    v[2 * i + 1] = (float)(a * s + b * c);
  }
}

/* NeoX-style RoPE (the Phi-3 forward, "Engine Architecture", "Architecture
   Detection"): pair i is dimensions (i, i + hd/2), turned by the same angle
   pos * theta^(-2i/hd) as adjacent pair i of the Llama form. */
void orc_rope_neox(float *v, int hd, int64_t pos, double theta) {
  const int h2 = hd / 2;
  for (int i = 0; i < h2; ++i) {
    const double freq = pow(theta, -2.0 * (double)i / (double)hd);
    const double phi = (double)pos * freq;
    const double c = cos(phi), s = sin(phi);
    const double a = v[i], b = v[i + h2];
    v[i] = (float)(a * c - b * s);
    v[i + h2] = (float)(a * s + b * c);
  }
}

/* Causal decode attention of all heads for the token at position p.
   K, V: [n_pos][n_kv][hd] (position-major), positions 0..p valid.
   Readings: query head h reads KV head h / (n_head / n_kv) (consecutive query
   heads share a KV head); with sliding_window W > 0 the token attends exactly
   the W positions p-W+1 .. p (sliding_window, 0 = disabled: "Config Parsing");
   scores are scaled by 1/sqrt(hd); softmax subtracts the maximum. */
void orc_attention(const float *q, const float *K, const float *V, int n_head, int n_kv, int hd,
                   int64_t p, int window, float *o) {
  const int group = n_head / n_kv;
  const int64_t lo = (window > 0 && p - window + 1 > 0) ? p - window + 1 : 0;
  const int64_t n = p - lo + 1;
  const double scale = 1.0 / sqrt((double)hd);
#pragma omp parallel
  {
    double *s = (double *)malloc((size_t)n * sizeof(double));
    double *acc = (double *)malloc((size_t)hd * sizeof(double));
#pragma omp for schedule(static)
    for (int h = 0; h < n_head; ++h) {
      const int g = h / group;
      const float *qh = q + (int64_t)h * hd;
      double mx = -INFINITY;
      for (int64_t j = 0; j < n; ++j) {
        const float *kj = K + ((lo + j) * n_kv + g) * hd;
        double d = 0.0;
        for (int t = 0; t < hd; ++t) d += (double)qh[t] * (double)kj[t];
        s[j] = d * scale;
        if (s[j] > mx) mx = s[j];
      }
      double z = 0.0;
      for (int64_t j = 0; j < n; ++j) {
        s[j] = exp(s[j] - mx);
        z += s[j];
      }
      for (int t = 0; t < hd; ++t) acc[t] = 0.0;
      for (int64_t j = 0; j < n; ++j) {
        const float *vj = V + ((lo + j) * n_kv + g) * hd;
        for (int t = 0; t < hd; ++t) acc[t] += s[j] * (double)vj[t];
      }
      for (int t = 0; t < hd; ++t) o[(int64_t)h * hd + t] = (float)(acc[t] / z);
    }
    free(s);
    free(acc);
  }
}

/* silu(z) = z / (1 + e^-z) */
double orc_silu(double z) { return z / (1.0 + exp(-z)); }

/* SwiGLU feed-forward: out = Wd (silu(Wg xn) * (Wu xn)); gate, up, act are fp32 vectors */
void orc_ffn(const orc_tensor *wg, const orc_tensor *wu, const orc_tensor *wd, int64_t n_embd,
             int64_t n_ff, int dtype, const float *xn, float *out) {
  float *gate = (float *)malloc((size_t)n_ff * sizeof(float));
  float *up = (float *)malloc((size_t)n_ff * sizeof(float));
  orc_matvec(wg, n_ff, n_embd, dtype, xn, gate);
  orc_matvec(wu, n_ff, n_embd, dtype, xn, up);
  for (int64_t i = 0; i < n_ff; ++i) gate[i] = (float)(orc_silu((double)gate[i]) * (double)up[i]);
  orc_matvec(wd, n_embd, n_ff, dtype, gate, out);
  free(gate);
  free(up);
}

/* MoE routing: pick the k largest router logits (lower expert index wins a
   tie) and softmax over the picked logits only (top-k router: expert_count > 0
   selects the MoE FFN, "Architecture Detection"; the arena reserves
   n_experts + 2*n_experts_used floats for it, "Scratch (arena) estimation"). */
void orc_topk_softmax(const float *r, int n_expert, int k, int32_t *idx, double *gate) {
  for (int i = 0; i < k; ++i) {
    int best = -1;
    for (int e = 0; e < n_expert; ++e) {
      int taken = 0;
      for (int j = 0; j < i; ++j) taken |= (idx[j] == e);
      if (taken) continue;
      if (best < 0 || r[e] > r[best]) best = e;
    }
    idx[i] = best;
  }
  double mx = -INFINITY, z = 0.0;
  for (int i = 0; i < k; ++i)
    if ((double)r[idx[i]] > mx) mx = (double)r[idx[i]];
  for (int i = 0; i < k; ++i) {
    gate[i] = exp((double)r[idx[i]] - mx);
    z += gate[i];
  }
  for (int i = 0; i < k; ++i) gate[i] /= z;
}

/* greedy pick: index of the largest value, lowest index on ties */
int32_t orc_argmax(const float *x, int64_t n) {
  int64_t best = 0;
  for (int64_t i = 1; i < n; ++i)
    if (x[i] > x[best]) best = i;
  return (int32_t)best;
}

/* Sampling ("Engine Architecture", "Sampling"): applied in the pages' order -
   (1) temperature: z = logit / T, T = 0 meaning the greedy argmax;
   (2) repetition penalty on the tokens of the recent window [READING: the
       pages name it only; each distinct recent token's z is divided by the
       penalty when positive and multiplied by it otherwise];
   (3) top-k: the k largest z, lower token id first on ties (k <= 0: all);
   (4) top-p: in that order, the tokens up to and including the first at
       which the cumulative probability exceeds p (p >= 1: all);
   (5) softmax over the kept tokens;
   (6) multinomial: the first kept token whose cumulative probability exceeds
       u times the kept total, u uniform in [0, 1).
   z, and so the order and the top-k set, are fp32, as the engine keeps its
   logits; a temperature <= 0 is greedy; probabilities and cumulative sums
   are fp64.  Returns the token;
   cand_idx / cand_cum (optional, n_vocab long) receive the kept tokens in
   draw order and their cumulative probabilities (normalised to the kept
   total), *n_cand their count. */
static int z_before(float za, int32_t a, float zb, int32_t b) { return za > zb || (za == zb && a < b); }

static int cmp_zi(const void *pa, const void *pb) {
  const float za = ((const float *)pa)[0], zb = ((const float *)pb)[0];
  int32_t a, b;
  memcpy(&a, (const float *)pa + 1, 4);
  memcpy(&b, (const float *)pb + 1, 4);
  return z_before(za, a, zb, b) ? -1 : (z_before(zb, b, za, a) ? 1 : 0);
}

int32_t orc_sample(const float *logits, int64_t V, float temperature, float repeat_penalty,
                   const int32_t *recent, int64_t n_recent, int64_t top_k, float top_p, double u,
                   int32_t *cand_idx, double *cand_cum, int64_t *n_cand) {
  if (temperature <= 0.0f) {
    if (n_cand) *n_cand = 0;
    return orc_argmax(logits, V);
  }
  float *z = (float *)malloc((size_t)V * sizeof(float));
  for (int64_t i = 0; i < V; ++i) z[i] = logits[i] / temperature;
  for (int64_t j = 0; j < n_recent; ++j) {
    const int32_t t = recent[j];
    int seen = 0;
    for (int64_t k = 0; k < j; ++k) seen |= recent[k] == t;
    if (seen || t < 0 || t >= V) continue;
    z[t] = z[t] > 0.0f ? z[t] / repeat_penalty : z[t] * repeat_penalty;
  }
  /* top-k: every token as a (z, id) pair in the draw order, then the first k */
  const int64_t k = (top_k <= 0 || top_k > V) ? V : top_k;
  float *pairs = (float *)malloc((size_t)V * 2 * sizeof(float));
  for (int64_t i = 0; i < V; ++i) {
    const int32_t id = (int32_t)i;
    pairs[2 * i] = z[i];
    memcpy(&pairs[2 * i + 1], &id, 4);
  }
  qsort(pairs, (size_t)V, 2 * sizeof(float), cmp_zi);
  float *kz = (float *)malloc((size_t)k * sizeof(float));
  int32_t *kid = (int32_t *)malloc((size_t)k * sizeof(int32_t));
  for (int64_t r = 0; r < k; ++r) {
    kz[r] = pairs[2 * r];
    memcpy(&kid[r], &pairs[2 * r + 1], 4);
  }
  free(pairs);
  /* softmax and cumulative probabilities in draw order (fp64) */
  double *cum = (double *)malloc((size_t)k * sizeof(double));
  double acc = 0.0;
  for (int64_t r = 0; r < k; ++r) {
    acc += exp((double)kz[r] - (double)kz[0]);
    cum[r] = acc;
  }
  /* top-p: up to and including the first token whose cumulative
     probability exceeds p */
  int64_t m = k;
  if (top_p < 1.0f) {
    m = 0;
    while (m < k && cum[m] <= (double)top_p * acc) ++m;
    m = m < k ? m + 1 : k;
  }
  const double total = cum[m - 1], target = u * total;
  int64_t pick = 0;
  while (pick < m - 1 && cum[pick] <= target) ++pick;
  if (cand_idx)
    for (int64_t r = 0; r < m; ++r) cand_idx[r] = kid[r];
  if (cand_cum)
    for (int64_t r = 0; r < m; ++r) cand_cum[r] = cum[r] / total;
  if (n_cand) *n_cand = m;
  const int32_t tok = kid[pick];
  free(cum);
  free(kz);
  free(kid);
  free(z);
  return tok;
}

/* the sampler's uniform draw: word `draw` of the SplitMix64 sequence of
   `seed` (Steele, Lea & Flood, OOPSLA 2014), top 24 bits scaled to [0, 1) */
double orc_sample_uniform(uint64_t seed, uint64_t draw) {
  uint64_t z = seed + (draw + 1ULL) * 0x9E3779B97F4A7C15ULL;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  z ^= z >> 31;
  return (double)(z >> 40) * (1.0 / 16777216.0);
}

/* ------------------------------------------------------ model / state */

orc_model *orc_model_new(const orc_config *cfg, const orc_tensor *glob, const orc_tensor *layers) {
  if (cfg->n_head <= 0 || cfg->n_kv_head <= 0 || cfg->n_embd % cfg->n_head) return NULL;
  if (cfg->n_head % cfg->n_kv_head) return NULL;
  if (cfg->expert_count > 256) return NULL;
  if (cfg->expert_count > 0 && (cfg->expert_used <= 0 || cfg->expert_used > cfg->expert_count))
    return NULL;
  orc_model *m = (orc_model *)calloc(1, sizeof(orc_model));
  m->cfg = *cfg;
  m->head_dim = cfg->n_embd / cfg->n_head;
  if (m->head_dim % 2) {
    free(m);
    return NULL;
  }
  m->n_ffn_sets = cfg->expert_count > 0 ? cfg->expert_count : 1;
  memcpy(m->glob, glob, sizeof(m->glob));
  const int64_t n = (int64_t)cfg->n_layer * layer_slots(m);
  m->layer = (orc_tensor *)malloc((size_t)n * sizeof(orc_tensor));
  memcpy(m->layer, layers, (size_t)n * sizeof(orc_tensor));
  return m;
}

void orc_model_free(orc_model *m) {
  if (!m) return;
  free(m->layer);
  free(m);
}

static int64_t kv_layer_elems(const orc_model *m) {
  return (int64_t)m->cfg.n_ctx * m->cfg.n_kv_head * m->head_dim;
}

/* pn_state_new: a zeroed KV cache of n_ctx positions and pos = 0 */
orc_state *orc_state_new(const orc_model *m) {
  orc_state *s = (orc_state *)calloc(1, sizeof(orc_state));
  const size_t n = (size_t)(kv_layer_elems(m) * m->cfg.n_layer);
  s->m = m;
  s->route_margin = INFINITY;
  s->k = (float *)calloc(n, sizeof(float));
  s->v = (float *)calloc(n, sizeof(float));
  if (!s->k || !s->v) {
    free(s->k);
    free(s->v);
    free(s);
    return NULL;
  }
  return s;
}

void orc_state_free(orc_state *s) {
  if (!s) return;
  free(s->k);
  free(s->v);
  free(s);
}

/* pn_state_reset: zero every K and V tensor, pos = 0 ("Core Engine API", "State lifecycle") */
void orc_state_reset(orc_state *s) {
  const size_t n = (size_t)(kv_layer_elems(s->m) * s->m->cfg.n_layer);
  memset(s->k, 0, n * sizeof(float));
  memset(s->v, 0, n * sizeof(float));
  s->pos = 0;
}

int64_t orc_state_pos(const orc_state *s) { return s->pos; }
double orc_state_route_margin(const orc_state *s) { return s->route_margin; }
void orc_state_set_pos(orc_state *s, int64_t pos) { s->pos = pos; }

/* [n_ctx][n_kv][hd] cache of one layer; kind 0 = K, 1 = V */
float *orc_state_kv(orc_state *s, int layer, int kind) {
  return (kind ? s->v : s->k) + (int64_t)layer * kv_layer_elems(s->m);
}

/* Pre-fill positions [j_lo, P) of every layer with generated cache contents
   (standard deviation sigma, storage type of the model) and set pos = P. */
int orc_state_prefill_synth(orc_state *s, uint64_t seed, uint32_t sub, int64_t j_lo, int64_t P,
                            float sigma) {
  const orc_config *c = &s->m->cfg;
  const int64_t per_pos = (int64_t)c->n_kv_head * s->m->head_dim;
  if (j_lo < 0 || P > c->n_ctx || j_lo > P) return -1;
  for (int l = 0; l < c->n_layer; ++l) {
    for (int kind = 0; kind < 2; ++kind) {
      const uint64_t key = synth_key(seed, kind ? SYNTH_VCACHE : SYNTH_KCACHE, (uint32_t)l, sub);
      float *dst = orc_state_kv(s, l, kind);
#pragma omp parallel for schedule(static)
      for (int64_t j = j_lo; j < P; ++j)
        for (int64_t e = 0; e < per_pos; ++e)
          dst[j * per_pos + e] = synth_value(key, (uint64_t)(j * per_pos + e), sigma,
                                             c->dtype == SYNTH_F32 ? SYNTH_F32 : SYNTH_BF16);
    }
  }
  s->pos = P;
  return 0;
}

/* ------------------------------------------------------------ forward */

/* Token embedding: x = row `token` of tok_embd (storage values as fp32).
   Returns 0, or -1 for a token outside [0, n_vocab). */
int orc_embed(const orc_model *m, int32_t token, float *x) {
  if (token < 0 || token >= m->cfg.n_vocab) return -1;
  get_row(&m->glob[ORC_G_TOK_EMBD], token, m->cfg.n_embd, m->cfg.dtype, x);
  return 0;
}

/* One transformer layer l for the token at position state->pos: attention
   block (RMSNorm, Q/K/V, RoPE, cache append, attention, output projection,
   residual) then feed-forward block (RMSNorm, SwiGLU or top-k MoE, residual),
   updating x [n_embd] in place.  Does not advance pos.  Returns -2 when the
   cache is full. */
int orc_layer(const orc_model *m, orc_state *s, int l, float *x) {
  const orc_config *c = &m->cfg;
  const int64_t E = c->n_embd, H = c->n_head, Hkv = c->n_kv_head, hd = m->head_dim;
  const int64_t F = c->n_ff;
  const int dt = c->dtype;
  const int64_t p = s->pos;
  if (p >= c->n_ctx) return -2;

  float *xn = (float *)malloc((size_t)E * sizeof(float));
  float *wbuf = (float *)malloc((size_t)E * sizeof(float));
  float *q = (float *)malloc((size_t)(H * hd) * sizeof(float));
  float *kn = (float *)malloc((size_t)(Hkv * hd) * sizeof(float));
  float *vn = (float *)malloc((size_t)(Hkv * hd) * sizeof(float));
  float *o = (float *)malloc((size_t)(H * hd) * sizeof(float));
  float *t = (float *)malloc((size_t)E * sizeof(float));
  float *t2 = (float *)malloc((size_t)E * sizeof(float));

  /* attention block */
  get_row(ltensor(m, l, ORC_L_ATTN_NORM), 0, E, 0, wbuf);
  orc_rmsnorm(x, wbuf, E, c->rms_norm_eps, xn);
  orc_matvec(ltensor(m, l, ORC_L_WQ), H * hd, E, dt, xn, q);
  orc_matvec(ltensor(m, l, ORC_L_WK), Hkv * hd, E, dt, xn, kn);
  orc_matvec(ltensor(m, l, ORC_L_WV), Hkv * hd, E, dt, xn, vn);
  if (c->qkv_bias) {
    /* Qwen2: q, k, v each get their bias before RoPE ("Engine Architecture",
       "Architecture Detection": attention biases set by config flags) */
    float *dst[3] = {q, kn, vn};
    const int64_t n[3] = {H * hd, Hkv * hd, Hkv * hd};
    for (int j = 0; j < 3; ++j) {
      float *b = (float *)malloc((size_t)n[j] * sizeof(float));
      get_row(ltensor(m, l, bias_slot(m, j)), 0, n[j], 0, b);
      for (int64_t e = 0; e < n[j]; ++e) dst[j][e] = dst[j][e] + b[e];
      free(b);
    }
  }
  for (int64_t h = 0; h < H; ++h)
    (c->rope_neox ? orc_rope_neox : orc_rope)(q + h * hd, (int)hd, p, c->rope_theta);
  for (int64_t g = 0; g < Hkv; ++g)
    (c->rope_neox ? orc_rope_neox : orc_rope)(kn + g * hd, (int)hd, p, c->rope_theta);
  float *Kl = orc_state_kv(s, l, 0), *Vl = orc_state_kv(s, l, 1);
  for (int64_t e = 0; e < Hkv * hd; ++e) {
    Kl[p * Hkv * hd + e] = dt ? orc_round_bf16(kn[e]) : kn[e];
    Vl[p * Hkv * hd + e] = dt ? orc_round_bf16(vn[e]) : vn[e];
  }
  orc_attention(q, Kl, Vl, (int)H, (int)Hkv, (int)hd, p, c->sliding_window, o);
  orc_matvec(ltensor(m, l, ORC_L_WO), E, H * hd, dt, o, t);
  for (int64_t i = 0; i < E; ++i) x[i] = x[i] + t[i];

  /* feed-forward block */
  get_row(ltensor(m, l, ORC_L_FFN_NORM), 0, E, 0, wbuf);
  orc_rmsnorm(x, wbuf, E, c->rms_norm_eps, xn);
  if (c->expert_count <= 0) {
    orc_ffn(ltensor(m, l, ORC_L_EXPERT0), ltensor(m, l, ORC_L_EXPERT0 + 1),
            ltensor(m, l, ORC_L_EXPERT0 + 2), E, F, dt, xn, t);
  } else {
    const int X = c->expert_count, k = c->expert_used;
    float r[256];
    int32_t idx[256];
    double g[256];
    orc_matvec(ltensor(m, l, ORC_L_WROUTER), X, E, dt, xn, r);
    orc_topk_softmax(r, X, k, idx, g);
    if (k < X) {
      /* how close the top-k choice came to a tie: the k-th chosen logit
         against the best unchosen one */
      float best_out = -INFINITY, amax = 0.f;
      for (int e = 0; e < X; ++e) {
        int chosen = 0;
        for (int i = 0; i < k; ++i) chosen |= (idx[i] == e);
        if (!chosen && r[e] > best_out) best_out = r[e];
        if (fabsf(r[e]) > amax) amax = fabsf(r[e]);
      }
      const double gap = ((double)r[idx[k - 1]] - (double)best_out) / (amax > 0.f ? (double)amax : 1.0);
      if (gap < s->route_margin) s->route_margin = gap;
    }
    double *acc = (double *)calloc((size_t)E, sizeof(double));
    for (int i = 0; i < k; ++i) {
      const int base = ORC_L_EXPERT0 + 3 * idx[i];
      orc_ffn(ltensor(m, l, base), ltensor(m, l, base + 1), ltensor(m, l, base + 2), E, F, dt, xn,
              t2);
      for (int64_t e = 0; e < E; ++e) acc[e] += g[i] * (double)t2[e];
    }
    for (int64_t e = 0; e < E; ++e) t[e] = (float)acc[e];
    free(acc);
  }
  for (int64_t i = 0; i < E; ++i) x[i] = x[i] + t[i];

  free(xn);
  free(wbuf);
  free(q);
  free(kn);
  free(vn);
  free(o);
  free(t);
  free(t2);
  return 0;
}

/* Final RMSNorm, LM head and greedy pick from the residual x [n_embd]. */
void orc_head(const orc_model *m, const float *x, float *logits, int32_t *argmax) {
  const int64_t E = m->cfg.n_embd, V = m->cfg.n_vocab;
  float *xn = (float *)malloc((size_t)E * sizeof(float));
  float *wbuf = (float *)malloc((size_t)E * sizeof(float));
  float *lg = (float *)malloc((size_t)V * sizeof(float));
  get_row(&m->glob[ORC_G_OUT_NORM], 0, E, 0, wbuf);
  orc_rmsnorm(x, wbuf, E, m->cfg.rms_norm_eps, xn);
  orc_matvec(&m->glob[ORC_G_OUTPUT], V, E, m->cfg.dtype, xn, lg);
  if (logits) memcpy(logits, lg, (size_t)V * sizeof(float));
  if (argmax) *argmax = orc_argmax(lg, V);
  free(xn);
  free(wbuf);
  free(lg);
}

/* One decode step for `token` at position state->pos: embedding, every
   layer, final norm + LM head; writes fp32 logits [n_vocab] (if logits !=
   NULL) and the greedy token (if argmax != NULL), then advances pos.
   Returns 0, -1 for a bad token, -2 when the cache is full. */
int orc_forward(const orc_model *m, orc_state *s, int32_t token, float *logits, int32_t *argmax) {
  if (token < 0 || token >= m->cfg.n_vocab) return -1;
  if (s->pos >= m->cfg.n_ctx) return -2;
  float *x = (float *)malloc((size_t)m->cfg.n_embd * sizeof(float));
  s->route_margin = INFINITY;
  orc_embed(m, token, x);
  for (int l = 0; l < m->cfg.n_layer; ++l) orc_layer(m, s, l, x);
  orc_head(m, x, logits, argmax);
  s->pos += 1;
  free(x);
  return 0;
}
