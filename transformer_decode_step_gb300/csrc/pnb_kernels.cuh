// pnb_kernels.cuh - argument blocks and launchers of the decode-step kernels.
//
// Every weight-streaming kernel is a row-split GEMV over one or more matrices
// that share a column count K: each CTA owns a contiguous range of output rows
// and streams those rows whole through a ring of shared-memory stages filled
// by 1-D bulk copies (one elected producer thread, mbarrier completion).  The
// first ring's worth is issued before griddepcontrol.wait, so a kernel's
// weight traffic overlaps the tail of the kernel before it.  Sixteen consumer
// warps multiply the staged rows by the fp32 activation vector, each lane
// holding its fixed column slice of that vector in registers, and fold the
// result into a fused epilogue.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pnb_device.cuh"

namespace pnb {

// Geometry of one streaming GEMV launch (host-computed).
struct Geom {
  int K;              // columns (elements)
  int es;             // weight storage type: 4 fp32, 2 bf16, 1 Q8
  int row_bytes;      // K * es (Q8: K + K / 16: the values, then one fp16 scale per 32)
  int vpr;            // weight vectors per row: 16-byte (K / 4, K / 8), Q8: 8-byte (K / 8)
  int rows_per_stage; // power of two <= 64: whole rows per ring slot
  int stage_bytes;    // ring slot size = rows_per_stage * row_bytes
  int nstages;        // ring slots
  int cw;             // warps sharing one row (its columns); 16 / cw rows in flight
  int nv;             // 16-byte vectors per lane per row (1, 2 or 4)
  int row_align;      // CTA row ranges are multiples of this
  int rows_cta_max;   // most rows any CTA owns (static row ranges)
  int nsum;           // matrices summed into the same rows (1 = concatenated rows)
  int n_items;        // ring items over all segments (dynamic claiming)
  int n_static_total; // items split evenly over the CTAs; the rest are claimed
  int cap_items;      // most items one CTA may take; 0 = static row ranges
  int inflight;       // bulk copies a producer keeps in flight at most
};

// The matrices of one launch.  Rows of segment i are virtual rows
// [i*rows, (i+1)*rows) (concatenated) or the same output rows (summed).
struct Segs {
  int n;
  int64_t rows;
  const void *w[kMaxSegments];
  // MoE: segment i is expert expert_idx[i] of `table` (device pointers), known
  // only after the router kernel has run
  const void *const *table;
  const int32_t *expert_idx;
};

struct SmemLayout {
  int ring, part, red, info, items, rope, bars, total;
};

__host__ __device__ inline int align_up(int v, int a) { return (v + a - 1) / a * a; }

__host__ __device__ inline SmemLayout smem_layout(const Geom &g) {
  SmemLayout L;
  L.ring = 0;
  L.part = align_up(g.nstages * g.stage_bytes, 128);
  const int part_rows = g.cap_items > 0 ? g.cap_items * g.rows_per_stage : g.rows_cta_max;
  L.red = align_up(L.part + part_rows * g.cw * g.nsum * 4, 16);
  // per ring slot: claimed item and its CTA-local index; then the CTA's
  // claimed items and their count
  L.info = align_up(L.red + 64 * 4, 16);
  L.items = L.info + 2 * g.nstages * 4;
  L.rope = align_up(L.items + (g.cap_items + 1) * 4, 16);   // 64 (cos, sin) pairs
  L.bars = L.rope + 64 * 8;
  L.total = L.bars + 2 * g.nstages * 8;
  return L;
}

// Optional per-CTA timestamps of the per-phase kernels (diagnostics): slot
// k of CTA c in launch `phase` is p[(phase * kTraceCtas + c) * 8 + k].
constexpr int kTraceCtas = 256;
struct KTrace {
  unsigned long long *p;
  int phase;
};

__device__ __forceinline__ void ktrace(const KTrace &t, int k) {
  if (t.p) {
    const unsigned c = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);
    if (c < (unsigned)kTraceCtas) t.p[((size_t)t.phase * kTraceCtas + c) * 8 + k] = global_ns();
  }
}

// ---------------------------------------------------------------- kernels

// layer input: RMSNorm(x) (or of the embedding row of io->token when emb is
// set) -> [Wq; Wk; Wv] -> RoPE on q and k -> q buffer, K/V cache slot of pos
struct QkvArgs {
  Geom g;
  Segs s;
  const float *x;
  const void *emb;     // token embedding table (first layer) or nullptr
  float *x_out;        // residual stream, written from the embedding row
  int n_vocab;
  const float *norm_w;
  float eps;
  int n_head, n_kv, head_dim;
  const double *inv_freq;  // [head_dim / 2] = rope_theta^(-2i/head_dim)
  const float *bias;       // [rows] q / k / v bias added before RoPE, or nullptr
  float *q;
  void *k_cache, *v_cache; // this layer's [n_kv][cap][head_dim]
  int cap, window;
  unsigned *work;      // [claim, done] item counters of this launch, zero between launches
  StepIO *io;
  KTrace tr;
};

// x[r] += (W v)[r]  (output projection, dense down projection)
struct ResidArgs {
  Geom g;
  Segs s;
  const float *vec;
  float *x;
  unsigned *work;      // [claim, done] item counters of this launch, zero between launches
  StepIO *io;
  KTrace tr;
};

// h[s][i] = silu((Wg xn)_i) * (Wu xn)_i with xn = RMSNorm(x); rows of W are
// gate/up interleaved; s runs over the segments (experts)
struct GateUpArgs {
  Geom g;
  Segs s;
  const float *x;
  const float *norm_w;
  float eps;
  float *h;  // [nseg][n_ff]
  int n_ff;
  unsigned *work;      // [claim, done] item counters of this launch, zero between launches
  StepIO *io;
  KTrace tr;
};

// x[r] += sum_s gate[s] * (W_s h_s)[r]  (MoE down projections, summed)
struct DownMoeArgs {
  Geom g;
  Segs s;
  const float *h;  // [nseg][n_ff]
  int n_ff;
  const float *gate;
  float *x;
  StepIO *io;
  KTrace tr;
};

// logits = W RMSNorm(x); greedy token; pos += 1
struct LmArgs {
  Geom g;
  Segs s;
  const float *x;
  const float *norm_w;
  float eps;
  float *logits;       // optional
  int32_t *argmax_out; // optional
  float *part_val;     // [gridDim.x]
  int32_t *part_idx;   // [gridDim.x]
  unsigned int *counter;
  unsigned *work;      // [claim, done] item counters of this launch, zero between launches
  StepIO *io;
  KTrace tr;
};

// router logits, top-k, softmax over the chosen logits
struct RouterArgs {
  const void *w;  // [n_expert][E]
  int n_expert, k, E;
  const float *x;
  const float *norm_w;
  float eps;
  int32_t *idx;
  float *gate;
  StepIO *io;
  KTrace tr;
};

struct BSlot;

// split-KV decode attention of the token at io->pos (grid: n_split x n_kv x zgroups)
struct AttnArgs {
  const float *q;        // [n_head][hd]
  const void *k_cache;   // this layer's [n_kv][cap][hd]
  const void *v_cache;
  int n_head, n_kv, cap, window;
  int n_split;
  float *part;           // [n_head][n_split][hd + 2]
  unsigned int *counter; // [n_kv * zgroups]
  float *out;            // [n_head][hd]
  float qscale;          // log2(e) / sqrt(hd)
  int stage_pos;         // positions per ring slot
  int nstages;           // ring slots
  StepIO *io;
  KTrace tr;
  // batched slots (null for one sequence): blockIdx.z = zgroup + zgroups * slot;
  // slot b's K / V are at slots[b].kv + kv_off / + kv_off + layer_kv_bytes, its
  // position is pos[b], its q / part / counters are offset by b, and the merged
  // output goes to the bf16 operand (rows b and bp + b hold hi and lo parts)
  const BSlot *slots;
  const int32_t *pos;
  size_t kv_off, layer_kv_bytes;
  __nv_bfloat16 *xop;
  int xop_ld, bp, nb;    // operand row pitch, padded slots, slots
  // prefill chunk (slots share one cache): the K / V of every position from
  // pos[0] on are new, and their stages are loaded after the dependency wait
  int shared_cache;
};

// One slot of a batched step (device table, written at the start of the step).
struct BSlot {
  uint8_t *kv;        // the slot's KV buffer [layer][K|V][n_kv][cap][hd]
  StepIO *io;         // the slot's token / position / error word
  const void *maps;   // the slot's [layer][K|V] tensor maps over that buffer (or null)
};

// Tensor-core decode attention (bf16 KV, head_dim 64 or 128, up to 8 query
// heads per KV head).  Grid (n_split, n_kv, slots); a CTA takes one KV head of
// one slot and 128-position tiles of its range.
struct AttnTcArgs {
  const float *q;          // [slots][n_head][hd]
  const void *maps;        // one sequence: its state's [layer][K|V] tensor maps
  int layer;
  int n_head, n_kv, cap, window;
  int n_split;             // CTAs per KV head (one cluster), 1 .. attn_tc_max_split()
  float qscale;            // log2(e) / sqrt(hd)
  float *out;              // one sequence: [n_head][hd]
  __nv_bfloat16 *xop;      // batched: o-proj operand rows b (hi) and bp + b (lo)
  int xop_ld, bp, nb;
  const BSlot *slots;      // batched (null for one sequence)
  const int32_t *pos;      // batched positions
  StepIO *io;              // one sequence
  int nstages;
  // Prefill chunk: the slots are one sequence's consecutive tokens sharing
  // one cache, so the preceding kernel wrote the K / V of every position from
  // pos[0] on; the tiles holding them are loaded after the dependency wait.
  // 0: each slot's own position is the only new one.
  int shared_cache;
  // Token groups (prefill chunks, whose virtual slots share one cache): one
  // CTA column block serves tok_group consecutive virtual slots, column
  // t * (n_head / n_kv) + j being query head j of slot group * tok_group + t,
  // each masked to its own positions; the grid's z is the group.  0 or 1:
  // one slot per z.
  int tok_group;
  // batched slots with their own caches (tok_group <= 1): grid z = rank, slot
  // order[rank]; ranked longest attended range first, so that in a grid of
  // several waves the long CTAs start first (any permutation is correct)
  uint8_t order[64];
  int use_order;
  // > 0: the persistent form (batched slots with their own caches, one split,
  // head_dim 128): min(items, persist) CTAs walk the (slot, KV head) items
  int persist;
  // persistent form: [claim, done] counters, zero before the launch and left
  // zero after it; null: a static item order
  unsigned *tp_claim;
  KTrace tr;
};

// group: columns per KV head (query heads per KV head, times tok_group)
cudaError_t launch_attn_tc(int head_dim, int group, const AttnTcArgs &a, cudaStream_t st, bool pdl);

// attention of a prefill chunk: n consecutive tokens of one sequence whose
// keys and values are already in its cache; one CTA per (KV head, 16 query
// rows) walks the attended positions once for all its rows
struct PAttnArgs {
  const float *q;              // [n][n_head][hd] rotated queries
  const __nv_bfloat16 *k, *v;  // this layer's cache [n_kv][cap][hd]
  const int32_t *pos;          // [n] the tokens' positions (ascending)
  int n, n_head, n_kv, cap, window;
  float qscale;                // log2(e) / sqrt(hd)
  __nv_bfloat16 *xop;          // o-proj operand: rows j (hi) and bp + j (lo)
  int xop_ld, bp;
};
cudaError_t launch_pattn(int head_dim, const PAttnArgs &a, cudaStream_t st, bool pdl);
cudaError_t prepare_pattn_kernels();
int attn_tc_smem(int head_dim, int nstages);
int attn_tc_stages(int head_dim);
int attn_tc_max_split();
cudaError_t prepare_attn_tc_kernels();

// Epilogues of the batched tensor-core GEMM
// kEpiResidGate: the residual add scaled per slot by gate[b * gate_ld] (0 =
// no add), for the MoE down projections of the batched step
// kEpiResidFix / kEpiResidGateFix: the same, K parts added in fixed point
// (the deterministic batched step; see acc below)
enum BEpi { kEpiQkv = 0, kEpiResid = 1, kEpiGateUp = 2, kEpiLm = 3, kEpiResidGate = 4,
            kEpiResidFix = 5, kEpiResidGateFix = 6 };

// Y[b][r] = sum_k W[r][k] * X[b][k] for the B slots of a batched step, on
// tcgen05 (tiles of 128 weight rows, slots as the MMA's N dimension with the
// operand split into bf16 hi and lo rows), split over K into ksplit parts
// whose partial tiles the last arriving CTA sums in a fixed order.
struct BGemmArgs {
  int rows, K, nchunks;  // weight rows, columns, 64-column chunks
  int tiles, ksplit, units;
  int B, bp;             // slots, padded slot count (16, 32 or 64)
  int kind;              // BEpi
  int nstages;           // ring slots
  float *part;           // [units][B][128] split-K partials
  unsigned *tile_cnt;    // [tiles] arrival counters, zero between launches
  // epilogue operands
  float *x;              // kEpiResid: residual streams [B][rows]
  float *q;              // kEpiQkv: queries [B][n_head * hd]
  const float2 *rope;    // kEpiQkv: (cos, sin) [B][hd / 2]
  const float *bias;     // kEpiQkv: q / k / v bias [rows] added before RoPE, or null
  const BSlot *slots;    // kEpiQkv / kEpiLm
  const int32_t *pos;    // [B]
  size_t kv_off, layer_kv_bytes;
  int n_head, n_kv, hd, cap;
  __nv_bfloat16 *xop;    // kEpiGateUp: next operand [2 * bp][xop_ld]
  int xop_ld;
  const float *gate;     // kEpiResidGate: per-slot scale gate[b * gate_ld] (0 = no add)
  int gate_ld;
  float *logits;         // kEpiLm: [B][rows] or null
  int32_t *argmax_out;   // kEpiLm: [B] or null
  float *am_val;         // kEpiLm: [B][gridDim.x]
  int32_t *am_idx;
  unsigned *am_cnt;
  int32_t *err;          // batch error word
  // residual kinds with ksplit > 1: each K part adds its share into x with
  // an fp32 atomic add (order not fixed), or (kEpiResidFix / kEpiResidGateFix)
  // into acc in 64-bit fixed point (units of 2^-32): an integer sum, the same
  // in any order, which the next k_bnorm folds into x and clears
  long long *acc;        // [B][rows]
  KTrace tr;
};

// MoE router of every slot of a batched step: RMSNorm of the slot's residual,
// the router logits, top-k (ties to the lower index) and the softmax over the
// chosen; gates[b][e] is expert e's weight for slot b, 0 when not chosen
struct BRouterArgs {
  const __nv_bfloat16 *w;  // [n_expert][E]
  int n_expert, k, E;
  const float *x;          // [B][E] residual streams
  const float *norm_w;
  float eps;
  float *gates;            // [B][n_expert]
  KTrace tr;
};
cudaError_t launch_brouter(const BRouterArgs &a, int B, cudaStream_t st, bool pdl);

// RMSNorm of every slot into the bf16 hi / lo operand; on the first layer
// also the embedding gather, the step's slot table and RoPE table
struct BNormArgs {
  const float *x;          // [B][E] residual streams (layers > 0)
  float *x_out;            // first layer: embedding rows written here
  const void *emb;         // first layer: token embedding table, else null
  const int32_t *tokens;   // first layer: tokens [B] or null (each slot's io->token)
  int n_vocab, E, B, bp;
  const float *norm_w;
  float eps;
  __nv_bfloat16 *xop;      // [2 * bp][E]
  BSlot *slots_dev;        // first layer: the table is written here
  int32_t *pos;            // first layer: positions [B] written here
  float2 *rope;            // first layer: [B][hd / 2]
  const double *inv_freq;  // [hd / 2]
  int hd, n_ctx;
  int32_t *err;
  // layers > 0 and the final norm: the residual GEMMs' fixed-point K-part
  // sums [B][E] (units of 2^-32), folded into x (written back) and cleared
  long long *acc;
  KTrace tr;
  BSlot slots[128];        // first layer: the slots of this step (prefill chunks: up to 128)
};

struct AttnGeom {
  int stage_pos;  // positions per ring slot
  int nstages;
  int heads_per_cta;
  int smem;       // dynamic shared memory bytes
};

// Launchers (dtype: 0 fp32, 1 bf16).  pdl = launch with programmatic stream
// serialization.  Return the CUDA error of the launch.
cudaError_t launch_qkv(int dtype, const QkvArgs &a, int grid, cudaStream_t st, bool pdl);
cudaError_t launch_resid(int dtype, const ResidArgs &a, int grid, cudaStream_t st, bool pdl);
cudaError_t launch_gateup(int dtype, const GateUpArgs &a, int grid, cudaStream_t st, bool pdl);
cudaError_t launch_down_moe(int dtype, const DownMoeArgs &a, int grid, cudaStream_t st, bool pdl);
cudaError_t launch_lmhead(int dtype, const LmArgs &a, int grid, cudaStream_t st, bool pdl);
cudaError_t launch_router(int dtype, const RouterArgs &a, cudaStream_t st, bool pdl);
cudaError_t launch_attn(int dtype, int head_dim, const AttnArgs &a, const AttnGeom &ag,
                        cudaStream_t st, bool pdl);
cudaError_t launch_set_token(StepIO *io, int32_t token, cudaStream_t st);
// diagnostic: a bounded wait on an mbarrier nothing arrives on, after a bulk
// copy of bytes (multiple of 16, <= kWaitProbeBytes) from src; sets the
// timeout bit in io->error when the wait gives up
constexpr int kWaitProbeBytes = 4096;
cudaError_t launch_wait_probe(const void *src, uint32_t bytes, unsigned long long limit_ns, StepIO *io,
                              cudaStream_t st);
cudaError_t launch_set_pos(StepIO *io, int32_t pos, cudaStream_t st);
cudaError_t launch_copy_token(StepIO *io, const int32_t *token, cudaStream_t st);
// prefill chunk of n <= 64 virtual slots: pio[b] = {pos: state->pos + b}; then
// the state takes pio[n - 1]'s token and position and every slot's error bits
cudaError_t launch_prefill_begin(StepIO *pio, const StepIO *state, int n, cudaStream_t st);
cudaError_t launch_prefill_end(StepIO *state, const StepIO *pio, int n, cudaStream_t st);

// batched step (tensor maps are CUtensorMap, passed by value)
cudaError_t launch_bnorm(const BNormArgs &a, cudaStream_t st, bool pdl);
cudaError_t launch_bgemm(const void *tmap_w, const void *tmap_x, const BGemmArgs &a, int grid,
                         int smem, cudaStream_t st, bool pdl);
int bgemm_smem(int bp, int nstages);
// sums the K parts of a split QKV / gate-up GEMM and applies its epilogue
cudaError_t launch_bmerge(const BGemmArgs &a, cudaStream_t st, bool pdl);
cudaError_t prepare_bgemm_kernels(int smem_bytes);

// the greedy pick after a 128-slot LM head (logits [B][V] written by it)
struct BArgmaxArgs {
  const float *logits;
  int V, B;
  const BSlot *slots;
  const int32_t *pos;
  int32_t *argmax_out;   // [B] or null
  int32_t *err;          // batch error word
};
cudaError_t launch_bargmax(const BArgmaxArgs &a, cudaStream_t st, bool pdl);

// raise the dynamic shared-memory limit of the kernels a model will launch
// (outside any stream capture)
cudaError_t prepare_gemv_kernels(int dtype, int smem_bytes);
cudaError_t prepare_attn_kernel(int dtype, int head_dim, const AttnGeom &ag);

// attention geometry for a head_dim / group size (host)
AttnGeom attn_geom(int dtype, int head_dim, int group);

// ------------------------------------------------------------------ sampler
// one sequence's sampling: logits [n_vocab] (overwritten with logit / T after
// the penalty), the recent tokens the penalty applies to, the parameters, the
// state's StepIO (its token becomes the sampled one, its draw counter picks u
// and is advanced) and an optional output word
struct SampleSlot {
  float *logits;
  const int32_t *recent;
  int32_t n_recent;
  int32_t top_k;
  float temperature, repeat_penalty, top_p;
  unsigned long long seed;
  StepIO *io;
  int32_t *out;
};
constexpr int kSampleMaxSlots = 64;
struct SampleArgs {
  int n_vocab;
  SampleSlot slot[kSampleMaxSlots];
};
size_t sample_smem_bytes(int n_vocab);
cudaError_t prepare_sample_kernel(int n_vocab);
// one CTA per slot (slots 0 .. n_slots - 1 of a)
cudaError_t launch_sample(const SampleArgs &a, int n_slots, cudaStream_t st);
cudaError_t launch_set_draws(StepIO *io, uint32_t draws, cudaStream_t st);

}  // namespace pnb
