/*
 * pnb.h - C ABI of the GB300 (sm_103a) transformer decode step.
 *
 * One call advances a sequence by one token through a Llama-family decoder
 * (Llama, Qwen2-style, Mistral sliding window, Mixtral top-k MoE) and returns
 * fp32 logits and/or the greedy token.  It is the decode seam of the Pantheon
 * engine pages: a forward function of type tm_tensor* (*)(pn_model*, uint32_t
 * token, pn_state*) that reads the token, appends to the state's KV cache,
 * advances state->pos and returns logits ("Core Engine API", section
 * "pn_model struct"), plus its batched form, in which several sequences with
 * their own states advance one token each ("Engine Architecture", section
 * "Continuous-Batch VLM Decoder": one M=B decode over all slots).
 *
 * Conventions for every entry point:
 *  - Pointers named *_dev are device pointers of the calling thread's current
 *    device, which must be the device current when the model was created.
 *    Weights, KV buffers, logits and token buffers are owned by the caller and
 *    must outlive the model / state that uses them.  Device pointers must be
 *    16-byte aligned (PNB_E_ALIGN otherwise).
 *  - Calls that take a stream are stream-ordered: they validate arguments on
 *    the host, enqueue work and return without waiting.  The caller
 *    synchronises (or records an event) to read results; pnb_forward_begin /
 *    pnb_forward_poll wrap this as the pages' begin / poll pair ("Core Engine
 *    API", section "Async forward-step seam").
 *  - At most one step may be in flight per state, and one batched step per
 *    model (the pages' per-model gen_lock gives the same guarantee).
 *  - Return value: PNB_OK (0) or a negative PNB_E_* code; nothing is enqueued
 *    when a call fails its host-side checks.  A step whose device-side checks
 *    fail (a token id out of range arriving through device memory, a bounded
 *    wait that expired) records an error word in the state, read with
 *    pnb_state_check().
 */
#ifndef PNB_H
#define PNB_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream (cudaStream_t); NULL is the legacy default stream. */
typedef struct CUstream_st *pnb_stream;

/* storage type of the weights; the KV cache is fp32 for PNB_F32 and bf16
   otherwise.  PNB_Q8_0: the pages' quantized weight mode ("Engine
   Architecture", "Weight Loading Modes": weights stay in their GGUF blocks
   and are dequantized per block inside the matvec), with GGUF Q8_0 blocks of
   32 int8 values and one fp16 scale (weight = scale * value), stored per row
   as all K values followed by the row's K / 32 scales (K + K / 16 bytes).
   PNB_Q4_0: the same mode with GGUF Q4_0 blocks of 32 4-bit codes u and one
   fp16 scale (weight = scale * (u - 8)), stored per row as K / 2 bytes of
   codes (byte j holds code 2j in its low and code 2j + 1 in its high nibble)
   followed by the row's K / 32 scales (K / 2 + K / 16 bytes). */
enum { PNB_F32 = 0, PNB_BF16 = 1, PNB_Q8_0 = 2, PNB_Q4_0 = 3 };

enum {
  PNB_OK = 0,
  PNB_E_INVAL = -1,       /* invalid configuration or argument */
  PNB_E_NULL = -2,        /* a required pointer is NULL */
  PNB_E_ALIGN = -3,       /* a device pointer is not 16-byte aligned */
  PNB_E_CTX_FULL = -4,    /* pos would reach n_ctx */
  PNB_E_UNSUPPORTED = -5, /* valid but not supported by this build (cf. the pages' -1) */
  PNB_E_CUDA = -6,        /* a CUDA runtime call failed */
  PNB_E_TOKEN = -7,       /* token id outside [0, n_vocab) */
  PNB_E_DEVICE = -8,      /* a device-side check failed (see pnb_state_check) */
  PNB_E_NOMEM = -9,       /* host or device allocation failed */
  PNB_E_WRONG_DEVICE = -10, /* current device differs from the model's */
  PNB_E_TOO_LARGE = -11,   /* needs more than PNB_STATIC_SCRATCH_BYTES of static scratch */
  PNB_E_BUSY = -12         /* the state has begun work that has not been polled to completion */
};

/* device-side error bits (pnb_state_check) */
enum {
  PNB_DEV_ERR_TOKEN = 1,   /* a token from device memory was out of range; id 0 was used */
  PNB_DEV_ERR_TIMEOUT = 2  /* a bounded wait inside a kernel expired; results are invalid */
};

/* Model dimensions: the config fields of the pages ("Engine Architecture",
   section "Config Parsing": n_vocab, n_embd, n_head, n_kv_head (default
   n_head), n_layer, n_ff, n_ctx (default 2048), rope_theta (default 10000),
   rms_norm_eps (default 1e-5), sliding_window (default 0 = disabled)) plus the
   MoE fields (expert_count > 0 selects the Mixtral FFN, "Architecture
   Detection"; the arena reserves n_experts + 2*n_experts_used floats for the
   router, "Core Engine API", section "Scratch (arena) estimation").
   The library applies no defaults: every field is used as given.
   head_dim = n_embd / n_head.
   rope_neox = 1 selects the NeoX-style rotation of the Phi-3 forward, which
   pairs dimension i of a head with dimension i + head_dim / 2 ("Engine
   Architecture", "Architecture Detection"); 0 the Llama form, adjacent pairs
   (2i, 2i + 1).  Both turn pair i by pos * rope_theta^(-2i/head_dim).  The
   kernels rotate adjacent pairs only: a NeoX model gives each head's Wq and
   Wk rows (and its q / k bias entries) in the order 0, hd/2, 1, hd/2 + 1,
   ..., hd/2 - 1, hd - 1, which makes each NeoX pair adjacent (the reordering
   a loader applies once), and its cached keys are in that order. */
typedef struct {
  int32_t n_vocab, n_embd, n_head, n_kv_head, n_layer, n_ff, n_ctx;
  double rope_theta, rms_norm_eps;
  int32_t sliding_window; /* 0 = attend to every position */
  int32_t expert_count;   /* 0 = dense SwiGLU FFN */
  int32_t expert_used;    /* top-k experts per token when expert_count > 0 */
  int32_t dtype;          /* PNB_F32, PNB_BF16, PNB_Q8_0 or PNB_Q4_0: weights (KV: fp32, else bf16) */
  int32_t rope_neox;      /* 0 Llama-style RoPE, 1 NeoX-style (see above) */
} pnb_config;

/* Device weights, caller-owned, in the library's layout (row-major; "dtype" =
   the config's storage type; norm vectors are always fp32, as the pages keep
   layer norms in F32: "Engine Architecture", section "Weight Loading Modes").
   Per-layer entries are HOST arrays of device pointers, read once by
   pnb_model_create.  With S = max(1, expert_count), E = n_embd, hd = head_dim:
     tok_embd            [n_vocab][E]                          dtype
     out_norm            [E]                                   fp32
     output              [n_vocab][E]                          dtype  (LM head)
     attn_norm[l]        [E]                                   fp32
     wqkv[l]             [(n_head + 2 n_kv_head) hd][E]        dtype  rows: Wq, then Wk, then Wv
     wo[l]               [E][n_head hd]                        dtype
     ffn_norm[l]         [E]                                   fp32
     w_router[l]         [expert_count][E]                     dtype  (NULL array when dense)
     w_gate_up[l*S + e]  [2 n_ff][E]                           dtype  row 2i = gate row i, 2i+1 = up row i
     w_down[l*S + e]     [E][n_ff]                             dtype
     bqkv[l]             [(n_head + 2 n_kv_head) hd]           fp32   q, k, v biases in wqkv's row order
                                                                      (Qwen2; NULL array: no biases)
   A model with biases runs the single-sequence and batched steps alike. */
typedef struct {
  const void *tok_embd;
  const float *out_norm;
  const void *output;
  const float *const *attn_norm;
  const void *const *wqkv;
  const void *const *wo;
  const float *const *ffn_norm;
  const void *const *w_router;
  const void *const *w_gate_up;
  const void *const *w_down;
  const float *const *bqkv;
} pnb_weights;

typedef struct pnb_model pnb_model;
typedef struct pnb_state pnb_state;

/* Create a model on the current device from a config and device weights
   (the pages' pn_model: config + weights + forward, "Core Engine API",
   section "pn_model struct"; Llama, Qwen2, Mistral and Mixtral share one
   forward, "Architecture registry").  Checks: n_embd = n_head * head_dim,
   head_dim even and in {32, 64, 128}, n_head % n_kv_head == 0, n_embd and
   n_ff multiples of 8, 0 < expert_used <= expert_count <= 64 when MoE,
   pointer non-NULL and 16-byte aligned.  PNB_Q8_0 and PNB_Q4_0 need n_embd and n_ff
   multiples of 256 (whole 16-byte vectors per row; PNB_E_UNSUPPORTED
   otherwise).  Every matrix of such a model is in the blocks, the MoE router
   and experts included (the pages dequantize only the embeddings and norms at
   load, "Weight Loading Modes"); its models run the single-sequence step only
   (no batched form; pnb_prefill goes one token per step).  *out is set on success. */
int pnb_model_create(const pnb_config *cfg, const pnb_weights *w, pnb_model **out);
void pnb_model_free(pnb_model *m);

/* Bytes of the KV buffer a state needs: n_layer * 2 * n_kv_head * cap *
   head_dim * (4 for PNB_F32, else 2), with cap = min(n_ctx, sliding_window) when the
   window is set, else n_ctx.  Layout, row-major:
     [n_layer][2 (K, V)][n_kv_head][cap][head_dim]
   Position j lives in slot j % cap (a ring when the window is set: the last
   `sliding_window` positions are all a step can attend).  Cache contents are
   raw, i.e. keys are stored after RoPE. */
size_t pnb_state_kv_bytes(const pnb_model *m);

/* Create a state over a caller-owned KV buffer (the pages' pn_state: KV cache
   and pos, "Core Engine API", section "pn_state struct").  The library
   allocates the state's device workspace (activations, split-KV partials,
   counters: the role of the pages' per-state arena, "Scratch (arena)
   estimation").  The new state has pos = 0; the KV buffer is not touched. */
int pnb_state_new(pnb_model *m, void *kv_dev, size_t kv_bytes, pnb_state **out);
void pnb_state_free(pnb_state *s);

/* Zero every K and V entry and set pos = 0 (pn_state_reset, "Core Engine
   API", section "State lifecycle"); also clears the device error word and
   the sampler's draw counter. */
int pnb_state_reset(pnb_state *s, pnb_stream stream);

/* Set pos, e.g. after the caller has filled cache positions [0, pos) itself.
   Requires 0 <= pos < n_ctx. */
int pnb_state_set_pos(pnb_state *s, int32_t pos, pnb_stream stream);

/* pos as of the last enqueued call (host bookkeeping, no device access). */
int pnb_state_get_pos(const pnb_state *s, int32_t *pos);

/* Synchronise the state's last stream work and read its device error word
   (PNB_DEV_ERR_* bits, 0 = none).  Returns PNB_E_DEVICE when it is nonzero. */
int pnb_state_check(pnb_state *s, int32_t *device_error);

/* Token value meaning "this state's current next token": the greedy token
   of its previous step, or the token pnb_sample drew after it. */
#define PNB_TOKEN_PREV (-1)

/* One decode step of one sequence (model->forward(model, token, state)).
   token: an id in [0, n_vocab), or PNB_TOKEN_PREV to feed back the argmax
   of this state's previous step without a host round trip.
   logits_dev: [n_vocab] fp32 output or NULL.  argmax_dev: [1] int32 output
   (greedy token, lowest id on ties; "Engine Architecture", section
   "Sampling": temperature 0 is argmax) or NULL.  Advances pos by one.
   Errors: PNB_E_TOKEN, PNB_E_CTX_FULL (pos = n_ctx - 1 already used). */
int pnb_forward(pnb_model *m, pnb_state *s, int32_t token, pnb_stream stream, float *logits_dev,
                int32_t *argmax_dev);

/* One decode step of B sequences together (pn_llama_forward_batch, "Engine
   Architecture", section "Vision-Language and Bulk OCR": one batched decode
   over all active slots; "Serve Layer Architecture", section "Batched
   Decode").  states: host array of B distinct states of this model; slot b
   reads tokens_dev[b] (device int32, or, when tokens_dev is NULL, its own
   previous argmax) and its own state's KV cache and pos, and advances that
   pos by one.  logits_dev: [B][n_vocab] fp32 or NULL; argmax_dev: [B] int32
   or NULL.  1 <= B <= 64.  Every weight is read once per step for all slots:
   the projections run on tcgen05 tensor cores with each activation split into
   a bf16 high and low part, so results equal B single-sequence steps to about
   1e-5 relative (not bitwise).  Supported: bf16 models with n_embd,
   n_head * head_dim and n_ff multiples of 64, dense or MoE; fp32 and Q8
   models return PNB_E_UNSUPPORTED (the pages' batched decoder returns -1
   for F32, and for MoE, which this one covers).  MoE: a router kernel gives
   every slot its top-k experts and their softmax weights (the
   single-sequence router's arithmetic per slot); each expert's gate/up and
   down projections then run over all slots, and the down projection adds
   weight * output to the slots that chose the expert - every expert's
   weights are streamed once per step.  B = 1 runs the single-sequence step
   (the faster path for one slot).  PNB_E_CTX_FULL when any slot's pos already reached n_ctx; a token
   outside [0, n_vocab) sets PNB_DEV_ERR_TOKEN in that slot's state.  The
   first call allocates the model's batched workspace (make it before any
   stream capture). */
int pnb_forward_batch(pnb_model *m, pnb_state *const *states, int32_t B, const int32_t *tokens_dev,
                      pnb_stream stream, float *logits_dev, int32_t *argmax_dev);

/* Capture each step into a CUDA graph and replay it (default 1), or launch
   the kernels one by one (0).  Results are identical either way. */
int pnb_model_set_graphs(pnb_model *m, int enable);

/* Bitwise reproducible batched steps (enable = 1) or the faster default (0).
   The batched step splits the output and down projections over K; by default
   each K part adds into the fp32 residual with an atomic add, so the last bits
   of the residual, and of the logits, can change from run to run.  Enabled,
   each part adds into a 64-bit fixed-point sum (units of 2^-32, exact and
   independent of the order), which the next norm folds into the residual
   once: the same steps from the same states then give the same bits, at
   3-4 % of step time (Llama-8B shapes: 4.2 % at B = 8, 3.2 % at B = 64; the
   64-bit adds and the fold).  The single-sequence step is reproducible either way.  Takes effect at the next
   batched step (its graph is re-captured). */
int pnb_model_set_deterministic_batch(pnb_model *m, int enable);

/* Decode attention on tcgen05 tensor cores (enable = 1, the default where
   the model allows it: bf16 weights and KV, head_dim 64 or 128, n_head /
   n_kv_head in {1, 2, 4, 8}, and with a sliding window a cache of a multiple
   of 128 positions) or on CUDA cores (0).  The scores and the weighted sum of
   V are MMAs whose fp32-side operands (queries, softmax weights) are split
   into bf16 high and low parts; results agree with the CUDA-core kernel to
   about 1e-5 relative.  Affects the single-sequence and batched steps.
   Returns PNB_E_UNSUPPORTED when enabling is not possible for this model. */
int pnb_model_set_tensor_attention(pnb_model *m, int enable);
int pnb_model_is_tensor_attention(const pnb_model *m);

/* Prefill: feed T >= 1 prompt tokens (tokens_dev [T], device int32) to a
   state, advancing its position by T, with every token's logits and greedy
   token written like a step's ("Core Engine API": the engine's prefill entry
   point; "Engine Architecture", "Chunked prefill").
   Chunks of up to 64 tokens run as one batched step of "virtual slots" that
   share the state's KV cache at positions pos .. pos + n - 1. Their K / V are
   stored by the chunk's QKV kernel before its attention kernel reads them,
   and each token attends to the positions up to its own. A sliding-window
   ring must not wrap inside a chunk, so once the ring is full the remaining
   tokens go one per step, as do models the batched step does not cover
   (fp32, Q8); a chunk of one token is a single-sequence step.
   logits_dev: optional [T][n_vocab] fp32 (16-byte aligned); argmax_dev:
   optional [T]. After the call the state's device token is the last token's
   argmax (PNB_TOKEN_PREV continues from it). Stream-ordered; it uses the
   model's batched workspace, so prefills and batched steps of one model must
   not overlap on the GPU. Returns PNB_E_CTX_FULL when pos + T > n_ctx and
   PNB_E_INVAL when T < 1. */
int pnb_prefill(pnb_model *m, pnb_state *s, const int32_t *tokens_dev, int32_t T, pnb_stream stream,
                float *logits_dev, int32_t *argmax_dev);

/* Sampling parameters ("Engine Architecture", section "Sampling": applied
   in the order temperature, repetition penalty, top-k, top-p, softmax,
   multinomial draw; the fields of the pages' pn_sampling_params). */
typedef struct {
  float temperature;    /* z = logit / temperature; <= 0: greedy argmax (lowest id on ties) */
  float repeat_penalty; /* > 0; each distinct recent token's z is divided by it when
                           positive, multiplied by it otherwise; 1 = off */
  int32_t top_k;        /* keep the k largest z; <= 0 or >= n_vocab: all */
  float top_p;          /* keep tokens in order until the cumulative probability
                           exceeds top_p (that token included); >= 1: all */
  uint64_t seed;        /* draw d of a state uses word d of SplitMix64(seed) */
} pnb_sampling_params;

/* Draw the next token from a step's logits (pn_sample_next_token, "Core
   Engine API", section "Sampler seam"), on the device, stream-ordered.
   logits_dev: [n_vocab] fp32, 16-byte aligned; as in the pages' sampler it is
   changed in place (it holds logit / temperature after the penalty when
   temperature > 0).  recent_dev: n_recent device int32 tokens the penalty
   applies to (ids outside [0, n_vocab) are ignored; NULL when n_recent is 0).
   The order of the candidates is z descending, lower id first on ties; the
   draw takes u = (word >> 40) * 2^-24 of SplitMix64 word d, where d is the
   state's draw counter (zeroed by pnb_state_reset, set by
   pnb_state_set_draw, advanced by one per call), and returns the first kept
   token whose cumulative probability exceeds u times the kept total.
   Probabilities are exp(z - max z) summed in 64-bit fixed point (units of
   2^-40), so the result is deterministic; it matches an exact computation
   except when u or top_p falls within about 1e-6 of a cumulative boundary.
   The token becomes the state's next token (pnb_forward with PNB_TOKEN_PREV,
   pnb_forward_batch with tokens_dev NULL) and is written to token_dev
   ([1] device int32) when given.  Logits must not be NaN and logit /
   temperature must be finite.  PNB_E_UNSUPPORTED when n_vocab >= 2^22 or
   its recent-token bitmap (n_vocab / 8 bytes) does not fit in shared memory
   beside the kernel's other 137 KB; PNB_E_INVAL for a NaN or infinite temperature,
   a penalty that is not a positive finite number or a NaN top_p. */
int pnb_sample(pnb_model *m, pnb_state *s, float *logits_dev, const pnb_sampling_params *params,
               const int32_t *recent_dev, int32_t n_recent, pnb_stream stream, int32_t *token_dev);

/* pnb_sample for B <= 64 distinct states at once (the pages' batch
   scheduler samples every slot after each batched step: "Serve Layer
   Architecture", section "L3 - in-driver sampling"), one launch: logits_dev
   [B][n_vocab]; params, recent_dev and n_recent are host arrays of B
   (recent_dev and n_recent may be NULL: no penalty window); tokens_dev [B]
   optional. */
int pnb_sample_batch(pnb_model *m, pnb_state *const *states, int32_t B, float *logits_dev,
                     const pnb_sampling_params *params, const int32_t *const *recent_dev,
                     const int32_t *n_recent, pnb_stream stream, int32_t *tokens_dev);

/* Set the state's draw counter (stream-ordered). */
int pnb_state_set_draw(pnb_state *s, uint32_t draw, pnb_stream stream);

/* Begin / poll ("Core Engine API", section "Async forward-step seam").
   pnb_forward_begin enqueues pnb_forward on the state's own non-blocking
   stream (pnb_state_stream; work for this state on other streams must be
   ordered before it by the caller), records an event and returns at once.
   pnb_sample_begin enqueues pnb_sample on the same stream and moves the
   event after it.  pnb_forward_poll returns 1 while the begun work runs;
   when it has finished, PNB_OK with *logits_out (if not NULL) set to the
   logits buffer of the begun step, PNB_E_DEVICE when the state's device
   error word is set, PNB_E_CUDA on a CUDA error - each of these ends the
   begun work.  Begin while work is outstanding returns PNB_E_BUSY; poll
   without begun work PNB_E_INVAL.  Every model supports it (the pages'
   begin answers 1, "unsupported", for all but one model family). */
int pnb_forward_begin(pnb_model *m, pnb_state *s, int32_t token, float *logits_dev,
                      int32_t *argmax_dev);
int pnb_sample_begin(pnb_model *m, pnb_state *s, float *logits_dev,
                     const pnb_sampling_params *params, const int32_t *recent_dev,
                     int32_t n_recent, int32_t *token_dev);
int pnb_forward_poll(pnb_model *m, pnb_state *s, float **logits_out);
int pnb_state_stream(pnb_state *s, pnb_stream *out);

/* Number of this library's kernels one step launches (single sequence when
   B == 0, batched otherwise). */
int pnb_step_kernel_count(const pnb_model *m, int32_t B);

/* The kernels of one decode step, in launch order within a layer. */
enum {
  PNB_KERNEL_QKV = 0,     /* RMSNorm (+ embedding in layer 0), Wqkv, RoPE, KV append */
  PNB_KERNEL_ATTN = 1,    /* split-KV attention with window, log-sum-exp merge */
  PNB_KERNEL_OPROJ = 2,   /* Wo + residual */
  PNB_KERNEL_ROUTER = 3,  /* MoE only: router logits, top-k, softmax */
  PNB_KERNEL_GATE_UP = 4, /* RMSNorm, gate/up (chosen experts), SwiGLU */
  PNB_KERNEL_DOWN = 5,    /* down projection(s) + residual */
  PNB_KERNEL_LM_HEAD = 6  /* final RMSNorm, LM head, argmax, pos += 1 */
};

/* Launch one kernel of the single-sequence step for `layer` in isolation
   (stream-ordered, no overlap with the previous kernel), reading and writing
   the state's workspace and KV cache exactly as inside a step: meant for
   per-kernel timing and checks.  The host position is not changed (the LM
   head kernel still advances the device position, as in a step). */
int pnb_step_kernel(pnb_model *m, pnb_state *s, int32_t kind, int32_t layer, pnb_stream stream);

/* Device pointers of a state's fp32 activation buffers after its last step
   (x: residual [n_embd]; q: rotated queries [n_head*hd]; attn: attention
   output [n_head*hd]; h: SwiGLU activations [max(1,expert_used)][n_ff]);
   meant for layer-level checks in tests. */
typedef struct {
  float *x, *q, *attn, *h;
} pnb_activations;
int pnb_state_activations(const pnb_state *s, pnb_activations *out);

/* Bytes of the device scratch array behind pnb_attention_decode_static. */
#define PNB_STATIC_SCRATCH_BYTES (2u << 20)

/* Split-KV decode attention of one layer for callers that may not allocate.
   No counterpart in the Pantheon pages: it exists for callers that cannot
   call cudaMalloc - code running where device allocation is forbidden after
   start-up, frameworks whose own pool owns all device memory, or plugins that
   only receive input and output buffers.  It allocates nothing (no
   cudaMalloc, cudaFree or allocating library call): its scratch (per-split
   partials, arrival counters, an I/O word) is one file-scope device array of
   PNB_STATIC_SCRATCH_BYTES that every GPU which loads this library holds
   until the process exits.
     q_dev   [n_head][head_dim] fp32 queries (already rotated), 16-byte aligned
     k_dev   one layer's K cache [n_kv_head][cap][head_dim], dtype (PNB_F32 / PNB_BF16)
     v_dev   the same layer's V cache, same layout
     out_dev [n_head][head_dim] fp32 output: softmax over positions
             [max(0, pos - window + 1), pos] (all of [0, pos] when window == 0)
             of q.k / sqrt(head_dim), applied to V; position j lives in slot j % cap
   head_dim in {32, 64, 128}; n_head % n_kv_head == 0; pos < cap unless
   window > 0 and cap >= window.  Returns PNB_E_TOO_LARGE when the partials
   of even one split, or the counters, do not fit the static scratch.
   The first call on each device looks up the array's device address with
   that device current (cudaGetSymbolAddress); make that first call before
   any stream capture.  Every call uses the same array and leaves its
   contents behind: each call clears the counters and I/O word it needs, and
   calls whose work overlaps on the GPU (concurrent streams) race on the
   array and must be serialised by the caller.
     err_dev optional device int32 (NULL: not written).  After the kernel, in
             stream order, it receives the call's device error bits
             (PNB_DEV_ERR_*, 0 = none): PNB_DEV_ERR_TIMEOUT means a bounded
             wait inside the kernel gave up and out_dev is not valid.  It is
             copied out of the static array before the next call clears it. */
int pnb_attention_decode_static(const float *q_dev, const void *k_dev, const void *v_dev,
                                int32_t dtype, int32_t n_head, int32_t n_kv_head, int32_t head_dim,
                                int32_t cap, int32_t window, int32_t pos, float *out_dev,
                                int32_t *err_dev, pnb_stream stream);

/* Diagnostics: have the step's kernels record globaltimer stamps (ns) into
   trace_dev, laid out [launch][256][8]: launch = 6 * layer + kernel kind
   (PNB_KERNEL_*), 6 * n_layer for the LM head; the CTA's linear index
   (< 256) picks the row; slots 0 = CTA start, 1 = compute warps past
   griddepcontrol.wait, 2 = activation prologue done, 3 = first ring slot
   arrived, 4 = all slots consumed, 5 = epilogue done, 6 / 7 = the producer
   reached / passed griddepcontrol.wait.  A batched step records into
   its first slot's buffer with launch = 7 * layer + (0 norm, 1 QKV,
   2 attention, 3 o-proj, 4 norm, 5 gate/up, 6 down), 7 * n_layer (+1) for the
   final norm (LM head); its GEMM slots are 0 start, 1 / 2 first / last MMA,
   3 first accumulator read, 4 epilogue done, 5 end, 6 / 7 producer done /
   past griddepcontrol.wait.  NULL turns it off.  bytes must cover
   (7 * n_layer + 2) * 256 * 8 words. */
int pnb_state_set_trace(pnb_state *s, uint64_t *trace_dev, size_t bytes);

/* Diagnostic: make a bounded device wait run out.  Enqueues one kernel that
   copies part of the state's workspace into shared memory with a bulk copy,
   then waits, with a limit of limit_ns (<= 1e9, else PNB_E_INVAL), on an
   mbarrier that nothing arrives on - the same bounded wait every kernel of
   the step uses, with a shorter limit.  When it gives up, the kernel sets
   PNB_DEV_ERR_TIMEOUT in the state's error word (pnb_state_check; a later
   pnb_forward_poll on the state answers PNB_E_DEVICE), waits for its copy to
   land and returns, so the context stays usable; pnb_state_reset clears the
   word.  The KV cache and activations are not touched. */
int pnb_state_wait_probe(pnb_state *s, uint64_t limit_ns, pnb_stream stream);

const char *pnb_strerror(int code);

#ifdef __cplusplus
}
#endif

#endif /* PNB_H */
