"""The decode-step workloads and their synthetic input recipe.

Shapes follow the five benchmark configurations of this project: a tiny fp32
Llama-style decoder, a Llama-7B-shaped dense decoder, a Mistral-7B-shaped GQA
decoder with a 4096-position sliding window, a Mixtral-shaped 8-expert top-2
MoE decoder and a Llama-8B-shaped batched-slot decoder.  The recipe:

* weights (embeddings, projections, router, LM head) ~ N(0, 0.02^2), stored in
  the model's dtype (Q8, Q4: blocks of 32 quantized as the generator defines);
  q / k / v biases (models with qkv_bias) ~ N(0, 0.5^2), fp32;
  every norm weight is 1.0 (fp32);
* the KV cache of positions below the start position ~ N(0, 1) in the cache
  dtype (raw cache contents, i.e. keys already rotated);
* prompt / start tokens uniform in [0, n_vocab); batched slot s starts at a
  position uniform in [512, 4096];
* all values come from ``synth`` keyed by (seed, tensor kind, layer, sub).
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace
from typing import List, Optional

from . import (ATTN_NORM, BF16, BK, BQ, BV, F32, FFN_NORM, OUT_NORM, OUTPUT, POSITIONS, Q4, Q8,
               TOK_EMBD, TOKENS, WDOWN, WGATE, WK, WO, WQ, WROUTER, WUP, WV, key, uniform_int)

WEIGHT_SIGMA = 0.02
BIAS_SIGMA = 0.5        # q / k / v biases (fp32), on the scale of the projections' outputs
KV_SIGMA = 1.0
NORM_VALUE = 1.0


@dataclass(frozen=True)
class Shape:
    n_vocab: int
    n_embd: int
    n_head: int
    n_kv_head: int
    n_layer: int
    n_ff: int
    n_ctx: int
    rope_theta: float = 10000.0
    rms_norm_eps: float = 1e-5
    sliding_window: int = 0
    expert_count: int = 0
    expert_used: int = 0
    dtype: int = BF16
    qkv_bias: bool = False    # Qwen2: bias vectors on q, k, v
    rope_neox: bool = False   # Phi-3: RoPE pairs dimension i with i + head_dim / 2

    @property
    def head_dim(self) -> int:
        return self.n_embd // self.n_head

    @property
    def kv_cap(self) -> int:
        """Positions the cache keeps: the window when one is set, else n_ctx."""
        if self.sliding_window > 0:
            return min(self.sliding_window, self.n_ctx)
        return self.n_ctx

    @property
    def elem_bytes(self) -> int:
        """Bytes of one KV-cache element (bf16 for bf16, Q8 and Q4 weights)."""
        return 4 if self.dtype == F32 else 2

    @property
    def kv_dtype(self) -> int:
        return F32 if self.dtype == F32 else BF16

    def matrix_bytes(self, rows: int, cols: int) -> int:
        """Bytes of a [rows][cols] weight matrix in the library's layout (Q8 rows:
        cols int8 values, then one fp16 scale per 32)."""
        if self.dtype == Q8:
            return rows * (cols + cols // 16)
        if self.dtype == Q4:
            return rows * (cols // 2 + cols // 16)
        return rows * cols * (4 if self.dtype == F32 else 2)

    @property
    def weight_bytes_per_param(self) -> float:
        return {F32: 4.0, BF16: 2.0, Q8: 1.0625, Q4: 0.5625}[self.dtype]

    def params_read_per_token(self) -> int:
        """Weight elements one decode step reads (top-k experts only for MoE)."""
        E, H, Hkv, hd, F, V, L = (self.n_embd, self.n_head, self.n_kv_head, self.head_dim,
                                  self.n_ff, self.n_vocab, self.n_layer)
        attn = (H + 2 * Hkv) * hd * E + E * H * hd
        ffn_sets = self.expert_used if self.expert_count > 0 else 1
        ffn = ffn_sets * 3 * F * E + (self.expert_count * E if self.expert_count > 0 else 0)
        return E + L * (attn + ffn) + V * E  # one embedding row + layers + LM head


@dataclass(frozen=True)
class Workload:
    name: str
    shape: Shape
    seed: int
    batch: int = 1
    prompt_len: int = 0       # tokens fed one by one before decoding (empty cache)
    prefill: int = 0          # cache positions pre-filled (B = 1)
    slot_pos_range: Optional[tuple] = None  # batched: start position uniform in [lo, hi]
    steps: int = 0            # greedy decode steps

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


TINY = Workload(
    "tiny_llama_f32",
    Shape(n_vocab=1024, n_embd=256, n_head=8, n_kv_head=4, n_layer=2, n_ff=688, n_ctx=128,
          rope_theta=10000.0, rms_norm_eps=1e-5, dtype=F32),
    seed=1, prompt_len=16, steps=48)

LLAMA7B = Workload(
    "llama7b_bf16",
    Shape(n_vocab=32000, n_embd=4096, n_head=32, n_kv_head=32, n_layer=32, n_ff=11008,
          n_ctx=2048 + 128, rope_theta=10000.0, rms_norm_eps=1e-5, dtype=BF16),
    seed=2, prefill=2048, steps=128)

MISTRAL7B = Workload(
    "mistral7b_bf16_w4096",
    Shape(n_vocab=32000, n_embd=4096, n_head=32, n_kv_head=8, n_layer=32, n_ff=14336,
          n_ctx=8192 + 128, rope_theta=1e6, rms_norm_eps=1e-5, sliding_window=4096, dtype=BF16),
    seed=3, prefill=8192, steps=128)

MIXTRAL = Workload(
    "mixtral8x_top2_bf16",
    Shape(n_vocab=32000, n_embd=4096, n_head=32, n_kv_head=8, n_layer=32, n_ff=14336,
          n_ctx=4096 + 128, rope_theta=1e6, rms_norm_eps=1e-5, expert_count=8, expert_used=2,
          dtype=BF16),
    seed=4, prefill=4096, steps=128)

LLAMA8B_BATCHED = Workload(
    "llama8b_bf16_batched",
    Shape(n_vocab=128256, n_embd=4096, n_head=32, n_kv_head=8, n_layer=32, n_ff=14336,
          n_ctx=4096 + 64, rope_theta=500000.0, rms_norm_eps=1e-5, dtype=BF16),
    seed=5, batch=64, slot_pos_range=(512, 4096), steps=64)

# the Llama-7B decode step with GGUF Q8_0-style weights (blocks of 32 int8
# values and an fp16 scale); bf16 KV cache
LLAMA7B_Q8 = Workload("llama7b_q8_0", replace(LLAMA7B.shape, dtype=Q8), seed=2, prefill=2048,
                      steps=128)

# the same with GGUF Q4_0-style weights (blocks of 32 4-bit codes and an fp16 scale)
LLAMA7B_Q4 = Workload("llama7b_q4_0", replace(LLAMA7B.shape, dtype=Q4), seed=2, prefill=2048,
                      steps=128)

# Mixtral's decode step with every matrix in Q8_0 / Q4_0 blocks (router and
# experts included; embeddings and norms as the dense quantized models)
MIXTRAL_Q8 = Workload("mixtral8x_top2_q8_0", replace(MIXTRAL.shape, dtype=Q8), seed=4,
                      prefill=4096, steps=128)
MIXTRAL_Q4 = Workload("mixtral8x_top2_q4_0", replace(MIXTRAL.shape, dtype=Q4), seed=4,
                      prefill=4096, steps=128)

ALL = [TINY, LLAMA7B, MISTRAL7B, MIXTRAL, LLAMA8B_BATCHED, LLAMA7B_Q8, LLAMA7B_Q4, MIXTRAL_Q8,
       MIXTRAL_Q4]
BY_NAME = {w.name: w for w in ALL}


# ---------------------------------------------------------------- the recipe

@dataclass(frozen=True)
class TensorSpec:
    """One logical weight tensor [rows][cols] (row-major logical index)."""
    name: str
    kind: int
    layer: int
    sub: int          # expert index (0 for dense tensors)
    rows: int
    cols: int
    const: Optional[float] = None   # constant tensors (norm weights)
    sigma: float = WEIGHT_SIGMA

    def key(self, seed: int) -> int:
        return key(seed, self.kind, self.layer, self.sub)


def weight_specs(shape: Shape) -> List[TensorSpec]:
    """Every logical weight tensor of the model, in a fixed order."""
    E, H, Hkv, hd, F, V = (shape.n_embd, shape.n_head, shape.n_kv_head, shape.head_dim,
                           shape.n_ff, shape.n_vocab)
    out = [TensorSpec("tok_embd", TOK_EMBD, 0, 0, V, E),
           TensorSpec("out_norm", OUT_NORM, 0, 0, 1, E, const=NORM_VALUE),
           TensorSpec("output", OUTPUT, 0, 0, V, E)]
    for l in range(shape.n_layer):
        out += [TensorSpec("attn_norm", ATTN_NORM, l, 0, 1, E, const=NORM_VALUE),
                TensorSpec("wq", WQ, l, 0, H * hd, E),
                TensorSpec("wk", WK, l, 0, Hkv * hd, E),
                TensorSpec("wv", WV, l, 0, Hkv * hd, E),
                TensorSpec("wo", WO, l, 0, E, H * hd),
                TensorSpec("ffn_norm", FFN_NORM, l, 0, 1, E, const=NORM_VALUE)]
        if shape.qkv_bias:
            out += [TensorSpec("bq", BQ, l, 0, 1, H * hd, sigma=BIAS_SIGMA),
                    TensorSpec("bk", BK, l, 0, 1, Hkv * hd, sigma=BIAS_SIGMA),
                    TensorSpec("bv", BV, l, 0, 1, Hkv * hd, sigma=BIAS_SIGMA)]
        if shape.expert_count > 0:
            out.append(TensorSpec("wrouter", WROUTER, l, 0, shape.expert_count, E))
        for e in range(max(1, shape.expert_count)):
            out += [TensorSpec("wgate", WGATE, l, e, F, E),
                    TensorSpec("wup", WUP, l, e, F, E),
                    TensorSpec("wdown", WDOWN, l, e, E, F)]
    return out


def prompt_tokens(w: Workload, slot: int = 0) -> List[int]:
    """Prompt ids (tiny workload) or the single start token (pre-filled workloads)."""
    n = w.prompt_len if w.prompt_len > 0 else 1
    return [int(t) for t in uniform_int(key(w.seed, TOKENS, 0, slot), 0, n, 0, w.shape.n_vocab)]


def slot_positions(w: Workload) -> List[int]:
    """Start position of every slot: the pre-fill length, or uniform in the slot range."""
    if w.slot_pos_range is None:
        return [w.prefill] * w.batch
    lo, hi = w.slot_pos_range
    return [int(p) for p in uniform_int(key(w.seed, POSITIONS, 0, 0), 0, w.batch, lo, hi - lo + 1)]


def kv_prefill_range(shape: Shape, start_pos: int):
    """Positions whose cache contents are generated: the last kv_cap below start_pos."""
    return max(0, start_pos - shape.kv_cap), start_pos
