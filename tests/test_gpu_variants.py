"""Architecture variants on the same decode seam, against the CPU oracle:
q / k / v biases (Qwen2) and NeoX-style RoPE (Phi-3).

The oracle adds the biases before RoPE and rotates the NeoX pairs (i, i + hd/2)
in their natural order; the GPU library rotates adjacent pairs of a layout in
which each head's Wq / Wk rows come interleaved (0, hd/2, 1, hd/2 + 1, ...),
which the test model generator produces from the same generated values.  So a
NeoX model's cache is in that interleaved order, and NeoX cases start from an
empty cache (the generated pre-filled caches follow the library's layout, not
the oracle's).  Bars as in the other parity tests: max|d logit| <= 2e-2 *
max|logit| for bf16 / Q8 weights and 1e-3 for fp32, argmax identical unless the
oracle's top-2 margin is inside that tolerance.
"""
import dataclasses

import numpy as np
import pytest

import oracle
import synth.workloads as wl
from synth import BF16, F32, Q8

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import transformer_decode_step_gb300 as pnb  # noqa: E402

DEV = torch.device("cuda:0")
SEED = 29

BASE = wl.Shape(n_vocab=3001, n_embd=512, n_head=8, n_kv_head=2, n_layer=2, n_ff=1024,
                n_ctx=160, rope_theta=1e6, rms_norm_eps=1e-6, dtype=BF16)
QWEN2 = dataclasses.replace(BASE, qkv_bias=True)
PHI3 = dataclasses.replace(BASE, n_kv_head=8, rope_theta=1e4, rope_neox=True)
BOTH = dataclasses.replace(BASE, qkv_bias=True, rope_neox=True, sliding_window=24)
QWEN2_Q8 = dataclasses.replace(QWEN2, dtype=Q8)
PHI3_F32 = dataclasses.replace(PHI3, dtype=F32, n_vocab=1000, n_layer=1)
QWEN2_HD128 = wl.Shape(n_vocab=1500, n_embd=1024, n_head=8, n_kv_head=4, n_layer=1, n_ff=1536,
                       n_ctx=300, rope_theta=1e6, rms_norm_eps=1e-6, dtype=BF16, qkv_bias=True)


def tol(shape):
    return 1e-3 if shape.dtype == F32 else 2e-2


def check(ref, ram, got, gam, what, t):
    scale = float(np.max(np.abs(ref)))
    err = float(np.max(np.abs(got - ref)))
    assert err <= t * scale, f"{what}: max|d|={err:.3e} > {t}*{scale:.3e}"
    if gam != ram:
        top = np.sort(ref)[-2:]
        assert float(top[1] - top[0]) <= t * scale, f"{what}: argmax {gam} vs {ram}"


def oracle_steps(shape, start, tokens, slot=0):
    m = oracle.Model(shape, seed=SEED)
    s = m.new_state()
    if start:
        lo, hi = wl.kv_prefill_range(shape, start)
        s.prefill_synth(SEED, slot, lo, hi)
    return [s.forward(int(t)) for t in tokens]


def gpu_steps(sm, start, tokens, slot=0):
    st = sm.new_state(start, slot=slot)
    V = sm.shape.n_vocab
    lg = torch.empty(V, dtype=torch.float32, device=DEV)
    am = torch.empty(1, dtype=torch.int32, device=DEV)
    out = []
    for t in tokens:
        st.forward(int(t), logits=lg, argmax=am)
        out.append((lg.cpu().numpy().copy(), int(am.item())))
    assert st.device_error() == 0
    return out


@pytest.mark.parametrize("name,shape,start,steps", [
    ("qwen2_gqa", QWEN2, 37, 12),
    ("qwen2_hd128", QWEN2_HD128, 120, 8),
    ("qwen2_q8", QWEN2_Q8, 21, 8),
    ("phi3_mha_neox", PHI3, 0, 24),
    ("phi3_neox_f32", PHI3_F32, 0, 20),
    ("bias_neox_window_ring", BOTH, 0, 40),     # a 24-slot ring, wrapped
])
def test_variant_models_match_oracle(name, shape, start, steps):
    rng = np.random.default_rng(steps + start)
    tokens = [int(t) for t in rng.integers(0, shape.n_vocab, size=steps)]
    sm = pnb.SynthModel(shape, SEED, device=DEV)
    got = gpu_steps(sm, start, tokens)
    ref = oracle_steps(shape, start, tokens)
    for i, ((g, ga), (r, ra)) in enumerate(zip(got, ref)):
        check(r, ra, g, ga, f"{name} step {i}", tol(shape))


def test_variant_flags_matter_on_the_gpu():
    """The same generated weights without the bias, or with the Llama rotation,
    give other logits: the kernels do use the bias and the layout."""
    rng = np.random.default_rng(4)
    tokens = [int(t) for t in rng.integers(0, BASE.n_vocab, size=6)]
    last = {}
    for name, shape in (("plain", BASE), ("bias", QWEN2), ("neox", dataclasses.replace(BASE, rope_neox=True))):
        last[name] = gpu_steps(pnb.SynthModel(shape, SEED, device=DEV), 0, tokens)[-1][0]
    for other in ("bias", "neox"):
        assert not np.allclose(last["plain"], last[other], atol=1e-3)


@pytest.mark.parametrize("shape", [QWEN2, BOTH])
def test_batched_variant_slots_equal_single_sequence_steps(shape):
    B = 5
    rng = np.random.default_rng(9)
    prompts = [[int(t) for t in rng.integers(0, shape.n_vocab, size=int(n))]
               for n in rng.integers(2, 9, size=B)]
    sm = pnb.SynthModel(shape, SEED, device=DEV)
    V = shape.n_vocab
    bstates, sstates = [], []
    for p in prompts:
        for lst in (bstates, sstates):
            st = sm.new_state(0)
            for t in p:
                st.forward(t)
            lst.append(st)
    toks = [int(t) for t in rng.integers(0, V, size=B)]
    lg = torch.empty(B, V, dtype=torch.float32, device=DEV)
    am = torch.empty(B, dtype=torch.int32, device=DEV)
    one = torch.empty(V, dtype=torch.float32, device=DEV)
    a1 = torch.empty(1, dtype=torch.int32, device=DEV)
    first = None
    for i in range(3):
        sm.model.forward_batch(bstates, tokens=torch.tensor(toks, dtype=torch.int32, device=DEV)
                               if i == 0 else None, logits=lg, argmax=am)
        got = lg.cpu().numpy()
        if i == 0:
            first = (got[0].copy(), int(am[0].item()))
        for b in range(B):
            sstates[b].forward(toks[b] if i == 0 else pnb.PNB_TOKEN_PREV, logits=one, argmax=a1)
            check(one.cpu().numpy(), int(a1.item()), got[b], int(am[b].item()),
                  f"step {i} slot {b}", 1e-3)
    assert all(st.device_error() == 0 for st in bstates + sstates)
    # slot 0's first batched step against the oracle fed the same tokens
    r, ra = oracle_steps(shape, 0, prompts[0] + [toks[0]])[-1]
    check(r, ra, first[0], first[1], "slot 0 against the oracle", tol(shape))


@pytest.mark.parametrize("shape", [QWEN2, dataclasses.replace(PHI3, n_ctx=200)])
def test_variant_prefill_matches_oracle(shape):
    rng = np.random.default_rng(13)
    T = 70                                     # two chunks
    tokens = [int(t) for t in rng.integers(0, shape.n_vocab, size=T)]
    sm = pnb.SynthModel(shape, SEED, device=DEV)
    st = sm.new_state(0)
    lg = torch.empty(T, shape.n_vocab, dtype=torch.float32, device=DEV)
    am = torch.empty(T, dtype=torch.int32, device=DEV)
    st.prefill(torch.tensor(tokens, dtype=torch.int32, device=DEV), logits=lg, argmax=am)
    assert st.device_error() == 0
    ref = oracle_steps(shape, 0, tokens)
    got, gam = lg.cpu().numpy(), am.cpu().numpy()
    for i, (r, ra) in enumerate(ref):
        check(r, ra, got[i], int(gam[i]), f"token {i}", tol(shape))


def test_neox_with_either_attention_kernel_matches_oracle():
    """Phi-3-style NeoX RoPE with the tensor-core and the CUDA-core attention."""
    rng = np.random.default_rng(21)
    tokens = [int(t) for t in rng.integers(0, PHI3.n_vocab, size=10)]
    ref = oracle_steps(PHI3, 0, tokens)
    sm = pnb.SynthModel(PHI3, SEED, device=DEV)
    kinds = [False] + ([True] if sm.model.tensor_attention else [])
    for tc in kinds:
        sm.model.set_tensor_attention(tc)
        for i, ((g, ga), (r, ra)) in enumerate(zip(gpu_steps(sm, 0, tokens), ref)):
            check(r, ra, g, ga, f"tensor attention {tc} step {i}", tol(PHI3))
