"""Q8 (GGUF Q8_0-style) weights: the decode step against the CPU oracle.

The oracle multiplies by exactly the weights the GPU holds (each block's fp16
scale times its int8 values, from the same seeded generator), so the only
difference is the GPU's fp32 accumulation and bf16 KV cache (MoE models: the
router and the experts in the same blocks): the bf16 bar
applies (argmax identical unless the oracle's top-2 margin is inside the
logit tolerance; max|d logit| <= 2e-2 * max|logit|).
"""
import dataclasses

import numpy as np
import pytest

import oracle
import synth
import synth.workloads as wl
from synth import Q8

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import transformer_decode_step_gb300 as pnb  # noqa: E402

DEV = torch.device("cuda:0")
TOL = 2e-2

# n_embd and n_ff multiples of 256 (whole 16-byte vectors of a Q8 row)
Q8_GQA = wl.Shape(n_vocab=3001, n_embd=512, n_head=8, n_kv_head=2, n_layer=2, n_ff=1024,
                  n_ctx=96, rope_theta=1e4, rms_norm_eps=1e-5, dtype=Q8)
Q8_WIN = dataclasses.replace(Q8_GQA, sliding_window=24, n_vocab=2000, rope_theta=1e6)
Q8_MHA128 = wl.Shape(n_vocab=1500, n_embd=1024, n_head=8, n_kv_head=8, n_layer=2, n_ff=1536,
                     n_ctx=300, rope_theta=5e5, rms_norm_eps=1e-5, dtype=Q8)
# MoE: router and experts in Q8 blocks too (top-2 of 4; top-2 of 8 with a window ring)
Q8_MOE = wl.Shape(n_vocab=1200, n_embd=512, n_head=8, n_kv_head=2, n_layer=2, n_ff=768,
                  n_ctx=96, rope_theta=1e6, rms_norm_eps=1e-5, expert_count=4, expert_used=2,
                  dtype=Q8)
Q8_MOE8_WIN = dataclasses.replace(Q8_MOE, expert_count=8, sliding_window=32, n_vocab=900)
# rows of 11008 values (the Llama-7B down projection): one row per ring slot
Q8_WIDE_FF = wl.Shape(n_vocab=1000, n_embd=512, n_head=4, n_kv_head=4, n_layer=1, n_ff=11008,
                      n_ctx=64, rope_theta=1e4, rms_norm_eps=1e-5, dtype=Q8)


def test_device_q8_fill_equals_host_fill():
    rows, cols = 37, 512
    rb = cols + cols // 16
    buf = torch.zeros(2 * rows * rb, dtype=torch.uint8, device=DEV)
    k = synth.key(9, synth.WGATE, 3, 1)
    synth.dev_fill_matrix(buf.data_ptr(), Q8, 1, 2, rows, cols, k, 0.02,
                          torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    raw, _ = synth.q8_rows(k, 0, rows, cols, 0.02)
    dev = buf.cpu().numpy().reshape(2 * rows, rb)
    assert np.array_equal(dev[1::2], raw)
    assert np.all(dev[0::2] == 0)


def run_both(shape, seed, start, tokens):
    sm = pnb.SynthModel(shape, seed, device=DEV)
    st = sm.new_state(start)
    V = shape.n_vocab
    lg = torch.empty(V, dtype=torch.float32, device=DEV)
    a = torch.empty(1, dtype=torch.int32, device=DEV)
    got, gam = [], []
    for t in tokens:
        st.forward(int(t), logits=lg, argmax=a)
        got.append(lg.cpu().numpy().copy())
        gam.append(int(a.item()))
    assert st.device_error() == 0
    m = oracle.Model(shape, seed=seed)
    s = m.new_state()
    if start:
        lo, hi = wl.kv_prefill_range(shape, start)
        s.prefill_synth(seed, 0, lo, hi)
    ref = [s.forward(int(t)) for t in tokens]
    return sm, got, gam, [r[0] for r in ref], [r[1] for r in ref]


def compare(got, gam, ref, ram, what):
    ties = 0
    for i, (g, r) in enumerate(zip(got, ref)):
        scale = float(np.max(np.abs(r)))
        err = float(np.max(np.abs(g - r)))
        assert err <= TOL * scale, f"{what} step {i}: max|d|={err:.3e} > {TOL}*{scale:.3e}"
        if gam[i] != ram[i]:
            top = np.sort(r)[-2:]
            assert float(top[1] - top[0]) <= TOL * scale, f"{what} step {i}: argmax"
            ties += 1
    return ties


@pytest.mark.parametrize("name,shape,start,steps", [
    ("gqa", Q8_GQA, 40, 12),
    ("window_ring", Q8_WIN, 40, 16),       # ring of 24 slots, already wrapped
    ("mha_hd128", Q8_MHA128, 250, 8),
    ("wide_ff", Q8_WIDE_FF, 9, 6),
    ("moe", Q8_MOE, 30, 10),
    ("moe8_window_ring", Q8_MOE8_WIN, 40, 12),   # ring of 32 slots, already wrapped
])
def test_small_q8_models_match_oracle(name, shape, start, steps):
    rng = np.random.default_rng(17)
    tokens = [int(t) for t in rng.integers(0, shape.n_vocab, size=steps)]
    _, got, gam, ref, ram = run_both(shape, 23, start, tokens)
    assert compare(got, gam, ref, ram, name) <= 1


def test_llama7b_q8_first_steps_match_oracle():
    """The Q8 benchmark model and cache: the first two greedy steps, teacher-forced."""
    w = wl.LLAMA7B_Q8
    m = oracle.Model(w.shape, seed=w.seed)
    s = m.new_state()
    lo, hi = wl.kv_prefill_range(w.shape, w.prefill)
    s.prefill_synth(w.seed, 0, lo, hi)
    tokens = [wl.prompt_tokens(w)[0]]
    ref, ram = [], []
    for i in range(2):
        lg, am = s.forward(tokens[-1])
        ref.append(lg)
        ram.append(am)
        tokens.append(am)
    del s, m
    sm = pnb.SynthModel(w.shape, w.seed, device=DEV)
    st = sm.new_state(w.prefill)
    V = w.shape.n_vocab
    lg = torch.empty(V, dtype=torch.float32, device=DEV)
    a = torch.empty(1, dtype=torch.int32, device=DEV)
    got, gam = [], []
    for t in tokens[:2]:
        st.forward(int(t), logits=lg, argmax=a)
        got.append(lg.cpu().numpy().copy())
        gam.append(int(a.item()))
    assert st.device_error() == 0
    assert compare(got, gam, ref, ram, w.name) == 0
    del st, sm
    torch.cuda.empty_cache()


def test_mixtral_q8_first_step_matches_oracle():
    """Mixtral with every matrix in Q8 blocks (router and experts included): the
    first greedy step from the pre-filled cache, teacher-forced."""
    w = wl.MIXTRAL_Q8
    m = oracle.Model(w.shape, seed=w.seed)
    s = m.new_state()
    lo, hi = wl.kv_prefill_range(w.shape, w.prefill)
    s.prefill_synth(w.seed, 0, lo, hi)
    tok = wl.prompt_tokens(w)[0]
    ref, ram = s.forward(tok)
    del s, m
    sm = pnb.SynthModel(w.shape, w.seed, device=DEV)
    st = sm.new_state(w.prefill)
    lg = torch.empty(w.shape.n_vocab, dtype=torch.float32, device=DEV)
    a = torch.empty(1, dtype=torch.int32, device=DEV)
    st.forward(int(tok), logits=lg, argmax=a)
    got = lg.cpu().numpy().copy()
    assert st.device_error() == 0
    assert compare([got], [int(a.item())], [ref], [ram], w.name) == 0
    del st, sm
    torch.cuda.empty_cache()


def test_q8_forms_and_limits():
    sm = pnb.SynthModel(Q8_GQA, 5, device=DEV)
    states = [sm.new_state(3), sm.new_state(4)]
    with pytest.raises(pnb.PnbError) as e:
        sm.model.forward_batch(states)
    assert e.value.code == -5
    # prefill goes one token per step and equals the steps
    toks = [3, 99, 1500, 7, 42]
    st = sm.new_state(10)
    lg = torch.empty(len(toks), Q8_GQA.n_vocab, dtype=torch.float32, device=DEV)
    st.prefill(torch.tensor(toks, dtype=torch.int32, device=DEV), logits=lg)
    st2 = sm.new_state(10)
    one = torch.empty(Q8_GQA.n_vocab, dtype=torch.float32, device=DEV)
    for i, t in enumerate(toks):
        st2.forward(t, logits=one)
        assert torch.equal(one, lg[i])
    with pytest.raises(pnb.PnbError) as e:   # rows not whole 16-byte vectors
        pnb.SynthModel(dataclasses.replace(Q8_GQA, n_ff=1056), 5, device=DEV)
    assert e.value.code == -5
    # MoE: no batched form either; prefill one token per step, equal to the steps
    sm = pnb.SynthModel(Q8_MOE, 5, device=DEV)
    with pytest.raises(pnb.PnbError) as e:
        sm.model.forward_batch([sm.new_state(3), sm.new_state(4)])
    assert e.value.code == -5
    st = sm.new_state(10)
    lg = torch.empty(len(toks), Q8_MOE.n_vocab, dtype=torch.float32, device=DEV)
    tk = [t % Q8_MOE.n_vocab for t in toks]
    st.prefill(torch.tensor(tk, dtype=torch.int32, device=DEV), logits=lg)
    st2 = sm.new_state(10)
    one = torch.empty(Q8_MOE.n_vocab, dtype=torch.float32, device=DEV)
    for i, t in enumerate(tk):
        st2.forward(t, logits=one)
        assert torch.equal(one, lg[i])
