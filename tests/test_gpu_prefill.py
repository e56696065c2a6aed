"""Prefill (pnb_prefill) against the CPU oracle and against single-sequence steps.

A prefill of T prompt tokens must leave the state exactly where T decode steps
would: the same KV cache contents, position and next token, with each token's
logits those of a step.  The oracle runs the tokens one at a time (its
definition of the forward).  Chunks of up to 64 tokens run as one batched step
of virtual slots sharing the state's cache, so the tolerances are the batched
step's: against the oracle, argmax identical unless the oracle's top-2 margin
is inside the logit tolerance and max|d logit| <= 2e-2 * max|logit| (bf16
weights); against the GPU's own single-sequence steps, 1e-3.
"""
import dataclasses

import numpy as np
import pytest

import oracle
import synth.workloads as wl
from synth import BF16

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import transformer_decode_step_gb300 as pnb  # noqa: E402

DEV = torch.device("cuda:0")
TOL = 2e-2
SEED = 41

# E, H * hd and F multiples of 64 (the batched GEMM's K chunks)
SHAPE = wl.Shape(n_vocab=3001, n_embd=512, n_head=8, n_kv_head=2, n_layer=2, n_ff=1024,
                 n_ctx=260, rope_theta=1e4, rms_norm_eps=1e-5, dtype=BF16)
SHAPE_HD128 = wl.Shape(n_vocab=1500, n_embd=1024, n_head=8, n_kv_head=8, n_layer=1, n_ff=1536,
                       n_ctx=300, rope_theta=5e5, rms_norm_eps=1e-5, dtype=BF16)
# a 48-slot ring: chunks stop where the ring would wrap, then one token per step
SHAPE_WIN = dataclasses.replace(SHAPE, sliding_window=48, n_ctx=200, n_vocab=2000, rope_theta=1e6)
# long prompts: chunks past position 256 run the tensor-core attention with
# token groups (2 tokens per KV-head pass at 4 query heads per KV head, 8 at MHA)
SHAPE_LONG = dataclasses.replace(SHAPE, n_ctx=600)
SHAPE_HD128_LONG = dataclasses.replace(SHAPE_HD128, n_ctx=600)
# MoE: chunks through the batched step's router and per-expert FFNs
SHAPE_MOE = wl.Shape(n_vocab=777, n_embd=256, n_head=4, n_kv_head=2, n_layer=2, n_ff=512,
                     n_ctx=128, rope_theta=1e6, rms_norm_eps=1e-5, expert_count=4, expert_used=2,
                     dtype=BF16)


def oracle_run(shape, start, tokens):
    """Teacher-forced logits of every token, then the greedy step after the last."""
    m = oracle.Model(shape, seed=SEED)
    s = m.new_state()
    lo, hi = wl.kv_prefill_range(shape, start)
    s.prefill_synth(SEED, 0, lo, hi)
    out = [s.forward(t) for t in tokens]
    nxt = s.forward(out[-1][1])
    return out, nxt


def check(ref, ram, got, gam, what, tol=TOL):
    scale = float(np.max(np.abs(ref)))
    err = float(np.max(np.abs(got - ref)))
    assert err <= tol * scale, f"{what}: max|d|={err:.3e} > {tol}*{scale:.3e}"
    if gam != ram:   # only a near-tie may differ
        top = np.sort(ref)[-2:]
        assert float(top[1] - top[0]) <= tol * scale, f"{what}: argmax {gam} vs {ram}"


def gpu_prefill(sm, start, tokens):
    V = sm.shape.n_vocab
    st = sm.new_state(start)
    tk = torch.tensor(tokens, dtype=torch.int32, device=DEV)
    lg = torch.empty(len(tokens), V, dtype=torch.float32, device=DEV)
    am = torch.empty(len(tokens), dtype=torch.int32, device=DEV)
    st.prefill(tk, logits=lg, argmax=am)
    assert st.pos == start + len(tokens)
    # the next step continues from the last token's argmax on the device
    lg1 = torch.empty(V, dtype=torch.float32, device=DEV)
    am1 = torch.empty(1, dtype=torch.int32, device=DEV)
    st.forward(pnb.PNB_TOKEN_PREV, logits=lg1, argmax=am1)
    out = (lg.cpu().numpy(), am.cpu().numpy(), lg1.cpu().numpy(), int(am1.item()))
    assert st.device_error() == 0
    return out, st


@pytest.mark.parametrize("name,shape,start,T", [
    ("gqa_one", SHAPE, 37, 1),
    ("gqa_7", SHAPE, 0, 7),
    ("gqa_64", SHAPE, 90, 64),
    ("gqa_100_two_chunks", SHAPE, 21, 100),
    ("mha_hd128_70", SHAPE_HD128, 150, 70),
    ("ring_fills_then_wraps", SHAPE_WIN, 0, 70),
    ("ring_partial_chunk", SHAPE_WIN, 30, 40),
    ("moe", SHAPE_MOE, 5, 9),
    ("gqa_512", SHAPE_LONG, 0, 512),
    ("mha_hd128_512", SHAPE_HD128_LONG, 0, 512),
    # a chunk that starts off the 64-token grid and crosses position 256: its
    # new K / V span two cache tiles, loaded only after the QKV kernel ends
    ("mha_hd128_unaligned", SHAPE_HD128, 150, 140),
    ("gqa_unaligned_from_cache", SHAPE_LONG, 230, 90),
])
def test_prefill_matches_oracle(name, shape, start, T):
    rng = np.random.default_rng(T + start)
    tokens = [int(t) for t in rng.integers(0, shape.n_vocab, size=T)]
    sm = pnb.SynthModel(shape, SEED, device=DEV)
    (lg, am, lg1, am1), _ = gpu_prefill(sm, start, tokens)
    ref, (rl1, ra1) = oracle_run(shape, start, tokens)
    for i, (rl, ra) in enumerate(ref):
        check(rl, ra, lg[i], int(am[i]), f"{name} token {i}")
    if int(am[-1]) == ref[-1][1]:   # same greedy token: the next step is comparable
        check(rl1, ra1, lg1, am1, f"{name} next step")


@pytest.mark.parametrize("shape,start,T", [(SHAPE, 11, 100), (SHAPE_HD128, 40, 64),
                                           (SHAPE_HD128_LONG, 200, 130)])
def test_prefill_equals_single_sequence_steps(shape, start, T):
    rng = np.random.default_rng(3)
    tokens = [int(t) for t in rng.integers(0, shape.n_vocab, size=T)]
    sm = pnb.SynthModel(shape, SEED, device=DEV)
    (lg, am, lg1, am1), _ = gpu_prefill(sm, start, tokens)
    st = sm.new_state(start)
    V = shape.n_vocab
    out = torch.empty(V, dtype=torch.float32, device=DEV)
    a1 = torch.empty(1, dtype=torch.int32, device=DEV)
    for i, t in enumerate(tokens):
        st.forward(t, logits=out, argmax=a1)
        check(out.cpu().numpy(), int(a1.item()), lg[i], int(am[i]), f"step {i}", tol=1e-3)
    st.forward(pnb.PNB_TOKEN_PREV, logits=out, argmax=a1)
    check(out.cpu().numpy(), int(a1.item()), lg1, am1, "next step", tol=1e-3)
    assert st.pos == start + T + 1


def test_prefill_without_outputs_and_errors():
    sm = pnb.SynthModel(SHAPE, SEED, device=DEV)
    st = sm.new_state(5)
    tk = torch.arange(20, dtype=torch.int32, device=DEV)
    st.prefill(tk)                       # no logits / argmax buffers
    assert st.pos == 25 and st.device_error() == 0
    # T < 1 (through the C ABI: an empty tensor has no data pointer)
    assert pnb.pnb_prefill(sm.model.handle, st._h, tk.data_ptr(), 0, None, None, None) == -1
    st.set_pos(SHAPE.n_ctx - 10)
    with pytest.raises(pnb.PnbError) as e:
        st.prefill(tk)                   # 20 tokens do not fit
    assert e.value.code == -4
    bad = torch.full((3,), SHAPE.n_vocab, dtype=torch.int32, device=DEV)
    st2 = sm.new_state(0)
    st2.prefill(bad)                     # out-of-range tokens: token 0 used, error bit set
    assert st2.device_error() & pnb.PNB_DEV_ERR_TOKEN
