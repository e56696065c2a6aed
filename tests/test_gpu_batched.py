"""Batched-slot decode step (pnb_forward_batch) against the CPU oracle.

Each slot is an independent sequence with its own KV cache and position; a
batched step must give every slot the logits that a single-sequence step of
that slot gives.  The oracle runs each slot on its own.  Tolerances as in the
single-sequence parity tests (argmax identical unless the oracle's top-2
margin is inside the logit tolerance; max|d logit| <= 2e-2 * max|logit| for
bf16 weights); against the GPU's own single-sequence step the bar is tighter
(1e-3), since both sides use the same weights and fp32 activations and differ
only in the tensor-core path's bf16 high / low split of the activations and
in summation order.
"""
import dataclasses

import numpy as np
import pytest

import oracle
import synth.workloads as wl
from synth import BF16, F32

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import transformer_decode_step_gb300 as pnb  # noqa: E402

DEV = torch.device("cuda:0")
TOL = 2e-2

# E, H * hd and F multiples of 64 (the GEMM's K chunks); V not a multiple of
# the 128-row tile, so the LM head ends in a ragged tile
SHAPE = wl.Shape(n_vocab=3001, n_embd=512, n_head=8, n_kv_head=2, n_layer=2, n_ff=1024,
                 n_ctx=160, rope_theta=1e4, rms_norm_eps=1e-5, dtype=BF16)
SHAPE_WIN = dataclasses.replace(SHAPE, sliding_window=48, n_ctx=200, n_vocab=2000, rope_theta=1e6)
SHAPE_HD128 = wl.Shape(n_vocab=1500, n_embd=1024, n_head=8, n_kv_head=8, n_layer=1, n_ff=1536,
                       n_ctx=300, rope_theta=5e5, rms_norm_eps=1e-5, dtype=BF16)
# head_dim 128 with 8 KV heads: from B = 20 on there are more (slot, KV head)
# items than SMs and the attention runs persistent CTAs that take several
# items each; the window variant reads a 128-slot ring (whole tiles, so the
# tensor-core attention takes it), wrapped for most slots
SHAPE_HD128_WIN = dataclasses.replace(SHAPE_HD128, sliding_window=128, n_ctx=320, rope_theta=1e6)
# MoE: 4 experts, top-2 (the router runs per slot, every expert's FFN over all slots)
SHAPE_MOE = wl.Shape(n_vocab=3001, n_embd=512, n_head=8, n_kv_head=2, n_layer=2, n_ff=1024,
                     n_ctx=160, rope_theta=1e6, rms_norm_eps=1e-5, expert_count=4, expert_used=2,
                     dtype=BF16)
SEED = 31


def starts_for(shape, B, seed):
    rng = np.random.default_rng(seed)
    return [int(p) for p in rng.integers(1, shape.n_ctx - 4, size=B)]


def oracle_slots(shape, starts):
    m = oracle.Model(shape, seed=SEED)
    out = []
    for b, p in enumerate(starts):
        s = m.new_state()
        lo, hi = wl.kv_prefill_range(shape, p)
        s.prefill_synth(SEED, b, lo, hi)
        out.append(s)
    return m, out


def check(ref, ram, got, gam, what, tol=TOL):
    scale = float(np.max(np.abs(ref)))
    err = float(np.max(np.abs(got - ref)))
    assert err <= tol * scale, f"{what}: max|d|={err:.3e} > {tol}*{scale:.3e}"
    if gam != ram:
        top = np.sort(ref)[-2:]
        assert float(top[1] - top[0]) <= tol * scale, f"{what}: argmax {gam} != {ram}"
        return 1
    return 0


def run(shape, B, steps=3):
    starts = starts_for(shape, B, 1000 + B)
    sm = pnb.SynthModel(shape, SEED, device=DEV)
    states = [sm.new_state(p, slot=b) for b, p in enumerate(starts)]
    _, ostates = oracle_slots(shape, starts)
    rng = np.random.default_rng(B)
    tokens = [int(t) for t in rng.integers(0, shape.n_vocab, size=B)]
    V = shape.n_vocab
    lg = torch.empty(B, V, dtype=torch.float32, device=DEV)
    am = torch.empty(B, dtype=torch.int32, device=DEV)
    tk = torch.empty(B, dtype=torch.int32, device=DEV)
    near = 0
    for i in range(steps):
        tk.copy_(torch.tensor(tokens, dtype=torch.int32))
        sm.model.forward_batch(states, tokens=tk, logits=lg, argmax=am)
        got, gam = lg.cpu().numpy(), am.cpu().numpy()
        nxt = []
        for b in range(B):
            ref, ram = ostates[b].forward(tokens[b])
            near += check(ref, ram, got[b], int(gam[b]), f"B={B} step {i} slot {b}")
            nxt.append(ram)
        tokens = nxt
    for b, s in enumerate(states):
        assert s.device_error() == 0
        assert s.pos == starts[b] + steps
    return near


@pytest.mark.parametrize("shape", [SHAPE, SHAPE_WIN, SHAPE_HD128, SHAPE_HD128_WIN, SHAPE_MOE],
                         ids=["gqa", "window", "mha_hd128", "window_hd128", "moe"])
@pytest.mark.parametrize("B", [1, 5, 20, 40])
def test_batched_step_matches_per_slot_oracle(shape, B):
    # argmax may differ only on near-ties (inside the logit tolerance); with
    # these seeds the dense shapes have none, the MoE shape at most one
    assert run(shape, B) <= (1 if shape.expert_count else 0)


@pytest.mark.parametrize("SHAPE", [SHAPE, SHAPE_MOE], ids=["dense", "moe"])
def test_batched_step_matches_single_sequence_steps(SHAPE):
    B = 12
    starts = starts_for(SHAPE, B, 7)
    sm = pnb.SynthModel(SHAPE, SEED, device=DEV)
    bstates = [sm.new_state(p, slot=b) for b, p in enumerate(starts)]
    sstates = [sm.new_state(p, slot=b) for b, p in enumerate(starts)]
    rng = np.random.default_rng(3)
    tokens = [int(t) for t in rng.integers(0, SHAPE.n_vocab, size=B)]
    V = SHAPE.n_vocab
    lg = torch.empty(B, V, dtype=torch.float32, device=DEV)
    am = torch.empty(B, dtype=torch.int32, device=DEV)
    tk = torch.tensor(tokens, dtype=torch.int32, device=DEV)
    one = torch.empty(V, dtype=torch.float32, device=DEV)
    a1 = torch.empty(1, dtype=torch.int32, device=DEV)
    for i in range(3):
        sm.model.forward_batch(bstates, tokens=tk if i == 0 else None, logits=lg, argmax=am)
        got = lg.cpu().numpy()
        for b in range(B):
            sstates[b].forward(tokens[b] if i == 0 else pnb.PNB_TOKEN_PREV, logits=one, argmax=a1)
            ref = one.cpu().numpy()
            check(ref, int(a1.item()), got[b], int(am[b].item()), f"step {i} slot {b}", tol=1e-3)
    assert all(s.device_error() == 0 for s in bstates + sstates)


@pytest.mark.parametrize("shape", [SHAPE, SHAPE_MOE], ids=["dense", "moe"])
@pytest.mark.parametrize("B", [5, 40])
def test_batched_step_is_bitwise_reproducible(shape, B):
    """With pnb_model_set_deterministic_batch the K parts of the residual
    projections add into a fixed-point sum, which does not depend on the order
    of the adds: the same steps from the same states give the same logits, bit
    for bit, and they agree with the default (fp32 atomic) step to rounding."""
    starts = starts_for(shape, B, 77)
    sm = pnb.SynthModel(shape, SEED, device=DEV)
    states = [sm.new_state(p, slot=b) for b, p in enumerate(starts)]
    tokens = [int(t) for t in np.random.default_rng(9).integers(0, shape.n_vocab, size=B)]
    tk = torch.tensor(tokens, dtype=torch.int32, device=DEV)
    lg = torch.empty(B, shape.n_vocab, dtype=torch.float32, device=DEV)
    runs = []
    for det in (True, True, False):
        sm.model.set_deterministic_batch(det)
        for b, st in enumerate(states):
            st.set_pos(starts[b])
        out = []
        for i in range(3):
            sm.model.forward_batch(states, tokens=tk if i == 0 else None, logits=lg)
            out.append(lg.clone())
        runs.append(torch.stack(out))
    sm.model.set_deterministic_batch(False)
    assert all(st.device_error() == 0 for st in states)
    assert torch.equal(runs[0], runs[1])
    scale = runs[0].abs().max().item()
    assert (runs[0] - runs[2]).abs().max().item() <= 1e-3 * scale


def test_batched_step_continues_from_each_slots_own_argmax():
    """tokens=None: every slot feeds back its previous greedy token on the device."""
    B = 6
    starts = starts_for(SHAPE, B, 11)
    sm = pnb.SynthModel(SHAPE, SEED, device=DEV)
    states = [sm.new_state(p, slot=b) for b, p in enumerate(starts)]
    _, ostates = oracle_slots(SHAPE, starts)
    tokens = [int(t) for t in np.random.default_rng(5).integers(0, SHAPE.n_vocab, size=B)]
    lg = torch.empty(B, SHAPE.n_vocab, dtype=torch.float32, device=DEV)
    am = torch.empty(B, dtype=torch.int32, device=DEV)
    sm.model.forward_batch(states, tokens=torch.tensor(tokens, dtype=torch.int32, device=DEV),
                           logits=lg, argmax=am)
    nxt = [ostates[b].forward(tokens[b])[1] for b in range(B)]
    assert am.cpu().tolist() == nxt
    for i in range(2):
        sm.model.forward_batch(states, logits=lg, argmax=am)
        got = lg.cpu().numpy()
        step = [ostates[b].forward(nxt[b]) for b in range(B)]
        for b in range(B):
            check(step[b][0], step[b][1], got[b], int(am[b].item()), f"step {i} slot {b}")
        nxt = [r[1] for r in step]


def test_batched_errors():
    sm = pnb.SynthModel(SHAPE, SEED, device=DEV)
    s0, s1 = sm.new_state(5), sm.new_state(9, slot=1)
    with pytest.raises(pnb.PnbError) as e:
        sm.model.forward_batch([s0, s0])
    assert e.value.code == -1
    with pytest.raises(pnb.PnbError) as e:
        sm.model.forward_batch([s0] * 65)
    assert e.value.code == -1
    f32 = dataclasses.replace(SHAPE, dtype=F32)
    fm = pnb.SynthModel(f32, 3, device=DEV)
    with pytest.raises(pnb.PnbError) as e:
        fm.model.forward_batch([fm.new_state(3)])
    assert e.value.code == -5
    full = sm.new_state(SHAPE.n_ctx - 1, slot=2)
    sm.model.forward_batch([s1, full])        # the last free position
    with pytest.raises(pnb.PnbError) as e:
        sm.model.forward_batch([s1, full])
    assert e.value.code == -4


def test_full_size_batched_first_step_matches_oracle():
    """The batched workload's own model: 64 slots at their seeded positions, one
    step; sampled slots against the oracle."""
    w = wl.LLAMA8B_BATCHED
    B = w.batch
    starts = wl.slot_positions(w)
    sm = pnb.SynthModel(w.shape, w.seed, device=DEV)
    states = [sm.new_state(p, slot=b) for b, p in enumerate(starts)]
    tokens = [wl.prompt_tokens(w, b)[0] for b in range(B)]
    lg = torch.empty(B, w.shape.n_vocab, dtype=torch.float32, device=DEV)
    am = torch.empty(B, dtype=torch.int32, device=DEV)
    sm.model.forward_batch(states, tokens=torch.tensor(tokens, dtype=torch.int32, device=DEV),
                           logits=lg, argmax=am)
    got, gam = lg.cpu().numpy(), am.cpu().numpy()
    assert all(s.device_error() == 0 for s in states)
    del states, sm
    torch.cuda.empty_cache()
    ref_model = oracle.Model(w.shape, seed=w.seed)
    for b in (0, 37, B - 1):
        s = ref_model.new_state()
        lo, hi = wl.kv_prefill_range(w.shape, starts[b])
        s.prefill_synth(w.seed, b, lo, hi)
        ref, ram = s.forward(tokens[b])
        assert check(ref, ram, got[b], int(gam[b]), f"slot {b}") == 0
