"""Tensor-core decode attention (tcgen05) against the oracle and against the
CUDA-core attention kernel, through the C ABI.

The tensor-core kernel covers bf16 caches with head_dim 64 or 128, 1, 2, 4 or
8 query heads per KV head, and sliding windows whose ring holds whole
128-position tiles.  Every shape here runs whole decode steps both ways:
against the oracle with the bf16 parity bar (argmax identical, max|d logit|
<= 2e-2 * max|logit|), and the two GPU attention kernels against each other
with a tighter bar (1e-3), since they differ only in the tensor-core path's
bf16 high / low split of the queries and softmax weights and in summation
order.
"""
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
SEED = 53

SHAPES = {
    # ring of 128 positions, wrapped several times (start 300)
    "window128_gqa4_hd64": (wl.Shape(n_vocab=1200, n_embd=512, n_head=8, n_kv_head=2, n_layer=2, n_ff=768,
                                     n_ctx=400, rope_theta=1e4, rms_norm_eps=1e-5, sliding_window=128,
                                     dtype=BF16), 300),
    "gqa4_hd128": (wl.Shape(n_vocab=1500, n_embd=1024, n_head=8, n_kv_head=2, n_layer=2, n_ff=1024,
                            n_ctx=700, rope_theta=1e6, rms_norm_eps=1e-5, dtype=BF16), 520),
    "mha_hd128": (wl.Shape(n_vocab=1000, n_embd=1024, n_head=8, n_kv_head=8, n_layer=1, n_ff=1024,
                           n_ctx=300, rope_theta=1e4, rms_norm_eps=1e-5, dtype=BF16), 131),
    "gqa8_hd128": (wl.Shape(n_vocab=800, n_embd=2048, n_head=16, n_kv_head=2, n_layer=1, n_ff=1024,
                            n_ctx=260, rope_theta=1e4, rms_norm_eps=1e-5, dtype=BF16), 200),
    "gqa2_hd64_short": (wl.Shape(n_vocab=900, n_embd=512, n_head=8, n_kv_head=4, n_layer=2, n_ff=512,
                                 n_ctx=64, rope_theta=1e4, rms_norm_eps=1e-5, dtype=BF16), 3),
}


def steps(sm, state, tokens):
    V = sm.shape.n_vocab
    lg = torch.empty(V, dtype=torch.float32, device=DEV)
    a = torch.empty(1, dtype=torch.int32, device=DEV)
    out = []
    for t in tokens:
        state.forward(int(t), logits=lg, argmax=a)
        out.append((lg.cpu().numpy().copy(), int(a.item())))
    assert state.device_error() == 0
    return out


def close(ref, got, tol, what):
    scale = float(np.max(np.abs(ref)))
    err = float(np.max(np.abs(got - ref)))
    assert err <= tol * scale, f"{what}: max|d|={err:.3e} > {tol}*{scale:.3e}"


@pytest.mark.parametrize("name", list(SHAPES))
def test_tensor_attention_matches_oracle_and_cuda_core_kernel(name):
    shape, start = SHAPES[name]
    sm = pnb.SynthModel(shape, SEED, device=DEV)
    assert sm.model.tensor_attention, "the tensor-core kernel should cover this shape"
    om = oracle.Model(shape, seed=SEED)
    os_ = om.new_state()
    lo, hi = wl.kv_prefill_range(shape, start)
    os_.prefill_synth(SEED, 0, lo, hi)
    tokens = [int(t) for t in np.random.default_rng(7).integers(0, shape.n_vocab, size=1)]
    ref = []
    for i in range(4):
        lg, am = os_.forward(tokens[-1])
        ref.append((lg, am))
        tokens.append(am)
    tokens = tokens[:4]
    tc = steps(sm, sm.new_state(start), tokens)
    sm.model.set_tensor_attention(False)
    cc = steps(sm, sm.new_state(start), tokens)
    sm.model.set_tensor_attention(True)
    for i, ((rl, ra), (tl, ta), (cl, ca)) in enumerate(zip(ref, tc, cc)):
        close(rl, tl, 2e-2, f"{name} step {i} tensor vs oracle")
        close(cl, tl, 1e-3, f"{name} step {i} tensor vs CUDA-core")
        if ta != ra:   # only inside the logit tolerance (a near-tie)
            top = np.sort(rl)[-2:]
            assert float(top[1] - top[0]) <= 2e-2 * float(np.max(np.abs(rl))), f"{name} step {i}: argmax"



def test_tensor_attention_batched_ring_matches_oracle():
    shape, _ = SHAPES["window128_gqa4_hd64"]
    B = 5
    rng = np.random.default_rng(19)
    starts = [int(p) for p in rng.integers(1, shape.n_ctx - 4, size=B)]
    sm = pnb.SynthModel(shape, SEED, device=DEV)
    states = [sm.new_state(p, slot=b) for b, p in enumerate(starts)]
    om = oracle.Model(shape, seed=SEED)
    ostates = []
    for b, p in enumerate(starts):
        s = om.new_state()
        lo, hi = wl.kv_prefill_range(shape, p)
        s.prefill_synth(SEED, b, lo, hi)
        ostates.append(s)
    tokens = [int(t) for t in rng.integers(0, shape.n_vocab, size=B)]
    lg = torch.empty(B, shape.n_vocab, dtype=torch.float32, device=DEV)
    am = torch.empty(B, dtype=torch.int32, device=DEV)
    tk = torch.empty(B, dtype=torch.int32, device=DEV)
    for i in range(3):
        tk.copy_(torch.tensor(tokens, dtype=torch.int32))
        sm.model.forward_batch(states, tokens=tk, logits=lg, argmax=am)
        got, gam = lg.cpu().numpy(), am.cpu().numpy()
        nxt = []
        for b in range(B):
            ref, ram = ostates[b].forward(tokens[b])
            close(ref, got[b], 2e-2, f"step {i} slot {b}")
            assert int(gam[b]) == ram
            nxt.append(ram)
        tokens = nxt
    assert all(s.device_error() == 0 for s in states)


def test_tensor_attention_setting_is_rejected_where_not_covered():
    shape = wl.Shape(n_vocab=500, n_embd=512, n_head=8, n_kv_head=2, n_layer=1, n_ff=512, n_ctx=96,
                     sliding_window=24, dtype=BF16)   # a 24-slot ring does not hold whole tiles
    sm = pnb.SynthModel(shape, 3, device=DEV)
    assert not sm.model.tensor_attention
    with pytest.raises(pnb.PnbError) as e:
        sm.model.set_tensor_attention(True)
    assert e.value.code == -5
