"""GPU decode step vs the CPU oracle, through the C ABI.

Tolerances: argmax identical; max |logit_gpu - logit_oracle| <= 1e-3 * max|logit|
for fp32 weights and <= 2e-2 * max|logit| for bf16 weights.  Both sides get the
same token sequence (teacher forcing), so every step's logits are compared; an
argmax mismatch is allowed only where the oracle's top-2 margin is inside the
logit tolerance (a near-tie), and such steps are counted and reported.
"""
import dataclasses
import os

import numpy as np
import pytest

import oracle
import synth
import synth.workloads as wl
from synth import BF16, F32

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import transformer_decode_step_gb300 as pnb  # noqa: E402

DEV = torch.device("cuda:0")
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def tol(shape):
    return 1e-3 if shape.dtype == F32 else 2e-2


def set_attention(sm, kind):
    """'tensor': decode attention on tcgen05 tensor cores; 'cuda': the CUDA-core
    kernel.  Both run inside the same per-phase step."""
    if kind == "tensor" and not sm.model.tensor_attention:
        try:
            sm.model.set_tensor_attention(True)
        except pnb.PnbError as e:
            if e.code == -5:
                pytest.skip("the tensor-core attention does not cover this shape")
            raise
    if kind == "cuda":
        sm.model.set_tensor_attention(False)
    assert sm.model.tensor_attention == (kind == "tensor")
    moe = sm.shape.expert_count > 0
    assert sm.model.step_kernel_count() == sm.shape.n_layer * (5 + (1 if moe else 0)) + 1


def gpu_run(sm, state, tokens, graphs=True):
    sm.model.set_graphs(graphs)
    V = sm.shape.n_vocab
    out, am = [], []
    lg = torch.empty(V, dtype=torch.float32, device=DEV)
    a = torch.empty(1, dtype=torch.int32, device=DEV)
    for t in tokens:
        state.forward(int(t), logits=lg, argmax=a)
        out.append(lg.cpu().numpy().copy())
        am.append(int(a.item()))
    assert state.device_error() == 0
    return out, am


def oracle_run(shape, seed, tokens, start_pos=0, slot=0):
    m = oracle.Model(shape, seed=seed)
    s = m.new_state()
    if start_pos:
        lo, hi = wl.kv_prefill_range(shape, start_pos)
        s.prefill_synth(seed, slot, lo, hi)
    res = [s.forward(int(t)) for t in tokens]
    return [r[0] for r in res], [r[1] for r in res]


def compare(shape, got, gam, ref, ram, what):
    t = tol(shape)
    near_ties = 0
    for i, (g, r) in enumerate(zip(got, ref)):
        scale = float(np.max(np.abs(r)))
        err = float(np.max(np.abs(g - r)))
        assert err <= t * scale, f"{what} step {i}: max|d|={err:.3e} > {t}*{scale:.3e}"
        if gam[i] != ram[i]:
            top = np.sort(r)[-2:]
            margin = float(top[1] - top[0])
            assert margin <= t * scale, f"{what} step {i}: argmax {gam[i]} != {ram[i]} (margin {margin})"
            near_ties += 1
    return near_ties


# ------------------------------------------------------------ device generator

@pytest.mark.parametrize("dtype", [F32, BF16])
def test_device_generator_equals_host_generator(dtype):
    rows, cols = 37, 264
    es = 4 if dtype == F32 else 2
    buf = torch.zeros(rows * 2 * cols * es, dtype=torch.uint8, device=DEV)
    k = synth.key(9, synth.WGATE, 3, 1)
    synth.dev_fill_matrix(buf.data_ptr(), dtype, 1, 2, rows, cols, k, 0.02,
                          torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    host = synth.values(k, 0, rows * cols, 0.02, dtype).reshape(rows, cols)
    if dtype == F32:
        dev = buf.view(torch.float32).reshape(2 * rows, cols).cpu().numpy()
    else:
        dev = buf.view(torch.bfloat16).float().reshape(2 * rows, cols).cpu().numpy()
    assert np.array_equal(dev[1::2], host)
    assert np.all(dev[0::2] == 0)


def test_device_kv_fill_uses_ring_slots():
    n_kv, cap, hd = 3, 10, 32
    buf = torch.zeros(n_kv * cap * hd, dtype=torch.bfloat16, device=DEV)
    k = synth.key(4, synth.KCACHE, 0, 2)
    synth.dev_fill_kv(buf.data_ptr(), BF16, n_kv, cap, hd, 13, 23, k, 1.0,
                      torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    dev = buf.float().reshape(n_kv, cap, hd).cpu().numpy()
    host = synth.values(k, 13 * n_kv * hd, 10 * n_kv * hd, 1.0, BF16).reshape(10, n_kv, hd)
    for j in range(13, 23):
        assert np.array_equal(dev[:, j % cap, :], host[j - 13])


# ---------------------------------------------------------------- tiny fp32

def _tiny_tokens():
    w = wl.TINY
    with open(os.path.join(GOLDEN, "tiny_oracle_greedy.txt")) as f:
        rows = dict(l.split(maxsplit=1) for l in f if not l.startswith("#"))
    prompt = [int(v) for v in rows["prompt"].split()]
    gen = [int(v) for v in rows["generated"].split()]
    assert prompt == wl.prompt_tokens(w)
    return prompt, gen


def test_tiny_teacher_forced_matches_oracle():
    w = wl.TINY
    prompt, gen = _tiny_tokens()
    tokens = prompt + gen[:-1]
    sm = pnb.SynthModel(w.shape, w.seed, device=DEV)
    got, gam = gpu_run(sm, sm.new_state(), tokens)
    ref, ram = oracle_run(w.shape, w.seed, tokens)
    assert compare(w.shape, got, gam, ref, ram, "tiny") == 0
    assert gam[len(prompt) - 1:] == gen


def test_tiny_free_running_greedy_matches_stored_oracle_run():
    w = wl.TINY
    prompt, gen = _tiny_tokens()
    sm = pnb.SynthModel(w.shape, w.seed, device=DEV)
    st = sm.new_state()
    a = torch.empty(len(gen), dtype=torch.int32, device=DEV)
    for t in prompt[:-1]:
        st.forward(t)
    st.forward(prompt[-1], argmax=a[0:1])
    for i in range(1, len(gen)):
        st.forward(pnb.PNB_TOKEN_PREV, argmax=a[i:i + 1])
    assert st.device_error() == 0
    assert a.cpu().tolist() == gen
    assert st.pos == len(prompt) + len(gen) - 1


@pytest.mark.parametrize("attention", ["cuda", "tensor"])
def test_graph_replay_equals_eager_launches_bitwise(attention):
    shape = SMALL_HD128 if attention == "tensor" else wl.TINY.shape
    seed = 11
    rng = np.random.default_rng(3)
    tokens = [int(t) for t in rng.integers(0, shape.n_vocab, size=12)]
    sm = pnb.SynthModel(shape, seed, device=DEV)
    set_attention(sm, attention)
    a, _ = gpu_run(sm, sm.new_state(), tokens, graphs=True)
    b, _ = gpu_run(sm, sm.new_state(), tokens, graphs=False)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def test_reset_then_replay_is_bitwise_identical():
    w = wl.TINY
    prompt, _ = _tiny_tokens()
    sm = pnb.SynthModel(w.shape, w.seed, device=DEV)
    st = sm.new_state()
    a, _ = gpu_run(sm, st, prompt)
    st.reset()
    assert st.pos == 0
    b, _ = gpu_run(sm, st, prompt)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def test_context_full_and_bad_token_are_host_errors():
    w = wl.TINY
    sm = pnb.SynthModel(w.shape, w.seed, device=DEV)
    st = sm.new_state()
    with pytest.raises(pnb.PnbError) as e:
        st.forward(w.shape.n_vocab)
    assert e.value.code == -7
    st.set_pos(w.shape.n_ctx - 1)
    st.forward(3)
    with pytest.raises(pnb.PnbError) as e:
        st.forward(3)
    assert e.value.code == -4
    assert st.device_error() == 0


# ------------------------------------------------- small bf16 models (tiles, ragged)

SMALL_WIN = wl.Shape(n_vocab=3001, n_embd=512, n_head=8, n_kv_head=2, n_layer=2, n_ff=1376,
                     n_ctx=96, rope_theta=1e4, rms_norm_eps=1e-5, sliding_window=24, dtype=BF16)
SMALL_MHA = dataclasses.replace(SMALL_WIN, n_kv_head=8, sliding_window=0, n_ff=1024,
                                n_vocab=2048, rope_theta=5e5)
SMALL_MOE = wl.Shape(n_vocab=777, n_embd=256, n_head=4, n_kv_head=2, n_layer=2, n_ff=512,
                     n_ctx=64, rope_theta=1e6, rms_norm_eps=1e-5, expert_count=4, expert_used=2,
                     dtype=BF16)
SMALL_G8 = wl.Shape(n_vocab=512, n_embd=2048, n_head=16, n_kv_head=2, n_layer=1, n_ff=1024,
                    n_ctx=64, rope_theta=1e4, rms_norm_eps=1e-5, dtype=BF16)
# KV-head counts that do not divide the SM count: attention ranges cross heads
SMALL_MHA32 = wl.Shape(n_vocab=1500, n_embd=2048, n_head=32, n_kv_head=32, n_layer=2, n_ff=1024,
                       n_ctx=400, rope_theta=1e4, rms_norm_eps=1e-5, dtype=BF16)
SMALL_KV5 = wl.Shape(n_vocab=700, n_embd=640, n_head=10, n_kv_head=5, n_layer=2, n_ff=768,
                     n_ctx=600, rope_theta=1e6, rms_norm_eps=1e-5, sliding_window=200, dtype=BF16)
SMALL_HD128 = wl.Shape(n_vocab=1000, n_embd=1024, n_head=8, n_kv_head=2, n_layer=1, n_ff=2816,
                       n_ctx=300, rope_theta=1e4, rms_norm_eps=1e-5, dtype=BF16)


@pytest.mark.parametrize("attention", ["tensor", "cuda"])
@pytest.mark.parametrize("name,shape,start,steps", [
    ("window_ring", SMALL_WIN, 40, 24),       # ring of 24 slots, pre-fill wraps it
    ("window_short", SMALL_WIN, 0, 30),       # empty cache, window fills then slides
    ("mha", SMALL_MHA, 17, 12),
    ("moe", SMALL_MOE, 9, 12),
    ("hd128", SMALL_HD128, 250, 8),
    ("hd128_gqa8", SMALL_G8, 40, 6),           # 8 query heads per KV head at head_dim 128
    ("mha32_cross", SMALL_MHA32, 300, 6),      # 32 KV heads: CTA ranges cross head boundaries
    ("kv5_window_cross", SMALL_KV5, 450, 6),   # 5 KV heads, window ring, crossing ranges
])
def test_small_bf16_models_match_oracle(name, shape, start, steps, attention):
    seed = 77
    sm = pnb.SynthModel(shape, seed, device=DEV)
    set_attention(sm, attention)
    st = sm.new_state(start_pos=start)
    rng = np.random.default_rng(5)
    tokens = [int(t) for t in rng.integers(0, shape.n_vocab, size=steps)]
    got, gam = gpu_run(sm, st, tokens)
    ref, ram = oracle_run(shape, seed, tokens, start_pos=start)
    ties = compare(shape, got, gam, ref, ram, name)
    assert ties <= 1


def test_tensor_and_cuda_core_attention_steps_agree():
    """Same model and tokens with either attention kernel: logits agree to fp32 rounding."""
    shape, seed = SMALL_HD128, 13
    tokens = [5, 17, 400, 300, 9, 9, 1]
    outs = []
    for attention in ("tensor", "cuda"):
        sm = pnb.SynthModel(shape, seed, device=DEV)
        set_attention(sm, attention)
        outs.append(gpu_run(sm, sm.new_state(start_pos=200), tokens))
    for a, b in zip(outs[0][0], outs[1][0]):
        assert np.max(np.abs(a - b)) <= 1e-4 * np.max(np.abs(a))


# ------------------------------------------------- full-size workloads, sampled steps

@pytest.mark.parametrize("w", [wl.LLAMA7B, wl.MISTRAL7B, wl.MIXTRAL], ids=lambda w: w.name)
def test_full_size_first_steps_match_oracle(w):
    """The benchmark's own model and cache: the first two greedy steps (one for
    the MoE model), teacher-forced, against the oracle."""
    nsteps = 1 if w.shape.expert_count else 2
    ref_model = oracle.Model(w.shape, seed=w.seed)
    os_ = ref_model.new_state()
    lo, hi = wl.kv_prefill_range(w.shape, w.prefill)
    os_.prefill_synth(w.seed, 0, lo, hi)
    tokens = [wl.prompt_tokens(w)[0]]
    ref, ram = [], []
    for i in range(nsteps):
        lg, am = os_.forward(tokens[-1])
        ref.append(lg)
        ram.append(am)
        if i + 1 < nsteps:
            tokens.append(am)
    del os_, ref_model
    sm = pnb.SynthModel(w.shape, w.seed, device=DEV)
    st = sm.new_state(start_pos=w.prefill)
    got, gam = gpu_run(sm, st, tokens)
    assert compare(w.shape, got, gam, ref, ram, w.name) == 0
    del st, sm
    torch.cuda.empty_cache()
