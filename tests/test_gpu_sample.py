"""The sampler (pnb_sample / pnb_sample_batch) against the CPU oracle, plus the
begin / poll seam.

Both sides order the candidates by the same fp32 z = logit / T (after the
penalty), so top-k is decided identically and z is compared bit for bit.  The
softmax masses differ by rounding (the kernel: fp32 exp in 64-bit fixed point;
the oracle: fp64), so where u or top_p lies within 1e-5 of a cumulative
boundary the token may be either neighbour: the test accepts the oracle's
token at u and top_p moved by +-1e-5, and nothing else.  u is the oracle's own
SplitMix64 word (pinned to the published sequence) at the state's draw index.
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
EPS = 1e-5

TINY = wl.Shape(n_vocab=1000, n_embd=64, n_head=2, n_kv_head=2, n_layer=1, n_ff=64, n_ctx=64,
                rope_theta=1e4, rms_norm_eps=1e-5, dtype=BF16)

_models = {}


def model_for(V):
    if V not in _models:
        _models[V] = pnb.SynthModel(dataclasses.replace(TINY, n_vocab=V), 3, device=DEV)
    return _models[V]


def lm_logits(rng, V, ties=False):
    """Logits shaped like a language model's: a heavy upper tail over a normal
    bulk; with ties, values on a coarse grid so many tokens share a value."""
    x = rng.normal(0.0, 2.0, size=V) + np.where(rng.random(V) < 0.01, rng.exponential(3.0, V), 0)
    if ties:
        x = np.round(x * 2) / 2
    return x.astype(np.float32)


def oracle_accepts(lg, T, pen, recent, k, p, u):
    main = oracle.sample(lg, T, pen, recent, k, p, u)[0]
    alts = {main}
    for dp in ((-EPS, 0.0, EPS) if p < 1.0 else (0.0,)):
        for du in (-EPS, 0.0, EPS):
            uu = min(max(u + du, 0.0), 1.0 - 2.0**-30)
            pp = min(max(p + dp, 0.0), 0.999999) if p < 1.0 else p
            alts.add(oracle.sample(lg, T, pen, recent, k, pp, uu)[0])
    return main, alts


def gpu_sample(st, lg_np, params, recent=None):
    lg = torch.from_numpy(lg_np).to(DEV)
    rec = torch.tensor(recent, dtype=torch.int32, device=DEV) if recent else None
    tok = torch.full((1,), -5, dtype=torch.int32, device=DEV)
    st.sample(lg, params, recent=rec, token=tok)
    torch.cuda.synchronize()
    return int(tok.item()), lg.cpu().numpy()


def expected_z(lg, T, pen, recent):
    z = (lg / np.float32(T)).astype(np.float32)
    for t in set(int(r) for r in recent if 0 <= r < lg.size):
        z[t] = z[t] / np.float32(pen) if z[t] > 0 else z[t] * np.float32(pen)
    return z


CASES = [
    # V, T, penalty, n_recent, top_k, top_p, ties
    (1000, 1.0, 1.0, 0, 0, 1.0, False),
    (1000, 0.7, 1.3, 40, 40, 0.9, False),
    (1000, 1.0, 1.0, 0, 0, 0.5, True),
    (1000, 1.5, 0.8, 10, 7, 1.0, True),
    (32000, 0.8, 1.1, 64, 40, 0.95, False),
    (32000, 1.0, 1.0, 0, 1, 1.0, False),
    (32000, 1.0, 1.0, 0, 4096, 1.0, False),      # the largest shared-memory candidate list
    (32000, 1.0, 1.0, 0, 4097, 0.8, False),      # candidates stay in global memory
    (32000, 2.0, 1.2, 100, 0, 0.9, False),       # no top-k: every token a candidate
    (32000, 0.9, 1.0, 0, 100, 0.7, True),
    (32000, 1.0, 1.0, 0, 0, 1.0, True),
    (50257, 0.6, 1.05, 256, 50, 0.92, False),
    (152064, 0.7, 1.1, 64, 20, 0.8, False),
    (152064, 1.0, 1.0, 0, 0, 0.99, False),
]


@pytest.mark.parametrize("V,T,pen,nrec,k,p,ties", CASES)
def test_sample_matches_oracle(V, T, pen, nrec, k, p, ties):
    sm = model_for(V)
    st = sm.new_state(0)
    rng = np.random.default_rng(V + nrec + k)
    seed = int(rng.integers(0, 2**63))
    params = pnb.sampling_params(T, pen, k, p, seed)
    exact = 0
    for draw in range(12):
        lg = lm_logits(rng, V, ties)
        recent = [int(t) for t in rng.integers(-3, V + 3, size=nrec)]
        recent += recent[: nrec // 4]   # repeated tokens count once
        u = oracle.sample_uniform(seed, draw)
        tok, z = gpu_sample(st, lg, params, recent)
        main, alts = oracle_accepts(lg, T, pen, recent, k, p, u)
        assert tok in alts, f"draw {draw}: gpu {tok}, oracle {main} (accepts {sorted(alts)})"
        exact += tok == main
        assert np.array_equal(z.view(np.uint32), expected_z(lg, T, pen, recent).view(np.uint32))
    assert exact >= 11
    assert st.device_error() == 0


def test_greedy_is_argmax_and_leaves_logits():
    sm = model_for(32000)
    st = sm.new_state(0)
    rng = np.random.default_rng(1)
    for T in (0.0, -2.0):
        lg = lm_logits(rng, 32000, ties=True)
        lg[[17, 900, 31999]] = lg.max() + 1.0   # tie at the top: the lowest id
        tok, out = gpu_sample(st, lg, pnb.sampling_params(T, 1.3, 5, 0.5, 9), [17, 900])
        assert tok == 17 and np.array_equal(out, lg)


def test_draw_counter_reset_and_set():
    sm = model_for(1000)
    st = sm.new_state(0)
    rng = np.random.default_rng(2)
    lg = lm_logits(rng, 1000)
    params = pnb.sampling_params(1.0, 1.0, 0, 1.0, 12345)
    first = [gpu_sample(st, lg, params)[0] for _ in range(20)]
    want = [oracle_accepts(lg, 1.0, 1.0, [], 0, 1.0, oracle.sample_uniform(12345, d))[1]
            for d in range(20)]
    assert all(t in w for t, w in zip(first, want))
    assert len(set(first)) > 3           # the draws move on
    st.reset()
    assert [gpu_sample(st, lg, params)[0] for _ in range(20)] == first
    st.set_draw(7)
    assert [gpu_sample(st, lg, params)[0] for _ in range(5)] == first[7:12]


def test_sampled_token_feeds_the_next_step():
    sm = model_for(1000)
    a, b = sm.new_state(0), sm.new_state(0)
    V = 1000
    lg = torch.empty(V, dtype=torch.float32, device=DEV)
    lb = torch.empty(V, dtype=torch.float32, device=DEV)
    tok = torch.empty(1, dtype=torch.int32, device=DEV)
    params = pnb.sampling_params(1.2, 1.0, 50, 0.95, 77)
    a.forward(5, logits=lg)
    b.forward(5, logits=lb)
    for step in range(6):
        raw = lg.cpu().numpy().copy()
        a.sample(lg, params, token=tok)
        t = int(tok.item())
        u = oracle.sample_uniform(77, step)
        assert t in oracle_accepts(raw, 1.2, 1.0, [], 50, 0.95, u)[1]
        a.forward(pnb.PNB_TOKEN_PREV, logits=lg)    # continues from the sampled token
        b.forward(t, logits=lb)
        assert torch.equal(lg, lb)
    assert a.device_error() == 0


def test_batch_equals_single_calls():
    V = 32000
    sm = model_for(V)
    B = 5
    rng = np.random.default_rng(5)
    lg = np.stack([lm_logits(rng, V, ties=(b % 2 == 1)) for b in range(B)])
    params = [pnb.sampling_params(0.5 + 0.3 * b, 1.0 + 0.1 * b, [0, 1, 40, 5000, 200][b],
                                  [1.0, 0.9, 0.8, 0.95, 0.3][b], 1000 + b) for b in range(B)]
    params[0] = pnb.sampling_params(0.0, 1.0, 0, 1.0, 1)   # one greedy slot
    recent = [torch.tensor(rng.integers(0, V, size=3 * b), dtype=torch.int32, device=DEV)
              for b in range(B)]
    states = [sm.new_state(0) for _ in range(B)]
    lt = torch.from_numpy(lg).to(DEV)
    toks = torch.empty(B, dtype=torch.int32, device=DEV)
    sm.model.sample_batch(states, lt, params, recent=recent, tokens=toks)
    single = []
    for b in range(B):
        st = sm.new_state(0)
        one = torch.from_numpy(lg[b].copy()).to(DEV)
        t = torch.empty(1, dtype=torch.int32, device=DEV)
        st.sample(one, params[b], recent=recent[b], token=t)
        single.append(int(t.item()))
        assert torch.equal(one, lt[b])
    assert toks.cpu().tolist() == single


def test_sampler_argument_errors():
    sm = model_for(1000)
    st = sm.new_state(0)
    lg = torch.zeros(1000, dtype=torch.float32, device=DEV)
    for bad in (pnb.sampling_params(float("nan")), pnb.sampling_params(float("inf")),
                pnb.sampling_params(1.0, 0.0), pnb.sampling_params(1.0, -1.0),
                pnb.sampling_params(1.0, 1.0, 0, float("nan"))):
        with pytest.raises(pnb.PnbError) as e:
            st.sample(lg, bad)
        assert e.value.code == -1
    with pytest.raises(pnb.PnbError) as e:
        st.sample(lg[1:], pnb.sampling_params(1.0))   # 4-byte offset: not 16-byte aligned
    assert e.value.code == -3
    assert pnb.pnb_sample(sm.model.handle, st.handle, lg.data_ptr(),
                          None, None, 0, None, None) == -2


def test_user_graph_of_step_and_sample_replays_the_eager_loop():
    sm = model_for(1000)
    sm.model.set_graphs(False)
    try:
        V = 1000
        params = pnb.sampling_params(1.0, 1.2, 30, 0.9, 4242)
        rec = torch.tensor([1, 2, 3, 4], dtype=torch.int32, device=DEV)

        def loop(st, lg, tok, n):
            out = []
            for _ in range(n):
                st.forward(pnb.PNB_TOKEN_PREV, logits=lg)
                st.sample(lg, params, recent=rec, token=tok)
                out.append(int(tok.item()))
            return out

        a = sm.new_state(0)
        lg = torch.empty(V, dtype=torch.float32, device=DEV)
        tok = torch.empty(1, dtype=torch.int32, device=DEV)
        a.forward(9, logits=lg)
        a.sample(lg, params, recent=rec, token=tok)
        eager = loop(a, lg, tok, 8)

        b = sm.new_state(0)
        lg2 = torch.empty(V, dtype=torch.float32, device=DEV)
        tok2 = torch.empty(1, dtype=torch.int32, device=DEV)
        b.forward(9, logits=lg2)
        b.sample(lg2, params, recent=rec, token=tok2)
        torch.cuda.synchronize()
        s = torch.cuda.Stream()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                b.forward(pnb.PNB_TOKEN_PREV, logits=lg2, stream=s)
                b.sample(lg2, params, recent=rec, token=tok2, stream=s)
        # capture enqueued nothing: b is still after its first sample
        replay = []
        for _ in range(8):
            g.replay()
            torch.cuda.synchronize()
            replay.append(int(tok2.item()))
        assert replay == eager
    finally:
        sm.model.set_graphs(True)


def test_begin_poll_seam():
    sm = model_for(1000)
    V = 1000
    a, b = sm.new_state(0), sm.new_state(0)
    lg = torch.empty(V, dtype=torch.float32, device=DEV)
    lb = torch.empty(V, dtype=torch.float32, device=DEV)
    am = torch.empty(1, dtype=torch.int32, device=DEV)
    torch.cuda.synchronize()             # begin runs on the state's own stream
    with pytest.raises(pnb.PnbError) as e:
        a.poll()                         # nothing begun
    assert e.value.code == -1
    a.forward_begin(11, logits=lg, argmax=am)
    with pytest.raises(pnb.PnbError) as e:
        a.forward_begin(12)              # one step in flight per state
    assert e.value.code == -12
    polls = 0
    while not a.poll():
        polls += 1
        assert polls < 10_000_000
    b.forward(11, logits=lb)
    torch.cuda.synchronize()
    assert torch.equal(lg, lb)
    # a step, then a sampling, then one poll for both
    tok = torch.empty(1, dtype=torch.int32, device=DEV)
    params = pnb.sampling_params(0.9, 1.0, 20, 0.9, 5)
    a.forward_begin(pnb.PNB_TOKEN_PREV, logits=lg)
    a.sample_begin(lg, params, token=tok)
    while not a.poll():
        pass
    b.forward(int(am.item()), logits=lb)
    torch.cuda.synchronize()
    raw = lb.cpu().numpy()
    assert int(tok.item()) in oracle_accepts(raw, 0.9, 1.0, [], 20, 0.9,
                                             oracle.sample_uniform(5, 0))[1]
    assert a.pos == 2 and a.stream() != 0
    # a device-side error surfaces through poll
    c = sm.new_state(0)
    c.prefill(torch.full((2,), V + 5, dtype=torch.int32, device=DEV))
    torch.cuda.synchronize()             # begin runs on the state's own stream
    c.forward_begin(3)
    with pytest.raises(pnb.PnbError) as e:
        while not c.poll():
            pass
    assert e.value.code == -8


# a model the batched step covers (bf16, dense, n_embd / n_head * hd / n_ff multiples of 64)
BATCH_SHAPE = wl.Shape(n_vocab=3001, n_embd=512, n_head=8, n_kv_head=2, n_layer=2, n_ff=1024,
                       n_ctx=160, rope_theta=1e4, rms_norm_eps=1e-5, dtype=BF16)


def test_continuous_batching_join_leave_with_in_loop_sampling():
    """The batch decoder loop of the pages' serve layer: sequences join (prefill,
    then a first sampled token) and leave (budget reached) between batched
    steps; after each step every active slot is sampled in one launch.  Each
    sequence, replayed alone with its recorded tokens, must see the same logits
    (1e-3: batched and single-sequence steps differ only in summation order and
    the tensor-core split of activations), and each recorded token must be a
    draw the oracle sampler accepts from the logits the slot had."""
    sm = pnb.SynthModel(BATCH_SHAPE, 19, device=DEV)
    V = BATCH_SHAPE.n_vocab
    rng = np.random.default_rng(12)
    reqs = []
    for r in range(6):
        reqs.append({"prompt": [int(t) for t in rng.integers(0, V, size=int(rng.integers(3, 20)))],
                     "budget": int(rng.integers(3, 9)),
                     "params": pnb.sampling_params(0.7 + 0.1 * r, 1.0 + 0.05 * r, [0, 20, 40][r % 3],
                                                   [0.9, 1.0, 0.8][r % 3], 900 + r),
                     "tokens": [], "logits": []})
    queue, active = list(range(6)), []
    states = {}
    max_active = 3
    sizes = []
    while queue or active:
        while queue and len(active) < max_active:             # join
            r = queue.pop(0)
            q = reqs[r]
            st = sm.new_state(0)
            T = len(q["prompt"])
            pl = torch.empty(T, V, dtype=torch.float32, device=DEV)
            st.prefill(torch.tensor(q["prompt"], dtype=torch.int32, device=DEV), logits=pl)
            last = pl[T - 1].clone()
            q["logits"].append(last.cpu().numpy())
            tok = torch.empty(1, dtype=torch.int32, device=DEV)
            st.sample(last, q["params"], token=tok)
            q["tokens"].append(int(tok.item()))
            states[r] = st
            active.append(r)
        B = len(active)
        sizes.append(B)
        lg = torch.empty(B, V, dtype=torch.float32, device=DEV)
        sm.model.forward_batch([states[r] for r in active], logits=lg)
        raw = lg.cpu().numpy()
        toks = torch.empty(B, dtype=torch.int32, device=DEV)
        sm.model.sample_batch([states[r] for r in active], lg, [reqs[r]["params"] for r in active],
                              tokens=toks)
        for j, r in enumerate(active):
            reqs[r]["logits"].append(raw[j].copy())
            reqs[r]["tokens"].append(int(toks[j].item()))
        for r in list(active):                                # leave
            if len(reqs[r]["tokens"]) >= reqs[r]["budget"]:
                active.remove(r)
                assert states.pop(r).device_error() == 0
    assert max(sizes) == max_active and min(sizes) < max_active   # membership changed
    for r, q in enumerate(reqs):
        p = q["params"]
        # every recorded token is a draw the oracle accepts from the slot's logits
        for d, (lgt, t) in enumerate(zip(q["logits"], q["tokens"])):
            assert t in oracle_accepts(lgt, p.temperature, p.repeat_penalty, [], p.top_k, p.top_p,
                                       oracle.sample_uniform(p.seed, d))[1], f"request {r} draw {d}"
        # alone, fed the recorded tokens, the sequence sees the same logits
        st = sm.new_state(0)
        one = torch.empty(V, dtype=torch.float32, device=DEV)
        for t in q["prompt"]:
            st.forward(t, logits=one)
        ref = [one.cpu().numpy()]
        for t in q["tokens"][:-1]:
            st.forward(t, logits=one)
            ref.append(one.cpu().numpy())
        for d, (a, b) in enumerate(zip(ref, q["logits"])):
            scale = float(np.max(np.abs(a)))
            assert float(np.max(np.abs(a - b))) <= 1e-3 * scale, f"request {r} step {d}"
