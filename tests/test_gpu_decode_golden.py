"""The benchmark workloads' own greedy decodes, every step, against the oracle.

The oracle's greedy decodes are stored by ``tests/golden/make_decode_golden.py``
(which calls only the CPU oracle and the seeded input generator):

* Llama-7B, Mistral-7B (4096-position window ring) and Mixtral (8 experts,
  top-2): 128 steps from the pre-filled positions 2048 / 8192 / 4096;
* Llama-7B with Q8_0 and Q4_0 weights (64 steps) and Mixtral with Q8_0 and
  Q4_0 weights (32 steps), every matrix in blocks;
* the batched Llama-8B workload: 64 steps of slots 0, 7, 15, 31 and 63.

The GPU decodes the same workload through the C ABI (``pnb_forward``, or
``pnb_forward_batch`` with B = 8, 16, 32 and 64 slots, in the launch
configuration the benchmark times), fed the oracle's tokens (teacher
forcing), and every step is compared:

* argmax identical, unless the oracle's top-2 margin is inside the logit
  tolerance (a near-tie, counted and printed, never hidden);
* max|d logit| <= 2e-2 * max|logit| (bf16 weights) on the top 8 logits and
  512 fixed ids of every step, on max|logit| itself, and on the full logit
  vectors stored for a few steps.

The "Engine Architecture" page's generation loop ("Generation Loop") is what
these decodes run: forward, then argmax at temperature 0.
"""
import os

import numpy as np
import pytest

import synth.workloads as wl

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import transformer_decode_step_gb300 as pnb  # noqa: E402

DEV = torch.device("cuda:0")
TOL = 2e-2
# A MoE step whose top-k routing came within this relative gap of a tie in the
# oracle (the smallest gap between a chosen and an unchosen router logit over the
# layers, relative to the layer's largest |logit|) may route one layer through
# another expert on the GPU: the residual streams of the two sides differ by
# about 1e-4 of their size (bf16 cache, summation order), and the router logits
# with them.  Such a step is a routing near-tie: reported, its logits not
# compared (the same rule as an argmax near-tie, for the router's decision).
ROUTE_TOL = 1e-3
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def golden(w):
    path = os.path.join(GOLDEN, f"decode_{w.name}.npz")
    if not os.path.exists(path):
        pytest.fail(f"{path} missing: run tests/golden/make_decode_golden.py")
    return dict(np.load(path))


class Recorder:
    """Collects, on the device, what each step is compared on; one copy at the end."""

    def __init__(self, g, gi, steps):
        self.ids = torch.as_tensor(g["sample_ids"].astype(np.int64), device=DEV)
        self.top = torch.as_tensor(g["top_idx"][gi].astype(np.int64), device=DEV)
        self.samp = torch.empty(steps, self.ids.numel(), device=DEV)
        self.topv = torch.empty(steps, self.top.shape[1], device=DEV)
        self.amax = torch.empty(steps, device=DEV)
        self.am = torch.empty(steps, dtype=torch.int32, device=DEV)
        self.full_steps = [int(s) for sl, s in zip(g["full_slot"], g["full_step"])
                           if sl == int(g["slots"][gi])]
        self.full = {}

    def record(self, i, logits, am):
        self.samp[i] = logits.index_select(0, self.ids)
        self.topv[i] = logits.index_select(0, self.top[i])
        self.amax[i] = logits.abs().max()
        self.am[i] = am
        if i in self.full_steps:
            self.full[i] = logits.clone()

    def check(self, g, gi, what):
        samp, topv = self.samp.cpu().numpy(), self.topv.cpu().numpy()
        amax, am = self.amax.cpu().numpy(), self.am.cpu().numpy()
        near, worst = [], 0.0
        route = g["route_margin"][gi] if "route_margin" in g else np.full(samp.shape[0], np.inf)
        routing_ties = [i for i in range(samp.shape[0]) if route[i] < ROUTE_TOL]
        for i in range(samp.shape[0]):
            if i in routing_ties:
                continue
            scale = float(g["maxabs"][gi][i])
            tol = TOL * scale
            err = max(float(np.max(np.abs(samp[i] - g["sample_val"][gi][i]))),
                      float(np.max(np.abs(topv[i] - g["top_val"][gi][i]))),
                      abs(float(amax[i]) - scale))
            worst = max(worst, err / scale)
            assert err <= tol, f"{what} step {i}: max|d|={err:.3e} > {TOL}*{scale:.3e}"
            if int(am[i]) != int(g["argmax"][gi][i]):
                margin = float(g["top1"][gi][i] - g["top2"][gi][i])
                assert margin <= tol, (f"{what} step {i}: argmax {int(am[i])} != "
                                       f"{int(g['argmax'][gi][i])} (oracle margin {margin:.3e})")
                near.append((i, int(am[i]), int(g["argmax"][gi][i]), margin))
        slot = int(g["slots"][gi])
        for k, (sl, st) in enumerate(zip(g["full_slot"], g["full_step"])):
            if sl != slot:
                continue
            if int(st) in routing_ties:
                continue
            ref = g["full_logits"][k]
            got = self.full[int(st)].cpu().numpy()
            scale = float(np.max(np.abs(ref)))
            err = float(np.max(np.abs(got - ref)))
            worst = max(worst, err / scale)
            assert err <= TOL * scale, f"{what} full logits of step {st}: {err:.3e}"
        print(f"\n{what}: {samp.shape[0]} steps, worst max|d|/max|logit| {worst:.2e}, "
              f"near-ties {len(near)} {near}, routing near-ties {len(routing_ties)} "
              f"{[(i, float(route[i])) for i in routing_ties]}")
        assert len(routing_ties) <= samp.shape[0] // 4, f"{what}: too many routing near-ties"
        return near


# the quantized forms: shorter stored decodes (Q8_0 / Q4_0 blocks, MoE router and
# experts included)
QUANT = [wl.LLAMA7B_Q8.with_(steps=64), wl.LLAMA7B_Q4.with_(steps=64),
         wl.MIXTRAL_Q8.with_(steps=32), wl.MIXTRAL_Q4.with_(steps=32)]


@pytest.mark.parametrize("w", [wl.LLAMA7B, wl.MISTRAL7B, wl.MIXTRAL] + QUANT, ids=lambda w: w.name)
def test_full_size_greedy_decode_matches_oracle(w):
    g = golden(w)
    tokens = g["tokens"][0]
    steps = tokens.size
    assert steps == w.steps and int(g["start_pos"][0]) == w.prefill
    # the stored run is greedy: each fed token is the previous step's argmax
    assert np.array_equal(tokens[1:], g["argmax"][0][:-1])
    assert int(tokens[0]) == wl.prompt_tokens(w)[0]
    sm = pnb.SynthModel(w.shape, w.seed, device=DEV)
    st = sm.new_state(start_pos=w.prefill)
    lg = torch.empty(w.shape.n_vocab, dtype=torch.float32, device=DEV)
    am = torch.empty(1, dtype=torch.int32, device=DEV)
    rec = Recorder(g, 0, steps)
    for i in range(steps):
        st.forward(int(tokens[i]), logits=lg, argmax=am)
        rec.record(i, lg, am[0])
    torch.cuda.synchronize()
    assert st.device_error() == 0
    assert st.pos == w.prefill + steps
    rec.check(g, 0, w.name)
    del st, sm
    torch.cuda.empty_cache()


@pytest.fixture(scope="module")
def batched_model():
    w = wl.LLAMA8B_BATCHED
    sm = pnb.SynthModel(w.shape, w.seed, device=DEV)
    yield w, sm
    del sm
    torch.cuda.empty_cache()


@pytest.mark.parametrize("B", [8, 16, 32, 64])
def test_full_size_batched_decode_matches_oracle(batched_model, B):
    """B slots at their seeded positions advance together for 64 steps; the
    stored slots among them are fed the oracle's tokens, the others their own
    greedy tokens."""
    w, sm = batched_model
    g = golden(w)
    starts = wl.slot_positions(w)
    assert [starts[s] for s in g["slots"]] == list(g["start_pos"])
    gis = [gi for gi, s in enumerate(g["slots"]) if s < B]
    steps = g["tokens"].shape[1]
    states = [sm.new_state(starts[b], slot=b) for b in range(B)]
    V = w.shape.n_vocab
    lg = torch.empty(B, V, dtype=torch.float32, device=DEV)
    am = torch.empty(B, dtype=torch.int32, device=DEV)
    tk = torch.tensor([wl.prompt_tokens(w, b)[0] for b in range(B)], dtype=torch.int32,
                      device=DEV)
    forced = torch.as_tensor(g["tokens"].astype(np.int32), device=DEV)   # [slot][step]
    bidx = torch.tensor([int(g["slots"][gi]) for gi in gis], dtype=torch.int64, device=DEV)
    recs = {gi: Recorder(g, gi, steps) for gi in gis}
    for i in range(steps):
        if i > 0:
            tk.copy_(am)                                  # free-running slots
        tk.index_copy_(0, bidx, forced[gis, i])           # stored slots: the oracle's tokens
        sm.model.forward_batch(states, tokens=tk, logits=lg, argmax=am)
        for gi in gis:
            b = int(g["slots"][gi])
            recs[gi].record(i, lg[b], am[b])
    torch.cuda.synchronize()
    assert all(s.device_error() == 0 for s in states)
    for gi in gis:
        recs[gi].check(g, gi, f"{w.name} B={B} slot {int(g['slots'][gi])}")
    del states
