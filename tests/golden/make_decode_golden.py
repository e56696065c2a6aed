"""Write decode_<workload>.npz: the oracle's greedy decodes of the benchmark workloads.

Calls only the CPU oracle and the seeded input generator (no GPU code).  Each
workload is decoded greedily from its start token and pre-filled cache, the
way the engine's generation loop runs ("Engine Architecture", "Generation
Loop": forward, then argmax at temperature 0, lowest id on ties):

* Llama-7B, Mistral-7B (sliding window 4096) and Mixtral (8 experts, top-2):
  128 steps from the pre-filled positions 2048 / 8192 / 4096;
* Llama-7B with Q8_0 and with Q4_0 weights (64 steps) and Mixtral with Q8_0
  and with Q4_0 weights, router and experts included (32 steps), from the
  same positions;
* the batched Llama-8B workload: 64 steps of slots 0, 7, 15, 31 and 63, each
  from its own seeded start position and token (a slot's sequence does not
  depend on which other slots share the batch, so one run per slot serves
  every batch size B in {8, 16, 32, 64}).

Stored per step (arrays [slot][step] for the batched workload): the token fed,
the oracle's argmax, its top-1 and top-2 logit values and max|logit|, the 8
largest logits with their ids, the logits at 512 fixed ids (seeded), the
smallest relative gap between chosen and unchosen router logits over the MoE
layers (inf for dense models; a routing near-tie when small); the
full logit vector of a few steps (``full_steps``).  The GPU test feeds the
stored tokens (teacher forcing) and compares every step.

Dense weights are handed to the oracle as explicit fp32 arrays generated once
from the same seeded recipe (for the quantized forms: the blocks' dequantized
weights, which the oracle's own block decoding equals bit for bit) (the values the oracle would otherwise generate on
every step), so a step costs one pass over memory; Mixtral's experts, too
large for host memory in fp32, stay seed-generated inside the oracle.  The
arithmetic is the oracle's either way.

Run from the repository root (about an hour and a half on 8 cores):
    python tests/golden/make_decode_golden.py [workload ...]
"""
import os
import sys
import time
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import numpy as np  # noqa: E402

import oracle  # noqa: E402
import synth  # noqa: E402
import synth.workloads as wl  # noqa: E402

N_SAMPLE = 512
N_TOP = 8
BATCHED_SLOTS = (0, 7, 15, 31, 63)


def path_for(w):
    return os.path.join(HERE, f"decode_{w.name}.npz")


def sample_ids(V):
    """The fixed logit ids compared at every step (seeded, sorted, distinct)."""
    rng = np.random.default_rng(20261202)
    return np.sort(rng.choice(V, size=N_SAMPLE, replace=False)).astype(np.int32)


def explicit_arrays(shape, seed, skip_experts):
    """Every generated (non-constant) weight of the model as a storage-valued fp32
    array, keyed as oracle.Model expects; MoE experts left out when asked."""
    specs = [s for s in wl.weight_specs(shape) if s.const is None
             and not (skip_experts and s.name in ("wgate", "wup", "wdown"))]
    out = {}

    def gen(spec):
        k = spec.key(seed)
        if shape.dtype in (synth.Q8, synth.Q4):
            # the dequantized block weights d * q (Q8) or d * (u - 8) (Q4)
            rows_fn = synth.q8_rows if shape.dtype == synth.Q8 else synth.q4_rows
            a = np.empty((spec.rows, spec.cols), dtype=np.float32)
            step = max(1, (1 << 22) // spec.cols)
            for r in range(0, spec.rows, step):
                n = min(step, spec.rows - r)
                a[r:r + n] = rows_fn(k, r, n, spec.cols, spec.sigma)[1]
            return spec, a
        a = np.empty(spec.rows * spec.cols, dtype=np.float32)
        step = 1 << 22
        for i in range(0, a.size, step):
            n = min(step, a.size - i)
            a[i:i + n] = synth.values(k, i, n, spec.sigma, shape.dtype)
        return spec, a.reshape(spec.rows, spec.cols)

    with ThreadPoolExecutor(max_workers=os.cpu_count()) as ex:
        for spec, a in ex.map(gen, specs):
            akey = spec.name if spec.name in ("tok_embd", "out_norm", "output") else \
                (spec.name, spec.layer, spec.sub)
            out[akey] = a
    return out


def decode(model, w, slot, start_pos, steps, full_at):
    """Greedy decode of one sequence; per-step records."""
    V = w.shape.n_vocab
    ids = sample_ids(V)
    s = model.new_state()
    lo, hi = wl.kv_prefill_range(w.shape, start_pos)
    s.prefill_synth(w.seed, slot, lo, hi)
    tok = wl.prompt_tokens(w, slot)[0]
    rec = {k: [] for k in ("tokens", "argmax", "top1", "top2", "maxabs", "top_idx", "top_val",
                           "sample_val", "route_margin")}
    full = []
    t0 = time.time()
    for i in range(steps):
        logits, am = s.forward(tok)
        order = np.argsort(-logits, kind="stable")[:N_TOP]
        srt = np.sort(logits)
        rec["tokens"].append(tok)
        rec["argmax"].append(am)
        rec["top1"].append(srt[-1])
        rec["top2"].append(srt[-2])
        rec["maxabs"].append(np.max(np.abs(logits)))
        rec["top_idx"].append(order.astype(np.int32))
        rec["top_val"].append(logits[order])
        rec["sample_val"].append(logits[ids])
        rec["route_margin"].append(s.route_margin)
        if i in full_at:
            full.append(logits.copy())
        tok = am
        if i % 16 == 15:
            print(f"  {w.name} slot {slot}: step {i + 1}/{steps} ({time.time() - t0:.0f} s)",
                  flush=True)
    dt = {"tokens": np.int32, "argmax": np.int32, "top_idx": np.int32, "route_margin": np.float64}
    out = {k: np.asarray(v, dtype=dt.get(k, np.float32)) for k, v in rec.items()}
    out["full_logits"] = np.asarray(full, dtype=np.float32).reshape(len(full), V)
    return out


def run(w):
    moe = w.shape.expert_count > 0
    t0 = time.time()
    arrays = explicit_arrays(w.shape, w.seed, skip_experts=moe)
    print(f"{w.name}: weights generated in {time.time() - t0:.0f} s", flush=True)
    model = oracle.Model(w.shape, seed=w.seed, arrays=arrays)
    if w.slot_pos_range is None:
        slots, starts, steps = [0], [w.prefill], w.steps
        full_at = {0: (0, steps - 1)}
    else:
        allpos = wl.slot_positions(w)
        slots = list(BATCHED_SLOTS)
        starts = [allpos[b] for b in slots]
        steps = w.steps
        full_at = {0: (steps - 1,), 63: (steps - 1,)}
    per = [decode(model, w, b, p, steps, full_at.get(b, ())) for b, p in zip(slots, starts)]
    res = {k: np.stack([r[k] for r in per]) for k in per[0] if k != "full_logits"}
    res["full_logits"] = np.concatenate([r["full_logits"] for r in per])
    res["full_slot"] = np.asarray([b for b in slots for _ in full_at.get(b, ())], dtype=np.int32)
    res["full_step"] = np.asarray([i for b in slots for i in full_at.get(b, ())], dtype=np.int32)
    res["slots"] = np.asarray(slots, dtype=np.int32)
    res["start_pos"] = np.asarray(starts, dtype=np.int32)
    res["sample_ids"] = sample_ids(w.shape.n_vocab)
    np.savez_compressed(path_for(w), **res)
    print(f"{w.name}: done in {time.time() - t0:.0f} s -> {path_for(w)}", flush=True)


# the quantized forms (every matrix in Q8_0 / Q4_0 blocks) over shorter decodes
QUANT_STEPS = {wl.LLAMA7B_Q8.name: 64, wl.LLAMA7B_Q4.name: 64, wl.MIXTRAL_Q8.name: 32,
               wl.MIXTRAL_Q4.name: 32}
WORKLOADS = [wl.LLAMA7B, wl.MISTRAL7B, wl.LLAMA8B_BATCHED, wl.MIXTRAL] + \
    [w.with_(steps=QUANT_STEPS[w.name]) for w in (wl.LLAMA7B_Q8, wl.LLAMA7B_Q4, wl.MIXTRAL_Q8,
                                                  wl.MIXTRAL_Q4)]

if __name__ == "__main__":
    names = sys.argv[1:] or [w.name for w in WORKLOADS]
    for w in WORKLOADS:
        if w.name in names:
            run(w)
