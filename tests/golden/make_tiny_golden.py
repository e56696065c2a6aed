"""Write tiny_oracle_greedy.txt: the oracle's greedy run of the tiny fp32 workload.

Calls only the CPU oracle and the seeded input generator (no GPU code).  The
workload: 16 prompt tokens fed one per forward, then 48 greedy steps
(argmax, lowest id on ties).  Stored: the prompt, the generated tokens, and
the top-5 (id, logit) of the step after the prompt.  Run from the repository
root:  python tests/golden/make_tiny_golden.py
"""
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import numpy as np  # noqa: E402

import oracle  # noqa: E402
import synth.workloads as wl  # noqa: E402


def run():
    w = wl.TINY
    m = oracle.Model(w.shape, seed=w.seed)
    s = m.new_state()
    prompt = wl.prompt_tokens(w)
    for t in prompt:
        logits, nxt = s.forward(t)
    first = logits.copy()
    gen = []
    for _ in range(w.steps):
        gen.append(nxt)
        logits, nxt = s.forward(nxt)
    top = np.argsort(-first, kind="stable")[:5]
    return prompt, gen, [(int(i), float(first[i])) for i in top]


if __name__ == "__main__":
    prompt, gen, top = run()
    with open(os.path.join(HERE, "tiny_oracle_greedy.txt"), "w") as f:
        f.write("# oracle greedy run of the tiny fp32 workload (written by make_tiny_golden.py)\n")
        f.write("prompt " + " ".join(map(str, prompt)) + "\n")
        f.write("generated " + " ".join(map(str, gen)) + "\n")
        f.write("top5 " + " ".join(f"{i}:{v:.9g}" for i, v in top) + "\n")
    print("prompt", prompt)
    print("generated", gen)
    print("top5", top)
