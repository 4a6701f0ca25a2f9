"""Write tests/golden/tiny_oracle.json from the CPU oracle alone.

The pages print no worked example (no logits or token ids), so this fixture
is not a value from the pages: it freezes the oracle's own output on the
tiny Qwen3-family member (hidden 256, 2 layers, 4 query / 2 KV heads,
head_dim 64, intermediate 768, vocab 4096; prompt of 8 seeded ids, 16
greedy new tokens) so that later changes to the oracle's arithmetic show up
as a diff that must name the passage justifying it.

It also writes tests/golden/tiny_sampling.json: the sampling chain's tokens
on the same model and prompt for three parameter sets ("Model-agnostic LLM
inference", section "Sampling"), with each step's draw u and the interval of
u that picks the frozen token.

Run:  python tests/golden/make_golden.py
"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
import synth   # noqa: E402
from oracle import sampling  # noqa: E402

SAMPLING_CASES = [
    {"temperature": 0.8, "top_k": 40, "top_p": 0.95, "min_p": 0.0, "repeat_penalty": 1.1},
    {"temperature": 1.3, "top_k": 0, "top_p": 1.0, "min_p": 0.05, "presence_penalty": 0.5,
     "frequency_penalty": 0.25},
    {"temperature": 0.5, "top_k": 8, "top_p": 0.7, "min_p": 0.0},
]
SAMPLING_SEED = 1234


def sampling_fixture(orc, prompt, n_new):
    cases = []
    for kw in SAMPLING_CASES:
        p = sampling.Params(**kw)
        toks = sampling.decode(orc, prompt, n_new, p, SAMPLING_SEED)
        s = orc.seq(len(prompt) + n_new)
        z = s.forward(np.asarray(prompt, np.int32))[-1]
        hist, us, iv = list(prompt), [], []
        for i, t in enumerate(toks):
            u = sampling.uniform(SAMPLING_SEED, 0, i)
            lo, hi = sampling.intervals(z, hist, p)[int(t)]
            us.append(u)
            iv.append([float(f"{lo:.12g}"), float(f"{hi:.12g}")])
            hist.append(int(t))
            z = s.forward(np.asarray([t], np.int32))[-1]
        cases.append({"params": kw, "tokens": [int(t) for t in toks], "u": us, "interval": iv})
    return cases


def main():
    w = synth.WORKLOADS["tiny-b1-p8-n16"]
    m = synth.make_model(w.shape, w.weight_seed)
    orc = oracle.Oracle(m, nthreads=1)
    prompt = synth.prompts(w)[0]
    gen = orc.greedy(prompt, w.new_tokens)
    z = orc.teacher_forced(np.concatenate([prompt, gen[:-1]]), len(prompt) - 1)
    top2 = np.sort(z, axis=1)[:, -2:]
    out = {
        "workload": w.name,
        "weight_seed": w.weight_seed,
        "prompt_seed": w.prompt_seed,
        "prompt": [int(t) for t in prompt],
        "greedy": [int(t) for t in gen],
        "logits_first8": [[float(f"{v:.7g}") for v in row[:8]] for row in z],
        "top1_minus_top2": [float(f"{a - b:.7g}") for b, a in top2],
        "note": "written by tests/golden/make_golden.py from the CPU oracle; not a value from the pages",
    }
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_oracle.json")
    with open(path, "w") as f:
        json.dump(out, f, indent=1)
    print("wrote", path)
    samp = {
        "workload": w.name,
        "seed": SAMPLING_SEED,
        "prompt": [int(t) for t in prompt],
        "cases": sampling_fixture(orc, prompt, w.new_tokens),
        "note": "written by tests/golden/make_golden.py from the CPU oracle; not a value from the pages",
    }
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_sampling.json")
    with open(path, "w") as f:
        json.dump(samp, f, indent=1)
    print("wrote", path)


if __name__ == "__main__":
    main()
