"""The oracle still reproduces its frozen tiny-model output (regression pin).
The fixture comes from tests/golden/make_golden.py, which calls only the
oracle and the input generator."""
import json
import os

import numpy as np

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "tiny_oracle.json")


def test_tiny_oracle_matches_frozen_fixture():
    g = json.load(open(GOLDEN))
    w = synth.WORKLOADS[g["workload"]]
    m = synth.make_model(w.shape, w.weight_seed)
    prompt = synth.prompts(w)[0]
    assert [int(t) for t in prompt] == g["prompt"]
    orc = oracle.Oracle(m, nthreads=2)
    frozen = np.array(g["greedy"], np.int32)
    z = orc.teacher_forced(np.concatenate([prompt, frozen[:-1]]), len(prompt) - 1)
    np.testing.assert_allclose(z[:, :8], np.array(g["logits_first8"]), rtol=1e-5, atol=1e-6)
    # argmax agrees wherever the frozen top-1/top-2 gap is not a near tie
    for i in range(len(frozen)):
        if g["top1_minus_top2"][i] > 1e-4:
            assert int(np.argmax(z[i])) == frozen[i], f"step {i}"
    # free-running greedy agrees up to the first near tie
    gen = orc.greedy(prompt, w.new_tokens)
    for i in range(len(frozen)):
        if g["top1_minus_top2"][i] <= 1e-4:
            break
        assert gen[i] == frozen[i], f"step {i}"


SAMPLING = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "tiny_sampling.json")


def test_sampling_oracle_matches_frozen_fixture():
    # the sampling chain ("Model-agnostic LLM inference", section "Sampling")
    # still draws the frozen tokens, with the frozen draws and intervals
    from oracle import sampling

    g = json.load(open(SAMPLING))
    w = synth.WORKLOADS[g["workload"]]
    orc = oracle.Oracle(synth.make_model(w.shape, w.weight_seed), nthreads=2)
    prompt = synth.prompts(w)[0]
    assert [int(t) for t in prompt] == g["prompt"]
    for case in g["cases"]:
        p = sampling.Params(**case["params"])
        us = [sampling.uniform(g["seed"], 0, i) for i in range(len(case["tokens"]))]
        assert us == case["u"]
        for (lo, hi), u in zip(case["interval"], us):
            assert lo <= u < hi
        toks = sampling.decode(orc, prompt, len(case["tokens"]), p, g["seed"])
        assert toks.tolist() == case["tokens"], case["params"]
