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
