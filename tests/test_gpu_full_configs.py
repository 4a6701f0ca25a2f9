"""GPU parity at full size for the batched (B = 16, 32), Qwen3-1.7B-shape and
long-context workloads, run the way the benchmark runs them: one whole
decode job through q3i8_decode.

The oracle re-scores every generated token in one teacher-forced pass per
sequence, streamed in chunks of 128 positions:
- for a batch, every sequence over every step;
- for the 1.7B job, every step;
- for the long-context job, every one of the 2048 steps.

Greedy tokens follow the tie rule at every re-scored step. Teacher-forced logits agree within 1e-2 on sampled
steps."""
import numpy as np
import pytest

import oracle
import synth
from gpu_common import LOGIT_ATOL, check_greedy_against_oracle, max_abs

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module")
def pkg():
    import torch

    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from decode_int8_weight_gb300 import build

    build.build()
    import decode_int8_weight_gb300 as p

    p.lib()
    return p


def gpu_job(pkg, model, prompts, n_new, max_ctx, logit_steps):
    """Decode the whole job, then the GPU's own teacher-forced logits at logit_steps (step i = the logits that
    predict generated token i)."""
    dec = pkg.Decoder(model, max_batch=len(prompts), max_ctx=max_ctx)
    ids, counts, stats = dec.decode(prompts, n_new)
    assert np.all(counts == n_new)
    keep = {}
    z = dec.prefill(prompts)
    if 0 in logit_steps:
        keep[0] = z
    last = max(logit_steps)
    for i in range(last):
        z = dec.step_logits(ids[:, i])
        if i + 1 in logit_steps:
            keep[i + 1] = z
    dec.close()
    return ids, keep, stats


def oracle_rescore(orc, prompt, gen, n_check, gpu_z, where):
    """Re-score gen[0:n_check] with the oracle, streaming the teacher-forced pass in chunks. The greedy tie rule
    applies at every step. Returns the largest logit difference at the steps in gpu_z ({step: logits})."""
    s = orc.seq(len(prompt) + n_check)
    worst = 0.0

    def consume(rows, step0):
        nonlocal worst
        for r in range(rows.shape[0]):
            i = step0 + r
            check_greedy_against_oracle(gen[i:i + 1], rows[r:r + 1], f"{where} step {i}")
            if i in gpu_z:
                worst = max(worst, max_abs(gpu_z[i], rows[r]))

    consume(s.forward(prompt), 0)  # logits at the last prompt position predict gen[0]
    for j in range(0, n_check - 1, 128):
        chunk = gen[j:min(j + 128, n_check - 1)]
        consume(s.forward(chunk, 0), j + 1)
    return worst


@pytest.mark.parametrize("B", [16, 32])
def test_batched_full_size(pkg, B):
    w = synth.WORKLOADS[f"0.6b-b{B}-p16to256-n128"]
    m = synth.make_model(w.shape, w.weight_seed)
    orc = oracle.Oracle(m)
    prompts = synth.prompts(w)
    steps = set(range(0, w.new_tokens, 16)) | {w.new_tokens - 1}
    ids, gz, _ = gpu_job(pkg, m, prompts, w.new_tokens, w.max_ctx, steps)
    worst = 0.0
    for b in range(B):
        worst = max(worst, oracle_rescore(orc, prompts[b], ids[b], w.new_tokens,
                                          {i: z[b] for i, z in gz.items()}, f"B={B} seq {b}"))
    assert worst <= LOGIT_ATOL, f"max |logit diff| {worst}"


def test_1p7b_full_job(pkg):
    w = synth.WORKLOADS["1.7b-b1-p256-n1024"]
    m = synth.make_model(w.shape, w.weight_seed)
    orc = oracle.Oracle(m)
    prompts = synth.prompts(w)
    steps = set(range(0, w.new_tokens, 64)) | {w.new_tokens - 1}
    ids, gz, _ = gpu_job(pkg, m, prompts, w.new_tokens, w.max_ctx, steps)
    worst = oracle_rescore(orc, prompts[0], ids[0], w.new_tokens, {i: z[0] for i, z in gz.items()}, "1.7b")
    assert worst <= LOGIT_ATOL, f"max |logit diff| {worst}"


def test_long_context_full_job(pkg):
    # 4096-token prompt, 2048 generated tokens (positions 4096..6143): the
    # oracle re-scores every one of them
    w = synth.WORKLOADS["0.6b-b1-p4096-n2048"]
    m = synth.make_model(w.shape, w.weight_seed)
    orc = oracle.Oracle(m)
    prompts = synth.prompts(w)
    steps = {0, 1, 1023, w.new_tokens - 1}
    ids, gz, _ = gpu_job(pkg, m, prompts, w.new_tokens, w.max_ctx, steps)
    worst = oracle_rescore(orc, prompts[0], ids[0], w.new_tokens, {i: z[0] for i, z in gz.items()}, "long context")
    assert worst <= LOGIT_ATOL, f"max |logit diff| {worst}"
