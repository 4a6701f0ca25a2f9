"""GPU parity: the CUDA path through the C ABI against the CPU oracle on the
same seeded inputs.  Integer work is compared bit for bit (argmax index on
clear maxima, KV cache slots); logits within 1e-2 absolute; greedy tokens
identical wherever the oracle's top-1/top-2 gap exceeds 1e-2."""
import numpy as np
import pytest

import oracle
import synth
from gpu_common import LOGIT_ATOL, check_greedy_against_oracle, max_abs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkg():
    import torch

    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from decode_int8_weight_gb300 import build

    build.build()
    import decode_int8_weight_gb300 as p

    p.lib()
    return p


_models = {}


def model_for(name, random_gains=False):
    key = (name, random_gains)
    if key not in _models:
        w = synth.WORKLOADS[name]
        m = synth.make_model(w.shape, w.weight_seed, random_gains=random_gains)
        _models[key] = (m, oracle.Oracle(m))
    return _models[key]


def _teacher_forced_check(pkg, name, B=None, random_gains=False, steps=None, max_ctx=None):
    w = synth.WORKLOADS[name]
    m, orc = model_for(name, random_gains)
    prompts = synth.prompts(w, B)
    n_new = steps or w.new_tokens
    dec = pkg.Decoder(m, max_batch=len(prompts), max_ctx=max_ctx or w.max_ctx)
    ids, counts, stats = dec.decode(prompts, n_new)
    assert np.all(counts == n_new)
    # teacher-forced GPU logits along the GPU's own tokens
    z0 = dec.prefill(prompts)
    gpu_z = [z0]
    for i in range(n_new - 1):
        gpu_z.append(dec.step_logits(ids[:, i]))
    gpu_z = np.stack(gpu_z, 1)  # [B, n_new, V]
    worst = 0.0
    for b, p in enumerate(prompts):
        zo = orc.teacher_forced(np.concatenate([p, ids[b, :-1]]), len(p) - 1)
        check_greedy_against_oracle(ids[b], zo, f"{name} seq {b}")
        worst = max(worst, max_abs(gpu_z[b], zo))
        # the decode path's tokens are the argmax of its own teacher-forced logits
        assert np.array_equal(np.argmax(gpu_z[b], axis=1), ids[b])
    assert worst <= LOGIT_ATOL, f"max |logit diff| {worst}"
    dec.close()
    return worst, stats


def test_tiny_b1_greedy_and_logits(pkg):
    worst, _ = _teacher_forced_check(pkg, "tiny-b1-p8-n16")
    assert worst < 1e-3


def test_tiny_one_attention_split(pkg):
    # a 64-position context is one KV chunk, so the decode attention runs one
    # split per kv head and writes its output itself, with no merge launch
    worst, _ = _teacher_forced_check(pkg, "tiny-b1-p8-n16", B=3, max_ctx=64)
    assert worst < 1e-3


def test_tiny_random_gains(pkg):
    _teacher_forced_check(pkg, "tiny-b1-p8-n16", random_gains=True)


def test_tiny_batched_ragged(pkg):
    w = synth.WORKLOADS["tiny-b1-p8-n16"]
    m, orc = model_for(w.name)
    prompts = [synth.ids(synth.key(77, b), n, w.shape.vocab) for b, n in enumerate([1, 5, 64, 65, 13, 130])]
    dec = pkg.Decoder(m, max_batch=8, max_ctx=512)
    ids, counts, _ = dec.decode(prompts, 12)
    for b, p in enumerate(prompts):
        zo = orc.teacher_forced(np.concatenate([p, ids[b, :-1]]), len(p) - 1)
        check_greedy_against_oracle(ids[b], zo, f"seq {b}")
    dec.close()


def test_kv_cache_slots_match_oracle_bits(pkg):
    w = synth.WORKLOADS["tiny-b1-p8-n16"]
    m, orc = model_for(w.name)
    prompt = synth.prompts(w)[0]
    dec = pkg.Decoder(m, max_batch=2, max_ctx=512)
    dec.prefill([prompt, prompt[:3]])
    s = orc.seq(len(prompt))
    s.forward(prompt)
    for layer in range(w.shape.n_layers):
        k, v = dec.read_kv(layer, 0, len(prompt))
        ko, vo = s.kv(layer)
        for a, b in ((k, ko), (v, vo)):
            # identical fp32 inputs give identical bf16 bits; otherwise at most 1 bf16 ulp
            d = np.abs(a.astype(np.int32) - b.astype(np.int32))
            assert d.max() <= 1, f"layer {layer}: bf16 bits differ by {d.max()}"
            assert (d == 0).mean() > 0.97
    dec.close()


def test_0p6b_b1_full(pkg):
    worst, stats = _teacher_forced_check(pkg, "0.6b-b1-p32-n128")
    print("0.6b b1 max |dlogit|", worst, stats)


def test_0p6b_b8_ragged(pkg):
    _teacher_forced_check(pkg, "0.6b-b8-p16to256-n128", steps=24)


def test_0p6b_b1_persistent_kernel(pkg, monkeypatch):
    # the persistent step kernel (staged operands, B <= 4) on the full job
    monkeypatch.setenv("Q3I8_PERSISTENT_MAX_BATCH", "4")
    worst, _ = _teacher_forced_check(pkg, "0.6b-b1-p32-n128")
    print("persistent 0.6b b1 max |dlogit|", worst)


def test_tiny_persistent_kernel_deterministic(pkg, monkeypatch):
    monkeypatch.setenv("Q3I8_PERSISTENT_MAX_BATCH", "4")
    _teacher_forced_check(pkg, "tiny-b1-p8-n16")
    w = synth.WORKLOADS["tiny-b1-p8-n16"]
    m, _ = model_for(w.name)
    dec = pkg.Decoder(m, max_batch=1, max_ctx=w.max_ctx)
    p = synth.prompts(w)
    a, _, _ = dec.decode(p, 16)
    b, _, _ = dec.decode(p, 16)
    assert np.array_equal(a, b)
    dec.close()


def test_0p6b_b8_persistent_operands_from_words(pkg, monkeypatch):
    # B > 4 decodes with the chained kernels by default; this keeps the
    # persistent kernel's wide-batch path (operands read from the flagged
    # words) under test
    monkeypatch.setenv("Q3I8_PERSISTENT_MAX_BATCH", "32")
    _teacher_forced_check(pkg, "0.6b-b8-p16to256-n128", steps=12)


def test_decode_is_deterministic(pkg):
    w = synth.WORKLOADS["tiny-b1-p8-n16"]
    m, _ = model_for(w.name)
    dec = pkg.Decoder(m, max_batch=1, max_ctx=w.max_ctx)
    p = synth.prompts(w)
    a, _, _ = dec.decode(p, 16)
    b, _, _ = dec.decode(p, 16)
    assert np.array_equal(a, b)
    dec.close()


def test_eos_counts_and_errors(pkg):
    w = synth.WORKLOADS["tiny-b1-p8-n16"]
    m, _ = model_for(w.name)
    dec = pkg.Decoder(m, max_batch=2, max_ctx=64)
    p = synth.prompts(w)
    ids, counts, _ = dec.decode(p, 8)
    eos = int(ids[0, 2])
    ids2, counts2, _ = dec.decode(p, 8, eos_id=eos)
    first = int(np.argmax(ids[0] == eos))
    assert counts2[0] == first + 1
    with pytest.raises(pkg.Q3Error) as e:
        dec.decode([np.array([], np.int32)], 4)
    assert e.value.status == "invalid_arguments"
    with pytest.raises(pkg.Q3Error) as e:
        dec.decode([np.array([w.shape.vocab], np.int32)], 4)
    assert e.value.status == "invalid_arguments"
    with pytest.raises(pkg.Q3Error) as e:
        dec.decode(p, 0)
    assert e.value.status == "invalid_arguments"
    with pytest.raises(pkg.Q3Error) as e:
        dec.decode(p * 3, 4)
    assert e.value.status == "invalid_arguments"
    with pytest.raises(pkg.Q3Error) as e:
        dec.decode(p, 70000)
    assert e.value.status == "context_past_ceiling"
    # context auto-raise past the initial 64 positions
    ids3, _, _ = dec.decode(p, 100)
    assert np.array_equal(ids3[0, :8], ids[0])
    dec.close()
    dec = pkg.Decoder(m, max_batch=1)
    with pytest.raises(pkg.Q3Error) as e:
        dec.step_logits(np.array([1], np.int32))
    assert e.value.status == "invalid_state"
    dec.close()
