"""Quantized load cache on the GPU ("Model-agnostic LLM inference", section
"The quantized load cache": cached and cold calls give byte-identical greedy
sequences).  A context initialised from a cache's tables decodes the same
ids and the same prefill logits, bit for bit, as one initialised from the
model's own arrays.  Collected after the parity tests."""
import numpy as np
import pytest

import synth

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


def _run(pkg, model, w, prompts, n_new):
    dec = pkg.Decoder(model, max_batch=len(prompts), max_ctx=w.max_ctx)
    ids, counts, _ = dec.decode(prompts, n_new)
    z = dec.prefill(prompts)
    dec.close()
    return ids, counts, np.ascontiguousarray(z)


@pytest.mark.parametrize("name,n_new", [("tiny-b1-p8-n16", 16), ("0.6b-b1-p32-n128", 16)])
def test_cached_and_cold_decode_are_byte_identical(pkg, tmp_path, name, n_new):
    w = synth.WORKLOADS[name]
    cold = synth.make_model(w.shape, w.weight_seed)
    manifest = f"{w.shape.name}/seed={w.weight_seed}".encode()
    path = str(tmp_path / "weights_i8.cache")
    pkg.cache_write(path, cold, manifest)
    cached, gate = pkg.cache_open(path, w.shape, manifest)
    assert gate == "valid"
    prompts = synth.prompts(w)
    ids0, counts0, z0 = _run(pkg, cold, w, prompts, n_new)
    ids1, counts1, z1 = _run(pkg, cached, w, prompts, n_new)
    cached.close()
    assert np.array_equal(counts0, counts1) and np.array_equal(ids0, ids1)
    assert z0.tobytes() == z1.tobytes()
