"""Host-side checks of the C ABI (no GPU): the library builds, loads and
exports every entry point the header declares; the architecture gates
("Model-agnostic LLM inference", section "Supported models") reject each
mismatch and name all of them; init without a GPU fails cleanly."""
import os
import re

import pytest

import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def pkg():
    from decode_int8_weight_gb300 import build

    build.build()
    import decode_int8_weight_gb300 as p

    p.lib()
    return p


def test_every_declared_symbol_is_exported(pkg):
    header = open(os.path.join(ROOT, "include", "q3i8.h")).read()
    declared = set(re.findall(r"\b(q3i8_[a-z_0-9]+)\s*\(", header))
    assert declared, "no declarations found"
    L = pkg.lib()
    for name in sorted(declared):
        assert hasattr(L, name), f"{name} is declared in q3i8.h but not exported"
    assert declared == set(pkg.EXPORTS)


def _dims(pkg, **kw):
    d = pkg.make_dims(synth.QWEN3_0_6B, max_batch=4)
    for k, v in kw.items():
        setattr(d, k, v)
    return d


def test_supported_shapes_pass(pkg):
    for sh in (synth.TINY, synth.QWEN3_0_6B, synth.QWEN3_1_7B):
        rc, msg = pkg.validate_dims(pkg.make_dims(sh, max_batch=32, max_ctx=6144))
        assert rc == 0, msg


@pytest.mark.parametrize("field,value,needle", [
    ("n_kv_heads", 3, "GQA"),
    ("hidden", 1000, "hidden % 32"),
    ("intermediate", 3000, "intermediate % 32"),
    ("head_dim", 96, "head_dim"),
    ("tie_word_embeddings", 0, "tie_word_embeddings"),
    ("attention_bias", 1, "bias"),
])
def test_each_gate_rejects(pkg, field, value, needle):
    rc, msg = pkg.validate_dims(_dims(pkg, **{field: value}))
    assert rc == 1 and needle in msg, (rc, msg)


def test_all_mismatches_are_named(pkg):
    rc, msg = pkg.validate_dims(_dims(pkg, hidden=1000, tie_word_embeddings=0, attention_bias=1))
    assert rc == 1
    for needle in ("hidden % 32", "tie_word_embeddings", "bias"):
        assert needle in msg
    assert msg.count(";") >= 2


def test_invalid_sizes(pkg):
    rc, msg = pkg.validate_dims(_dims(pkg, vocab=0))
    assert rc == 2 and "vocab" in msg
    rc, msg = pkg.validate_dims(_dims(pkg, max_batch=0))
    assert rc == 2
    rc, msg = pkg.validate_dims(_dims(pkg, max_ctx=70000))
    assert rc == 3


def test_status_names(pkg):
    L = pkg.lib()
    for code, name in pkg.STATUS.items():
        assert L.q3i8_status_name(code).decode() == name


def test_init_without_gpu_reports_no_device(pkg):
    import torch

    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    m = synth.make_model(synth.TINY, 3)
    with pytest.raises(pkg.Q3Error) as e:
        pkg.Decoder(m, max_batch=1)
    assert e.value.status == "no_device"


def test_init_rejects_bad_shape_before_touching_the_device(pkg):
    m = synth.make_model(synth.Shape("odd", 256, 1, 4, 3, 64, 768, 512), 3)
    with pytest.raises(pkg.Q3Error) as e:
        pkg.Decoder(m, max_batch=1)
    assert e.value.status == "unsupported_architecture" and "GQA" in str(e.value)


def test_wait_probe_rejects_missing_status_before_touching_the_device(pkg):
    with pytest.raises(pkg.Q3Error) as e:
        pkg.op_wait_probe(False, 0, None)
    assert e.value.status == "invalid_arguments" and "d_status" in str(e.value)
