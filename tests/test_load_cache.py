"""Quantized load cache ("Model-agnostic LLM inference", section "The
quantized load cache"), host side: the file holds exactly the bytes the
model's arrays hold, its size is the page's cache size for the 0.6B and
1.7B shapes, and the gate (magic + dims + SHA-256 of the manifest + exact
length) refuses every mismatch.  No GPU."""
import hashlib
import os

import numpy as np
import pytest

import synth


@pytest.fixture(scope="module")
def pkg():
    from decode_int8_weight_gb300 import build

    build.build()
    import decode_int8_weight_gb300 as p

    p.lib()
    return p


@pytest.fixture(scope="module")
def tiny():
    return synth.make_model(synth.TINY, 7, random_gains=True)


def _arrays(m):
    """Every array of a model in the cache's file order."""
    out = [m.embed.q, m.embed.s, m.final_norm]
    for ly in m.layers:
        for w in (ly.wq, ly.wk, ly.wv, ly.wo, ly.wg, ly.wu, ly.wd):
            out += [w.q, w.s]
        out += [ly.attn_norm, ly.ffn_norm, ly.q_norm, ly.k_norm]
    return out


def test_payload_size_is_the_pages_cache_size(pkg):
    # the page's table: 0.598 GB (Qwen3-0.6B-Base) and 1.724 GB (Qwen3-1.7B);
    # int8 weights + fp32 scales + fp32 gains, tied embedding counted once
    assert pkg.cache_payload_bytes(synth.QWEN3_0_6B) == 598_230_528
    assert pkg.cache_payload_bytes(synth.QWEN3_1_7B) == 1_723_848_192
    assert pkg.cache_payload_bytes(synth.TINY) == 2_664_448


def test_roundtrip_holds_the_same_bytes(pkg, tiny, tmp_path):
    path = str(tmp_path / "weights_i8.cache")
    pkg.cache_write(path, tiny, b"tiny manifest")
    assert os.path.getsize(path) == 128 + pkg.cache_payload_bytes(synth.TINY)
    cm, gate = pkg.cache_open(path, synth.TINY, b"tiny manifest")
    assert gate == "valid" and cm is not None
    a, b = _arrays(tiny), _arrays(cm)
    assert len(a) == len(b)
    for x, y in zip(a, b):
        assert x.shape == y.shape and x.dtype == y.dtype
        assert np.asarray(x).tobytes() == np.asarray(y).tobytes()
    # the payload is the arrays back to back after the 128-byte header
    raw = open(path, "rb").read()
    assert raw[128:] == b"".join(np.ascontiguousarray(x).tobytes() for x in a)
    cm.close()


def test_header_fields(pkg, tiny, tmp_path):
    path = str(tmp_path / "c")
    manifest = b'{"model": "tiny", "seed": 7}'
    pkg.cache_write(path, tiny, manifest)
    head = open(path, "rb").read(128)
    assert head[:8] == b"Q3I8WC01"
    assert int.from_bytes(head[8:12], "little") == 1
    assert int.from_bytes(head[12:16], "little") == 128
    sh = synth.TINY
    words = [int.from_bytes(head[16 + 4 * i:20 + 4 * i], "little") for i in range(11)]
    assert words[:7] == [sh.hidden, sh.n_layers, sh.n_heads, sh.n_kv_heads, sh.head_dim, sh.intermediate, sh.vocab]
    assert words[7] == int(np.float32(sh.rope_theta).view(np.uint32))
    assert words[8] == int(np.float32(sh.rms_eps).view(np.uint32))
    assert head[60:92] == hashlib.sha256(manifest).digest()
    assert int.from_bytes(head[92:100], "little") == pkg.cache_payload_bytes(sh)
    assert head[100:128] == bytes(28)


@pytest.mark.parametrize("n", [0, 1, 3, 55, 56, 57, 63, 64, 65, 119, 120, 127, 128, 129, 1000, 65537])
def test_manifest_digest_is_sha256(pkg, tiny, tmp_path, n):
    # FIPS 180-4 SHA-256 of manifests across the padding boundaries (55/56/64
    # bytes in the last block) against Python's hashlib
    manifest = bytes((i * 131 + 7) & 255 for i in range(n))
    path = str(tmp_path / f"c{n}")
    pkg.cache_write(path, tiny, manifest)
    assert open(path, "rb").read(92)[60:92] == hashlib.sha256(manifest).digest()


def _gate(pkg, path, shape=synth.TINY, manifest=b"m"):
    cm, gate = pkg.cache_open(path, shape, manifest)
    if cm is not None:
        cm.close()
    return gate


def test_gate_refuses_every_mismatch(pkg, tiny, tmp_path):
    path = str(tmp_path / "c")
    assert _gate(pkg, path) == "absent"
    pkg.cache_write(path, tiny, b"m")
    assert _gate(pkg, path) == "valid"
    # another checkpoint's manifest never passes
    assert _gate(pkg, path, manifest=b"n") == "manifest"
    assert _gate(pkg, path, manifest=b"") == "manifest"
    # other dims (each a gated field)
    import dataclasses
    for field, value in [("vocab", 2048), ("intermediate", 512), ("rms_eps", 1e-5), ("rope_theta", 1e4),
                         ("n_layers", 3)]:
        other = dataclasses.replace(synth.TINY, **{field: value})
        assert _gate(pkg, path, shape=other) == "dims", field
    raw = open(path, "rb").read()
    # truncated and extended files
    for bad in (raw[:-1], raw + b"\0", raw[:128], raw[:100]):
        open(path, "wb").write(bad)
        assert _gate(pkg, path) == "length"
    # not a cache, or another format version
    for bad in (b"", b"Q3I8", b"X" + raw[1:], raw[:8] + (2).to_bytes(4, "little") + raw[12:]):
        open(path, "wb").write(bad)
        assert _gate(pkg, path) == "bad_magic"
    # a header that announces another payload size
    open(path, "wb").write(raw[:92] + (12345).to_bytes(8, "little") + raw[100:])
    assert _gate(pkg, path) == "length"


def test_load_cached_builds_once_then_restores(pkg, tiny, tmp_path):
    path = str(tmp_path / "weights_i8.cache")
    calls = []

    def build():
        calls.append(1)
        return tiny

    m1, gate1 = pkg.load_cached(path, synth.TINY, b"tiny/7", build)
    assert gate1 == "absent" and m1 is tiny and len(calls) == 1
    m2, gate2 = pkg.load_cached(path, synth.TINY, b"tiny/7", build)
    assert gate2 == "valid" and len(calls) == 1
    assert all(np.array_equal(x, y) for x, y in zip(_arrays(tiny), _arrays(m2)))
    m2.close()
    # a different checkpoint rebuilds and rewrites the cache
    m3, gate3 = pkg.load_cached(path, synth.TINY, b"tiny/8", build)
    assert gate3 == "manifest" and len(calls) == 2
    m4, gate4 = pkg.load_cached(path, synth.TINY, b"tiny/8", build)
    assert gate4 == "valid" and len(calls) == 2
    m4.close()


def test_write_and_open_errors(pkg, tiny, tmp_path):
    import dataclasses

    bad = dataclasses.replace(synth.TINY, n_kv_heads=3)  # GQA gate
    with pytest.raises(pkg.Q3Error) as e:
        pkg.cache_open(str(tmp_path / "c"), bad, b"")
    assert e.value.status == "unsupported_architecture"
    with pytest.raises(pkg.Q3Error) as e:
        pkg.cache_write(str(tmp_path / "no_such_dir" / "c"), tiny, b"")
    assert e.value.status == "invalid_arguments"
    assert not any(p.name.startswith("c.tmp") for p in tmp_path.iterdir())


def test_cached_model_feeds_the_decoder_tables(pkg, tiny, tmp_path):
    # the host tables q3i8_init would receive point at the cache's bytes and
    # hold the model's values (init itself needs a GPU)
    path = str(tmp_path / "c")
    pkg.cache_write(path, tiny, b"")
    cm, gate = pkg.cache_open(path, synth.TINY, b"")
    assert gate == "valid"
    emb, layers, fin, keep = pkg._host_tables(cm)
    import ctypes

    def view(addr, ctype, n):
        return np.ctypeslib.as_array(ctypes.cast(addr, ctypes.POINTER(ctype)), shape=(n,))

    sh = synth.TINY
    assert np.array_equal(view(emb.w, ctypes.c_int8, sh.vocab * sh.hidden), tiny.embed.q.ravel())
    assert np.array_equal(view(fin, ctypes.c_float, sh.hidden), tiny.final_norm)
    last = layers[sh.n_layers - 1]
    assert np.array_equal(view(last.down.w, ctypes.c_int8, sh.hidden * sh.intermediate), tiny.layers[-1].wd.q.ravel())
    assert np.array_equal(view(last.k_norm, ctypes.c_float, sh.head_dim), tiny.layers[-1].k_norm)
    import torch

    if not torch.cuda.is_available():
        with pytest.raises(pkg.Q3Error) as e:
            pkg.Decoder(cm, max_batch=1)
        assert e.value.status == "no_device"
    cm.close()
