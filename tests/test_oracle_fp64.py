"""Whole-model pin of the oracle: the tiny config evaluated in float64 from
the decoder's definition, in plain numpy, against the fp32 oracle's
teacher-forced logits (within 1e-4).

The float64 pass follows the same definition, including its two fixed
roundings: K (after the per-head RMSNorm and RoPE) and V are rounded to bf16
(round to nearest even) before they enter the cache, and the RoPE cos/sin
table holds float64 values rounded to fp32 ("Model-agnostic LLM inference",
section "Supported models"; "Run local LLM decode", section "Limitations").
Everything else is float64, so the gap measures the oracle's fp32 error.

A cache element whose float64 value lies next to the midpoint between two
bf16 neighbours may round the other way in the oracle's fp32 arithmetic.
Those elements are allowed to differ only where the float64 value is within
fp32 error of that midpoint; the logits are then compared with the float64
pass taking the oracle's rounding of exactly those elements."""
import numpy as np

import oracle
import synth

TOL = 1e-4


def _bf16_rne(x):
    """Round float64 values to the nearest bf16 value (8 significant bits, ties to even)."""
    m, e = np.frexp(x)  # x = m 2^e, 0.5 <= |m| < 1
    return np.ldexp(np.rint(np.ldexp(m, 8)), e - 8)


def _rmsnorm(x, g, eps):
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps) * g


def _rope_table(n, hd, theta):
    half = hd // 2
    freq = theta ** (-2.0 * np.arange(half) / hd)
    ang = np.arange(n)[:, None] * freq[None, :]
    return np.cos(ang).astype(np.float32).astype(np.float64), np.sin(ang).astype(np.float32).astype(np.float64)


def _rope(v, c, s):
    half = v.shape[-1] // 2
    a, b = v[..., :half], v[..., half:]
    return np.concatenate([a * c - b * s, b * c + a * s], axis=-1)


def _w(m):
    return m.q.astype(np.float64) * m.s.astype(np.float64)[:, None]


# How close to a bf16 rounding midpoint a value must be to round either way
# in fp32, measured against its row's RMS: the fp32 error of an element of a
# dot-product row scales with the row, not with the element (an element near
# zero comes from cancellation and carries the row's absolute error).
MIDPOINT_REL = 1e-5


def _match_oracle_rounding(x, bits, where):
    """x: float64 values before the bf16 rounding; bits: the oracle's bf16 bit
    patterns for them.  Returns the rounded values, taking the oracle's choice
    where the two differ, after checking each such element sits at a midpoint."""
    ours = _bf16_rne(x)
    theirs = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    diff = ours != theirs
    if diff.any():
        mid = 0.5 * (ours[diff] + theirs[diff])
        row_rms = np.broadcast_to(np.sqrt(np.mean(x * x, axis=-1, keepdims=True)), x.shape)
        off = np.abs(x[diff] - mid) / row_rms[diff]
        assert np.all(off <= MIDPOINT_REL), f"{where}: a bf16 rounding differs away from a midpoint ({off.max():.2e})"
        assert diff.mean() < 1e-2, f"{where}: {int(diff.sum())} of {diff.size} roundings differ"
    return np.where(diff, theirs, ours)


def forward_fp64(model, ids, oracle_kv=None):
    """Logits [n, vocab] at every position of one causal pass over ids.
    oracle_kv: optional per-layer (k_bits, v_bits) [n_kv, n, hd] of the
    oracle's cache, whose rounding is taken at midpoint elements."""
    sh = model.shape
    n, hd, nh, nkv = len(ids), sh.head_dim, sh.n_heads, sh.n_kv_heads
    group = nh // nkv
    E = _w(model.embed)
    x = E[np.asarray(ids)]
    cos, sin = _rope_table(n, hd, sh.rope_theta)
    causal = np.tril(np.ones((n, n), bool))
    for li, ly in enumerate(model.layers):
        h = _rmsnorm(x, ly.attn_norm.astype(np.float64), sh.rms_eps)
        q = (h @ _w(ly.wq).T).reshape(n, nh, hd)
        k = (h @ _w(ly.wk).T).reshape(n, nkv, hd)
        v = (h @ _w(ly.wv).T).reshape(n, nkv, hd)
        q = _rmsnorm(q, ly.q_norm.astype(np.float64), sh.rms_eps)
        k = _rmsnorm(k, ly.k_norm.astype(np.float64), sh.rms_eps)
        q = _rope(q, cos[:, None, :], sin[:, None, :])
        k = _rope(k, cos[:, None, :], sin[:, None, :])
        if oracle_kv is None:
            k, v = _bf16_rne(k), _bf16_rne(v)
        else:
            kb, vb = oracle_kv[li]
            k = _match_oracle_rounding(k, kb.transpose(1, 0, 2), f"layer {li} K")
            v = _match_oracle_rounding(v, vb.transpose(1, 0, 2), f"layer {li} V")
        o = np.empty((n, nh, hd))
        for j in range(nh):
            g = j // group
            sc = q[:, j, :] @ k[:, g, :].T / np.sqrt(hd)
            sc = np.where(causal, sc, -np.inf)
            p = np.exp(sc - sc.max(axis=1, keepdims=True))
            o[:, j, :] = (p / p.sum(axis=1, keepdims=True)) @ v[:, g, :]
        x = x + o.reshape(n, nh * hd) @ _w(ly.wo).T
        h = _rmsnorm(x, ly.ffn_norm.astype(np.float64), sh.rms_eps)
        gate, up = h @ _w(ly.wg).T, h @ _w(ly.wu).T
        x = x + (gate / (1.0 + np.exp(-gate)) * up) @ _w(ly.wd).T
    h = _rmsnorm(x, model.final_norm.astype(np.float64), sh.rms_eps)
    return h @ E.T


def _check(model, ids):
    orc = oracle.Oracle(model)
    s = orc.seq(len(ids))
    z32 = s.forward(ids, 0).astype(np.float64)
    z64 = forward_fp64(model, ids, [s.kv(l) for l in range(model.shape.n_layers)])
    gap = float(np.max(np.abs(z64 - z32)))
    assert gap <= TOL, f"oracle vs float64: max |logit diff| {gap}"
    return gap


def test_oracle_within_1e4_of_float64_tiny():
    w = synth.WORKLOADS["tiny-b1-p8-n16"]
    m = synth.make_model(w.shape, w.weight_seed)
    prompt = synth.prompts(w)[0]
    gen = oracle.Oracle(m).greedy(prompt, w.new_tokens)
    _check(m, np.concatenate([prompt, gen[:-1]]))


def test_oracle_within_1e4_of_float64_tiny_random_gains():
    w = synth.WORKLOADS["tiny-b1-p8-n16"]
    m = synth.make_model(w.shape, w.weight_seed, random_gains=True)
    ids = synth.ids(synth.key(99, 0), 24, w.shape.vocab)
    _check(m, ids)


def test_float64_pass_is_sensitive_to_a_dropped_rounding():
    # the bf16 rounding of the cache is part of the definition: leaving it
    # out of the float64 pass moves the logits by far more than the tolerance,
    # so the pin above does see that step
    w = synth.WORKLOADS["tiny-b1-p8-n16"]
    m = synth.make_model(w.shape, w.weight_seed)
    ids = synth.ids(synth.key(98, 0), 24, w.shape.vocab)
    keep = _bf16_rne.__code__
    try:
        globals()["_bf16_rne"] = lambda x: x
        z_no_round = forward_fp64(m, ids)
    finally:
        globals()["_bf16_rne"] = _bf16_rne_impl
    z = forward_fp64(m, ids)
    assert float(np.max(np.abs(z - z_no_round))) > 10 * TOL
    del keep


_bf16_rne_impl = _bf16_rne
