"""Pins of the CPU oracle against closed forms, invariants, library routines
and brute force (no GPU).  Every oracle function is covered here; see the
oracle's header for which passage each follows.

A plausible mistake anywhere in the oracle (a dropped gain or residual, a
wrong sign or pairing in RoPE, a wrong GQA index, a transposed weight, a
misplaced bf16 rounding, an off-by-one position) fails at least one test.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import synth

rng = np.random.default_rng(1234)


# ----------------------------------------------------------------- bf16 rounding

def test_bf16_round_half_even_exact_cases():
    # 1 + 2^-8 is exactly halfway between bf16 1.0 and 1 + 2^-7: ties to even (1.0)
    assert oracle.bf16_bits(1.0) == 0x3F80
    assert oracle.bf16_bits(1.0 + 2 ** -8) == 0x3F80
    # 1 + 3*2^-8 is halfway between 1 + 2^-7 (odd mantissa) and 1 + 2^-6: goes up
    assert oracle.bf16_bits(1.0 + 3 * 2 ** -8) == 0x3F82
    assert oracle.bf16_bits(-2.0) == 0xC000
    assert oracle.bf16_value(0x3F80) == 1.0


def test_bf16_matches_library_conversion():
    x = (rng.standard_normal(4096) * np.exp(rng.uniform(-20, 20, 4096))).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.bf16_bits(float(v)) for v in x], np.uint16)
    assert np.array_equal(got, ref)


# ----------------------------------------------------------------- RMSNorm

@pytest.mark.parametrize("c", [1.0, -3.5, 1e-3, 2.0e-3])
def test_rmsnorm_constant_vector_closed_form(c):
    # x = c * ones: mean(x^2) = c^2, y = c / sqrt(c^2 + eps) * g = sign(c) g / sqrt(1 + eps / c^2)
    n, eps = 64, 1e-6
    g = rng.uniform(0.5, 1.5, n).astype(np.float32)
    y = oracle.rmsnorm(np.full(n, c, np.float32), g, eps)
    expect = math.copysign(1.0, c) * g.astype(np.float64) / math.sqrt(1.0 + eps / (c * c))
    np.testing.assert_allclose(y, expect, rtol=2e-6)


def test_rmsnorm_scale_invariance_and_gain():
    n, eps = 1024, 1e-6
    x = rng.standard_normal(n).astype(np.float32)
    g = rng.uniform(0.5, 1.5, n).astype(np.float32)
    y1 = oracle.rmsnorm(x, g, eps)
    y2 = oracle.rmsnorm(np.float32(8.0) * x, g, eps)
    np.testing.assert_allclose(y1, y2, rtol=1e-5, atol=1e-6)
    # unit rms output before the gain
    ones = oracle.rmsnorm(x, np.ones(n, np.float32), eps)
    assert abs(np.sqrt(np.mean(ones.astype(np.float64) ** 2)) - 1.0) < 1e-5
    np.testing.assert_allclose(y1, ones * g, rtol=1e-6)


# ----------------------------------------------------------------- RoPE

def test_rope_position_zero_is_identity():
    v = rng.standard_normal(128).astype(np.float32)
    assert np.array_equal(oracle.rope(v, 0, 1e6), v)


def test_rope_hand_computed_2d():
    # hd = 2: the only frequency is theta^0 = 1, so position p rotates (a, b) by p radians
    for p in (1, 2, 7, 1000):
        a, b = 0.75, -0.25
        got = oracle.rope(np.array([a, b], np.float32), p, 1e6)
        c, s = math.cos(p), math.sin(p)
        np.testing.assert_allclose(got, [a * c - b * s, b * c + a * s], rtol=1e-6, atol=1e-7)


def test_rope_rotate_half_pairing_and_frequencies():
    # hd = 4, theta = 1e6: pairs (0, 2) at frequency 1 and (1, 3) at frequency 1e6^(-1/2) = 1e-3
    p = 5
    v = np.array([1.0, 2.0, 3.0, 4.0], np.float32)
    got = oracle.rope(v, p, 1e6)
    f1 = 1e6 ** (-2.0 / 4.0)
    e = np.empty(4)
    for i, f in ((0, 1.0), (1, f1)):
        c, s = math.cos(p * f), math.sin(p * f)
        e[i] = v[i] * c - v[i + 2] * s
        e[i + 2] = v[i + 2] * c + v[i] * s
    np.testing.assert_allclose(got, e, rtol=1e-6, atol=1e-7)


def test_rope_preserves_norm_and_is_relative():
    hd = 128
    q = rng.standard_normal(hd).astype(np.float32)
    k = rng.standard_normal(hd).astype(np.float32)
    for p in (1, 17, 4095):
        assert abs(np.linalg.norm(oracle.rope(q, p, 1e6)) - np.linalg.norm(q)) < 1e-4
    # <R_p q, R_p' k> depends only on p - p'
    d1 = float(np.dot(oracle.rope(q, 10, 1e6).astype(np.float64), oracle.rope(k, 3, 1e6)))
    d2 = float(np.dot(oracle.rope(q, 107, 1e6).astype(np.float64), oracle.rope(k, 100, 1e6)))
    assert abs(d1 - d2) < 1e-4


# ----------------------------------------------------------------- SiLU

def test_silu_special_values_and_double():
    assert oracle.silu(0.0) == 0.0
    assert abs(oracle.silu(30.0) - 30.0) < 1e-5
    assert abs(oracle.silu(-30.0)) < 1e-10
    for z in np.linspace(-12, 12, 97):
        z32 = float(np.float32(z))
        ref = z32 / (1.0 + math.exp(-z32))
        assert abs(oracle.silu(z32) - ref) <= 4e-7 * max(1.0, abs(ref))


# ----------------------------------------------------------------- int8 matmul

def test_matmul_i8_matches_library_matmul_non_square():
    rows, cols, m = 37, 96, 5
    q = rng.integers(-127, 128, (rows, cols), dtype=np.int8)
    s = rng.uniform(1e-4, 1e-2, rows).astype(np.float32)
    x = rng.standard_normal((m, cols)).astype(np.float32)
    y = oracle.matmul_i8(q, s, x, nthreads=3)
    ref = (x.astype(np.float64) @ q.astype(np.float64).T) * s.astype(np.float64)
    np.testing.assert_allclose(y, ref, rtol=2e-5, atol=1e-7)
    # single vector and the many-token path agree exactly (same per-output summation)
    assert np.array_equal(oracle.matmul_i8(q, s, x[2]), y[2])
    # more than 64 tokens crosses the token-block boundary
    xb = rng.standard_normal((130, cols)).astype(np.float32)
    yb = oracle.matmul_i8(q, s, xb, nthreads=2)
    assert np.array_equal(yb[129], oracle.matmul_i8(q, s, xb[129]))


# ----------------------------------------------------------------- attention

def _bits(a):
    return np.array([oracle.bf16_bits(float(v)) for v in np.ravel(a)], np.uint16).reshape(np.shape(a))


def _vals(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32)


def test_attention_single_position_returns_v_of_its_group():
    nh, nkv, hd = 8, 2, 16
    q = rng.standard_normal((nh, hd)).astype(np.float32)
    k = _bits(rng.standard_normal((nkv, 1, hd)))
    v = _bits(rng.standard_normal((nkv, 1, hd)))
    out = oracle.attention(q, k, v, 1)
    group = nh // nkv
    for j in range(nh):
        # consecutive query heads share a kv head: j // group, not j % n_kv
        assert np.array_equal(out[j], _vals(v[j // group, 0]))


def test_attention_equal_scores_give_mean_of_v():
    nh, nkv, hd, n = 4, 4, 8, 5
    q = np.zeros((nh, hd), np.float32)
    k = _bits(rng.standard_normal((nkv, n, hd)))
    v = _bits(rng.standard_normal((nkv, n, hd)))
    out = oracle.attention(q, k, v, n)
    np.testing.assert_allclose(out, _vals(v).astype(np.float64).mean(axis=1), rtol=1e-6, atol=1e-7)


def test_attention_brute_force_double():
    nh, nkv, hd = 4, 2, 4
    for n in range(1, 6):
        q = rng.standard_normal((nh, hd)).astype(np.float32) * 2
        k = _bits(rng.standard_normal((nkv, 6, hd)))
        v = _bits(rng.standard_normal((nkv, 6, hd)))
        out = oracle.attention(q, k, v, n)
        kf, vf = _vals(k).astype(np.float64), _vals(v).astype(np.float64)
        for j in range(nh):
            g = j // (nh // nkv)
            sc = np.array([np.dot(q[j].astype(np.float64), kf[g, t]) / math.sqrt(hd) for t in range(n)])
            p = np.exp(sc - sc.max())
            p /= p.sum()
            ref = (p[:, None] * vf[g, :n]).sum(axis=0)
            np.testing.assert_allclose(out[j], ref, rtol=1e-5, atol=1e-6)


def test_attention_gqa_equals_duplicated_mha():
    nh, nkv, hd, n = 6, 2, 8, 4
    q = rng.standard_normal((nh, hd)).astype(np.float32)
    k = _bits(rng.standard_normal((nkv, n, hd)))
    v = _bits(rng.standard_normal((nkv, n, hd)))
    gqa = oracle.attention(q, k, v, n)
    kd = np.repeat(k, nh // nkv, axis=0)
    vd = np.repeat(v, nh // nkv, axis=0)
    assert np.array_equal(gqa, oracle.attention(q, kd, vd, n))
    # identical queries inside one group give identical outputs
    q2 = q.copy()
    q2[1] = q2[0]
    o2 = oracle.attention(q2, k, v, n)
    assert np.array_equal(o2[0], o2[1])


# ----------------------------------------------------------------- argmax

def test_argmax_planted_and_ties():
    z = rng.standard_normal(1000).astype(np.float32)
    z[0] = 10
    assert oracle.argmax(z) == 0
    z[0] = 0
    z[999] = 10
    assert oracle.argmax(z) == 999
    z[500] = 10
    assert oracle.argmax(z) == 500          # lowest index of the tie
    assert oracle.argmax(np.zeros(17, np.float32)) == 0
    assert oracle.argmax(np.full(17, -np.inf, np.float32)) == 0


# ----------------------------------------------------------------- quantiser (input preparation)

def test_quantiser_round_trip_and_extremes():
    bits = synth.normal_bf16(synth.key(5, 0), 64 * 300)
    w = synth.bf16_bits_to_f32(bits).reshape(64, 300)
    q, s = synth.quantize_rows(bits.reshape(64, 300))
    deq = q.astype(np.float64) * s[:, None]
    # fp32 quotient w/s carries one rounding, so the half-step bound holds to ~1e-5
    assert np.all(np.abs(deq - w) <= s[:, None] * (0.5 + 1e-5))
    assert np.all(np.abs(q).max(axis=1) == 127)           # the amax element maps to +-127
    amax_col = np.abs(w).argmax(axis=1)
    assert np.all(np.abs(q[np.arange(64), amax_col]) == 127)
    q2, s2 = synth.quantize_rows((q.astype(np.float32) * s[:, None]).astype(np.float32))
    assert np.array_equal(q2, q)                           # re-quantising is exact
    np.testing.assert_allclose(s2, s, rtol=1e-6)
    z = np.zeros((2, 32), np.float32)
    qz, sz = synth.quantize_rows(z)
    assert np.all(qz == 0) and np.all(sz == 1.0)


# ----------------------------------------------------------------- whole model

def _small_model(layers=1, random_gains=True, seed=77):
    sh = synth.Shape("pin-small", 64, layers, 4, 2, 16, 96, 200)
    return synth.make_model(sh, seed, sigma=0.05, random_gains=random_gains)


def test_zero_layers_reduce_to_embedding_lm_head_closed_form():
    m = _small_model(layers=2)
    for ly in m.layers:
        for name in ("wq", "wk", "wv", "wo", "wg", "wu", "wd"):
            getattr(ly, name).q[:] = 0
    orc = oracle.Oracle(m, nthreads=2)
    ids = np.array([3, 150, 7], np.int32)
    z = orc.teacher_forced(ids, 0)
    E = m.embed.q.astype(np.float64) * m.embed.s[:, None].astype(np.float64)
    for t, tok in enumerate(ids):
        x = E[tok]
        h = x / np.sqrt(np.mean(x * x) + 1e-6) * m.final_norm
        ref = E @ h
        np.testing.assert_allclose(z[t], ref, rtol=1e-4, atol=1e-6)


def _layer_from_pieces(m, ly, x, pos_list, kc, vc):
    """One decoder layer for the rows of x at positions pos_list, using only
    oracle pieces (each pinned above) and numpy glue."""
    sh = m.shape
    hd, nh, nkv = sh.head_dim, sh.n_heads, sh.n_kv_heads
    out = []
    for t, pos in enumerate(pos_list):
        h = oracle.rmsnorm(x[t], ly.attn_norm, sh.rms_eps)
        q = oracle.matmul_i8(ly.wq.q, ly.wq.s, h).reshape(nh, hd)
        k = oracle.matmul_i8(ly.wk.q, ly.wk.s, h).reshape(nkv, hd)
        v = oracle.matmul_i8(ly.wv.q, ly.wv.s, h).reshape(nkv, hd)
        q = np.stack([oracle.rope(oracle.rmsnorm(q[j], ly.q_norm, sh.rms_eps), pos, sh.rope_theta)
                      for j in range(nh)])
        k = np.stack([oracle.rope(oracle.rmsnorm(k[g], ly.k_norm, sh.rms_eps), pos, sh.rope_theta)
                      for g in range(nkv)])
        kc[:, pos] = _bits(k)
        vc[:, pos] = _bits(v)
        o = oracle.attention(q, kc, vc, pos + 1).reshape(-1)
        x1 = x[t] + oracle.matmul_i8(ly.wo.q, ly.wo.s, o)
        h2 = oracle.rmsnorm(x1, ly.ffn_norm, sh.rms_eps)
        g = oracle.matmul_i8(ly.wg.q, ly.wg.s, h2)
        u = oracle.matmul_i8(ly.wu.q, ly.wu.s, h2)
        a = np.array([oracle.silu(float(gi)) for gi in g], np.float32) * u
        out.append(x1 + oracle.matmul_i8(ly.wd.q, ly.wd.s, a))
    return np.stack(out)


def test_model_composition_matches_pinned_pieces():
    m = _small_model(layers=2)
    sh = m.shape
    orc = oracle.Oracle(m, nthreads=2)
    ids = np.array([5, 199, 0, 42], np.int32)
    z = orc.teacher_forced(ids, 0)
    x = np.stack([m.embed.q[t].astype(np.float32) * m.embed.s[t] for t in ids])
    kcs = [np.zeros((sh.n_kv_heads, len(ids), sh.head_dim), np.uint16) for _ in m.layers]
    vcs = [np.zeros_like(kcs[0]) for _ in m.layers]
    for li, ly in enumerate(m.layers):
        x = _layer_from_pieces(m, ly, x, list(range(len(ids))), kcs[li], vcs[li])
    for t in range(len(ids)):
        h = oracle.rmsnorm(x[t], m.final_norm, sh.rms_eps)
        ref = oracle.matmul_i8(m.embed.q, m.embed.s, h)
        np.testing.assert_allclose(z[t], ref, rtol=1e-5, atol=1e-6)
    # the stored cache holds exactly the bf16 K / V of the composition
    s = orc.seq(len(ids))
    s.forward(ids)
    for li in range(sh.n_layers):
        k, v = s.kv(li)
        assert np.array_equal(k, kcs[li]) and np.array_equal(v, vcs[li])


def test_teacher_forced_equals_step_by_step_and_is_causal():
    m = _small_model(layers=2, random_gains=False)
    orc = oracle.Oracle(m, nthreads=3)
    ids = synth.ids(synth.key(9, 0), 12, m.shape.vocab)
    full = orc.teacher_forced(ids, 0)
    s = orc.seq(12)
    rows = [s.forward(ids[:5], 0)]
    for t in range(5, 12):
        rows.append(s.forward(ids[t:t + 1], 0))
    step = np.concatenate(rows)
    assert np.array_equal(full, step)                      # bit-exact
    ids2 = ids.copy()
    ids2[8] = (ids2[8] + 1) % m.shape.vocab
    full2 = orc.teacher_forced(ids2, 0)
    assert np.array_equal(full[:8], full2[:8])             # earlier positions unaffected
    assert not np.array_equal(full[8], full2[8])


def test_greedy_is_argmax_of_teacher_forced():
    m = _small_model(layers=2)
    orc = oracle.Oracle(m, nthreads=2)
    prompt = np.array([1, 2, 3], np.int32)
    gen = orc.greedy(prompt, 6)
    z = orc.teacher_forced(np.concatenate([prompt, gen[:-1]]), len(prompt) - 1)
    assert [int(np.argmax(r)) for r in z] == list(gen)
    assert len(orc.greedy(prompt, 6, eos_id=int(gen[1]))) == 2
