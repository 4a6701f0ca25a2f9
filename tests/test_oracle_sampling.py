"""Pins of the sampling-chain oracle ("Model-agnostic LLM inference", section
"Sampling") to facts fixed outside it: SplitMix64's published first outputs
and the input generator's independent C implementation, closed forms of the
penalties and of the draw's distribution, planted cut-offs of top-k / min-p /
top-p, the order of the chain, and the page's two properties (the same seed
gives the same tokens; top_k = 1 gives the greedy sequence at any
temperature).  No GPU."""
import numpy as np
import pytest

import oracle
import synth
from oracle import sampling as S


def test_splitmix64_published_outputs():
    # the first outputs of SplitMix64 started at seed 0, as printed wherever
    # the generator is used to seed xorshift-family generators
    assert [S.splitmix64_output(0, n) for n in (1, 2, 3)] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4,
                                                             0x06C45D188009454F]


@pytest.mark.parametrize("seed", [0, 1, 1234, 2**63 + 5, 2**64 - 1])
def test_splitmix64_matches_the_generators_c_code(seed):
    # synth/gen.c draws counter c as output c + 1 of the same generator
    d = synth.draws(seed, 64)
    assert [S.splitmix64_output(seed, c + 1) for c in range(64)] == [int(x) for x in d]


def test_uniform_grid_and_streams():
    us = [S.uniform(1234, b, i) for b in range(4) for i in range(64)]
    assert all(0.0 <= u < 1.0 for u in us)
    assert all((u * 2**24).is_integer() for u in us)
    assert len(set(us)) > 250  # (sequence, step) pairs draw distinct values
    assert S.uniform(1234, 2, 7) == S.uniform(1234, 2, 7)
    assert S.uniform(1234, 2, 7) != S.uniform(1235, 2, 7)
    # counter = step * 2^20 + sequence
    assert S.uniform(9, 3, 5) == (S.splitmix64_output(9, 5 * 2**20 + 3 + 1) >> 40) / 2**24


def test_penalties_closed_form():
    z = np.array([2.0, -1.0, 0.5, 3.0, -2.0])
    p = S.Params(temperature=1.0, repeat_penalty=2.0, presence_penalty=0.25, frequency_penalty=0.5)
    out = S.apply_penalties(z, [0, 1, 1, 1, 3], p)
    # token 0 (once, positive): 2/2 - 0.25 - 0.5; token 1 (three times,
    # negative): -1*2 - 0.25 - 1.5; token 3 (once): 3/2 - 0.75; unseen unchanged
    assert out.tolist() == [0.25, -3.75, 0.5, 0.75, -2.0]
    # repetition first, then presence: (2/2) - 1, not (2 - 1)/2
    q = S.Params(temperature=1.0, repeat_penalty=2.0, presence_penalty=1.0)
    assert S.apply_penalties(np.array([2.0]), [0], q)[0] == 0.0
    # neutral settings change nothing
    assert S.apply_penalties(z, [0, 1, 2], S.Params(temperature=1.0)).tolist() == z.tolist()


def test_draw_distribution_is_the_softmax():
    rng = np.random.default_rng(5)
    z = rng.normal(size=12)
    for T in (0.5, 1.0, 2.0):
        p = S.Params(temperature=T)
        iv = S.intervals(z, [], p)
        want = np.exp(z / T - np.max(z / T))
        want /= want.sum()
        # every token survives; interval lengths are its probabilities, in
        # the order (z descending, token ascending), covering [0, 1)
        assert sorted(iv) == list(range(12))
        for t, (lo, hi) in iv.items():
            assert abs((hi - lo) - want[t]) < 1e-15
        ends = sorted(iv.values())
        assert ends[0][0] == 0.0 and abs(ends[-1][1] - 1.0) < 1e-15
        assert all(abs(a[1] - b[0]) == 0.0 for a, b in zip(ends, ends[1:]))
        order = [t for t, _ in sorted(iv.items(), key=lambda kv: kv[1][0])]
        assert order == sorted(range(12), key=lambda t: (-z[t], t))
        # the draw picks the token whose interval holds u (brute force over a grid)
        N = 4096
        counts = np.bincount([S.sample(z, [], p, (i + 0.5) / N) for i in range(N)], minlength=12)
        assert np.all(np.abs(counts - want * N) <= 1.0)


def test_top_k_with_ties():
    z = np.array([1.0, 3.0, 3.0, 2.0])
    assert set(S.intervals(z, [], S.Params(temperature=1.0, top_k=2))) == {1, 2}
    assert list(S.intervals(z, [], S.Params(temperature=1.0, top_k=1))) == [1]  # lowest index among ties
    assert set(S.intervals(z, [], S.Params(temperature=1.0, top_k=3))) == {1, 2, 3}
    assert len(S.intervals(z, [], S.Params(temperature=1.0, top_k=0))) == 4


def test_candidate_order_is_taken_before_the_temperature():
    # two adjacent float64 logits whose quotients by T = 1.5 round to the
    # same value: the order stays the logits' own (the larger first), so
    # top_k = 1 keeps token 1, not the lower index of a tie the division made
    z = np.array([1.9563777446746826, np.nextafter(1.9563777446746826, 3.0)])
    assert z[0] < z[1] and z[0] / 1.5 == z[1] / 1.5
    assert list(S.intervals(z, [], S.Params(temperature=1.5, top_k=1))) == [1]
    assert list(S.intervals(z, [], S.Params(temperature=1.5))) == [1, 0]


def _planted(probs):
    return np.log(np.asarray(probs, np.float64))


def test_min_p_cut():
    z = _planted([0.5, 0.25, 0.15, 0.1])
    assert set(S.intervals(z, [], S.Params(temperature=1.0, min_p=0.35))) == {0, 1}     # >= 0.175
    assert set(S.intervals(z, [], S.Params(temperature=1.0, min_p=0.25))) == {0, 1, 2}  # >= 0.125
    assert set(S.intervals(z, [], S.Params(temperature=1.0, min_p=0.9))) == {0}


def test_top_p_cut_and_renormalisation():
    z = _planted([0.5, 0.25, 0.15, 0.1])
    assert set(S.intervals(z, [], S.Params(temperature=1.0, top_p=0.45))) == {0}
    assert set(S.intervals(z, [], S.Params(temperature=1.0, top_p=0.6))) == {0, 1}
    assert set(S.intervals(z, [], S.Params(temperature=1.0, top_p=0.8))) == {0, 1, 2}
    iv = S.intervals(z, [], S.Params(temperature=1.0, top_p=0.6))
    assert abs(iv[0][1] - 2 / 3) < 1e-15 and iv[1] == (iv[0][1], 1.0)


def test_chain_order_top_k_before_top_p():
    # top-k 3 renormalises to 4/9, 3/9, 2/9; top-p 0.75 then keeps two.  On
    # the full distribution (0.4, 0.3, 0.2, 0.1) top-p 0.75 would keep three.
    z = _planted([0.4, 0.3, 0.2, 0.1])
    assert set(S.intervals(z, [], S.Params(temperature=1.0, top_k=3, top_p=0.75))) == {0, 1}
    # min-p 0.3 keeps probabilities >= 0.3 * 0.4 = 0.12: all but 0.1
    assert set(S.intervals(z, [], S.Params(temperature=1.0, top_k=4, min_p=0.3))) == {0, 1, 2}


def test_temperature_scales_the_logits():
    z = np.array([0.0, np.log(4.0)])
    iv = S.intervals(z, [], S.Params(temperature=2.0))  # probabilities 2:1 at T = 2
    assert abs((iv[1][1] - iv[1][0]) - 2 / 3) < 1e-15


def test_top_k_one_is_greedy_at_any_temperature():
    rng = np.random.default_rng(11)
    for _ in range(50):
        z = rng.normal(size=64).astype(np.float32)
        for T in (0.1, 0.7, 1.0, 5.0):
            for u in (0.0, 0.3, 0.999):
                assert S.sample(z, [1, 2, 3], S.Params(temperature=T, top_k=1), u) == int(np.argmax(z))
    assert S.sample(np.array([1.0, 5.0, 5.0]), [], S.Params(), 0.5) == 1  # temperature 0: argmax, lowest index


def test_sampled_decode_properties_on_the_tiny_model():
    m = synth.make_model(synth.TINY, 3)
    orc = oracle.Oracle(m, nthreads=1)
    prompt = synth.ids(synth.key(9, 0), 8, synth.TINY.vocab)
    p = S.Params(temperature=0.8, top_k=40, top_p=0.95, min_p=0.0, repeat_penalty=1.1)
    a = S.decode(orc, prompt, 24, p, seed=1234)
    b = S.decode(orc, prompt, 24, p, seed=1234)
    c = S.decode(orc, prompt, 24, p, seed=4321)
    assert a.tolist() == b.tolist()          # same seed, same tokens
    assert a.tolist() != c.tolist()          # another seed draws another sequence here
    # top_k = 1 reproduces the greedy sequence at any temperature
    g = orc.greedy(prompt, 24)
    for T in (0.3, 1.0, 3.0):
        assert S.decode(orc, prompt, 24, S.Params(temperature=T, top_k=1), seed=7).tolist() == g.tolist()
    # every sampled token lies in the support the chain allows at its step
    s = orc.seq(len(prompt) + 24)
    z = s.forward(np.asarray(prompt, np.int32))[-1]
    hist = list(prompt)
    for i, t in enumerate(a):
        iv = S.intervals(z, hist, p)
        u = S.uniform(1234, 0, i)
        assert iv[int(t)][0] <= u < iv[int(t)][1]
        hist.append(int(t))
        z = s.forward(np.asarray([t], np.int32))[-1]
