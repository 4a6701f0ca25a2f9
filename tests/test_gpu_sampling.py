"""GPU parity of the seeded sampling chain ("Model-agnostic LLM inference",
section "Sampling") against the CPU oracle's chain (oracle.sampling), through
the C ABI.

Two levels.  The op (q3i8_op_sample) on seeded synthetic logits at the full
Qwen3 vocabulary, with histories for the penalties and planted ties: every
drawn token must be the oracle's, whose float64 arithmetic it shares step
for step.  And the whole sampled decode (q3i8_decode_sample): the decode's
own logits are re-computed teacher-forced on the GPU (the same kernels, so
the same bits), and every sampled token must be the oracle chain's draw on
those logits with the draw u of its (seed, sequence, step).  The only
allowed difference is a draw within 1e-12 of the boundary between two
tokens' intervals, where the summation order of the probabilities decides;
the tests count such cases and expect none on these inputs.
"""
import numpy as np
import pytest

import oracle
import synth
from oracle import sampling as S

pytestmark = pytest.mark.gpu

BOUNDARY = 1e-12


@pytest.fixture(scope="module")
def pkg():
    import torch

    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from decode_int8_weight_gb300 import build

    build.build()
    import decode_int8_weight_gb300 as p

    p.lib()
    return p


SETTINGS = [
    dict(temperature=0.8, top_k=40, top_p=0.95, min_p=0.0, repeat_penalty=1.1),
    dict(temperature=1.3, top_k=4096, top_p=1.0, min_p=0.05, presence_penalty=0.5, frequency_penalty=0.25),
    dict(temperature=0.5, top_k=8, top_p=0.7),
    dict(temperature=2.0, top_k=1000, top_p=0.9, repeat_penalty=1.3, frequency_penalty=0.1),
    dict(temperature=1.0, top_k=1),
]


def _params(kw):
    return S.Params(**kw)


def _settings(pkg, kw, seed):
    return pkg.sampling(seed=seed, **kw)


def _expect(z, hist, p, u, got, where):
    """The oracle's draw on logits z; a different token is accepted only when
    u sits within BOUNDARY of the two tokens' shared interval end."""
    want = S.sample(z, hist, p, u)
    if want == got:
        return 0
    iv = S.intervals(z, hist, p)
    assert got in iv, f"{where}: token {got} is not a candidate (oracle drew {want})"
    lo, hi = iv[got]
    assert min(abs(u - lo), abs(u - hi)) <= BOUNDARY, f"{where}: drew {got}, oracle {want}, u {u}"
    return 1


def _logits(rng, B, V, ties=0):
    z = (rng.standard_normal((B, V)) * 2.5).astype(np.float32)
    if ties:
        # the same top value on `ties` tokens of each row: the top-k boundary
        # falls inside the tie, which the lowest token ids must win
        for b in range(B):
            idx = rng.choice(V, ties, replace=False)
            z[b, idx] = z[b].max() + 1.0
    return z


def _histories(rng, B, V, n):
    return [rng.integers(0, V, size=n).tolist() + rng.integers(0, min(50, V), size=n // 4).tolist() for _ in range(B)]


def _counts(hists, V):
    c = np.zeros((len(hists), V), np.int32)
    for b, h in enumerate(hists):
        np.add.at(c[b], h, 1)
    return c


@pytest.mark.parametrize("kw", SETTINGS, ids=lambda kw: f"T{kw['temperature']}-k{kw['top_k']}")
@pytest.mark.parametrize("V,ties", [(151936, 0), (151936, 64), (4096, 0), (1000, 3), (1001, 2), (37, 0)])
def test_op_sample_matches_oracle_chain(pkg, kw, V, ties):
    import torch

    # V = 1001: rows not 16-byte aligned, the one-token-per-lane path; V = 37: fewer tokens than top_k
    rng = np.random.default_rng(V + ties + int(kw["temperature"] * 10) + kw["top_k"])
    B, seed = 3, 0xC0FFEE + V
    z = _logits(rng, B, V, ties)
    hists = _histories(rng, B, V, 64)
    cnt = _counts(hists, V)
    dev = torch.device("cuda")
    dz = torch.from_numpy(z).to(dev)
    dc = torch.from_numpy(cnt).to(dev)
    tok = torch.full((B,), -1, dtype=torch.int32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = torch.empty(pkg.op_sample_workspace(B, V), dtype=torch.uint8, device=dev)
    p = _params(kw)
    near = 0
    for step in range(3):
        before = dc.cpu().numpy()
        pkg.op_sample(dz, dc, _settings(pkg, kw, seed), step, tok, ws, st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        got = tok.cpu().numpy()
        after = dc.cpu().numpy()
        for b in range(B):
            u = S.uniform(seed, b, step)
            near += _expect(z[b], hists[b], p, u, int(got[b]), f"V={V} b={b} step={step}")
            # the drawn token is counted, nothing else changes
            diff = after[b] - before[b]
            assert diff[got[b]] == 1 and np.count_nonzero(diff) == 1
            hists[b].append(int(got[b]))
    assert near == 0


def test_op_sample_ties_go_to_the_lowest_tokens(pkg):
    import torch

    V, B = 151936, 2
    z = np.zeros((B, V), np.float32)
    z[0, [9, 70000, 5, 151935, 33]] = 3.0      # five equal maxima: top_k = 3 keeps 5, 9, 33; 4 adds 70000
    z[1, :] = 1.0                               # everything tied: top_k = k keeps 0 .. k-1
    dev = torch.device("cuda")
    dz = torch.from_numpy(z).to(dev)
    ws = torch.empty(pkg.op_sample_workspace(B, V), dtype=torch.uint8, device=dev)
    seen = {(b, k): set() for b in range(B) for k in (3, 4)}
    for seed in range(60):
        k = 3 if seed % 2 else 4
        dc = torch.zeros((B, V), dtype=torch.int32, device=dev)
        tok = torch.full((B,), -1, dtype=torch.int32, device=dev)
        pkg.op_sample(dz, dc, pkg.sampling(temperature=1.0, top_k=k, seed=seed), 0, tok, ws)
        torch.cuda.synchronize()
        got = tok.cpu().numpy()
        for b in range(B):
            assert int(got[b]) == S.sample(z[b], [], S.Params(temperature=1.0, top_k=k), S.uniform(seed, b, 0))
            seen[(b, k)].add(int(got[b]))
    assert seen[(0, 3)] == {5, 9, 33} and seen[(0, 4)] == {5, 9, 33, 70000}
    assert seen[(1, 3)] == {0, 1, 2} and seen[(1, 4)] == {0, 1, 2, 3}


def test_op_sample_is_reproducible(pkg):
    import torch

    V, B = 151936, 4
    rng = np.random.default_rng(3)
    z = _logits(rng, B, V)
    dev = torch.device("cuda")
    dz = torch.from_numpy(z).to(dev)
    ws = torch.empty(pkg.op_sample_workspace(B, V), dtype=torch.uint8, device=dev)
    outs = []
    for _ in range(3):
        dc = torch.zeros((B, V), dtype=torch.int32, device=dev)
        tok = torch.zeros(B, dtype=torch.int32, device=dev)
        seq = []
        for step in range(8):
            pkg.op_sample(dz, dc, pkg.sampling(temperature=1.1, top_k=200, top_p=0.9, repeat_penalty=1.2, seed=77),
                          step, tok, ws)
            seq.append(tok.cpu().numpy().copy())
        outs.append(np.stack(seq))
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])


def test_op_sample_rejects_bad_settings(pkg):
    import torch

    dev = torch.device("cuda")
    z = torch.zeros((1, 100), device=dev)
    c = torch.zeros((1, 100), dtype=torch.int32, device=dev)
    t = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = torch.empty(pkg.op_sample_workspace(1, 100), dtype=torch.uint8, device=dev)
    bad = [dict(temperature=0.0, top_k=5), dict(temperature=1.0, top_k=0), dict(temperature=1.0, top_k=4097),
           dict(temperature=1.0, top_k=5, top_p=0.0), dict(temperature=1.0, top_k=5, min_p=1.5),
           dict(temperature=1.0, top_k=5, repeat_penalty=0.0), dict(temperature=float("nan"), top_k=5),
           dict(temperature=-1.0, top_k=5)]
    for kw in bad:
        with pytest.raises(pkg.Q3Error):
            pkg.op_sample(z, c, pkg.sampling(**kw), 0, t, ws)
    with pytest.raises(pkg.Q3Error, match="workspace"):
        pkg.op_sample(z, c, pkg.sampling(temperature=1.0, top_k=5), 0, t, ws[:16])


# ---------------------------------------------------------------- the sampled decode

_models = {}


def _model(name):
    if name not in _models:
        w = synth.WORKLOADS[name]
        _models[name] = synth.make_model(w.shape, w.weight_seed)
    return _models[name]


def _decode_logits(dec, prompts, ids):
    """The decode's logits before each generated token, teacher-forced on the GPU."""
    z = [dec.prefill(prompts)]
    for i in range(ids.shape[1] - 1):
        z.append(dec.step_logits(ids[:, i]))
    return np.stack(z, 1)


def _check_decode(pkg, name, B, n_new, kw, seed):
    m = _model(name)
    w = synth.WORKLOADS[name]
    prompts = synth.prompts(w, B)
    dec = pkg.Decoder(m, max_batch=B, max_ctx=w.max_ctx)
    ids, counts, _ = dec.decode_sample(prompts, n_new, _settings(pkg, kw, seed))
    assert np.all(counts == n_new)
    z = _decode_logits(dec, prompts, ids)
    p = _params(kw)
    near = 0
    for b in range(B):
        hist = [int(t) for t in prompts[b]]
        for i in range(n_new):
            near += _expect(z[b, i], hist, p, S.uniform(seed, b, i), int(ids[b, i]), f"{name} seq {b} step {i}")
            hist.append(int(ids[b, i]))
    dec.close()
    assert near == 0
    return ids


@pytest.mark.parametrize("kw", SETTINGS[:4], ids=lambda kw: f"T{kw['temperature']}-k{kw['top_k']}")
def test_sampled_decode_tiny_batched(pkg, kw):
    _check_decode(pkg, "tiny-b1-p8-n16", 4, 24, kw, seed=1234)


def test_sampled_decode_0p6b_shape(pkg):
    # the full vocabulary inside the decode graph (fused small-batch step)
    _check_decode(pkg, "0.6b-b1-p32-n128", 2, 12, SETTINGS[0], seed=99)


def test_sampled_decode_0p6b_b8_chained_step(pkg):
    # B = 8 decodes with the chained step kernels
    _check_decode(pkg, "0.6b-b8-p16to256-n128", 8, 6, SETTINGS[3], seed=5)


def test_sampled_decode_seed_and_greedy_properties(pkg):
    name = "tiny-b1-p8-n16"
    m = _model(name)
    w = synth.WORKLOADS[name]
    prompts = [synth.ids(synth.key(41, b), 6 + b, w.shape.vocab) for b in range(3)]
    dec = pkg.Decoder(m, max_batch=3, max_ctx=w.max_ctx)
    kw = dict(temperature=0.9, top_k=50, top_p=0.95)
    a = dec.decode_sample(prompts, 20, pkg.sampling(seed=11, **kw))[0]
    b = dec.decode_sample(prompts, 20, pkg.sampling(seed=11, **kw))[0]
    c = dec.decode_sample(prompts, 20, pkg.sampling(seed=12, **kw))[0]
    assert np.array_equal(a, b)            # same seed, same tokens
    assert not np.array_equal(a, c)        # another seed draws other tokens here
    g = dec.decode(prompts, 20)[0]
    for T in (0.3, 1.0, 3.0):              # top_k = 1 is greedy at any temperature
        assert np.array_equal(dec.decode_sample(prompts, 20, pkg.sampling(temperature=T, top_k=1, seed=3))[0], g)
    # temperature 0 is the greedy call itself
    assert np.array_equal(dec.decode_sample(prompts, 20, pkg.sampling(temperature=0.0, top_k=0))[0], g)
    # the greedy path still works after sampled calls (separate graphs)
    assert np.array_equal(dec.decode(prompts, 20)[0], g)
    dec.close()


def test_sampled_decode_rejects_bad_settings(pkg):
    name = "tiny-b1-p8-n16"
    dec = pkg.Decoder(_model(name), max_batch=1, max_ctx=64)
    prompt = [np.arange(5, dtype=np.int32)]
    for kw in (dict(temperature=1.0, top_k=0), dict(temperature=1.0, top_k=10, top_p=1.5),
               dict(temperature=float("inf"), top_k=10)):
        with pytest.raises(pkg.Q3Error):
            dec.decode_sample(prompt, 4, pkg.sampling(**kw))
    # the context still decodes
    assert dec.decode_sample(prompt, 4, pkg.sampling(temperature=1.0, top_k=10))[0].shape == (1, 4)
    dec.close()


def test_sampled_decode_eos_stops(pkg):
    # eos_id is the first sampled token of sequence 0: its count is 1
    name = "tiny-b1-p8-n16"
    dec = pkg.Decoder(_model(name), max_batch=2, max_ctx=128)
    prompts = [synth.ids(synth.key(51, b), 7, 4096) for b in range(2)]
    st = pkg.sampling(temperature=0.7, top_k=20, seed=8)
    ids, _, _ = dec.decode_sample(prompts, 40, st)
    eos = int(ids[0, 0])
    ids2, counts, _ = dec.decode_sample(prompts, 40, st, eos_id=eos)
    assert counts[0] == 1
    n1 = int(counts[1])
    assert np.array_equal(ids2[1, :n1], ids[1, :n1])
    assert n1 == 40 or ids2[1, n1 - 1] == eos
    dec.close()
