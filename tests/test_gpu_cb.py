"""Continuous batching on the GPU ("LLM inference overview", section
"Workload characteristics": one weight sweep per step serves every sequence
in flight): the scheduler's plan executed by q3i8_cb_prefill / q3i8_cb_step
and the native loop q3i8_sched_run, through the C ABI.

Each request's tokens must be its own greedy sequence: checked against the
oracle (teacher-forced on the GPU's tokens, identical wherever the oracle's
top-1/top-2 gap exceeds 1e-2).  Where a sequence's prompt is prefilled alone
and its steps run on the small-batch step kernels (at most 2 rows), its
tokens must also equal a plain single-sequence decode bit for bit: every
row of those kernels is computed independently of the others
(column-independent MMAs, per-row attention, integer accumulation of the
residual stream), whatever the other rows and slots are."""
import numpy as np
import pytest

import oracle
import synth
from gpu_common import check_greedy_against_oracle

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


@pytest.fixture(scope="module")
def tiny():
    w = synth.WORKLOADS["tiny-b1-p8-n16"]
    m = synth.make_model(w.shape, w.weight_seed)
    return m, oracle.Oracle(m)


def _requests(n, vocab, seed=0):
    rng = np.random.default_rng(seed)
    reqs = []
    for i in range(n):
        plen = int(rng.integers(1, 40))
        reqs.append((synth.ids(synth.key(500 + seed, i), plen, vocab), int(rng.integers(1, 30))))
    return reqs


def _serve(pkg, dec, reqs, max_batch, max_ctx, eos=-1):
    s = pkg.Scheduler(max_batch, max_ctx)
    ids = [s.submit(p, n, eos) for p, n in reqs]
    stats = dec.sched_run(s)
    out = [s.result(i) for i in ids]
    s.close()
    assert all(done for _, done in out)
    return [t for t, _ in out], stats


@pytest.mark.parametrize("max_batch", [1, 3, 4])
def test_sched_run_gives_each_request_its_greedy_sequence(pkg, tiny, max_batch):
    m, orc = tiny
    reqs = _requests(9, m.shape.vocab, seed=max_batch)
    dec = pkg.Decoder(m, max_batch=max_batch, max_ctx=128)
    got, stats = _serve(pkg, dec, reqs, max_batch, 96)
    assert stats["decode_steps"] > 0 and stats["prefill_tokens"] == sum(len(p) for p, _ in reqs)
    for (p, n), g in zip(reqs, got):
        assert len(g) == n
        zo = orc.teacher_forced(np.concatenate([p, g[:-1]]), len(p) - 1)
        check_greedy_against_oracle(g, zo, f"request of {len(p)} tokens")
    if max_batch == 1:  # every prompt prefilled alone, every step one row: the plain decode's bits
        single = pkg.Decoder(m, max_batch=1, max_ctx=128)
        for (p, n), g in zip(reqs, got):
            assert np.array_equal(g, single.decode([p], n)[0][0])
        single.close()
    dec.close()


def test_sched_run_with_the_chained_step(pkg, tiny):
    # up to 8 rows: batches above 4 decode with the chained step kernels
    m, orc = tiny
    reqs = _requests(14, m.shape.vocab, seed=21)
    dec = pkg.Decoder(m, max_batch=8, max_ctx=128)
    got, _ = _serve(pkg, dec, reqs, 8, 96)
    for (p, n), g in zip(reqs, got):
        assert len(g) == n
        zo = orc.teacher_forced(np.concatenate([p, g[:-1]]), len(p) - 1)
        check_greedy_against_oracle(g, zo, f"request of {len(p)} tokens")
    dec.close()


def test_eos_retires_requests_early(pkg, tiny):
    m, _ = tiny
    reqs = _requests(6, m.shape.vocab, seed=33)
    # one slot: every request runs alone, so the runs differ only where eos cuts them
    dec = pkg.Decoder(m, max_batch=1, max_ctx=128)
    full, _ = _serve(pkg, dec, reqs, 1, 96)
    eos = int(full[0][min(2, len(full[0]) - 1)])  # a token the first request produces
    cut, _ = _serve(pkg, dec, reqs, 1, 96, eos=eos)
    for f, c in zip(full, cut):
        hit = np.nonzero(f == eos)[0]
        n = hit[0] + 1 if hit.size else len(f)
        assert np.array_equal(c, f[:n])
    dec.close()


def test_cb_calls_keep_other_slots(pkg, tiny):
    m, _ = tiny
    dec = pkg.Decoder(m, max_batch=4, max_ctx=128)
    dec.cb_reserve(128)
    pa = synth.ids(synth.key(71, 0), 11, m.shape.vocab)
    pb = synth.ids(synth.key(71, 1), 5, m.shape.vocab)
    single = pkg.Decoder(m, max_batch=1, max_ctx=128)
    want_a = single.decode([pa], 12)[0][0]
    want_b = single.decode([pb], 6)[0][0]
    # sequence a in slot 2: prefill and three steps alone
    t = dec.cb_prefill([2], [pa])
    got_a = [int(t[0])]
    for i in range(3):
        got_a.append(int(dec.cb_step([2], [len(pa) + i], [got_a[-1]])[0]))
    # sequence b joins in slot 0; both decode together (rows in any order)
    tb = dec.cb_prefill([0], [pb])
    got_b = [int(tb[0])]
    for i in range(5):
        pos_a, pos_b = len(pa) + 3 + i, len(pb) + i
        nxt = dec.cb_step([0, 2], [pos_b, pos_a], [got_b[-1], got_a[-1]])
        got_b.append(int(nxt[0]))
        got_a.append(int(nxt[1]))
    for i in range(3):
        got_a.append(int(dec.cb_step([2], [len(pa) + 8 + i], [got_a[-1]])[0]))
    assert got_a == want_a.tolist()
    assert got_b == want_b.tolist()
    # the plain calls still decode as before (their rows point at slots 0..B-1 again)
    assert np.array_equal(dec.decode([pa], 12)[0][0], want_a)
    single.close()
    dec.close()


def test_cb_errors(pkg, tiny):
    m, _ = tiny
    dec = pkg.Decoder(m, max_batch=2, max_ctx=64)
    p = synth.ids(synth.key(72, 0), 4, m.shape.vocab)
    dec.cb_reserve(64)
    dec.cb_prefill([1], [p])
    with pytest.raises(pkg.Q3Error):
        dec.cb_prefill([0, 0], [p, p])      # repeated slot
    with pytest.raises(pkg.Q3Error):
        dec.cb_prefill([2], [p])            # slot out of range
    with pytest.raises(pkg.Q3Error):
        dec.cb_step([1], [0], [1])          # position 0 has no earlier token
    with pytest.raises(pkg.Q3Error):
        dec.cb_step([1], [1 << 20], [1])    # past the reserved positions
    with pytest.raises(pkg.Q3Error):
        dec.cb_step([1], [4], [m.shape.vocab])
    assert dec.cb_step([1], [4], [1]).shape == (1,)  # the context still works
    s = pkg.Scheduler(4, 64)
    with pytest.raises(pkg.Q3Error, match="slots"):
        dec.sched_run(s)                     # more slots than the context's max_batch
    s.close()
    dec.close()
