"""Continuous-batching scheduler (q3i8_sched_*), host side.  The decode
work is done here by the CPU oracle, one KV cache per slot, so the test
checks the scheduler's bookkeeping against ground truth: every request,
however its steps interleave with others', generates exactly the tokens of
its own greedy decode ("Run local LLM decode", section "Limitations": each
token is the argmax at its step), with the positions and input tokens the
scheduler hands out.  No GPU."""
import numpy as np
import pytest

import oracle
import synth


@pytest.fixture(scope="module")
def pkg():
    from decode_int8_weight_gb300 import build

    build.build()
    import decode_int8_weight_gb300 as p

    p.lib()
    return p


@pytest.fixture(scope="module")
def orc():
    return oracle.Oracle(synth.make_model(synth.TINY, 21), nthreads=1)


def _serve(pkg, orc, requests, max_batch, max_ctx):
    """Run the scheduler's loop with the oracle as the engine.  Returns the
    outputs per request and the largest number of rows in one step."""
    s = pkg.Scheduler(max_batch, max_ctx)
    ids = [s.submit(p, n, eos) for p, n, eos in requests]
    kv = {}  # slot -> the oracle sequence holding that slot's cache
    widest, steps = 0, 0
    while not s.idle():
        adm, rows = s.plan()
        firsts = []
        for rid, slot in adm:
            assert slot not in {r[1] for r in rows}  # a slot in use is never handed out
            kv[slot] = orc.seq(max_ctx)
            z = kv[slot].forward(np.asarray(requests[rid][0], np.int32))[-1]
            firsts.append(int(np.argmax(z)))
        toks = []
        for rid, slot, pos, tok in rows:
            seq = kv[slot]
            assert seq.length == pos  # the position is the slot's cache length
            z = seq.forward(np.asarray([tok], np.int32))[-1]
            toks.append(int(np.argmax(z)))
        s.complete_prefill([a[0] for a in adm], firsts)
        s.complete_step(toks)
        widest = max(widest, len(rows))
        steps += 1
        assert steps < 10_000
    outs = []
    for rid in ids:
        out, done = s.result(rid)
        assert done
        outs.append(out)
    s.close()
    return outs, widest


def _requests(n, seed, vocab, lens=(1, 12), new=(1, 20), eos=-1):
    rng = np.random.default_rng(seed)
    return [(rng.integers(0, vocab, size=int(rng.integers(lens[0], lens[1] + 1))).astype(np.int32),
             int(rng.integers(new[0], new[1] + 1)), eos) for _ in range(n)]


@pytest.mark.parametrize("max_batch", [1, 3, 8])
def test_each_request_gets_its_own_greedy_sequence(pkg, orc, max_batch):
    reqs = _requests(11, 5 + max_batch, synth.TINY.vocab)
    outs, widest = _serve(pkg, orc, reqs, max_batch, 64)
    assert widest <= max_batch
    if max_batch > 1:
        assert widest > 1  # sequences really share steps
    for (p, n, eos), out in zip(reqs, outs):
        assert out.tolist() == orc.greedy(p, n, eos).tolist()


def test_eos_retires_early_and_frees_the_slot(pkg, orc):
    # pick as eos a token that one request's greedy run emits early
    reqs = _requests(6, 77, synth.TINY.vocab, new=(12, 16))
    g = orc.greedy(reqs[0][0], reqs[0][1])
    eos = int(g[3])
    reqs = [(p, n, eos) for p, n, _ in reqs]
    outs, _ = _serve(pkg, orc, reqs, 2, 64)
    for (p, n, e), out in zip(reqs, outs):
        want = orc.greedy(p, n, e)
        assert out.tolist() == want.tolist()
    assert outs[0][-1] == eos and len(outs[0]) <= 4


def test_single_token_requests_finish_at_prefill(pkg, orc):
    reqs = _requests(5, 3, synth.TINY.vocab, new=(1, 1))
    outs, widest = _serve(pkg, orc, reqs, 2, 64)
    assert widest == 0  # never reach a decode step
    for (p, n, eos), out in zip(reqs, outs):
        assert out.tolist() == orc.greedy(p, 1, eos).tolist()


def test_fifo_admission_into_the_lowest_free_slots(pkg):
    s = pkg.Scheduler(2, 32)
    a = s.submit([1, 2, 3], 3)
    b = s.submit([4], 1)
    c = s.submit([5, 6], 2)
    adm, rows = s.plan()
    assert adm == [(a, 0), (b, 1)] and rows == []
    s.complete_prefill([b, a], [40, 10])  # any order; b is done after one token
    adm, rows = s.plan()
    assert adm == [(c, 1)]                                  # c takes the slot b freed
    assert rows == [(a, 0, 3, 10)]                          # a: prompt 3 + 1 generated - 1
    s.complete_prefill([c], [50])
    s.complete_step([11])
    adm, rows = s.plan()
    assert adm == [] and rows == [(a, 0, 4, 11), (c, 1, 2, 50)]
    s.complete_step([12, 51])                               # a: 3 tokens, c: 2 tokens -> both done
    assert s.idle()
    assert s.result(a)[0].tolist() == [10, 11, 12] and s.result(b)[0].tolist() == [40]
    assert s.result(c)[0].tolist() == [50, 51]


def test_errors(pkg):
    s = pkg.Scheduler(2, 16)
    with pytest.raises(pkg.Q3Error) as e:
        s.submit([], 4)
    assert e.value.status == "invalid_arguments"
    with pytest.raises(pkg.Q3Error) as e:
        s.submit([1], 0)
    assert e.value.status == "invalid_arguments"
    with pytest.raises(pkg.Q3Error) as e:
        s.submit(list(range(10)), 8)  # 10 + 8 - 1 = 17 positions > 16
    assert e.value.status == "context_past_ceiling"
    s.submit(list(range(10)), 7)      # 16 positions fit
    s.plan()
    with pytest.raises(pkg.Q3Error) as e:
        s.plan()                      # the admission's prefill was not reported
    assert e.value.status == "invalid_state"
    with pytest.raises(pkg.Q3Error) as e:
        s.complete_prefill([5], [1])  # not an admitted request
    assert e.value.status == "invalid_state"
    with pytest.raises(pkg.Q3Error):
        pkg.Scheduler(0, 16)
