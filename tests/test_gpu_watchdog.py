"""Device time-outs: the bounded mbarrier wait that the attention and prefill
kernels use gives up, reports Q3_ERR_TIMEOUT and returns, and the context
stays usable.  The wait runs on a barrier phase that nothing completes (no
fault, no endless loop): q3i8_op_wait_probe."""
import numpy as np
import pytest

import oracle
import synth
from gpu_common import check_greedy_against_oracle

pytestmark = pytest.mark.gpu

Q3_ERR_TIMEOUT = 7
WALL_LIMIT_NS = 1_000_000_000  # the kernels' own wall-time limit of a wait (q3::kWaitWallNs)


@pytest.fixture(scope="module")
def pkg():
    import torch

    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from decode_int8_weight_gb300 import build

    build.build()
    import decode_int8_weight_gb300 as p

    p.lib()
    return p


@pytest.fixture()
def bufs():
    import torch

    return (torch.full((1,), -1, dtype=torch.int32, device="cuda"),
            torch.zeros((1,), dtype=torch.int64, device="cuda"))


def _probe(pkg, arrive, limit, status, elapsed):
    """Returns (rc, device status, elapsed ns of the wait)."""
    try:
        pkg.op_wait_probe(arrive, limit, status, elapsed)
        rc = 0
    except pkg.Q3Error as e:
        rc = e.code
    return rc, int(status.item()), int(elapsed.item())


def test_completed_phase_is_seen(pkg, bufs):
    rc, st, _ = _probe(pkg, True, -1, *bufs)
    assert (rc, st) == (0, 0)


def test_limit_zero_times_out_at_once(pkg, bufs):
    rc, st, ns = _probe(pkg, False, 0, *bufs)
    assert (rc, st) == (Q3_ERR_TIMEOUT, Q3_ERR_TIMEOUT)
    assert 0 <= ns < 50_000_000
    # limit 0 gives up without polling even when the phase has completed
    rc, st, _ = _probe(pkg, True, 0, *bufs)
    assert (rc, st) == (Q3_ERR_TIMEOUT, Q3_ERR_TIMEOUT)


def test_small_limit_times_out_and_context_survives(pkg, bufs):
    rc, st, ns = _probe(pkg, False, 4096, *bufs)
    assert (rc, st) == (Q3_ERR_TIMEOUT, Q3_ERR_TIMEOUT)
    assert 0 < ns < 1_000_000_000
    # the same call with the phase completed succeeds afterwards
    rc, st, _ = _probe(pkg, True, 4096, *bufs)
    assert (rc, st) == (0, 0)
    # and a whole decode on the same context still matches the oracle
    w = synth.WORKLOADS["tiny-b1-p8-n16"]
    m = synth.make_model(w.shape, w.weight_seed)
    prompts = synth.prompts(w)
    dec = pkg.Decoder(m, max_batch=1, max_ctx=w.max_ctx)
    ids, counts, _ = dec.decode(prompts, w.new_tokens)
    dec.close()
    assert np.all(counts == w.new_tokens)
    zo = oracle.Oracle(m).teacher_forced(np.concatenate([prompts[0], ids[0, :-1]]), len(prompts[0]) - 1)
    check_greedy_against_oracle(ids[0], zo, "after time-outs")


def test_kernels_own_limits_run_out(pkg, bufs):
    # the kernels' own limits: 2^22 polls or one second of wall time,
    # whichever comes first; either way the wait ends within about a second
    rc, _, ns4k = _probe(pkg, False, 4096, *bufs)
    assert rc == Q3_ERR_TIMEOUT
    rc, st, ns = _probe(pkg, False, -1, *bufs)
    assert (rc, st) == (Q3_ERR_TIMEOUT, Q3_ERR_TIMEOUT)
    assert ns < WALL_LIMIT_NS + 500_000_000
    print(f"\n4096 polls: {ns4k / 1e6:.2f} ms; own limits ran out after {ns / 1e6:.1f} ms")
