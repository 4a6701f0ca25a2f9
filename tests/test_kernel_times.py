"""The per-kernel step table of decode_int8_weight_gb300.kernel_times, on
hand-made kernel records (no GPU): launches per step, mean durations, and the
exclusive times that split each step's span between its kernels."""
import pytest

from decode_int8_weight_gb300.kernel_times import step_table


def _records():
    ev = []
    t = 0.0
    for step in range(4):
        # a: 0..5, b overlaps a (starts early at 3, ends at 9), lm_head 8..12
        ev.append(("void q3::a_kernel(Args)", t, t + 5))
        ev.append(("void q3::b_kernel<2>(Args)", t + 3, t + 9))
        ev.append(("q3::lm_head_kernel(LmHeadArgs)", t + 8, t + 12))
        t += 12
    return ev


def test_step_table_splits_the_span():
    steps, span, table = step_table(_records())
    assert steps == 2  # the first step is skipped, the rest run between lm_head launches
    assert span == pytest.approx(12.0)
    n, dur, exc = table["a_kernel"]
    assert n == 1 and dur == pytest.approx(5.0) and exc == pytest.approx(5.0)
    n, dur, exc = table["b_kernel<2>"]
    assert n == 1 and dur == pytest.approx(6.0) and exc == pytest.approx(4.0)  # 5..9
    n, dur, exc = table["lm_head_kernel"]
    assert exc == pytest.approx(3.0)  # 9..12
    assert sum(x for _, _, x in table.values()) == pytest.approx(span)


def test_too_few_steps():
    with pytest.raises(RuntimeError):
        step_table(_records()[:6])
