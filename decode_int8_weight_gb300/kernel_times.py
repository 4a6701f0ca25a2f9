"""Per-kernel device times of the decode step inside its CUDA graph.

ncu serialises kernels and replays them with cold caches, so its per-launch
times leave out what programmatic dependent launch overlaps.  This tool
records the kernels of real graph replays instead (CUPTI kernel records
through torch.profiler) and reports, per kernel name and per decode step:

- ``n/step``: launches per step;
- ``dur``: mean time from a launch's first CTA starting to its last CTA
  ending (a launch may start early and wait for its predecessor);
- ``excl/step``: the time per step during which that kernel was the one
  whose end moved the step forward (the step's span split between the
  kernels; the column sums to the step time).

    python -m decode_int8_weight_gb300.kernel_times [--workload NAME] [--new-tokens N]

Workloads are the seeded synthetic ones of ``synth`` (random int8 weights of
the named shape); a step is one graph replay of the greedy decode.
"""
from __future__ import annotations

import argparse
import collections
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def _is_step_end(name: str) -> bool:
    # the last kernel of a decode step: the lm_head sweep (or the sampling kernel after it)
    return ("lm_head" in name) or ("gemv_kernel<" in name and ", 3>" in name) or ("sample_kernel" in name)


def step_table(events, n_skip: int = 1):
    """events: [(name, start_us, end_us)] of one decode call.  Returns
    (steps, span_us_per_step, {kernel: (launches/step, mean dur us, excl us/step)})."""
    ev = sorted(events, key=lambda e: e[1])
    ends = [i for i, e in enumerate(ev) if _is_step_end(e[0])]
    if len(ends) < n_skip + 2:
        raise RuntimeError("too few decode steps recorded")
    seg = ev[ends[n_skip] + 1: ends[-1] + 1]
    steps = len(ends) - n_skip - 1
    dur = collections.defaultdict(float)
    exc = collections.defaultdict(float)
    cnt = collections.Counter()
    prev_end = seg[0][1]
    for name, s, e in seg:
        k = name.split("(")[0].replace("void ", "").replace("q3::", "")
        dur[k] += e - s
        cnt[k] += 1
        if e > prev_end:
            exc[k] += e - max(prev_end, s)
            prev_end = e
    span = seg[-1][2] - seg[0][1]
    table = {k: (cnt[k] / steps, dur[k] / cnt[k], exc[k] / steps) for k in cnt}
    return steps, span / steps, table


def main(argv=None) -> int:
    import torch
    from torch.profiler import ProfilerActivity, profile

    import synth
    import decode_int8_weight_gb300 as q3

    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--workload", default="0.6b-b1-p32-n128", choices=sorted(synth.WORKLOADS))
    ap.add_argument("--new-tokens", type=int, default=16)
    args = ap.parse_args(argv)
    w = synth.WORKLOADS[args.workload]
    model = synth.make_model(w.shape, w.weight_seed)
    prompts = synth.prompts(w)
    dec = q3.Decoder(model, max_batch=len(prompts), max_ctx=w.max_ctx)
    for _ in range(2):  # graphs built, caches warm
        dec.decode(prompts, args.new_tokens)
    with profile(activities=[ProfilerActivity.CUDA]):  # the first profiled region starts CUPTI up
        torch.ones(4, device="cuda").sum()
    torch.cuda.synchronize()
    with profile(activities=[ProfilerActivity.CUDA]) as prof:
        stats = dec.decode(prompts, args.new_tokens)[2]
    torch.cuda.synchronize()
    events = [(e.name, e.time_range.start, e.time_range.end) for e in prof.events()
              if e.device_type == torch.autograd.DeviceType.CUDA]
    dec.close()
    steps, span, table = step_table(events)
    print(f"{args.workload}: step_us (CUDA events) {stats['step_us']:.1f}, "
          f"{steps} profiled steps, span per step {span:.1f} us")
    print(f"{'kernel':52s} {'n/step':>7s} {'dur us':>8s} {'excl us/step':>13s}")
    for k, (n, d, x) in sorted(table.items(), key=lambda kv: -kv[1][2]):
        print(f"{k[:52]:52s} {n:7.1f} {d:8.2f} {x:13.1f}")
    return 0


if __name__ == "__main__":
    sys.exit(main())
