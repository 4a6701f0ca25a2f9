"""Benchmark of int8 weight-only Qwen3-family greedy decode on GB300.

One bench step = one whole decode job of the workload: prefill of every
prompt plus the greedy decode of all new tokens for all B sequences, through
the library's C ABI.  ``value`` is whole-job throughput (generated tokens per
second over all ranks) with prompts and weights resident on the device when
the timed region starts; ``e2e`` is the same metric through ``q3i8_decode``
with host buffers (prompt upload and id download inside the timed region).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

Under torchrun (N > 1) every rank runs its own replica of the workload on its
GPU (the decode step does not shard; no collective on the data path); the
time is the maximum over ranks.  ``--impl reference`` times the CPU oracle on
the host cores on a bounded sample of the same workload (rank 0 only).
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

# DRAM bytes (read + write) of one decode step (the graph's kernels summed),
# from an ncu launch list of the bench workload (the decode-step summary
# under profiles/).  A figure holds only for the sources it was taken on,
# identified by kernel_source_id(); for any other build the roofline
# reports null.
NCU_TRAFFIC = {("2fda45da04582310", "0.6b-b1-p32-n128", 1): 609_032_704}


def kernel_source_id() -> str:
    """Hash of every CUDA source and header of the library."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "decode_int8_weight_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if f.endswith((".cu", ".cuh", ".h")):
            with open(os.path.join(csrc, f), "rb") as fh:
                h.update(f.encode() + b"\0" + fh.read())
    return h.hexdigest()[:16]


METRIC = "decode tok/s at B=1/8/32 (Qwen3-0.6B shape) and achieved HBM GB/s per step"
DEFAULT_WORKLOAD = "0.6b-b1-p32-n128"
L2_BYTES = 126 * 2 ** 20


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def bf16_sustained_tflops() -> float:
    """Measured sustained dense bf16 throughput (the prefill's tensor roofline); the profiling fallback else."""
    try:
        return float(json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))["bf16_tflops_sustained"])
    except Exception:
        return 1700.0


BF16_SUSTAINED_TFLOPS = bf16_sustained_tflops()


# ---------------------------------------------------------------- clocks sampling

class ClockSampler:
    """nvidia-smi SM clocks and throttle reasons sampled during the timed region."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits", "-lms", "100"]
        if self.gpu_id:
            cmd += ["--id=" + self.gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(power) if power else None}


def gpu_uuid():
    try:
        import torch

        u = str(torch.cuda.get_device_properties(torch.cuda.current_device()).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return None


# ---------------------------------------------------------------- distributed

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def init_dist(ws, local, backend):
    import torch.distributed as dist

    if ws > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)
    return dist


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(x: float, ws: int, device=None) -> float:
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------- reference arm (CPU oracle)

def oracle_sample(w, model, n_decode: int, nthreads: int):
    """Time the CPU oracle on prefill of every prompt + n_decode greedy steps
    per sequence (a bounded sample of the workload).  Returns (tokens, seconds)."""
    import oracle

    orc = oracle.Oracle(model, nthreads=nthreads)
    prompts = synth.prompts(w)
    t0 = time.perf_counter()
    toks = 0
    for p in prompts:
        s = orc.seq(len(p) + n_decode + 1)
        z = s.forward(p)
        tok = int(np.argmax(z[-1]))
        toks += 1
        for _ in range(n_decode):
            z = s.forward(np.array([tok], np.int32), 0)
            tok = int(np.argmax(z[-1]))
            toks += 1
    return toks, time.perf_counter() - t0


def sample_steps(w) -> int:
    # keep one oracle sample in the ~10 s range on 16 host cores
    base = {"qwen3-tiny": 15, "qwen3-0.6b": 16, "qwen3-1.7b": 6}[w.shape.name]
    return max(2, base // max(1, w.batch // 4)) if w.batch > 1 else base


def run_reference(args, w):
    ws, rank, local = dist_env()
    if rank != 0:
        return 0
    model = synth.make_model(w.shape, w.weight_seed)
    import oracle

    nthreads = oracle.default_threads()
    n_dec = sample_steps(w)
    times, toks = [], 0
    for i in range(args.warmup + args.steps):
        t, s = oracle_sample(w, model, n_dec, nthreads)
        if i >= args.warmup:
            times.append(s)
            toks = t
    tot = sum(times)
    value = toks * len(times) / tot
    sample = (f"prefill of all {w.batch} prompt(s) + {n_dec} greedy decode steps per sequence "
              f"({toks} tokens), per step")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tok/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot / len(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded random int8 weights and prompt ids)",
        "config": {"workload": w.name, "batch": w.batch, "new_tokens": w.new_tokens, "sample": sample},
        "cpu_baseline": {"value": value, "unit": "tok/s", "cores": nthreads, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- GPU arm

def batched_sweep(q3, dev, hbm_peak, batches=(8, 16, 32)):
    """Decode jobs of the batched workloads (one untimed job, then one timed): decode tok/s, step time and the
    step's HBM roofline fraction, with the KV bytes of each sequence's positions."""
    import torch

    out = {}
    for B in batches:
        wb = synth.WORKLOADS[f"0.6b-b{B}-p16to256-n128"]
        mb = synth.make_model(wb.shape, wb.weight_seed)
        pb = synth.prompts(wb)
        lens = np.array([len(p) for p in pb], np.int32)
        dec = q3.Decoder(mb, max_batch=B, max_ctx=wb.max_ctx)
        d_ids = torch.from_numpy(np.concatenate(pb).astype(np.int32)).to(dev)
        d_out = torch.empty((B, wb.new_tokens), dtype=torch.int32, device=dev)
        dec.decode_device(d_ids, lens, wb.new_tokens, d_out)
        st = dec.decode_device(d_ids, lens, wb.new_tokens, d_out)
        sb = float(np.mean([dec.step_bytes(lens + i) for i in range(wb.new_tokens - 1)]))
        gbs = sb / (st["step_us"] * 1e-6) / 1e9
        out[f"b{B}"] = {"decode_tok_s": st["decode_tokens_per_sec"], "step_us": st["step_us"],
                        "step_bytes_mean": sb, "achieved_gbs": gbs, "frac": gbs / hbm_peak,
                        "prefill_tok_s": st["prefill_tokens_per_sec"]}
        dec.close()
    return out


def long_jobs(q3, dev, hbm_peak, names=("1.7b-b1-p256-n1024", "0.6b-b1-p4096-n2048")):
    """One whole job of each B = 1 long workload (after a prefill-only warm-up): prefill tok/s, decode tok/s,
    mean step time and the decode step's HBM roofline fraction, with the weight / KV split of its bytes."""
    import torch

    out = {}
    for name in names:
        wl = synth.WORKLOADS[name]
        ml = synth.make_model(wl.shape, wl.weight_seed)
        pl = synth.prompts(wl)
        lens = np.array([len(p) for p in pl], np.int32)
        dec = q3.Decoder(ml, max_batch=len(pl), max_ctx=wl.max_ctx)
        d_ids = torch.from_numpy(np.concatenate(pl).astype(np.int32)).to(dev)
        d_out = torch.empty((len(pl), wl.new_tokens), dtype=torch.int32, device=dev)
        dec.decode_device(d_ids, lens, 2, d_out)
        st = dec.decode_device(d_ids, lens, wl.new_tokens, d_out)
        wbytes = wl.shape.weight_bytes()
        sb = float(np.mean([dec.step_bytes(lens + i) for i in range(0, wl.new_tokens - 1, 16)]))
        gbs = sb / (st["step_us"] * 1e-6) / 1e9
        # prefill work: the projections (2 flops per weight per token, lm_head excluded) and causal attention
        sh, M = wl.shape, int(lens.sum())
        proj = 2.0 * sh.n_layers * ((sh.dq + 2 * sh.dkv) * sh.hidden + sh.hidden * sh.dq + 3 * sh.intermediate * sh.hidden)
        attn = 4.0 * sh.n_heads * sh.head_dim * float((lens.astype(np.float64) ** 2).sum()) / 2 * sh.n_layers
        pf_tflops = (proj * M + attn) / (st["prefill_ms"] * 1e-3) / 1e12 if st["prefill_ms"] > 0 else 0.0
        out[name] = {"prefill_tok_s": st["prefill_tokens_per_sec"], "prefill_tflops": pf_tflops,
                     "prefill_frac_bf16_sustained": pf_tflops / BF16_SUSTAINED_TFLOPS,
                     "decode_tok_s": st["decode_tokens_per_sec"],
                     "step_us": st["step_us"], "step_bytes_mean": sb, "weight_bytes": wbytes,
                     "kv_bytes_mean": sb - wbytes, "achieved_gbs": gbs, "frac": gbs / hbm_peak}
        dec.close()
    return out


def run_gpu(args, w):
    import torch

    ws, rank, local = dist_env()
    if ws > 1:
        torch.cuda.set_device(local)
    init_dist(ws, local, "nccl")
    dev = torch.device("cuda", torch.cuda.current_device())

    import decode_int8_weight_gb300 as q3

    model = synth.make_model(w.shape, w.weight_seed)
    prompts = synth.prompts(w)
    B = len(prompts)
    lens = np.array([len(p) for p in prompts], np.int32)
    flat = np.concatenate(prompts).astype(np.int32)
    dec = q3.Decoder(model, max_batch=B, max_ctx=w.max_ctx)
    d_ids = torch.from_numpy(flat).to(dev)
    d_out = torch.empty((B, w.new_tokens), dtype=torch.int32, device=dev)
    n_tok = B * w.new_tokens

    # warm-up (also captures the step graph)
    for _ in range(args.warmup):
        dec.decode_device(d_ids, lens, w.new_tokens, d_out)
    torch.cuda.synchronize()

    # timed region: K whole jobs, device-resident
    sampler = ClockSampler(gpu_uuid()) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    barrier(ws)
    torch.cuda.synchronize()
    launches0 = dec.launch_count()
    stats = []
    t0 = time.perf_counter()
    for _ in range(args.steps):
        stats.append(dec.decode_device(d_ids, lens, w.new_tokens, d_out))
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    barrier(ws)
    launches = dec.launch_count() - launches0
    clocks = sampler.stop() if sampler else None
    dev_s = sum((s["prefill_ms"] + s["decode_ms"]) * 1e-3 for s in stats)
    dev_s_max = max_over_ranks(dev_s, ws, dev)
    value = ws * n_tok * args.steps / dev_s_max

    # per-step roofline of the decode step (CUDA events on the library's stream)
    step_us = statistics.median(s["step_us"] for s in stats)
    nsteps = w.new_tokens - 1
    pos_bytes = [dec.step_bytes(lens + i) for i in range(nsteps)]  # positions of step i+1
    step_bytes = float(np.mean(pos_bytes)) if pos_bytes else 0.0
    weight_bytes = w.shape.weight_bytes()
    hbm_peak, peak_kind = peaks()
    achieved = step_bytes / (step_us * 1e-6) / 1e9 if step_us > 0 else 0.0

    # the batched decode workloads (B = 8 / 16 / 32), outside the timed region
    batched = batched_sweep(q3, dev, hbm_peak) if (rank == 0 and not args.no_batched and w.batch == 1) else None
    longer = long_jobs(q3, dev, hbm_peak) if (rank == 0 and not args.no_batched and w.batch == 1) else None

    # e2e through the public API with host buffers
    out_e2e = None
    e2e_times = []
    for i in range(max(1, min(args.steps, 3)) + 1):
        torch.cuda.synchronize()
        t1 = time.perf_counter()
        out_e2e, _, _ = dec.decode(prompts, w.new_tokens)
        e2e_times.append(time.perf_counter() - t1)
    e2e_s = max_over_ranks(statistics.median(e2e_times[1:]), ws, dev)
    e2e_val = ws * n_tok / e2e_s
    same = bool(np.array_equal(out_e2e, d_out.cpu().numpy()))

    line = None
    if rank == 0:
        cpu = None
        if not args.no_cpu_baseline:
            import oracle

            nthreads = oracle.default_threads()
            n_dec = sample_steps(w)
            toks, secs = oracle_sample(w, model, n_dec, nthreads)
            cpu = {"value": toks / secs, "unit": "tok/s", "cores": nthreads, "kind": "oracle",
                   "sample": f"prefill of all {B} prompt(s) + {n_dec} greedy decode steps per sequence "
                             f"({toks} tokens, {secs:.1f} s)"}
        pf_tok_s = statistics.median(s["prefill_tokens_per_sec"] for s in stats)
        line = {
            "metric": METRIC, "value": value, "unit": "tok/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * dev_s_max / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "i8w_f32acc",
            "data": "synthetic (seeded random int8 weights and prompt ids)",
            "config": {"workload": w.name, "shape": w.shape.name, "batch": B, "prompt_lens": sorted(set(lens.tolist()))
                       if len(set(lens.tolist())) <= 4 else [int(lens.min()), int(lens.max())],
                       "new_tokens": w.new_tokens, "kv": "bf16", "parallelism": f"replicas x{ws}",
                       "l2": f"weights {weight_bytes / 1e6:.0f} MB per step > L2 {L2_BYTES / 2**20:.0f} MiB; no flush"},
            "decode_tok_s": statistics.median(s["decode_tokens_per_sec"] for s in stats),
            "step_us": step_us, "prefill_tok_s": pf_tok_s,
            "step_bytes": {"weights": weight_bytes, "kv_mean": step_bytes - weight_bytes, "total_mean": step_bytes},
            "roofline": {"kernel": "decode step (CUDA graph replay)", "bound": "hbm", "achieved": achieved,
                         "peak": hbm_peak, "unit": "GB/s", "frac": achieved / hbm_peak,
                         "traffic": NCU_TRAFFIC.get((kernel_source_id(), w.name, B)), "traffic_unit": "bytes/launch",
                         "peak_kind": peak_kind},
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_val, "unit": "tok/s", "h2d_bytes_per_step": int(flat.nbytes + 8 * flat.size + 12 * B),
                    "d2h_bytes_per_step": int(n_tok * 4), "ids_match_device_run": same},
            "batched_decode": batched,
            "long_jobs": longer,
            "gpu_launches": int(launches),
            "wall_s": wall,
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    dec.close()
    if ws > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(synth.WORKLOADS))
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-batched", action="store_true",
                    help="skip the extra jobs (B = 8 / 16 / 32 decode, the 1.7B and long-context jobs)")
    ap.add_argument("--new-tokens", type=int, default=None,
                    help="override the workload's generated tokens per sequence (e.g. to profile its prefill)")
    args = ap.parse_args()
    w = synth.WORKLOADS[args.workload]
    if args.new_tokens is not None:
        w = dataclasses.replace(w, new_tokens=max(1, args.new_tokens))
    if args.impl == "reference":
        return run_reference(args, w)
    return run_gpu(args, w)


if __name__ == "__main__":
    sys.exit(main())
