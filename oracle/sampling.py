"""CPU oracle of the sampling chain -- TEST INFRASTRUCTURE (see the package
docstring for who may import it).

"Model-agnostic LLM inference", section "Sampling": with temperature > 0
every token is drawn from the model's distribution through the chain
repetition / presence / frequency penalties -> temperature -> top-k -> min-p
-> top-p -> seeded weighted draw; the same seed reproduces the same tokens,
and top_k = 1 reproduces the greedy sequence at any temperature.

The page names the chain but no formulas; each step below is the plainest
conventional reading, written out in float64 on plain numpy arrays:

* penalties, over the tokens already in the sequence (prompt and generated
  tokens before this step), t seen c_t >= 1 times:
  repetition r: z_t / r if z_t > 0 else z_t * r; then
  presence a_p and frequency a_f: z_t - a_p - a_f * c_t;
* temperature T > 0: z / T.  T = 0 is the default greedy call: the argmax
  of the raw logits (lowest index on ties), with no step of the chain;
* candidates in the order (z descending, token ascending); top-k keeps the
  first k of them (k = 0: all).  The order is taken on the penalised logits,
  before the division by T: for T > 0 it is the order of z / T, and taking
  it first keeps a float64 rounding of the quotient from merging two
  distinct values into a tie;
* min-p keeps candidates whose softmax probability over the current
  candidates is at least min_p times the largest;
* top-p keeps the shortest prefix whose softmax probabilities over the
  current candidates sum to at least top_p (at least one candidate);
* the draw: with the survivors' renormalised probabilities q_1.. in that
  order, the token is the first i with u < q_1 + .. + q_i (the last one if
  rounding leaves none), u in [0, 1).

u is the seeded draw of ``uniform``: output c + 1 of SplitMix64 (Steele, Lea
and Flood, "Fast splittable pseudorandom number generators", OOPSLA 2014)
started at the seed, with counter c = step * 2^20 + sequence, its top 24 bits
scaled by 2^-24 (exact in float32 and float64).
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

_M64 = (1 << 64) - 1


def splitmix64_output(seed: int, n: int) -> int:
    """Output number n (n >= 1) of SplitMix64 started at `seed`: the state
    advances by the golden-ratio increment and each output is the state's
    mix (the published algorithm's two xor-shift-multiply rounds and final
    xor-shift)."""
    z = (seed + n * 0x9E3779B97F4A7C15) & _M64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _M64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _M64
    return z ^ (z >> 31)


def uniform(seed: int, sequence: int, step: int) -> float:
    """The draw u in [0, 1) of `sequence` (< 2^20) at generated position `step`."""
    c = step * (1 << 20) + sequence
    return (splitmix64_output(seed & _M64, c + 1) >> 40) * 2.0 ** -24


@dataclass(frozen=True)
class Params:
    temperature: float = 0.0
    top_k: int = 0
    top_p: float = 1.0
    min_p: float = 0.0
    repeat_penalty: float = 1.0
    presence_penalty: float = 0.0
    frequency_penalty: float = 0.0


def apply_penalties(z: np.ndarray, history, p: Params) -> np.ndarray:
    """Penalised logits (float64 copy)."""
    z = np.asarray(z, np.float64).copy()
    ids, counts = np.unique(np.asarray(history, np.int64), return_counts=True)
    for t, c in zip(ids, counts):
        v = z[t]
        if p.repeat_penalty != 1.0:
            v = v / p.repeat_penalty if v > 0 else v * p.repeat_penalty
        z[t] = v - p.presence_penalty - p.frequency_penalty * c
    return z


def _softmax(v: np.ndarray) -> np.ndarray:
    e = np.exp(v - np.max(v))
    return e / np.sum(e)


def candidates(z: np.ndarray, history, p: Params):
    """(tokens, q): the tokens that survive penalties, temperature, top-k,
    min-p and top-p, in draw order, with their renormalised probabilities.
    Only for temperature > 0."""
    assert p.temperature > 0
    pen = apply_penalties(z, history, p)
    order = np.lexsort((np.arange(pen.size), -pen))  # z descending, token ascending
    v = pen / p.temperature
    if 0 < p.top_k < v.size:
        order = order[:p.top_k]
    if p.min_p > 0:
        q = _softmax(v[order])
        order = order[q >= p.min_p * q.max()]
    if p.top_p < 1.0:
        q = _softmax(v[order])
        cum = np.cumsum(q)
        n = int(np.searchsorted(cum, p.top_p, side="left")) + 1  # first prefix with sum >= top_p
        order = order[:min(n, order.size)]
    return order, _softmax(v[order])


def sample(z: np.ndarray, history, p: Params, u: float) -> int:
    """One token from logits z (the whole vocabulary), the sequence so far
    and the draw u."""
    if p.temperature == 0.0:
        return int(np.argmax(np.asarray(z, np.float64)))  # np.argmax: lowest index on ties
    tokens, q = candidates(z, history, p)
    cum = np.cumsum(q)
    i = int(np.searchsorted(cum, u, side="right"))  # first i with u < cum[i]
    return int(tokens[min(i, tokens.size - 1)])


def intervals(z: np.ndarray, history, p: Params):
    """{token: (lo, hi)}: the draws u in [lo, hi) that pick each surviving
    token (lo and hi are float64 partial sums of the draw order)."""
    tokens, q = candidates(z, history, p)
    cum = np.cumsum(q)
    lo = np.concatenate([[0.0], cum[:-1]])
    return {int(t): (float(a), float(b)) for t, a, b in zip(tokens, lo, cum)}


def decode(orc, prompt, max_new: int, p: Params, seed: int, sequence: int = 0, eos_id: int = -1) -> np.ndarray:
    """Sampled decode of one sequence with the oracle model `orc`: every
    token, the first included, drawn by ``sample`` from the logits of the
    sequence so far, with draw ``uniform(seed, sequence, i)`` for generated
    token i; stops after max_new tokens or at eos_id (kept)."""
    prompt = [int(t) for t in prompt]
    s = orc.seq(len(prompt) + max_new)
    z = s.forward(np.asarray(prompt, np.int32))[-1]
    history, out = list(prompt), []
    for i in range(max_new):
        t = sample(z, history, p, uniform(seed, sequence, i))
        out.append(t)
        history.append(t)
        if t == eos_id or i + 1 == max_new:
            break
        z = s.forward(np.asarray([t], np.int32))[-1]
    return np.asarray(out, np.int32)
