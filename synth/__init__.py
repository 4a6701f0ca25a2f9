"""Seeded synthetic inputs: model shapes, random int8 weights, prompts.

Input preparation only, shared by the CUDA path's tests and benchmark and by
the CPU oracle's tests.  Nothing here computes any part of the decoder; the
one transformation applied to the random draws is the offline per-row int8
quantiser that produces what the library's ``init`` consumes (int8 weights +
one fp32 scale per output channel; "Model-agnostic LLM inference", section
"The quantized load cache").

Shapes follow the Qwen3 family as the pages list it ("Run local LLM decode",
section "Limitations": hidden 1024, 28 layers, 16 query heads, 8 key/value
heads, head_dim 128, vocab 151936, tied embeddings) plus the 1.7B sibling
served by the model-agnostic path, and a tiny member for fast checks.

Weights are N(0, 0.02) rounded to bf16 and quantised per row; RMSNorm gains
are 1.0 unless a caller asks for random gains (used by tests so that a
dropped gain cannot go unnoticed).  Seeds: weights ``1000 + k`` and prompts
``2000 + k`` for workload number ``k`` below.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "_build", "libsynth.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile gen.c into synth/_build/libsynth.so with gcc (host code only)."""
    src = os.path.join(_HERE, "gen.c")
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(src):
        os.makedirs(os.path.dirname(_SO), exist_ok=True)
        tmp = _SO + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
                               "-o", tmp, src, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            u64, i64, i32, dbl, vp = (ctypes.c_uint64, ctypes.c_int64, ctypes.c_int32,
                                      ctypes.c_double, ctypes.c_void_p)
            lib.synth_key.restype = u64
            lib.synth_key.argtypes = [u64, u64]
            lib.synth_draws.argtypes = [u64, u64, i64, vp]
            lib.synth_normal_bf16.argtypes = [u64, i64, dbl, vp]
            lib.synth_normal_f32.argtypes = [u64, i64, dbl, dbl, vp]
            lib.synth_quantize_rows_bf16.argtypes = [vp, i64, i64, vp, vp]
            lib.synth_quantize_rows_f32.argtypes = [vp, i64, i64, vp, vp]
            lib.synth_matrix_i8.argtypes = [u64, i64, i64, dbl, vp, vp]
            lib.synth_ids.argtypes = [u64, i64, i32, vp]
            lib.synth_lengths.argtypes = [u64, i64, i32, i32, vp]
            _lib = lib
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


# --------------------------------------------------------------------------- draws

def key(seed: int, index: int) -> int:
    return int(_load().synth_key(seed, index))


def draws(k: int, n: int, start: int = 0) -> np.ndarray:
    out = np.empty(n, np.uint64)
    _load().synth_draws(k, start, n, _p(out))
    return out


def normal_bf16(k: int, n: int, sigma: float = 0.02) -> np.ndarray:
    """bf16 bit patterns (uint16) of sigma * N(0, 1)."""
    out = np.empty(n, np.uint16)
    _load().synth_normal_bf16(k, n, sigma, _p(out))
    return out


def normal_f32(k: int, n: int, mean: float = 0.0, sigma: float = 1.0) -> np.ndarray:
    out = np.empty(n, np.float32)
    _load().synth_normal_f32(k, n, mean, sigma, _p(out))
    return out


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)


def quantize_rows(w: np.ndarray):
    """Per-row symmetric int8 quantisation of a bf16-bit (uint16) or fp32 matrix."""
    w = np.ascontiguousarray(w)
    rows, cols = w.shape
    q = np.empty((rows, cols), np.int8)
    s = np.empty(rows, np.float32)
    if w.dtype == np.uint16:
        _load().synth_quantize_rows_bf16(_p(w), rows, cols, _p(q), _p(s))
    elif w.dtype == np.float32:
        _load().synth_quantize_rows_f32(_p(w), rows, cols, _p(q), _p(s))
    else:
        raise TypeError(w.dtype)
    return q, s


def matrix_i8(k: int, rows: int, cols: int, sigma: float = 0.02):
    """Draw a bf16 N(0, sigma) [rows, cols] matrix and quantise it per row."""
    assert cols <= 16384
    q = np.empty((rows, cols), np.int8)
    s = np.empty(rows, np.float32)
    _load().synth_matrix_i8(k, rows, cols, sigma, _p(q), _p(s))
    return q, s


def ids(k: int, n: int, vocab: int) -> np.ndarray:
    out = np.empty(n, np.int32)
    _load().synth_ids(k, n, vocab, _p(out))
    return out


def lengths(k: int, n: int, lo: int, hi: int) -> np.ndarray:
    out = np.empty(n, np.int32)
    _load().synth_lengths(k, n, lo, hi, _p(out))
    return out


# --------------------------------------------------------------------------- shapes

@dataclass(frozen=True)
class Shape:
    name: str
    hidden: int
    n_layers: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    intermediate: int
    vocab: int
    rope_theta: float = 1.0e6
    rms_eps: float = 1.0e-6

    @property
    def dq(self) -> int:
        return self.n_heads * self.head_dim

    @property
    def dkv(self) -> int:
        return self.n_kv_heads * self.head_dim

    def weight_bytes(self) -> int:
        """int8 weights + fp32 scales + fp32 norm gains read once per decode step."""
        H, I, V, L = self.hidden, self.intermediate, self.vocab, self.n_layers
        per_layer_w = (self.dq + 2 * self.dkv) * H + H * self.dq + 2 * I * H + H * I
        per_layer_s = (self.dq + 2 * self.dkv) + H + 2 * I + H
        per_layer_g = 2 * H + 2 * self.head_dim
        return (V * H + L * per_layer_w) + 4 * (V + L * per_layer_s) + 4 * (L * per_layer_g + H)

    def kv_bytes_per_position(self) -> int:
        """bf16 K and V over all layers for one position of one sequence."""
        return self.n_layers * 2 * self.dkv * 2


TINY = Shape("qwen3-tiny", 256, 2, 4, 2, 64, 768, 4096)
QWEN3_0_6B = Shape("qwen3-0.6b", 1024, 28, 16, 8, 128, 3072, 151936)
QWEN3_1_7B = Shape("qwen3-1.7b", 2048, 28, 16, 8, 128, 6144, 151936)
SHAPES = {s.name: s for s in (TINY, QWEN3_0_6B, QWEN3_1_7B)}


@dataclass(frozen=True)
class Workload:
    """One measured decode workload: shape, batch, prompt lengths, new tokens."""
    name: str
    number: int
    shape: Shape
    batch: int
    prompt_len: int | None          # fixed prompt length, or None for drawn lengths
    prompt_range: tuple | None      # (lo, hi) inclusive when lengths are drawn
    new_tokens: int
    max_ctx: int                    # per-sequence KV capacity

    @property
    def weight_seed(self) -> int:
        return 1000 + self.number

    @property
    def prompt_seed(self) -> int:
        return 2000 + self.number


def _ctx(n: int) -> int:
    # context sizing rule: max(512, prompt + new)
    return max(512, n)


WORKLOADS = {
    w.name: w for w in [
        Workload("tiny-b1-p8-n16", 1, TINY, 1, 8, None, 16, _ctx(24)),
        Workload("0.6b-b1-p32-n128", 2, QWEN3_0_6B, 1, 32, None, 128, _ctx(160)),
        Workload("0.6b-b8-p16to256-n128", 3, QWEN3_0_6B, 8, None, (16, 256), 128, 512),
        Workload("0.6b-b16-p16to256-n128", 3, QWEN3_0_6B, 16, None, (16, 256), 128, 512),
        Workload("0.6b-b32-p16to256-n128", 3, QWEN3_0_6B, 32, None, (16, 256), 128, 512),
        Workload("1.7b-b1-p256-n1024", 4, QWEN3_1_7B, 1, 256, None, 1024, _ctx(1280)),
        Workload("0.6b-b1-p4096-n2048", 5, QWEN3_0_6B, 1, 4096, None, 2048, _ctx(6144)),
    ]
}


# --------------------------------------------------------------------------- models

@dataclass
class Mat:
    q: np.ndarray   # int8 [out, in], row-major (nn.Linear order)
    s: np.ndarray   # fp32 [out]


@dataclass
class Layer:
    wq: Mat
    wk: Mat
    wv: Mat
    wo: Mat
    wg: Mat
    wu: Mat
    wd: Mat
    attn_norm: np.ndarray
    ffn_norm: np.ndarray
    q_norm: np.ndarray
    k_norm: np.ndarray


@dataclass
class Model:
    shape: Shape
    embed: Mat                    # tied: embedding gather and lm_head
    layers: list = field(default_factory=list)
    final_norm: np.ndarray | None = None


def make_model(shape: Shape, seed: int, sigma: float = 0.02, random_gains: bool = False) -> Model:
    """Random-init model.  Tensor stream order: E, then per layer q, k, v, o,
    gate, up, down (stream index 0, 1 + 7l + j); gains use streams after those."""
    H, I = shape.hidden, shape.intermediate
    t = 0

    def mat(rows, cols):
        nonlocal t
        q, s = matrix_i8(key(seed, t), rows, cols, sigma)
        t += 1
        return Mat(q, s)

    embed = mat(shape.vocab, H)
    layers = []
    for _ in range(shape.n_layers):
        wq, wk, wv = mat(shape.dq, H), mat(shape.dkv, H), mat(shape.dkv, H)
        wo = mat(H, shape.dq)
        wg, wu = mat(I, H), mat(I, H)
        wd = mat(H, I)
        layers.append(Layer(wq, wk, wv, wo, wg, wu, wd,
                            np.ones(H, np.float32), np.ones(H, np.float32),
                            np.ones(shape.head_dim, np.float32), np.ones(shape.head_dim, np.float32)))
    final = np.ones(H, np.float32)
    if random_gains:
        g = 10_000

        def gain(n):
            nonlocal g
            v = normal_f32(key(seed, g), n, 1.0, 0.1)
            g += 1
            return v

        for ly in layers:
            ly.attn_norm, ly.ffn_norm = gain(H), gain(H)
            ly.q_norm, ly.k_norm = gain(shape.head_dim), gain(shape.head_dim)
        final = gain(H)
    return Model(shape, embed, layers, final)


def prompts(w: Workload, batch: int | None = None):
    """Prompt id arrays for a workload (list of int32 arrays, one per sequence)."""
    B = w.batch if batch is None else batch
    if w.prompt_len is not None:
        lens = np.full(B, w.prompt_len, np.int32)
    else:
        lens = lengths(key(w.prompt_seed, 0), B, *w.prompt_range)
    return [ids(key(w.prompt_seed, 1 + b), int(lens[b]), w.shape.vocab) for b in range(B)]
