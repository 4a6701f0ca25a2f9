"""CPU oracle for int8 weight-only Qwen3-family decode -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library and its Python binding
never touch it, and it imports nothing from them.

The arithmetic lives in ``orc.c`` (plain fp32 C, one sequential accumulator
per dot product, no fused multiply-add); this module only compiles it with
gcc and marshals numpy arrays through ctypes.  What each function follows:

* ``rmsnorm``, ``rope``, ``silu``, ``attention``, ``matmul_i8``: the decoder
  block of "Model-agnostic LLM inference", section "Supported models"
  (grouped-query attention with RMSNorm on Q/K, RoPE, SiLU-gated FFN, tied
  embeddings, no attention bias) with int8 weights and per-row scales (same
  page, section "The quantized load cache").
* ``argmax`` / ``greedy``: "Run local LLM decode", section "Limitations"
  (each generated token is the argmax at its step).
* ``Oracle.forward``: prefill builds the KV cache from the whole prompt and a
  decode step adds one token ("LLM inference overview", sections "Results"
  and "Workload characteristics"); both are the same causal pass here.
* ``sampling``: the sampling chain of "Model-agnostic LLM inference",
  section "Sampling" (penalties, temperature, top-k, min-p, top-p, seeded
  draw), in float64 numpy; see its module docstring for the readings.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "_build", "liborc.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile orc.c into oracle/_build/liborc.so (gcc, OpenMP, no FMA contraction)."""
    srcs = [os.path.join(_HERE, "orc.c"), os.path.join(_HERE, "orc.h")]
    if force or not os.path.exists(_SO) or any(os.path.getmtime(_SO) < os.path.getmtime(s) for s in srcs):
        os.makedirs(os.path.dirname(_SO), exist_ok=True)
        tmp = _SO + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O3", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
                               "-o", tmp, srcs[0], "-lm"])
        os.replace(tmp, _SO)
    return _SO


class _Dims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("hidden", "n_layers", "n_heads", "n_kv_heads", "head_dim", "intermediate", "vocab")] + \
               [("rope_theta", ctypes.c_float), ("rms_eps", ctypes.c_float)]


class _Mat(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("s", ctypes.c_void_p)]


class _Layer(ctypes.Structure):
    _fields_ = [(n, _Mat) for n in ("wq", "wk", "wv", "wo", "wg", "wu", "wd")] + \
               [(n, ctypes.c_void_p) for n in ("attn_norm", "ffn_norm", "q_norm", "k_norm")]


class _Model(ctypes.Structure):
    _fields_ = [("d", _Dims), ("embed", _Mat), ("layers", ctypes.POINTER(_Layer)),
                ("final_norm", ctypes.c_void_p)]


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            vp, i32, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
            lib.orc_bf16_bits.restype = ctypes.c_uint16
            lib.orc_bf16_bits.argtypes = [f32]
            lib.orc_bf16_value.restype = f32
            lib.orc_bf16_value.argtypes = [ctypes.c_uint16]
            lib.orc_rmsnorm.argtypes = [vp, vp, i32, f32, vp]
            lib.orc_rope.argtypes = [vp, i32, i32, f32]
            lib.orc_silu.restype = f32
            lib.orc_silu.argtypes = [f32]
            lib.orc_matmul_i8.argtypes = [ctypes.POINTER(_Mat), i32, i32, vp, i32, vp, i32]
            lib.orc_attention.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, vp]
            lib.orc_argmax.restype = i32
            lib.orc_argmax.argtypes = [vp, i32]
            lib.orc_cache_new.restype = vp
            lib.orc_cache_new.argtypes = [ctypes.POINTER(_Model), i32]
            lib.orc_cache_free.argtypes = [vp]
            lib.orc_cache_len.restype = i32
            lib.orc_cache_len.argtypes = [vp]
            lib.orc_cache_read.argtypes = [vp, i32, vp, vp]
            lib.orc_forward_block.restype = i32
            lib.orc_forward_block.argtypes = [ctypes.POINTER(_Model), vp, vp, i32, i32, vp, i32]
            lib.orc_greedy.restype = i32
            lib.orc_greedy.argtypes = [ctypes.POINTER(_Model), vp, i32, i32, ctypes.c_int32, vp, i32]
            _lib = lib
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "arrays passed to the oracle must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count() or 1)


# ------------------------------------------------------------------- pieces

def bf16_bits(x: float) -> int:
    return int(_load().orc_bf16_bits(float(x)))


def bf16_value(bits: int) -> float:
    return float(_load().orc_bf16_value(int(bits)))


def rmsnorm(x: np.ndarray, g: np.ndarray, eps: float) -> np.ndarray:
    x = np.ascontiguousarray(x, np.float32)
    g = np.ascontiguousarray(g, np.float32)
    y = np.empty_like(x)
    _load().orc_rmsnorm(_p(x), _p(g), x.size, eps, _p(y))
    return y


def rope(v: np.ndarray, pos: int, theta: float) -> np.ndarray:
    v = np.array(v, np.float32, copy=True, order="C")
    _load().orc_rope(_p(v), v.size, pos, theta)
    return v


def silu(z: float) -> float:
    return float(_load().orc_silu(float(z)))


def matmul_i8(q: np.ndarray, s: np.ndarray, x: np.ndarray, nthreads: int = 1) -> np.ndarray:
    """y[t] = s * (q @ x[t]) for x of shape [m, cols] (or [cols])."""
    q = np.ascontiguousarray(q, np.int8)
    s = np.ascontiguousarray(s, np.float32)
    x2 = np.ascontiguousarray(np.atleast_2d(x), np.float32)
    rows, cols = q.shape
    y = np.empty((x2.shape[0], rows), np.float32)
    m = _Mat(q.ctypes.data, s.ctypes.data)
    _load().orc_matmul_i8(ctypes.byref(m), rows, cols, _p(x2), x2.shape[0], _p(y), nthreads)
    return y if x.ndim == 2 else y[0]


def attention(q: np.ndarray, k_bits: np.ndarray, v_bits: np.ndarray, length: int | None = None) -> np.ndarray:
    """q [n_heads, hd] fp32; k_bits, v_bits [n_kv, cap, hd] bf16 bit patterns (uint16)."""
    q = np.ascontiguousarray(q, np.float32)
    k_bits = np.ascontiguousarray(k_bits, np.uint16)
    v_bits = np.ascontiguousarray(v_bits, np.uint16)
    nh, hd = q.shape
    nkv, cap, _ = k_bits.shape
    length = cap if length is None else length
    out = np.empty_like(q)
    _load().orc_attention(_p(q), _p(k_bits), _p(v_bits), length, cap, nh, nkv, hd, _p(out))
    return out


def argmax(z: np.ndarray) -> int:
    z = np.ascontiguousarray(z, np.float32)
    return int(_load().orc_argmax(_p(z), z.size))


# ------------------------------------------------------------------- model

class Oracle:
    """Holds ctypes views of a model (numpy arrays stay referenced here)."""

    def __init__(self, model, nthreads: int | None = None):
        _load()
        sh = model.shape
        self.shape = sh
        self.nthreads = nthreads or default_threads()
        self._keep = []

        def mat(m):
            q = np.ascontiguousarray(m.q, np.int8)
            s = np.ascontiguousarray(m.s, np.float32)
            self._keep += [q, s]
            return _Mat(q.ctypes.data, s.ctypes.data)

        def vec(a):
            a = np.ascontiguousarray(a, np.float32)
            self._keep.append(a)
            return a.ctypes.data

        layers = (_Layer * sh.n_layers)()
        for i, ly in enumerate(model.layers):
            layers[i] = _Layer(mat(ly.wq), mat(ly.wk), mat(ly.wv), mat(ly.wo), mat(ly.wg), mat(ly.wu),
                               mat(ly.wd), vec(ly.attn_norm), vec(ly.ffn_norm), vec(ly.q_norm),
                               vec(ly.k_norm))
        self._layers = layers
        dims = _Dims(sh.hidden, sh.n_layers, sh.n_heads, sh.n_kv_heads, sh.head_dim, sh.intermediate,
                     sh.vocab, sh.rope_theta, sh.rms_eps)
        self._m = _Model(dims, mat(model.embed), layers, vec(model.final_norm))

    # one sequence with its own KV cache
    class Seq:
        def __init__(self, orc: "Oracle", capacity: int):
            self.orc = orc
            self.h = _lib.orc_cache_new(ctypes.byref(orc._m), capacity)
            self.capacity = capacity

        def __del__(self):
            if getattr(self, "h", None):
                _lib.orc_cache_free(self.h)
                self.h = None

        @property
        def length(self) -> int:
            return int(_lib.orc_cache_len(self.h))

        def forward(self, ids, logits_from: int | None = None) -> np.ndarray | None:
            """Append ids (causal); return logits [n - logits_from, vocab] (default: last row)."""
            ids = np.ascontiguousarray(ids, np.int32)
            n = ids.size
            lf = n - 1 if logits_from is None else logits_from
            out = np.empty((max(n - lf, 0), self.orc.shape.vocab), np.float32) if lf < n else None
            rc = _lib.orc_forward_block(ctypes.byref(self.orc._m), self.h, _p(ids), n, lf,
                                        _p(out) if out is not None else None, self.orc.nthreads)
            if rc != 0:
                raise ValueError("oracle KV cache overflow")
            return out

        def kv(self, layer: int):
            """bf16 bit patterns [n_kv, len, hd] of K and V for one layer."""
            sh = self.orc.shape
            n = self.length
            k = np.empty((sh.n_kv_heads, n, sh.head_dim), np.uint16)
            v = np.empty_like(k)
            _lib.orc_cache_read(self.h, layer, _p(k), _p(v))
            return k, v

    def seq(self, capacity: int) -> "Oracle.Seq":
        return Oracle.Seq(self, capacity)

    def teacher_forced(self, ids, logits_from: int) -> np.ndarray:
        """Logits at every position >= logits_from of one causal pass over ids."""
        s = self.seq(len(ids))
        return s.forward(ids, logits_from)

    def greedy(self, prompt, max_new: int, eos_id: int = -1) -> np.ndarray:
        prompt = np.ascontiguousarray(prompt, np.int32)
        out = np.empty(max_new, np.int32)
        n = _lib.orc_greedy(ctypes.byref(self._m), _p(prompt), prompt.size, max_new, eos_id, _p(out),
                            self.nthreads)
        return out[:n]
