"""Python binding of libq3i8.so: int8 weight-only Qwen3-family decode on GB300.

Argument marshalling only.  Every step of the decode path runs in the CUDA
kernels of ``libq3i8.so`` (built in-tree by ``build.py``); there is no CPU or
PyTorch fallback.  If the library is missing, importing its functions raises.

The call surface mirrors the C ABI in ``include/q3i8.h``:

* ``Decoder(model, max_batch, max_ctx)``          -> ``q3i8_init``
* ``Decoder.decode(prompts, max_new_tokens)``     -> ``q3i8_decode`` (host ids)
* ``Decoder.decode_device(ids, lens, n, out)``    -> ``q3i8_decode_device``
* ``Decoder.prefill`` / ``Decoder.step_logits``   -> teacher-forced checking
* ``validate_dims``                               -> ``q3i8_validate_dims``
* ``op_gemm_i8``                                  -> ``q3i8_op_gemm_i8``
* ``op_attention``                                -> ``q3i8_op_attention``
* ``op_attention_static``                         -> ``q3i8_op_attention_static``

A model is any object with ``shape`` (hidden, n_layers, n_heads, n_kv_heads,
head_dim, intermediate, vocab, rope_theta, rms_eps), ``embed.q``/``embed.s``,
``final_norm`` and ``layers[i]`` holding ``wq wk wv wo wg wu wd`` (each with
int8 ``q`` [out, in] and fp32 ``s`` [out]) and the gains ``attn_norm
ffn_norm q_norm k_norm``.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.environ.get("Q3I8_LIB") or os.path.join(_HERE, "_build", "libq3i8.so")

STATUS = {0: "ok", 1: "unsupported_architecture", 2: "invalid_arguments", 3: "context_past_ceiling",
          4: "no_device", 5: "out_of_memory", 6: "cuda_error", 7: "device_wait_timeout", 8: "invalid_state"}

EXPORTS = ["q3i8_validate_dims", "q3i8_init", "q3i8_decode", "q3i8_decode_sample", "q3i8_decode_device", "q3i8_prefill",
           "q3i8_step_logits", "q3i8_read_kv", "q3i8_step_bytes", "q3i8_step_launches", "q3i8_launch_count", "q3i8_last_error",
           "q3i8_status_name", "q3i8_destroy", "q3i8_trace_step", "q3i8_op_gemm_i8", "q3i8_op_gemm_i8_splitk_workspace",
           "q3i8_op_gemm_i8_splitk", "q3i8_op_attention_workspace", "q3i8_op_attention",
           "q3i8_op_attention_static", "q3i8_op_sample_workspace", "q3i8_op_sample", "q3i8_op_wait_probe",
           "q3i8_cache_payload_bytes", "q3i8_cache_write",
           "q3i8_cache_open", "q3i8_cache_tables", "q3i8_cache_close", "q3i8_sched_new", "q3i8_sched_destroy",
           "q3i8_sched_submit", "q3i8_sched_plan", "q3i8_sched_complete_prefill", "q3i8_sched_complete_step",
           "q3i8_sched_idle", "q3i8_sched_result", "q3i8_cb_reserve", "q3i8_cb_prefill", "q3i8_cb_step",
           "q3i8_sched_run"]

# q3i8_cache_open gate results
CACHE_GATE = {0: "valid", 1: "absent", 2: "bad_magic", 3: "dims", 4: "manifest", 5: "length"}


class Q3Error(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{STATUS.get(code, code)}: {msg}")
        self.code = code
        self.status = STATUS.get(code, str(code))


class Dims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("hidden", "n_layers", "n_heads", "n_kv_heads", "head_dim", "intermediate", "vocab")] + \
               [("rope_theta", ctypes.c_float), ("rms_eps", ctypes.c_float)] + \
               [(n, ctypes.c_int32) for n in ("max_batch", "max_ctx", "tie_word_embeddings", "attention_bias")]


class Mat(ctypes.Structure):
    _fields_ = [("w", ctypes.c_void_p), ("scale", ctypes.c_void_p)]


class Layer(ctypes.Structure):
    _fields_ = [(n, Mat) for n in ("q", "k", "v", "o", "gate", "up", "down")] + \
               [(n, ctypes.c_void_p) for n in ("attn_norm", "ffn_norm", "q_norm", "k_norm")]


class Stats(ctypes.Structure):
    _fields_ = [(n, ctypes.c_double) for n in ("prefill_ms", "decode_ms", "prefill_tokens_per_sec",
                                               "decode_tokens_per_sec", "step_us")] + \
               [("prefill_tokens", ctypes.c_int64), ("decode_steps", ctypes.c_int64)]

    def as_dict(self):
        return {f: getattr(self, f) for f, _ in self._fields_}


class Sampling(ctypes.Structure):
    """Settings of the device sampling chain (q3i8_sampling)."""
    _fields_ = [(n, ctypes.c_double) for n in ("temperature", "top_p", "min_p", "repeat_penalty",
                                               "presence_penalty", "frequency_penalty")] + \
               [("top_k", ctypes.c_int32), ("reserved", ctypes.c_int32), ("seed", ctypes.c_uint64)]


def sampling(temperature: float, top_k: int, top_p: float = 1.0, min_p: float = 0.0, repeat_penalty: float = 1.0,
             presence_penalty: float = 0.0, frequency_penalty: float = 0.0, seed: int = 0) -> Sampling:
    return Sampling(temperature=temperature, top_p=top_p, min_p=min_p, repeat_penalty=repeat_penalty,
                    presence_penalty=presence_penalty, frequency_penalty=frequency_penalty, top_k=top_k, reserved=0,
                    seed=seed & ((1 << 64) - 1))


_lib = None
_lock = threading.Lock()


def lib():
    """The loaded libq3i8.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise ImportError(f"libq3i8.so is not built ({LIB_PATH}); run "
                                  "`python -m decode_int8_weight_gb300.build`")
            L = ctypes.CDLL(LIB_PATH)
            vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
            L.q3i8_validate_dims.argtypes = [ctypes.POINTER(Dims), ctypes.c_char_p, sz]
            L.q3i8_init.argtypes = [ctypes.POINTER(Dims), ctypes.POINTER(Mat), ctypes.POINTER(Layer), vp, vp,
                                    ctypes.POINTER(vp)]
            L.q3i8_decode.argtypes = [vp, i32, ctypes.POINTER(vp), vp, i32, i32, vp, vp, ctypes.POINTER(Stats)]
            L.q3i8_decode_sample.argtypes = [vp, i32, ctypes.POINTER(vp), vp, i32, i32, ctypes.POINTER(Sampling),
                                             vp, vp, ctypes.POINTER(Stats)]
            L.q3i8_op_sample_workspace.restype = sz
            L.q3i8_op_sample_workspace.argtypes = [i32, i32]
            L.q3i8_op_sample.argtypes = [vp, i32, i32, vp, ctypes.POINTER(Sampling), i32, vp, vp, sz, vp, vp]
            L.q3i8_decode_device.argtypes = [vp, i32, vp, vp, i32, vp, ctypes.POINTER(Stats)]
            L.q3i8_prefill.argtypes = [vp, i32, ctypes.POINTER(vp), vp, vp]
            L.q3i8_step_logits.argtypes = [vp, vp, vp]
            L.q3i8_read_kv.argtypes = [vp, i32, i32, i32, vp, vp]
            L.q3i8_step_bytes.restype = i64
            L.q3i8_step_bytes.argtypes = [vp, i32, vp]
            L.q3i8_step_launches.restype = i32
            L.q3i8_step_launches.argtypes = [vp, i32]
            L.q3i8_launch_count.restype = i64
            L.q3i8_launch_count.argtypes = [vp]
            L.q3i8_last_error.restype = ctypes.c_char_p
            L.q3i8_last_error.argtypes = [vp]
            L.q3i8_status_name.restype = ctypes.c_char_p
            L.q3i8_status_name.argtypes = [ctypes.c_int]
            L.q3i8_destroy.argtypes = [vp]
            L.q3i8_trace_step.argtypes = [vp, vp, vp, sz, ctypes.POINTER(i32), ctypes.POINTER(i32)]
            L.q3i8_op_gemm_i8.argtypes = [vp, vp, vp, i32, i32, i32, vp, vp, vp]
            L.q3i8_op_gemm_i8_splitk_workspace.restype = sz
            L.q3i8_op_gemm_i8_splitk_workspace.argtypes = [i32, i32, i32]
            L.q3i8_op_gemm_i8_splitk.argtypes = [vp, vp, vp, i32, i32, i32, vp, vp, sz, vp, vp]
            L.q3i8_op_attention_workspace.restype = sz
            L.q3i8_op_attention_workspace.argtypes = [i32, i32, i32, i32]
            L.q3i8_op_attention.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, vp, vp, sz, vp, vp]
            L.q3i8_op_attention_static.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, vp, vp, vp]
            L.q3i8_op_wait_probe.argtypes = [i32, i32, vp, vp, vp]
            L.q3i8_cache_payload_bytes.restype = ctypes.c_uint64
            L.q3i8_cache_payload_bytes.argtypes = [ctypes.POINTER(Dims)]
            L.q3i8_cache_write.argtypes = [ctypes.c_char_p, ctypes.POINTER(Dims), ctypes.POINTER(Mat),
                                           ctypes.POINTER(Layer), vp, ctypes.c_char_p, sz]
            L.q3i8_cache_open.argtypes = [ctypes.c_char_p, ctypes.POINTER(Dims), ctypes.c_char_p, sz,
                                          ctypes.POINTER(vp), ctypes.POINTER(i32)]
            L.q3i8_cache_tables.argtypes = [vp, ctypes.POINTER(Mat), ctypes.POINTER(Layer), ctypes.POINTER(vp)]
            L.q3i8_cache_close.argtypes = [vp]
            L.q3i8_sched_new.argtypes = [i32, i32, ctypes.POINTER(vp)]
            L.q3i8_sched_destroy.argtypes = [vp]
            L.q3i8_sched_submit.argtypes = [vp, vp, i32, i32, i32, ctypes.POINTER(i32)]
            L.q3i8_sched_plan.argtypes = [vp, ctypes.POINTER(i32), vp, vp, ctypes.POINTER(i32), vp, vp, vp, vp]
            L.q3i8_sched_complete_prefill.argtypes = [vp, i32, vp, vp]
            L.q3i8_sched_complete_step.argtypes = [vp, i32, vp]
            L.q3i8_sched_idle.restype = i32
            L.q3i8_sched_idle.argtypes = [vp]
            L.q3i8_cb_reserve.argtypes = [vp, i32]
            L.q3i8_cb_prefill.argtypes = [vp, i32, vp, ctypes.POINTER(vp), vp, vp]
            L.q3i8_cb_step.argtypes = [vp, i32, vp, vp, vp, vp]
            L.q3i8_sched_run.argtypes = [vp, vp, ctypes.POINTER(Stats)]
            L.q3i8_sched_result.argtypes = [vp, i32, vp, i32, ctypes.POINTER(i32), ctypes.POINTER(i32)]
            _lib = L
    return _lib


def _check(rc: int, ctx=None):
    if rc != 0:
        raise Q3Error(rc, lib().q3i8_last_error(ctx).decode(errors="replace"))


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def make_dims(shape, max_batch: int = 1, max_ctx: int = 0, tie_word_embeddings: int = 1,
              attention_bias: int = 0) -> Dims:
    return Dims(shape.hidden, shape.n_layers, shape.n_heads, shape.n_kv_heads, shape.head_dim, shape.intermediate,
                shape.vocab, shape.rope_theta, shape.rms_eps, max_batch, max_ctx, tie_word_embeddings,
                attention_bias)


def validate_dims(dims: Dims):
    """(status, message) of the host-only architecture check (no GPU needed)."""
    buf = ctypes.create_string_buffer(2048)
    rc = lib().q3i8_validate_dims(ctypes.byref(dims), buf, len(buf))
    return rc, buf.value.decode()


def _tptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _host_tables(model):
    """q3i8_init's host argument tables for a model (synth.Model layout).
    Returns (embed Mat, Layer array, final_norm address, arrays to keep alive)."""
    keep = []

    def mat(m):
        q = np.ascontiguousarray(m.q, np.int8)
        s = np.ascontiguousarray(m.s, np.float32)
        keep.extend([q, s])
        return Mat(q.ctypes.data, s.ctypes.data)

    def vec(a):
        a = np.ascontiguousarray(a, np.float32)
        keep.append(a)
        return a.ctypes.data

    layers = (Layer * model.shape.n_layers)()
    for i, ly in enumerate(model.layers):
        layers[i] = Layer(mat(ly.wq), mat(ly.wk), mat(ly.wv), mat(ly.wo), mat(ly.wg), mat(ly.wu), mat(ly.wd),
                          vec(ly.attn_norm), vec(ly.ffn_norm), vec(ly.q_norm), vec(ly.k_norm))
    emb = mat(model.embed)
    fin = vec(model.final_norm)
    return emb, layers, fin, keep


class Decoder:
    """One q3i8 context: weights resident on the current CUDA device."""

    def __init__(self, model, max_batch: int = 1, max_ctx: int = 0, stream=None):
        sh = model.shape
        self.shape = sh
        self.max_batch = max_batch
        dims = make_dims(sh, max_batch, max_ctx)
        emb, layers, fin, keep = _host_tables(model)
        h = ctypes.c_void_p()
        rc = lib().q3i8_init(ctypes.byref(dims), ctypes.byref(emb), layers, ctypes.c_void_p(fin),
                             ctypes.c_void_p(stream) if stream else None, ctypes.byref(h))
        _check(rc, None)
        self._h = h
        del keep  # weights were copied to the device

    def close(self):
        if getattr(self, "_h", None):
            lib().q3i8_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def _prompts(self, prompts):
        arrs = [np.ascontiguousarray(p, np.int32) for p in prompts]
        ptrs = (ctypes.c_void_p * len(arrs))(*[a.ctypes.data for a in arrs])
        lens = np.array([a.size for a in arrs], np.int32)
        return arrs, ptrs, lens

    def decode(self, prompts, max_new_tokens: int, eos_id: int = -1):
        """Greedy decode (host buffers).  Returns (ids [B, max_new], counts [B], stats dict)."""
        arrs, ptrs, lens = self._prompts(prompts)
        B = len(arrs)
        out = np.zeros((B, max_new_tokens), np.int32)
        counts = np.zeros(B, np.int32)
        st = Stats()
        rc = lib().q3i8_decode(self._h, B, ptrs, _p(lens), max_new_tokens, eos_id, _p(out), _p(counts),
                               ctypes.byref(st))
        _check(rc, self._h)
        return out, counts, st.as_dict()

    def decode_sample(self, prompts, max_new_tokens: int, settings: Sampling, eos_id: int = -1):
        """Sampled decode (host buffers; see q3i8_decode_sample).  Returns (ids, counts, stats dict)."""
        arrs, ptrs, lens = self._prompts(prompts)
        B = len(arrs)
        out = np.zeros((B, max_new_tokens), np.int32)
        counts = np.zeros(B, np.int32)
        st = Stats()
        rc = lib().q3i8_decode_sample(self._h, B, ptrs, _p(lens), max_new_tokens, eos_id, ctypes.byref(settings),
                                      _p(out), _p(counts), ctypes.byref(st))
        _check(rc, self._h)
        return out, counts, st.as_dict()

    def decode_device(self, d_ids, lens, max_new_tokens: int, d_out):
        """Greedy decode on device buffers (torch int32 CUDA tensors).  Returns stats."""
        lens = np.ascontiguousarray(lens, np.int32)
        st = Stats()
        rc = lib().q3i8_decode_device(self._h, lens.size, _tptr(d_ids), _p(lens), max_new_tokens, _tptr(d_out),
                                      ctypes.byref(st))
        _check(rc, self._h)
        return st.as_dict()

    def prefill(self, prompts, want_logits: bool = True):
        arrs, ptrs, lens = self._prompts(prompts)
        out = np.zeros((len(arrs), self.shape.vocab), np.float32) if want_logits else None
        rc = lib().q3i8_prefill(self._h, len(arrs), ptrs, _p(lens), _p(out) if out is not None else None)
        _check(rc, self._h)
        return out

    def step_logits(self, tokens):
        tokens = np.ascontiguousarray(tokens, np.int32)
        out = np.zeros((tokens.size, self.shape.vocab), np.float32)
        rc = lib().q3i8_step_logits(self._h, _p(tokens), _p(out))
        _check(rc, self._h)
        return out

    def read_kv(self, layer: int, seq: int, n_pos: int):
        sh = self.shape
        k = np.zeros((sh.n_kv_heads, n_pos, sh.head_dim), np.uint16)
        v = np.zeros_like(k)
        _check(lib().q3i8_read_kv(self._h, layer, seq, n_pos, _p(k), _p(v)), self._h)
        return k, v

    def step_bytes(self, positions) -> int:
        positions = np.ascontiguousarray(positions, np.int32)
        return int(lib().q3i8_step_bytes(self._h, positions.size, _p(positions)))

    def step_launches(self, B: int) -> int:
        return int(lib().q3i8_step_launches(self._h, B))

    def trace_step(self, tokens):
        """One traced decode step: per-CTA %globaltimer stamps [grid, stride] (ns)."""
        tokens = np.ascontiguousarray(tokens, np.int32)
        grid, stride = ctypes.c_int32(), ctypes.c_int32()
        lib().q3i8_trace_step(self._h, _p(tokens), None, 0, ctypes.byref(grid), ctypes.byref(stride))
        out = np.zeros((grid.value, stride.value), np.uint64)
        _check(lib().q3i8_trace_step(self._h, _p(tokens), _p(out), out.size, ctypes.byref(grid),
                                     ctypes.byref(stride)), self._h)
        return out

    def launch_count(self) -> int:
        return int(lib().q3i8_launch_count(self._h))

    # continuous batching on the device (q3i8_cb_*, q3i8_sched_run)
    def cb_reserve(self, max_ctx: int):
        _check(lib().q3i8_cb_reserve(self._h, max_ctx), self._h)

    def cb_prefill(self, slots, prompts):
        arrs, ptrs, lens = self._prompts(prompts)
        slots = np.ascontiguousarray(slots, np.int32)
        out = np.zeros(len(arrs), np.int32)
        _check(lib().q3i8_cb_prefill(self._h, len(arrs), _p(slots), ptrs, _p(lens), _p(out)), self._h)
        return out

    def cb_step(self, slots, positions, tokens):
        slots = np.ascontiguousarray(slots, np.int32)
        positions = np.ascontiguousarray(positions, np.int32)
        tokens = np.ascontiguousarray(tokens, np.int32)
        out = np.zeros(slots.size, np.int32)
        _check(lib().q3i8_cb_step(self._h, slots.size, _p(slots), _p(positions), _p(tokens), _p(out)), self._h)
        return out

    def sched_run(self, sched):
        """Run a Scheduler to idle on this context's GPU; returns the stats dict."""
        st = Stats()
        _check(lib().q3i8_sched_run(self._h, sched._h, ctypes.byref(st)), self._h)
        return st.as_dict()


def op_gemm_i8(a_planes, w, scale, y, status=None, stream=None):
    """Tensor-core projection on torch CUDA tensors (see q3i8_op_gemm_i8): a_planes [M, 2K] (f16 bits as int16 or
    float16), w [N, K] int8, scale [N] fp32, y [M, N] fp32."""
    M, K2 = a_planes.shape
    N, K = w.shape
    assert K2 == 2 * K
    rc = lib().q3i8_op_gemm_i8(_tptr(a_planes), _tptr(w), _tptr(scale), M, N, K, _tptr(y), _tptr(status),
                               ctypes.c_void_p(stream) if stream else None)
    _check(rc, None)


def op_gemm_i8_splitk_workspace(M: int, N: int, K: int) -> int:
    return int(lib().q3i8_op_gemm_i8_splitk_workspace(M, N, K))


def op_gemm_i8_splitk(a_planes, w, scale, y, workspace=None, status=None, stream=None):
    """op_gemm_i8 with K split over CTAs when the shape calls for it (see q3i8_op_gemm_i8_splitk); workspace: a
    torch CUDA tensor of at least op_gemm_i8_splitk_workspace(M, N, K) bytes, or None when that is 0."""
    M, K2 = a_planes.shape
    N, K = w.shape
    assert K2 == 2 * K
    nbytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    rc = lib().q3i8_op_gemm_i8_splitk(_tptr(a_planes), _tptr(w), _tptr(scale), M, N, K, _tptr(y), _tptr(workspace),
                                      nbytes, _tptr(status), ctypes.c_void_p(stream) if stream else None)
    _check(rc, None)


def op_attention_workspace(R: int, n_heads: int, hd: int, splits: int) -> int:
    return int(lib().q3i8_op_attention_workspace(R, n_heads, hd, splits))


def op_attention(q, k, v, row_seq, row_len, n_kv_heads: int, splits: int, out, workspace, status=None,
                 stream=None):
    """Split-KV decode attention on torch CUDA tensors (see q3i8_op_attention)."""
    R, nh, hd = q.shape
    cap = k.shape[2]
    rc = lib().q3i8_op_attention(_tptr(q), _tptr(k), _tptr(v), _tptr(row_seq), _tptr(row_len), R, nh, n_kv_heads,
                                 hd, cap, splits, _tptr(out), _tptr(workspace),
                                 workspace.numel() * workspace.element_size(), _tptr(status),
                                 ctypes.c_void_p(stream) if stream else None)
    _check(rc, None)


def op_sample_workspace(B: int, V: int) -> int:
    return int(lib().q3i8_op_sample_workspace(B, V))


def op_sample(logits, counts, settings: Sampling, step: int, tokens, workspace, status=None, stream=None):
    """The sampling chain on one step's logits (see q3i8_op_sample): logits [B, V] fp32, counts [B, V] int32
    (updated), tokens [B] int32, workspace uint8 of op_sample_workspace(B, V) bytes; torch CUDA tensors."""
    B, V = logits.shape
    rc = lib().q3i8_op_sample(_tptr(logits), B, V, _tptr(counts), ctypes.byref(settings), step, _tptr(tokens),
                              _tptr(workspace), workspace.numel() * workspace.element_size(), _tptr(status),
                              ctypes.c_void_p(stream) if stream else None)
    _check(rc, None)


#: Largest scratch, in bytes, that ``op_attention_static`` may need.
OP_ATTENTION_STATIC_SCRATCH_BYTES = 4 << 20


def op_attention_static(q, k, v, row_seq, row_len, n_kv_heads: int, splits: int, out, status=None, stream=None):
    """``op_attention`` without a workspace: the partial states go to scratch
    compiled into the library, so nothing is allocated (see
    q3i8_op_attention_static).  Calls that overlap on one device race."""
    R, nh, hd = q.shape
    cap = k.shape[2]
    rc = lib().q3i8_op_attention_static(_tptr(q), _tptr(k), _tptr(v), _tptr(row_seq), _tptr(row_len), R, nh,
                                        n_kv_heads, hd, cap, splits, _tptr(out), _tptr(status),
                                        ctypes.c_void_p(stream) if stream else None)
    _check(rc, None)


def op_wait_probe(arrive: bool, limit: int, status, elapsed_ns=None, stream=None):
    """Run the library's bounded mbarrier wait on a phase that completes only
    when ``arrive`` is set, with at most ``limit`` polls (negative: the
    kernels' own limit).  ``status`` is a device int32 tensor, ``elapsed_ns``
    an optional device int64 tensor.  Raises Q3Error (code Q3_ERR_TIMEOUT)
    when the wait ran out (see q3i8_op_wait_probe)."""
    rc = lib().q3i8_op_wait_probe(1 if arrive else 0, int(limit), _tptr(status), _tptr(elapsed_ns),
                                  ctypes.c_void_p(stream) if stream else None)
    _check(rc, None)


# ------------------------------------------------------------ quantized load cache

class _CMat:
    def __init__(self, q, s):
        self.q, self.s = q, s


class _CLayer:
    pass


class CachedModel:
    """A model (synth.Model layout) whose arrays are views of an open cache's
    bytes (q3i8_cache_open); the cache stays open while this object lives."""

    def __init__(self, shape, handle):
        self.shape = shape
        self._h = handle
        L = lib()
        n = shape.n_layers
        emb, layers, fin = Mat(), (Layer * n)(), ctypes.c_void_p()
        _check(L.q3i8_cache_tables(handle, ctypes.byref(emb), layers, ctypes.byref(fin)), None)
        H, I, hd = shape.hidden, shape.intermediate, shape.head_dim
        Dq, Dkv = shape.n_heads * hd, shape.n_kv_heads * hd

        def arr(addr, ctype, shp):
            return np.ctypeslib.as_array(ctypes.cast(addr, ctypes.POINTER(ctype)), shape=shp)

        def mat(m, rows, cols):
            return _CMat(arr(m.w, ctypes.c_int8, (rows, cols)), arr(m.scale, ctypes.c_float, (rows,)))

        self.embed = mat(emb, shape.vocab, H)
        self.final_norm = arr(fin.value, ctypes.c_float, (H,))
        self.layers = []
        for ly in layers:
            c = _CLayer()
            c.wq, c.wk, c.wv = mat(ly.q, Dq, H), mat(ly.k, Dkv, H), mat(ly.v, Dkv, H)
            c.wo = mat(ly.o, H, Dq)
            c.wg, c.wu, c.wd = mat(ly.gate, I, H), mat(ly.up, I, H), mat(ly.down, H, I)
            c.attn_norm, c.ffn_norm = arr(ly.attn_norm, ctypes.c_float, (H,)), arr(ly.ffn_norm, ctypes.c_float, (H,))
            c.q_norm, c.k_norm = arr(ly.q_norm, ctypes.c_float, (hd,)), arr(ly.k_norm, ctypes.c_float, (hd,))
            self.layers.append(c)

    def close(self):
        if getattr(self, "_h", None):
            lib().q3i8_cache_close(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def cache_payload_bytes(shape) -> int:
    d = make_dims(shape, 1)
    return int(lib().q3i8_cache_payload_bytes(ctypes.byref(d)))


def cache_write(path: str, model, manifest: bytes = b""):
    """Write the model's post-quantization arrays to a cache file (q3i8_cache_write)."""
    d = make_dims(model.shape, 1)
    emb, layers, fin, keep = _host_tables(model)
    rc = lib().q3i8_cache_write(os.fsencode(path), ctypes.byref(d), ctypes.byref(emb), layers,
                                ctypes.c_void_p(fin), manifest, len(manifest))
    _check(rc, None)
    del keep


def cache_open(path: str, shape, manifest: bytes = b""):
    """(CachedModel or None, gate name): the cache at path if it passes the
    gate for this shape and manifest (q3i8_cache_open)."""
    d = make_dims(shape, 1)
    h, gate = ctypes.c_void_p(), ctypes.c_int32(-1)
    rc = lib().q3i8_cache_open(os.fsencode(path), ctypes.byref(d), manifest, len(manifest), ctypes.byref(h),
                               ctypes.byref(gate))
    _check(rc, None)
    if gate.value != 0:
        return None, CACHE_GATE[gate.value]
    return CachedModel(shape, h), "valid"


def load_cached(path: str, shape, manifest: bytes, build):
    """The page's flow: restore the cache when it passes the gate, otherwise
    call build() (the full path: convert and quantize), write a fresh cache
    and return the built model.  Returns (model, gate name of the cache that
    was found)."""
    model, gate = cache_open(path, shape, manifest)
    if model is not None:
        return model, gate
    model = build()
    cache_write(path, model, manifest)
    return model, gate


# ------------------------------------------------------------ continuous batching

class Scheduler:
    """Host scheduler of a continuous batch (q3i8_sched_*): FIFO admission
    into free KV slots between steps, retirement at max_new_tokens or eos."""

    def __init__(self, max_batch: int, max_ctx: int):
        self.max_batch = max_batch
        h = ctypes.c_void_p()
        _check(lib().q3i8_sched_new(max_batch, max_ctx, ctypes.byref(h)), None)
        self._h = h

    def close(self):
        if getattr(self, "_h", None):
            lib().q3i8_sched_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def submit(self, prompt, max_new_tokens: int, eos_id: int = -1) -> int:
        p = np.ascontiguousarray(prompt, np.int32)
        rid = ctypes.c_int32()
        _check(lib().q3i8_sched_submit(self._h, _p(p), p.size, max_new_tokens, eos_id, ctypes.byref(rid)), None)
        return rid.value

    def plan(self):
        """(admissions [(request, slot)], rows [(request, slot, position, token)])."""
        n = self.max_batch
        na, nr = ctypes.c_int32(), ctypes.c_int32()
        ar, asl = np.zeros(n, np.int32), np.zeros(n, np.int32)
        rr, rs, rp, rt = (np.zeros(n, np.int32) for _ in range(4))
        _check(lib().q3i8_sched_plan(self._h, ctypes.byref(na), _p(ar), _p(asl), ctypes.byref(nr), _p(rr), _p(rs),
                                     _p(rp), _p(rt)), None)
        adm = [(int(ar[i]), int(asl[i])) for i in range(na.value)]
        rows = [(int(rr[i]), int(rs[i]), int(rp[i]), int(rt[i])) for i in range(nr.value)]
        return adm, rows

    def complete_prefill(self, request_ids, first_tokens):
        r = np.ascontiguousarray(request_ids, np.int32)
        t = np.ascontiguousarray(first_tokens, np.int32)
        assert r.size == t.size
        _check(lib().q3i8_sched_complete_prefill(self._h, r.size, _p(r), _p(t)), None)

    def complete_step(self, tokens):
        t = np.ascontiguousarray(tokens, np.int32)
        _check(lib().q3i8_sched_complete_step(self._h, t.size, _p(t)), None)

    def idle(self) -> bool:
        return bool(lib().q3i8_sched_idle(self._h))

    def result(self, request_id: int):
        """(tokens generated so far, finished)."""
        n, done = ctypes.c_int32(), ctypes.c_int32()
        _check(lib().q3i8_sched_result(self._h, request_id, None, 0, ctypes.byref(n), ctypes.byref(done)), None)
        out = np.zeros(max(n.value, 1), np.int32)
        _check(lib().q3i8_sched_result(self._h, request_id, _p(out), n.value, ctypes.byref(n), ctypes.byref(done)),
               None)
        return out[:n.value], bool(done.value)
