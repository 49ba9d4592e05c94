"""ctypes binding to the C oracle (``gpt2_ref.c``).

TEST INFRASTRUCTURE ONLY: the test suite, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference leg are the only callers.  The oracle is
single-threaded C99 in binary32 (the LeanExe GPT-2 README fixes binary32
arithmetic), built with ``-O2 -ffp-contract=off``; it shares no code with the
CUDA library.  Status names mirror the C codes; they are compared by name.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gpt2_ref.c")
_OUT = os.path.join(_HERE, "_build", "libgpt2ref.so")

STATUS = {0: "ok", 1: "weights_len", 2: "token", 3: "position", 4: "cache_len",
          5: "tokens_len", 6: "nonfinite", 7: "config", 8: "nomem"}


def build(src: str = _SRC, out: str = _OUT, extra=()) -> str:
    """Compile the oracle into a shared library with gcc; returns its path."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    cmd = ["gcc", "-std=c99", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
           *extra, "-o", out, src, "-lm"]
    subprocess.run(cmd, check=True)
    return out


class _Cfg(C.Structure):
    _fields_ = [(n, C.c_uint32) for n in
                ("n_layer", "d_model", "n_head", "d_ff", "vocab", "n_pos", "max_pos")]


def _cfg(shape) -> _Cfg:
    return _Cfg(*shape.as_tuple())


_f32p = np.ctypeslib.ndpointer(np.float32, flags="C_CONTIGUOUS")
_i8p = np.ctypeslib.ndpointer(np.int8, flags="C_CONTIGUOUS")
_i32p = np.ctypeslib.ndpointer(np.int32, flags="C_CONTIGUOUS")


class Oracle:
    """Loaded oracle library.  ``path`` selects a build (the tests also load
    deliberately broken builds to check that the pins catch them)."""

    def __init__(self, path: str | None = None):
        if path is None:
            path = _OUT
            if not os.path.exists(path) or os.path.getmtime(path) < os.path.getmtime(_SRC):
                build()
        L = C.CDLL(path)
        self.lib = L
        L.ref_weight_words.argtypes = [C.POINTER(_Cfg)]
        L.ref_weight_words.restype = C.c_size_t
        L.ref_cache_words_per_position.argtypes = [C.POINTER(_Cfg)]
        L.ref_cache_words_per_position.restype = C.c_size_t
        L.ref_layernorm.argtypes = [_f32p, _f32p, _f32p, C.c_int, _f32p]
        L.ref_gelu.argtypes = [C.c_float]
        L.ref_gelu.restype = C.c_float
        L.ref_argmax.argtypes = [_f32p, C.c_size_t, C.POINTER(C.c_uint32)]
        L.ref_group_scale.argtypes = [_f32p, C.c_int]
        L.ref_group_scale.restype = C.c_float
        L.ref_quantize.argtypes = [_f32p, C.c_int, C.c_float, _i8p]
        L.ref_quantize_groups.argtypes = [_f32p, C.c_int, _i8p, _f32p]
        L.ref_quantize_row.argtypes = [_f32p, C.c_int, _i8p, _f32p]
        L.ref_q8_group_dots.argtypes = [_i8p, _i8p, C.c_int, _i32p]
        L.ref_linear_f32.argtypes = [_f32p, _f32p, C.c_void_p, C.c_int, C.c_int, _f32p]
        L.ref_linear_q8.argtypes = [_f32p, _i8p, _f32p, C.c_void_p, C.c_int, C.c_int, _f32p]
        L.ref_linear_q8_rowx.argtypes = [_f32p, _i8p, _f32p, C.c_void_p, C.c_int, C.c_int, _f32p]
        L.ref_attention_head.argtypes = [_f32p, C.c_void_p, C.c_void_p, C.c_int, C.c_int, C.c_size_t,
                                         _f32p, C.c_void_p]
        L.ref_model_create.argtypes = [C.POINTER(_Cfg), C.c_void_p, C.c_size_t, C.c_int, C.POINTER(C.c_int)]
        L.ref_model_create.restype = C.c_void_p
        L.ref_model_free.argtypes = [C.c_void_p]
        L.ref_model_get_q8.argtypes = [C.c_void_p, C.c_int, _i8p, _f32p]
        L.ref_model_cached_step.argtypes = [C.c_void_p, C.c_void_p, C.c_size_t, C.c_uint32, C.c_uint32,
                                            C.c_void_p, C.POINTER(C.c_size_t), C.c_void_p,
                                            C.POINTER(C.c_size_t), C.c_void_p]
        L.ref_model_infer.argtypes = [C.c_void_p, C.c_void_p, C.c_size_t, C.c_void_p, C.POINTER(C.c_size_t)]
        L.ref_cached_step.argtypes = [C.POINTER(_Cfg), C.c_void_p, C.c_size_t, C.c_void_p, C.c_size_t,
                                      C.c_uint32, C.c_uint32, C.c_void_p, C.POINTER(C.c_size_t), C.c_void_p,
                                      C.POINTER(C.c_size_t)]
        L.ref_infer.argtypes = [C.POINTER(_Cfg), C.c_void_p, C.c_size_t, C.c_void_p, C.c_size_t, C.c_void_p,
                                C.POINTER(C.c_size_t)]

    # ---- sizes -------------------------------------------------------
    def weight_words(self, shape) -> int:
        return int(self.lib.ref_weight_words(C.byref(_cfg(shape))))

    def cache_words_per_position(self, shape) -> int:
        return int(self.lib.ref_cache_words_per_position(C.byref(_cfg(shape))))

    # ---- primitives --------------------------------------------------
    def layernorm(self, x, g, b):
        x, g, b = (np.ascontiguousarray(v, np.float32) for v in (x, g, b))
        y = np.empty_like(x)
        self.lib.ref_layernorm(x, g, b, x.size, y)
        return y

    def gelu(self, x: float) -> float:
        return float(self.lib.ref_gelu(C.c_float(x)))

    def argmax(self, x):
        x = np.ascontiguousarray(x, np.float32)
        idx = C.c_uint32()
        st = self.lib.ref_argmax(x, x.size, C.byref(idx))
        return STATUS[st], int(idx.value)

    def group_scale(self, x) -> float:
        x = np.ascontiguousarray(x, np.float32)
        return float(self.lib.ref_group_scale(x, x.size))

    def quantize(self, x, s: float):
        x = np.ascontiguousarray(x, np.float32)
        q = np.empty(x.size, np.int8)
        self.lib.ref_quantize(x, x.size, C.c_float(s), q)
        return q

    def quantize_groups(self, x):
        x = np.ascontiguousarray(x, np.float32)
        q = np.empty(x.size, np.int8)
        s = np.empty(x.size // 64, np.float32)
        self.lib.ref_quantize_groups(x, x.size, q, s)
        return q, s

    def quantize_row(self, x):
        """One scale for the whole vector (the rejected per-activation-row
        design of the quantized GPT-2 abstract): (codes, scale per group slot)."""
        x = np.ascontiguousarray(x, np.float32)
        q = np.empty(x.size, np.int8)
        s = np.empty(x.size // 64, np.float32)
        self.lib.ref_quantize_row(x, x.size, q, s)
        return q, s

    def q8_group_dots(self, xq, wq):
        xq = np.ascontiguousarray(xq, np.int8)
        wq = np.ascontiguousarray(wq, np.int8)
        acc = np.empty(xq.size // 64, np.int32)
        self.lib.ref_q8_group_dots(xq, wq, xq.size, acc)
        return acc

    def linear_f32(self, x, w_in_out, b=None):
        x = np.ascontiguousarray(x, np.float32)
        w = np.ascontiguousarray(w_in_out, np.float32)
        n_in, n_out = w.shape
        y = np.empty(n_out, np.float32)
        bb = None if b is None else np.ascontiguousarray(b, np.float32)
        self.lib.ref_linear_f32(x, w, None if bb is None else bb.ctypes.data, n_in, n_out, y)
        return y

    def linear_q8(self, x, wq_out_in, ws, b=None, per_row_x=False):
        x = np.ascontiguousarray(x, np.float32)
        wq = np.ascontiguousarray(wq_out_in, np.int8)
        ws = np.ascontiguousarray(ws, np.float32)
        n_out, n_in = wq.shape
        y = np.empty(n_out, np.float32)
        bb = None if b is None else np.ascontiguousarray(b, np.float32)
        f = self.lib.ref_linear_q8_rowx if per_row_x else self.lib.ref_linear_q8
        f(x, wq, ws, None if bb is None else bb.ctypes.data, n_in, n_out, y)
        return y

    def attention_head(self, q, keys, values):
        """keys/values: [n_src][dh] float32.  Returns (out[dh], weights[n_src])."""
        q = np.ascontiguousarray(q, np.float32)
        k = np.ascontiguousarray(keys, np.float32)
        v = np.ascontiguousarray(values, np.float32)
        n, dh = k.shape
        out = np.empty(dh, np.float32)
        w = np.empty(n, np.float32)
        self.lib.ref_attention_head(q, k.ctypes.data, v.ctypes.data, n, dh, dh, out, w.ctypes.data)
        return out, w

    # ---- byte-level entries (binary32) -------------------------------
    def cached_step(self, shape, weights, cache, token, position):
        """Returns (status, logits, cache_out); outputs are empty on failure."""
        w = np.ascontiguousarray(weights)
        c = np.ascontiguousarray(cache)
        row = self.cache_words_per_position(shape)
        logits = np.empty(shape.vocab, np.float32)
        cout = np.empty(c.nbytes // 4 + row, np.float32)
        ll, cl = C.c_size_t(), C.c_size_t()
        st = self.lib.ref_cached_step(C.byref(_cfg(shape)), w.ctypes.data, w.nbytes, c.ctypes.data, c.nbytes,
                                      token & 0xFFFFFFFF, position & 0xFFFFFFFF, logits.ctypes.data,
                                      C.byref(ll), cout.ctypes.data, C.byref(cl))
        return STATUS[st], logits[:ll.value], cout[:cl.value // 4]

    def infer(self, shape, weights, tokens_bytes):
        w = np.ascontiguousarray(weights)
        t = np.frombuffer(bytes(tokens_bytes), np.uint8).copy()
        logits = np.empty(shape.vocab, np.float32)
        ll = C.c_size_t()
        st = self.lib.ref_infer(C.byref(_cfg(shape)), w.ctypes.data, w.nbytes,
                                t.ctypes.data if t.size else None, t.size, logits.ctypes.data, C.byref(ll))
        return STATUS[st], logits[:ll.value]

    def model(self, shape, weights, quant: int = 0) -> "OracleModel":
        return OracleModel(self, shape, weights, quant)


def round_f16(shape, weights) -> np.ndarray:
    """The half-precision weight option (gpt2.s page, half-precision weight
    paragraph, read as: the weight matrices are stored in binary16 and widened
    to binary32 for the arithmetic): a copy of the packed checkpoint whose
    tied embedding and 48 block matrices are rounded to the nearest binary16
    value (ties to even, numpy's IEEE conversion); wpe, the LayerNorm
    parameters and the biases keep their binary32 values.  The model computed
    on this checkpoint in binary32 is the binary16-weight model."""
    d, f, V = shape.d_model, shape.d_ff, shape.vocab
    w = np.array(weights, dtype=np.float32, copy=True)

    def rnd(o, n):
        w[o:o + n] = w[o:o + n].astype(np.float16).astype(np.float32)

    rnd(0, V * d)  # wte
    o = V * d + shape.n_pos * d
    for _ in range(shape.n_layer):
        o += 2 * d  # ln_1
        rnd(o, d * 3 * d)
        o += d * 3 * d + 3 * d
        rnd(o, d * d)
        o += d * d + d + 2 * d  # w_o, b_o, ln_2
        rnd(o, d * f)
        o += d * f + f
        rnd(o, f * d)
        o += f * d + d
    assert o + 2 * d == w.size
    return w


class OracleModel:
    """A parsed oracle model: quant=0 binary32, quant=1 int8 group-64,
    quant=2 binary16 weights (binary32 arithmetic on round_f16's checkpoint),
    quant=3 int8 with one weight scale per output row, quant=4 int8 with
    per-row weight scales and one scale per projection input."""

    def __init__(self, o: Oracle, shape, weights, quant: int):
        self.o, self.shape, self.quant = o, shape, quant
        w = np.ascontiguousarray(weights)
        if quant == 2:
            w, quant = round_f16(shape, w), 0
        st = C.c_int()
        self._cfg = _cfg(shape)
        self.h = o.lib.ref_model_create(C.byref(self._cfg), w.ctypes.data, w.nbytes, quant, C.byref(st))
        if not self.h:
            raise ValueError(f"oracle model_create: {STATUS[st.value]}")
        self.row = o.cache_words_per_position(shape)

    def close(self):
        if self.h:
            self.o.lib.ref_model_free(self.h)
            self.h = None

    def __del__(self):
        self.close()

    def cached_step(self, cache, token, position, trace=False):
        """Returns (status, logits, cache_out[, trace[n_layer][d]])."""
        c = np.ascontiguousarray(cache, np.float32)
        logits = np.empty(self.shape.vocab, np.float32)
        cout = np.empty(c.size + self.row, np.float32)
        tr = np.empty((self.shape.n_layer, self.shape.d_model), np.float32) if trace else None
        ll, cl = C.c_size_t(), C.c_size_t()
        st = self.o.lib.ref_model_cached_step(self.h, c.ctypes.data, c.nbytes, token & 0xFFFFFFFF,
                                              position & 0xFFFFFFFF, logits.ctypes.data, C.byref(ll),
                                              cout.ctypes.data, C.byref(cl),
                                              None if tr is None else tr.ctypes.data)
        out = (STATUS[st], logits[:ll.value], cout[:cl.value // 4])
        return out + (tr,) if trace else out

    def infer(self, tokens):
        t = np.ascontiguousarray(tokens, np.uint32)
        logits = np.empty(self.shape.vocab, np.float32)
        ll = C.c_size_t()
        st = self.o.lib.ref_model_infer(self.h, t.ctypes.data if t.size else None, t.nbytes,
                                        logits.ctypes.data, C.byref(ll))
        return STATUS[st], logits[:ll.value]

    def q8_matrix(self, index: int):
        """int8 copy of matrix ``index`` (4*layer + {qkv,o,fc,p}, 4*n_layer = wte):
        returns (q[out][in], s[out][in/64])."""
        s = self.shape
        d, F, L = s.d_model, s.d_ff, s.n_layer
        if index == 4 * L:
            n_in, n_out = d, s.vocab
        else:
            n_in, n_out = [(d, 3 * d), (d, d), (d, F), (F, d)][index % 4]
        q = np.empty((n_out, n_in), np.int8)
        sc = np.empty((n_out, n_in // 64), np.float32)
        st = self.o.lib.ref_model_get_q8(self.h, index, q, sc)
        if st != 0:
            raise ValueError(STATUS[st])
        return q, sc

    def session(self, tokens_in, n_steps, p0=0, cache=None):
        """Runs positions p0..p0+n_steps-1: token tokens_in[s] when given
        (>= 0), else the previous step's greedy choice.  Returns
        (logits[n_steps][vocab], chosen[n_steps], cache)."""
        cache = np.zeros(0, np.float32) if cache is None else cache
        logits = np.empty((n_steps, self.shape.vocab), np.float32)
        chosen = np.empty(n_steps, np.int64)
        prev = None
        for s in range(n_steps):
            tok = int(tokens_in[s]) if s < len(tokens_in) and tokens_in[s] >= 0 else prev
            st, lg, cache = self.cached_step(cache, tok, p0 + s)
            if st != "ok":
                raise RuntimeError(st)
            logits[s] = lg
            ast, prev = self.o.argmax(lg)
            chosen[s] = prev
        return logits, chosen, cache
