"""ctypes binding to libgpt2gb.so (include/gpt2.h).  Argument marshalling
only: every step of the computation runs in the library's CUDA kernels.
Device buffers are passed as torch CUDA tensors (their data pointers); torch
is used for device memory and streams, nothing else.

Importing this module loads the library and raises if it has not been built
(``python -m stream_decode_gb300.build``); there is no fallback.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_build", "libgpt2gb.so")

if not os.path.exists(_LIB_PATH):
    raise ImportError(f"libgpt2gb.so is not built ({_LIB_PATH}); run python -m stream_decode_gb300.build")

lib = C.CDLL(_LIB_PATH)

GREEDY = 0xFFFFFFFF
F32, INT8_G64, F16, INT8_ROW, INT8_ROW_ACT = 0, 1, 2, 3, 4
STATUS = {0: "ok", 1: "weights_len", 2: "token", 3: "position", 4: "cache_len", 5: "tokens_len",
          6: "nonfinite", 7: "config", 8: "nomem", 9: "timeout", 10: "cuda", 11: "arg", 12: "scratch"}


class Config(C.Structure):
    _fields_ = [(n, C.c_uint32) for n in ("n_layer", "d_model", "n_head", "d_ff", "vocab", "n_pos", "max_pos")]


def config(shape) -> Config:
    return Config(*shape.as_tuple())


_vp, _sz, _u32, _i32 = C.c_void_p, C.c_size_t, C.c_uint32, C.c_int
_cfgp = C.POINTER(Config)
_szp = C.POINTER(C.c_size_t)
_SIGS = {
    "gpt2_weight_words": ([_cfgp], _sz),
    "gpt2_cache_words_per_position": ([_cfgp], _sz),
    "gpt2_infer": ([_cfgp, _vp, _sz, _vp, _sz, _vp, _szp], _i32),
    "gpt2_cached_step": ([_cfgp, _vp, _sz, _vp, _sz, _u32, _u32, _vp, _szp, _vp, _szp], _i32),
    "gpt2_model_create": ([_cfgp, _vp, _sz, _i32, _i32, C.POINTER(_vp)], _i32),
    "gpt2_model_destroy": ([_vp], None),
    "gpt2_model_read_q8": ([_vp, _i32, _vp, _vp], _i32),
    "gpt2_model_step_kernel": ([_vp, C.POINTER(_u32), C.POINTER(_u32)], _i32),
    "gpt2_session_create": ([_vp, C.POINTER(_vp)], _i32),
    "gpt2_session_destroy": ([_vp], None),
    "gpt2_session_position": ([_vp], _u32),
    "gpt2_session_load_cache": ([_vp, _vp, _sz], _i32),
    "gpt2_session_read_cache": ([_vp, _vp, _sz, _szp], _i32),
    "gpt2_session_rewind": ([_vp, _u32], _i32),
    "gpt2_session_run": ([_vp, _vp, _u32, _vp, _sz, _vp, _vp], _i32),
    "gpt2_session_prefill": ([_vp, _vp, _u32, _vp, _vp, _vp], _i32),
    "gpt2_session_step": ([_vp, _u32, _vp, _vp, _vp], _i32),
    "gpt2_session_step_host": ([_vp, _u32, _vp, _vp], _i32),
    "gpt2_session_run_host": ([_vp, _vp, _u32, _vp, _vp], _i32),
    "gpt2_session_sync": ([_vp], _i32),
    "gpt2_session_set_trace": ([_vp, _vp], _i32),
    "gpt2_session_inject_stall": ([_vp, _u32, C.c_uint64], _i32),
    "gpt2_session_set_timing": ([_vp, _vp], _i32),
    "gpt2_debug_project": ([_vp, _i32, _vp, _vp, _vp], _i32),
    "gpt2_debug_argmax": ([_vp, _u32, _vp, _vp, _vp], _i32),
    "gpt2_cached_step_noalloc": ([_vp, _vp, _u32, _u32, _vp, _vp, _vp], _i32),
    "gpt2_batch_create": ([_vp, _u32, C.POINTER(_vp)], _i32),
    "gpt2_batch_destroy": ([_vp], None),
    "gpt2_batch_size": ([_vp], _u32),
    "gpt2_batch_position": ([_vp, _u32], _u32),
    "gpt2_batch_load_cache": ([_vp, _u32, _vp, _sz], _i32),
    "gpt2_batch_read_cache": ([_vp, _u32, _vp, _sz, _szp], _i32),
    "gpt2_batch_run": ([_vp, _vp, _u32, _vp, _sz, _vp, _vp], _i32),
    "gpt2_batch_sync": ([_vp], _i32),
    "gpt2_batch_rewind": ([_vp, _u32, _vp], _i32),
    "gpt2_status_name": ([_i32], C.c_char_p),
    "gpt2_last_cuda_error": ([C.POINTER(C.c_char_p)], _i32),
}
for _name, (_args, _res) in _SIGS.items():
    _f = getattr(lib, _name)
    _f.argtypes = _args
    _f.restype = _res


def _ptr(t) -> int | None:
    """Device pointer of a torch CUDA tensor (None passes NULL)."""
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else stream


def weight_words(shape) -> int:
    return int(lib.gpt2_weight_words(C.byref(config(shape))))


def cache_words_per_position(shape) -> int:
    return int(lib.gpt2_cache_words_per_position(C.byref(config(shape))))


def infer(shape, weights: np.ndarray, tokens_bytes: bytes):
    """README ``infer`` on host buffers: returns (status, logits)."""
    w = np.ascontiguousarray(weights)
    t = np.frombuffer(bytes(tokens_bytes), np.uint8).copy()
    logits = np.empty(shape.vocab, np.float32)
    n = C.c_size_t()
    st = lib.gpt2_infer(C.byref(config(shape)), w.ctypes.data, w.nbytes, t.ctypes.data if t.size else None,
                        t.size, logits.ctypes.data, C.byref(n))
    return STATUS[st], logits[:n.value]


def cached_step(shape, weights: np.ndarray, cache: np.ndarray, token: int, position: int):
    """README ``cachedStep`` on host buffers: returns (status, logits, cache_out)."""
    w = np.ascontiguousarray(weights)
    c = np.ascontiguousarray(cache)
    row = cache_words_per_position(shape)
    logits = np.empty(shape.vocab, np.float32)
    cout = np.empty(c.nbytes // 4 + row, np.float32)
    nl, nc = C.c_size_t(), C.c_size_t()
    st = lib.gpt2_cached_step(C.byref(config(shape)), w.ctypes.data, w.nbytes, c.ctypes.data if c.size else None,
                              c.nbytes, token & 0xFFFFFFFF, position & 0xFFFFFFFF, logits.ctypes.data,
                              C.byref(nl), cout.ctypes.data, C.byref(nc))
    return STATUS[st], logits[:nl.value], cout[:nc.value // 4]


class GPT2Error(RuntimeError):
    def __init__(self, where: str, status: int):
        super().__init__(f"{where}: {STATUS.get(status, status)}")
        self.status = STATUS.get(status, str(status))


def _check(where: str, st: int):
    if st != 0:
        raise GPT2Error(where, st)


class Model:
    """Device-resident model (gpt2_model_create)."""

    def __init__(self, shape, weights: np.ndarray, quant: int = F32, grid_ctas: int = 0):
        self.shape, self.quant = shape, quant
        w = np.ascontiguousarray(weights)
        h = C.c_void_p()
        self._cfg = config(shape)
        _check("gpt2_model_create", lib.gpt2_model_create(C.byref(self._cfg), w.ctypes.data, w.nbytes, quant,
                                                          grid_ctas, C.byref(h)))
        self.h = h

    def read_q8(self, index: int):
        s = self.shape
        d, F, L = s.d_model, s.d_ff, s.n_layer
        n_in, n_out = (d, s.vocab) if index == 4 * L else [(d, 3 * d), (d, d), (d, F), (F, d)][index % 4]
        q = np.empty((n_out, n_in), np.int8)
        sc = np.empty((n_out, n_in // 64), np.float32)
        _check("gpt2_model_read_q8", lib.gpt2_model_read_q8(self.h, index, q.ctypes.data, sc.ctypes.data))
        return q, sc

    @property
    def step_kernel(self):
        """(kind, clusters, cluster_size): kind "cluster" or "phase"
        (gpt2_model_step_kernel); for "phase" clusters is 0 and cluster_size
        the CTA count."""
        nc, cs = C.c_uint32(), C.c_uint32()
        k = lib.gpt2_model_step_kernel(self.h, C.byref(nc), C.byref(cs))
        return ("cluster" if k == 1 else "phase"), nc.value, cs.value

    def debug_project(self, index: int, x, y, stream=None) -> str:
        """Test hook: projection `index` of x (CUDA tensor) into y (CUDA tensor)."""
        return STATUS[lib.gpt2_debug_project(self.h, index, _ptr(x), _ptr(y), _stream(stream))]

    def cached_step_noalloc(self, cache, position: int, token: int, logits=None, next_token=None,
                            stream=None) -> str:
        """One step that allocates nothing (gpt2_cached_step_noalloc): `cache`
        is a caller-owned CUDA tensor in the cachedStep layout with room for
        position + 1 positions; logits / next_token are CUDA tensors or None."""
        return STATUS[lib.gpt2_cached_step_noalloc(self.h, _ptr(cache), position, token, _ptr(logits),
                                                   _ptr(next_token), _stream(stream))]

    def close(self):
        if getattr(self, "h", None):
            lib.gpt2_model_destroy(self.h)
            self.h = None

    def __del__(self):
        self.close()


class Session:
    """Device KV cache plus step state (gpt2_session_*)."""

    def __init__(self, model: Model):
        self.model = model
        h = C.c_void_p()
        _check("gpt2_session_create", lib.gpt2_session_create(model.h, C.byref(h)))
        self.h = h

    @property
    def position(self) -> int:
        return int(lib.gpt2_session_position(self.h))

    def load_cache(self, cache: np.ndarray) -> str:
        c = np.ascontiguousarray(cache, np.float32)
        return STATUS[lib.gpt2_session_load_cache(self.h, c.ctypes.data if c.size else None, c.nbytes)]

    def rewind(self, position: int) -> str:
        return STATUS[lib.gpt2_session_rewind(self.h, position)]

    def read_cache(self) -> np.ndarray:
        n = self.position * cache_words_per_position(self.model.shape)
        out = np.empty(n, np.float32)
        got = C.c_size_t()
        _check("gpt2_session_read_cache", lib.gpt2_session_read_cache(self.h, out.ctypes.data if n else None,
                                                                      out.nbytes, C.byref(got)))
        return out[:got.value // 4]

    def run(self, tokens_in, n_steps: int, logits=None, stride: int = 0, tokens_out=None, stream=None) -> str:
        return STATUS[lib.gpt2_session_run(self.h, _ptr(tokens_in), n_steps, _ptr(logits), stride,
                                           _ptr(tokens_out), _stream(stream))]

    def prefill(self, tokens, n: int, logits=None, next_token=None, stream=None) -> str:
        """Tensor-core prefill of n device token ids from an empty session (gpt2_session_prefill)."""
        return STATUS[lib.gpt2_session_prefill(self.h, _ptr(tokens), n, _ptr(logits), _ptr(next_token),
                                               _stream(stream))]

    def step(self, token: int, logits=None, next_token=None, stream=None) -> str:
        return STATUS[lib.gpt2_session_step(self.h, token & 0xFFFFFFFF, _ptr(logits), _ptr(next_token),
                                            _stream(stream))]

    def step_host(self, token: int, logits_host=None, next_host=None) -> str:
        """logits_host: numpy float32[vocab] or a pinned CPU torch tensor."""
        lp = None if logits_host is None else (logits_host.data_ptr() if hasattr(logits_host, "data_ptr")
                                               else logits_host.ctypes.data)
        npt = None if next_host is None else (next_host.data_ptr() if hasattr(next_host, "data_ptr")
                                              else next_host.ctypes.data)
        return STATUS[lib.gpt2_session_step_host(self.h, token & 0xFFFFFFFF, lp, npt)]

    def run_host(self, tokens_host, n_steps: int, logits_host=None, tokens_out_host=None) -> str:
        """Host buffers (numpy arrays or pinned CPU torch tensors): tokens_host
        uint32/int32[n_steps]; logits_host float32[n_steps][vocab]; tokens_out_host
        uint32/int32[n_steps]."""
        def hp(t):
            if t is None:
                return None
            return t.data_ptr() if hasattr(t, "data_ptr") else t.ctypes.data
        return STATUS[lib.gpt2_session_run_host(self.h, hp(tokens_host), n_steps, hp(logits_host),
                                                hp(tokens_out_host))]

    def sync(self) -> str:
        return STATUS[lib.gpt2_session_sync(self.h)]

    def set_trace(self, trace) -> str:
        return STATUS[lib.gpt2_session_set_trace(self.h, _ptr(trace))]

    def set_timing(self, stamps) -> str:
        """Profiling: next run records (phase, CTA, 8) stamps (see gpt2_session_set_timing) into a CUDA int64 tensor."""
        return STATUS[lib.gpt2_session_set_timing(self.h, _ptr(stamps))]

    def inject_stall(self, phase: int, wait_limit_ns: int) -> str:
        return STATUS[lib.gpt2_session_inject_stall(self.h, phase, wait_limit_ns)]

    def close(self):
        if getattr(self, "h", None):
            lib.gpt2_session_destroy(self.h)
            self.h = None

    def __del__(self):
        self.close()


class Batch:
    """B independent decode sessions of one binary32 model stepped together
    (gpt2_batch_*)."""

    def __init__(self, model: Model, n_sessions: int):
        self.model = model
        h = C.c_void_p()
        _check("gpt2_batch_create", lib.gpt2_batch_create(model.h, n_sessions, C.byref(h)))
        self.h = h
        self.size = int(lib.gpt2_batch_size(h))

    def position(self, index: int) -> int:
        return int(lib.gpt2_batch_position(self.h, index))

    def load_cache(self, index: int, cache: np.ndarray) -> str:
        c = np.ascontiguousarray(cache, np.float32)
        return STATUS[lib.gpt2_batch_load_cache(self.h, index, c.ctypes.data if c.size else None, c.nbytes)]

    def read_cache(self, index: int) -> np.ndarray:
        n = self.position(index) * cache_words_per_position(self.model.shape)
        out = np.empty(n, np.float32)
        got = C.c_size_t()
        _check("gpt2_batch_read_cache", lib.gpt2_batch_read_cache(self.h, index, out.ctypes.data if n else None,
                                                                  out.nbytes, C.byref(got)))
        return out[:got.value // 4]

    def run(self, tokens_in, n_steps: int, logits=None, stride: int = 0, tokens_out=None, stream=None) -> str:
        """tokens_in: CUDA int32/uint32 tensor [n_steps][B]; logits: CUDA
        float tensor (step s, session b at s * stride + b * vocab)."""
        return STATUS[lib.gpt2_batch_run(self.h, _ptr(tokens_in), n_steps, _ptr(logits), stride, _ptr(tokens_out),
                                         _stream(stream))]

    def rewind(self, position: int, stream=None) -> str:
        return STATUS[lib.gpt2_batch_rewind(self.h, position, _stream(stream))]

    def sync(self) -> str:
        return STATUS[lib.gpt2_batch_sync(self.h)]

    def close(self):
        if getattr(self, "h", None):
            lib.gpt2_batch_destroy(self.h)
            self.h = None

    def __del__(self):
        self.close()


def debug_argmax(values, index, nonfinite, stream=None) -> str:
    """Test hook: the step kernel's greedy choice over a CUDA float tensor."""
    return STATUS[lib.gpt2_debug_argmax(_ptr(values), values.numel(), _ptr(index), _ptr(nonfinite),
                                        _stream(stream))]


def last_cuda_error() -> tuple[int, str]:
    """(code, name) of the CUDA error behind the last 'cuda' / 'nomem' status."""
    name = C.c_char_p()
    code = lib.gpt2_last_cuda_error(C.byref(name))
    return code, (name.value or b"").decode()


def trace_words(shape) -> int:
    """Size of a trace buffer (gpt2_session_set_trace)."""
    return shape.n_layer * (8 * shape.d_model + shape.d_ff) + 2 * shape.d_model
