"""The C ABI library loads and exports every symbol include/gpt2.h declares,
and its host-side size helpers agree with the pages (CPU only: no compute)."""
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from stream_decode_gb300 import build
    if not os.path.exists(build.LIB):
        build.build()
    from stream_decode_gb300 import gpt2
    return gpt2


def declared_functions():
    with open(os.path.join(ROOT, "include", "gpt2.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gpt2_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("gpt2_infer", "gpt2_cached_step", "gpt2_model_create", "gpt2_session_run",
                 "gpt2_session_step", "gpt2_session_step_host"):
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in declared_functions() if not hasattr(lib.lib, n)]
    assert not missing, missing


def test_size_helpers_match_pages(lib):
    from stream_decode_gb300 import synth
    assert lib.weight_words(synth.GPT2_124M) == 124439808
    assert lib.cache_words_per_position(synth.GPT2_124M) == 12 * 1536
    assert lib.weight_words(synth.GPT2_TINY) == synth.weight_words(synth.GPT2_TINY)


def test_status_names(lib):
    assert lib.lib.gpt2_status_name(0) == b"ok"
    assert lib.lib.gpt2_status_name(9) == b"timeout"


def test_validation_needs_no_gpu(lib, oracle):
    """Byte-level validation returns before any device work, with empty outputs,
    in the order weights_len, token, position, cache_len (README cachedStep
    paragraph) -- runnable without a GPU."""
    import numpy as np
    from stream_decode_gb300 import synth
    s = synth.GPT2_TINY
    w = synth.checkpoint(s, synth.SEED_TINY)
    row = lib.cache_words_per_position(s)
    cases = [
        (w[:-1], np.zeros(3 * row, np.float32), 1, 3),
        (w, np.zeros(3 * row, np.float32), s.vocab, 3),
        (w, np.zeros(3 * row, np.float32), 0xFFFFFFFF, 3),
        (w, np.zeros(s.max_pos * row, np.float32), 1, s.max_pos),
        (w, np.zeros(3 * row - 1, np.float32), 1, 3),
        (w[:-1], np.zeros(3 * row - 1, np.float32), s.vocab, s.max_pos),
        (w, np.zeros(3 * row - 1, np.float32), s.vocab, s.max_pos),
        (w, np.zeros(3 * row, np.float32), 1, s.max_pos),
    ]
    for ww, cc, t, p in cases:
        st, lg, co = lib.cached_step(s, ww, cc, t, p)
        ost, olg, oco = oracle.cached_step(s, ww, cc, t, p)
        assert st == ost and lg.size == 0 and co.size == 0, (st, ost)
    toks = synth.tokens(s.vocab, 4)
    for tb in (b"", toks.astype("<u4").tobytes()[:-2], np.zeros(s.max_pos + 1, "<u4").tobytes(),
               np.array([3, s.vocab], "<u4").tobytes(), np.array([s.vocab], "<u4").tobytes() + b"\x00"):
        st, lg = lib.infer(s, w, tb)
        ost, _ = oracle.infer(s, w, tb)
        assert st == ost and lg.size == 0
    st, lg = lib.infer(s, w[:-1], toks.astype("<u4").tobytes())
    assert st == "weights_len" and lg.size == 0
