"""GPU parity at the full GPT-2 124M shapes, in the launch configuration the
benchmark times (one persistent launch per decode run, one CTA per SM)."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

from gpu_util import AGREE_MIN, GREEDY, LOGIT_TOL, run  # noqa: E402
from stream_decode_gb300 import synth  # noqa: E402


@pytest.fixture(scope="module")
def g():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from stream_decode_gb300 import gpt2
    return gpt2


def _decode_run(g, oracle, w, quant):
    """16 uniform random prompt tokens through cachedStep at positions 0..15,
    then 112 greedy steps up to position 127, all in one launch; the oracle
    recomputes every step on the GPU's token sequence."""
    s = synth.GPT2_124M
    toks = synth.tokens(s.vocab, 16)
    model = g.Model(s, w, quant=quant)
    sess = g.Session(model)
    logits, ch = run(sess, list(toks) + [GREEDY] * 112, 128)
    seq = np.concatenate([toks, ch[15:127]])
    om = oracle.model(s, w, quant=quant)
    ref, ref_ch, ref_cache = om.session(list(seq), 128)
    cache = sess.read_cache()
    om.close()
    return logits, ch, ref, cache, ref_cache


def test_124m_f32_decode_128_positions(g, oracle, w124m):
    logits, ch, ref, cache, ref_cache = _decode_run(g, oracle, w124m, 0)
    err = np.abs(logits - ref).max(axis=1)
    assert err.max() <= LOGIT_TOL, err.max()
    assert np.mean(np.argmax(ref, 1) == ch) >= AGREE_MIN
    assert cache.size == 128 * 12 * 1536 and np.abs(cache - ref_cache).max() <= LOGIT_TOL


def test_124m_int8_decode_128_positions(g, oracle, w124m):
    logits, ch, ref, cache, ref_cache = _decode_run(g, oracle, w124m, 1)
    err = np.abs(logits - ref).max(axis=1)
    assert err.max() <= LOGIT_TOL, err.max()
    assert np.mean(np.argmax(ref, 1) == ch) >= AGREE_MIN


def test_124m_long_context_positions(g, oracle, w124m):
    """Cache of 1023 prior positions from 1023 uniform random tokens (built by
    one GPU launch), then single steps at p = 128, 512, 1023 compared with the
    oracle given the same cache prefix."""
    s = synth.GPT2_124M_LONG
    toks = synth.tokens(s.vocab, 1024, seed=1234)
    model = g.Model(s, w124m)
    sess = g.Session(model)
    run(sess, list(toks[:1023]), 1023, want_logits=False)
    full = sess.read_cache()
    row = g.cache_words_per_position(s)
    om = oracle.model(s, w124m)
    for p in (128, 512, 1023):
        prefix = full[:p * row]
        st, ol, ocache = om.cached_step(prefix, int(toks[p]), p)
        assert st == "ok"
        s2 = g.Session(model)
        assert s2.load_cache(prefix) == "ok"
        lg, ch = run(s2, [int(toks[p])], 1)
        assert np.abs(lg[0] - ol).max() <= LOGIT_TOL, p
        assert ch[0] == np.argmax(ol) or abs(np.sort(ol)[-1] - np.sort(ol)[-2]) < LOGIT_TOL
        newrow = s2.read_cache()[p * row:]
        assert np.abs(newrow - ocache[p * row:]).max() <= LOGIT_TOL
    om.close()
