"""The tensor-core prefill (gpt2_session_prefill, and gpt2_infer through it):
the full-prefix forward pass of a prompt (LeanExe GPT-2 README, infer
paragraph) against the oracle's infer, plus the KV cache it leaves, which
must equal the cache the oracle's cachedSteps build over the same tokens
(the pages' cached-versus-full agreement), within the binary32 logit
tolerance.  Every expected value comes from the oracle on seeded inputs."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

from gpu_util import (GREEDY, LOGIT_TOL, dev_tokens, disagreements_are_near_ties,  # noqa: E402
                      oracle_teacher_forced, run)
from stream_decode_gb300 import synth  # noqa: E402

# 192 wide, 3 heads of 64, 256 positions: two 128-row tiles for n > 128.
MID = synth.Shape(2, 192, 3, 384, 512, 256, 256)


@pytest.fixture(scope="module")
def g():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from stream_decode_gb300 import gpt2
    return gpt2


def _prefill(g, model, toks):
    """Returns (status, logits, cache, greedy choice) of one prefill."""
    sess = g.Session(model)
    V = model.shape.vocab
    lg = torch.full((V,), float("nan"), dtype=torch.float32, device="cuda")
    nxt = torch.full((1,), -7, dtype=torch.int32, device="cuda")
    st = sess.prefill(dev_tokens(toks), len(toks), lg, nxt)
    if st == "ok":
        st = sess.sync()
    out = (st, lg.cpu().numpy(), sess.read_cache() if st == "ok" else None, int(nxt.item()) & 0xFFFFFFFF)
    assert sess.position == (len(toks) if st == "ok" else sess.position)
    sess.close()
    return out


def _check_against_oracle(g, oracle, shape, w, toks):
    om = oracle.model(shape, w)
    ref_logits, ref_ch, ref_cache = oracle_teacher_forced(om, toks)
    ost, olg = om.infer(np.asarray(toks, np.uint32))
    om.close()
    assert ost == "ok"
    # the oracle's own cached-versus-full identity
    assert np.array_equal(olg, ref_logits[-1])
    model = g.Model(shape, w)
    st, lg, cache, nxt = _prefill(g, model, toks)
    model.close()
    assert st == "ok", st
    assert np.abs(lg - olg).max() <= LOGIT_TOL, np.abs(lg - olg).max()
    assert cache.size == ref_cache.size
    assert np.abs(cache - ref_cache).max() <= LOGIT_TOL
    top2 = np.sort(olg)[-2:]
    assert nxt == int(np.argmax(olg)) or top2[1] - top2[0] <= LOGIT_TOL


@pytest.mark.parametrize("variant", ["plain", "rich"])
def test_prefill_tiny_every_length(g, oracle, variant):
    shape = synth.GPT2_TINY
    w = synth.checkpoint(shape, synth.SEED_TINY, variant)
    toks = [int(t) for t in synth.tokens(shape.vocab, 16)]
    for n in range(1, 17):
        _check_against_oracle(g, oracle, shape, w, toks[:n])


@pytest.mark.parametrize("n", [129, 200])
def test_prefill_two_row_tiles(g, oracle, n):
    w = synth.checkpoint(MID, 0x5EED0192, "rich")
    toks = [int(t) for t in synth.tokens(MID.vocab, n, seed=7)]
    _check_against_oracle(g, oracle, MID, w, toks)


def test_prefill_124m_128_tokens(g, oracle, w124m):
    """The 128-token prefill of the benchmark's prompt shape at full size."""
    s = synth.GPT2_124M
    toks = [int(t) for t in synth.tokens(s.vocab, 128, seed=11)]
    om = oracle.model(s, w124m)
    # the oracle's infer is its cachedSteps over the prefix (bit-identical
    # logits, checked on the tiny model above); the steps also give the cache
    ref_logits, _, ref_cache = oracle_teacher_forced(om, toks)
    om.close()
    olg = ref_logits[-1]
    model = g.Model(s, w124m)
    st, lg, cache, _ = _prefill(g, model, toks)
    model.close()
    assert st == "ok", st
    assert np.abs(lg - olg).max() <= LOGIT_TOL, np.abs(lg - olg).max()
    assert np.abs(cache - ref_cache).max() <= LOGIT_TOL


def test_prefill_then_decode_continues(g, oracle, tiny_rich):
    """Prefill of an 8-token prompt, then greedy cachedSteps on the device
    from the prefill's choice: the oracle's greedy session over the same
    prompt fixes every logit."""
    shape = synth.GPT2_TINY
    toks = [int(t) for t in synth.tokens(shape.vocab, 8)]
    om = oracle.model(shape, tiny_rich)
    ref_logits, ref_ch, _ = om.session(toks + [GREEDY] * 8, 16)
    om.close()
    model = g.Model(shape, tiny_rich)
    sess = g.Session(model)
    assert sess.prefill(dev_tokens(toks), 8) == "ok"
    logits, ch = run(sess, [GREEDY] * 8, 8)
    assert np.abs(logits - ref_logits[8:]).max() <= LOGIT_TOL
    assert disagreements_are_near_ties(ref_logits[8:], ch, LOGIT_TOL)
    sess.close()
    model.close()


def test_prefill_rejects_bad_arguments(g, tiny_plain):
    shape = synth.GPT2_TINY
    model = g.Model(shape, tiny_plain)
    sess = g.Session(model)
    t = dev_tokens([1, 2, 3])
    assert sess.prefill(t, 0) == "tokens_len"
    assert sess.prefill(dev_tokens([1] * 17), 17) == "tokens_len"
    assert sess.prefill(t, 3) == "ok" and sess.sync() == "ok"
    assert sess.prefill(t, 3) == "position"  # only from an empty session
    sess.close()
    q8 = g.Model(shape, tiny_plain, quant=g.INT8_G64)
    s8 = g.Session(q8)
    assert s8.prefill(t, 3) == "config"
    s8.close()
    q8.close()
    # an out-of-range token id is reported by the next sync
    sess = g.Session(model)
    assert sess.prefill(dev_tokens([1, shape.vocab, 2]), 3) == "ok"
    assert sess.sync() == "token"
    sess.close()
    model.close()
