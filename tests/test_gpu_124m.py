"""GPU parity at the full GPT-2 124M shapes, in the launch configuration the
benchmark times (one persistent launch per decode run, one CTA per SM).

The oracle runs first, on seeded inputs only; the GPU is then fed the same
inputs (the oracle's greedy token sequence, seeded synthetic caches)."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

from gpu_util import (AGREE_MIN, GREEDY, LOGIT_TOL, disagreements_are_near_ties,  # noqa: E402
                      greedy_agreement, int8_tolerance, oracle_greedy, run)
from stream_decode_gb300 import synth  # noqa: E402


@pytest.fixture(scope="module")
def g():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from stream_decode_gb300 import gpt2
    return gpt2


@pytest.fixture(params=["phase", "cluster"])
def kernel(request, monkeypatch):
    """Runs a binary32 / binary16 test on each step kernel (the variable is
    read when a model is created)."""
    monkeypatch.setenv("GPT2_STEP_KERNEL", request.param)
    return request.param


@pytest.fixture(scope="module")
def ref_f32(oracle, w124m):
    """The oracle's greedy session: 16 uniform random prompt tokens at
    positions 0..15, then 112 greedy steps up to position 127."""
    s = synth.GPT2_124M
    om = oracle.model(s, w124m)
    out = oracle_greedy(om, synth.tokens(s.vocab, 16), 128)
    om.close()
    return out


def test_124m_f32_decode_128_positions(g, w124m, ref_f32, kernel):
    s = synth.GPT2_124M
    seq, ref, ref_ch, ref_cache = ref_f32
    model = g.Model(s, w124m)
    logits, ch = run(g.Session(model), list(seq), 128)
    err = np.abs(logits - ref).max(axis=1)
    assert err.max() <= LOGIT_TOL, err.max()
    assert greedy_agreement(ref, ch) >= AGREE_MIN
    assert disagreements_are_near_ties(ref, ch, LOGIT_TOL)
    sess = g.Session(model)
    run(sess, list(seq), 128, want_logits=False)
    cache = sess.read_cache()
    assert cache.size == 128 * 12 * 1536 and np.abs(cache - ref_cache).max() <= LOGIT_TOL
    # device-side greedy feedback from the same prompt follows the oracle
    _, gch = run(g.Session(model), list(seq[:16]) + [GREEDY] * 112, 128, want_logits=False)
    d = np.nonzero(gch != ref_ch)[0]
    if d.size:
        top2 = np.sort(ref[d[0]])[-2:]
        assert top2[1] - top2[0] <= LOGIT_TOL, f"greedy run left the oracle's path at step {d[0]}"


@pytest.mark.parametrize("quant", [1, 3], ids=["group64", "per_row"])
def test_124m_int8_decode_128_positions(g, oracle, w124m, ref_f32, quant):
    s = synth.GPT2_124M
    om = oracle.model(s, w124m, quant=quant)
    seq, ref, ref_ch, _ = oracle_greedy(om, synth.tokens(s.vocab, 16), 128)
    om.close()
    of = oracle.model(s, w124m)
    ref_f32_same, _, _ = of.session(list(seq), 128)
    of.close()
    tol = int8_tolerance(ref, ref_f32_same)
    logits, ch = run(g.Session(g.Model(s, w124m, quant=quant)), list(seq), 128)
    err = np.abs(logits - ref).max(axis=1)
    assert err.max() <= tol, (err.max(), tol)
    assert disagreements_are_near_ties(ref, ch, tol)
    print(f"int8: max|gpu-oracle| {err.max():.4g}, tolerance {tol:.4g}, "
          f"greedy agreement {greedy_agreement(ref, ch):.3f}")


def test_124m_f16_decode_128_positions(g, oracle, w124m, kernel):
    """Binary16 weight storage at full size: against the oracle's
    binary16-weight model, to the binary32 bar."""
    s = synth.GPT2_124M
    om = oracle.model(s, w124m, quant=2)
    seq, ref, ref_ch, ref_cache = oracle_greedy(om, synth.tokens(s.vocab, 16), 128)
    om.close()
    model = g.Model(s, w124m, quant=g.F16)
    sess = g.Session(model)
    logits, ch = run(sess, list(seq), 128)
    err = np.abs(logits - ref).max(axis=1)
    assert err.max() <= LOGIT_TOL, err.max()
    assert greedy_agreement(ref, ch) >= AGREE_MIN
    assert disagreements_are_near_ties(ref, ch, LOGIT_TOL)
    cache = sess.read_cache()
    assert np.abs(cache - ref_cache).max() <= LOGIT_TOL


@pytest.mark.parametrize("quant", [0, 1, 2, 3, 4], ids=["f32", "int8", "f16", "int8_row", "int8_row_act"])
def test_124m_projections_on_identical_inputs(g, oracle, w124m, quant):
    from test_gpu_decode import check_projections
    L = 12
    check_projections(g, oracle, synth.GPT2_124M, w124m, quant, [0, 1, 2, 3, 4 * 5 + 2, 4 * 11 + 3, 4 * L])


@pytest.mark.parametrize("p", [128, 512, 1023])
def test_124m_long_context_positions(g, oracle, w124m, p, kernel):
    """A seeded synthetic cache of p prior positions (keys/values ~ N(0, 0.25),
    the magnitude N(0,0.02) weights give), then one step at position p with
    token = the p-th uniform random token, on both sides."""
    s = synth.GPT2_124M_LONG
    row = g.cache_words_per_position(s)
    cache = synth.cache(s, p, seed=4242 + p)
    tok = int(synth.tokens(s.vocab, 1024, seed=1234)[p])
    om = oracle.model(s, w124m)
    st, ol, ocache = om.cached_step(cache, tok, p)
    om.close()
    assert st == "ok"
    model = g.Model(s, w124m)
    sess = g.Session(model)
    assert sess.load_cache(cache) == "ok"
    lg, ch = run(sess, [tok], 1)
    assert np.abs(lg[0] - ol).max() <= LOGIT_TOL
    assert disagreements_are_near_ties(ol[None], ch, LOGIT_TOL)
    out = sess.read_cache()
    assert np.array_equal(out[:p * row].view(np.uint32), cache.view(np.uint32))
    assert np.abs(out[p * row:] - ocache[p * row:]).max() <= LOGIT_TOL


@pytest.fixture(scope="module")
def ref_long(oracle, w124m):
    """The long-context configuration as the workload defines it: 1024
    uniform random tokens fed through the oracle's own cached steps, so its
    cache of 1023 prior positions is the model's, not a synthetic one.
    Returns (tokens, logits at positions 128, 512 and 1023, final cache)."""
    s = synth.GPT2_124M_LONG
    toks = [int(t) for t in synth.tokens(s.vocab, 1024, seed=1234)]
    om = oracle.model(s, w124m)
    logits, _, cache = om.session(toks, 1024)
    om.close()
    return toks, {p: logits[p].copy() for p in (128, 512, 1023)}, cache


def test_124m_long_context_model_built_cache(g, w124m, ref_long, kernel):
    """GPU and oracle are fed the same 1024 tokens (one launch on the GPU):
    logits at positions 128, 512 and 1023 and every cache row agree."""
    s = synth.GPT2_124M_LONG
    toks, ref, ref_cache = ref_long
    model = g.Model(s, w124m)
    sess = g.Session(model)
    logits, ch = run(sess, toks, 1024)
    for p, ol in ref.items():
        assert np.abs(logits[p] - ol).max() <= LOGIT_TOL, p
        assert disagreements_are_near_ties(ol[None], ch[p:p + 1], LOGIT_TOL), p
    cache = sess.read_cache()
    assert cache.size == ref_cache.size and np.abs(cache - ref_cache).max() <= LOGIT_TOL
    sess.close()
    model.close()


def test_124m_offset_residual_decode(g, oracle, kernel):
    """GPT-2 124M on the offset_residual checkpoint (residual channels near
    100, a drifting common offset): 32 positions teacher-forced on the
    oracle's greedy sequence, to the binary32 bar."""
    s = synth.GPT2_124M
    w = synth.checkpoint(s, synth.SEED_124M, "offset_residual")
    om = oracle.model(s, w)
    seq, ref, ref_ch, ref_cache = oracle_greedy(om, synth.tokens(s.vocab, 8), 32)
    om.close()
    model = g.Model(s, w)
    sess = g.Session(model)
    logits, ch = run(sess, list(seq), 32)
    assert np.abs(logits - ref).max() <= LOGIT_TOL, np.abs(logits - ref).max()
    assert disagreements_are_near_ties(ref, ch, LOGIT_TOL)
    cache = sess.read_cache()
    assert np.abs(cache - ref_cache[:cache.size]).max() <= LOGIT_TOL
    sess.close()
    model.close()
