"""GPU parity: the CUDA step kernel through the C ABI against the CPU oracle.

Tolerances: binary32 logits max |delta| <= 2e-3 and greedy agreement >= 99%
(teacher-forced on the GPU's own choices); cache indexing, argmax on
identical logits, int8 codes/scales and int8 projections on identical inputs
are compared bit for bit.
"""
import hashlib

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

from gpu_util import AGREE_MIN, GREEDY, LOGIT_TOL, dev_tokens, greedy_agreement, run  # noqa: E402
from stream_decode_gb300 import synth  # noqa: E402

import oracle_pins as P  # noqa: E402


@pytest.fixture(scope="module")
def g():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from stream_decode_gb300 import gpt2
    return gpt2


def _session_case(g, oracle, shape, seed, variant, quant, grid, n_prompt=8):
    w = synth.checkpoint(shape, seed, variant)
    n = shape.max_pos
    toks = synth.tokens(shape.vocab, n_prompt)
    model = g.Model(shape, w, quant=quant, grid_ctas=grid)
    sess = g.Session(model)
    logits, ch = run(sess, list(toks) + [GREEDY] * (n - n_prompt), n)
    seq = np.concatenate([toks, ch[n_prompt - 1:n - 1]])
    om = oracle.model(shape, w, quant=quant)
    ref, ref_ch, ref_cache = om.session(list(seq), n)
    cache = sess.read_cache()
    return logits, ch, ref, ref_ch, cache, ref_cache


@pytest.mark.parametrize("grid", [0, 1, 3, 7, 37])
def test_tiny_f32_session(g, oracle, grid):
    logits, ch, ref, ref_ch, cache, ref_cache = _session_case(g, oracle, synth.GPT2_TINY, synth.SEED_TINY, "rich",
                                                              0, grid)
    assert np.abs(logits - ref).max() <= LOGIT_TOL
    assert np.array_equal(ch[:len(ref_ch)], np.argmax(logits, 1)), "argmax of the GPU's own logits"
    assert greedy_agreement(ref, ch) >= AGREE_MIN
    assert cache.size == ref_cache.size and np.abs(cache - ref_cache).max() <= LOGIT_TOL


@pytest.mark.parametrize("grid", [0, 5])
def test_small_shape_f32_session(g, oracle, grid):
    logits, ch, ref, _, cache, ref_cache = _session_case(g, oracle, P.SMALL, P.SEED_SMALL, "rich", 0, grid)
    assert np.abs(logits - ref).max() <= LOGIT_TOL
    assert greedy_agreement(ref, ch) >= AGREE_MIN
    assert np.abs(cache - ref_cache).max() <= LOGIT_TOL


def test_argmax_bit_exact_on_gpu_logits(g, oracle):
    """The device's greedy choice equals the oracle's argmax rule applied to
    the very logits the device produced (ties to the lowest index)."""
    shape = synth.GPT2_TINY
    w = synth.checkpoint(shape, synth.SEED_TINY, "plain")
    sess = g.Session(g.Model(shape, w))
    logits, ch = run(sess, list(synth.tokens(shape.vocab, 16, seed=3)), 16)
    for s in range(16):
        st, idx = oracle.argmax(logits[s])
        assert st == "ok" and idx == ch[s]


def test_cache_indexing_bit_exact(g, oracle):
    """Index-tagged cache: the returned cache keeps the incoming words bit for
    bit and appends one position at word (p*L + l)*2d + offset."""
    shape = synth.GPT2_TINY
    w = synth.checkpoint(shape, synth.SEED_TINY, "plain")
    row = g.cache_words_per_position(shape)
    for p in (0, 1, 5, shape.max_pos - 1):
        tagged = (np.arange(p * row, dtype=np.float32) * 1e-4).astype(np.float32)
        st, lg, cout = g.cached_step(shape, w, tagged, 3, p)
        ost, olg, ocout = oracle.cached_step(shape, w, tagged, 3, p)
        assert st == ost == "ok"
        assert cout.size == (p + 1) * row
        assert np.array_equal(cout[:p * row].view(np.uint32), tagged.view(np.uint32))
        assert np.abs(cout[p * row:] - ocout[p * row:]).max() <= 1e-4
        assert np.abs(lg - olg).max() <= LOGIT_TOL


def test_byte_level_infer_matches_cached_chain(g, oracle):
    """README: tests compare cached and full-prefix execution."""
    shape = synth.GPT2_TINY
    w = synth.checkpoint(shape, synth.SEED_TINY, "rich")
    toks = synth.tokens(shape.vocab, shape.max_pos, seed=5)
    cache = np.zeros(0, np.float32)
    for p in range(shape.max_pos):
        st, lg, cache = g.cached_step(shape, w, cache, int(toks[p]), p)
        assert st == "ok"
        if p in (0, 3, shape.max_pos - 1):
            sti, li = g.infer(shape, w, toks[:p + 1].astype("<u4").tobytes())
            assert sti == "ok" and np.abs(li - lg).max() <= LOGIT_TOL
            ost, ol = oracle.infer(shape, w, toks[:p + 1].astype("<u4").tobytes())
            assert np.abs(li - ol).max() <= LOGIT_TOL


def test_byte_level_validation_matches_oracle(g, oracle):
    P.check_validation(g)  # the pins' validation table, run against the GPU library


def test_step_apis_agree(g, oracle):
    shape = synth.GPT2_TINY
    w = synth.checkpoint(shape, synth.SEED_TINY, "rich")
    toks = synth.tokens(shape.vocab, 6, seed=8)
    model = g.Model(shape, w)
    a, b = g.Session(model), g.Session(model)
    la, _ = run(a, list(toks), 6)
    d_logits = torch.empty(shape.vocab, dtype=torch.float32, device="cuda")
    d_next = torch.empty(1, dtype=torch.int32, device="cuda")
    host = np.empty(shape.vocab, np.float32)
    nxt = np.zeros(1, np.uint32)
    for p, t in enumerate(toks):
        if p % 2:
            assert b.step(int(t), d_logits, d_next) == "ok"
            assert b.sync() == "ok"
            lb = d_logits.cpu().numpy()
        else:
            assert b.step_host(int(t), host, nxt) == "ok"
            lb = host.copy()
        assert np.array_equal(lb.view(np.uint32), la[p].view(np.uint32)), "same kernel, same bits"
    assert b.position == 6
    assert b.step(shape.vocab, d_logits, d_next) == "token"


def test_greedy_token_without_history_is_an_error(g):
    shape = synth.GPT2_TINY
    sess = g.Session(g.Model(shape, synth.checkpoint(shape, synth.SEED_TINY)))
    tin = dev_tokens([GREEDY, GREEDY])
    assert sess.run(tin, 2, None, 0, None) == "ok"
    assert sess.sync() == "token"


def test_nonfinite_logits_reported(g):
    shape = synth.GPT2_TINY
    w = synth.checkpoint(shape, synth.SEED_TINY)
    lay = synth.layout(shape)
    w[lay["lnf_g"][0] + 5] = np.nan
    sess = g.Session(g.Model(shape, w))
    tout = torch.zeros(3, dtype=torch.int32, device="cuda")
    assert sess.run(dev_tokens([1, 2, 3]), 3, None, 0, tout) == "ok"
    assert sess.sync() == "nonfinite"
    assert (int(tout.cpu().numpy()[0]) & 0xFFFFFFFF) == 0xFFFFFFFF


def test_stalled_phase_times_out_and_session_recovers(g):
    """A CTA that never publishes a phase makes the others' bounded waits
    expire: the run ends with 'timeout' (no hang, no fault) and the session is
    usable again after the status is read."""
    shape = synth.GPT2_TINY
    w = synth.checkpoint(shape, synth.SEED_TINY)
    sess = g.Session(g.Model(shape, w, grid_ctas=8))
    assert sess.inject_stall(3, 50_000_000) == "ok"
    assert sess.run(dev_tokens([1, 2]), 2, None, 0, None) == "ok"
    assert sess.sync() == "timeout"
    sess2 = g.Session(sess.model)
    logits, _ = run(sess2, [1, 2], 2)
    assert np.isfinite(logits).all()


def test_run_to_run_determinism(g):
    shape = synth.GPT2_TINY
    w = synth.checkpoint(shape, synth.SEED_TINY, "rich")
    model = g.Model(shape, w)
    digests = []
    for _ in range(2):
        logits, _ = run(g.Session(model), list(synth.tokens(shape.vocab, 8)) + [GREEDY] * 8, 16)
        digests.append(hashlib.sha256(logits.tobytes()).hexdigest())
    assert digests[0] == digests[1]


# ------------------------------------------------------------------ int8
@pytest.mark.parametrize("shape,seed", [(synth.GPT2_TINY, synth.SEED_TINY), (P.SMALL, P.SEED_SMALL)],
                         ids=["tiny", "small"])
def test_int8_weight_codes_bit_exact(g, oracle, shape, seed):
    w = synth.checkpoint(shape, seed, "rich")
    model = g.Model(shape, w, quant=g.INT8_G64)
    om = oracle.model(shape, w, quant=1)
    for idx in range(4 * shape.n_layer + 1):
        q, s = model.read_q8(idx)
        oq, os_ = om.q8_matrix(idx)
        assert np.array_equal(q, oq), idx
        assert np.array_equal(s.view(np.uint32), os_.view(np.uint32)), idx


def _trace(g, shape, model, tokens):
    sess = g.Session(model)
    tr = torch.zeros(g.trace_words(shape), dtype=torch.float32, device="cuda")
    sess.set_trace(tr)
    logits, _ = run(sess, tokens, 1)
    return tr.cpu().numpy(), logits[0]


@pytest.mark.parametrize("shape,seed", [(synth.GPT2_TINY, synth.SEED_TINY), (P.SMALL, P.SEED_SMALL)],
                         ids=["tiny", "small"])
def test_int8_projections_bit_exact_on_identical_inputs(g, oracle, shape, seed):
    """Feed the oracle's int8 projection the exact input vectors the device
    formed (from the device trace): quantized codes, int32 group sums and the
    fixed rescale order make the outputs identical bit for bit."""
    w = synth.checkpoint(shape, seed, "rich")
    model = g.Model(shape, w, quant=g.INT8_G64)
    om = oracle.model(shape, w, quant=1)
    tr, logits = _trace(g, shape, model, [7])
    d, F, L = shape.d_model, shape.d_ff, shape.n_layer
    per = 8 * d + F
    lay = synth.layout(shape)
    bits = lambda a: np.asarray(a, np.float32).view(np.uint32)
    for l in range(L):
        base = l * per
        x_in, xn1 = tr[base:base + d], tr[base + d:base + 2 * d]
        qkv, o = tr[base + 2 * d:base + 5 * d], tr[base + 5 * d:base + 6 * d]
        x_mid, xn2 = tr[base + 6 * d:base + 7 * d], tr[base + 7 * d:base + 8 * d]
        u = tr[base + 8 * d:base + 8 * d + F]
        b = lambda name: w[lay[f"h{l}.{name}"][0]:lay[f"h{l}.{name}"][0] + lay[f"h{l}.{name}"][1]]
        q, s = om.q8_matrix(4 * l + 0)
        assert np.array_equal(bits(oracle.linear_q8(xn1, q, s, b("b_qkv"))), bits(qkv)), f"qkv layer {l}"
        q, s = om.q8_matrix(4 * l + 1)
        y = oracle.linear_q8(o, q, s, b("b_o"))
        assert np.array_equal(bits(x_in + y), bits(x_mid)), f"out-proj layer {l}"
        q, s = om.q8_matrix(4 * l + 3)
        y = oracle.linear_q8(u, q, s, b("b_p"))
        x_next = tr[(l + 1) * per:(l + 1) * per + d] if l + 1 < L else tr[L * per:L * per + d]
        assert np.array_equal(bits(x_mid + y), bits(x_next)), f"mlp-proj layer {l}"
    xnf = tr[L * per + d:L * per + 2 * d]
    q, s = om.q8_matrix(4 * L)
    assert np.array_equal(bits(oracle.linear_q8(xnf, q, s)), bits(logits)), "vocab projection"


@pytest.mark.parametrize("shape,seed", [(synth.GPT2_TINY, synth.SEED_TINY), (P.SMALL, P.SEED_SMALL)],
                         ids=["tiny", "small"])
def test_int8_session(g, oracle, shape, seed):
    logits, ch, ref, _, cache, ref_cache = _session_case(g, oracle, shape, seed, "rich", 1, 0)
    assert np.abs(logits - ref).max() <= LOGIT_TOL
    assert greedy_agreement(ref, ch) >= AGREE_MIN
    assert np.abs(cache - ref_cache).max() <= LOGIT_TOL


def test_f32_traced_stages_close_to_oracle(g, oracle):
    """Stage-by-stage binary32 check on the 192-wide shape from the trace."""
    shape = P.SMALL
    w = synth.checkpoint(shape, P.SEED_SMALL, "rich")
    tr, logits = _trace(g, shape, g.Model(shape, w), [9])
    st, ol, _, otr = oracle.model(shape, w).cached_step(np.zeros(0, np.float32), 9, 0, trace=True)
    d, F = shape.d_model, shape.d_ff
    per = 8 * d + F
    for l in range(shape.n_layer):
        nxt = tr[(l + 1) * per:(l + 1) * per + d] if l + 1 < shape.n_layer else tr[shape.n_layer * per:
                                                                                    shape.n_layer * per + d]
        assert np.abs(nxt - otr[l]).max() < 1e-4, l
    assert np.abs(logits - ol).max() <= LOGIT_TOL
