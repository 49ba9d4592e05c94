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

from gpu_util import (AGREE_MIN, GREEDY, LOGIT_TOL, dev_tokens, disagreements_are_near_ties,  # noqa: E402
                      greedy_agreement, int8_tolerance, oracle_greedy, run)
from stream_decode_gb300 import synth  # noqa: E402

import oracle_pins as P  # noqa: E402
from oracle import round_f16  # noqa: E402


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


def _session_case(g, oracle, shape, seed, variant, quant, grid, n_prompt=8):
    """The oracle runs its own greedy session from a seeded prompt; the GPU is
    fed that token sequence (one launch), and separately runs greedily on the
    device from the same prompt."""
    w = synth.checkpoint(shape, seed, variant)
    n = shape.max_pos
    toks = synth.tokens(shape.vocab, n_prompt)
    om = oracle.model(shape, w, quant=quant)
    seq, ref, ref_ch, ref_cache = oracle_greedy(om, toks, n)
    model = g.Model(shape, w, quant=quant, grid_ctas=grid)
    sess = g.Session(model)
    logits, ch = run(sess, list(seq), n)
    cache = sess.read_cache()
    greedy_sess = g.Session(model)
    _, greedy_ch = run(greedy_sess, list(toks) + [GREEDY] * (n - n_prompt), n, want_logits=False)
    return logits, ch, ref, ref_ch, cache, ref_cache, greedy_ch, seq


def _first_divergence(a, b):
    d = np.nonzero(np.asarray(a) != np.asarray(b))[0]
    return int(d[0]) if d.size else len(a)


def _check_f32_session(out):
    logits, ch, ref, ref_ch, cache, ref_cache, greedy_ch, _ = out
    assert np.abs(logits - ref).max() <= LOGIT_TOL
    assert greedy_agreement(ref, ch) >= AGREE_MIN
    assert disagreements_are_near_ties(ref, ch, LOGIT_TOL)
    assert cache.size == ref_cache.size and np.abs(cache - ref_cache).max() <= LOGIT_TOL
    # greedy on the device follows the oracle's choices up to the first near tie
    k = _first_divergence(greedy_ch, ref_ch)
    if k < len(ref_ch):
        top2 = np.sort(ref[k])[-2:]
        assert top2[1] - top2[0] <= LOGIT_TOL, f"greedy run left the oracle's path at step {k}"


@pytest.mark.parametrize("grid", [0, 1, 3, 7, 37])
def test_tiny_f32_session(g, oracle, grid, kernel):
    _check_f32_session(_session_case(g, oracle, synth.GPT2_TINY, synth.SEED_TINY, "rich", 0, grid))


@pytest.mark.parametrize("grid", [0, 5])
def test_small_shape_f32_session(g, oracle, grid, kernel):
    _check_f32_session(_session_case(g, oracle, P.SMALL, P.SEED_SMALL, "rich", 0, grid))


@pytest.mark.parametrize("shape,seed", [(synth.GPT2_TINY, synth.SEED_TINY), (P.SMALL, P.SEED_SMALL)],
                         ids=["tiny", "small"])
def test_offset_residual_f32_session(g, oracle, shape, seed, kernel):
    """LayerNorm on a residual stream with channels near 100 and a common
    offset that drifts from layer to layer (synthetic variant
    offset_residual): the README applies LayerNorm to whatever the weights
    make of the stream, and a variance formed as E[x^2] - mean^2 would lose
    most of its bits here."""
    _check_f32_session(_session_case(g, oracle, shape, seed, "offset_residual", 0, 0))


def test_argmax_bit_exact(g, oracle):
    """The device's greedy-choice routine against the oracle's on identical
    seeded values: random rows, planted ties (lowest index wins), -0.0 vs
    +0.0, and NaN / +-Inf (non-finite status)."""
    cases = []
    for k in range(6):
        cases.append(synth.uniform_f32(100 + k, 50257, -4.0, 4.0))
    tie = synth.uniform_f32(7, 5000, -1.0, 1.0)
    tie[[4321, 17, 999]] = 2.0
    cases.append(tie)
    z = np.full(300, -1.0, np.float32)
    z[40], z[7] = 0.0, -0.0
    cases.append(z)
    for bad in (np.nan, np.inf, -np.inf):
        v = synth.uniform_f32(9, 777)
        v[500] = bad
        cases.append(v)
    cases.append(np.array([3.5], np.float32))
    for v in cases:
        dv = torch.tensor(v, device="cuda")
        idx = torch.zeros(1, dtype=torch.int32, device="cuda")
        nf = torch.zeros(1, dtype=torch.int32, device="cuda")
        assert g.debug_argmax(dv, idx, nf) == "ok"
        torch.cuda.synchronize()
        st, oidx = oracle.argmax(v)
        assert (int(idx.item()) & 0xFFFFFFFF) == oidx
        assert bool(nf.item()) == (st == "nonfinite")


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


@pytest.mark.parametrize("shape,quant", [(synth.GPT2_TINY, 0), (synth.GPT2_TINY, 2), (P.SMALL, 0), (synth.GPT2_TINY, 1),
                                         (synth.GPT2_TINY, 3)],
                         ids=["tiny-f32", "tiny-f16", "small-f32", "tiny-int8", "tiny-int8row"])
def test_step_kernel_in_use(g, shape, quant, kernel):
    """binary32 and binary16 models step on the kernel GPT2_STEP_KERNEL
    names (so the session tests run on each); int8 models on the per-phase
    kernel."""
    model = g.Model(shape, synth.checkpoint(shape, synth.SEED_TINY if shape is synth.GPT2_TINY else P.SEED_SMALL),
                    quant=quant)
    k, nc, cs = model.step_kernel
    kind = kernel if quant in (0, 2) else "phase"
    assert k == kind
    if kind == "cluster":
        assert nc >= 1 and cs >= 1 and shape.d_model % cs == 0
    model.close()


def test_step_apis_agree(g, oracle, kernel):
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


def test_run_host_matches_device_run(g, kernel):
    """gpt2_session_run_host (host token ids in, every step's logits and
    choices back in host memory) gives the device run's bits, with greedy
    feedback, and checks its host tokens before any launch."""
    shape = synth.GPT2_TINY
    w = synth.checkpoint(shape, synth.SEED_TINY, "rich")
    model = g.Model(shape, w)
    toks = [int(t) for t in synth.tokens(shape.vocab, 4, seed=9)] + [GREEDY] * 8
    a, b = g.Session(model), g.Session(model)
    la, ca = run(a, toks, 12)
    hl = np.full((12, shape.vocab), np.nan, np.float32)
    ho = np.zeros(12, np.uint32)
    assert b.run_host(np.array(toks, np.int64).astype(np.uint32), 12, hl, ho) == "ok"
    assert np.array_equal(hl.view(np.uint32), la.view(np.uint32)), "same kernel, same bits"
    assert np.array_equal(ho.astype(np.int64), np.asarray(ca, np.int64) & 0xFFFFFFFF)
    assert b.position == 12
    c = g.Session(model)
    assert c.run_host(np.array([1, shape.vocab], np.uint32), 2) == "token" and c.position == 0
    assert c.run_host(np.zeros(shape.max_pos + 1, np.uint32), shape.max_pos + 1) == "position"
    assert c.run_host(np.array([3], np.uint32), 1) == "ok" and c.position == 1  # outputs optional
    for sess in (a, b, c):
        sess.close()
    model.close()


def test_greedy_token_without_history_is_an_error(g, kernel):
    shape = synth.GPT2_TINY
    sess = g.Session(g.Model(shape, synth.checkpoint(shape, synth.SEED_TINY)))
    tin = dev_tokens([GREEDY, GREEDY])
    assert sess.run(tin, 2, None, 0, None) == "ok"
    assert sess.sync() == "token"


def test_nonfinite_logits_reported(g, kernel):
    shape = synth.GPT2_TINY
    w = synth.checkpoint(shape, synth.SEED_TINY)
    lay = synth.layout(shape)
    w[lay["lnf_g"][0] + 5] = np.nan
    sess = g.Session(g.Model(shape, w))
    tout = torch.zeros(3, dtype=torch.int32, device="cuda")
    assert sess.run(dev_tokens([1, 2, 3]), 3, None, 0, tout) == "ok"
    assert sess.sync() == "nonfinite"
    assert (int(tout.cpu().numpy()[0]) & 0xFFFFFFFF) == 0xFFFFFFFF


def test_stalled_phase_times_out_and_session_recovers(g, kernel):
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


@pytest.mark.parametrize("shape,seed", [(synth.GPT2_TINY, synth.SEED_TINY), (P.SMALL, P.SEED_SMALL)],
                         ids=["tiny", "small"])
def test_rewind_and_resume_are_bit_identical(g, shape, seed, kernel):
    """The session recurrence (README cachedStep paragraph: each returned
    cache is passed to the next position): rewinding to a position and
    stepping again, or taking the cache at a position into a new session
    and continuing there, gives the uninterrupted run's bits."""
    w = synth.checkpoint(shape, seed, "rich")
    model = g.Model(shape, w)
    n, half = shape.max_pos, shape.max_pos // 2
    toks = [int(t) for t in synth.tokens(shape.vocab, n, seed=21)]
    full, full_ch = run(g.Session(model), toks, n)
    # rewind: the second half again on the same session
    a = g.Session(model)
    run(a, toks, n)
    assert a.rewind(half) == "ok" and a.position == half
    again, again_ch = run(a, toks[half:], n - half)
    assert np.array_equal(again.view(np.uint32), full[half:].view(np.uint32))
    assert np.array_equal(again_ch, full_ch[half:])
    # snapshot at half: the cache into a fresh session, then continue
    b = g.Session(model)
    run(b, toks[:half], half)
    snap = b.read_cache()
    c = g.Session(model)
    assert c.load_cache(snap) == "ok" and c.position == half
    cont, cont_ch = run(c, toks[half:], n - half)
    assert np.array_equal(cont.view(np.uint32), full[half:].view(np.uint32))
    assert np.array_equal(cont_ch, full_ch[half:])
    assert np.array_equal(c.read_cache().view(np.uint32), a.read_cache().view(np.uint32))
    for s_ in (a, b, c):
        s_.close()
    model.close()


def test_writes_stay_inside_their_buffers(g, kernel):
    """Canaries: a caller-owned cache filled with a pattern keeps it past
    the positions stepped; logits written with a stride above vocab leave
    the gaps between steps untouched; the choices buffer past the run is
    untouched."""
    shape = synth.GPT2_TINY
    w = synth.checkpoint(shape, synth.SEED_TINY, "rich")
    model = g.Model(shape, w)
    V, row, n = shape.vocab, g.cache_words_per_position(shape), 5
    canary = np.uint32(0x7FC0DEAD)  # a NaN payload no step can produce
    cache = torch.tensor(np.full(shape.max_pos * row, canary, np.uint32).view(np.float32), device="cuda")
    out = torch.empty(V, dtype=torch.float32, device="cuda")
    for p, t in enumerate(synth.tokens(V, n, seed=3)):
        assert model.cached_step_noalloc(cache, p, int(t), out) == "ok"
    torch.cuda.synchronize()
    c = cache.cpu().numpy().view(np.uint32)
    assert (c[n * row:] == canary).all(), "a step wrote past its position's cache row"
    assert not (c[:n * row] == canary).any()
    stride = V + 37
    lg = torch.tensor(np.full(n * stride + 11, canary, np.uint32).view(np.float32), device="cuda")
    tout = torch.full((n + 9,), -12345, dtype=torch.int32, device="cuda")
    sess = g.Session(model)
    assert sess.run(dev_tokens(list(synth.tokens(V, n, seed=4))), n, lg, stride, tout) == "ok"
    assert sess.sync() == "ok"
    l = lg.cpu().numpy().view(np.uint32)
    for s_ in range(n):
        assert not (l[s_ * stride:s_ * stride + V] == canary).any()
        assert (l[s_ * stride + V:(s_ + 1) * stride] == canary).all(), f"logits gap after step {s_}"
    assert (l[n * stride:] == canary).all()
    assert (tout.cpu().numpy()[n:] == -12345).all()
    sess.close()
    model.close()


def test_run_to_run_determinism(g, kernel):
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
@pytest.mark.parametrize("quant", [1, 3], ids=["group64", "per_row"])
def test_int8_weight_codes_bit_exact(g, oracle, shape, seed, quant):
    w = synth.checkpoint(shape, seed, "rich")
    model = g.Model(shape, w, quant=quant)
    om = oracle.model(shape, w, quant=quant)
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


def _matrix_bias(shape, w, idx):
    L = shape.n_layer
    if idx == 4 * L:
        return None
    lay = synth.layout(shape)
    name = f"h{idx // 4}." + ["b_qkv", "b_o", "b_fc", "b_p"][idx % 4]
    o, n = lay[name]
    return w[o:o + n]


def check_projections(g, oracle, shape, w, quant, indices, seed=31):
    """Every projection of the model on a seeded input vector: int8 models
    bit for bit against the oracle's int8 projection (codes, int32 group
    sums, fixed-order rescale, bias); binary32 models within 1e-5, and
    binary16-weight models within 1e-5 of the binary32 projection with the
    oracle's rounded weights.  quant 4 quantizes the input with one scale
    for the whole vector."""
    model = g.Model(shape, w, quant=quant)
    q8 = quant in (1, 3, 4)
    om = oracle.model(shape, w, quant=quant) if q8 else None
    p = None
    for idx in indices:
        n_in = shape.d_ff if (idx % 4 == 3 and idx != 4 * shape.n_layer) else shape.d_model
        x = (2.0 * synth.normals(seed + idx, 0, n_in)).astype(np.float32)
        x[::97] *= 3.0
        dx = torch.tensor(x, device="cuda")
        q, s = (om.q8_matrix(idx) if q8 else (None, None))
        n_out = q.shape[0] if q8 else None
        if not q8:
            if p is None:
                import torch_gpt2
                p = torch_gpt2.parse(shape, round_f16(shape, w) if quant == 2 else w)
            if idx == 4 * shape.n_layer:
                wm = p["wte"].numpy().T
            else:
                wm = p["blocks"][idx // 4][["w_qkv", "w_o", "w_fc", "w_p"][idx % 4]].numpy()
            n_out = wm.shape[1]
        dy = torch.full((n_out,), float("nan"), device="cuda")
        assert model.debug_project(idx, dx, dy) == "ok"
        torch.cuda.synchronize()
        y = dy.cpu().numpy()
        b = _matrix_bias(shape, w, idx)
        if q8:
            ref = oracle.linear_q8(x, q, s, b, per_row_x=quant == 4)
            assert np.array_equal(y.view(np.uint32), ref.view(np.uint32)), f"matrix {idx}"
        else:
            ref = oracle.linear_f32(x, wm.astype(np.float32), b)
            assert np.abs(y - ref).max() <= 1e-5 * max(1.0, np.abs(ref).max()), f"matrix {idx}"
    model.close()
    if om is not None:
        om.close()


@pytest.mark.parametrize("shape,seed", [(synth.GPT2_TINY, synth.SEED_TINY), (P.SMALL, P.SEED_SMALL)],
                         ids=["tiny", "small"])
@pytest.mark.parametrize("quant", [0, 1, 2, 3, 4], ids=["f32", "int8", "f16", "int8_row", "int8_row_act"])
def test_projections_on_identical_inputs(g, oracle, shape, seed, quant):
    w = synth.checkpoint(shape, seed, "rich")
    check_projections(g, oracle, shape, w, quant, range(4 * shape.n_layer + 1))


def test_int8_activation_codes_near_ties(g, oracle):
    """The int8 activation quantizer on inputs whose quotients x / s sit
    at, or a few ulp either side of, the half-integers where nearest-even
    rounding changes its answer (the quantization rule of the quantized
    GPT-2 abstract): every code must equal the oracle's, so the int8
    projection of such a vector is bit-identical to the oracle's."""
    shape = P.SMALL
    w = synth.checkpoint(shape, P.SEED_SMALL, "rich")
    model = g.Model(shape, w, quant=1)
    om = oracle.model(shape, w, quant=1)
    rng = np.random.default_rng(2024)
    for idx in (0, 3):
        n_in = shape.d_ff if idx % 4 == 3 else shape.d_model
        x = np.empty(n_in, np.float32)
        for g0 in range(0, n_in, 64):
            m = np.float32(rng.uniform(0.25, 4.0))
            sc = np.float32(m / np.float32(127.0))
            k = rng.integers(-126, 126, 64).astype(np.float32)
            v = ((k + np.float32(0.5)) * sc).astype(np.float32)
            steps = rng.integers(-3, 4, 64)
            for i in range(64):
                for _ in range(abs(int(steps[i]))):
                    v[i] = np.nextafter(v[i], np.float32(np.inf) if steps[i] > 0 else np.float32(-np.inf))
            v[rng.integers(0, 64)] = m if rng.random() < 0.5 else -m  # the group's largest magnitude
            x[g0:g0 + 64] = v
        q, s_ = om.q8_matrix(idx)
        dx = torch.tensor(x, device="cuda")
        dy = torch.full((q.shape[0],), float("nan"), device="cuda")
        assert model.debug_project(idx, dx, dy) == "ok"
        torch.cuda.synchronize()
        ref = oracle.linear_q8(x, q, s_, _matrix_bias(shape, w, idx))
        assert np.array_equal(dy.cpu().numpy().view(np.uint32), ref.view(np.uint32)), f"matrix {idx}"
    model.close()
    om.close()


@pytest.mark.parametrize("shape,seed", [(synth.GPT2_TINY, synth.SEED_TINY), (P.SMALL, P.SEED_SMALL)],
                         ids=["tiny", "small"])
@pytest.mark.parametrize("quant", [1, 3, 4], ids=["group64", "per_row", "per_row_act"])
def test_int8_session(g, oracle, shape, seed, quant):
    logits, ch, ref, ref_ch, cache, ref_cache, greedy_ch, seq = _session_case(g, oracle, shape, seed, "rich", quant,
                                                                               0)
    w = synth.checkpoint(shape, seed, "rich")
    ref_f32, _, _ = oracle.model(shape, w).session(list(seq), shape.max_pos)
    tol = int8_tolerance(ref, ref_f32)
    assert np.abs(logits - ref).max() <= tol
    assert disagreements_are_near_ties(ref, ch, tol)
    assert np.abs(cache - ref_cache).max() <= tol


def test_f32_traced_stages_close_to_oracle(g, oracle, kernel):
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


# ------------------------------------------------------------------ binary16 weights
@pytest.mark.parametrize("shape,seed,grid", [(synth.GPT2_TINY, synth.SEED_TINY, 0), (synth.GPT2_TINY, synth.SEED_TINY, 7),
                                             (P.SMALL, P.SEED_SMALL, 0)], ids=["tiny", "tiny-grid7", "small"])
def test_f16_session(g, oracle, shape, seed, grid, kernel):
    """Binary16 weight storage: the oracle's binary16-weight model (binary32
    arithmetic on the rounded checkpoint) is matched to the binary32 bar."""
    _check_f32_session(_session_case(g, oracle, shape, seed, "rich", 2, grid))
