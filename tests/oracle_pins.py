"""Pins that tie the oracle to something other than itself.

Each ``check_*`` takes an ``Oracle`` and raises AssertionError on a
mismatch.  ``test_oracle.py`` runs them against the real oracle;
``test_oracle_mutants.py`` runs them against deliberately broken copies of
the oracle source and requires that every planted mistake trips at least one.

What pins what (sources by page title and paragraph):
* sizes -- numbers printed in the LeanExe GPT-2 README and the quantized-GPT-2
  abstract (``golden/page_identities.json``);
* the whole forward pass and the cache layout -- an independent float64
  full-prefix restatement from torch library primitives (``torch_gpt2.py``);
* cached vs full-prefix -- the README's statement that tests compare cached
  and full-prefix execution (exact here: same per-row code);
* LayerNorm, GELU, attention -- closed forms, invariants and library routines;
* zero blocks -- every block is the identity, so the logits reduce to one
  float64 matrix-vector product;
* argmax -- brute force with planted ties and non-finite values;
* int8 -- hand-worked quantizer vectors (``golden/int8_quantizer_cases.json``),
  int64 brute-force group sums, an integer-exact special case, and the
  quantization error bound against float64.
"""
from __future__ import annotations

import json
import os

import numpy as np
import torch
import torch.nn.functional as F

from stream_decode_gb300 import synth

import torch_gpt2

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")

# A shape with several int8 groups per row (d = 3 groups, F = 6 groups).
SMALL = synth.Shape(n_layer=2, d_model=192, n_head=3, d_ff=384, vocab=640, n_pos=16, max_pos=16)
SEED_SMALL = 0x5EED0192


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ------------------------------------------------------------------ sizes
def check_sizes(o):
    g = _golden("page_identities.json")
    s = synth.GPT2_124M
    assert o.weight_words(s) == g["checkpoint_words_124m"]["value"]
    assert o.weight_words(s) * 4 == g["checkpoint_bytes_124m"]["value"]
    assert o.cache_words_per_position(s) == g["cache_words_per_position"]["value"]
    assert o.cache_words_per_position(s) == s.n_layer * g["cache_row_words"]["value"]
    assert 128 * s.vocab == g["session_logits_128"]["value"]
    assert s.n_pos == g["stored_position_rows"]["value"]
    assert s.max_pos == g["accepted_positions"]["value"]
    # tiny: wte + wpe + 2 blocks + final LN, counted by hand
    assert o.weight_words(synth.GPT2_TINY) == 512 * 64 + 16 * 64 + 2 * 49984 + 128


# ----------------------------------------------------- whole forward pass
def check_forward_vs_torch(o, shape=synth.GPT2_TINY, seed=synth.SEED_TINY, variant="rich", n=16, tol=1e-5):
    w = synth.checkpoint(shape, seed, variant)
    m = o.model(shape, w)
    toks = synth.tokens(shape.vocab, n)
    logits, _, cache = m.session(list(toks), n)
    ref, K, V = torch_gpt2.forward(shape, w, toks)
    err = np.abs(logits - ref).max()
    assert err < tol, f"logits differ from float64 restatement by {err}"
    # cache layout: word (source*L + layer)*2d + offset, keys then values
    d, L = shape.d_model, shape.n_layer
    c = cache.reshape(n, L, 2, d)
    assert np.abs(c[:, :, 0, :].transpose(1, 0, 2) - K).max() < tol
    assert np.abs(c[:, :, 1, :].transpose(1, 0, 2) - V).max() < tol


def check_cached_equals_infer(o, shape=synth.GPT2_TINY, seed=synth.SEED_TINY):
    w = synth.checkpoint(shape, seed, "rich")
    m = o.model(shape, w)
    toks = synth.tokens(shape.vocab, shape.max_pos, seed=7)
    logits, _, _ = m.session(list(toks), shape.max_pos)
    for n in (1, 2, 5, shape.max_pos):
        st, li = o.infer(shape, w, toks[:n].astype("<u4").tobytes())
        assert st == "ok"
        assert np.array_equal(li.view(np.uint32), logits[n - 1].view(np.uint32)), f"prefix {n}"


def check_cache_prefix_kept(o, shape=synth.GPT2_TINY, seed=synth.SEED_TINY):
    """Index-tagged cache: word w holds float(w); the returned cache must be
    those words unchanged, followed by exactly one new position."""
    w = synth.checkpoint(shape, seed, "plain")
    row = o.cache_words_per_position(shape)
    p = 5
    tagged = (np.arange(p * row, dtype=np.float32) * 1e-4).astype(np.float32)
    st, logits, cout = o.cached_step(shape, w, tagged, 3, p)
    assert st == "ok" and cout.size == (p + 1) * row
    assert np.array_equal(cout[:p * row].view(np.uint32), tagged.view(np.uint32))
    # the new position's layer-0 keys/values depend only on the embedding, so
    # they equal the float64 restatement's layer-0 k/v for token 3 at position p
    toks = np.zeros(p + 1, np.int64)
    toks[p] = 3
    _, K, V = torch_gpt2.forward(shape, w, toks)
    new = cout[p * row:].reshape(shape.n_layer, 2, shape.d_model)
    assert np.abs(new[0, 0] - K[0, p]).max() < 1e-5
    assert np.abs(new[0, 1] - V[0, p]).max() < 1e-5


def check_zero_blocks(o, shape=synth.GPT2_TINY, seed=synth.SEED_TINY):
    """Zero block matrices and biases make every block the identity; the
    logits are then wte . LN_f(wte[t] + wpe[p])."""
    w = synth.checkpoint(shape, seed, "zero_blocks")
    m = o.model(shape, w)
    toks = synth.tokens(shape.vocab, 4, seed=11)
    logits, _, _ = m.session(list(toks), 4)
    p = torch_gpt2.parse(shape, w)
    for pos in range(4):
        x = p["wte"][int(toks[pos])] + p["wpe"][pos]
        xf = F.layer_norm(x, (shape.d_model,), p["lnf_g"], p["lnf_b"], eps=1e-5)
        ref = torch.mv(p["wte"], xf).numpy()
        assert np.abs(logits[pos] - ref).max() < 1e-5


# ------------------------------------------------------------- primitives
def check_layernorm(o):
    rng = np.random.default_rng(1)
    n = 768
    g = np.ones(n, np.float32)
    b = np.zeros(n, np.float32)
    c = np.full(n, 0.5, np.float32)
    bb = rng.standard_normal(n).astype(np.float32)
    assert np.array_equal(o.layernorm(c, g, bb), bb), "constant input must give the shift exactly"
    x = (3.0 + 2.0 * rng.standard_normal(n)).astype(np.float32)
    y = o.layernorm(x, g, b).astype(np.float64)
    assert abs(y.mean()) < 1e-5  # binary32 sums of 768 values near 3
    assert abs(y.var() - 4.0 / (4.0 + 1e-5)) < 1e-4
    gg = (1 + 0.1 * rng.standard_normal(n)).astype(np.float32)
    ref = F.layer_norm(torch.from_numpy(x.astype(np.float64)), (n,), torch.from_numpy(gg.astype(np.float64)),
                       torch.from_numpy(bb.astype(np.float64)), eps=1e-5).numpy()
    assert np.abs(o.layernorm(x, gg, bb) - ref).max() < 1e-5


def check_gelu(o):
    assert o.gelu(0.0) == 0.0
    assert o.gelu(10.0) == 10.0
    assert o.gelu(-10.0) == 0.0
    xs = np.linspace(-6, 6, 241)
    ref = F.gelu(torch.from_numpy(xs), approximate="tanh").numpy()
    got = np.array([o.gelu(float(np.float32(v))) for v in xs])
    ref32 = F.gelu(torch.from_numpy(xs.astype(np.float32).astype(np.float64)), approximate="tanh").numpy()
    assert np.abs(got - ref32).max() < 2e-6, np.abs(got - ref).max()


def check_attention(o):
    rng = np.random.default_rng(2)
    dh = 64
    for n in (1, 2, 7, 128):
        q = rng.standard_normal(dh).astype(np.float32)
        k = rng.standard_normal((n, dh)).astype(np.float32)
        v = rng.standard_normal((n, dh)).astype(np.float32)
        out, wts = o.attention_head(q, k, v)
        assert abs(float(wts.astype(np.float64).sum()) - 1.0) <= n * 2.0 ** -23 + 1e-7
        if n == 1:
            assert np.array_equal(out, v[0]), "one source: the output is that value row exactly"
        ref = F.scaled_dot_product_attention(torch.from_numpy(q[None, None].astype(np.float64)),
                                             torch.from_numpy(k[None].astype(np.float64)),
                                             torch.from_numpy(v[None].astype(np.float64))).numpy()[0, 0]
        assert np.abs(out - ref).max() < 1e-5
    # equal keys: uniform weights 1/n
    n = 9
    k = np.tile(rng.standard_normal(dh).astype(np.float32), (n, 1))
    v = rng.standard_normal((n, dh)).astype(np.float32)
    _, wts = o.attention_head(rng.standard_normal(dh).astype(np.float32), k, v)
    assert np.all(wts == np.float32(1.0) / np.float32(n))


def check_linear_f32(o):
    rng = np.random.default_rng(3)
    x = rng.standard_normal(96).astype(np.float32)
    w = rng.standard_normal((96, 40)).astype(np.float32)
    b = rng.standard_normal(40).astype(np.float32)
    ref = x.astype(np.float64) @ w.astype(np.float64) + b
    assert np.abs(o.linear_f32(x, w, b) - ref).max() < 1e-4


def check_argmax(o):
    rng = np.random.default_rng(4)
    for _ in range(20):
        x = rng.standard_normal(1000).astype(np.float32)
        st, i = o.argmax(x)
        assert st == "ok" and i == int(np.argmax(x))
    x = np.zeros(50, np.float32)
    x[[7, 13, 40]] = 3.0
    assert o.argmax(x) == ("ok", 7), "ties go to the lowest index"
    x = np.full(8, -1.0, np.float32)
    x[2], x[5] = -0.0, 0.0
    assert o.argmax(x) == ("ok", 2), "-0.0 and +0.0 compare equal"
    for bad in (np.nan, np.inf, -np.inf):
        x = rng.standard_normal(64).astype(np.float32)
        x[30] = bad
        assert o.argmax(x) == ("nonfinite", 0xFFFFFFFF)


# ------------------------------------------------------------------ int8
def check_quantizer(o):
    cases = _golden("int8_quantizer_cases.json")
    for c in cases["fixed_scale"]:
        got = o.quantize(np.array(c["x"], np.float32), c["s"])
        assert got.tolist() == c["q"], (c["why"], got.tolist())
    ramp = np.concatenate([np.arange(-63, 64, 2, dtype=np.float32)[:63], [127.0]]).astype(np.float32)
    q, s = o.quantize_groups(ramp)
    assert s[0] == 1.0 and np.array_equal(q.astype(np.float32), ramp)
    q, s = o.quantize_groups(np.zeros(64, np.float32))
    assert s[0] == 0.0 and not q.any()
    x = np.random.default_rng(5).uniform(-1, 1, 64).astype(np.float32)
    x[17] = -1.5
    q, s = o.quantize_groups(x)
    assert q[17] == -127 and s[0] == np.float32(1.5) / np.float32(127.0)
    nan = np.ones(64, np.float32)
    nan[3] = np.nan
    q, s = o.quantize_groups(nan)
    assert q[3] == 0 and s[0] == np.float32(1.0) / np.float32(127.0) and q[0] == 127


def check_q8_group_dots(o):
    rng = np.random.default_rng(6)
    for n in (64, 768, 3072):
        xq = rng.integers(-127, 128, n).astype(np.int8)
        wq = rng.integers(-127, 128, n).astype(np.int8)
        acc = o.q8_group_dots(xq, wq)
        ref = (xq.astype(np.int64) * wq.astype(np.int64)).reshape(-1, 64).sum(1)
        assert np.array_equal(acc.astype(np.int64), ref)
    xq = np.full(64, -127, np.int8)
    assert o.q8_group_dots(xq, xq)[0] == 64 * 127 * 127


def check_linear_q8_exact(o):
    """Integer-valued inputs whose every group holds a +-127: both scales are
    exactly 1 and the result is the exact integer dot product."""
    rng = np.random.default_rng(7)
    n_in, n_out = 192, 24
    x = rng.integers(-126, 127, n_in).astype(np.float32)
    x[::64] = 127.0
    wq = rng.integers(-126, 127, (n_out, n_in)).astype(np.int8)
    wq[:, 5::64] = -127
    ws = np.ones((n_out, n_in // 64), np.float32)
    b = rng.integers(-50, 50, n_out).astype(np.float32)
    y = o.linear_q8(x, wq, ws, b)
    ref = wq.astype(np.int64) @ x.astype(np.int64) + b.astype(np.int64)
    assert np.array_equal(y.astype(np.int64), ref)


def check_linear_q8_bound(o):
    """Quantization error bound: with per-group scales s_x, s_w, the result
    differs from the float64 product by at most
    sum_i |x_i| s_w/2 + |w_i| s_x/2 + s_x s_w/4 (+ float32 rounding)."""
    rng = np.random.default_rng(8)
    n_in, n_out = 384, 48
    x = rng.standard_normal(n_in).astype(np.float32)
    w = (0.02 * rng.standard_normal((n_out, n_in))).astype(np.float32)
    ng = n_in // 64
    ws = np.abs(w).reshape(n_out, ng, 64).max(2) / np.float32(127.0)
    wq = np.clip(np.rint(w / np.repeat(ws, 64, 1)), -127, 127).astype(np.int8)
    y = o.linear_q8(x, wq, ws.astype(np.float32))
    sx = (np.abs(x).reshape(ng, 64).max(1) / 127.0)
    wdq = wq.astype(np.float64) * np.repeat(ws, 64, 1)
    exact = wdq @ x.astype(np.float64)
    bound = (np.abs(wdq) * np.repeat(sx, 64)[None, :] / 2).sum(1) * 1.0001 + 1e-6
    assert np.all(np.abs(y - exact) <= bound)
    # the scales must be the ones of *this* row and group: wrong pairing blows the bound
    assert np.abs(y - exact).max() < 0.25 * bound.max() + 1e-6


def check_q8_model(o, shape=SMALL, seed=SEED_SMALL):
    """Weight groups run over 64 consecutive inputs of one output row; every
    dequantized weight lies within half a step of the binary32 weight; the
    int8 model tracks the binary32 model; the int8 embedding is the
    dequantized wte row plus the position row."""
    w = synth.checkpoint(shape, seed, "rich")
    p = torch_gpt2.parse(shape, w)
    m = o.model(shape, w, quant=1)
    L = shape.n_layer
    for idx in (0, 1, 2, 3, 4 * L):
        q, s = m.q8_matrix(idx)
        if idx == 4 * L:
            wf = p["wte"].numpy()
        else:
            wf = p["blocks"][0][["w_qkv", "w_o", "w_fc", "w_p"][idx]].numpy().T
        wf32 = wf.astype(np.float32)
        n_out, n_in = wf32.shape
        mx = np.abs(wf32).reshape(n_out, n_in // 64, 64).max(2)
        assert np.array_equal(s, mx / np.float32(127.0))
        deq = q.astype(np.float64) * np.repeat(s.astype(np.float64), 64, 1)
        # half a step, plus the rounding of the quotient w/s (127 * 2^-23 steps)
        assert np.all(np.abs(deq - wf) <= np.repeat(s, 64, 1) * (0.5 + 127 * 2.0 ** -23))
    toks = synth.tokens(shape.vocab, 8, seed=9)
    lq, _, _ = m.session(list(toks), 8)
    lf, _, _ = o.model(shape, w).session(list(toks), 8)
    assert np.abs(lq - lf).max() < 0.1
    assert np.corrcoef(lq.ravel(), lf.ravel())[0, 1] > 0.995
    # embedding through identity blocks
    wz = synth.checkpoint(shape, seed, "zero_blocks")
    mz = o.model(shape, wz, quant=1)
    qe, se = mz.q8_matrix(4 * L)
    pz = torch_gpt2.parse(shape, wz)
    for pos, t in enumerate((5, 600)):
        cache = np.zeros(pos * o.cache_words_per_position(shape), np.float32)
        st, _, _, tr = mz.cached_step(cache, t, pos, trace=True)
        emb = (qe[t].astype(np.float32) * np.repeat(se[t], 64)).astype(np.float32) + \
            pz["wpe"][pos].numpy().astype(np.float32)
        assert np.array_equal(tr[-1], emb.astype(np.float32))


# ------------------------------------------------------------- validation
def check_validation(o, shape=synth.GPT2_TINY, seed=synth.SEED_TINY):
    w = synth.checkpoint(shape, seed, "plain")
    row = o.cache_words_per_position(shape)
    ok_cache = np.zeros(3 * row, np.float32)
    assert o.cached_step(shape, w, ok_cache, 1, 3)[0] == "ok"
    bad = [
        (w[:-1], ok_cache, 1, 3, "weights_len"),
        (np.concatenate([w, w[:1]]), ok_cache, 1, 3, "weights_len"),
        (w, ok_cache, shape.vocab, 3, "token"),
        (w, ok_cache, 0xFFFFFFFF, 3, "token"),
        (w, np.zeros(shape.max_pos * row, np.float32), 1, shape.max_pos, "position"),
        (w, ok_cache[:-1], 1, 3, "cache_len"),
        (w, np.zeros(4 * row, np.float32), 1, 3, "cache_len"),
    ]
    # several invalid inputs at once: the first condition in the order the
    # README's cachedStep paragraph names them (weight length, token,
    # position, cache length) decides the status; the outputs are empty in
    # every case (reading R17)
    bad += [
        (w[:-1], np.zeros(shape.max_pos * row + 1, np.float32), shape.vocab, shape.max_pos + 1, "weights_len"),
        (w, np.zeros(shape.max_pos * row + 1, np.float32), shape.vocab, shape.max_pos + 1, "token"),
        (w, ok_cache, 1, shape.max_pos, "position"),
    ]
    for ww, cc, t, pos, want in bad:
        st, lg, co = o.cached_step(shape, ww, cc, t, pos)
        assert st == want and lg.size == 0 and co.size == 0, (want, st)
    toks = synth.tokens(shape.vocab, 4)
    assert o.infer(shape, w, toks.astype("<u4").tobytes())[0] == "ok"
    bad_inf = [
        (w[:-1], toks.astype("<u4").tobytes(), "weights_len"),
        (w, b"", "tokens_len"),
        (w, toks.astype("<u4").tobytes()[:-1], "tokens_len"),
        (w, np.zeros(shape.max_pos + 1, "<u4").tobytes(), "tokens_len"),
        (w, np.array([1, shape.vocab], "<u4").tobytes(), "token"),
        # several at once (infer paragraph: weight length, then the token
        # array, its length before its entries; reading R17)
        (w[:-1], np.array([shape.vocab], "<u4").tobytes()[:-1], "weights_len"),
        (w, np.array([shape.vocab], "<u4").tobytes() + b"\x00", "tokens_len"),
    ]
    for ww, tb, want in bad_inf:
        st, lg = o.infer(shape, ww, tb)
        assert st == want and lg.size == 0, (want, st)
    assert o.infer(shape, w, np.zeros(shape.max_pos, "<u4").tobytes())[0] == "ok"


# ------------------------------------------------------------- binary16 weights
def _binary16_representable(x: np.ndarray) -> np.ndarray:
    """True where x is a binary16 value: at most 11 significant bits with an
    exponent in range, or a multiple of 2^-24 below 2^-14 (subnormals);
    decided with frexp and integer tests, not with a float16 conversion."""
    x = x.astype(np.float64)
    m, e = np.frexp(x)  # x = m * 2^e, 0.5 <= |m| < 1
    normal = (np.abs(x) >= 2.0 ** -14) & (np.abs(x) <= 65504.0)
    sig = m * 2.0 ** 11
    ok_normal = normal & (sig == np.round(sig))
    sub = x * 2.0 ** 24
    ok_sub = (np.abs(x) < 2.0 ** -14) & (sub == np.round(sub))
    return ok_normal | ok_sub


def check_round_f16(o, shape=synth.GPT2_TINY, seed=synth.SEED_TINY):
    """The binary16-weight checkpoint: hand-worked round-to-nearest-even
    cases, which tensors are rounded (layout by name), representability and
    the half-ulp error bound (2^-11 relative for normal values)."""
    from oracle import round_f16
    w = synth.checkpoint(shape, seed, "rich")
    lay = synth.layout(shape)
    o_te = lay["wte"][0]
    # planted values and their hand-rounded binary16 images
    cases = [
        (1.0 + 2.0 ** -11, 1.0),                  # tie, 1 is even
        (1.0 + 3 * 2.0 ** -11, 1.0 + 2.0 ** -9),  # tie, 1 + 2 ulp is even
        (1.0 + 2.0 ** -11 + 2.0 ** -20, 1.0 + 2.0 ** -10),  # above the tie
        (-(1.0 + 2.0 ** -11), -1.0),
        (2.0 ** -25, 0.0),                        # tie with 0 below the least subnormal
        (3 * 2.0 ** -25, 2.0 ** -23),             # subnormal tie to even
        (0.1, 1638.0 / 16384.0),                  # 0.1 -> 0x2E66
        (65504.0, 65504.0),                       # largest finite
    ]
    for i, (v, _) in enumerate(cases):
        w[o_te + i] = v
    r = round_f16(shape, w)
    for i, (v, want) in enumerate(cases):
        assert r[o_te + i] == np.float32(want), (v, r[o_te + i], want)
    for name, v in lay.items():
        if name == "_words":
            continue
        off, n = v
        a, b = w[off:off + n], r[off:off + n]
        if name == "wte" or name.split(".")[-1].startswith("w_"):
            assert _binary16_representable(b).all(), name
            big = np.abs(a) >= 2.0 ** -14
            rel = np.abs(b[big].astype(np.float64) - a[big]) / np.abs(a[big].astype(np.float64))
            assert rel.max() <= 2.0 ** -11, name
            assert (np.abs(b[~big].astype(np.float64) - a[~big]) <= 2.0 ** -25).all(), name
            assert not np.array_equal(a, b), name  # random weights do move
        else:
            assert np.array_equal(a.view(np.uint32), b.view(np.uint32)), name
    # the quant=2 model is the binary32 model on the rounded checkpoint and stays near it
    w = synth.checkpoint(shape, seed, "rich")  # without the planted values
    r = round_f16(shape, w)
    toks = list(synth.tokens(shape.vocab, 4))
    lh, _, _ = o.model(shape, w, quant=2).session(toks, 4)
    lr, _, _ = o.model(shape, r, quant=0).session(toks, 4)
    lf, _, _ = o.model(shape, w, quant=0).session(toks, 4)
    assert np.array_equal(lh.view(np.uint32), lr.view(np.uint32))
    assert 0 < np.abs(lh - lf).max() < 0.05


# ------------------------------------------------------------- per-row int8 scales
def check_q8_row_scales(o, shape=SMALL, seed=SEED_SMALL):
    """Per-row weight scales (quant 3) and per-activation-row scales (quant
    4, the quantized GPT-2 abstract's rejected first design): every matrix
    row has one scale, 127 times it is the row's largest magnitude, the
    largest code is 127 and every code is within half a step of its weight
    (checked in float64 against the checkpoint); the per-row activation
    quantizer on a hand-worked vector; and the ablation changes the model's
    logits."""
    w = synth.checkpoint(shape, seed, "rich")
    p = torch_gpt2.parse(shape, w)
    L = shape.n_layer
    m3 = o.model(shape, w, quant=3)
    m1 = o.model(shape, w, quant=1)
    differ = False
    for idx in range(4 * L + 1):
        if idx == 4 * L:
            W = p["wte"].numpy()  # [out][in]
        else:
            W = p["blocks"][idx // 4][["w_qkv", "w_o", "w_fc", "w_p"][idx % 4]].numpy().T  # [out][in]
        q, sc = m3.q8_matrix(idx)
        s = sc[:, :1].astype(np.float64)
        assert (sc == sc[:, :1]).all(), idx  # one scale per row
        mx = np.abs(W).max(axis=1, keepdims=True)
        assert (np.abs(127.0 * s - mx) <= 1e-6 * mx).all(), idx
        assert (np.abs(q).max(axis=1) == 127).all(), idx
        assert (np.abs(q * s - W) <= 0.5 * s * (1 + 1e-6)).all(), idx
        differ |= not np.array_equal(m1.q8_matrix(idx)[1], sc)
    assert differ  # group scales are not per-row scales on this shape
    # hand-worked per-row activation codes: the largest magnitude sits in the
    # second group; one scale 2/127 for the whole vector
    x = np.zeros(128, np.float32)
    x[64], x[0], x[1], x[2], x[65] = -2.0, 1.0, -1.0, 0.001, 0.5
    qx, sx = o.quantize_row(x)
    assert np.array_equal(sx, np.full(2, np.float32(2.0) / np.float32(127.0), np.float32))
    want = np.zeros(128, np.int8)
    # 1/(2/127) = 63.5 -> 64 (even); 0.001 -> 0.0635 -> 0; 0.5 -> 31.75 -> 32
    want[64], want[0], want[1], want[2], want[65] = -127, 64, -64, 0, 32
    assert np.array_equal(qx, want)
    # the ablation changes the logits; both stay near the binary32 model
    toks = list(synth.tokens(shape.vocab, 4))
    lf, _, _ = o.model(shape, w, quant=0).session(toks, 4)
    l3, _, _ = m3.session(toks, 4)
    m4 = o.model(shape, w, quant=4)
    l4, _, _ = m4.session(toks, 4)
    assert not np.array_equal(l3, l4)
    # already the first block's output differs (the block projections take
    # one activation scale, not only the vocabulary projection)
    row = o.cache_words_per_position(shape)
    t3 = m3.cached_step(np.zeros(row, np.float32), int(toks[1]), 1, trace=True)[3]
    t4 = m4.cached_step(np.zeros(row, np.float32), int(toks[1]), 1, trace=True)[3]
    assert not np.array_equal(t3[0], t4[0])
    m4.close()
    assert np.abs(l3 - lf).max() < 0.2 and np.abs(l4 - lf).max() < 0.5
    m1.close()
    m3.close()


FAST_CHECKS = [check_sizes, check_forward_vs_torch, check_cached_equals_infer, check_cache_prefix_kept,
               check_zero_blocks, check_layernorm, check_gelu, check_attention, check_linear_f32,
               check_argmax, check_quantizer, check_q8_group_dots, check_linear_q8_exact,
               check_linear_q8_bound, check_q8_model, check_round_f16, check_q8_row_scales,
               check_validation]
