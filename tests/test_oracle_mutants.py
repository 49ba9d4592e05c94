"""Plant plausible mistakes in copies of the oracle and require that the pins
catch every one.  The mistakes are planted in a temporary copy of the C
source, on the CPU; the oracle in the repository is never modified."""
import os
import tempfile

import pytest

import oracle_pins as P
from oracle import Oracle, build, _SRC

# (name, exact text in gpt2_ref.c, replacement)
MUTANTS = [
    ("drop_qkv_bias", "project(m, 4 * l + 0, a, b->w_qkv, b->b_qkv, d, 3 * d, qkv);",
     "project(m, 4 * l + 0, a, b->w_qkv, NULL, d, 3 * d, qkv);"),
    ("unbiased_variance", "float var = sq / (float)n;", "float var = sq / (float)(n - 1);"),
    ("wrong_eps", "#define REF_LN_EPS 1e-5f", "#define REF_LN_EPS 1e-3f"),
    ("ln_gain_dropped", "y[i] = (x[i] - mean) / den * g[i] + b[i];", "y[i] = (x[i] - mean) / den + b[i];"),
    ("score_scale_1_over_dh", "float scale_den = sqrtf((float)dh);", "float scale_den = (float)dh;"),
    ("head_slice_offset", "const float *k0 = cache + (size_t)l * 2 * d + h * dh;",
     "const float *k0 = cache + (size_t)l * 2 * d + h;"),
    ("keys_from_values", "mine[i] = qkv[d + i];", "mine[i] = qkv[2 * d + i];"),
    ("gelu_constant", "0.044715f", "0.44715f"),
    ("no_position_embedding", "x[i] = m->wte[(size_t)token * d + i] + m->wpe[(size_t)pos * d + i];",
     "x[i] = m->wte[(size_t)token * d + i];"),
    ("transposed_projection", "y[j] += xi * row[j];", "y[j] += xi * w[(size_t)j * n_in + i];"),
    ("mlp_residual_dropped", "project(m, 4 * l + 3, u, b->w_p, b->b_p, f, d, y);\n        for (int i = 0; i < d; i++) x[i] = x[i] + y[i];",
     "project(m, 4 * l + 3, u, b->w_p, b->b_p, f, d, y);\n        for (int i = 0; i < d; i++) x[i] = y[i];"),
    ("softmax_no_normalise", "for (int j = 0; j < n_src; j++) e[j] = e[j] / z;", ""),
    ("argmax_last_tie", "if (x[i] > x[best]) best = i;", "if (x[i] >= x[best]) best = i;"),
    ("argmax_accepts_inf", "if (!isfinite(x[i])) {", "if (isnan(x[i])) {"),
    ("round_half_away", "if (s != 0.0f) r = rintf(x[i] / s);", "if (s != 0.0f) r = roundf(x[i] / s);"),
    ("no_saturation", "if (r > 127.0f) r = 127.0f;", "if (r > 128.0f) r = 127.0f;"),
    ("scale_over_128", "return m / 127.0f;", "return m / 128.0f;"),
    ("first_group_scale_only", "sum += ((float)acc[g] * xs[g]) * ws[(size_t)j * ng + g];",
     "sum += ((float)acc[g] * xs[g]) * ws[(size_t)j * ng];"),
    ("embedding_group0_scale",
     "float w = (float)e->q[(size_t)token * d + i] * e->s[(size_t)token * ng + i / REF_GROUP];",
     "float w = (float)e->q[(size_t)token * d + i] * e->s[(size_t)token * ng];"),
    ("infer_positions_zero", "forward_token(m, work, load_le_u32(tb + 4 * t), (uint32_t)t,",
     "forward_token(m, work, load_le_u32(tb + 4 * t), (uint32_t)0,"),
    ("cache_prefix_not_returned", "for (size_t i = 0; i < ((size_t)position + 1) * row; i++) store_le_f32",
     "for (size_t i = (size_t)position * row; i < ((size_t)position + 1) * row; i++) store_le_f32"),
    ("position_bound_off_by_one", "if (position >= c->max_pos) return REF_ERR_POSITION;",
     "if (position > c->max_pos) return REF_ERR_POSITION;"),
    ("row_scale_from_first_group", "float s = ref_group_scale(row, n_in);",
     "float s = ref_group_scale(row, REF_GROUP);"),
    ("row_scale_in_slot0_only", "for (int g = 0; g < ng; g++) m->s[(size_t)j * ng + g] = s;",
     "m->s[(size_t)j * ng] = s;"),
    ("row_gather_transposed", "row[i] = in_out ? w[(size_t)i * n_out + j] : w[(size_t)j * n_in + i];",
     "row[i] = in_out ? w[(size_t)j * n_in + i] : w[(size_t)j * n_in + i];"),
    ("activation_row_scale_first_group", "float sr = ref_group_scale(x, n);",
     "float sr = ref_group_scale(x, REF_GROUP);"),
    ("ablation_ignored", "linear_q8(x, q->q, q->s, b, n_in, n_out, y, m->quant == 4);",
     "linear_q8(x, q->q, q->s, b, n_in, n_out, y, 0);"),
    ("token_bound_off_by_one", "if (token >= c->vocab) return REF_ERR_TOKEN;",
     "if (token > c->vocab) return REF_ERR_TOKEN;"),
    ("attention_residual_dropped",
     "project(m, 4 * l + 1, o, b->w_o, b->b_o, d, d, y);\n        for (int i = 0; i < d; i++) x[i] = x[i] + y[i];",
     "project(m, 4 * l + 1, o, b->w_o, b->b_o, d, d, y);\n        for (int i = 0; i < d; i++) x[i] = y[i];"),
    ("ln1_takes_ln2_parameters", "ref_layernorm(x, b->ln1_g, b->ln1_b, d, a);",
     "ref_layernorm(x, b->ln2_g, b->ln2_b, d, a);"),
    ("final_layernorm_dropped", "ref_layernorm(x, m->lnf_g, m->lnf_b, d, a);", "memcpy(a, x, sizeof(float) * d);"),
    ("out_projection_bias_dropped", "project(m, 4 * l + 1, o, b->w_o, b->b_o, d, d, y);",
     "project(m, 4 * l + 1, o, b->w_o, NULL, d, d, y);"),
    ("fc_bias_dropped", "project(m, 4 * l + 2, a, b->w_fc, b->b_fc, d, f, u);",
     "project(m, 4 * l + 2, a, b->w_fc, NULL, d, f, u);"),
    ("current_position_not_attended", "ref_attention_head(qkv + h * dh, k0, v0, (int)pos + 1, dh, row, o + h * dh, NULL);",
     "ref_attention_head(qkv + h * dh, k0, v0, pos ? (int)pos : 1, dh, row, o + h * dh, NULL);"),
    ("values_read_at_key_offset", "const float *v0 = cache + (size_t)l * 2 * d + d + h * dh;",
     "const float *v0 = cache + (size_t)l * 2 * d + h * dh;"),
    ("signed_group_maximum", "float a = fabsf(x[i]);", "float a = x[i];"),
    ("activation_scale_dropped", "sum += ((float)acc[g] * xs[g]) * ws[(size_t)j * ng + g];",
     "sum += (float)acc[g] * ws[(size_t)j * ng + g];"),
    ("group_dot_skips_first_term", "for (int i = g * REF_GROUP; i < (g + 1) * REF_GROUP; i++) a +=",
     "for (int i = g * REF_GROUP + 1; i < (g + 1) * REF_GROUP; i++) a +="),
    ("int8_bias_dropped", "y[j] = b ? sum + b[j] : sum;", "y[j] = sum;"),
    ("negative_saturation_at_128", "if (r < -127.0f) r = -127.0f;", "if (r < -128.0f) r = -128.0f;"),
    ("position_checked_before_token",
     "    if (token >= c->vocab) return REF_ERR_TOKEN;\n    if (position >= c->max_pos) return REF_ERR_POSITION;",
     "    if (position >= c->max_pos) return REF_ERR_POSITION;\n    if (token >= c->vocab) return REF_ERR_TOKEN;"),
    ("cache_length_checked_before_position",
     "    if (position >= c->max_pos) return REF_ERR_POSITION;\n    size_t row = ref_cache_words_per_position(c);\n"
     "    if (cache_len != (size_t)position * row * 4) return REF_ERR_CACHE_LEN;",
     "    size_t row = ref_cache_words_per_position(c);\n"
     "    if (cache_len != (size_t)position * row * 4) return REF_ERR_CACHE_LEN;\n"
     "    if (position >= c->max_pos) return REF_ERR_POSITION;"),
    ("softmax_without_max_shift", "e[j] = expf(e[j] - m);", "e[j] = expf(e[j]);"),
    ("infer_returns_first_row", "t + 1 == n ? logits_out : NULL", "t == 0 ? logits_out : NULL"),
]


@pytest.fixture(scope="module")
def source():
    with open(_SRC) as f:
        return f.read()


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(source, name, old, new):
    assert source.count(old) == 1, f"mutation site for {name} must be unique"
    with tempfile.TemporaryDirectory() as td:
        src = os.path.join(td, "mutant.c")
        with open(src, "w") as f:
            f.write(source.replace(old, new))
        lib = build(src, os.path.join(td, "mutant.so"))
        o = Oracle(lib)
        caught = []
        for check in P.FAST_CHECKS:
            try:
                check(o)
            except (AssertionError, ValueError, RuntimeError) as e:  # noqa: PERF203
                caught.append(check.__name__)
        assert caught, f"no pin caught mutant {name}"


def _round_f16_mutants():
    """Plausible mistakes in the binary16-weight checkpoint (oracle.round_f16,
    gpt2.s page, half-precision weight paragraph), built around the real
    function: rounding toward zero instead of to nearest, rounding every
    tensor (LayerNorm parameters and biases too), leaving wte in binary32."""
    import numpy as np
    import oracle
    from stream_decode_gb300 import synth
    real = oracle.round_f16

    def toward_zero(shape, weights):
        w = np.asarray(weights, np.float32)
        r = real(shape, weights)
        away = np.abs(r) > np.abs(w)
        r[away] = np.nextafter(r[away].astype(np.float16), np.float16(0)).astype(np.float32)
        return r

    def every_tensor(shape, weights):
        return np.asarray(weights, np.float32).astype(np.float16).astype(np.float32)

    def wte_kept(shape, weights):
        r = real(shape, weights)
        off, n = synth.layout(shape)["wte"]
        r[off:off + n] = np.asarray(weights, np.float32)[off:off + n]
        return r

    return [("round_toward_zero", toward_zero), ("every_tensor_rounded", every_tensor), ("wte_not_rounded", wte_kept)]


@pytest.mark.parametrize("name,fn", _round_f16_mutants(), ids=[m[0] for m in _round_f16_mutants()])
def test_round_f16_pin_catches_mutant(monkeypatch, name, fn):
    import oracle
    monkeypatch.setattr(oracle, "round_f16", fn)
    o = Oracle(oracle.build())
    with pytest.raises(AssertionError):
        P.check_round_f16(o)
