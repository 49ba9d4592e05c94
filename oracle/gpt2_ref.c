/*
 * gpt2_ref.c -- the oracle: a plain, slow, single-threaded C99 implementation
 * of the GPT-2 cached decode step, its full-prefix twin and the int8
 * grouped-quantized variant.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this code.  It shares no code, header,
 * table or helper with the CUDA library, and never calls it.
 *
 * Arithmetic: binary32 storage and binary32 operations, as the LeanExe GPT-2
 * README fixes ("binary32 arithmetic"), in naive loops with ascending
 * summation indices.  Build with -O2 -ffp-contract=off so that no multiply
 * and add are fused.  libm expf/tanhf/sqrtf/rintf are used.
 *
 * Sources (cited by page title and section):
 *  [P1] LeanExe GPT-2 README: model description paragraph (block structure),
 *       packed checkpoint paragraph (word order, 124,439,808 words), the
 *       `infer` and `cachedStep` paragraphs (inputs, cache layout, validation),
 *       the CLI paragraph (nonfinite logits rejected).
 *  [P2] "Quantized GPT-2 Inference with Exact WebAssembly Proofs" (marXiv
 *       2609.00018), abstract: signed 8-bit weights and projection inputs,
 *       32-bit integer accumulation, binary32 elsewhere; scales for
 *       consecutive groups of 64 coordinates; nearest-even rounding;
 *       saturation; a fixed order for every rescaling.
 *  [P3] gpt2.s documentation, weight-layout paragraph: the Hugging Face
 *       checkpoint stores block matrices as [input][output].
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *  R1 block-internal tensor order = Hugging Face GPT-2 state-dict order.
 *  R2 LayerNorm: eps = 1e-5, biased variance, (x-mean)/sqrtf(var+eps)*g+b.
 *  R3 heads are contiguous 64-wide slices of q, k and v.
 *  R4 attention score = (q.k) / sqrtf(head_dim); softmax with max shift;
 *     weights = e_j / Z; output = sum_j weight_j * v_j.
 *  R5 GELU = GPT-2 tanh form 0.5x(1+tanh(0.7978845608(x+0.044715x^3))).
 *  R6 argmax: largest value, lowest index on ties; any NaN/Inf logit makes
 *     the status NONFINITE.
 *  R7 int8: group scale s = maxabs/127 (IEEE division); q = rint(x/s)
 *     (nearest-even), saturated to [-127,127]; s == 0 or NaN quotient -> 0.
 *     Weights are grouped by 64 consecutive input coordinates of each output
 *     row; the 48 block matrices and the tied wte are quantized; the
 *     embedding lookup uses the dequantized wte row (float)q*s.  A projection
 *     output is y_j = (sum over groups g ascending, from 0.0f, of
 *     ((float)acc_g * s_x[g]) * s_w[j][g]) + b_j.
 *  R8 max_pos is a configuration field (128 for the pages' entry points,
 *     1024 for the long-context configuration).
 *  R15 per-row weight scales (quant 3): one scale per output row, maxabs over
 *     the row's inputs / 127, codes as in R7; the rescale keeps R7's order
 *     with the row's scale in every group's place: y_j = (sum over g
 *     ascending of ((float)acc_g * s_x[g]) * s_w[j]) + b_j.  Activations keep
 *     their group-64 scales.
 *  R16 per-activation-row scales (quant 4, the abstract's rejected first
 *     design): as R15, and every projection input quantized with one scale
 *     for the whole vector (maxabs / 127), s_x[g] = that scale for all g.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    uint32_t n_layer, d_model, n_head, d_ff, vocab, n_pos, max_pos;
} ref_config;

enum {
    REF_OK = 0,
    REF_ERR_WEIGHTS_LEN = 1,
    REF_ERR_TOKEN = 2,
    REF_ERR_POSITION = 3,
    REF_ERR_CACHE_LEN = 4,
    REF_ERR_TOKENS_LEN = 5,
    REF_ERR_NONFINITE = 6,
    REF_ERR_CONFIG = 7,
    REF_ERR_NOMEM = 8
};

#define REF_GROUP 64
#define REF_LN_EPS 1e-5f

/* ------------------------------------------------------------------ */
/* Checkpoint layout [P1 packed checkpoint paragraph, P3 layout, R1]   */
/* ------------------------------------------------------------------ */

static size_t block_words(const ref_config *c) {
    size_t d = c->d_model, f = c->d_ff;
    return 2 * d + d * 3 * d + 3 * d + d * d + d + 2 * d + d * f + f + f * d + d;
}

size_t ref_weight_words(const ref_config *c) {
    size_t d = c->d_model;
    return (size_t)c->vocab * d + (size_t)c->n_pos * d + (size_t)c->n_layer * block_words(c) + 2 * d;
}

/* Words of one cached position: every layer's keys then values [P1 cachedStep]. */
size_t ref_cache_words_per_position(const ref_config *c) {
    return (size_t)c->n_layer * 2 * c->d_model;
}

typedef struct {
    const float *ln1_g, *ln1_b, *w_qkv, *b_qkv, *w_o, *b_o;
    const float *ln2_g, *ln2_b, *w_fc, *b_fc, *w_p, *b_p;
} ref_block;

/* int8 copy of one projection: q[out][in], s[out][in/64] [R7] */
typedef struct {
    int8_t *q;
    float *s;
    int n_in, n_out;
} ref_q8_matrix;

typedef struct {
    ref_config cfg;
    int quant; /* 0 = binary32, 1 = int8 group-64, 3 = int8 per-row weight scales (R15),
                  4 = int8 per-row weight and activation scales (R16) */
    float *words;
    const float *wte, *wpe, *lnf_g, *lnf_b;
    ref_block *blocks;
    ref_q8_matrix *q8; /* 4 per layer (qkv, o, fc, p) then wte; NULL if fp32 */
} ref_model;

static int config_ok(const ref_config *c) {
    if (!c || c->n_layer == 0 || c->d_model == 0 || c->n_head == 0 || c->d_ff == 0 || c->vocab == 0 ||
        c->n_pos == 0 || c->max_pos == 0)
        return 0;
    if (c->d_model % c->n_head) return 0;
    if (c->max_pos > c->n_pos) return 0;
    if (c->d_model % REF_GROUP || c->d_ff % REF_GROUP) return 0;
    return 1;
}

static float load_le_f32(const unsigned char *p) {
    uint32_t u = (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16) | ((uint32_t)p[3] << 24);
    float f;
    memcpy(&f, &u, 4);
    return f;
}

static void store_le_f32(unsigned char *p, float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    p[0] = (unsigned char)(u & 0xFF);
    p[1] = (unsigned char)((u >> 8) & 0xFF);
    p[2] = (unsigned char)((u >> 16) & 0xFF);
    p[3] = (unsigned char)((u >> 24) & 0xFF);
}

static uint32_t load_le_u32(const unsigned char *p) {
    return (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16) | ((uint32_t)p[3] << 24);
}

/* ------------------------------------------------------------------ */
/* Numerical primitives [P1 "Numerical functions"; R2, R5, R6, R7]     */
/* ------------------------------------------------------------------ */

/* LayerNorm with biased variance [R2]. */
void ref_layernorm(const float *x, const float *g, const float *b, int n, float *y) {
    float sum = 0.0f;
    for (int i = 0; i < n; i++) sum += x[i];
    float mean = sum / (float)n;
    float sq = 0.0f;
    for (int i = 0; i < n; i++) {
        float t = x[i] - mean;
        sq += t * t;
    }
    float var = sq / (float)n;
    float den = sqrtf(var + REF_LN_EPS);
    for (int i = 0; i < n; i++) y[i] = (x[i] - mean) / den * g[i] + b[i];
}

/* GPT-2 tanh-form GELU [R5]. */
float ref_gelu(float x) {
    float inner = 0.7978845608f * (x + 0.044715f * x * x * x);
    return 0.5f * x * (1.0f + tanhf(inner));
}

/* Greedy choice [P1 CLI paragraph; R6].  Returns REF_ERR_NONFINITE (and
 * *idx = 0xFFFFFFFF) when any value is NaN or infinite. */
int ref_argmax(const float *x, size_t n, uint32_t *idx) {
    for (size_t i = 0; i < n; i++) {
        if (!isfinite(x[i])) {
            *idx = 0xFFFFFFFFu;
            return REF_ERR_NONFINITE;
        }
    }
    size_t best = 0;
    for (size_t i = 1; i < n; i++)
        if (x[i] > x[best]) best = i;
    *idx = (uint32_t)best;
    return REF_OK;
}

/* Group scale [R7]: maxabs / 127 in IEEE binary32 division. */
float ref_group_scale(const float *x, int n) {
    float m = 0.0f;
    for (int i = 0; i < n; i++) {
        float a = fabsf(x[i]);
        if (a > m) m = a;
    }
    return m / 127.0f;
}

/* Quantize with a given scale [R7]: nearest-even, saturate to [-127,127]. */
void ref_quantize(const float *x, int n, float s, int8_t *q) {
    for (int i = 0; i < n; i++) {
        float r = 0.0f;
        if (s != 0.0f) r = rintf(x[i] / s);
        if (r != r) r = 0.0f;
        if (r > 127.0f) r = 127.0f;
        if (r < -127.0f) r = -127.0f;
        q[i] = (int8_t)r;
    }
}

/* Quantize a vector in groups of 64 consecutive coordinates [P2; R7]. */
void ref_quantize_groups(const float *x, int n, int8_t *q, float *s) {
    for (int g = 0; g < n / REF_GROUP; g++) {
        s[g] = ref_group_scale(x + g * REF_GROUP, REF_GROUP);
        ref_quantize(x + g * REF_GROUP, REF_GROUP, s[g], q + g * REF_GROUP);
    }
}

/* Quantize a whole vector with one scale [R16]: maxabs over all n / 127;
 * the scale is written to each of the n/64 group slots. */
void ref_quantize_row(const float *x, int n, int8_t *q, float *s) {
    float sr = ref_group_scale(x, n);
    ref_quantize(x, n, sr, q);
    for (int g = 0; g < n / REF_GROUP; g++) s[g] = sr;
}

/* int32 accumulators of one row against a quantized input, per group [P2]. */
void ref_q8_group_dots(const int8_t *xq, const int8_t *wq, int n, int32_t *acc) {
    for (int g = 0; g < n / REF_GROUP; g++) {
        int32_t a = 0;
        for (int i = g * REF_GROUP; i < (g + 1) * REF_GROUP; i++) a += (int32_t)xq[i] * (int32_t)wq[i];
        acc[g] = a;
    }
}

/* ------------------------------------------------------------------ */
/* Projections                                                         */
/* ------------------------------------------------------------------ */

/* y_j = (sum_i x_i W[i][j], i ascending) + b_j, with W stored [in][out]
 * [P3].  The loop runs i outside j so memory is walked in order; each y_j
 * still receives its terms in ascending i. */
void ref_linear_f32(const float *x, const float *w, const float *b, int n_in, int n_out, float *y) {
    for (int j = 0; j < n_out; j++) y[j] = 0.0f;
    for (int i = 0; i < n_in; i++) {
        const float *row = w + (size_t)i * n_out;
        float xi = x[i];
        for (int j = 0; j < n_out; j++) y[j] += xi * row[j];
    }
    if (b)
        for (int j = 0; j < n_out; j++) y[j] = y[j] + b[j];
}

/* int8 projection [P2; R7]: quantize x per group (per_row_x: one scale for
 * all of x [R16]), int32 group sums, then the fixed rescale order. */
static void linear_q8(const float *x, const int8_t *wq, const float *ws, const float *b, int n_in, int n_out,
                      float *y, int per_row_x) {
    int ng = n_in / REF_GROUP;
    int8_t *xq = (int8_t *)malloc((size_t)n_in);
    float *xs = (float *)malloc(sizeof(float) * (size_t)ng);
    int32_t *acc = (int32_t *)malloc(sizeof(int32_t) * (size_t)ng);
    if (per_row_x)
        ref_quantize_row(x, n_in, xq, xs);
    else
        ref_quantize_groups(x, n_in, xq, xs);
    for (int j = 0; j < n_out; j++) {
        ref_q8_group_dots(xq, wq + (size_t)j * n_in, n_in, acc);
        float sum = 0.0f;
        for (int g = 0; g < ng; g++) sum += ((float)acc[g] * xs[g]) * ws[(size_t)j * ng + g];
        y[j] = b ? sum + b[j] : sum;
    }
    free(xq);
    free(xs);
    free(acc);
}

void ref_linear_q8(const float *x, const int8_t *wq, const float *ws, const float *b, int n_in, int n_out,
                   float *y) {
    linear_q8(x, wq, ws, b, n_in, n_out, y, 0);
}

/* The same with the input quantized with one scale [R16]. */
void ref_linear_q8_rowx(const float *x, const int8_t *wq, const float *ws, const float *b, int n_in, int n_out,
                        float *y) {
    linear_q8(x, wq, ws, b, n_in, n_out, y, 1);
}

/* One attention head over n_src cached rows [P1 model paragraph; R4].
 * keys/values: row j starts at keys + j*stride.  weights_out (optional)
 * receives the softmax weights. */
void ref_attention_head(const float *q, const float *keys, const float *values, int n_src, int dh, size_t stride,
                        float *out, float *weights_out) {
    float *e = (float *)malloc(sizeof(float) * (size_t)n_src);
    float scale_den = sqrtf((float)dh);
    for (int j = 0; j < n_src; j++) {
        const float *k = keys + (size_t)j * stride;
        float dot = 0.0f;
        for (int t = 0; t < dh; t++) dot += q[t] * k[t];
        e[j] = dot / scale_den;
    }
    float m = e[0];
    for (int j = 1; j < n_src; j++)
        if (e[j] > m) m = e[j];
    float z = 0.0f;
    for (int j = 0; j < n_src; j++) {
        e[j] = expf(e[j] - m);
        z += e[j];
    }
    for (int j = 0; j < n_src; j++) e[j] = e[j] / z;
    for (int t = 0; t < dh; t++) {
        float o = 0.0f;
        for (int j = 0; j < n_src; j++) o += e[j] * values[(size_t)j * stride + t];
        out[t] = o;
    }
    if (weights_out) memcpy(weights_out, e, sizeof(float) * (size_t)n_src);
    free(e);
}

/* ------------------------------------------------------------------ */
/* Model                                                               */
/* ------------------------------------------------------------------ */

static void q8_from_in_out(const float *w, int n_in, int n_out, ref_q8_matrix *m) {
    /* w is [in][out]; groups run over 64 consecutive inputs of one output. */
    int ng = n_in / REF_GROUP;
    m->n_in = n_in;
    m->n_out = n_out;
    m->q = (int8_t *)malloc((size_t)n_in * n_out);
    m->s = (float *)malloc(sizeof(float) * (size_t)ng * n_out);
    float col[REF_GROUP];
    for (int j = 0; j < n_out; j++)
        for (int g = 0; g < ng; g++) {
            for (int t = 0; t < REF_GROUP; t++) col[t] = w[(size_t)(g * REF_GROUP + t) * n_out + j];
            float s = ref_group_scale(col, REF_GROUP);
            m->s[(size_t)j * ng + g] = s;
            ref_quantize(col, REF_GROUP, s, m->q + (size_t)j * n_in + g * REF_GROUP);
        }
}

/* Per-row weight scales [R15]: row j (output j) = w[.][j] of an [in][out]
 * matrix, or w[j][.] of an [out][in] one; one scale for the whole row,
 * written to each of its group slots. */
static void q8_rows(const float *w, int n_in, int n_out, int in_out, ref_q8_matrix *m) {
    int ng = n_in / REF_GROUP;
    m->n_in = n_in;
    m->n_out = n_out;
    m->q = (int8_t *)malloc((size_t)n_in * n_out);
    m->s = (float *)malloc(sizeof(float) * (size_t)ng * n_out);
    float *row = (float *)malloc(sizeof(float) * (size_t)n_in);
    for (int j = 0; j < n_out; j++) {
        for (int i = 0; i < n_in; i++) row[i] = in_out ? w[(size_t)i * n_out + j] : w[(size_t)j * n_in + i];
        float s = ref_group_scale(row, n_in);
        ref_quantize(row, n_in, s, m->q + (size_t)j * n_in);
        for (int g = 0; g < ng; g++) m->s[(size_t)j * ng + g] = s;
    }
    free(row);
}

static void q8_from_out_in(const float *w, int n_in, int n_out, ref_q8_matrix *m) {
    /* w is [out][in] (the tied wte). */
    int ng = n_in / REF_GROUP;
    m->n_in = n_in;
    m->n_out = n_out;
    m->q = (int8_t *)malloc((size_t)n_in * n_out);
    m->s = (float *)malloc(sizeof(float) * (size_t)ng * n_out);
    for (int j = 0; j < n_out; j++)
        for (int g = 0; g < ng; g++) {
            const float *src = w + (size_t)j * n_in + g * REF_GROUP;
            float s = ref_group_scale(src, REF_GROUP);
            m->s[(size_t)j * ng + g] = s;
            ref_quantize(src, REF_GROUP, s, m->q + (size_t)j * n_in + g * REF_GROUP);
        }
}

void ref_model_free(ref_model *m) {
    if (!m) return;
    if (m->q8) {
        int nm = 4 * (int)m->cfg.n_layer + 1;
        for (int i = 0; i < nm; i++) {
            free(m->q8[i].q);
            free(m->q8[i].s);
        }
        free(m->q8);
    }
    free(m->blocks);
    free(m->words);
    free(m);
}

/* Parse the packed checkpoint [P1 packed checkpoint paragraph; R1] and, for
 * quant 1, 3 or 4, build the int8 copies [P2; R7; R15].  Returns NULL with *status set
 * on a bad configuration or weight length. */
ref_model *ref_model_create(const ref_config *c, const void *weights, size_t weights_len, int quant, int *status) {
    *status = REF_OK;
    if (!config_ok(c) || (quant != 0 && quant != 1 && quant != 3 && quant != 4)) {
        *status = REF_ERR_CONFIG;
        return NULL;
    }
    size_t nw = ref_weight_words(c);
    if (!weights || weights_len != nw * 4) {
        *status = REF_ERR_WEIGHTS_LEN;
        return NULL;
    }
    ref_model *m = (ref_model *)calloc(1, sizeof(ref_model));
    if (!m) {
        *status = REF_ERR_NOMEM;
        return NULL;
    }
    m->cfg = *c;
    m->quant = quant;
    m->words = (float *)malloc(nw * 4);
    m->blocks = (ref_block *)calloc(c->n_layer, sizeof(ref_block));
    if (!m->words || !m->blocks) {
        ref_model_free(m);
        *status = REF_ERR_NOMEM;
        return NULL;
    }
    const unsigned char *src = (const unsigned char *)weights;
    for (size_t i = 0; i < nw; i++) m->words[i] = load_le_f32(src + 4 * i);

    size_t d = c->d_model, f = c->d_ff;
    const float *p = m->words;
    m->wte = p;
    p += (size_t)c->vocab * d;
    m->wpe = p;
    p += (size_t)c->n_pos * d;
    for (uint32_t l = 0; l < c->n_layer; l++) {
        ref_block *b = &m->blocks[l];
        b->ln1_g = p; p += d;
        b->ln1_b = p; p += d;
        b->w_qkv = p; p += d * 3 * d;
        b->b_qkv = p; p += 3 * d;
        b->w_o = p; p += d * d;
        b->b_o = p; p += d;
        b->ln2_g = p; p += d;
        b->ln2_b = p; p += d;
        b->w_fc = p; p += d * f;
        b->b_fc = p; p += f;
        b->w_p = p; p += f * d;
        b->b_p = p; p += d;
    }
    m->lnf_g = p; p += d;
    m->lnf_b = p; p += d;

    if (quant == 1) {
        int nm = 4 * (int)c->n_layer + 1;
        m->q8 = (ref_q8_matrix *)calloc((size_t)nm, sizeof(ref_q8_matrix));
        for (uint32_t l = 0; l < c->n_layer; l++) {
            const ref_block *b = &m->blocks[l];
            q8_from_in_out(b->w_qkv, (int)d, (int)(3 * d), &m->q8[4 * l + 0]);
            q8_from_in_out(b->w_o, (int)d, (int)d, &m->q8[4 * l + 1]);
            q8_from_in_out(b->w_fc, (int)d, (int)f, &m->q8[4 * l + 2]);
            q8_from_in_out(b->w_p, (int)f, (int)d, &m->q8[4 * l + 3]);
        }
        q8_from_out_in(m->wte, (int)d, (int)c->vocab, &m->q8[4 * c->n_layer]);
    } else if (quant == 3 || quant == 4) {
        int nm = 4 * (int)c->n_layer + 1;
        m->q8 = (ref_q8_matrix *)calloc((size_t)nm, sizeof(ref_q8_matrix));
        for (uint32_t l = 0; l < c->n_layer; l++) {
            const ref_block *b = &m->blocks[l];
            q8_rows(b->w_qkv, (int)d, (int)(3 * d), 1, &m->q8[4 * l + 0]);
            q8_rows(b->w_o, (int)d, (int)d, 1, &m->q8[4 * l + 1]);
            q8_rows(b->w_fc, (int)d, (int)f, 1, &m->q8[4 * l + 2]);
            q8_rows(b->w_p, (int)f, (int)d, 1, &m->q8[4 * l + 3]);
        }
        q8_rows(m->wte, (int)d, (int)c->vocab, 0, &m->q8[4 * c->n_layer]);
    }
    return m;
}

/* Copy out one int8 matrix (index 4*layer + {0:qkv,1:o,2:fc,3:p}, or
 * 4*n_layer for wte) as q[out][in] and s[out][in/64]. */
int ref_model_get_q8(const ref_model *m, int index, int8_t *q, float *s) {
    if (!m->q8 || index < 0 || index > 4 * (int)m->cfg.n_layer) return REF_ERR_CONFIG;
    const ref_q8_matrix *x = &m->q8[index];
    memcpy(q, x->q, (size_t)x->n_in * x->n_out);
    memcpy(s, x->s, sizeof(float) * (size_t)x->n_out * (x->n_in / REF_GROUP));
    return REF_OK;
}

static void project(const ref_model *m, int qindex, const float *x, const float *w, const float *b, int n_in,
                    int n_out, float *y) {
    if (m->q8) {
        const ref_q8_matrix *q = &m->q8[qindex];
        linear_q8(x, q->q, q->s, b, n_in, n_out, y, m->quant == 4);
    } else {
        ref_linear_f32(x, w, b, n_in, n_out, y);
    }
}

/* One token through the model at `pos`, given a cache holding rows for
 * positions 0..pos-1 and room for row pos [P1 model paragraph, cachedStep
 * paragraph].  Writes the new keys/values into row pos.  logits may be NULL
 * (the row is then not projected).  trace (optional) receives the residual
 * stream after each block, n_layer x d words. */
static void forward_token(const ref_model *m, float *cache, uint32_t token, uint32_t pos, float *logits,
                          float *trace) {
    const ref_config *c = &m->cfg;
    int d = (int)c->d_model, f = (int)c->d_ff, L = (int)c->n_layer, H = (int)c->n_head, dh = d / H;
    size_t row = ref_cache_words_per_position(c);
    float *x = (float *)malloc(sizeof(float) * d);
    float *a = (float *)malloc(sizeof(float) * d);
    float *o = (float *)malloc(sizeof(float) * d);
    float *y = (float *)malloc(sizeof(float) * d);
    float *qkv = (float *)malloc(sizeof(float) * 3 * d);
    float *u = (float *)malloc(sizeof(float) * f);

    /* Embedding: token row plus position row [P1 model paragraph; R7 for int8]. */
    if (m->q8) {
        const ref_q8_matrix *e = &m->q8[4 * L];
        int ng = d / REF_GROUP;
        for (int i = 0; i < d; i++) {
            float w = (float)e->q[(size_t)token * d + i] * e->s[(size_t)token * ng + i / REF_GROUP];
            x[i] = w + m->wpe[(size_t)pos * d + i];
        }
    } else {
        for (int i = 0; i < d; i++) x[i] = m->wte[(size_t)token * d + i] + m->wpe[(size_t)pos * d + i];
    }

    for (int l = 0; l < L; l++) {
        const ref_block *b = &m->blocks[l];
        /* normalization, then query/key/value projection */
        ref_layernorm(x, b->ln1_g, b->ln1_b, d, a);
        project(m, 4 * l + 0, a, b->w_qkv, b->b_qkv, d, 3 * d, qkv);
        /* append this position's keys and values [P1 cachedStep paragraph] */
        float *mine = cache + ((size_t)pos * L + l) * 2 * d;
        for (int i = 0; i < d; i++) {
            mine[i] = qkv[d + i];
            mine[d + i] = qkv[2 * d + i];
        }
        /* causal attention over positions 0..pos */
        for (int h = 0; h < H; h++) {
            const float *k0 = cache + (size_t)l * 2 * d + h * dh;
            const float *v0 = cache + (size_t)l * 2 * d + d + h * dh;
            ref_attention_head(qkv + h * dh, k0, v0, (int)pos + 1, dh, row, o + h * dh, NULL);
        }
        /* output projection and residual addition */
        project(m, 4 * l + 1, o, b->w_o, b->b_o, d, d, y);
        for (int i = 0; i < d; i++) x[i] = x[i] + y[i];
        /* normalization, GELU feed-forward network, residual addition */
        ref_layernorm(x, b->ln2_g, b->ln2_b, d, a);
        project(m, 4 * l + 2, a, b->w_fc, b->b_fc, d, f, u);
        for (int i = 0; i < f; i++) u[i] = ref_gelu(u[i]);
        project(m, 4 * l + 3, u, b->w_p, b->b_p, f, d, y);
        for (int i = 0; i < d; i++) x[i] = x[i] + y[i];
        if (trace) memcpy(trace + (size_t)l * d, x, sizeof(float) * d);
    }

    if (logits) {
        /* final normalization and tied vocabulary projection (no bias) */
        ref_layernorm(x, m->lnf_g, m->lnf_b, d, a);
        if (m->q8) {
            const ref_q8_matrix *e = &m->q8[4 * L];
            linear_q8(a, e->q, e->s, NULL, d, (int)c->vocab, logits, m->quant == 4);
        } else {
            for (uint32_t j = 0; j < c->vocab; j++) {
                const float *w = m->wte + (size_t)j * d;
                float acc = 0.0f;
                for (int i = 0; i < d; i++) acc += a[i] * w[i];
                logits[j] = acc;
            }
        }
    }
    free(x); free(a); free(o); free(y); free(qkv); free(u);
}

/* cachedStep [P1 cachedStep paragraph]: validates, then returns the logits
 * and the incoming cache with this position's rows appended.  cache_out must
 * hold cache_len + n_layer*2*d*4 bytes; it may be the same buffer as cache.
 * On a validation failure both output lengths are 0. */
int ref_model_cached_step(const ref_model *m, const void *cache, size_t cache_len, uint32_t token,
                          uint32_t position, float *logits_out, size_t *logits_len, void *cache_out,
                          size_t *cache_out_len, float *trace) {
    const ref_config *c = &m->cfg;
    *logits_len = 0;
    *cache_out_len = 0;
    if (token >= c->vocab) return REF_ERR_TOKEN;
    if (position >= c->max_pos) return REF_ERR_POSITION;
    size_t row = ref_cache_words_per_position(c);
    if (cache_len != (size_t)position * row * 4) return REF_ERR_CACHE_LEN;

    float *work = (float *)malloc(sizeof(float) * row * ((size_t)position + 1));
    if (!work) return REF_ERR_NOMEM;
    const unsigned char *src = (const unsigned char *)cache;
    for (size_t i = 0; i < (size_t)position * row; i++) work[i] = load_le_f32(src + 4 * i);
    forward_token(m, work, token, position, logits_out, trace);
    unsigned char *dst = (unsigned char *)cache_out;
    for (size_t i = 0; i < ((size_t)position + 1) * row; i++) store_le_f32(dst + 4 * i, work[i]);
    free(work);
    *logits_len = c->vocab;
    *cache_out_len = ((size_t)position + 1) * row * 4;
    return REF_OK;
}

/* infer [P1 infer paragraph]: full-prefix recompute of up to max_pos tokens,
 * final row's logits.  Implemented as successive positions through the same
 * per-row code, so its logits equal the last cachedStep's bit for bit. */
int ref_model_infer(const ref_model *m, const void *tokens, size_t tokens_len, float *logits_out,
                    size_t *logits_len) {
    const ref_config *c = &m->cfg;
    *logits_len = 0;
    if (tokens_len == 0 || tokens_len % 4 != 0 || tokens_len / 4 > c->max_pos) return REF_ERR_TOKENS_LEN;
    size_t n = tokens_len / 4;
    const unsigned char *tb = (const unsigned char *)tokens;
    for (size_t t = 0; t < n; t++)
        if (load_le_u32(tb + 4 * t) >= c->vocab) return REF_ERR_TOKEN;
    size_t row = ref_cache_words_per_position(c);
    float *work = (float *)malloc(sizeof(float) * row * n);
    if (!work) return REF_ERR_NOMEM;
    for (size_t t = 0; t < n; t++)
        forward_token(m, work, load_le_u32(tb + 4 * t), (uint32_t)t, t + 1 == n ? logits_out : NULL, NULL);
    free(work);
    *logits_len = c->vocab;
    return REF_OK;
}

/* Byte-level entries with the pages' signatures (binary32 model). */
int ref_cached_step(const ref_config *c, const void *weights, size_t weights_len, const void *cache,
                    size_t cache_len, uint32_t token, uint32_t position, float *logits_out, size_t *logits_len,
                    void *cache_out, size_t *cache_out_len) {
    int st;
    *logits_len = 0;
    *cache_out_len = 0;
    ref_model *m = ref_model_create(c, weights, weights_len, 0, &st);
    if (!m) return st;
    st = ref_model_cached_step(m, cache, cache_len, token, position, logits_out, logits_len, cache_out,
                               cache_out_len, NULL);
    ref_model_free(m);
    return st;
}

int ref_infer(const ref_config *c, const void *weights, size_t weights_len, const void *tokens, size_t tokens_len,
              float *logits_out, size_t *logits_len) {
    int st;
    *logits_len = 0;
    ref_model *m = ref_model_create(c, weights, weights_len, 0, &st);
    if (!m) return st;
    st = ref_model_infer(m, tokens, tokens_len, logits_out, logits_len);
    ref_model_free(m);
    return st;
}
