// api.cu -- the C ABI declared in include/gpt2.h: validation (LeanExe GPT-2
// README, infer and cachedStep paragraphs), device memory ownership, and the
// launches of the step kernel.
#include <cuda_runtime.h>

#include <cstdlib>
#include <cstring>
#include <new>
#include <vector>

#include "../../include/gpt2.h"
#include "gpt2_dev.cuh"
#include "model_internal.h"
#include "prefill.h"

namespace gpt2 {
cudaError_t launch_step(const StepPlan& P, int wq, cudaStream_t stream);
int step_max_ctas(int D, int FF, int DH, int wq, int max_pos);
bool step_shape_supported(int D, int FF, int DH);
cudaError_t repack_matrix(const float* src_in_out, uint8_t* dst, int K, int N, int wf, bool per_row,
                          cudaStream_t st);
cudaError_t rows_to_f16(const float* src, uint8_t* dst, size_t n, cudaStream_t st);
cudaError_t quantize_rows(const float* src_out_in, uint8_t* dst, int K, int N, bool per_row, cudaStream_t st);
cudaError_t fold_rows(const uint8_t* rows, int K, int N, int wf, const float* g, const float* b, const float* bias,
                      float* c, float* d, cudaStream_t st);
cudaError_t launch_project(const uint8_t* rows, int K, int N, int wq, const float* x, const float* bias, float* y,
                           int stream, int act_row, cudaStream_t st);
cudaError_t launch_argmax(const float* v, unsigned n, uint32_t* idx, int* nonfinite, cudaStream_t st);
bool cstep_supported(int D, int FF, int DH, int wf);
cudaError_t cgeo_make(int L, int D, int H, int FF, int wf, int want_ctas, CGeo* out);
cudaError_t cstream_build(const uint8_t* wstream, uint64_t layer_bytes, const uint64_t mat_off[4], int L, int D,
                          int H, int FF, int wf, const CGeo& g, uint8_t* dst, cudaStream_t st);
cudaError_t launch_cstep(const CPlan& P, int wf, cudaStream_t stream);
bool noalloc_prepare();
}  // namespace gpt2

using namespace gpt2;

struct gpt2_session {
    gpt2_model* m;
    float* d_cache;
    unsigned char* d_scratch;  // ScratchLayout or CScratch: status words, last token, tagged exchange buffers
    ScratchLayout lay;
    CScratch clay;
    size_t xoff, xtotal;       // the tagged exchange words: [xoff, xtotal) of d_scratch
    int* d_words;  // [0] status, [1] abort
    uint32_t* d_last_token;
    float* d_logits;       // session-owned logits for gpt2_session_step_host
    uint32_t* d_next;      // session-owned next token
    cudaStream_t own;      // session stream for host-buffer steps
    cudaStream_t last;     // last stream work was enqueued on
    unsigned epoch;
    uint32_t position;
    float* trace_next;
    uint64_t* timing_next;
    int stall_phase;
    uint64_t wait_limit_ns;
    PrefillWs pf;  // tensor-core prefill workspace, allocated on first use
    // gpt2_session_run_host buffers (grown on demand): tokens in, logits, choices
    uint32_t* d_run_in = nullptr;
    float* d_run_logits = nullptr;
    uint32_t* d_run_out = nullptr;
    uint32_t run_cap = 0;
};

namespace {

constexpr uint64_t kDefaultWaitNs = 2000000000ull;  // 2 s
// Whether binary32 and binary16 models step on the cluster kernel unless
// GPT2_STEP_KERNEL says otherwise.
constexpr bool kClusterStepDefault = true;

size_t words_of(const gpt2_config* c) {
    size_t d = c->d_model, f = c->d_ff;
    size_t block = 2 * d + d * 3 * d + 3 * d + d * d + d + 2 * d + d * f + f + f * d + d;
    return (size_t)c->vocab * d + (size_t)c->n_pos * d + (size_t)c->n_layer * block + 2 * d;
}

size_t row_words(const gpt2_config* c) { return (size_t)c->n_layer * 2 * c->d_model; }

bool config_ok(const gpt2_config* c) {
    if (!c || c->n_layer == 0 || c->n_layer > (uint32_t)kMaxLayers || c->n_head == 0 || c->vocab == 0 ||
        c->n_pos == 0 || c->max_pos == 0 || c->max_pos > c->n_pos)
        return false;
    if (c->d_model % c->n_head) return false;
    return step_shape_supported((int)c->d_model, (int)c->d_ff, (int)(c->d_model / c->n_head));
}

int g_last_cuda_error = 0;

gpt2_status cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return GPT2_OK;
    g_last_cuda_error = (int)e;
    if (e == cudaErrorMemoryAllocation) return GPT2_ERR_NOMEM;
    return GPT2_ERR_CUDA;
}

#define CK(x)                                  \
    do {                                       \
        cudaError_t e_ = (x);                  \
        if (e_ != cudaSuccess) {               \
            st = cuda_status(e_);              \
            goto fail;                         \
        }                                      \
    } while (0)

void fill_plan(const gpt2_session* s, StepPlan& P) {
    const gpt2_model* m = s->m;
    const gpt2_config& c = m->cfg;
    memset(&P, 0, sizeof(P));
    P.L = (int)c.n_layer;
    P.D = (int)c.d_model;
    P.H = (int)c.n_head;
    P.FF = (int)c.d_ff;
    P.V = (int)c.vocab;
    P.n_pos = (int)c.n_pos;
    P.max_pos = (int)c.max_pos;
    P.G = m->G;
    P.packed = m->d_packed;
    P.fold = m->d_fold;
    P.wstream = m->d_wstream;
    P.layer_bytes = m->layer_bytes;
    for (int i = 0; i < 4; ++i) P.mat_off[i] = m->mat_off[i];
    P.vocab = m->wfmt != kWF32 ? m->d_vocab : reinterpret_cast<const uint8_t*>(m->d_packed + m->wte_off);
    P.wte_off = m->wte_off;
    P.wpe_off = m->wpe_off;
    P.lnf_g = m->lnf_g;
    P.lnf_b = m->lnf_b;
    for (uint32_t l = 0; l < c.n_layer; ++l) P.lp[l] = m->lp[l];
    P.cache = s->d_cache;
    P.xa = reinterpret_cast<uint64_t*>(s->d_scratch + s->lay.xa);
    P.xb = reinterpret_cast<uint64_t*>(s->d_scratch + s->lay.xb);
    P.qkv = reinterpret_cast<uint64_t*>(s->d_scratch + s->lay.qkv);
    P.u = reinterpret_cast<uint64_t*>(s->d_scratch + s->lay.u);
    P.attn_part = reinterpret_cast<uint64_t*>(s->d_scratch + s->lay.attn);
    P.arg_part = reinterpret_cast<uint64_t*>(s->d_scratch + s->lay.arg);
    P.status = s->d_words;
    P.abort_flag = s->d_words + 1;
    P.last_token = s->d_last_token;
    P.wait_limit_ns = s->wait_limit_ns;
    P.stall_phase = -1;
    P.prefetch_chunks = 0;
    P.pace_ns = kDefaultPaceNs;
    P.act_row = m->quant == GPT2_INT8_ROW_ACT;
}

unsigned phases_per_step(const gpt2_model* m) {
    return m->ckern ? 2u * m->cfg.n_layer + 1u : 5u * m->cfg.n_layer + 1u;
}

// The cluster kernel's plan: the shared StepPlan fields, its geometry and
// its exchange buffers.
void fill_cplan(const gpt2_model* m, unsigned char* scratch, const CScratch& k, float* cache, CPlan& C) {
    C.g = m->cg;
    C.cstream = m->d_cstream;
    C.partO = reinterpret_cast<uint64_t*>(scratch + k.partO);
    C.partP = reinterpret_cast<uint64_t*>(scratch + k.partP);
    StepPlan& P = C.s;
    P.xa = P.xb = P.qkv = P.u = P.attn_part = nullptr;
    P.arg_part = reinterpret_cast<uint64_t*>(scratch + k.arg);
    P.status = reinterpret_cast<int*>(scratch + k.words);
    P.abort_flag = reinterpret_cast<int*>(scratch + k.words) + 1;
    P.last_token = reinterpret_cast<uint32_t*>(scratch + k.last_token);
    P.cache = cache;
}

// Enqueue one run; the caller has validated sizes.
gpt2_status enqueue_run(gpt2_session* s, const uint32_t* d_tokens_in, uint32_t token0, uint32_t n_steps,
                        float* d_logits, size_t stride, uint32_t* d_tokens_out, cudaStream_t stream) {
    StepPlan P;
    fill_plan(s, P);
    const unsigned need = n_steps * phases_per_step(s->m);
    if (s->epoch > (1u << 30)) {
        // tags restart: clear every exchanged word so no stale tag can match
        cudaError_t e = cudaMemsetAsync(s->d_scratch + s->xoff, 0, s->xtotal - s->xoff, stream);
        if (e != cudaSuccess) return cuda_status(e);
        s->epoch = 0;
    }
    P.epoch = s->epoch;
    P.p0 = (int)s->position;
    P.n_steps = (int)n_steps;
    P.tokens_in = d_tokens_in;
    P.token0 = token0;
    P.tokens_out = d_tokens_out;
    P.logits = d_logits;
    P.logits_stride = stride;
    P.trace = s->trace_next;
    P.timing = s->timing_next;
    P.stall_phase = s->stall_phase;
    if (s->stall_phase >= 0) P.wait_limit_ns = s->wait_limit_ns;
    const char* pf = getenv("GPT2_PREFETCH_CHUNKS");
    if (pf) P.prefetch_chunks = atoi(pf);
    const char* pace = getenv("GPT2_PACE_NS");
    if (pace) P.pace_ns = (uint32_t)atoi(pace);
    cudaError_t e;
    if (s->m->ckern) {
        CPlan C;
        memset(&C, 0, sizeof(C));
        C.s = P;
        fill_cplan(s->m, s->d_scratch, s->clay, s->d_cache, C);
        e = launch_cstep(C, s->m->wfmt, stream);
    } else {
        e = launch_step(P, s->m->wfmt, stream);
    }
    if (e != cudaSuccess) return cuda_status(e);
    s->trace_next = nullptr;
    s->timing_next = nullptr;
    s->stall_phase = -1;
    s->epoch += need;
    s->position += n_steps;
    s->last = stream;
    return GPT2_OK;
}

}  // namespace

extern "C" {

size_t gpt2_weight_words(const gpt2_config* cfg) { return cfg ? words_of(cfg) : 0; }

size_t gpt2_cache_words_per_position(const gpt2_config* cfg) { return cfg ? row_words(cfg) : 0; }

int gpt2_last_cuda_error(const char** name) {
    if (name) *name = cudaGetErrorName((cudaError_t)g_last_cuda_error);
    return g_last_cuda_error;
}

const char* gpt2_status_name(gpt2_status st) {
    switch (st) {
        case GPT2_OK: return "ok";
        case GPT2_ERR_WEIGHTS_LEN: return "weights_len";
        case GPT2_ERR_TOKEN: return "token";
        case GPT2_ERR_POSITION: return "position";
        case GPT2_ERR_CACHE_LEN: return "cache_len";
        case GPT2_ERR_TOKENS_LEN: return "tokens_len";
        case GPT2_ERR_NONFINITE: return "nonfinite";
        case GPT2_ERR_CONFIG: return "config";
        case GPT2_ERR_NOMEM: return "nomem";
        case GPT2_ERR_TIMEOUT: return "timeout";
        case GPT2_ERR_CUDA: return "cuda";
        case GPT2_ERR_ARG: return "arg";
        case GPT2_ERR_SCRATCH: return "scratch";
    }
    return "unknown";
}

gpt2_status gpt2_model_create(const gpt2_config* cfg, const void* weights, size_t weights_len, int quant,
                              int grid_ctas, gpt2_model** out) {
    if (!out) return GPT2_ERR_ARG;
    *out = nullptr;
    if (!config_ok(cfg) || (quant != GPT2_F32 && quant != GPT2_INT8_G64 && quant != GPT2_F16 &&
                            quant != GPT2_INT8_ROW && quant != GPT2_INT8_ROW_ACT))
        return GPT2_ERR_CONFIG;
    if (!weights || weights_len != words_of(cfg) * 4) return GPT2_ERR_WEIGHTS_LEN;
    const int D = (int)cfg->d_model, FF = (int)cfg->d_ff, L = (int)cfg->n_layer;
    // the weight format of the device streams: per-row int8 scales use the
    // grouped layout with the row's scale in every group slot
    const int wfmt = (quant == GPT2_INT8_ROW || quant == GPT2_INT8_ROW_ACT) ? kWQ8 : quant;
    const bool q8 = wfmt == kWQ8, per_row = quant == GPT2_INT8_ROW || quant == GPT2_INT8_ROW_ACT;
    const int maxc = step_max_ctas(D, FF, D / (int)cfg->n_head, wfmt, (int)cfg->max_pos);
    if (maxc <= 0) return GPT2_ERR_CUDA;
    if (grid_ctas < 0 || grid_ctas > maxc) return GPT2_ERR_CONFIG;

    gpt2_status st = GPT2_OK;
    gpt2_model* m = new (std::nothrow) gpt2_model();
    if (!m) return GPT2_ERR_NOMEM;
    m->cfg = *cfg;
    m->quant = quant;
    m->wfmt = wfmt;
    m->G = grid_ctas ? grid_ctas : maxc;
    {
        // word offsets of the packed checkpoint (README packed checkpoint
        // paragraph; Hugging Face block order)
        uint64_t o = 0;
        m->wte_off = o; o += (uint64_t)cfg->vocab * D;
        m->wpe_off = o; o += (uint64_t)cfg->n_pos * D;
        std::vector<uint64_t> wq(L), wo(L), wf(L), wp(L);
        for (int l = 0; l < L; ++l) {
            LayerParams& p = m->lp[l];
            p.ln1_g = o; o += D;
            p.ln1_b = o; o += D;
            wq[l] = o; o += (uint64_t)D * 3 * D;
            p.b_qkv = o; o += 3 * D;
            wo[l] = o; o += (uint64_t)D * D;
            p.b_o = o; o += D;
            p.ln2_g = o; o += D;
            p.ln2_b = o; o += D;
            wf[l] = o; o += (uint64_t)D * FF;
            p.b_fc = o; o += FF;
            wp[l] = o; o += (uint64_t)FF * D;
            p.b_p = o; o += D;
        }
        m->lnf_g = o; o += D;
        m->lnf_b = o; o += D;

        const uint64_t rbd = row_bytes(D, wfmt), rbf = row_bytes(FF, wfmt);
        m->mat_off[kQKV] = 0;
        m->mat_off[kO] = m->mat_off[kQKV] + 3ull * D * rbd;
        m->mat_off[kFC] = m->mat_off[kO] + (uint64_t)D * rbd;
        m->mat_off[kP] = m->mat_off[kFC] + (uint64_t)FF * rbd;
        m->layer_bytes = m->mat_off[kP] + (uint64_t)D * rbf;

        CK(cudaMalloc(&m->d_packed, weights_len));
        CK(cudaMemcpy(m->d_packed, weights, weights_len, cudaMemcpyHostToDevice));
        CK(cudaMalloc(&m->d_wstream, m->layer_bytes * L));
        CK(cudaMemset(m->d_wstream, 0, m->layer_bytes * L));
        for (int l = 0; l < L; ++l) {
            uint8_t* base = m->d_wstream + (uint64_t)l * m->layer_bytes;
            CK(repack_matrix(m->d_packed + wq[l], base + m->mat_off[kQKV], D, 3 * D, wfmt, per_row, 0));
            CK(repack_matrix(m->d_packed + wo[l], base + m->mat_off[kO], D, D, wfmt, per_row, 0));
            CK(repack_matrix(m->d_packed + wf[l], base + m->mat_off[kFC], D, FF, wfmt, per_row, 0));
            CK(repack_matrix(m->d_packed + wp[l], base + m->mat_off[kP], FF, D, wfmt, per_row, 0));
        }
        if (!q8) {
            const uint64_t fw = fold_layer_words(D, FF);
            CK(cudaMalloc(&m->d_fold, fw * L * sizeof(float)));
            for (int l = 0; l < L; ++l) {
                const uint8_t* base = m->d_wstream + (uint64_t)l * m->layer_bytes;
                float* f = m->d_fold + (uint64_t)l * fw;
                const LayerParams& p = m->lp[l];
                const float* pk = m->d_packed;
                CK(fold_rows(base + m->mat_off[kQKV], D, 3 * D, wfmt, pk + p.ln1_g, pk + p.ln1_b, pk + p.b_qkv, f,
                             f + 3 * D, 0));
                CK(fold_rows(base + m->mat_off[kFC], D, FF, wfmt, pk + p.ln2_g, pk + p.ln2_b, pk + p.b_fc, f + 6 * D,
                             f + 6 * D + FF, 0));
            }
        }
        if (q8) {
            CK(cudaMalloc(&m->d_vocab, (uint64_t)cfg->vocab * rbd));
            CK(cudaMemset(m->d_vocab, 0, (uint64_t)cfg->vocab * rbd));
            CK(quantize_rows(m->d_packed + m->wte_off, m->d_vocab, D, (int)cfg->vocab, per_row, 0));
        } else if (wfmt == kWF16) {
            CK(cudaMalloc(&m->d_vocab, (uint64_t)cfg->vocab * rbd));
            CK(rows_to_f16(m->d_packed + m->wte_off, m->d_vocab, (size_t)cfg->vocab * D, 0));
        }
        // decode steps: GPT2_STEP_KERNEL=cluster selects the cluster step
        // kernel where it supports the shape and weight format, =phase the
        // per-phase kernel; unset, kClusterStepDefault decides
        const char* sk = getenv("GPT2_STEP_KERNEL");
        const bool want_cluster = sk ? strcmp(sk, "cluster") == 0 : kClusterStepDefault;
        // (a geometry the GPU cannot hold, e.g. too few co-resident
        // clusters, leaves the model on the per-phase kernel)
        bool use_cluster = want_cluster && cstep_supported(D, FF, D / (int)cfg->n_head, wfmt);
        if (use_cluster && cgeo_make(L, D, (int)cfg->n_head, FF, wfmt, grid_ctas, &m->cg) != cudaSuccess) {
            use_cluster = false;
            (void)cudaGetLastError();  // an occupancy query that failed leaves no error behind
        }
        if (use_cluster) {
            CK(cudaMalloc(&m->d_cstream, m->cg.layer_bytes * L));
            CK(cstream_build(m->d_wstream, m->layer_bytes, m->mat_off, L, D, (int)cfg->n_head, FF, wfmt, m->cg,
                             m->d_cstream, 0));
            m->ckern = 1;
            m->G = m->cg.G;
        }
        CK(cudaDeviceSynchronize());
        // the no-allocation entry point's scratch array, set up here so that
        // its calls do none
        if (!noalloc_prepare()) CK(cudaErrorInitializationError);
    }
    *out = m;
    return GPT2_OK;
fail:
    gpt2_model_destroy(m);
    return st;
}

void gpt2_model_destroy(gpt2_model* m) {
    if (!m) return;
    cudaFree(m->d_packed);
    cudaFree(m->d_wstream);
    cudaFree(m->d_vocab);
    cudaFree(m->d_fold);
    cudaFree(m->d_wlo);
    cudaFree(m->d_wte_lo);
    cudaFree(m->d_cstream);
    delete m;
}

int gpt2_model_step_kernel(const gpt2_model* m, uint32_t* clusters, uint32_t* cluster_size) {
    if (!m) return -1;
    if (clusters) *clusters = m->ckern ? (uint32_t)m->cg.NC : 0u;
    if (cluster_size) *cluster_size = m->ckern ? (uint32_t)m->cg.CS : (uint32_t)m->G;
    return m->ckern;
}

gpt2_status gpt2_model_read_q8(gpt2_model* m, int index, int8_t* q_host, float* s_host) {
    if (!m || !q_host || !s_host) return GPT2_ERR_ARG;
    if (m->wfmt != kWQ8) return GPT2_ERR_CONFIG;
    const int D = (int)m->cfg.d_model, FF = (int)m->cfg.d_ff, L = (int)m->cfg.n_layer;
    if (index < 0 || index > 4 * L) return GPT2_ERR_ARG;
    int K, N;
    const uint8_t* src;
    if (index == 4 * L) {
        K = D; N = (int)m->cfg.vocab; src = m->d_vocab;
    } else {
        const int l = index / 4, k = index % 4;
        K = (k == kP) ? FF : D;
        N = (k == kQKV) ? 3 * D : (k == kFC ? FF : D);
        src = m->d_wstream + (uint64_t)l * m->layer_bytes + m->mat_off[k];
    }
    const int rb = row_bytes(K, true), ng = K / kGroup;
    std::vector<uint8_t> buf((size_t)N * rb);
    cudaError_t e = cudaMemcpy(buf.data(), src, buf.size(), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_status(e);
    for (int n = 0; n < N; ++n) {
        memcpy(q_host + (size_t)n * K, buf.data() + (size_t)n * rb, K);
        memcpy(s_host + (size_t)n * ng, buf.data() + (size_t)n * rb + K, sizeof(float) * ng);
    }
    return GPT2_OK;
}

gpt2_status gpt2_session_create(gpt2_model* m, gpt2_session** out) {
    if (!m || !out) return GPT2_ERR_ARG;
    *out = nullptr;
    gpt2_status st = GPT2_OK;
    gpt2_session* s = new (std::nothrow) gpt2_session();
    if (!s) return GPT2_ERR_NOMEM;
    s->m = m;
    s->wait_limit_ns = kDefaultWaitNs;
    s->stall_phase = -1;
    {
        const gpt2_config& c = m->cfg;
        s->lay = scratch_layout((int)c.d_model, (int)c.n_head, (int)c.d_ff, m->G);
        size_t words_off = s->lay.words, last_off = s->lay.last_token;
        s->xoff = s->lay.xa;
        s->xtotal = s->lay.total;
        if (m->ckern) {
            s->clay = cscratch_layout((int)c.d_model, (int)c.n_head, m->cg.NC, m->cg.G);
            words_off = s->clay.words;
            last_off = s->clay.last_token;
            s->xoff = s->clay.partO;
            s->xtotal = s->clay.total;
        }
        CK(cudaMalloc(&s->d_cache, sizeof(float) * row_words(&c) * c.max_pos));
        CK(cudaMemset(s->d_cache, 0, sizeof(float) * row_words(&c) * c.max_pos));
        CK(cudaMalloc(&s->d_scratch, s->xtotal));
        CK(cudaMemset(s->d_scratch, 0, s->xtotal));
        s->d_words = reinterpret_cast<int*>(s->d_scratch + words_off);
        s->d_last_token = reinterpret_cast<uint32_t*>(s->d_scratch + last_off);
        CK(cudaMemset(s->d_last_token, 0xFF, sizeof(uint32_t) * 2));
        CK(cudaMalloc(&s->d_logits, sizeof(float) * c.vocab));
        CK(cudaMalloc(&s->d_next, sizeof(uint32_t)));
        CK(cudaStreamCreateWithFlags(&s->own, cudaStreamNonBlocking));
        s->last = s->own;
    }
    *out = s;
    return GPT2_OK;
fail:
    gpt2_session_destroy(s);
    return st;
}

void gpt2_session_destroy(gpt2_session* s) {
    if (!s) return;
    if (s->last) cudaStreamSynchronize(s->last);
    cudaFree(s->d_cache);
    cudaFree(s->d_scratch);
    prefill_free(&s->pf);
    cudaFree(s->d_logits);
    cudaFree(s->d_next);
    cudaFree(s->d_run_in);
    cudaFree(s->d_run_logits);
    cudaFree(s->d_run_out);
    if (s->own) cudaStreamDestroy(s->own);
    delete s;
}

uint32_t gpt2_session_position(const gpt2_session* s) { return s ? s->position : 0; }

gpt2_status gpt2_session_sync(gpt2_session* s) {
    if (!s) return GPT2_ERR_ARG;
    cudaError_t e = cudaStreamSynchronize(s->last);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s->own);
    if (e != cudaSuccess) return cuda_status(e);
    int words[2] = {0, 0};
    e = cudaMemcpy(words, s->d_words, sizeof(words), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_status(e);
    if (words[0] == 0 && words[1] == 0) return GPT2_OK;
    // A failed run leaves exchanged words mid-sequence: clear them and restart the tags.
    e = cudaMemset(s->d_words, 0, sizeof(int) * 4);
    if (e == cudaSuccess) e = cudaMemset(s->d_scratch + s->xoff, 0, s->xtotal - s->xoff);
    if (e != cudaSuccess) return cuda_status(e);
    s->epoch = 0;
    return words[0] ? (gpt2_status)words[0] : GPT2_ERR_TIMEOUT;
}

gpt2_status gpt2_session_load_cache(gpt2_session* s, const void* cache, size_t len) {
    if (!s || (!cache && len)) return GPT2_ERR_ARG;
    const size_t rowb = row_words(&s->m->cfg) * 4;
    if (len % rowb || len / rowb >= s->m->cfg.max_pos) return GPT2_ERR_CACHE_LEN;
    cudaError_t e = cudaStreamSynchronize(s->last);
    if (e == cudaSuccess && len) e = cudaMemcpy(s->d_cache, cache, len, cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaMemset(s->d_last_token, 0xFF, sizeof(uint32_t));
    if (e != cudaSuccess) return cuda_status(e);
    s->position = (uint32_t)(len / rowb);
    return GPT2_OK;
}

gpt2_status gpt2_session_rewind(gpt2_session* s, uint32_t position) {
    if (!s) return GPT2_ERR_ARG;
    if (position > s->position) return GPT2_ERR_POSITION;
    cudaError_t e = cudaMemsetAsync(s->d_last_token, 0xFF, sizeof(uint32_t), s->last);
    if (e != cudaSuccess) return cuda_status(e);
    s->position = position;
    return GPT2_OK;
}

gpt2_status gpt2_session_read_cache(gpt2_session* s, void* out, size_t capacity, size_t* len) {
    if (!s || !len) return GPT2_ERR_ARG;
    *len = 0;
    const size_t bytes = row_words(&s->m->cfg) * 4 * s->position;
    if (capacity < bytes || (!out && bytes)) return GPT2_ERR_ARG;
    cudaError_t e = cudaStreamSynchronize(s->last);
    if (e == cudaSuccess && bytes) e = cudaMemcpy(out, s->d_cache, bytes, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_status(e);
    *len = bytes;
    return GPT2_OK;
}

gpt2_status gpt2_session_run(gpt2_session* s, const uint32_t* d_tokens_in, uint32_t n_steps, float* d_logits,
                             size_t stride, uint32_t* d_tokens_out, void* stream) {
    if (!s || !d_tokens_in) return GPT2_ERR_ARG;
    if (n_steps == 0) return GPT2_ERR_TOKENS_LEN;
    if ((uint64_t)s->position + n_steps > s->m->cfg.max_pos) return GPT2_ERR_POSITION;
    return enqueue_run(s, d_tokens_in, 0, n_steps, d_logits, stride, d_tokens_out, (cudaStream_t)stream);
}

gpt2_status gpt2_session_step(gpt2_session* s, uint32_t token, float* d_logits, uint32_t* d_next_token,
                              void* stream) {
    if (!s) return GPT2_ERR_ARG;
    if (token != GPT2_TOKEN_GREEDY && token >= s->m->cfg.vocab) return GPT2_ERR_TOKEN;
    if (s->position >= s->m->cfg.max_pos) return GPT2_ERR_POSITION;
    return enqueue_run(s, nullptr, token, 1, d_logits, 0, d_next_token, (cudaStream_t)stream);
}

gpt2_status gpt2_session_step_host(gpt2_session* s, uint32_t token, float* logits_host, uint32_t* next_host) {
    if (!s) return GPT2_ERR_ARG;
    if (token != GPT2_TOKEN_GREEDY && token >= s->m->cfg.vocab) return GPT2_ERR_TOKEN;
    if (s->position >= s->m->cfg.max_pos) return GPT2_ERR_POSITION;
    gpt2_status st = enqueue_run(s, nullptr, token, 1, s->d_logits, 0, s->d_next, s->own);
    if (st != GPT2_OK) return st;
    cudaError_t e = cudaSuccess;
    if (logits_host)
        e = cudaMemcpyAsync(logits_host, s->d_logits, sizeof(float) * s->m->cfg.vocab, cudaMemcpyDeviceToHost,
                            s->own);
    if (e == cudaSuccess && next_host)
        e = cudaMemcpyAsync(next_host, s->d_next, sizeof(uint32_t), cudaMemcpyDeviceToHost, s->own);
    if (e != cudaSuccess) return cuda_status(e);
    return gpt2_session_sync(s);
}

gpt2_status gpt2_session_run_host(gpt2_session* s, const uint32_t* tokens_host, uint32_t n_steps, float* logits_host,
                                  uint32_t* tokens_out_host) {
    if (!s || !tokens_host) return GPT2_ERR_ARG;
    const gpt2_config& c = s->m->cfg;
    if (n_steps == 0) return GPT2_ERR_TOKENS_LEN;
    if ((uint64_t)s->position + n_steps > c.max_pos) return GPT2_ERR_POSITION;
    for (uint32_t i = 0; i < n_steps; ++i)
        if (tokens_host[i] != GPT2_TOKEN_GREEDY && tokens_host[i] >= c.vocab) return GPT2_ERR_TOKEN;
    cudaError_t e = cudaStreamSynchronize(s->last);
    if (e == cudaSuccess && n_steps > s->run_cap) {
        cudaFree(s->d_run_in);
        cudaFree(s->d_run_logits);
        cudaFree(s->d_run_out);
        s->d_run_in = s->d_run_out = nullptr;
        s->d_run_logits = nullptr;
        s->run_cap = 0;
        e = cudaMalloc(&s->d_run_in, sizeof(uint32_t) * n_steps);
        if (e == cudaSuccess) e = cudaMalloc(&s->d_run_out, sizeof(uint32_t) * n_steps);
        if (e == cudaSuccess) e = cudaMalloc(&s->d_run_logits, sizeof(float) * c.vocab * n_steps);
        if (e == cudaSuccess) s->run_cap = n_steps;
    }
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(s->d_run_in, tokens_host, sizeof(uint32_t) * n_steps, cudaMemcpyHostToDevice, s->own);
    if (e != cudaSuccess) return cuda_status(e);
    gpt2_status st = enqueue_run(s, s->d_run_in, 0, n_steps, logits_host ? s->d_run_logits : nullptr, c.vocab,
                                 s->d_run_out, s->own);
    if (st != GPT2_OK) return st;
    if (logits_host)
        e = cudaMemcpyAsync(logits_host, s->d_run_logits, sizeof(float) * c.vocab * n_steps, cudaMemcpyDeviceToHost,
                            s->own);
    if (e == cudaSuccess && tokens_out_host)
        e = cudaMemcpyAsync(tokens_out_host, s->d_run_out, sizeof(uint32_t) * n_steps, cudaMemcpyDeviceToHost,
                            s->own);
    if (e != cudaSuccess) return cuda_status(e);
    return gpt2_session_sync(s);
}

gpt2_status gpt2_session_set_trace(gpt2_session* s, float* d_trace) {
    if (!s) return GPT2_ERR_ARG;
    s->trace_next = d_trace;
    return GPT2_OK;
}

gpt2_status gpt2_session_set_timing(gpt2_session* s, uint64_t* d_stamps) {
    if (!s) return GPT2_ERR_ARG;
    s->timing_next = d_stamps;
    return GPT2_OK;
}

gpt2_status gpt2_session_inject_stall(gpt2_session* s, uint32_t phase, uint64_t wait_limit_ns) {
    if (!s || phase == 0 || wait_limit_ns == 0) return GPT2_ERR_ARG;
    s->stall_phase = (int)phase;
    s->wait_limit_ns = wait_limit_ns;
    return GPT2_OK;
}

gpt2_status gpt2_debug_project(gpt2_model* m, int index, const float* d_x, float* d_y, void* stream) {
    if (!m || !d_x || !d_y) return GPT2_ERR_ARG;
    const int D = (int)m->cfg.d_model, FF = (int)m->cfg.d_ff, L = (int)m->cfg.n_layer;
    if (index < 0 || index > 4 * L) return GPT2_ERR_ARG;
    int K, N;
    const uint8_t* rows;
    const float* bias = nullptr;
    if (index == 4 * L) {
        K = D;
        N = (int)m->cfg.vocab;
        rows = m->wfmt != kWF32 ? m->d_vocab : reinterpret_cast<const uint8_t*>(m->d_packed + m->wte_off);
    } else {
        const int l = index / 4, k = index % 4;
        K = (k == kP) ? FF : D;
        N = (k == kQKV) ? 3 * D : (k == kFC ? FF : D);
        rows = m->d_wstream + (uint64_t)l * m->layer_bytes + m->mat_off[k];
        const LayerParams& lp = m->lp[l];
        const uint64_t b = (k == kQKV) ? lp.b_qkv : (k == kO ? lp.b_o : (k == kFC ? lp.b_fc : lp.b_p));
        bias = m->d_packed + b;
    }
    // the path the step kernel takes for this matrix at one CTA per SM: streaming for the vocabulary
    return cuda_status(launch_project(rows, K, N, m->wfmt, d_x, bias, d_y, index == 4 * L ? 1 : 0,
                                      m->quant == GPT2_INT8_ROW_ACT, (cudaStream_t)stream));
}

gpt2_status gpt2_debug_argmax(const float* d_values, uint32_t n, uint32_t* d_index, int* d_nonfinite,
                              void* stream) {
    if (!d_values || !d_index || !d_nonfinite || n == 0) return GPT2_ERR_ARG;
    return cuda_status(launch_argmax(d_values, n, d_index, d_nonfinite, (cudaStream_t)stream));
}

// ------------------------------------------------------- byte-level entries
gpt2_status gpt2_cached_step(const gpt2_config* cfg, const void* weights, size_t weights_len, const void* cache,
                             size_t cache_len, uint32_t token, uint32_t position, float* logits_out,
                             size_t* logits_len, void* cache_out, size_t* cache_out_len) {
    if (!logits_len || !cache_out_len) return GPT2_ERR_ARG;
    *logits_len = 0;
    *cache_out_len = 0;
    if (!config_ok(cfg)) return GPT2_ERR_CONFIG;
    if (!weights || weights_len != words_of(cfg) * 4) return GPT2_ERR_WEIGHTS_LEN;
    if (token >= cfg->vocab) return GPT2_ERR_TOKEN;
    if (position >= cfg->max_pos) return GPT2_ERR_POSITION;
    const size_t rowb = row_words(cfg) * 4;
    if (cache_len != (size_t)position * rowb) return GPT2_ERR_CACHE_LEN;
    if (!logits_out || !cache_out || (!cache && cache_len)) return GPT2_ERR_ARG;

    gpt2_model* m = nullptr;
    gpt2_session* s = nullptr;
    gpt2_status st = gpt2_model_create(cfg, weights, weights_len, GPT2_F32, 0, &m);
    if (st == GPT2_OK) st = gpt2_session_create(m, &s);
    if (st == GPT2_OK) st = gpt2_session_load_cache(s, cache, cache_len);
    if (st == GPT2_OK) st = gpt2_session_step_host(s, token, logits_out, nullptr);
    size_t got = 0;
    if (st == GPT2_OK) st = gpt2_session_read_cache(s, cache_out, cache_len + rowb, &got);
    gpt2_session_destroy(s);
    gpt2_model_destroy(m);
    if (st != GPT2_OK) return st;
    *logits_len = cfg->vocab;
    *cache_out_len = got;
    return GPT2_OK;
}

gpt2_status gpt2_session_prefill(gpt2_session* s, const uint32_t* d_tokens, uint32_t n, float* d_logits,
                                 uint32_t* d_next_token, void* stream) {
    if (!s || !d_tokens) return GPT2_ERR_ARG;
    gpt2_model* m = s->m;
    const gpt2_config& c = m->cfg;
    if (m->quant != GPT2_F32 || !prefill_shape_supported(c)) return GPT2_ERR_CONFIG;
    if (n == 0 || n > c.max_pos) return GPT2_ERR_TOKENS_LEN;
    if (s->position != 0) return GPT2_ERR_POSITION;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = prefill_make_lo(m, st);
    if (e == cudaSuccess) e = prefill_alloc(&s->pf, (int)c.max_pos, (int)c.d_model, (int)c.d_ff);
    if (e == cudaSuccess)
        e = prefill_enqueue(m, &s->pf, d_tokens, (int)n, s->d_cache, d_logits ? d_logits : s->d_logits, s->d_words,
                            s->d_last_token, d_next_token, st);
    if (e != cudaSuccess) return cuda_status(e);
    s->position = n;
    s->last = st;
    return GPT2_OK;
}

gpt2_status gpt2_infer(const gpt2_config* cfg, const void* weights, size_t weights_len, const void* tokens,
                       size_t tokens_len, float* logits_out, size_t* logits_len) {
    if (!logits_len) return GPT2_ERR_ARG;
    *logits_len = 0;
    if (!config_ok(cfg)) return GPT2_ERR_CONFIG;
    if (!weights || weights_len != words_of(cfg) * 4) return GPT2_ERR_WEIGHTS_LEN;
    if (tokens_len == 0 || tokens_len % 4 || tokens_len / 4 > cfg->max_pos || !tokens) return GPT2_ERR_TOKENS_LEN;
    const size_t n = tokens_len / 4;
    std::vector<uint32_t> ids(n);
    const unsigned char* tb = static_cast<const unsigned char*>(tokens);
    for (size_t i = 0; i < n; ++i) {
        ids[i] = (uint32_t)tb[4 * i] | ((uint32_t)tb[4 * i + 1] << 8) | ((uint32_t)tb[4 * i + 2] << 16) |
                 ((uint32_t)tb[4 * i + 3] << 24);
        if (ids[i] >= cfg->vocab) return GPT2_ERR_TOKEN;
    }
    if (!logits_out) return GPT2_ERR_ARG;

    gpt2_model* m = nullptr;
    gpt2_session* s = nullptr;
    uint32_t* d_ids = nullptr;
    gpt2_status st = gpt2_model_create(cfg, weights, weights_len, GPT2_F32, 0, &m);
    if (st == GPT2_OK) st = gpt2_session_create(m, &s);
    if (st == GPT2_OK) {
        cudaError_t e = cudaMalloc(&d_ids, sizeof(uint32_t) * n);
        if (e == cudaSuccess) e = cudaMemcpy(d_ids, ids.data(), sizeof(uint32_t) * n, cudaMemcpyHostToDevice);
        st = cuda_status(e);
    }
    if (st == GPT2_OK) st = gpt2_session_prefill(s, d_ids, (uint32_t)n, s->d_logits, nullptr, s->own);
    if (st == GPT2_OK) st = gpt2_session_sync(s);
    if (st == GPT2_OK)
        st = cuda_status(cudaMemcpy(logits_out, s->d_logits, sizeof(float) * cfg->vocab, cudaMemcpyDeviceToHost));
    cudaFree(d_ids);
    gpt2_session_destroy(s);
    gpt2_model_destroy(m);
    if (st != GPT2_OK) return st;
    *logits_len = cfg->vocab;
    return GPT2_OK;
}

}  // extern "C"
