// batch.cu -- B independent decode sessions stepped together: one cached
// step (LeanExe GPT-2 README, cachedStep paragraph) for every session of the
// batch, each at its own position, on its own KV cache.
//
// With B sessions the projections of a step are B-row matrix products, so
// they run on the tensor cores: the prefill's 3xTF32 tcgen05 GEMM (one
// weight read per step for all B rows), its LayerNorm (+ residual) and
// split-reduce kernels, with the key/value columns of the QKV reduce
// appended to row b's own cache at row b's position.  Around them: the
// embedding of each session's token at its position, a decode attention
// kernel (one block per (head, session) over that session's keys), the tied
// vocabulary projection as one more GEMM (N = vocab, padded to 64 with
// zero rows), and the greedy choice (chunks of each row in parallel, then
// one thread per session, which also advances the positions).  A step is
// one CUDA graph (captured once per set of output buffers) replayed once
// per step; every kernel after the step's first is a programmatic
// dependent launch (chain.cuh).
#include <cuda_runtime.h>

#include <cmath>
#include <cstring>
#include <new>
#include <vector>

#include "../../include/gpt2.h"
#include "gpt2_dev.cuh"
#include "model_internal.h"
#include "prefill.h"
#include "rows.cuh"

namespace gpt2 {
namespace {

// Row b of the step: token t = tokens_in[step * B + b] (GPT2_TOKEN_GREEDY:
// the session's previous choice), X[b][:] = wte[t] + wpe[pos[b]].  An
// out-of-range token (or a greedy token with no previous choice) sets the
// status and leaves the row unwritten.
__global__ void batch_embed_kernel(const float* __restrict__ packed, uint64_t wte_off, uint64_t wpe_off,
                                   const uint32_t* __restrict__ tokens_in, const int* __restrict__ step,
                                   const uint32_t* __restrict__ last, const int* __restrict__ pos, int D,
                                   uint32_t vocab, float* __restrict__ X, int* status) {
    chain_enter();
    const int b = blockIdx.x, B = gridDim.x;
    uint32_t t = tokens_in[(size_t)(*step) * B + b];
    if (t == 0xFFFFFFFFu) t = last[b];
    if (t >= vocab) {
        if (threadIdx.x == 0) atomicCAS(status, 0, (int)kDevToken);
        return;
    }
    const float* te = packed + wte_off + (uint64_t)t * D;
    const float* pe = packed + wpe_off + (uint64_t)pos[b] * D;
    for (int j = threadIdx.x; j < D; j += blockDim.x) X[(size_t)b * D + j] = __fadd_rn(te[j], pe[j]);
}

constexpr int kBAttnThreads = 128;
constexpr int kLanesPerKey = 8;
constexpr int kKeySlots = kBAttnThreads / kLanesPerKey;  // keys per pass
constexpr int kPassGroup = 4;                            // passes whose loads are issued together

template <int N>
__device__ __forceinline__ void load_n(const float* p, float (&r)[N]) {
    if constexpr (N % 4 == 0) {
#pragma unroll
        for (int i = 0; i < N; i += 4) {
            const float4 v = *reinterpret_cast<const float4*>(p + i);
            r[i] = v.x;
            r[i + 1] = v.y;
            r[i + 2] = v.z;
            r[i + 3] = v.w;
        }
    } else {
#pragma unroll
        for (int i = 0; i < N; i += 2) {
            const float2 v = *reinterpret_cast<const float2*>(p + i);
            r[i] = v.x;
            r[i + 1] = v.y;
        }
    }
}

// Attention of session b (blockIdx.y), head h (blockIdx.x) at its position
// p = pos[b]: s_j = (q . k_j) / sqrt(DH) over the keys j = 0..p of layer l
// in the session's cache (this step's key and value were appended by the
// QKV reduce), softmax, o = sum_j a_j v_j.  Key j goes to slot j mod 16;
// the 8 lanes of a slot hold DH / 8 coordinates each and keep an online
// max, sum and weighted value sum over their slot's keys; the 16 slots are
// merged with the log-sum-exp rule in shared memory.
template <int DH>
__global__ void __launch_bounds__(kBAttnThreads) batch_attention_kernel(const float* __restrict__ QKV,
                                                                        const float* __restrict__ cache,
                                                                        size_t session_words,
                                                                        const int* __restrict__ pos, int L, int l,
                                                                        int D, float* __restrict__ O,
                                                                        float* __restrict__ Olo) {
    constexpr int DPL = DH / kLanesPerKey;
    static_assert(DPL >= 2 && DPL % 2 == 0, "head width");
    __shared__ float sm[kKeySlots], sz[kKeySlots];
    __shared__ float so[kKeySlots][DH];
    chain_enter();
    const int h = blockIdx.x, b = blockIdx.y, t = threadIdx.x;
    const int slot = t / kLanesPerKey, e8 = t % kLanesPerKey;
    const int p = pos[b];
    float q[DPL];
    load_n<DPL>(QKV + (size_t)b * 3 * D + (size_t)h * DH + e8 * DPL, q);
    const float scale = 1.0f / sqrtf((float)DH);
    const size_t row = (size_t)L * 2 * D;  // words between positions
    const float* kb = cache + (size_t)b * session_words + (size_t)l * 2 * D + (size_t)h * DH + e8 * DPL;
    float m = -INFINITY, z = 0.0f, o[DPL];
#pragma unroll
    for (int d = 0; d < DPL; ++d) o[d] = 0.0f;
    // Every lane of the block makes the same number of passes (the shuffles
    // below name the whole warp); a slot whose key of this pass lies past p
    // takes part in the shuffles and skips the update.  The keys and values
    // of kPassGroup passes are loaded before the first of them is used, so
    // their cache round trips overlap.
    for (int jg = 0; jg <= p; jg += kPassGroup * kKeySlots) {
        float k[kPassGroup][DPL], v[kPassGroup][DPL];
#pragma unroll
        for (int g = 0; g < kPassGroup; ++g) {
            const int j = jg + g * kKeySlots + slot;
            if (j <= p) {
                load_n<DPL>(kb + (size_t)j * row, k[g]);
                load_n<DPL>(kb + (size_t)j * row + D, v[g]);
            } else {
#pragma unroll
                for (int d = 0; d < DPL; ++d) k[g][d] = v[g][d] = 0.0f;
            }
        }
#pragma unroll
        for (int g = 0; g < kPassGroup; ++g) {
            const bool have = jg + g * kKeySlots + slot <= p;
            float s = 0.0f;
#pragma unroll
            for (int d = 0; d < DPL; ++d) s = fmaf(q[d], k[g][d], s);
#pragma unroll
            for (int off = 1; off < kLanesPerKey; off <<= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
            if (have) {
                s *= scale;
                const float mn = fmaxf(m, s);
                const float corr = expf(m - mn);  // 0 while m is -inf
                const float e = expf(s - mn);
                z = fmaf(z, corr, e);
#pragma unroll
                for (int d = 0; d < DPL; ++d) o[d] = fmaf(o[d], corr, e * v[g][d]);
                m = mn;
            }
        }
    }
    if (e8 == 0) {
        sm[slot] = m;
        sz[slot] = z;
    }
#pragma unroll
    for (int d = 0; d < DPL; ++d) so[slot][e8 * DPL + d] = o[d];
    __syncthreads();
    for (int e = t; e < DH; e += kBAttnThreads) {
        float M = -INFINITY;
#pragma unroll
        for (int s = 0; s < kKeySlots; ++s) M = fmaxf(M, sm[s]);
        float num = 0.0f, den = 0.0f;
#pragma unroll
        for (int s = 0; s < kKeySlots; ++s) {
            const float w = expf(sm[s] - M);  // 0 for a slot without keys
            num = fmaf(so[s][e], w, num);
            den = fmaf(sz[s], w, den);
        }
        const float y = num / den;
        O[(size_t)b * D + (size_t)h * DH + e] = y;
        Olo[(size_t)b * D + (size_t)h * DH + e] = tf32_lo(y);
    }
}

constexpr int kBChoiceThreads = 256;
constexpr int kChoiceChunk = 4096;  // logits of one row per block of the logits kernel

// Block (c, b): logits n of row b in chunk c ([c * 4096, (c + 1) * 4096) and
// n < V) = the sum over the vocabulary GEMM's splits of part[s][b][n] (part
// rows are ldp floats apart, a multiple of 64; B rows a split), copied to
// out + step * stride + b * V when out is given; the chunk's greedy
// candidate (largest, lowest index on ties, any non-finite value flagged)
// goes to cand_v / cand_i / cand_nf[b * C + c].
__global__ void __launch_bounds__(kBChoiceThreads) batch_logits_kernel(
    const float* __restrict__ part, int splits, int ldp, int V, float* __restrict__ out, size_t stride,
    const int* __restrict__ step, float* __restrict__ cand_v, unsigned* __restrict__ cand_i,
    int* __restrict__ cand_nf) {
    __shared__ float s_v[kBChoiceThreads / 32];
    __shared__ unsigned s_i[kBChoiceThreads / 32];
    __shared__ int s_nf[kBChoiceThreads / 32];
    chain_enter();
    const int c = blockIdx.x, C = gridDim.x, b = blockIdx.y, B = gridDim.y;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    float* o = out ? out + (size_t)(*step) * stride + (size_t)b * V : nullptr;
    float bv = -INFINITY;
    unsigned bi = 0xFFFFFFFFu;
    int nf = 0;
    const int n_end = min(V, (c + 1) * kChoiceChunk);
    for (int n = c * kChoiceChunk + 4 * tid; n < n_end; n += 4 * kBChoiceThreads) {
        // 16-byte loads: rows start on 64-float boundaries and n is a multiple of 4
        float4 x = *reinterpret_cast<const float4*>(part + (size_t)b * ldp + n);
        for (int sp = 1; sp < splits; ++sp) {
            const float4 y = *reinterpret_cast<const float4*>(part + ((size_t)sp * B + b) * ldp + n);
            x.x += y.x;
            x.y += y.y;
            x.z += y.z;
            x.w += y.w;
        }
        const float xv[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int k = 0; k < 4; ++k)
            if (n + k < n_end) {
                if (o) o[n + k] = xv[k];
                choice_take(xv[k], (unsigned)(n + k), bv, bi, nf);
            }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
        const unsigned oi = __shfl_xor_sync(0xffffffffu, bi, off);
        nf |= __shfl_xor_sync(0xffffffffu, nf, off);
        if (ov > bv || (ov == bv && oi < bi)) {
            bv = ov;
            bi = oi;
        }
    }
    if (lane == 0) {
        s_v[warp] = bv;
        s_i[warp] = bi;
        s_nf[warp] = nf;
    }
    __syncthreads();
    if (tid == 0) {
        for (int w = 1; w < kBChoiceThreads / 32; ++w) {
            nf |= s_nf[w];
            if (s_v[w] > bv || (s_v[w] == bv && s_i[w] < bi)) {
                bv = s_v[w];
                bi = s_i[w];
            }
        }
        cand_v[(size_t)b * C + c] = bv;
        cand_i[(size_t)b * C + c] = bi;
        cand_nf[(size_t)b * C + c] = nf;
    }
}

// One block of B threads: thread b combines row b's C chunk candidates
// (same rule), writes the choice (0xFFFFFFFF and the status if any logit
// was not finite) to tokens_out[step * B + b] when given and to last[b],
// and advances pos[b]; then the step counter advances.
__global__ void batch_pick_kernel(const float* __restrict__ cand_v, const unsigned* __restrict__ cand_i,
                                  const int* __restrict__ cand_nf, int C, uint32_t* __restrict__ tokens_out,
                                  uint32_t* __restrict__ last, int* __restrict__ pos, int* step, int* status) {
    __shared__ int s_step;
    chain_enter();
    const int b = threadIdx.x, B = blockDim.x;
    if (b == 0) s_step = *step;
    __syncthreads();
    const int st = s_step;
    float bv = -INFINITY;
    unsigned bi = 0xFFFFFFFFu;
    int nf = 0;
    for (int c = 0; c < C; ++c) {
        const float v = cand_v[(size_t)b * C + c];
        const unsigned i = cand_i[(size_t)b * C + c];
        nf |= cand_nf[(size_t)b * C + c];
        if (v > bv || (v == bv && i < bi)) {
            bv = v;
            bi = i;
        }
    }
    const uint32_t ch = nf ? 0xFFFFFFFFu : bi;
    if (tokens_out) tokens_out[(size_t)st * B + b] = ch;
    last[b] = ch;
    pos[b] += 1;
    if (nf) atomicCAS(status, 0, (int)kDevNonfinite);
    __syncthreads();
    if (b == 0) *step = st + 1;
}

// Every session back to position p with no previous choice.
__global__ void batch_rewind_kernel(int* __restrict__ pos, uint32_t* __restrict__ last, int p, int B) {
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b < B) {
        pos[b] = p;
        last[b] = 0xFFFFFFFFu;
    }
}

}  // namespace
}  // namespace gpt2

// ---------------------------------------------------------------- host side
struct gpt2_batch {
    gpt2_model* m;
    int B;
    int v_pad;              // vocabulary rounded up to the GEMM's 64-column tiles
    size_t session_words;   // cache words of one session (max_pos rows)
    float* d_cache;         // [B][max_pos][L][2d]
    float* X = nullptr;     // [B][d] residual rows
    float* A = nullptr;     // [B][d] projection input and its TF32 remainder
    float* Alo = nullptr;
    float* QKV = nullptr;   // [B][3d]
    float* U = nullptr;     // [B][d_ff] GELU output and remainder
    float* Ulo = nullptr;
    float* part = nullptr;  // split-K partials of the block projections
    float* vpart = nullptr; // [B][v_pad] vocabulary products
    float* cand = nullptr;  // [3][B][chunks] greedy candidates of the logits chunks (value, index, non-finite)
    int* d_pos = nullptr;   // [B] positions
    uint32_t* d_last = nullptr;  // [B] previous greedy choices
    int* d_words = nullptr;      // [0] status, [1] step counter
    std::vector<uint32_t> pos;   // host copy of the positions
    cudaStream_t cs = nullptr, last = nullptr;
    cudaEvent_t ev_in = nullptr, ev_out = nullptr;
    cudaGraphExec_t exec = nullptr;
    const void* key[4] = {};
};

namespace gpt2 {
namespace {

constexpr int kBatchMaxSplits = 16;

// Every launch of one batched step on stream st.  Each kernel after the
// first is a programmatic dependent launch (chain.cuh): 16 / 64 / 256
// sessions measured 593 / 735 / 1,373 against 617 / 778 / 1,432 us per step
// with plain launches.
cudaError_t batch_launches(gpt2_batch* bt, const uint32_t* d_tokens_in, float* d_logits, size_t stride,
                           uint32_t* d_tokens_out, cudaStream_t st) {
    gpt2_model* m = bt->m;
    const gpt2_config& c = m->cfg;
    const int D = (int)c.d_model, FF = (int)c.d_ff, L = (int)c.n_layer, H = (int)c.n_head, DH = D / H;
    const int B = bt->B;
    const float* P = m->d_packed;
    int* status = bt->d_words;
    cudaError_t e = cudaSuccess;

    auto gemm = [&](const float* A, const float* Alo, int K, int N, int l, int mat, int* sp) {
        const uint64_t off = (uint64_t)l * m->layer_bytes + m->mat_off[mat];
        const float* W = reinterpret_cast<const float*>(m->d_wstream + off);
        const float* Wlo = reinterpret_cast<const float*>(reinterpret_cast<const uint8_t*>(m->d_wlo) + off);
        return tc_gemm(A, Alo, B, W, Wlo, N, K, N, kBatchMaxSplits, sp, bt->part, status, st, true);
    };
    auto reduce = [&](int splits, int N, uint64_t bias_off, int kind, float* out, float* out_lo, int l) {
        const size_t total = (size_t)B * N;
        const int blocks = (int)((total + 255) / 256 < 4096 ? (total + 255) / 256 : 4096);
        return chain_launch(true, reduce_kernel, dim3(blocks), dim3(256), 0, st, (const float*)bt->part, splits, B, N,
                            P + bias_off, kind, out, out_lo, bt->X, bt->d_cache, L, l, D, (const int*)bt->d_pos,
                            bt->session_words);
    };
    auto ln = [&](uint64_t g_off, uint64_t b_off, int splits, uint64_t bias_off) {
        return chain_launch(true, ln_split_kernel, dim3(B), dim3(kLnThreads), 0, st, bt->X, P + g_off, P + b_off, D,
                            bt->A, bt->Alo, (const float*)(splits ? bt->part : nullptr), splits, B, P + bias_off);
    };

    // the first kernel of the chain: a plain launch after the previous step
    e = chain_launch(false, batch_embed_kernel, dim3(B), dim3(256), 0, st, P, m->wte_off, m->wpe_off, d_tokens_in,
                     (const int*)(bt->d_words + 1), (const uint32_t*)bt->d_last, (const int*)bt->d_pos, D, c.vocab,
                     bt->X, status);
    if (e == cudaSuccess) e = ln(m->lp[0].ln1_g, m->lp[0].ln1_b, 0, 0);
    int sp = 1;
    for (int l = 0; l < L && e == cudaSuccess; ++l) {
        const LayerParams& lp = m->lp[l];
        if ((e = gemm(bt->A, bt->Alo, D, 3 * D, l, kQKV, &sp)) != cudaSuccess) break;
        if ((e = reduce(sp, 3 * D, lp.b_qkv, kRedQKV, bt->QKV, nullptr, l)) != cudaSuccess) break;
        const dim3 agrid(H, B);
        auto attn = DH == 64 ? batch_attention_kernel<64> : DH == 32 ? batch_attention_kernel<32>
                                                                     : batch_attention_kernel<16>;
        if ((e = chain_launch(true, attn, agrid, dim3(kBAttnThreads), 0, st, (const float*)bt->QKV,
                              (const float*)bt->d_cache, bt->session_words, (const int*)bt->d_pos, L, l, D, bt->A,
                              bt->Alo)) != cudaSuccess)
            break;
        if ((e = gemm(bt->A, bt->Alo, D, D, l, kO, &sp)) != cudaSuccess) break;
        if ((e = ln(lp.ln2_g, lp.ln2_b, sp, lp.b_o)) != cudaSuccess) break;  // residual + LN2
        if ((e = gemm(bt->A, bt->Alo, D, FF, l, kFC, &sp)) != cudaSuccess) break;
        if ((e = reduce(sp, FF, lp.b_fc, kRedGelu, bt->U, bt->Ulo, l)) != cudaSuccess) break;
        if ((e = gemm(bt->U, bt->Ulo, FF, D, l, kP, &sp)) != cudaSuccess) break;
        if (l + 1 < L) e = ln(m->lp[l + 1].ln1_g, m->lp[l + 1].ln1_b, sp, lp.b_p);  // residual + next LN1
        else e = ln(m->lnf_g, m->lnf_b, sp, lp.b_p);                              // residual + LN_f
    }
    if (e != cudaSuccess) return e;
    // tied vocabulary projection: logits[b][n] = wte[n] . LN_f(x_b), one split
    int vs = 1;
    e = tc_gemm(bt->A, bt->Alo, B, P + m->wte_off, m->d_wte_lo, (int)c.vocab, D, bt->v_pad, 1, &vs, bt->vpart,
                status, st, true);
    if (e != cudaSuccess) return e;
    const int C = (bt->v_pad + kChoiceChunk - 1) / kChoiceChunk;
    float* cv = bt->cand;
    unsigned* ci = reinterpret_cast<unsigned*>(bt->cand + (size_t)B * C);
    int* cnf = reinterpret_cast<int*>(bt->cand + 2 * (size_t)B * C);
    e = chain_launch(true, batch_logits_kernel, dim3(C, B), dim3(kBChoiceThreads), 0, st, (const float*)bt->vpart, vs,
                     bt->v_pad, (int)c.vocab, d_logits, stride, (const int*)(bt->d_words + 1), cv, ci, cnf);
    if (e != cudaSuccess) return e;
    return chain_launch(true, batch_pick_kernel, dim3(1), dim3(B), 0, st, (const float*)cv, (const unsigned*)ci,
                        (const int*)cnf, C, d_tokens_out, bt->d_last, bt->d_pos, bt->d_words + 1, status);
}

gpt2_status batch_status(cudaError_t e) {
    if (e == cudaSuccess) return GPT2_OK;
    return e == cudaErrorMemoryAllocation ? GPT2_ERR_NOMEM : GPT2_ERR_CUDA;
}

}  // namespace
}  // namespace gpt2

using namespace gpt2;

extern "C" {

gpt2_status gpt2_batch_create(gpt2_model* m, uint32_t n_sessions, gpt2_batch** out) {
    if (!m || !out) return GPT2_ERR_ARG;
    *out = nullptr;
    const gpt2_config& c = m->cfg;
    if (m->quant != GPT2_F32 || !prefill_shape_supported(c)) return GPT2_ERR_CONFIG;
    if (n_sessions == 0 || n_sessions > GPT2_BATCH_MAX) return GPT2_ERR_ARG;
    if (!tc_ready()) return GPT2_ERR_CUDA;
    gpt2_batch* bt = new (std::nothrow) gpt2_batch();
    if (!bt) return GPT2_ERR_NOMEM;
    bt->m = m;
    bt->B = (int)n_sessions;
    bt->v_pad = (int)((c.vocab + 63) / 64 * 64);
    bt->session_words = (size_t)c.n_layer * 2 * c.d_model * c.max_pos;
    bt->pos.assign(n_sessions, 0);
    const size_t B = n_sessions, D = c.d_model, FF = c.d_ff, N = FF > 3 * D ? FF : 3 * D;
    cudaError_t e = cudaStreamCreateWithFlags(&bt->cs, cudaStreamNonBlocking);
    bt->last = bt->cs;
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&bt->ev_in, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&bt->ev_out, cudaEventDisableTiming);
    if (e == cudaSuccess) e = prefill_make_lo(m, bt->cs);
    if (e == cudaSuccess && !m->d_wte_lo) {
        e = cudaMalloc(&m->d_wte_lo, sizeof(float) * c.vocab * D);
        if (e == cudaSuccess) e = split_lo(m->d_packed + m->wte_off, m->d_wte_lo, (size_t)c.vocab * D, bt->cs);
    }
    if (e == cudaSuccess) e = cudaMalloc(&bt->d_cache, sizeof(float) * B * bt->session_words);
    if (e == cudaSuccess) e = cudaMemset(bt->d_cache, 0, sizeof(float) * B * bt->session_words);
    if (e == cudaSuccess) e = cudaMalloc(&bt->X, sizeof(float) * B * D);
    if (e == cudaSuccess) e = cudaMalloc(&bt->A, sizeof(float) * B * D);
    if (e == cudaSuccess) e = cudaMalloc(&bt->Alo, sizeof(float) * B * D);
    if (e == cudaSuccess) e = cudaMalloc(&bt->QKV, sizeof(float) * B * 3 * D);
    if (e == cudaSuccess) e = cudaMalloc(&bt->U, sizeof(float) * B * FF);
    if (e == cudaSuccess) e = cudaMalloc(&bt->Ulo, sizeof(float) * B * FF);
    if (e == cudaSuccess) e = cudaMalloc(&bt->part, sizeof(float) * kBatchMaxSplits * B * N);
    if (e == cudaSuccess) e = cudaMalloc(&bt->vpart, sizeof(float) * B * bt->v_pad);
    if (e == cudaSuccess)
        e = cudaMalloc(&bt->cand, sizeof(float) * 3 * B * ((bt->v_pad + kChoiceChunk - 1) / kChoiceChunk));
    if (e == cudaSuccess) e = cudaMalloc(&bt->d_pos, sizeof(int) * B);
    if (e == cudaSuccess) e = cudaMemset(bt->d_pos, 0, sizeof(int) * B);
    if (e == cudaSuccess) e = cudaMalloc(&bt->d_last, sizeof(uint32_t) * B);
    if (e == cudaSuccess) e = cudaMemset(bt->d_last, 0xFF, sizeof(uint32_t) * B);
    if (e == cudaSuccess) e = cudaMalloc(&bt->d_words, sizeof(int) * 4);
    if (e == cudaSuccess) e = cudaMemset(bt->d_words, 0, sizeof(int) * 4);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
        gpt2_batch_destroy(bt);
        return batch_status(e);
    }
    *out = bt;
    return GPT2_OK;
}

void gpt2_batch_destroy(gpt2_batch* bt) {
    if (!bt) return;
    if (bt->last) cudaStreamSynchronize(bt->last);
    if (bt->cs) cudaStreamSynchronize(bt->cs);
    if (bt->exec) cudaGraphExecDestroy(bt->exec);
    if (bt->ev_in) cudaEventDestroy(bt->ev_in);
    if (bt->ev_out) cudaEventDestroy(bt->ev_out);
    if (bt->cs) cudaStreamDestroy(bt->cs);
    cudaFree(bt->d_cache);
    cudaFree(bt->X);
    cudaFree(bt->A);
    cudaFree(bt->Alo);
    cudaFree(bt->QKV);
    cudaFree(bt->U);
    cudaFree(bt->Ulo);
    cudaFree(bt->part);
    cudaFree(bt->vpart);
    cudaFree(bt->cand);
    cudaFree(bt->d_pos);
    cudaFree(bt->d_last);
    cudaFree(bt->d_words);
    delete bt;
}

uint32_t gpt2_batch_size(const gpt2_batch* bt) { return bt ? (uint32_t)bt->B : 0; }

uint32_t gpt2_batch_position(const gpt2_batch* bt, uint32_t index) {
    return (bt && index < (uint32_t)bt->B) ? bt->pos[index] : 0;
}

gpt2_status gpt2_batch_load_cache(gpt2_batch* bt, uint32_t index, const void* cache, size_t len) {
    if (!bt || index >= (uint32_t)bt->B || (!cache && len)) return GPT2_ERR_ARG;
    const gpt2_config& c = bt->m->cfg;
    const size_t rowb = (size_t)c.n_layer * 2 * c.d_model * 4;
    if (len % rowb || len / rowb >= c.max_pos) return GPT2_ERR_CACHE_LEN;
    cudaError_t e = cudaStreamSynchronize(bt->last);
    if (e == cudaSuccess && len)
        e = cudaMemcpy(bt->d_cache + (size_t)index * bt->session_words, cache, len, cudaMemcpyHostToDevice);
    const int p = (int)(len / rowb);
    const uint32_t none = 0xFFFFFFFFu;
    if (e == cudaSuccess) e = cudaMemcpy(bt->d_pos + index, &p, sizeof(int), cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaMemcpy(bt->d_last + index, &none, sizeof(uint32_t), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return batch_status(e);
    bt->pos[index] = (uint32_t)p;
    return GPT2_OK;
}

gpt2_status gpt2_batch_read_cache(gpt2_batch* bt, uint32_t index, void* out, size_t capacity, size_t* len) {
    if (!bt || !len || index >= (uint32_t)bt->B) return GPT2_ERR_ARG;
    *len = 0;
    const gpt2_config& c = bt->m->cfg;
    const size_t bytes = (size_t)c.n_layer * 2 * c.d_model * 4 * bt->pos[index];
    if (capacity < bytes || (!out && bytes)) return GPT2_ERR_ARG;
    cudaError_t e = cudaStreamSynchronize(bt->last);
    if (e == cudaSuccess && bytes)
        e = cudaMemcpy(out, bt->d_cache + (size_t)index * bt->session_words, bytes, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return batch_status(e);
    *len = bytes;
    return GPT2_OK;
}

gpt2_status gpt2_batch_run(gpt2_batch* bt, const uint32_t* d_tokens_in, uint32_t n_steps, float* d_logits,
                           size_t stride, uint32_t* d_tokens_out, void* stream) {
    if (!bt || !d_tokens_in) return GPT2_ERR_ARG;
    if (n_steps == 0) return GPT2_ERR_TOKENS_LEN;
    const uint32_t max_pos = bt->m->cfg.max_pos;
    for (int b = 0; b < bt->B; ++b)
        if ((uint64_t)bt->pos[b] + n_steps > max_pos) return GPT2_ERR_POSITION;
    if (d_logits && stride && stride < (size_t)bt->B * bt->m->cfg.vocab) return GPT2_ERR_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaSuccess;
    const void* key[4] = {d_tokens_in, d_logits, reinterpret_cast<const void*>(stride), d_tokens_out};
    bool same = bt->exec != nullptr;
    for (int i = 0; i < 4 && same; ++i) same = key[i] == bt->key[i];
    if (!same) {
        if (bt->exec) {
            cudaGraphExecDestroy(bt->exec);
            bt->exec = nullptr;
        }
        cudaGraph_t graph = nullptr;
        e = cudaStreamBeginCapture(bt->cs, cudaStreamCaptureModeThreadLocal);
        if (e != cudaSuccess) return batch_status(e);
        const cudaError_t el = batch_launches(bt, d_tokens_in, d_logits, stride, d_tokens_out, bt->cs);
        e = cudaStreamEndCapture(bt->cs, &graph);
        if (el != cudaSuccess) e = el;
        if (e == cudaSuccess) e = cudaGraphInstantiate(&bt->exec, graph, 0);
        if (graph) cudaGraphDestroy(graph);
        if (e != cudaSuccess) {
            bt->exec = nullptr;
            return batch_status(e);
        }
        for (int i = 0; i < 4; ++i) bt->key[i] = key[i];
    }
    e = cudaEventRecord(bt->ev_in, st);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(bt->cs, bt->ev_in, 0);
    if (e == cudaSuccess) e = cudaMemsetAsync(bt->d_words + 1, 0, sizeof(int), bt->cs);  // step counter
    for (uint32_t s = 0; s < n_steps && e == cudaSuccess; ++s) e = cudaGraphLaunch(bt->exec, bt->cs);
    if (e == cudaSuccess) e = cudaEventRecord(bt->ev_out, bt->cs);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(st, bt->ev_out, 0);
    if (e != cudaSuccess) return batch_status(e);
    for (int b = 0; b < bt->B; ++b) bt->pos[b] += n_steps;
    bt->last = st;
    return GPT2_OK;
}

gpt2_status gpt2_batch_rewind(gpt2_batch* bt, uint32_t position, void* stream) {
    if (!bt) return GPT2_ERR_ARG;
    for (int b = 0; b < bt->B; ++b)
        if (bt->pos[b] < position) return GPT2_ERR_POSITION;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    batch_rewind_kernel<<<(bt->B + 255) / 256, 256, 0, st>>>(bt->d_pos, bt->d_last, (int)position, bt->B);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return batch_status(e);
    for (int b = 0; b < bt->B; ++b) bt->pos[b] = position;
    bt->last = st;
    return GPT2_OK;
}

gpt2_status gpt2_batch_sync(gpt2_batch* bt) {
    if (!bt) return GPT2_ERR_ARG;
    cudaError_t e = cudaStreamSynchronize(bt->last);
    if (e == cudaSuccess) e = cudaStreamSynchronize(bt->cs);
    if (e != cudaSuccess) return batch_status(e);
    int w = 0;
    e = cudaMemcpy(&w, bt->d_words, sizeof(int), cudaMemcpyDeviceToHost);
    if (e == cudaSuccess && w) e = cudaMemset(bt->d_words, 0, sizeof(int));
    if (e != cudaSuccess) return batch_status(e);
    return (gpt2_status)w;
}

}  // extern "C"
