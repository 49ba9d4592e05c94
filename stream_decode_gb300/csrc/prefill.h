// prefill.h -- the tensor-core prompt prefill (full-prefix forward pass)
// shared between prefill.cu and the C ABI in api.cu.
#pragma once
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "../../include/gpt2.h"

struct gpt2_model;

namespace gpt2 {

constexpr int kPrefillMaxSplits = 16;  // K splits of one projection at most

// Per-session prefill workspace for up to `cap` prompt rows.
struct PrefillWs {
    int cap = 0;
    float* X = nullptr;     // [cap][d] residual stream
    float* A = nullptr;     // [cap][d] projection input (LN output or attention output)
    float* Alo = nullptr;   // its TF32 remainder
    float* QKV = nullptr;   // [cap][3d]
    float* U = nullptr;     // [cap][d_ff] GELU output
    float* Ulo = nullptr;   // its TF32 remainder
    float* part = nullptr;  // split-K partial tiles
    // The prefill's launches, captured once per (model, buffers, length) and
    // replayed as one CUDA graph on the workspace's stream, ordered after and
    // before the caller's stream by events.
    cudaGraphExec_t exec = nullptr;
    cudaStream_t cs = nullptr;
    cudaEvent_t ev_in = nullptr, ev_out = nullptr;
    const void* key[9] = {};
};

bool prefill_shape_supported(const gpt2_config& c);

// The 3xTF32 tensor-core GEMM shared by the prefill and the batched decode
// step.  tc_ready() looks up the tensor-map encoder and the SM count once
// and sets the kernel's shared-memory size; false if either is missing.
bool tc_ready();
int tc_sm_count();
// part[split][m][n] for m < m_rows, n < N: the split's K range of
// A[m][:] . W[n][:] with both operands K-major binary32 ([rows][K]) and
// their TF32 remainders Alo, Wlo beside them.  W has w_rows <= N rows; the
// columns n >= w_rows read zeros.  K a multiple of 32, N of 64; base
// addresses 16-byte aligned.  *splits_out = the number of K splits chosen
// (at most max_splits); part holds splits x m_rows x N floats.  pdl: a
// programmatic dependent launch (chain.cuh) after the kernel before it on st.
cudaError_t tc_gemm(const float* A, const float* Alo, int m_rows, const float* W, const float* Wlo, int w_rows, int K,
                    int N, int max_splits, int* splits_out, float* part, int* status, cudaStream_t st, bool pdl);
// lo[i] = w[i] - (w[i] with its low 13 mantissa bits cleared), i < n.
cudaError_t split_lo(const float* w, float* lo, size_t n, cudaStream_t st);
// The model's block-matrix TF32 remainders (made once, on stream st).
cudaError_t prefill_make_lo(gpt2_model* m, cudaStream_t st);
cudaError_t prefill_alloc(PrefillWs* w, int cap, int D, int FF);
void prefill_free(PrefillWs* w);
// Enqueues the prefill of n device token ids; writes cache rows 0..n-1,
// the logits of row n-1, the greedy choice of those logits into *d_choice
// (0xFFFFFFFF and status GPT2_ERR_NONFINITE-coded if any logit is not
// finite) and, if d_next is not null, into *d_next too.
cudaError_t prefill_enqueue(gpt2_model* m, PrefillWs* w, const uint32_t* d_tok, int n, float* cache, float* logits,
                            int* status, uint32_t* d_choice, uint32_t* d_next, cudaStream_t st);

}  // namespace gpt2
