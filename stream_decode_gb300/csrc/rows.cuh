// rows.cuh -- row-wise kernels shared by the tensor-core paths (the prompt
// prefill and the batched decode step): TF32 splitting, LayerNorm (with
// the preceding residual add), the split-K reduce with its epilogues, and
// the greedy-choice rule.  Everything here has internal linkage; each
// translation unit that includes it gets its own copy.
#pragma once
#include <cuda_runtime.h>

#include <cstdint>

#include "chain.cuh"
#include "gpt2_dev.cuh"

namespace gpt2 {
namespace {

__device__ __forceinline__ float tf32_hi(float x) { return __uint_as_float(__float_as_uint(x) & ~0x1FFFu); }
__device__ __forceinline__ float tf32_lo(float x) { return __fsub_rn(x, tf32_hi(x)); }

__device__ __forceinline__ float warp_sum32(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ float warp_max32(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float gelu(float x) {
    const float inner = 0.7978845608f * (x + 0.044715f * x * x * x);
    return 0.5f * x * (1.0f + tanhf(inner));
}

// lo[i] = w[i] - hi(w[i]) over n floats.
__global__ void split_lo_kernel(const float* __restrict__ w, float* __restrict__ lo, size_t n) {
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
        lo[i] = tf32_lo(w[i]);
}

// X[i][:] = wte[tok_i] + wpe[i]; an out-of-range token sets the status and
// leaves its row unwritten.
__global__ void embed_kernel(const float* __restrict__ packed, uint64_t wte_off, uint64_t wpe_off,
                             const uint32_t* __restrict__ tok, int D, uint32_t vocab, float* __restrict__ X,
                             int* status) {
    chain_enter();
    const int i = blockIdx.x;
    const uint32_t t = tok[i];
    if (t >= vocab) {
        if (threadIdx.x == 0) atomicCAS(status, 0, (int)kDevToken);
        return;
    }
    for (int j = threadIdx.x; j < D; j += blockDim.x)
        X[(size_t)i * D + j] = __fadd_rn(packed[wte_off + (uint64_t)t * D + j], packed[wpe_off + (uint64_t)i * D + j]);
}

constexpr int kLnThreads = 256;

// Y = LN(X) (mean, then the biased variance of the deviations; eps 1e-5)
// and its TF32 remainder, one block of 256 threads per row (up to 8 values a
// thread: D <= 2048).
// With part != nullptr the row is first completed as the residual add of a
// projection: X[i][j] += (sum over splits s = 0, 1, ... of part[s][i][j]) +
// bias[j], in the split reduce's order, and written back.
__global__ void __launch_bounds__(kLnThreads) ln_split_kernel(float* __restrict__ X, const float* __restrict__ g,
                                                             const float* __restrict__ b, int D,
                                                             float* __restrict__ Y, float* __restrict__ Ylo,
                                                             const float* __restrict__ part, int splits, int n,
                                                             const float* __restrict__ bias) {
    __shared__ float red[kLnThreads / 32];
    chain_enter();
    const int row = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    float* x = X + (size_t)row * D;
    float v[8];
    if (part) {
        // split sums in split order; eight splits' loads are issued together
        float y[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) y[k] = 0.0f;
        int sp = 0;
        for (; sp + 8 <= splits; sp += 8) {
            float a[8][8];
#pragma unroll
            for (int u = 0; u < 8; ++u)
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const int i = tid + kLnThreads * k;
                    a[u][k] = i < D ? part[((size_t)(sp + u) * n + row) * D + i] : 0.0f;
                }
#pragma unroll
            for (int u = 0; u < 8; ++u)
#pragma unroll
                for (int k = 0; k < 8; ++k) y[k] += a[u][k];
        }
        for (; sp < splits; ++sp)
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int i = tid + kLnThreads * k;
                if (i < D) y[k] += part[((size_t)sp * n + row) * D + i];
            }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int i = tid + kLnThreads * k;
            v[k] = 0.0f;
            if (i < D) {
                v[k] = __fadd_rn(x[i], __fadd_rn(y[k], bias[i]));
                x[i] = v[k];
            }
        }
    } else {
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int i = tid + kLnThreads * k;
            v[k] = i < D ? x[i] : 0.0f;
        }
    }
    float s = 0.0f;
#pragma unroll
    for (int k = 0; k < 8; ++k) s += v[k];
    s = warp_sum32(s);
    if (lane == 0) red[warp] = s;
    __syncthreads();
    float t = 0.0f;
#pragma unroll
    for (int w = 0; w < kLnThreads / 32; ++w) t += red[w];
    const float mean = t / (float)D;
    __syncthreads();
    float q = 0.0f;
#pragma unroll
    for (int k = 0; k < 8; ++k)
        if (tid + kLnThreads * k < D) {
            const float d = v[k] - mean;
            q = fmaf(d, d, q);
        }
    q = warp_sum32(q);
    if (lane == 0) red[warp] = q;
    __syncthreads();
    float u = 0.0f;
#pragma unroll
    for (int w = 0; w < kLnThreads / 32; ++w) u += red[w];
    const float den = sqrtf(u / (float)D + kLnEps);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const int i = tid + kLnThreads * k;
        if (i < D) {
            const float y = (v[k] - mean) / den * g[i] + b[i];
            Y[(size_t)row * D + i] = y;
            Ylo[(size_t)row * D + i] = tf32_lo(y);
        }
    }
}

enum ReduceKind : int { kRedQKV = 0, kRedResidual = 1, kRedGelu = 2 };

// y[i][j] = (sum over splits s = 0, 1, ... of part[s][i][j]) + bias[j], then
// QKV: out[i][j] = y and, for key/value columns, a KV-cache word: with
// pos == nullptr row i is prompt position i of one cache; otherwise row i
// is session i, whose cache starts session_words words after the previous
// one, at position pos[i]; residual: X[i][j] += y; GELU: out = gelu(y) and
// its remainder.
__global__ void reduce_kernel(const float* __restrict__ part, int splits, int n, int N,
                              const float* __restrict__ bias, int kind, float* __restrict__ out,
                              float* __restrict__ out_lo, float* __restrict__ X, float* __restrict__ cache, int L,
                              int l, int D, const int* __restrict__ pos, size_t session_words) {
    chain_enter();
    const size_t total = (size_t)n * N;
    for (size_t idx = blockIdx.x * (size_t)blockDim.x + threadIdx.x; idx < total;
         idx += (size_t)gridDim.x * blockDim.x) {
        const int i = (int)(idx / N), j = (int)(idx - (size_t)i * N);
        float y = 0.0f;
        for (int s = 0; s < splits; ++s) y += part[((size_t)s * n + i) * N + j];
        y = __fadd_rn(y, bias[j]);
        if (kind == kRedQKV) {
            out[idx] = y;
            if (j >= D) {
                const size_t row = pos ? (size_t)i * session_words + ((size_t)pos[i] * L + l) * 2 * D
                                       : ((size_t)i * L + l) * 2 * D;
                cache[row + (j - D)] = y;
            }
        } else if (kind == kRedResidual) {
            X[idx] = __fadd_rn(X[idx], y);
        } else {
            const float u = gelu(y);
            out[idx] = u;
            out_lo[idx] = tf32_lo(u);
        }
    }
}

// Greedy choice rule: largest value, lowest index on ties; a non-finite
// value sets nf.
__device__ __forceinline__ void choice_take(float x, unsigned j, float& bv, unsigned& bi, int& nf) {
    if (!isfinite(x)) nf = 1;
    else if (x > bv || (x == bv && j < bi)) { bv = x; bi = j; }
}
}  // namespace
}  // namespace gpt2
