// repack.cu -- load-time construction of the device weight streams.
//
// The packed checkpoint stores block matrices [in][out] (gpt2.s page,
// weight-layout paragraph).  The step kernel wants each output's weights
// contiguous (K-major rows) so that a CTA's share of outputs is one byte
// range.  binary32 models get a transposed copy, binary16 models a
// transposed copy rounded to nearest-even half precision (and a binary16
// copy of the tied embedding); int8 models get, per output
// row, K int8 codes followed by the K/64 group scales (padded to 16 bytes),
// quantized with the rule of the quantized GPT-2 abstract: scale =
// maxabs/127 over 64 consecutive inputs of the row, nearest-even, saturate
// (or, with per-row weight scales, one scale over the whole row, repeated
// in every group slot).
#include <cuda_runtime.h>

#include "gpt2_dev.cuh"

namespace gpt2 {

// src [K][N] row-major -> dst rows of N outputs, each K floats (row pitch rb bytes).
__global__ void transpose_kernel(const float* __restrict__ src, uint8_t* __restrict__ dst, int K, int N, int rb) {
    __shared__ float tile[32][33];
    const int n0 = blockIdx.x * 32, k0 = blockIdx.y * 32;
    for (int dy = threadIdx.y; dy < 32; dy += blockDim.y) {
        const int k = k0 + dy, n = n0 + threadIdx.x;
        tile[dy][threadIdx.x] = (k < K && n < N) ? src[(size_t)k * N + n] : 0.0f;
    }
    __syncthreads();
    for (int dy = threadIdx.y; dy < 32; dy += blockDim.y) {
        const int n = n0 + dy, k = k0 + threadIdx.x;
        if (n < N && k < K) reinterpret_cast<float*>(dst + (size_t)n * rb)[k] = tile[threadIdx.x][dy];
    }
}

// The same into rows of K binary16 values (nearest-even).
__global__ void transpose_f16_kernel(const float* __restrict__ src, uint8_t* __restrict__ dst, int K, int N, int rb) {
    __shared__ float tile[32][33];
    const int n0 = blockIdx.x * 32, k0 = blockIdx.y * 32;
    for (int dy = threadIdx.y; dy < 32; dy += blockDim.y) {
        const int k = k0 + dy, n = n0 + threadIdx.x;
        tile[dy][threadIdx.x] = (k < K && n < N) ? src[(size_t)k * N + n] : 0.0f;
    }
    __syncthreads();
    for (int dy = threadIdx.y; dy < 32; dy += blockDim.y) {
        const int n = n0 + dy, k = k0 + threadIdx.x;
        if (n < N && k < K) reinterpret_cast<__half*>(dst + (size_t)n * rb)[k] = __float2half_rn(tile[threadIdx.x][dy]);
    }
}

// Rows already K-major (the tied wte [N][K]) to binary16 rows.
__global__ void to_f16_kernel(const float* __restrict__ src, __half* __restrict__ dst, size_t n) {
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
        dst[i] = __float2half_rn(src[i]);
}

// One thread per (output n, group g): weights W[64g .. 64g+63][n] of a [K][N] matrix.
__global__ void quantize_in_out_kernel(const float* __restrict__ src, uint8_t* __restrict__ dst, int K, int N,
                                       int rb) {
    const int n = blockIdx.x * blockDim.x + threadIdx.x;
    const int g = blockIdx.y;
    if (n >= N) return;
    float m = 0.0f;
    for (int t = 0; t < kGroup; ++t) {
        const float a = fabsf(src[(size_t)(g * kGroup + t) * N + n]);
        if (a > m) m = a;
    }
    const float s = __fdiv_rn(m, 127.0f);
    int8_t* q = reinterpret_cast<int8_t*>(dst + (size_t)n * rb);
    for (int t = 0; t < kGroup; ++t) q[g * kGroup + t] = (int8_t)quantize_one(src[(size_t)(g * kGroup + t) * N + n], s);
    reinterpret_cast<float*>(dst + (size_t)n * rb + K)[g] = s;
}

// One thread per (row n, group g) of an [N][K] matrix (the tied wte).
__global__ void quantize_out_in_kernel(const float* __restrict__ src, uint8_t* __restrict__ dst, int K, int N,
                                       int rb) {
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const int ng = K / kGroup;
    if (i >= (long long)N * ng) return;
    const int n = (int)(i / ng), g = (int)(i % ng);
    const float* row = src + (size_t)n * K + g * kGroup;
    float m = 0.0f;
    for (int t = 0; t < kGroup; ++t) {
        const float a = fabsf(row[t]);
        if (a > m) m = a;
    }
    const float s = __fdiv_rn(m, 127.0f);
    int8_t* q = reinterpret_cast<int8_t*>(dst + (size_t)n * rb);
    for (int t = 0; t < kGroup; ++t) q[g * kGroup + t] = (int8_t)quantize_one(row[t], s);
    reinterpret_cast<float*>(dst + (size_t)n * rb + K)[g] = s;
}

// Per-row weight scales, one thread per output n of a [K][N] matrix: one
// scale for the row's K weights (maxabs / 127), written to each of the K/64
// group slots, so the grouped kernels read it unchanged.
__global__ void quantize_in_out_row_kernel(const float* __restrict__ src, uint8_t* __restrict__ dst, int K, int N,
                                           int rb) {
    const int n = blockIdx.x * blockDim.x + threadIdx.x;
    if (n >= N) return;
    float m = 0.0f;
    for (int k = 0; k < K; ++k) {
        const float a = fabsf(src[(size_t)k * N + n]);
        if (a > m) m = a;
    }
    const float s = __fdiv_rn(m, 127.0f);
    int8_t* q = reinterpret_cast<int8_t*>(dst + (size_t)n * rb);
    for (int k = 0; k < K; ++k) q[k] = (int8_t)quantize_one(src[(size_t)k * N + n], s);
    for (int g = 0; g < K / kGroup; ++g) reinterpret_cast<float*>(dst + (size_t)n * rb + K)[g] = s;
}

// The same for the rows of an [N][K] matrix (the tied wte), one thread per row.
__global__ void quantize_out_in_row_kernel(const float* __restrict__ src, uint8_t* __restrict__ dst, int K, int N,
                                           int rb) {
    const int n = blockIdx.x * blockDim.x + threadIdx.x;
    if (n >= N) return;
    const float* row = src + (size_t)n * K;
    float m = 0.0f;
    for (int k = 0; k < K; ++k) {
        const float a = fabsf(row[k]);
        if (a > m) m = a;
    }
    const float s = __fdiv_rn(m, 127.0f);
    int8_t* q = reinterpret_cast<int8_t*>(dst + (size_t)n * rb);
    for (int k = 0; k < K; ++k) q[k] = (int8_t)quantize_one(row[k], s);
    for (int g = 0; g < K / kGroup; ++g) reinterpret_cast<float*>(dst + (size_t)n * rb + K)[g] = s;
}

// The LayerNorm folds of one K-major matrix (rows of K binary32 or binary16
// values, the latter the model's weights as stored):
// c_j = sum_i W_ji g_i and d_j = bias_j + sum_i W_ji b_i, one warp per
// row, summed in binary64 and rounded once.
template <typename T>
__global__ void fold_kernel(const uint8_t* __restrict__ rows, int K, int N, const float* __restrict__ g,
                            const float* __restrict__ b, const float* __restrict__ bias, float* __restrict__ c_out,
                            float* __restrict__ d_out) {
    const int j = (int)((blockIdx.x * (size_t)blockDim.x + threadIdx.x) >> 5), lane = threadIdx.x & 31;
    if (j >= N) return;
    const T* w = reinterpret_cast<const T*>(rows) + (size_t)j * K;
    double c = 0.0, d = 0.0;
    for (int i = lane; i < K; i += 32) {
        const double wi = (double)(float)w[i];
        c += wi * (double)g[i];
        d += wi * (double)b[i];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        c += __shfl_xor_sync(0xffffffffu, c, o);
        d += __shfl_xor_sync(0xffffffffu, d, o);
    }
    if (lane == 0) {
        c_out[j] = (float)c;
        d_out[j] = (float)((double)bias[j] + d);
    }
}

cudaError_t fold_rows(const uint8_t* rows, int K, int N, int wf, const float* g, const float* b, const float* bias,
                      float* c, float* d, cudaStream_t st) {
    const int threads = 256, per_block = threads / 32;
    if (wf == kWF16)
        fold_kernel<__half><<<(N + per_block - 1) / per_block, threads, 0, st>>>(rows, K, N, g, b, bias, c, d);
    else
        fold_kernel<float><<<(N + per_block - 1) / per_block, threads, 0, st>>>(rows, K, N, g, b, bias, c, d);
    return cudaGetLastError();
}

cudaError_t rows_to_f16(const float* src, uint8_t* dst, size_t n, cudaStream_t st) {
    to_f16_kernel<<<1024, 256, 0, st>>>(src, reinterpret_cast<__half*>(dst), n);
    return cudaGetLastError();
}

cudaError_t repack_matrix(const float* src_in_out, uint8_t* dst, int K, int N, int wf, bool per_row,
                          cudaStream_t st) {
    const int rb = row_bytes(K, wf);
    if (wf == kWQ8 && per_row) {
        quantize_in_out_row_kernel<<<(N + 127) / 128, 128, 0, st>>>(src_in_out, dst, K, N, rb);
        return cudaGetLastError();
    }
    if (wf == kWF32) {
        dim3 grid((N + 31) / 32, (K + 31) / 32), block(32, 8);
        transpose_kernel<<<grid, block, 0, st>>>(src_in_out, dst, K, N, rb);
    } else if (wf == kWF16) {
        dim3 grid((N + 31) / 32, (K + 31) / 32), block(32, 8);
        transpose_f16_kernel<<<grid, block, 0, st>>>(src_in_out, dst, K, N, rb);
    } else {
        dim3 grid((N + 127) / 128, K / kGroup), block(128);
        quantize_in_out_kernel<<<grid, block, 0, st>>>(src_in_out, dst, K, N, rb);
    }
    return cudaGetLastError();
}

cudaError_t quantize_rows(const float* src_out_in, uint8_t* dst, int K, int N, bool per_row, cudaStream_t st) {
    const int rb = row_bytes(K, kWQ8);
    if (per_row) {
        quantize_out_in_row_kernel<<<(N + 127) / 128, 128, 0, st>>>(src_out_in, dst, K, N, rb);
        return cudaGetLastError();
    }
    const long long n = (long long)N * (K / kGroup);
    quantize_out_in_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(src_out_in, dst, K, N, rb);
    return cudaGetLastError();
}

}  // namespace gpt2
