// prefill.cu -- the full-prefix forward pass of a prompt ("infer", LeanExe
// GPT-2 README, infer paragraph) on the tensor cores, writing the session's
// KV cache for every prompt position on the way.
//
// Per layer: LN1 -> QKV projection (+ KV-cache rows) -> causal attention ->
// out-projection + residual -> LN2 -> FC + GELU -> MLP projection +
// residual; then LN_f and the tied vocabulary projection of the last row
// only.  The four projections are 3xTF32 tcgen05 GEMMs (tc_gemm.cuh) over
// 128-row x 64-column tiles, split along K over about two thirds of the
// SMs; the splits are summed in split order by the projection's epilogue
// kernel (QKV + KV-cache rows; GELU), or, for a residual add, by the
// LayerNorm kernel of the next block input (one row-wise kernel).  Every
// GEMM input is written with its TF32 remainder (x - hi(x)) next to it; the
// weights' remainders are made once per model.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>

#include "gpt2_dev.cuh"
#include "model_internal.h"
#include "prefill.h"
#include "rows.cuh"
#include "tc_gemm.cuh"

namespace gpt2 {

namespace {

constexpr int kAttnWarps = 8;
constexpr int kAttnRows = 8;           // query rows per block (one per warp)
constexpr int kMaxPrefillKeys = 1024;  // longest prompt (the keys of a block are staged in chunks of kKeyTile)
constexpr int kKeyTile = 64;

// Causal attention of head h for query rows [r0, r0 + 16) of the prompt:
// s_j = (q . k_j) / sqrt(dh) over keys j <= i, softmax, o = sum_j a_j v_j.
// The keys and values are staged in shared memory in tiles of 64 (keys
// padded to DH + 1 floats a row: conflict-free reads down a column); each
// warp takes 2 query rows and keeps, per row, the scores of the current
// tile, an online max / sum and its output coordinates (lane, lane + 32).
// Dot products and the weighted value sums run in four independent chains.
template <int DH>
__global__ void __launch_bounds__(kAttnWarps * 32) attention_kernel(const float* __restrict__ QKV, int n, int D,
                                                                    float* __restrict__ O, float* __restrict__ Olo) {
    static_assert(DH % 4 == 0 && DH <= 64, "head width");
    constexpr int DPL = (DH + 31) / 32;  // output coordinates per lane
    __shared__ float ks[kKeyTile][DH + 1];
    __shared__ __align__(16) float vs[kKeyTile][DH];
    __shared__ float qs[kAttnRows][DH];
    __shared__ float ps[kAttnWarps][kKeyTile];
    chain_enter();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int h = blockIdx.x, r0 = blockIdx.y * kAttnRows;
    const size_t N3 = 3 * (size_t)D;
    const float scale = 1.0f / sqrtf((float)DH);
    const int rmax = min(r0 + kAttnRows, n);  // rows r0..rmax-1; keys 0..rmax-1
    for (int i = threadIdx.x; i < kAttnRows * DH; i += blockDim.x) {
        const int r = i / DH, e = i - r * DH;
        qs[r][e] = r0 + r < n ? QKV[(size_t)(r0 + r) * N3 + (size_t)h * DH + e] : 0.0f;
    }
    constexpr int RPW = kAttnRows / kAttnWarps;  // query rows per warp
    float m[RPW], z[RPW], o[RPW][DPL];
#pragma unroll
    for (int t = 0; t < RPW; ++t) {
        m[t] = -INFINITY;
        z[t] = 0.0f;
#pragma unroll
        for (int d = 0; d < DPL; ++d) o[t][d] = 0.0f;
    }
    for (int j0 = 0; j0 < rmax; j0 += kKeyTile) {
        const int jn = min(kKeyTile, rmax - j0);
        __syncthreads();
        for (int i = threadIdx.x; i < jn * (DH / 4); i += blockDim.x) {
            const int j = i / (DH / 4), e = 4 * (i - j * (DH / 4));
            const size_t base = (size_t)(j0 + j) * N3 + (size_t)h * DH + e;
            const float4 kv = *reinterpret_cast<const float4*>(QKV + base + D);
            const float4 vv = *reinterpret_cast<const float4*>(QKV + base + 2 * D);
            ks[j][e] = kv.x;
            ks[j][e + 1] = kv.y;
            ks[j][e + 2] = kv.z;
            ks[j][e + 3] = kv.w;
            *reinterpret_cast<float4*>(&vs[j][e]) = vv;
        }
        __syncthreads();
#pragma unroll
        for (int t = 0; t < RPW; ++t) {
            const int r = warp * RPW + t, i = r0 + r;
            if (i >= n) continue;
            const int kend = min(jn, i - j0 + 1);  // keys of this tile at or before row i
            if (kend <= 0) continue;
            // scores of this tile: lane takes keys lane, lane + 32
            float tmax = -INFINITY;
#pragma unroll
            for (int jj = 0; jj < kKeyTile; jj += 32) {
                const int j = jj + lane;
                if (j < kend) {
                    float d0 = 0.0f, d1 = 0.0f, d2 = 0.0f, d3 = 0.0f;
#pragma unroll
                    for (int e = 0; e < DH; e += 4) {
                        d0 = fmaf(qs[r][e], ks[j][e], d0);
                        d1 = fmaf(qs[r][e + 1], ks[j][e + 1], d1);
                        d2 = fmaf(qs[r][e + 2], ks[j][e + 2], d2);
                        d3 = fmaf(qs[r][e + 3], ks[j][e + 3], d3);
                    }
                    const float sc = ((d0 + d1) + (d2 + d3)) * scale;
                    ps[warp][j] = sc;
                    tmax = fmaxf(tmax, sc);
                }
            }
            tmax = warp_max32(tmax);
            const float mn = fmaxf(m[t], tmax);
            const float corr = expf(m[t] - mn);  // 0 while m is -inf
            float tz = 0.0f;
#pragma unroll
            for (int jj = 0; jj < kKeyTile; jj += 32) {
                const int j = jj + lane;
                if (j < kend) {
                    const float e = expf(ps[warp][j] - mn);
                    ps[warp][j] = e;
                    tz += e;
                }
            }
            tz = warp_sum32(tz);
            __syncwarp();
            // weighted values: four chains over keys j = 4u + c
            float acc[DPL][4];
#pragma unroll
            for (int d = 0; d < DPL; ++d)
#pragma unroll
                for (int c = 0; c < 4; ++c) acc[d][c] = 0.0f;
            int j = 0;
            for (; j + 4 <= kend; j += 4) {
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const float pj = ps[warp][j + c];
#pragma unroll
                    for (int d = 0; d < DPL; ++d)
                        if (lane + 32 * d < DH) acc[d][c] = fmaf(pj, vs[j + c][lane + 32 * d], acc[d][c]);
                }
            }
            for (; j < kend; ++j) {
                const float pj = ps[warp][j];
#pragma unroll
                for (int d = 0; d < DPL; ++d)
                    if (lane + 32 * d < DH) acc[d][0] = fmaf(pj, vs[j][lane + 32 * d], acc[d][0]);
            }
            __syncwarp();
#pragma unroll
            for (int d = 0; d < DPL; ++d)
                o[t][d] = fmaf(o[t][d], corr, (acc[d][0] + acc[d][1]) + (acc[d][2] + acc[d][3]));
            z[t] = fmaf(z[t], corr, tz);
            m[t] = mn;
        }
    }
#pragma unroll
    for (int t = 0; t < RPW; ++t) {
        const int i = r0 + warp * RPW + t;
        if (i >= n) continue;
#pragma unroll
        for (int d = 0; d < DPL; ++d) {
            const int e = lane + 32 * d;
            if (e < DH) {
                const float v = o[t][d] / z[t];
                O[(size_t)i * D + (size_t)h * DH + e] = v;
                Olo[(size_t)i * D + (size_t)h * DH + e] = tf32_lo(v);
            }
        }
    }
}

constexpr int kHeadThreads = 256;

// Greedy choice over the logits (largest value, lowest index on ties; any
// non-finite value makes the choice 0xFFFFFFFF and sets the status).  One
// block of 1024 threads; float4 loads when the logits are 16-byte aligned.
constexpr int kChoiceThreads = 1024;
__global__ void __launch_bounds__(kChoiceThreads) choice_kernel(const float* __restrict__ v, unsigned n,
                                                                uint32_t* choice, uint32_t* next, int* status) {
    __shared__ float s_v[kChoiceThreads / 32];
    __shared__ unsigned s_i[kChoiceThreads / 32];
    __shared__ int s_nf[kChoiceThreads / 32];
    chain_enter();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    float bv = -INFINITY;
    unsigned bi = 0xFFFFFFFFu;
    int nf = 0;
    unsigned done = 0;
    if ((reinterpret_cast<uintptr_t>(v) & 15u) == 0) {
        const unsigned n4 = n / 4;
        const float4* v4 = reinterpret_cast<const float4*>(v);
        for (unsigned q = tid; q < n4; q += kChoiceThreads) {
            const float4 x = v4[q];
            choice_take(x.x, 4 * q, bv, bi, nf);
            choice_take(x.y, 4 * q + 1, bv, bi, nf);
            choice_take(x.z, 4 * q + 2, bv, bi, nf);
            choice_take(x.w, 4 * q + 3, bv, bi, nf);
        }
        done = 4 * n4;
    }
    for (unsigned j = done + tid; j < n; j += kChoiceThreads) choice_take(v[j], j, bv, bi, nf);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const unsigned oi = __shfl_xor_sync(0xffffffffu, bi, o);
        nf |= __shfl_xor_sync(0xffffffffu, nf, o);
        if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
    }
    if (lane == 0) { s_v[warp] = bv; s_i[warp] = bi; s_nf[warp] = nf; }
    __syncthreads();
    if (tid == 0) {
        for (int w = 1; w < kChoiceThreads / 32; ++w) {
            nf |= s_nf[w];
            if (s_v[w] > bv || (s_v[w] == bv && s_i[w] < bi)) { bv = s_v[w]; bi = s_i[w]; }
        }
        const uint32_t c = nf ? 0xFFFFFFFFu : bi;
        *choice = c;
        if (next) *next = c;
        if (nf) atomicCAS(status, 0, (int)kDevNonfinite);
    }
}

// logits[r] = wte[r] . LN_f(X[last]) for r < V; every block recomputes the
// final LayerNorm of the last row into shared memory (D = 4 * NV <= 1024).
// A warp takes two rows at a time with all of their float4 loads issued
// before the first multiply, so enough bytes are in flight to stream the
// tied embedding at HBM speed.
template <int NV>
__global__ void __launch_bounds__(kHeadThreads) head_kernel(const float* __restrict__ X, int last,
                                                            const float* __restrict__ g,
                                                            const float* __restrict__ b,
                                                            const float* __restrict__ wte, int V,
                                                            float* __restrict__ logits) {
    constexpr int D = 4 * NV, PL = (NV + 31) / 32;  // float4 per lane per row
    static_assert(D <= 1024, "row width");
    __shared__ __align__(16) float xs[D];
    __shared__ float red[kHeadThreads / 32];
    chain_enter();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const float* x = X + (size_t)last * D;
    float s = 0.0f;
    for (int i = tid; i < D; i += kHeadThreads) s += x[i];
    s = warp_sum32(s);
    if (lane == 0) red[warp] = s;
    __syncthreads();
    float t = 0.0f;
    for (int w = 0; w < kHeadThreads / 32; ++w) t += red[w];
    const float mean = t / (float)D;
    __syncthreads();
    float q = 0.0f;
    for (int i = tid; i < D; i += kHeadThreads) {
        const float d = x[i] - mean;
        q = fmaf(d, d, q);
    }
    q = warp_sum32(q);
    if (lane == 0) red[warp] = q;
    __syncthreads();
    float v = 0.0f;
    for (int w = 0; w < kHeadThreads / 32; ++w) v += red[w];
    const float den = sqrtf(v / (float)D + kLnEps);
    for (int i = tid; i < D; i += kHeadThreads) xs[i] = (x[i] - mean) / den * g[i] + b[i];
    __syncthreads();
    const float4* x4 = reinterpret_cast<const float4*>(xs);
    float4 xr[PL];
#pragma unroll
    for (int p = 0; p < PL; ++p) {
        const int c = lane + 32 * p;
        xr[p] = c < NV ? x4[c] : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    }
    const int gw = blockIdx.x * (kHeadThreads / 32) + warp, nw = gridDim.x * (kHeadThreads / 32);
    for (int r = gw; r < V; r += 2 * nw) {
        const int r2 = r + nw;
        const float4* w0 = reinterpret_cast<const float4*>(wte + (size_t)r * D);
        const float4* w1 = reinterpret_cast<const float4*>(wte + (size_t)(r2 < V ? r2 : r) * D);
        float4 a0[PL], a1[PL];
#pragma unroll
        for (int p = 0; p < PL; ++p) {
            const int c = lane + 32 * p;
            a0[p] = c < NV ? __ldcs(w0 + c) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            a1[p] = c < NV ? __ldcs(w1 + c) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        }
        float acc0 = 0.0f, acc1 = 0.0f;
#pragma unroll
        for (int p = 0; p < PL; ++p) {
            acc0 = fmaf(a0[p].x, xr[p].x, acc0);
            acc0 = fmaf(a0[p].y, xr[p].y, acc0);
            acc0 = fmaf(a0[p].z, xr[p].z, acc0);
            acc0 = fmaf(a0[p].w, xr[p].w, acc0);
            acc1 = fmaf(a1[p].x, xr[p].x, acc1);
            acc1 = fmaf(a1[p].y, xr[p].y, acc1);
            acc1 = fmaf(a1[p].z, xr[p].z, acc1);
            acc1 = fmaf(a1[p].w, xr[p].w, acc1);
        }
        acc0 = warp_sum32(acc0);
        acc1 = warp_sum32(acc1);
        if (lane == 0) {
            logits[r] = acc0;
            if (r2 < V) logits[r2] = acc1;
        }
    }
}

}  // namespace

// ---------------------------------------------------------------- host side
namespace {
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;
int g_sms = 0;

bool encode_ready() {
    std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return g_encode != nullptr;
}

// K-major fp32 matrix [rows][K] (row stride K floats) with a {32, box_rows} box.
bool kmajor_map(CUtensorMap* map, const float* base, int K, int rows, int box_rows) {
    cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)K * 4};
    cuuint32_t box[2] = {(cuuint32_t)tc::kBlockK, (cuuint32_t)box_rows};
    cuuint32_t es[2] = {1, 1};
    return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(base), dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// K splits for an (m tiles x n tiles) grid.
int choose_splits(int m_tiles, int n_tiles, int K, int TN) {
    const int nkb = K / tc::kBlockK;
    const int tiles = m_tiles * n_tiles;
    // about two thirds of the SMs for one row tile of 64-wide tiles: longer K
    // ranges per CTA keep its 4-stage pipeline full (measured best between
    // 36 and 300 CTAs on 152 SMs for the 128-row prefill); every SM for the
    // 128-wide tiles of up to 64 rows and for several row tiles (the batched
    // step at 16, 64 and 256 sessions measured best so)
    const int want = (TN == 128 || m_tiles > 1) ? g_sms : (2 * g_sms + 2) / 3;
    int s = (want + tiles / 2) / tiles;
    if (s < 1) s = 1;
    if (s > nkb) s = nkb;
    if (s > kPrefillMaxSplits) s = kPrefillMaxSplits;
    return s;
}

}  // namespace

bool tc_ready() {
    if (!encode_ready()) return false;
    if (!g_sms) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&g_sms, cudaDevAttrMultiProcessorCount, dev);
        if (g_sms <= 0) g_sms = 1;
    }
    return cudaFuncSetAttribute(tc::tf32x3_gemm_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)tc::tc_smem(64)) == cudaSuccess &&
           cudaFuncSetAttribute(tc::tf32x3_gemm_kernel<128, 64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)tc::tc_smem(128)) == cudaSuccess;
}

int tc_sm_count() { return g_sms; }

cudaError_t tc_gemm(const float* A, const float* Alo, int m_rows, const float* W, const float* Wlo, int w_rows, int K,
                    int N, int max_splits, int* splits_out, float* part, int* status, cudaStream_t st, bool pdl) {
    if (K % tc::kBlockK || N % tc::kTileN || w_rows > N || m_rows <= 0) return cudaErrorInvalidValue;
    // 128 output features per tile for up to 64 rows where N allows (half
    // the activation reads of the 64-wide tile; measured faster for 16 and
    // 64 sessions, slower for the 128-row prefill), else 64
    const int TN = (N % 128 == 0 && m_rows <= tc::kTileM / 2) ? 128 : 64;
    tc::TcMaps maps;
    const int a_rows = m_rows <= tc::kTileM / 2 ? tc::kTileM / 2 : tc::kTileM;  // A rows loaded per tile
    if (!kmajor_map(&maps.a_hi, A, K, m_rows, a_rows) || !kmajor_map(&maps.a_lo, Alo, K, m_rows, a_rows) ||
        !kmajor_map(&maps.b_hi, W, K, w_rows, TN) || !kmajor_map(&maps.b_lo, Wlo, K, w_rows, TN))
        return cudaErrorInvalidValue;
    const int m_tiles = (m_rows + tc::kTileM - 1) / tc::kTileM, n_tiles = N / TN;
    int splits = choose_splits(m_tiles, n_tiles, K, TN);
    if (splits > max_splits) splits = max_splits < 1 ? 1 : max_splits;
    *splits_out = splits;
    // (128-wide tiles only for up to 64 rows: 64-row A tiles)
    return chain_launch(pdl, TN == 128 ? tc::tf32x3_gemm_kernel<128, 64> : tc::tf32x3_gemm_kernel<64>,
                        dim3(n_tiles, splits, m_tiles), dim3(tc::kTcThreads), tc::tc_smem(TN), st, maps, K, N, m_rows,
                        splits, part, status, (int)kDevTimeout, a_rows);
}

cudaError_t split_lo(const float* w, float* lo, size_t n, cudaStream_t st) {
    split_lo_kernel<<<1024, 256, 0, st>>>(w, lo, n);
    return cudaGetLastError();
}


size_t prefill_part_floats(int cap, int D, int FF) {
    const int n = cap, N = FF > 3 * D ? FF : 3 * D;
    return (size_t)kPrefillMaxSplits * n * N;
}

cudaError_t prefill_make_lo(gpt2_model* m, cudaStream_t st) {
    if (m->d_wlo) return cudaSuccess;
    const size_t bytes = m->layer_bytes * m->cfg.n_layer;
    cudaError_t e = cudaMalloc(&m->d_wlo, bytes);
    if (e != cudaSuccess) return e;
    return split_lo(reinterpret_cast<const float*>(m->d_wstream), m->d_wlo, bytes / 4, st);
}

cudaError_t prefill_alloc(PrefillWs* w, int cap, int D, int FF) {
    if (w->cap >= cap) return cudaSuccess;
    prefill_free(w);
    cudaError_t es = cudaStreamCreateWithFlags(&w->cs, cudaStreamNonBlocking);
    if (es == cudaSuccess) es = cudaEventCreateWithFlags(&w->ev_in, cudaEventDisableTiming);
    if (es == cudaSuccess) es = cudaEventCreateWithFlags(&w->ev_out, cudaEventDisableTiming);
    if (es != cudaSuccess) {
        prefill_free(w);
        return es;
    }
    const size_t nd = (size_t)cap * D, nf = (size_t)cap * FF;
    cudaError_t e = cudaMalloc(&w->X, nd * 4);
    if (e == cudaSuccess) e = cudaMalloc(&w->A, nd * 4);
    if (e == cudaSuccess) e = cudaMalloc(&w->Alo, nd * 4);
    if (e == cudaSuccess) e = cudaMalloc(&w->QKV, 3 * nd * 4);
    if (e == cudaSuccess) e = cudaMalloc(&w->U, nf * 4);
    if (e == cudaSuccess) e = cudaMalloc(&w->Ulo, nf * 4);
    if (e == cudaSuccess) e = cudaMalloc(&w->part, prefill_part_floats(cap, D, FF) * 4);
    if (e != cudaSuccess) {
        prefill_free(w);
        return e;
    }
    w->cap = cap;
    return cudaSuccess;
}

void prefill_free(PrefillWs* w) {
    if (w->cs) cudaStreamSynchronize(w->cs);
    if (w->exec) cudaGraphExecDestroy(w->exec);
    if (w->ev_in) cudaEventDestroy(w->ev_in);
    if (w->ev_out) cudaEventDestroy(w->ev_out);
    if (w->cs) cudaStreamDestroy(w->cs);
    cudaFree(w->X);
    cudaFree(w->A);
    cudaFree(w->Alo);
    cudaFree(w->QKV);
    cudaFree(w->U);
    cudaFree(w->Ulo);
    cudaFree(w->part);
    *w = PrefillWs{};
}

bool prefill_shape_supported(const gpt2_config& c) {
    const int D = (int)c.d_model, FF = (int)c.d_ff, DH = D / (int)c.n_head;
    return D % tc::kTileN == 0 && FF % tc::kTileN == 0 && (D == 64 || D == 192 || D == 768) &&
           (DH == 16 || DH == 32 || DH == 64) &&
           c.max_pos <= kMaxPrefillKeys;
}

namespace {

// Programmatic dependent launches (chain.cuh) in the prefill: for the
// GEMMs only, whose CTAs then initialise their barriers and tensor memory
// while the kernel before them drains.  Per 128-token prefill, same box:
// 0.817 ms with the GEMMs chained, 0.854 with plain launches, 0.94 with
// every kernel chained and 0.98 with every kernel but the GEMMs chained.
// The other kernels' successors are plain launches, so each GEMM still
// completes before the kernel after it starts.
constexpr bool kPrefillGemmPdl = true;
constexpr bool kPrefillPdl = false;

// Every launch of one prefill, enqueued on stream st.
cudaError_t prefill_launches(gpt2_model* m, PrefillWs* w, const uint32_t* d_tok, int n, float* cache, float* logits,
                             int* status, uint32_t* d_choice, uint32_t* d_next, cudaStream_t st) {
    const gpt2_config& c = m->cfg;
    const int D = (int)c.d_model, FF = (int)c.d_ff, L = (int)c.n_layer, H = (int)c.n_head, DH = D / H;
    cudaError_t e = cudaSuccess;
    const float* P = m->d_packed;

    // C[n][N] partials of A[n][K] x W[N][K] (W = block matrix `mat` of layer l)
    auto gemm = [&](const float* A, const float* Alo, int K, int N, int l, int mat, int* splits_out) -> cudaError_t {
        const uint64_t off = (uint64_t)l * m->layer_bytes + m->mat_off[mat];
        const float* W = reinterpret_cast<const float*>(m->d_wstream + off);
        const float* Wlo = reinterpret_cast<const float*>(reinterpret_cast<const uint8_t*>(m->d_wlo) + off);
        return tc_gemm(A, Alo, n, W, Wlo, N, K, N, kPrefillMaxSplits, splits_out, w->part, status, st, kPrefillGemmPdl);
    };
    auto reduce = [&](int splits, int N, uint64_t bias_off, int kind, float* out, float* out_lo, int l) {
        const size_t total = (size_t)n * N;
        const int blocks = (int)((total + 255) / 256 < 4096 ? (total + 255) / 256 : 4096);
        return chain_launch(kPrefillPdl, reduce_kernel, dim3(blocks), dim3(256), 0, st, (const float*)w->part, splits, n, N,
                            P + bias_off, kind, out, out_lo, w->X, cache, L, l, D, (const int*)nullptr, (size_t)0);
    };

    // LayerNorm of the residual rows into A (+ remainder); with a projection's
    // partials, the residual add of that projection first (one kernel)
    auto ln = [&](uint64_t g_off, uint64_t b_off, int splits, uint64_t bias_off) {
        return chain_launch(kPrefillPdl, ln_split_kernel, dim3(n), dim3(kLnThreads), 0, st, w->X, P + g_off, P + b_off, D,
                            w->A, w->Alo, (const float*)(splits ? w->part : nullptr), splits, n, P + bias_off);
    };

    // the first kernel of the chain: a plain launch
    e = chain_launch(false, embed_kernel, dim3(n), dim3(256), 0, st, P, m->wte_off, m->wpe_off, d_tok, D, c.vocab,
                     w->X, status);
    if (e == cudaSuccess) e = ln(m->lp[0].ln1_g, m->lp[0].ln1_b, 0, 0);
    for (int l = 0; l < L && e == cudaSuccess; ++l) {
        const LayerParams& lp = m->lp[l];
        int sp = 1;
        if ((e = gemm(w->A, w->Alo, D, 3 * D, l, kQKV, &sp)) != cudaSuccess) break;
        if ((e = reduce(sp, 3 * D, lp.b_qkv, kRedQKV, w->QKV, nullptr, l)) != cudaSuccess) break;
        const dim3 agrid(H, (n + kAttnRows - 1) / kAttnRows);
        auto attn = DH == 64 ? attention_kernel<64> : DH == 32 ? attention_kernel<32> : attention_kernel<16>;
        if ((e = chain_launch(kPrefillPdl, attn, agrid, dim3(kAttnWarps * 32), 0, st, (const float*)w->QKV, n, D, w->A,
                              w->Alo)) != cudaSuccess)
            break;
        if ((e = gemm(w->A, w->Alo, D, D, l, kO, &sp)) != cudaSuccess) break;
        if ((e = ln(lp.ln2_g, lp.ln2_b, sp, lp.b_o)) != cudaSuccess) break;  // residual + LN2
        if ((e = gemm(w->A, w->Alo, D, FF, l, kFC, &sp)) != cudaSuccess) break;
        if ((e = reduce(sp, FF, lp.b_fc, kRedGelu, w->U, w->Ulo, l)) != cudaSuccess) break;
        if ((e = gemm(w->U, w->Ulo, FF, D, l, kP, &sp)) != cudaSuccess) break;
        if (l + 1 < L) e = ln(m->lp[l + 1].ln1_g, m->lp[l + 1].ln1_b, sp, lp.b_p);  // residual + next LN1
        else e = reduce(sp, D, lp.b_p, kRedResidual, nullptr, nullptr, l);
    }
    if (e != cudaSuccess) return e;
    const float* lg = P + m->lnf_g;
    const float* lb = P + m->lnf_b;
    const float* wte = P + m->wte_off;
    const int hb = 2 * tc_sm_count();  // two blocks per SM
    if (D != 768 && D != 192 && D != 64) return cudaErrorInvalidValue;
    auto head = D == 768 ? head_kernel<192> : D == 192 ? head_kernel<48> : head_kernel<16>;
    e = chain_launch(kPrefillPdl, head, dim3(hb), dim3(kHeadThreads), 0, st, (const float*)w->X, n - 1, lg, lb, wte,
                     (int)c.vocab, logits);
    if (e != cudaSuccess) return e;
    return chain_launch(kPrefillPdl, choice_kernel, dim3(1), dim3(kChoiceThreads), 0, st, (const float*)logits, c.vocab,
                        d_choice, d_next, status);
}

}  // namespace

cudaError_t prefill_enqueue(gpt2_model* m, PrefillWs* w, const uint32_t* d_tok, int n, float* cache, float* logits,
                            int* status, uint32_t* d_choice, uint32_t* d_next, cudaStream_t st) {
    if (!tc_ready()) return cudaErrorNotSupported;
    cudaError_t e = cudaSuccess;
    const void* key[9] = {m, d_tok, reinterpret_cast<const void*>((uintptr_t)n), cache, logits, status, d_choice, d_next,
                          w->part};
    bool same = w->exec != nullptr;
    for (int i = 0; i < 9 && same; ++i) same = key[i] == w->key[i];
    if (!same) {
        if (w->exec) {
            cudaGraphExecDestroy(w->exec);
            w->exec = nullptr;
        }
        cudaGraph_t graph = nullptr;
        e = cudaStreamBeginCapture(w->cs, cudaStreamCaptureModeThreadLocal);
        if (e != cudaSuccess) return e;
        const cudaError_t el = prefill_launches(m, w, d_tok, n, cache, logits, status, d_choice, d_next, w->cs);
        e = cudaStreamEndCapture(w->cs, &graph);
        if (el != cudaSuccess) e = el;
        if (e == cudaSuccess) e = cudaGraphInstantiate(&w->exec, graph, 0);
        if (graph) cudaGraphDestroy(graph);
        if (e != cudaSuccess) {
            w->exec = nullptr;
            return e;
        }
        for (int i = 0; i < 9; ++i) w->key[i] = key[i];
    }
    e = cudaEventRecord(w->ev_in, st);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(w->cs, w->ev_in, 0);
    if (e == cudaSuccess) e = cudaGraphLaunch(w->exec, w->cs);
    if (e == cudaSuccess) e = cudaEventRecord(w->ev_out, w->cs);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(st, w->ev_out, 0);
    return e;
}

}  // namespace gpt2
