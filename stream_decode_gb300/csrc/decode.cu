// decode.cu -- the persistent GPT-2 step kernel.
//
// One cooperative launch runs n_steps cached steps (LeanExe GPT-2 README,
// cachedStep paragraph; model description paragraph for the block order):
//   embed -> per layer [LN1 + QKV, KV append, attention, out-proj + residual,
//   LN2 + FC + GELU, MLP-proj + residual] -> LN_f + tied vocab projection ->
//   greedy argmax.
//
// Work split: every projection is split by OUTPUT rows across the G CTAs.
// The device keeps every block matrix K-major ([out][in], one contiguous row
// per output), so CTA c's share of a matrix is one contiguous byte range.
// Each CTA has one producer warp that streams its shares of all matrices, in
// step order, through a ring of shared-memory slots with cp.async.bulk and
// mbarriers; it never waits on activations, so weight streaming runs ahead
// of the grid-wide dependencies (bounded only by the ring depth and an
// optional L2 bulk prefetch further ahead).  Eight consumer warps take the
// chunks round-robin and compute complete dot products from shared memory,
// so no cross-CTA reduction is needed.  Phases are ordered by per-CTA epoch
// flags (release/acquire at gpu scope); every spin-wait is bounded by a
// wall-clock limit after which the kernel records GPT2_ERR_TIMEOUT, sets a
// global abort word, drains its own bulk copies and returns.
//
// Attention is split along the key axis ("flash-decoding" split-KV, lean /
// llm-web page, GPU-path paragraph): CTA c owns (head, key range) units and
// writes an unnormalised partial (max, sum, o[64]); the out-projection phase
// merges the partials of every head before its GEMV.
//
// int8 (quantized GPT-2 abstract): projection inputs are quantized per group
// of 64 coordinates right after they are formed (in shared memory); the
// weights come as int8 rows followed by their group scales; int32 group sums
// use __dp4a and the rescale runs in the fixed order
//   y = sum_{g ascending} ((float)acc_g * s_x[g]) * s_w[g], then + bias,
// with explicitly rounded operations so no multiply-add is fused.
#include <cuda_runtime.h>

#include <cstdio>
#include <type_traits>

#include "gpt2_dev.cuh"

namespace gpt2 {

// ----------------------------------------------------------- smem layout
struct SmemLayout {
    uint32_t ring, full, empty, xs, vin, vq, vs, red, ored, qh, rsc, stage, bias, geot, misc, total;
};

__host__ __device__ constexpr uint32_t align16(uint32_t x) { return (x + 15u) & ~15u; }

// `stage` holds, at different times: the attention warp merge
// [warps][8 lanes][2 + 8] (head dim 64), the (max, sum) pairs of every
// attention unit (2 * 12 heads * kMaxSplits), and the per-CTA greedy choices
// [256 + kMaxGrid].
constexpr int kStageFloats = 640;
// int8 rescale terms of one window: [32 rows][48 groups] at most.
constexpr int kCoopTaskFloats = 32 * 48;
static_assert(kConsumerWarps * 8 * (2 + 8) <= kStageFloats, "attention warp merge fits in stage");
static_assert(2 * 16 * kMaxSplits <= kStageFloats, "unit (max, sum) pairs fit in stage");
static_assert(256 + kMaxGrid <= kStageFloats, "greedy choices fit in stage");
constexpr int kMaxChunkRows = 32;

__host__ __device__ inline SmemLayout smem_layout(int D, int FF, bool q8, int max_pos) {
    SmemLayout s{};
    int kmax = D > FF ? D : FF;
    uint32_t o = 0;
    s.ring = o; o += kSlots * kSlotBytes;
    s.full = o; o += kSlots * 8;
    s.empty = o; o += kSlots * 8;
    s.xs = o; o = align16(o + D * 4);
    s.vin = o; o = align16(o + kmax * 4);
    s.vq = o; o = align16(o + (q8 ? kmax : 0));
    s.vs = o; o = align16(o + (kmax / kGroup) * 4);
    s.red = o; o = align16(o + 64 * 4);
    s.ored = o; o = align16(o + kConsumerWarps * 32 * 4);
    s.qh = o; o = align16(o + 3 * 64 * 4);  // q_h, k_p, v_p of one attention unit
    s.rsc = o; o = align16(o + (q8 ? kCoopTaskFloats * 4 : 0));  // int8 rescale terms
    s.stage = o; o = align16(o + kStageFloats * 4);  // attention warp merge; (max, sum) pairs; greedy choices
    s.bias = o; o = align16(o + kConsumerWarps * 32 * 4);
    s.geot = o; o = align16(o + 5 * 32);  // GeoRow table
    s.misc = o; o = align16(o + 64 * 4);
    s.total = o;
    return s;
}

// ------------------------------------------------------- phase geometry
// Phase index within a step: 4*l + {kQKV, kO, kFC, kP} for the projections
// of layer l, 4*L for the vocabulary projection.
struct Geo {
    const uint8_t* base;  // first byte of this CTA's rows
    int r0, nrows;        // first output row and row count of this CTA
    int rb;               // bytes per row
    int rpc;              // rows per chunk
    int nchunks;
};

__device__ __forceinline__ Geo phase_geo(const StepPlan& P, int ph, int cta, bool q8) {
    int N, K;
    const uint8_t* mat;
    if (ph == 4 * P.L) {
        N = P.V; K = P.D; mat = P.vocab;
    } else {
        int l = ph >> 2, m = ph & 3;
        N = (m == kQKV) ? 3 * P.D : (m == kFC ? P.FF : P.D);
        K = (m == kP) ? P.FF : P.D;
        mat = P.wstream + (uint64_t)l * P.layer_bytes + P.mat_off[m];
    }
    Geo g;
    g.rb = row_bytes(K, q8);
    g.r0 = (int)(((long long)cta * N) / P.G);
    int r1 = (int)(((long long)(cta + 1) * N) / P.G);
    g.nrows = r1 - g.r0;
    int rpc = kSlotBytes / g.rb;
    g.rpc = rpc > kMaxChunkRows ? kMaxChunkRows : rpc;
    g.nchunks = (g.nrows + g.rpc - 1) / g.rpc;
    g.base = mat + (uint64_t)g.r0 * g.rb;
    return g;
}

// The same geometry without divisions: one row per matrix kind
// (kQKV, kO, kFC, kP, kVocab), filled once per CTA at kernel start.
struct GeoRow {
    int r0, nrows, rb, rpc, nchunks, pad0, pad1, pad2;
};

__device__ __forceinline__ Geo geo_of(const StepPlan& P, const GeoRow* t, int ph) {
    const int m = (ph == 4 * P.L) ? (int)kVocab : (ph & 3);
    const GeoRow& e = t[m];
    const uint8_t* mat = (m == kVocab) ? P.vocab : P.wstream + (uint64_t)(ph >> 2) * P.layer_bytes + P.mat_off[m];
    Geo g;
    g.base = mat + (uint64_t)e.r0 * e.rb;
    g.r0 = e.r0;
    g.nrows = e.nrows;
    g.rb = e.rb;
    g.rpc = e.rpc;
    g.nchunks = e.nchunks;
    return g;
}

// ------------------------------------------------------- small helpers
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// Deterministic sum over the 256 consumer threads (fixed order).
__device__ __forceinline__ float block_sum(float v, float* red, int tid) {
    v = warp_sum(v);
    if ((tid & 31) == 0) red[tid >> 5] = v;
    consumers_sync();
    float t = 0.0f;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) t += red[w];
    consumers_sync();
    return t;
}

__device__ __forceinline__ float block_max(float v, float* red, int tid) {
    v = warp_max(v);
    if ((tid & 31) == 0) red[tid >> 5] = v;
    consumers_sync();
    float t = -INFINITY;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) t = fmaxf(t, red[w]);
    consumers_sync();
    return t;
}

__device__ __forceinline__ float gelu_tanh(float x) {
    float inner = 0.7978845608f * (x + 0.044715f * x * x * x);
    return 0.5f * x * (1.0f + tanhf(inner));
}

__device__ __forceinline__ void record_error(const StepPlan& P, int code) {
    atomicCAS(P.status, 0, code);
    atomicExch(P.abort_flag, 1);
}

// Greedy choice order: larger value first, then lower index.
__device__ __forceinline__ bool arg_better(float v, unsigned i, float bv, unsigned bi) {
    return v > bv || (v == bv && i < bi);
}

// Running greedy choice: best finite value (lowest index on ties) and a
// flag for any NaN or infinite value seen.
struct ArgBest {
    float v;
    unsigned i;
    int nf;
};

__device__ __forceinline__ ArgBest arg_init() { return ArgBest{-INFINITY, 0xFFFFFFFFu, 0}; }

__device__ __forceinline__ void arg_update(ArgBest& b, float v, unsigned j) {
    if (!isfinite(v)) b.nf = 1;
    else if (arg_better(v, j, b.v, b.i)) { b.v = v; b.i = j; }
}

__device__ __forceinline__ void arg_merge(ArgBest& b, float v, unsigned i, int nf) {
    b.nf |= nf;
    if (arg_better(v, i, b.v, b.i)) { b.v = v; b.i = i; }
}

__device__ __forceinline__ void arg_warp_reduce(ArgBest& b) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, b.v, o);
        const unsigned oi = __shfl_xor_sync(0xffffffffu, b.i, o);
        const int onf = __shfl_xor_sync(0xffffffffu, b.nf, o);
        arg_merge(b, ov, oi, onf);
    }
}

// LayerNorm of x (smem, N values) into y (smem); biased variance, eps 1e-5.
template <int N>
__device__ __forceinline__ void layernorm(const float* x, const float* __restrict__ g, const float* __restrict__ b,
                                          float* y, float* red, int tid) {
    float s = 0.0f;
    for (int i = tid; i < N; i += kConsumerWarps * 32) s += x[i];
    const float mean = block_sum(s, red, tid) / (float)N;
    float q = 0.0f;
    for (int i = tid; i < N; i += kConsumerWarps * 32) {
        float t = x[i] - mean;
        q += t * t;
    }
    const float var = block_sum(q, red, tid) / (float)N;
    const float den = sqrtf(var + kLnEps);
    for (int i = tid; i < N; i += kConsumerWarps * 32) y[i] = (x[i] - mean) / den * __ldg(g + i) + __ldg(b + i);
}

// Quantize v[0..N) per group of 64 into q/s (int8 path).  Warp w owns groups
// w, w + warps, ...; its groups are loaded, reduced and quantized together
// so the shuffles and divisions of different groups overlap.
template <int N>
__device__ __forceinline__ void quantize_vec(const float* v, int8_t* q, float* s, int warp, int lane) {
    constexpr int NG = N / kGroup;
    constexpr int GPW = (NG + kConsumerWarps - 1) / kConsumerWarps;  // groups per warp (at most)
    float a[GPW], b[GPW], m[GPW];
#pragma unroll
    for (int k = 0; k < GPW; ++k) {
        const int gi = warp + kConsumerWarps * k;
        a[k] = gi < NG ? v[gi * kGroup + lane] : 0.0f;
        b[k] = gi < NG ? v[gi * kGroup + 32 + lane] : 0.0f;
        // max of |v| starting from 0; NaN never wins a comparison, as in a plain compare loop
        m[k] = fmaxf(fmaxf(fabsf(a[k]), fabsf(b[k])), 0.0f);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
#pragma unroll
        for (int k = 0; k < GPW; ++k) m[k] = fmaxf(m[k], __shfl_xor_sync(0xffffffffu, m[k], o));
#pragma unroll
    for (int k = 0; k < GPW; ++k) {
        const int gi = warp + kConsumerWarps * k;
        if (gi < NG) {
            const float sc = __fdiv_rn(m[k], 127.0f);
            q[gi * kGroup + lane] = (int8_t)quantize_one(a[k], sc);
            q[gi * kGroup + 32 + lane] = (int8_t)quantize_one(b[k], sc);
            if (lane == 0) s[gi] = sc;
        }
    }
}

// Warp transpose-reduction: every lane holds partials v[0..N) of N rows
// (N a power of two, at most 32).  Plain butterflies fold the lane bits above
// log2(N), then transpose steps halve the values per lane; lane l ends with
// the warp's total of row l % N (fixed order).
template <int N>
__device__ __forceinline__ float warp_transpose_sum(float (&v)[N], int lane) {
#pragma unroll
    for (int o = 16; o >= N; o >>= 1)
#pragma unroll
        for (int i = 0; i < N; ++i) v[i] += __shfl_xor_sync(0xffffffffu, v[i], o);
#pragma unroll
    for (int o = N / 2; o >= 1; o >>= 1) {
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < o; ++i) {
            const float send = up ? v[i] : v[i + o];
            const float keep = up ? v[i + o] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
    }
    return v[0];
}

// Rows per ring chunk and per window for input width K.  A window is a run
// of whole chunks (at most 8, at most 32 rows; 8 rows for binary32 K = 3072,
// which keeps the accumulators in registers) that all warps compute together.
template <int K, bool Q8>
struct WinGeo {
    static constexpr int RB = row_bytes(K, Q8);
    static constexpr int RPC0 = kSlotBytes / RB;
    static constexpr int RPC = RPC0 > kMaxChunkRows ? kMaxChunkRows : RPC0;  // rows per chunk
    static constexpr int MAXW = (!Q8 && K > 2048) ? 8 : 32;                  // rows per window, at most
    static constexpr int CPW0 = MAXW / RPC < 1 ? 1 : MAXW / RPC;
    static constexpr int CPW = CPW0 > 8 ? 8 : CPW0;                          // chunks per window
    static constexpr int WR = CPW * RPC;                                      // rows per window
    static constexpr int MR = WR > 8 ? 32 : 8;                                // padded for the transpose-sum
};

// binary32 window: thread t covers float4 columns t, t + NT, ... of every
// row; the warps' partial sums meet through wpart.  Thread r < wn returns
// row r's dot product with x.  Window row r lives in chunk c0 + r / RPC.
template <int K>
__device__ __forceinline__ float win_f32(const uint8_t* ring, uint32_t c0, int wn, const float* x, float* wpart,
                                         int tid, int lane, int warp) {
    using W = WinGeo<K, false>;
    constexpr int NT = kConsumerWarps * 32;
    constexpr int NV = K / 4;
    constexpr int FPT = (NV + NT - 1) / NT;
    const float4* x4 = reinterpret_cast<const float4*>(x);
    float4 xv[FPT];
#pragma unroll
    for (int i = 0; i < FPT; ++i) {
        const int f = tid + NT * i;
        xv[i] = f < NV ? x4[f] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float acc[W::MR];
#pragma unroll
    for (int r = 0; r < W::MR; ++r) {
        acc[r] = 0.0f;
        // a compiler-only fence every 8 rows bounds the shared loads in flight
        if ((r & 7) == 0) asm volatile("" ::: "memory");
        if (r < wn) {
            const int c = r / W::RPC, rr = r - c * W::RPC;
            const float4* w4 = reinterpret_cast<const float4*>(ring + (size_t)((c0 + c) % kSlots) * kSlotBytes +
                                                              (size_t)rr * W::RB);
#pragma unroll
            for (int i = 0; i < FPT; ++i) {
                const int f = tid + NT * i;
                if (f < NV) {
                    const float4 wv = w4[f];
                    acc[r] = fmaf(xv[i].x, wv.x, acc[r]);
                    acc[r] = fmaf(xv[i].y, wv.y, acc[r]);
                    acc[r] = fmaf(xv[i].z, wv.z, acc[r]);
                    acc[r] = fmaf(xv[i].w, wv.w, acc[r]);
                }
            }
        }
    }
    const float tot = warp_transpose_sum<W::MR>(acc, lane);
    if (lane < W::MR) wpart[warp * 32 + lane] = tot;
    consumers_sync();
    float y = 0.0f;
    if (tid < wn)
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) y += wpart[w * 32 + tid];
    return y;
}

// int8 window: (row, group) tasks over all warps give the exact int32 group
// sums; t_g = ((float)acc_g * s_x[g]) * s_w[g] is parked in tsm, and thread
// r < wn returns its row's terms summed in ascending group order from 0.0f
// (the fixed rescale order), explicitly rounded so nothing is fused.
template <int K>
__device__ __forceinline__ float win_q8(const uint8_t* ring, uint32_t c0, int wn, const int8_t* xq, const float* xs,
                                        float* tsm, int tid) {
    using W = WinGeo<K, true>;
    constexpr int NT = kConsumerWarps * 32;
    constexpr int NG = K / kGroup;
    const int tasks = wn * NG;
    for (int tk = tid; tk < tasks; tk += NT) {
        const int r = tk / NG, g = tk - r * NG;
        const int c = r / W::RPC, rr = r - c * W::RPC;
        const uint8_t* row = ring + (size_t)((c0 + c) % kSlots) * kSlotBytes + (size_t)rr * W::RB;
        const int4* wv = reinterpret_cast<const int4*>(row + g * kGroup);
        const int4* xv = reinterpret_cast<const int4*>(xq + g * kGroup);
        int acc = 0;
#pragma unroll
        for (int v = 0; v < 4; ++v) {
            const int4 a = wv[v], b = xv[v];
            acc = __dp4a(a.x, b.x, acc);
            acc = __dp4a(a.y, b.y, acc);
            acc = __dp4a(a.z, b.z, acc);
            acc = __dp4a(a.w, b.w, acc);
        }
        const float sw = reinterpret_cast<const float*>(row + K)[g];
        tsm[tk] = __fmul_rn(__fmul_rn(__int2float_rn(acc), xs[g]), sw);
    }
    consumers_sync();
    float sum = 0.0f;
    if (tid < wn)
        for (int g = 0; g < NG; ++g) sum = __fadd_rn(sum, tsm[tid * NG + g]);
    return sum;
}

// -------------------------------------------------------------- kernel
// Waits until every word k with bit k set in `pending` carries `tag`,
// leaving the raw words in w[] (decode with val_of).  MAXC bounds k at
// compile time so the words stay in registers; all pending words are
// reloaded together, so one round costs one L2 round trip.  Returns false
// when the run is abandoned (another CTA gave up, or the wait exceeded its
// limit).
template <int MAXC, typename Addr>
__device__ __forceinline__ bool tagged_wait(uint64_t (&w)[MAXC], uint64_t pending, unsigned tag, Addr addr,
                                            const StepPlan& P) {
    uint64_t t0 = 0;
    uint32_t rounds = 0;
    while (pending) {
#pragma unroll
        for (int k = 0; k < MAXC; ++k)
            if ((pending >> k) & 1ull) w[k] = ld_tagged(addr(k));
#pragma unroll
        for (int k = 0; k < MAXC; ++k)
            if (((pending >> k) & 1ull) && tag_of(w[k]) == tag) pending &= ~(1ull << k);
        if (pending && (++rounds & 7u) == 0) {
            if (ld_volatile_int(P.abort_flag)) return false;
            const uint64_t now = globaltimer_ns();
            if (t0 == 0) t0 = now;
            else if (now - t0 > P.wait_limit_ns) {
                record_error(P, kDevTimeout);
                return false;
            }
        }
    }
    return true;
}

// Bits of the words of an N-word vector that thread tid owns (tid + NT*k).
template <int MAXC>
__device__ __forceinline__ uint64_t own_words(int N, int tid) {
    constexpr int NT = kConsumerWarps * 32;
    uint64_t m = 0;
#pragma unroll
    for (int k = 0; k < MAXC; ++k)
        if (tid + NT * k < N) m |= 1ull << k;
    return m;
}

// Copies a tagged N-word vector into shared memory once every word carries `tag`.
template <int MAXC>
__device__ __forceinline__ bool gather_vec(const uint64_t* src, int N, unsigned tag, float* dst, int tid,
                                           const StepPlan& P) {
    constexpr int NT = kConsumerWarps * 32;
    uint64_t w[MAXC];
    const bool ok = tagged_wait<MAXC>(w, own_words<MAXC>(N, tid), tag, [&](int k) { return src + tid + NT * k; }, P);
#pragma unroll
    for (int k = 0; k < MAXC; ++k)
        if (tid + NT * k < N) dst[tid + NT * k] = val_of(w[k]);
    return ok;
}

// LayerNorm with this thread's gains/shifts already in registers (loaded
// before the wait for x, so their latency hides behind it).
template <int N, int PN>
__device__ __forceinline__ void layernorm_regs(const float* x, const float (&g)[PN], const float (&b)[PN], float* y,
                                               float* red, int tid) {
    // one block reduction of (sum x, sum x^2); var = E[x^2] - mean^2 (biased)
    constexpr int NT = kConsumerWarps * 32;
    float s1 = 0.0f, s2 = 0.0f;
#pragma unroll
    for (int k = 0; k < PN; ++k)
        if (tid + NT * k < N) {
            const float v = x[tid + NT * k];
            s1 += v;
            s2 = fmaf(v, v, s2);
        }
    s1 = warp_sum(s1);
    s2 = warp_sum(s2);
    if ((tid & 31) == 0) {
        red[tid >> 5] = s1;
        red[32 + (tid >> 5)] = s2;
    }
    consumers_sync();
    float t1 = 0.0f, t2 = 0.0f;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) {
        t1 += red[w];
        t2 += red[32 + w];
    }
    const float mean = t1 / (float)N;
    const float var = fmaxf(t2 / (float)N - mean * mean, 0.0f);
    const float den = sqrtf(var + kLnEps);
#pragma unroll
    for (int k = 0; k < PN; ++k)
        if (tid + NT * k < N) y[tid + NT * k] = (x[tid + NT * k] - mean) / den * g[k] + b[k];
}

template <int N, int PN>
__device__ __forceinline__ void load_ln(const float* g, const float* b, float (&gr)[PN], float (&br)[PN], int tid) {
    constexpr int NT = kConsumerWarps * 32;
#pragma unroll
    for (int k = 0; k < PN; ++k) {
        const int i = tid + NT * k;
        gr[k] = i < N ? __ldg(g + i) : 0.0f;
        br[k] = i < N ? __ldg(b + i) : 0.0f;
    }
}

template <int D, int FF, int DH, bool Q8>
__global__ void __launch_bounds__(kThreads, 1) step_kernel(const __grid_constant__ StepPlan P) {
    extern __shared__ __align__(128) uint8_t smem[];
    const SmemLayout lay = smem_layout(D, FF, Q8, P.max_pos);
    uint8_t* ring = smem + lay.ring;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + lay.full);
    uint64_t* empty = reinterpret_cast<uint64_t*>(smem + lay.empty);
    float* xs = reinterpret_cast<float*>(smem + lay.xs);
    float* vin = reinterpret_cast<float*>(smem + lay.vin);
    int8_t* vq = reinterpret_cast<int8_t*>(smem + lay.vq);
    float* vs = reinterpret_cast<float*>(smem + lay.vs);
    float* red = reinterpret_cast<float*>(smem + lay.red);
    float* ored = reinterpret_cast<float*>(smem + lay.ored);
    GeoRow* geot = reinterpret_cast<GeoRow*>(smem + lay.geot);
    float* qh = reinterpret_cast<float*>(smem + lay.qh);  // q_h, k_p, v_p
    float* rsc = reinterpret_cast<float*>(smem + lay.rsc);
    float* stage = reinterpret_cast<float*>(smem + lay.stage);
    float* bias_s = reinterpret_cast<float*>(smem + lay.bias);
    volatile int* s_abort = reinterpret_cast<volatile int*>(smem + lay.misc);
    volatile int* s_fail = s_abort + 1;  // two slots, alternating per agreement point
    unsigned* s_tok = reinterpret_cast<unsigned*>(smem + lay.misc) + 4;
    volatile int* s_nf = s_abort + 5;
    float* s_arg = reinterpret_cast<float*>(smem + lay.misc) + 8;  // [warps][3]

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int cta = blockIdx.x;
    const int L = P.L;
    const int phases_per_step = 4 * L + 1;  // weight phases per step (producer)

    if (tid == 0) {
        for (int i = 0; i < kSlots; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        *s_abort = ld_volatile_int(P.abort_flag);
        s_fail[0] = 0;
        s_fail[1] = 0;
        for (int m = 0; m < 5; ++m) {
            const Geo g0 = phase_geo(P, m == kVocab ? 4 * L : m, cta, Q8);
            geot[m] = GeoRow{g0.r0, g0.nrows, g0.rb, g0.rpc, g0.nchunks, 0, 0, 0};
        }
        fence_mbar_init();
    }
    __syncthreads();
    if (*s_abort) return;  // an earlier run of this session failed and was not cleared
    // ================================================= producer warp
    if (warp == kConsumerWarps) {
        if (lane != 0) return;
        const uint64_t pol = policy_evict_first();
        uint32_t gi = 0;  // chunks issued
        bool stop = false;
        // L2 prefetch cursor: walks the same chunk sequence prefetch_chunks ahead.
        int pf_s = 0, pf_ph = 0, pf_k = 0;
        Geo pf_g = geo_of(P, geot, 0);
        uint32_t pf_issued = 0;
        auto pf_advance = [&]() {
            // issue one prefetch at the cursor, then move it
            while (pf_s < P.n_steps && pf_k >= pf_g.nchunks) {
                pf_k = 0;
                if (++pf_ph == phases_per_step) { pf_ph = 0; ++pf_s; }
                if (pf_s < P.n_steps) pf_g = geo_of(P, geot, pf_ph);
            }
            if (pf_s >= P.n_steps) return;
            const int r = pf_k * pf_g.rpc;
            const int n = min(pf_g.rpc, pf_g.nrows - r);
            bulk_prefetch_l2(pf_g.base + (uint64_t)r * pf_g.rb, (uint32_t)(n * pf_g.rb));
            ++pf_k;
            ++pf_issued;
        };
        for (int i = 0; i < P.prefetch_chunks; ++i) pf_advance();
        for (int s = 0; s < P.n_steps && !stop; ++s) {
            for (int ph = 0; ph < phases_per_step && !stop; ++ph) {
                const Geo g = geo_of(P, geot, ph);
                for (int k = 0; k < g.nchunks; ++k) {
                    const int slot = gi % kSlots;
                    const uint32_t fill = gi / kSlots;
                    if (fill > 0) {
                        uint64_t t0 = 0;
                        uint32_t spins = 0;
                        while (!mbar_try_wait(&empty[slot], (fill - 1) & 1)) {
                            if (*s_abort) { stop = true; break; }
                            if ((++spins & 255) == 0) {
                                const uint64_t now = globaltimer_ns();
                                if (t0 == 0) t0 = now;
                                else if (now - t0 > 2 * P.wait_limit_ns) {
                                    // Only consumer warps write s_abort (they read it after named
                                    // barriers); the producer reports through the global words.
                                    record_error(P, kDevTimeout);
                                    stop = true;
                                    break;
                                }
                            }
                        }
                        if (stop) break;
                    }
                    const int r = k * g.rpc;
                    const int n = min(g.rpc, g.nrows - r);
                    const uint32_t bytes = (uint32_t)(n * g.rb);
                    mbar_arrive_expect_tx(&full[slot], bytes);
                    bulk_load(ring + (size_t)slot * kSlotBytes, g.base + (uint64_t)r * g.rb, bytes, &full[slot], pol);
                    ++gi;
                    if (P.prefetch_chunks > 0) pf_advance();
                }
            }
        }
        // Drain: every issued copy must have landed before this thread exits.
        const uint32_t nslot = gi < (uint32_t)kSlots ? gi : (uint32_t)kSlots;
        for (uint32_t i = 0; i < nslot; ++i) {
            const uint32_t last = gi - 1 - i;  // the most recent fill of slot last % kSlots
            const int slot = last % kSlots;
            uint64_t t0 = 0;
            uint32_t spins = 0;
            while (!mbar_try_wait(&full[slot], (last / kSlots) & 1)) {
                if ((++spins & 255) == 0) {
                    const uint64_t now = globaltimer_ns();
                    if (t0 == 0) t0 = now;
                    else if (now - t0 > 2 * P.wait_limit_ns) { record_error(P, kDevTimeout); break; }
                }
            }
        }
        (void)pf_issued;
        return;
    }


    // ================================================= consumer warps
    constexpr int NT = kConsumerWarps * 32;
    constexpr int PD = (D + NT - 1) / NT;      // D-vector words per thread
    constexpr int PF = (FF + NT - 1) / NT;     // FF-vector words per thread
    constexpr int P3 = (3 * D + NT - 1) / NT;  // qkv words per thread (trace)
    constexpr int PM = PD * kMaxSplits;        // attention partial words per thread (merge)
    static_assert(PM <= 64 && PF <= 64 && P3 <= 64, "tagged gathers hold at most 64 words per thread");
    uint32_t gi = 0;  // chunks consumed (same sequence as the producer)
    const int S = attn_splits(P.G, P.H);  // splits the scratch holds per head
    const unsigned per_step = 5u * (unsigned)L + 1u;
    const bool tracer = (P.trace != nullptr) && cta == 0;
    const int trace_layer = 8 * D + FF;
    // Profiling hook: globaltimer stamps of step 0, per (phase, CTA): phase
    // start, inputs ready, outputs stored.
    int tph = 0;
    // per (phase, CTA): globaltimer at start / inputs ready / outputs stored,
    // then SM clock64 at start / ready / transform done / first chunk in / stored
    // (10 slots: + clock64 after warp 0's first chunk body, after its last chunk)
    constexpr int kStamps = 10;
    auto stamp = [&](int s_now, int point) {
        if (P.timing && s_now == 0 && tid == 0) {
            uint64_t* e = P.timing + ((size_t)tph * P.G + cta) * kStamps;
            const int ci = point == 0 ? 3 : point == 1 ? 4 : point == 3 ? 5 : point == 4 ? 6 : 9;
            e[ci] = (uint64_t)clock64();
            if (point <= 2) e[point] = globaltimer_ns();
        }
        if (point == 2) ++tph;
    };
    bool stamp_chunk = false;  // warp 0 stamps point 4 when its first chunk of the phase has landed
    // Test hook: CTA 0 tags one phase's outputs one too low, so nobody accepts them.
    const unsigned stall_tag = P.stall_phase >= 0 ? P.epoch + (unsigned)P.stall_phase : 0u;
    auto out_tag = [&](unsigned t) -> unsigned { return (cta == 0 && t == stall_tag) ? t - 1u : t; };

    // Every consumer thread reaches each agreement point; a failure anywhere
    // in the CTA becomes everyone's decision (two slots, so the next point's
    // write can never race this point's reads).
    int agree_no = 0;
    auto agree = [&](bool ok) -> bool {
        volatile int* slot = s_fail + (agree_no & 1);
        ++agree_no;
        if (!ok) *slot = 1;
        consumers_sync();
        return *slot == 0;
    };

    // Epilogue of one output row j (run by the thread that owns the row):
    // QKV: + bias, tagged store, KV append; O and P: + bias + residual; FC:
    // + bias, GELU; vocabulary: logits and the running greedy choice.
    struct Epi {
        int kind;
        unsigned tag;
        uint64_t bias;   // word offset of the bias in the packed checkpoint (unused for the vocabulary)
        float* kv_row;   // QKV: this position's cache row
        float* logits;   // vocabulary: this step's logits or null
    };
    ArgBest best = arg_init();
    auto apply_epi = [&](const Epi& e, const Geo& g, int j, float acc) {
        if (e.kind == kVocab) {
            if (e.logits) e.logits[j] = acc;
            arg_update(best, acc, (unsigned)j);
            return;
        }
        const float b = g.nrows <= NT ? bias_s[j - g.r0] : __ldg(P.packed + e.bias + j);
        const float y = __fadd_rn(acc, b);
        if (e.kind == kQKV) {
            st_tagged(P.qkv + j, e.tag, y);
            if (j >= D) e.kv_row[j - D] = y;
        } else if (e.kind == kO) {
            st_tagged(P.xb + j, e.tag, __fadd_rn(xs[j], y));
        } else if (e.kind == kFC) {
            st_tagged(P.u + j, e.tag, gelu_tanh(y));
        } else {
            st_tagged(P.xa + j, e.tag, __fadd_rn(xs[j], y));
        }
    };
    // Runs weight phase `ph` over this CTA's rows, one window of whole ring
    // chunks at a time (all warps on every row of the window); the producer
    // fills the next window's slots meanwhile.  Returns false if a chunk
    // never arrived (the run is then abandoned at the next agreement).
    auto run_phase = [&](auto kk, int ph, const Epi& e) -> bool {
        constexpr int KK = decltype(kk)::value;
        using W = WinGeo<KK, Q8>;
        const Geo g = geo_of(P, geot, ph);
        bool ok = true;
        for (int w0 = 0; w0 < g.nrows; w0 += W::WR) {
            const int wn = min(W::WR, g.nrows - w0);
            const uint32_t c0 = gi + (uint32_t)(w0 / W::RPC);
            const int nc = (wn + W::RPC - 1) / W::RPC;
            for (int c = 0; c < nc && ok; ++c) {
                const uint32_t cc = c0 + c;
                const int slot = cc % kSlots;
                uint64_t t0 = 0;
                uint32_t spins = 0;
                // every lane observes the completed phase (acquire) before reading the slot
                while (!__all_sync(0xffffffffu, mbar_try_wait(&full[slot], (cc / kSlots) & 1))) {
                    if ((++spins & 255) == 0) {
                        int give_up = 0;
                        if (ld_volatile_int(P.abort_flag)) give_up = 1;
                        const uint64_t now = globaltimer_ns();
                        if (t0 == 0) t0 = now;
                        else if (now - t0 > P.wait_limit_ns) {
                            if (lane == 0) record_error(P, kDevTimeout);
                            give_up = 1;
                        }
                        if (__shfl_sync(0xffffffffu, give_up, 0)) { ok = false; break; }
                    }
                }
            }
            const bool st0 = w0 == 0 && stamp_chunk && P.timing && tid == 0 && tph < (int)per_step;
            if (st0) P.timing[((size_t)tph * P.G + cta) * kStamps + 6] = (uint64_t)clock64();
            float y;
            if constexpr (Q8) y = win_q8<KK>(ring, c0, wn, vq, vs, rsc, tid);
            else y = win_f32<KK>(ring, c0, wn, vin, stage, tid, lane, warp);
            if (st0) P.timing[((size_t)tph * P.G + cta) * kStamps + 7] = (uint64_t)clock64();
            if (ok && tid < wn) apply_epi(e, g, g.r0 + w0 + tid, y);
            consumers_sync();  // the window's slots are read and its scratch is free again
            if (tid == 0)
                for (int c = 0; c < nc; ++c) mbar_arrive(&empty[(c0 + c) % kSlots]);
        }
        stamp_chunk = false;
        if (P.timing && tid == 0 && tph < (int)per_step)
            P.timing[((size_t)tph * P.G + cta) * kStamps + 8] = (uint64_t)clock64();
        gi += g.nchunks;
        return ok;
    };
    using KD = std::integral_constant<int, D>;
    using KF = std::integral_constant<int, FF>;
    // Bias rows of this CTA's share of a phase: loaded into a register before
    // the phase's wait, parked in shared memory after it.
    auto bias_prefetch = [&](const Geo& g, uint64_t off) -> float {
        return (g.nrows <= NT && tid < g.nrows) ? __ldg(P.packed + off + g.r0 + tid) : 0.0f;
    };
    auto bias_park = [&](const Geo& g, float v) {
        if (g.nrows <= NT && tid < g.nrows) bias_s[tid] = v;
    };
    auto trace_vec = [&](int offset, const float* v, int n) {
        for (int i = tid; i < n; i += NT) P.trace[offset + i] = v[i];
    };
    auto quantize_in = [&](int n) {
        if constexpr (Q8) {
            if (n == FF) quantize_vec<FF>(vin, vq, vs, warp, lane);
            else quantize_vec<D>(vin, vq, vs, warp, lane);
            consumers_sync();
        }
    };
    // The previous step's per-CTA greedy choices (tag `tag`), reduced here.
    // The acquire pairs with each CTA's release of its choice, so the KV rows
    // that step wrote are visible to this step's attention.
    auto reduce_choice = [&](unsigned tag) -> bool {
        bool ok = true;
        if (tid < P.G) {
            const uint64_t* ap = P.arg_part + 2 * (size_t)tid;
            uint64_t t0 = 0;
            uint32_t rounds = 0;
            uint64_t w0 = ld_tagged_acquire(ap);
            while (tag_of(w0) != tag) {
                if ((++rounds & 7u) == 0) {
                    if (ld_volatile_int(P.abort_flag)) { ok = false; break; }
                    const uint64_t now = globaltimer_ns();
                    if (t0 == 0) t0 = now;
                    else if (now - t0 > P.wait_limit_ns) {
                        record_error(P, kDevTimeout);
                        ok = false;
                        break;
                    }
                }
                w0 = ld_tagged_acquire(ap);
            }
            if (ok) {
                const uint64_t w1 = ld_tagged(ap + 1);  // written before w0's release
                if (tag_of(w1) != tag) {
                    record_error(P, kDevTimeout);
                    ok = false;
                }
                stage[tid] = val_of(w0);
                stage[256 + tid] = val_of(w1);
            }
        }
        if (!agree(ok)) return false;
        if (warp == 0) {
            ArgBest b = arg_init();
            for (int c = lane; c < P.G; c += 32) {
                const unsigned iw = __float_as_uint(stage[256 + c]);
                arg_merge(b, stage[c], iw & 0x7FFFFFFFu, (int)(iw >> 31));
            }
            arg_warp_reduce(b);
            if (lane == 0) {
                *s_tok = b.nf ? 0xFFFFFFFFu : b.i;
                *s_nf = b.nf;
            }
        }
        consumers_sync();
        return true;
    };
    auto publish_choice = [&](int s_done, unsigned choice, int nf) {
        if (tid == 0 && cta == 0) {
            if (P.tokens_out) P.tokens_out[s_done] = choice;
            *P.last_token = choice;
            if (nf) atomicCAS(P.status, 0, (int)kDevNonfinite);
        }
    };

    unsigned prev_choice = *P.last_token;
    bool alive = true;
    int s = 0;
    for (; s < P.n_steps && alive; ++s) {
        const int p = P.p0 + s;
        const unsigned base = P.epoch + (unsigned)s * per_step;
        const bool trace_step = tracer && s == 0;
        if (s > 0) {
            if (!reduce_choice(base)) { alive = false; break; }
            prev_choice = *s_tok;
            const int nf = *s_nf;
            publish_choice(s - 1, prev_choice, nf);
            if (nf) { alive = false; break; }  // same decision in every CTA
        }
        // ---- token of this step
        unsigned tok = P.tokens_in ? P.tokens_in[s] : P.token0;
        if (tok == 0xFFFFFFFFu) tok = prev_choice;
        if (tok >= (unsigned)P.V) {
            if (tid == 0 && cta == 0) record_error(P, kDevToken);
            alive = false;
            break;
        }
        for (int l = 0; l < L && alive; ++l) {
            const LayerParams& lp = P.lp[l];
            const unsigned tQKV = base + 5u * (unsigned)l + 1u, tATT = tQKV + 1u, tO = tQKV + 2u, tFC = tQKV + 3u,
                           tP = tQKV + 4u;
            // ---------------- LN1 + QKV (+ KV append)
            {
                stamp(s, 0);
                float gr[PD], br[PD];
                load_ln<D>(P.packed + lp.ln1_g, P.packed + lp.ln1_b, gr, br, tid);
                const Geo g = geo_of(P, geot, 4 * l + kQKV);
                const float bv = bias_prefetch(g, lp.b_qkv);
                bool ok = true;
                if (l == 0) {
                    for (int i = tid; i < D; i += NT) {
                        const float pe = __ldg(P.packed + P.wpe_off + (uint64_t)p * D + i);
                        if constexpr (Q8) {
                            const uint8_t* row = P.vocab + (uint64_t)tok * row_bytes(D, true);
                            const float qv = (float)reinterpret_cast<const int8_t*>(row)[i];
                            const float sv = reinterpret_cast<const float*>(row + D)[i / kGroup];
                            xs[i] = __fadd_rn(__fmul_rn(qv, sv), pe);
                        } else {
                            xs[i] = __fadd_rn(__ldg(P.packed + P.wte_off + (uint64_t)tok * D + i), pe);
                        }
                    }
                } else {
                    ok = gather_vec<PD>(P.xa, D, tQKV - 1u, xs, tid, P);
                }
                bias_park(g, bv);
                if (!agree(ok)) { alive = false; break; }
                stamp(s, 1);
                layernorm_regs<D>(xs, gr, br, vin, red, tid);
                consumers_sync();
                quantize_in(D);
                if (trace_step) {
                    trace_vec(l * trace_layer, xs, D);
                    trace_vec(l * trace_layer + D, vin, D);
                }
                const Epi e{kQKV, out_tag(tQKV), lp.b_qkv, P.cache + ((uint64_t)p * L + l) * 2 * D, nullptr};
                stamp(s, 3);
                stamp_chunk = (s == 0);
                if (!agree(run_phase(KD{}, 4 * l + kQKV, e))) { alive = false; break; }
                stamp(s, 2);
            }
            // ---------------- attention over positions 0..p, split along keys
            // Unit (head h, split sp) covers keys [k0, k1).  A warp takes 8 keys
            // per pass (4 lanes per key, DH/4 dims per lane) and every lane keeps
            // an online softmax (running max, sum, weighted values).  Keys and
            // values of positions < p do not depend on this step, so the first
            // passes are loaded before waiting for q; position p's key and value
            // come from this step's tagged qkv words.
            const int S_eff = attn_splits_for(p + 1, S);
            {
                stamp(s, 0);
                const unsigned tg = out_tag(tATT);
                bool ok = true;
                bool first_unit = true;
                constexpr int LPK = DH >= 32 ? 8 : 4;    // lanes per key
                constexpr int KPW = 32 / LPK;            // keys per warp per pass
                constexpr int DPL = DH / LPK;            // dims per lane
                constexpr int F4 = DPL / 4;              // float4 per lane per row
                constexpr int KPP = kConsumerWarps * KPW;  // keys per pass over the CTA
                constexpr int PRE = 2;                   // passes loaded before the wait for q
                static_assert(DPL % 4 == 0, "a lane holds whole float4s of a head row");
                const int ks = lane / LPK, dc = lane % LPK;
                for (int u = cta; u < P.H * S_eff; u += P.G) {
                    const int h = u / S_eff, sp = u - h * S_eff;
                    const int n = p + 1;
                    const int k0 = (int)(((long long)sp * n) / S_eff), k1 = (int)(((long long)(sp + 1) * n) / S_eff);
                    const bool has_p = (k1 == n);  // the last split holds this position's key
                    float4 kr[PRE][F4], vr[PRE][F4];
#pragma unroll
                    for (int ps = 0; ps < PRE; ++ps) {
                        const int j = k0 + (ps * kConsumerWarps + warp) * KPW + ks;
                        if (j < k1 && j < p) {
                            const float* row = P.cache + ((uint64_t)j * L + l) * 2 * D + h * DH + dc * DPL;
#pragma unroll
                            for (int f = 0; f < F4; ++f) {
                                kr[ps][f] = __ldcg(reinterpret_cast<const float4*>(row) + f);
                                vr[ps][f] = __ldcg(reinterpret_cast<const float4*>(row + D) + f);
                            }
                        }
                    }
                    // q_h (threads 0..DH-1); k_p, v_p (DH..3DH-1) when this unit holds key p
                    uint64_t mine = 0;
                    const uint64_t* src = nullptr;
                    if (tid < DH) src = P.qkv + h * DH + tid;
                    else if (has_p && tid < 2 * DH) src = P.qkv + D + h * DH + (tid - DH);
                    else if (has_p && tid < 3 * DH) src = P.qkv + 2 * D + h * DH + (tid - 2 * DH);
                    if (src) mine = 1;
                    uint64_t wq[1];
                    const bool got = tagged_wait<1>(wq, mine, tQKV, [&](int) { return src; }, P);
                    if (src) qh[tid] = val_of(wq[0]);
                    if (!agree(got)) { ok = false; break; }
                    if (first_unit) stamp(s, 1);
                    first_unit = false;
                    const float4* q4 = reinterpret_cast<const float4*>(qh + dc * DPL);  // read from smem per key
                    const float den = sqrtf((float)DH);
                    float m = -INFINITY, z = 0.0f;
                    float acc[DPL];
#pragma unroll
                    for (int d = 0; d < DPL; ++d) acc[d] = 0.0f;
                    auto consume = [&](int j, const float4 (&kk)[F4], const float4 (&vv)[F4]) {
                        float dot = 0.0f;
#pragma unroll
                        for (int f = 0; f < F4; ++f) {
                            const float4 qf = q4[f];
                            dot += qf.x * kk[f].x + qf.y * kk[f].y + qf.z * kk[f].z + qf.w * kk[f].w;
                        }
#pragma unroll
                        for (int o = 1; o < LPK; o <<= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
                        if (j < k1) {
                            const float sc = dot / den;
                            const float mn = fmaxf(m, sc);
                            const float corr = expf(m - mn);  // 0 while m is -inf
                            const float e = expf(sc - mn);
                            z = fmaf(z, corr, e);
#pragma unroll
                            for (int f = 0; f < F4; ++f) {
                                acc[4 * f + 0] = fmaf(acc[4 * f + 0], corr, e * vv[f].x);
                                acc[4 * f + 1] = fmaf(acc[4 * f + 1], corr, e * vv[f].y);
                                acc[4 * f + 2] = fmaf(acc[4 * f + 2], corr, e * vv[f].z);
                                acc[4 * f + 3] = fmaf(acc[4 * f + 3], corr, e * vv[f].w);
                            }
                            m = mn;
                        }
                    };
                    auto fetch = [&](int j, float4 (&kk)[F4], float4 (&vv)[F4]) {
                        if (j < k1) {
                            if (j < p) {
                                const float* row = P.cache + ((uint64_t)j * L + l) * 2 * D + h * DH + dc * DPL;
#pragma unroll
                                for (int f = 0; f < F4; ++f) {
                                    kk[f] = __ldcg(reinterpret_cast<const float4*>(row) + f);
                                    vv[f] = __ldcg(reinterpret_cast<const float4*>(row + D) + f);
                                }
                            } else {
#pragma unroll
                                for (int f = 0; f < F4; ++f) {
                                    kk[f] = reinterpret_cast<const float4*>(qh + DH + dc * DPL)[f];
                                    vv[f] = reinterpret_cast<const float4*>(qh + 2 * DH + dc * DPL)[f];
                                }
                            }
                        }
                    };
#pragma unroll
                    for (int ps = 0; ps < PRE; ++ps) {
                        const int j = k0 + (ps * kConsumerWarps + warp) * KPW + ks;
                        if (j == p && j < k1) fetch(j, kr[ps], vr[ps]);
                        consume(j, kr[ps], vr[ps]);
                    }
                    for (int jb = k0 + PRE * KPP + warp * KPW; jb < k1; jb += KPP) {
                        float4 kk[F4], vv[F4];
                        fetch(jb + ks, kk, vv);
                        consume(jb + ks, kk, vv);
                    }
                    // merge the key slots of the warp (lanes with the same dc)
#pragma unroll
                    for (int o = LPK; o < 32; o <<= 1) {
                        const float om = __shfl_xor_sync(0xffffffffu, m, o);
                        const float oz = __shfl_xor_sync(0xffffffffu, z, o);
                        const float mn = fmaxf(m, om);
                        const float c1 = (m == -INFINITY) ? 0.0f : expf(m - mn);
                        const float c2 = (om == -INFINITY) ? 0.0f : expf(om - mn);
                        z = z * c1 + oz * c2;
#pragma unroll
                        for (int d = 0; d < DPL; ++d) {
                            const float oa = __shfl_xor_sync(0xffffffffu, acc[d], o);
                            acc[d] = acc[d] * c1 + oa * c2;
                        }
                        m = mn;
                    }
                    // then the warps: stage[w][dc][2 + DPL]
                    if (ks == 0) {
                        float* st = stage + (warp * LPK + dc) * (2 + DPL);
                        st[0] = m;
                        st[1] = z;
#pragma unroll
                        for (int d = 0; d < DPL; ++d) st[2 + d] = acc[d];
                    }
                    consumers_sync();
                    if (tid < DH) {
                        const int c = tid / DPL, d = tid - c * DPL;
                        float M = -INFINITY;
                        for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, stage[(w * LPK + c) * (2 + DPL)]);
                        float Z = 0.0f, O = 0.0f;
                        for (int w = 0; w < kConsumerWarps; ++w) {
                            const float* st = stage + (w * LPK + c) * (2 + DPL);
                            if (st[0] == -INFINITY) continue;
                            const float cw = expf(st[0] - M);
                            Z = fmaf(st[1], cw, Z);
                            O = fmaf(st[2 + d], cw, O);
                        }
                        uint64_t* part = P.attn_part + (size_t)u * (DH + 2);
                        st_tagged(part + 2 + tid, tg, O);
                        if (tid == 0) {
                            st_tagged(part, tg, M);
                            st_tagged(part + 1, tg, Z);
                        }
                    }
                    consumers_sync();
                }
                if (!ok) { alive = false; break; }
                if (first_unit) stamp(s, 1);
                stamp(s, 3);
                stamp(s, 2);
            }
            // ---------------- merge the heads' partials, out-projection + residual
            {
                stamp(s, 0);
                const Geo g = geo_of(P, geot, 4 * l + kO);
                const float bv = bias_prefetch(g, lp.b_o);
                const int units_eff = P.H * S_eff;
                // (max, sum) of every unit into stage[2u], stage[2u+1]
                const int nmz = 2 * units_eff;
                uint64_t wmz[2];
                const bool ok1 = tagged_wait<2>(
                    wmz, own_words<2>(nmz, tid), tATT,
                    [&](int k) {
                        const int w = tid + NT * k;
                        return P.attn_part + (size_t)(w >> 1) * (DH + 2) + (w & 1);
                    },
                    P);
#pragma unroll
                for (int k = 0; k < 2; ++k)
                    if (tid + NT * k < nmz) stage[tid + NT * k] = val_of(wmz[k]);
                // this thread's output coordinates idx = tid + NT*i: every split's o[e]
                uint64_t ov[PM];
                uint64_t want = 0;
#pragma unroll
                for (int i = 0; i < PD; ++i)
                    if (tid + NT * i < D)
                        for (int sp = 0; sp < S_eff; ++sp) want |= 1ull << (i * kMaxSplits + sp);
                const bool ok2 = tagged_wait<PM>(
                    ov, want, tATT,
                    [&](int k) {
                        const int idx = tid + NT * (k / kMaxSplits), sp = k % kMaxSplits;
                        const int h = idx / DH, e = idx - h * DH;
                        return P.attn_part + (size_t)(h * S_eff + sp) * (DH + 2) + 2 + e;
                    },
                    P);
                bias_park(g, bv);
                if (!agree(ok1 && ok2)) { alive = false; break; }
                stamp(s, 1);
                // weight of each (head, split): exp(m - M_h) / Z_h, once per CTA
                if (tid < units_eff) {
                    const int h = tid / S_eff;
                    float M = -INFINITY;
                    for (int sp = 0; sp < S_eff; ++sp) M = fmaxf(M, stage[2 * (h * S_eff + sp)]);
                    float Z = 0.0f;
                    for (int sp = 0; sp < S_eff; ++sp) {
                        const float ms = stage[2 * (h * S_eff + sp)];
                        if (ms != -INFINITY) Z = fmaf(expf(ms - M), stage[2 * (h * S_eff + sp) + 1], Z);
                    }
                    const float ms = stage[2 * tid];
                    ored[tid] = (ms == -INFINITY) ? 0.0f : expf(ms - M) / Z;
                }
                consumers_sync();
#pragma unroll
                for (int i = 0; i < PD; ++i) {
                    const int idx = tid + NT * i;
                    if (idx >= D) continue;
                    const int h = idx / DH;
                    float O = 0.0f;
#pragma unroll
                    for (int sp = 0; sp < kMaxSplits; ++sp) {
                        if (sp >= S_eff) break;
                        O = fmaf(ored[h * S_eff + sp], val_of(ov[i * kMaxSplits + sp]), O);
                    }
                    vin[idx] = O;
                }
                consumers_sync();
                quantize_in(D);
                if (trace_step) {
                    const bool okq = gather_vec<P3>(P.qkv, 3 * D, tQKV, P.trace + l * trace_layer + 2 * D, tid, P);
                    if (!agree(okq)) { alive = false; break; }
                    trace_vec(l * trace_layer + 5 * D, vin, D);
                }
                const Epi e{kO, out_tag(tO), lp.b_o, nullptr, nullptr};
                stamp(s, 3);
                stamp_chunk = (s == 0);
                if (!agree(run_phase(KD{}, 4 * l + kO, e))) { alive = false; break; }
                stamp(s, 2);
            }
            // ---------------- LN2 + FC + GELU
            {
                stamp(s, 0);
                float gr[PD], br[PD];
                load_ln<D>(P.packed + lp.ln2_g, P.packed + lp.ln2_b, gr, br, tid);
                const Geo g = geo_of(P, geot, 4 * l + kFC);
                const float bv = bias_prefetch(g, lp.b_fc);
                const bool ok = gather_vec<PD>(P.xb, D, tO, xs, tid, P);
                bias_park(g, bv);
                if (!agree(ok)) { alive = false; break; }
                stamp(s, 1);
                layernorm_regs<D>(xs, gr, br, vin, red, tid);
                consumers_sync();
                quantize_in(D);
                if (trace_step) {
                    trace_vec(l * trace_layer + 6 * D, xs, D);
                    trace_vec(l * trace_layer + 7 * D, vin, D);
                }
                const Epi e{kFC, out_tag(tFC), lp.b_fc, nullptr, nullptr};
                stamp(s, 3);
                stamp_chunk = (s == 0);
                if (!agree(run_phase(KD{}, 4 * l + kFC, e))) { alive = false; break; }
                stamp(s, 2);
            }
            // ---------------- MLP projection + residual
            {
                stamp(s, 0);
                const Geo g = geo_of(P, geot, 4 * l + kP);
                const float bv = bias_prefetch(g, lp.b_p);
                const bool ok = gather_vec<PF>(P.u, FF, tFC, vin, tid, P);
                bias_park(g, bv);
                if (!agree(ok)) { alive = false; break; }
                stamp(s, 1);
                quantize_in(FF);
                if (trace_step) trace_vec(l * trace_layer + 8 * D, vin, FF);
                const Epi e{kP, out_tag(tP), lp.b_p, nullptr, nullptr};
                stamp(s, 3);
                stamp_chunk = (s == 0);
                if (!agree(run_phase(KF{}, 4 * l + kP, e))) { alive = false; break; }
                stamp(s, 2);
            }
        }
        if (!alive) break;
        // ---------------- final LN + tied vocabulary projection + greedy choice
        {
            stamp(s, 0);
            const unsigned tVOC = base + per_step;
            float gr[PD], br[PD];
            load_ln<D>(P.packed + P.lnf_g, P.packed + P.lnf_b, gr, br, tid);
            const bool ok = gather_vec<PD>(P.xa, D, tVOC - 1u, xs, tid, P);
            if (!agree(ok)) { alive = false; break; }
            stamp(s, 1);
            layernorm_regs<D>(xs, gr, br, vin, red, tid);
            consumers_sync();
            quantize_in(D);
            if (trace_step) {
                trace_vec(L * trace_layer, xs, D);
                trace_vec(L * trace_layer + D, vin, D);
            }
            best = arg_init();
            const Epi e{kVocab, 0u, 0ull, nullptr, P.logits ? P.logits + (uint64_t)s * P.logits_stride : nullptr};
            stamp(s, 3);
            stamp_chunk = (s == 0);
            if (!agree(run_phase(KD{}, 4 * L, e))) { alive = false; break; }
            stamp(s, 2);
            arg_warp_reduce(best);
            if (lane == 0) {
                s_arg[warp * 3 + 0] = best.v;
                s_arg[warp * 3 + 1] = __uint_as_float(best.i);
                s_arg[warp * 3 + 2] = (float)best.nf;
            }
            consumers_sync();
            if (tid == 0) {
                for (int w = 1; w < kConsumerWarps; ++w)
                    arg_merge(best, s_arg[w * 3 + 0], __float_as_uint(s_arg[w * 3 + 1]), s_arg[w * 3 + 2] != 0.0f);
                const unsigned tg = out_tag(tVOC);
                uint64_t* ap = P.arg_part + 2 * (size_t)cta;
                const unsigned iw = (best.i & 0x7FFFFFFFu) | (best.nf ? 0x80000000u : 0u);
                st_tagged(ap + 1, tg, __uint_as_float(iw));
                // release: this CTA's KV rows and choice become visible with it
                st_tagged_release(ap, tag_pack(tg, best.v));
            }
        }
    }
    // The last step's greedy choice (CTA 0 reports it).
    if (alive && s == P.n_steps && cta == 0) {
        if (reduce_choice(P.epoch + (unsigned)P.n_steps * per_step)) publish_choice(s - 1, *s_tok, *s_nf);
    }
    // Make the producer stop if the consumers left early.
    if (tid == 0) *s_abort = 1;
}

// ------------------------------------------------------------ test hooks
// One projection of the model on a given input vector, with the step
// kernel's own routines: the activation quantizer and the window GEMV
// (win_f32 / win_q8), then the epilogue's bias add.  Block: the consumer
// warps, one window of rows copied into a ring-shaped shared buffer.
template <int K, bool Q8>
__host__ __device__ constexpr uint32_t project_smem_bytes() {
    using W = WinGeo<K, Q8>;
    return (uint32_t)W::CPW * kSlotBytes + align16(K * 4) + align16(K) + align16((K / kGroup) * 4) +
           (uint32_t)kCoopTaskFloats * 4;
}

template <int K, bool Q8>
__global__ void __launch_bounds__(kConsumerWarps * 32) project_kernel(const uint8_t* __restrict__ rows, int N,
                                                                      const float* __restrict__ x,
                                                                      const float* __restrict__ bias,
                                                                      float* __restrict__ y) {
    using W = WinGeo<K, Q8>;
    extern __shared__ __align__(128) uint8_t sm[];
    uint8_t* ring = sm;
    float* vin = reinterpret_cast<float*>(sm + W::CPW * kSlotBytes);
    int8_t* vq = reinterpret_cast<int8_t*>(reinterpret_cast<uint8_t*>(vin) + align16(K * 4));
    float* vs = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(vq) + align16(K));
    float* scratch = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(vs) + align16((K / kGroup) * 4));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int w0 = blockIdx.x * W::WR;
    const int wn = min(W::WR, N - w0);
    // rows w0 .. w0+wn-1 into "slots": row r at slot r / RPC, offset (r % RPC) * RB
    for (int i = tid; i < wn * (W::RB / 16); i += blockDim.x) {
        const int r = i / (W::RB / 16), q = i - r * (W::RB / 16);
        const int4 v = reinterpret_cast<const int4*>(rows + (size_t)(w0 + r) * W::RB)[q];
        reinterpret_cast<int4*>(ring + (size_t)(r / W::RPC) * kSlotBytes + (size_t)(r % W::RPC) * W::RB)[q] = v;
    }
    for (int i = tid; i < K; i += blockDim.x) vin[i] = x[i];
    __syncthreads();
    if constexpr (Q8) quantize_vec<K>(vin, vq, vs, warp, lane);
    __syncthreads();
    float out;
    if constexpr (Q8) out = win_q8<K>(ring, 0, wn, vq, vs, scratch, tid);
    else out = win_f32<K>(ring, 0, wn, vin, scratch, tid, lane, warp);
    if (tid < wn) y[w0 + tid] = bias ? __fadd_rn(out, bias[w0 + tid]) : out;
}

// The step kernel's greedy-choice routine over n values (one block).
__global__ void __launch_bounds__(kConsumerWarps * 32) argmax_kernel(const float* __restrict__ v, unsigned n,
                                                                     uint32_t* idx, int* nonfinite) {
    __shared__ float s_arg[kConsumerWarps * 3];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    ArgBest b = arg_init();
    for (unsigned j = tid; j < n; j += blockDim.x) arg_update(b, v[j], j);
    arg_warp_reduce(b);
    if (lane == 0) {
        s_arg[warp * 3 + 0] = b.v;
        s_arg[warp * 3 + 1] = __uint_as_float(b.i);
        s_arg[warp * 3 + 2] = (float)b.nf;
    }
    __syncthreads();
    if (tid == 0) {
        for (int w = 1; w < kConsumerWarps; ++w)
            arg_merge(b, s_arg[w * 3 + 0], __float_as_uint(s_arg[w * 3 + 1]), s_arg[w * 3 + 2] != 0.0f);
        *idx = b.nf ? 0xFFFFFFFFu : b.i;
        *nonfinite = b.nf;
    }
}

template <int K, bool Q8>
static cudaError_t project_t(const uint8_t* rows, int N, const float* x, const float* bias, float* y,
                             cudaStream_t st) {
    constexpr int rows_per_block = WinGeo<K, Q8>::WR;
    constexpr uint32_t smem = project_smem_bytes<K, Q8>();
    cudaError_t e = cudaFuncSetAttribute(project_kernel<K, Q8>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    project_kernel<K, Q8><<<(N + rows_per_block - 1) / rows_per_block, kConsumerWarps * 32, smem, st>>>(rows, N, x,
                                                                                                      bias, y);
    return cudaGetLastError();
}

cudaError_t launch_project(const uint8_t* rows, int K, int N, bool q8, const float* x, const float* bias, float* y,
                           cudaStream_t st) {
#define GPT2_PROJ(KK)                                                                             \
    if (K == KK) return q8 ? project_t<KK, true>(rows, N, x, bias, y, st) : project_t<KK, false>(rows, N, x, bias, y, st);
    GPT2_PROJ(64) GPT2_PROJ(192) GPT2_PROJ(256) GPT2_PROJ(384) GPT2_PROJ(768) GPT2_PROJ(3072)
#undef GPT2_PROJ
    return cudaErrorInvalidValue;
}

cudaError_t launch_argmax(const float* v, unsigned n, uint32_t* idx, int* nonfinite, cudaStream_t st) {
    argmax_kernel<<<1, kConsumerWarps * 32, 0, st>>>(v, n, idx, nonfinite);
    return cudaGetLastError();
}

// ------------------------------------------------------------ launcher
template <int D, int FF, int DH, bool Q8>
static cudaError_t launch_t(const StepPlan& P, cudaStream_t stream) {
    const SmemLayout lay = smem_layout(D, FF, Q8, P.max_pos);
    auto kern = step_kernel<D, FF, DH, Q8>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)lay.total);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(P.G);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = lay.total;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, P);
}

template <int D, int FF, int DH, bool Q8>
static int max_ctas_t(int max_pos) {
    const SmemLayout lay = smem_layout(D, FF, Q8, max_pos);
    auto kern = step_kernel<D, FF, DH, Q8>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)lay.total) != cudaSuccess)
        return 0;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, lay.total) != cudaSuccess) return 0;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    return per_sm * sms < kMaxGrid ? per_sm * sms : kMaxGrid;
}

bool step_shape_supported(int D, int FF, int DH) {
    return (D == 768 && FF == 3072 && DH == 64) || (D == 192 && FF == 384 && DH == 64) ||
           (D == 64 && FF == 256 && DH == 16);
}

uint32_t step_smem_bytes(int D, int FF, bool q8, int max_pos) { return smem_layout(D, FF, q8, max_pos).total; }

#define GPT2_DISPATCH(FN, ...)                                                                  \
    if (D == 768 && FF == 3072 && DH == 64)                                                      \
        return q8 ? FN<768, 3072, 64, true>(__VA_ARGS__) : FN<768, 3072, 64, false>(__VA_ARGS__); \
    if (D == 192 && FF == 384 && DH == 64)                                                       \
        return q8 ? FN<192, 384, 64, true>(__VA_ARGS__) : FN<192, 384, 64, false>(__VA_ARGS__);   \
    if (D == 64 && FF == 256 && DH == 16)                                                        \
        return q8 ? FN<64, 256, 16, true>(__VA_ARGS__) : FN<64, 256, 16, false>(__VA_ARGS__);

cudaError_t launch_step(const StepPlan& P, bool q8, cudaStream_t stream) {
    const int D = P.D, FF = P.FF, DH = P.D / P.H;
    GPT2_DISPATCH(launch_t, P, stream)
    return cudaErrorInvalidValue;
}

int step_max_ctas(int D, int FF, int DH, bool q8, int max_pos) {
    GPT2_DISPATCH(max_ctas_t, max_pos)
    return 0;
}

}  // namespace gpt2
