// decode.cu -- the persistent GPT-2 step kernel.
//
// One cooperative launch runs n_steps cached steps (LeanExe GPT-2 README,
// cachedStep paragraph; model description paragraph for the block order):
//   embed -> per layer [LN1 + QKV, KV append, attention, out-proj + residual,
//   LN2 + FC + GELU, MLP-proj + residual] -> LN_f + tied vocab projection ->
//   greedy argmax.
//
// This is the step kernel for int8 models (and for every format when
// GPT2_STEP_KERNEL=legacy); binary32 and binary16 models step on the cluster
// kernel in cstep.cu.
//
// Work split: every projection is split by OUTPUT rows across the G CTAs
// (one per SM).  The device keeps every block matrix K-major ([out][in], one
// contiguous row per output), so CTA c's share of a matrix is one contiguous
// byte range.  Each CTA has 7 consumer warps and 1 producer warp; the
// producer streams this CTA's shares of all matrices, in step order, through
// a ring of shared-memory slots with cp.async.bulk and mbarriers and never
// waits on activations, so weight streaming runs ahead of the grid-wide
// dependencies (bounded by the ring depth).  Small shares are computed
// cooperatively by the whole CTA from registers; the vocabulary streams one
// warp per chunk.  Complete dot products need no cross-CTA reduction.
//
// Exchange between phases: every value a phase publishes is one 64-bit
// tagged word (phase tag << 32 | float bits), stored relaxed at gpu scope
// and polled by its consumers until the tag matches; a 64-bit word is
// single-copy atomic, so no flag or fence is needed per phase.  The only
// release/acquire is one per step, on the greedy partials, which orders the
// plain KV-cache stores before the next step's attention.  Every spin-wait
// is bounded by a wall-clock limit after which the kernel records
// GPT2_ERR_TIMEOUT, sets a global abort word, drains its own bulk copies and
// returns.
//
// Attention is split along the key axis ("flash-decoding" split-KV, lean /
// llm-web page, GPU-path paragraph): a unit is (head, key split), one split
// per 128 keys.  Up to 128 keys a head is a single unit whose output is
// normalised, and the out-projection gathers it like any vector; with
// several splits each unit stores (max, sum, unnormalised o) and the
// out-projection merges them by the log-sum-exp rule before its GEMV.
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
    uint32_t ring, full, empty, xs, vin, vq, vs, red, ored, qh, rsc, stage, fpart, bias, geot, misc, plan, total;
};

__host__ __device__ constexpr uint32_t align16(uint32_t x) { return (x + 15u) & ~15u; }

// `stage` holds, at different times: the attention warp merge
// [warps][8 lanes][2 + 8] (head dim 64), the (max, sum) pairs of every
// attention unit (2 * 12 heads * kMaxSplits), and the per-CTA greedy choices
// [256 + kMaxGrid].
constexpr int kStageFloats = 640;
// int8 rescale terms, per consumer warp: [rows][groups] of one pass.
constexpr int kWarpScratch = 192;
constexpr int kCoopTaskFloats = kConsumerWarps * kWarpScratch;
static_assert(kConsumerWarps * 8 * (2 + 8) <= kStageFloats, "attention warp merge fits in stage");
static_assert(2 * 16 * kMaxSplits <= kStageFloats, "unit (max, sum) pairs fit in stage");
static_assert(256 + kMaxGrid <= kStageFloats, "greedy choices fit in stage");
constexpr int kMaxChunkRows = 32;
// Rows of a spread share (computed by the whole CTA once its chunks landed).
constexpr int kSpreadRows = 32;
// Fast phases alternate between two sets of [warps][kSpreadRows] row
// partials and [warps] (sum x, sum x^2) pairs, so that one phase's partials
// can be written while slower threads still read the previous phase's.
constexpr int kFastSet = kConsumerWarps * kSpreadRows + 2 * kConsumerWarps;
constexpr int kFastPartFloats = 2 * kFastSet;

__host__ __device__ inline SmemLayout smem_layout(int D, int FF, bool q8, int max_pos) {
    SmemLayout s{};
    int kmax = D > FF ? D : FF;
    uint32_t o = 0;
    s.ring = o; o += kSlots * kSlotBytes;
    s.full = o; o += kSlots * 8;
    s.empty = o; o += kSlots * 8;
    s.xs = o; o = align16(o + D * 4);
    s.vin = o; o = align16(o + (kmax > kMaxSplits * D ? kmax : kMaxSplits * D) * 4);  // also every split's head outputs
    s.vq = o; o = align16(o + (q8 ? kmax : 0));
    s.vs = o; o = align16(o + (kmax / kGroup) * 4);
    s.red = o; o = align16(o + 64 * 4);
    s.ored = o; o = align16(o + kConsumerWarps * 32 * 4);
    s.qh = o; o = align16(o + 3 * 64 * 4);  // q_h, k_p, v_p of one attention unit
    s.rsc = o; o = align16(o + (q8 ? kCoopTaskFloats * 4 : 0));  // int8 rescale terms
    s.stage = o; o = align16(o + kStageFloats * 4);  // attention warp merge; (max, sum) pairs; greedy choices
    s.fpart = o; o = align16(o + kFastPartFloats * 4);  // fast phases: two alternating sets of row partials + LN sums
    s.bias = o; o = align16(o + kConsumerWarps * 32 * 4);
    s.geot = o; o = align16(o + 5 * 32);  // GeoRow table
    s.misc = o; o = align16(o + 64 * 4);
    s.plan = o; o = align16(o + (uint32_t)sizeof(StepPlan));  // the launch's plan, copied once
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

__device__ __forceinline__ Geo phase_geo(const StepPlan& P, int ph, int cta, int wf) {
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
    g.rb = row_bytes(K, wf);
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

// Quantize v[0..N) per group of 64 into q/s (int8 path).  Warp w owns groups
// w, w + warps, ...; its groups are loaded, reduced and quantized together so
// the shuffles and divisions of different groups overlap.
// With row set, one scale for the whole vector instead (the largest |v| of
// all N, reduced through red[kConsumerWarps] with one consumer barrier),
// written to every group's slot.
__device__ __forceinline__ float row_absmax(float m, float* red, int warp, int lane) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0) red[warp] = m;
    consumers_sync();
    float r = 0.0f;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) r = fmaxf(r, red[w]);
    return r;
}

template <int N>
__device__ __forceinline__ void quantize_vec(const float* v, int8_t* q, float* s, int warp, int lane, bool row,
                                             float* red) {
    constexpr int NG = N / kGroup;
    constexpr int GPW = (NG + kConsumerWarps - 1) / kConsumerWarps;  // groups per warp (at most)
    float mrow = 0.0f;
    if (row) {
        float m = 0.0f;
        for (int i = warp * 32 + lane; i < N; i += kConsumerWarps * 32) m = fmaxf(m, fabsf(v[i]));
        mrow = row_absmax(m, red, warp, lane);
    }
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
            const float sc = __fdiv_rn(row ? mrow : m[k], 127.0f), inv = __frcp_rn(sc);
            q[gi * kGroup + lane] = (int8_t)quantize_fast(a[k], sc, inv);
            q[gi * kGroup + 32 + lane] = (int8_t)quantize_fast(b[k], sc, inv);
            if (lane == 0) s[gi] = sc;
        }
    }
}

// Quantize a K-vector held in the quad layout (thread tid owns float4
// columns tid + NT*k) per group of 64 into q/s: a group is 16 consecutive
// columns, i.e. one half-warp, so its largest |v| is four shuffles away.
// Same rule as quantize_vec; the maximum is exact in any order.  Every
// consumer thread calls it (the shuffles take all lanes).
template <int K>
__device__ __forceinline__ void quantize_quads(const float (&x)[4 * ((K / 4 + kConsumerWarps * 32 - 1) /
                                                                      (kConsumerWarps * 32))],
                                               int8_t* q, float* s, int tid, bool row, float* red) {
    constexpr int NT = kConsumerWarps * 32, NV = K / 4, NC = (NV + NT - 1) / NT;
    static_assert(K % kGroup == 0 && NT % 16 == 0, "groups are whole half-warps");
    auto absmax4 = [&](int cc) {
        // max of |v| starting from 0; NaN never wins a comparison
        return fmaxf(fmaxf(fmaxf(fabsf(x[4 * cc]), fabsf(x[4 * cc + 1])), fmaxf(fabsf(x[4 * cc + 2]), fabsf(x[4 * cc + 3]))),
                     0.0f);
    };
    float mrow = 0.0f;
    if (row) {
        float m = 0.0f;
#pragma unroll
        for (int cc = 0; cc < NC; ++cc)
            if (tid + NT * cc < NV) m = fmaxf(m, absmax4(cc));
        mrow = row_absmax(m, red, tid >> 5, tid & 31);
    }
#pragma unroll
    for (int cc = 0; cc < NC; ++cc) {
        const int col = tid + NT * cc;
        float m = absmax4(cc);
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        if (row) m = mrow;
        if (col < NV) {
            const float sc = __fdiv_rn(m, 127.0f), inv = __frcp_rn(sc);
            const uint32_t b0 = (uint32_t)(uint8_t)(int8_t)quantize_fast(x[4 * cc], sc, inv);
            const uint32_t b1 = (uint32_t)(uint8_t)(int8_t)quantize_fast(x[4 * cc + 1], sc, inv);
            const uint32_t b2 = (uint32_t)(uint8_t)(int8_t)quantize_fast(x[4 * cc + 2], sc, inv);
            const uint32_t b3 = (uint32_t)(uint8_t)(int8_t)quantize_fast(x[4 * cc + 3], sc, inv);
            reinterpret_cast<uint32_t*>(q)[col] = b0 | (b1 << 8) | (b2 << 16) | (b3 << 24);
            if ((col & 15) == 0) s[col >> 4] = sc;
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

// ---------------------------------------------------------- projection cores
// A phase share (this CTA's rows of one matrix, input width K) arrives in
// ring chunks of RPC rows of RB bytes; chunk c of the ring sequence sits in
// slot c % kSlots.
//
// Spread shares (all chunks fit in half the ring, at most kSpreadRows rows)
// are computed cooperatively by the whole CTA once every chunk has landed:
// each weight byte is read from shared memory once and every thread works.
// Longer shares (the vocabulary) stream: one warp per chunk, chunks
// released as they are used.
template <int K, int WF>
struct Rows {
    static constexpr int RB = row_bytes(K, WF);                               // bytes per row
    static constexpr int RPC0 = kSlotBytes / RB;
    static constexpr int RPC = RPC0 > kMaxChunkRows ? kMaxChunkRows : RPC0;  // rows per chunk
    static constexpr int NG = K / kGroup;                                     // int8 groups per row
};

__host__ __device__ constexpr bool share_spread(int nchunks, int nrows, int K, bool q8) {
    return nchunks <= kSlots / 2 && nrows <= kSpreadRows && (!q8 || nrows * (K / kGroup) <= kCoopTaskFloats) &&
           (q8 || K / 4 <= kConsumerWarps * 32 || nrows <= 8);  // rows longer than the CTA: groups of 4 + 4
}

// Column layout of a spread binary32 share: thread t takes the float4
// columns t, t + NT, ... of every row of the share.
template <int K>
struct Pre {
    static constexpr int NT = kConsumerWarps * 32;
    static constexpr int NV = K / 4;                 // float4 columns per row
    static constexpr int NC = (NV + NT - 1) / NT;    // columns per thread
};

template <int K, int WF = kWF32>
__device__ __forceinline__ uint32_t share_row_off(uint32_t c0, int r) {
    using R = Rows<K, WF>;
    return ((c0 + (uint32_t)(r / R::RPC)) % kSlots) * (uint32_t)kSlotBytes + (uint32_t)((r % R::RPC) * R::RB);
}

// The cooperative projection of a spread share, rows R0..R0+NR-1 that are
// below nrows, against x held in registers (this thread's float4 columns,
// quad layout), weights from shared memory; the warp's partial of row r
// goes to part[warp][r].  (Variants that keep more values live -- weight
// rows held in registers across the input wait, or every load of a row
// group issued before its multiply-adds -- measured slower: the step kernel
// is at its register limit and the extra live values spill.)
// Four consecutive weights of a binary32 or binary16 row, as binary32.
template <int WF>
__device__ __forceinline__ float4 weight4(const uint8_t* row, int col) {
    if constexpr (WF == kWF16) {
        const uint2 h = *reinterpret_cast<const uint2*>(row + 8u * (uint32_t)col);
        const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&h.x));
        const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&h.y));
        return make_float4(a.x, a.y, b.x, b.y);
    } else {
        return *reinterpret_cast<const float4*>(row + 16u * (uint32_t)col);
    }
}

template <int K, int NR, int R0, int WF = kWF32>
__device__ __forceinline__ void coop_reg_part(const uint8_t* ring, uint32_t c0, int nrows,
                                              const float (&x)[4 * Pre<K>::NC], float* part, int tid) {
    using Q = Pre<K>;
    const int warp = tid >> 5, lane = tid & 31;
    // whole warps past the row have no columns: their partials are zero
    if ((Q::NV % Q::NT) != 0 && Q::NC == 1 && (warp * 32) >= Q::NV) {
        if (lane < NR && R0 + lane < nrows) part[warp * kSpreadRows + R0 + lane] = 0.0f;
        return;
    }
    float acc[NR];
#pragma unroll
    for (int i = 0; i < NR; ++i) acc[i] = 0.0f;
#pragma unroll
    for (int cc = 0; cc < Q::NC; ++cc) {
        const int col = tid + Q::NT * cc;
        if (col < Q::NV) {
            const float4 xv = make_float4(x[4 * cc], x[4 * cc + 1], x[4 * cc + 2], x[4 * cc + 3]);
#pragma unroll
            for (int i = 0; i < NR; ++i) {
                const int r = R0 + i;
                if (r < nrows) {
                    const float4 wv = weight4<WF>(ring + share_row_off<K, WF>(c0, r), col);
                    acc[i] = fmaf(xv.x, wv.x, acc[i]);
                    acc[i] = fmaf(xv.y, wv.y, acc[i]);
                    acc[i] = fmaf(xv.z, wv.z, acc[i]);
                    acc[i] = fmaf(xv.w, wv.w, acc[i]);
                }
            }
        }
    }
    const float t = warp_transpose_sum<NR>(acc, lane);
    if (lane < NR && R0 + lane < nrows) part[warp * kSpreadRows + R0 + lane] = t;
}

// Rows 0..nrows-1 (<= kSpreadRows) of a spread share against x (quad
// layout, registers), in power-of-two row groups: the warps' partials of
// every row to part; the caller's barrier then lets the row's thread sum
// them in warp order.
template <int K, int WF = kWF32>
__device__ __forceinline__ void coop_reg(const uint8_t* ring, uint32_t c0, int nrows, const float (&x)[4 * Pre<K>::NC],
                                         float* part, int tid) {
    if constexpr (Pre<K>::NC == 1) {
        // rows of at most the CTA's width: groups of 16, the tail in 8
        if (nrows > 16) {
            coop_reg_part<K, 16, 0, WF>(ring, c0, nrows, x, part, tid);
            if (nrows > 24) coop_reg_part<K, 16, 16, WF>(ring, c0, nrows, x, part, tid);
            else coop_reg_part<K, 8, 16, WF>(ring, c0, nrows, x, part, tid);
        } else if (nrows > 8) {
            coop_reg_part<K, 16, 0, WF>(ring, c0, nrows, x, part, tid);
        } else {
            coop_reg_part<K, 8, 0, WF>(ring, c0, nrows, x, part, tid);
        }
    } else {
        // long rows (at most 8 per spread share): groups of 4 and 2 waste fewer loads
        if (nrows > 4) {
            coop_reg_part<K, 4, 0, WF>(ring, c0, nrows, x, part, tid);
            if (nrows > 6) coop_reg_part<K, 4, 4, WF>(ring, c0, nrows, x, part, tid);
            else coop_reg_part<K, 2, 4, WF>(ring, c0, nrows, x, part, tid);
        } else {
            coop_reg_part<K, 4, 0, WF>(ring, c0, nrows, x, part, tid);
        }
    }
}

// This thread's float4 columns of a K-vector in shared memory (quad layout).
template <int K>
__device__ __forceinline__ void load_quads(const float* v, float (&x)[4 * Pre<K>::NC], int tid) {
    using Q = Pre<K>;
#pragma unroll
    for (int cc = 0; cc < Q::NC; ++cc) {
        const int col = tid + Q::NT * cc;
        const float4 t = col < Q::NV ? reinterpret_cast<const float4*>(v)[col] : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        x[4 * cc] = t.x;
        x[4 * cc + 1] = t.y;
        x[4 * cc + 2] = t.z;
        x[4 * cc + 3] = t.w;
    }
}

// Row r's total from the warps' partials, summed in warp order.
__device__ __forceinline__ float sum_warp_parts(const float* part, int r) {
    float y = 0.0f;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) y += part[w * kSpreadRows + r];
    return y;
}

// Exact int32 sum of the 64 products of one group (two independent dp4a
// chains; integer addition is exact in any order).  The four 16-byte
// quarters are read starting at quarter rot: lanes whose groups lie 64
// bytes apart then hit eight distinct bank groups per load instead of two.
__device__ __forceinline__ int group_dot(const uint8_t* w, const int8_t* x, int rot) {
    const int4* wv = reinterpret_cast<const int4*>(w);
    const int4* xv = reinterpret_cast<const int4*>(x);
    int a0 = 0, a1 = 0;
#pragma unroll
    for (int v = 0; v < 4; v += 2) {
        const int j0 = (v + rot) & 3, j1 = (v + 1 + rot) & 3;
        const int4 p = wv[j0], q = xv[j0], r = wv[j1], s = xv[j1];
        a0 = __dp4a(p.x, q.x, a0);
        a1 = __dp4a(r.x, s.x, a1);
        a0 = __dp4a(p.y, q.y, a0);
        a1 = __dp4a(r.y, s.y, a1);
        a0 = __dp4a(p.z, q.z, a0);
        a1 = __dp4a(r.z, s.z, a1);
        a0 = __dp4a(p.w, q.w, a0);
        a1 = __dp4a(r.w, s.w, a1);
    }
    return a0 + a1;
}

// The rescale term of one (row, group): ((float)acc * s_x[g]) * s_w[g],
// explicitly rounded; rot: the caller's lane-dependent quarter rotation.
__device__ __forceinline__ float group_term(const uint8_t* row, int g, int K, const int8_t* xq, const float* xs,
                                           int rot) {
    const int acc = group_dot(row + g * kGroup, xq + g * kGroup, rot);
    return __fmul_rn(__fmul_rn(__int2float_rn(acc), xs[g]), reinterpret_cast<const float*>(row + K)[g]);
}

// Ordered rescale sum of one row: t[0] + t[1] + ... from 0.0f, explicitly
// rounded (the fixed int8 rescale order).
template <int NG>
__device__ __forceinline__ float ordered_sum(const float* t) {
    float sum = 0.0f;
    if constexpr ((NG & 3) == 0) {
#pragma unroll
        for (int g = 0; g < NG; g += 4) {
            const float4 v = *reinterpret_cast<const float4*>(t + g);
            sum = __fadd_rn(__fadd_rn(__fadd_rn(__fadd_rn(sum, v.x), v.y), v.z), v.w);
        }
    } else {
#pragma unroll
        for (int g = 0; g < NG; ++g) sum = __fadd_rn(sum, t[g]);
    }
    return sum;
}

// int8, cooperative: the (row, group) tasks of the share are spread over
// every consumer thread; task terms go to scr[row][group]; thread r < nrows
// returns row r's ordered sum, others 0.  Contains a barrier over the
// consumer warps.
template <int K>
__device__ __forceinline__ float coop_q8(const uint8_t* ring, uint32_t c0, int nrows, const int8_t* xq,
                                         const float* xs, float* scr, int tid) {
    using R = Rows<K, true>;
    constexpr int NT = kConsumerWarps * 32;
    for (int tk = tid; tk < nrows * R::NG; tk += NT) {
        const int i = tk / R::NG, g = tk - i * R::NG;
        const uint8_t* row = ring + (size_t)((c0 + (uint32_t)(i / R::RPC)) % kSlots) * kSlotBytes +
                             (size_t)((i % R::RPC) * R::RB);
        scr[tk] = group_term(row, g, K, xq, xs, (tid >> 1) & 3);
    }
    consumers_sync();
    return tid < nrows ? ordered_sum<R::NG>(scr + tid * R::NG) : 0.0f;
}

// Rows one streaming call covers: binary32 keeps four accumulators per
// lane; int8 is bounded by the warp's rescale scratch.
template <int K, bool Q8>
__host__ __device__ constexpr int dot_rows() {
    return !Q8 ? 4 : ((kWarpScratch / (K / kGroup)) < 32 ? (kWarpScratch / (K / kGroup)) : 32);
}

// binary32 or binary16 weights, streaming: m <= 4 consecutive rows at w against x[0..K); lane
// i < m returns row i's total.  Lanes stride float4 columns; one butterfly
// transpose per call.
template <int K, int WF = kWF32>
__device__ __forceinline__ float dot_f32(const uint8_t* w, int m, const float* x, int lane) {
    using R = Rows<K, WF>;
    constexpr int NV = K / 4, T = (NV + 31) / 32;
    const float4* x4 = reinterpret_cast<const float4*>(x);
    float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll 2
    for (int t = 0; t < T; ++t) {
        const int idx = lane + 32 * t;
        if ((NV % 32) == 0 || idx < NV) {
            const float4 xv = x4[idx];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                if (i < m) {
                    const float4 wv = weight4<WF>(w + (size_t)i * R::RB, idx);
                    acc[i] = fmaf(xv.x, wv.x, acc[i]);
                    acc[i] = fmaf(xv.y, wv.y, acc[i]);
                    acc[i] = fmaf(xv.z, wv.z, acc[i]);
                    acc[i] = fmaf(xv.w, wv.w, acc[i]);
                }
            }
        }
    }
    return warp_transpose_sum<4>(acc, lane);
}

// int8, streaming: m consecutive rows at w (m * K/64 <= kWarpScratch);
// lanes take (row, group) tasks; lane i < m returns row i's ordered sum.
// scr: this warp's scratch.
template <int K>
__device__ __forceinline__ float dot_q8(const uint8_t* w, int m, const int8_t* xq, const float* xs, float* scr,
                                        int lane) {
    using R = Rows<K, true>;
#pragma unroll 2
    for (int tk = lane; tk < m * R::NG; tk += 32) {
        const int i = tk / R::NG, g = tk - i * R::NG;
        scr[tk] = group_term(w + (size_t)i * R::RB, g, K, xq, xs, (lane >> 1) & 3);
    }
    __syncwarp();
    const float sum = lane < m ? ordered_sum<R::NG>(scr + lane * R::NG) : 0.0f;
    __syncwarp();
    return sum;
}

// -------------------------------------------------------------- kernel
// Waits until every word k with bit k set in `pending` carries `tag`,
// leaving the raw words in w[] (decode with val_of).  MAXC bounds k at
// compile time so the words stay in registers; all pending words are
// reloaded together, so one round costs one L2 round trip.  Returns false
// when the run is abandoned (another CTA gave up, or the wait exceeded its
// limit).
// Every spin-wait reads the grid's abort word only once it has lasted
// kAbortCheckNs: one word polled by every thread of every CTA makes a hot L2
// line that slows every exchange; no wait of a healthy run lasts this long.
constexpr uint64_t kAbortCheckNs = 20000;
__device__ __forceinline__ bool waited_long(uint64_t elapsed_ns) { return elapsed_ns > kAbortCheckNs; }

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
            const uint64_t now = globaltimer_ns();
            if (t0 == 0) t0 = now;
            else if (waited_long(now - t0) && ld_volatile_int(P.abort_flag)) return false;
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

// Pair layout of a vector held in registers: thread tid owns the word
// pairs q = tid + NT*k (k < PP), i.e. elements 2q and 2q + 1, so that each
// tagged load moves 16 bytes (two words) and a warp's loads are contiguous.
template <int N>
struct Pairs {
    static constexpr int NT = kConsumerWarps * 32;
    static constexpr int NP = N / 2;                   // pairs in the vector
    static constexpr int PP = (NP + NT - 1) / NT;      // pairs per thread (at most)
};

// Waits until both words of each of this thread's pairs carry `tag` and
// returns their values in v[2k], v[2k + 1]; addr(q) is the first word of
// pair q (16-byte aligned).  Returns false when the run is abandoned.
template <int PP, typename Addr>
__device__ __forceinline__ bool gather_pairs(float (&v)[2 * PP], int npairs, unsigned tag, Addr addr, int tid,
                                             const StepPlan& P) {
    constexpr int NT = kConsumerWarps * 32;
    uint32_t pending = 0;
#pragma unroll
    for (int k = 0; k < PP; ++k) {
        v[2 * k] = 0.0f;
        v[2 * k + 1] = 0.0f;
        if (tid + NT * k < npairs) pending |= 1u << k;
    }
    uint64_t t0 = 0;
    uint32_t rounds = 0;
    while (pending) {
        uint64_t a[PP], b[PP];
#pragma unroll
        for (int k = 0; k < PP; ++k)
            if ((pending >> k) & 1u) ld_tagged_x2(addr(tid + NT * k), a[k], b[k]);
#pragma unroll
        for (int k = 0; k < PP; ++k)
            if (((pending >> k) & 1u) && tag_of(a[k]) == tag && tag_of(b[k]) == tag) {
                v[2 * k] = val_of(a[k]);
                v[2 * k + 1] = val_of(b[k]);
                pending &= ~(1u << k);
            }
        if (pending && (++rounds & 7u) == 0) {
            const uint64_t now = globaltimer_ns();
            if (t0 == 0) t0 = now;
            else if (waited_long(now - t0) && ld_volatile_int(P.abort_flag)) return false;
            else if (now - t0 > P.wait_limit_ns) {
                record_error(P, kDevTimeout);
                return false;
            }
        }
    }
    return true;
}

// Waits until the four words of each of this thread's quads (float4
// columns c = tid + NT*k, k < NQ, c < nquads) carry `tag` and returns
// their values in x[4k .. 4k+3]; addr(c) is the first word of quad c (four
// consecutive words, 16-byte aligned).  Returns false when the run is
// abandoned.
template <int NQ, typename Addr>
__device__ __forceinline__ bool gather_quads(float (&x)[4 * NQ], int nquads, unsigned tag, Addr addr, int tid,
                                             const StepPlan& P) {
    constexpr int NT = kConsumerWarps * 32;
    uint32_t pending = 0;
#pragma unroll
    for (int k = 0; k < NQ; ++k) {
#pragma unroll
        for (int e = 0; e < 4; ++e) x[4 * k + e] = 0.0f;
        if (tid + NT * k < nquads) pending |= 1u << k;
    }
    uint64_t t0 = 0;
    uint32_t rounds = 0;
    while (pending) {
        uint64_t w[NQ][4];
#pragma unroll
        for (int k = 0; k < NQ; ++k)
            if ((pending >> k) & 1u) {
                const uint64_t* a = addr(tid + NT * k);
                ld_tagged_x2(a, w[k][0], w[k][1]);
                ld_tagged_x2(a + 2, w[k][2], w[k][3]);
            }
#pragma unroll
        for (int k = 0; k < NQ; ++k)
            if (((pending >> k) & 1u) && tag_of(w[k][0]) == tag && tag_of(w[k][1]) == tag && tag_of(w[k][2]) == tag &&
                tag_of(w[k][3]) == tag) {
#pragma unroll
                for (int e = 0; e < 4; ++e) x[4 * k + e] = val_of(w[k][e]);
                pending &= ~(1u << k);
            }
        if (pending && (++rounds & 7u) == 0) {
            const uint64_t now = globaltimer_ns();
            if (t0 == 0) t0 = now;
            else if (waited_long(now - t0) && ld_volatile_int(P.abort_flag)) return false;
            else if (now - t0 > P.wait_limit_ns) {
                record_error(P, kDevTimeout);
                return false;
            }
        }
    }
    return true;
}

// LayerNorm parameters of this thread's pairs (loaded before the input wait).
template <int N, int PP>
__device__ __forceinline__ void load_ln_pairs(const float* g, const float* b, float (&gr)[2 * PP], float (&br)[2 * PP],
                                              int tid) {
    constexpr int NT = kConsumerWarps * 32;
#pragma unroll
    for (int k = 0; k < PP; ++k) {
        const int q = tid + NT * k;
        float2 gv = make_float2(0.0f, 0.0f), bv = make_float2(0.0f, 0.0f);
        if (q < N / 2) {
            gv = __ldg(reinterpret_cast<const float2*>(g) + q);
            bv = __ldg(reinterpret_cast<const float2*>(b) + q);
        }
        gr[2 * k] = gv.x;
        gr[2 * k + 1] = gv.y;
        br[2 * k] = bv.x;
        br[2 * k + 1] = bv.y;
    }
}

// LayerNorm of the pair-held coordinates into y (shared memory): one block
// reduction of (sum x, sum x^2); biased variance E[x^2] - mean^2; eps 1e-5.
template <int N, int PP>
__device__ __forceinline__ void layernorm_pairs(const float (&v)[2 * PP], const float (&g)[2 * PP],
                                                const float (&b)[2 * PP], float* y, float* red, int tid) {
    constexpr int NT = kConsumerWarps * 32;
    float s1 = 0.0f, s2 = 0.0f;
#pragma unroll
    for (int k = 0; k < PP; ++k)
        if (tid + NT * k < N / 2) {
            s1 += v[2 * k] + v[2 * k + 1];
            s2 = fmaf(v[2 * k], v[2 * k], fmaf(v[2 * k + 1], v[2 * k + 1], s2));
        }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        s1 += __shfl_xor_sync(0xffffffffu, s1, o);
        s2 += __shfl_xor_sync(0xffffffffu, s2, o);
    }
    if ((tid & 31) == 0) reinterpret_cast<float2*>(red)[tid >> 5] = make_float2(s1, s2);
    consumers_sync();
    float t1 = 0.0f, t2 = 0.0f;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) {
        const float2 r = reinterpret_cast<const float2*>(red)[w];
        t1 += r.x;
        t2 += r.y;
    }
    constexpr float inv_n = 1.0f / (float)N;
    const float mean = t1 * inv_n;
    const float rstd = rsqrtf(fmaxf(fmaf(t2, inv_n, -mean * mean), 0.0f) + kLnEps);
#pragma unroll
    for (int k = 0; k < PP; ++k) {
        const int q = tid + NT * k;
        if (q < N / 2)
            reinterpret_cast<float2*>(y)[q] = make_float2(fmaf((v[2 * k] - mean) * rstd, g[2 * k], b[2 * k]),
                                                          fmaf((v[2 * k + 1] - mean) * rstd, g[2 * k + 1], b[2 * k + 1]));
    }
}

// Phase kinds of a step, in order: per layer LN1 + QKV, attention,
// out-projection, LN2 + FC, MLP projection; then LN_f + vocabulary.
enum PhaseKind : int { kPhQKV = 0, kPhAtt = 1, kPhO = 2, kPhFC = 3, kPhP = 4, kPhVocab = 5 };

// Profiling stamps per (phase of step 0, CTA): globaltimer at phase start,
// inputs complete, outputs stored; clock64 at inputs complete, projection
// start, warp 0's last row stored, outputs stored, warp 0's first weight
// chunk landed.
constexpr int kStamps = 8;

// The consumer side is one loop over the phases of a step with a runtime
// dispatch on the phase kind, so that every routine (gather, LayerNorm, head
// merge, quantizer, dot products, epilogue, attention) exists once in the
// binary: a layer executes far more code than an SM's instruction cache
// holds when each phase carries inlined copies of its own.
template <int D, int FF, int DH, int WQ>
__global__ void __launch_bounds__(kThreads, 1) step_kernel(const __grid_constant__ StepPlan plan) {
    constexpr bool Q8 = WQ == kWQ8;
    extern __shared__ __align__(128) uint8_t smem[];
    const SmemLayout lay = smem_layout(D, FF, Q8, plan.max_pos);
    // Every field of the plan is read from a shared-memory copy: kernel
    // parameters live in the constant bank, whose cache misses cost an L2
    // round trip in the middle of a phase's critical path.
    {
        const uint32_t* src = reinterpret_cast<const uint32_t*>(&plan);
        uint32_t* dst = reinterpret_cast<uint32_t*>(smem + lay.plan);
        static_assert(sizeof(StepPlan) % 4 == 0, "plan copies as words");
        for (int i = threadIdx.x; i < (int)(sizeof(StepPlan) / 4); i += blockDim.x) dst[i] = src[i];
        __syncthreads();
    }
    const StepPlan& P = *reinterpret_cast<const StepPlan*>(smem + lay.plan);
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
            const Geo g0 = phase_geo(P, m == kVocab ? 4 * L : m, cta, WQ);
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
        };
        for (int i = 0; i < P.prefetch_chunks; ++i) pf_advance();
        // Pacing: the chunks of the block matrices are issued at least pace_ns
        // apart, so that the refills released together at a phase boundary do
        // not saturate HBM while the next phase exchanges its activations
        // (loaded memory raises the latency of every exchange).  The
        // vocabulary streams unpaced.
        uint64_t next_issue = 0;
        for (int s = 0; s < P.n_steps && !stop; ++s) {
            for (int ph = 0; ph < phases_per_step && !stop; ++ph) {
                const Geo g = geo_of(P, geot, ph);
                const bool paced = P.pace_ns != 0 && ph != phases_per_step - 1;
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
                    if (paced) {
                        uint64_t now = globaltimer_ns();
                        while (now < next_issue && !*s_abort) {
                            __nanosleep(64);
                            now = globaltimer_ns();
                        }
                        next_issue = (now > next_issue ? now : next_issue) + P.pace_ns;
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
        return;
    }

    // ================================================= consumer warps
    constexpr int NT = kConsumerWarps * 32;
    constexpr int PPD = Pairs<D>::PP;          // word pairs per thread of a D-vector
    constexpr int PPS = Pairs<kMaxSplits * D>::PP;  // ... of every key split's head outputs
    constexpr int PPQ = Pairs<3 * D>::PP;      // ... of the qkv vector (trace)
    constexpr int PPF = Pairs<FF>::PP;         // word pairs per thread of an FF-vector
    static_assert(PPF <= 32 && PPS <= 32 && D % 2 == 0 && FF % 2 == 0 && DH % 2 == 0, "pair gathers");
    uint32_t gi = 0;  // chunks consumed (same sequence as the producer)
    using KD = std::integral_constant<int, D>;
    using KF = std::integral_constant<int, FF>;
    static_assert(kSlots / 2 <= 32, "a spread share's chunks are released by one warp's lanes");
    const int S = attn_splits(P.G, P.H);  // splits the scratch holds per head
    const int nph = 5 * L + 1;
    const unsigned per_step = (unsigned)nph;
    const bool tracer = (P.trace != nullptr) && cta == 0;
    const int trace_layer = 8 * D + FF;
    uint64_t* stp = nullptr;  // this phase's stamps (thread 0, step 0, when profiling)
    auto gstamp = [&](int k) { if (stp) stp[k] = globaltimer_ns(); };
    auto cstamp = [&](int k) { if (stp) stp[k] = (uint64_t)clock64(); };
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

    // Lane i < n of a warp waits (bounded) until ring chunk c0 + i has
    // landed.  The caller's next CTA barrier orders the observed copies
    // before every consumer thread's reads.  Warp-uniform result.
    auto wait_chunks = [&](uint32_t c0, int n) -> bool {
        const uint32_t cc = c0 + (uint32_t)lane;
        uint64_t t0 = 0;
        uint32_t spins = 0;
        while (!__all_sync(0xffffffffu, lane >= n || mbar_try_wait(&full[cc % kSlots], (cc / kSlots) & 1))) {
            if ((++spins & 255) == 0) {
                int give_up = 0;
                const uint64_t now = globaltimer_ns();
                if (t0 == 0) t0 = now;
                else if (waited_long(now - t0) && ld_volatile_int(P.abort_flag)) give_up = 1;
                if (t0 != now && now - t0 > P.wait_limit_ns) {
                    if (lane == 0) record_error(P, kDevTimeout);
                    give_up = 1;
                }
                if (__shfl_sync(0xffffffffu, give_up, 0)) return false;
            }
        }
        return true;
    };

    ArgBest best = arg_init();
    // One streamed projection phase over this CTA's share of rows (input
    // width KK; the vocabulary, or a block matrix whose share is too long to
    // be spread), one warp per chunk, with the epilogue of each output row j
    // run by the lane that holds it: QKV: + bias, tagged store, KV append; O
    // and P: + bias + residual; FC: + bias, GELU; vocabulary: logits and the
    // running greedy choice.  Chunks are released by the warp that used
    // them, with a named barrier per round of chunks so warp skew stays below
    // one ring length (*release stays 0).
    auto run_gemv = [&](auto kk, int kind, const Geo& g, unsigned tag, uint64_t boff, float* kv_row, float* lg,
                        int* release) -> bool {
        constexpr int KK = decltype(kk)::value;
        using R = Rows<KK, WQ>;
        auto epilogue = [&](int j, float y) {
            if (kind == kPhVocab) {
                if (lg) lg[j] = y;
                arg_update(best, y, (unsigned)j);
                return;
            }
            const float b = g.nrows <= NT ? bias_s[j - g.r0] : __ldg(P.packed + boff + j);
            const float v = __fadd_rn(y, b);
            if (kind == kPhQKV) {
                st_tagged(P.qkv + j, tag, v);
                if (j >= D) kv_row[j - D] = v;
            } else if (kind == kPhFC) {
                st_tagged(P.u + j, tag, gelu_tanh(v));
            } else {
                st_tagged((kind == kPhO ? P.xb : P.xa) + j, tag, __fadd_rn(xs[j], v));
            }
        };
        *release = 0;
        bool ok = true;
        constexpr int MR = dot_rows<KK, Q8>();
        static_assert(2 * kConsumerWarps <= kSlots, "a round must stay within one ring length");
        for (int k0 = 0; k0 < g.nchunks; k0 += kConsumerWarps) {
            const int k = k0 + warp;
            if (ok && k < g.nchunks) {
                const uint32_t c = gi + (uint32_t)k;
                ok = wait_chunks(c, 1);
                __syncwarp();
                if (k0 == 0) cstamp(7);
                if (ok) {
                    const uint8_t* w = ring + (size_t)(c % kSlots) * kSlotBytes;
                    const int n = min(R::RPC, g.nrows - k * R::RPC);
                    for (int q = 0; q < n; q += MR) {
                        const int m = min(MR, n - q);
                        float y;
                        if constexpr (Q8)
                            y = dot_q8<KK>(w + (size_t)q * R::RB, m, vq, vs, rsc + warp * kWarpScratch, lane);
                        else
                            y = dot_f32<KK, WQ>(w + (size_t)q * R::RB, m, vin, lane);
                        if (lane < m) epilogue(g.r0 + k * R::RPC + q + lane, y);
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&empty[c % kSlots]);
                }
            }
            if (k0 + kConsumerWarps < g.nchunks) consumers_sync();
        }
        cstamp(5);
        gi += g.nchunks;
        return ok;
    };

    // One binary32 fast phase (LN1 + QKV, single-split out-projection,
    // LN2 + FC, MLP projection) over a spread share: the input is gathered
    // in the quad layout straight into the registers that the dot products
    // use; LayerNorm is folded into the projection (row constants c, d) and
    // its mean and variance are reduced alongside the dot products; one
    // barrier per phase, after which the share's ring slots are released and
    // thread r runs row r's epilogue.
    float* fpart = reinterpret_cast<float*>(smem + lay.fpart);
    int fast_no = 0;
    // int8 models trace step 0 from the fast path itself, in every CTA: the
    // vectors the fast path quantizes (CTA 0; every CTA forms the same ones)
    // and each CTA's own QKV rows.  (binary32 / binary16 traced steps take
    // the general path in CTA 0.)
    bool q8_trace_now = false;
    // With from_vin the input is the vector already formed in vin (the
    // LayerNorm output or merged attention heads of the general path) and
    // the epilogue adds the plain bias.
    auto fast_phase = [&](auto kk, int kind, int l, int p, unsigned tok, const Geo& g, unsigned tag,
                          bool from_vin) -> bool {
        constexpr int KK = decltype(kk)::value;
        using Q = Pre<KK>;
        constexpr bool kLnWidth = KK == D;  // LayerNorm phases project D-vectors
        const bool has_ln = kLnWidth && !from_vin && (kind == kPhQKV || kind == kPhFC);
        const LayerParams& lp = P.lp[l];
        const bool row = tid < g.nrows;
        const int j = g.r0 + tid;
        // row constants: the LayerNorm folds (binary32), or the bias
        float cj = 0.0f, dj = 0.0f;
        if (row) {
            if (!Q8 && has_ln) {
                const int N = kind == kPhQKV ? 3 * D : FF;
                const float* f = P.fold + (uint64_t)l * fold_layer_words(D, FF) + (kind == kPhQKV ? 0 : 6 * D);
                cj = __ldg(f + j);
                dj = __ldg(f + N + j);
            } else {
                const uint64_t bo = kind == kPhQKV ? lp.b_qkv : kind == kPhO ? lp.b_o : kind == kPhFC ? lp.b_fc : lp.b_p;
                dj = __ldg(P.packed + bo + j);
            }
        }
        float gq[4 * Q::NC], bq[4 * Q::NC];
        if constexpr (kLnWidth) {
            if (has_ln) {
                load_quads<KK>(P.packed + (kind == kPhQKV ? lp.ln1_g : lp.ln2_g), gq, tid);
                if constexpr (Q8) load_quads<KK>(P.packed + (kind == kPhQKV ? lp.ln1_b : lp.ln2_b), bq, tid);
            }
        }
        // the share's chunks were issued phases ago
        bool ok = wait_chunks(gi, g.nchunks);
        __syncwarp();
        cstamp(7);
        // inputs
        float x[4 * Q::NC];
        if (from_vin) {
            load_quads<KK>(vin, x, tid);
        } else if (kind == kPhQKV && l == 0) {
            // token + position embedding (int8 models: the tied embedding's
            // int8 row times its group scale; binary16 models: its binary16 row)
            const float4* te = reinterpret_cast<const float4*>(P.packed + P.wte_off + (uint64_t)tok * D);
            const float4* pe = reinterpret_cast<const float4*>(P.packed + P.wpe_off + (uint64_t)p * D);
#pragma unroll
            for (int cc = 0; cc < Q::NC; ++cc) {
                const int col = tid + Q::NT * cc;
                float4 a = make_float4(0.0f, 0.0f, 0.0f, 0.0f), b = a;
                if (col < Q::NV) {
                    if constexpr (Q8) {
                        const uint8_t* row = P.vocab + (uint64_t)tok * row_bytes(D, kWQ8);
                        const char4 qv = reinterpret_cast<const char4*>(row)[col];
                        const float sv = reinterpret_cast<const float*>(row + D)[(4 * col) / kGroup];
                        a = make_float4(__fmul_rn((float)qv.x, sv), __fmul_rn((float)qv.y, sv),
                                        __fmul_rn((float)qv.z, sv), __fmul_rn((float)qv.w, sv));
                    } else if constexpr (WQ == kWF16) {
                        a = weight4<kWF16>(P.vocab + (uint64_t)tok * row_bytes(D, kWF16), col);
                    } else {
                        a = __ldg(te + col);
                    }
                    b = __ldg(pe + col);
                }
                x[4 * cc] = __fadd_rn(a.x, b.x);
                x[4 * cc + 1] = __fadd_rn(a.y, b.y);
                x[4 * cc + 2] = __fadd_rn(a.z, b.z);
                x[4 * cc + 3] = __fadd_rn(a.w, b.w);
            }
        } else if (kind == kPhO) {
            ok = ok & gather_quads<Q::NC>(
                          x, Q::NV, tag - 1u,
                          [&](int c) {
                              const int idx = 4 * c, h = idx / DH;
                              return P.attn_part + (size_t)h * (DH + 2) + 2 + (idx - h * DH);
                          },
                          tid, P);
        } else {
            const uint64_t* src = kind == kPhQKV ? P.xa : kind == kPhFC ? P.xb : P.u;
            ok = ok & gather_quads<Q::NC>(x, Q::NV, tag - 1u, [&](int c) { return src + 4 * (size_t)c; }, tid, P);
        }
        gstamp(1);
        cstamp(3);
        float* part = fpart + (fast_no & 1) * kFastSet;
        float2* lns = reinterpret_cast<float2*>(part + kConsumerWarps * kSpreadRows);
        ++fast_no;
        float s1 = 0.0f, s2 = 0.0f;
        if (kLnWidth && has_ln) {
            // the residual stream for the later residual add and the
            // LayerNorm sums; binary32 then takes g * x for the folded
            // projection
#pragma unroll
            for (int cc = 0; cc < Q::NC; ++cc) {
                const int col = tid + Q::NT * cc;
                if (col < Q::NV) {
                    reinterpret_cast<float4*>(xs)[col] = make_float4(x[4 * cc], x[4 * cc + 1], x[4 * cc + 2], x[4 * cc + 3]);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        s1 += x[4 * cc + e];
                        s2 = fmaf(x[4 * cc + e], x[4 * cc + e], s2);
                        if constexpr (!Q8) x[4 * cc + e] *= gq[4 * cc + e];
                    }
                }
            }
        }
        cstamp(4);
        if constexpr (!Q8) coop_reg<KK, WQ>(ring, gi, g.nrows, x, part, tid);
        if (kLnWidth && has_ln) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                s1 += __shfl_xor_sync(0xffffffffu, s1, o);
                s2 += __shfl_xor_sync(0xffffffffu, s2, o);
            }
            if (lane == 0) lns[warp] = make_float2(s1, s2);
        }
        cstamp(5);
        volatile int* slot = s_fail + (agree_no & 1);
        ++agree_no;
        if (!ok) *slot = 1;
        // (an int8 phase without LayerNorm agrees at its quantization barrier)
        if (!Q8 || (kLnWidth && has_ln)) {
            consumers_sync();
            if (*slot != 0) return false;
        }
        // the mean and inverse deviation of the LayerNorm input
        auto ln_stats = [&](float& mean, float& rstd) {
            float t1 = 0.0f, t2 = 0.0f;
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) {
                const float2 r = lns[w];
                t1 += r.x;
                t2 += r.y;
            }
            constexpr float inv_n = 1.0f / (float)D;
            mean = t1 * inv_n;
            rstd = rsqrtf(fmaxf(fmaf(t2, inv_n, -mean * mean), 0.0f) + kLnEps);
        };
        float y = 0.0f;
        if constexpr (Q8) {
            // int8: LayerNorm in registers, then the quantized input to
            // shared memory for the (row, group) dot-product tasks
            if (kLnWidth && has_ln) {
                float mean, rstd;
                ln_stats(mean, rstd);
#pragma unroll
                for (int e = 0; e < 4 * Q::NC; ++e) x[e] = fmaf((x[e] - mean) * rstd, gq[e], bq[e]);
            }
            if (q8_trace_now && cta == 0) {
                // trace offsets per layer: x 0, LN1 D, attention output 5D, x_mid 6D, LN2 7D, GELU output 8D
                const size_t tb = (size_t)l * (8 * D + FF);
                const int oin = kind == kPhQKV ? D : kind == kPhO ? 5 * D : kind == kPhFC ? 7 * D : 8 * D;
#pragma unroll
                for (int cc = 0; cc < Q::NC; ++cc) {
                    const int col = tid + Q::NT * cc;
                    if (col < Q::NV)
#pragma unroll
                        for (int e = 0; e < 4; ++e) P.trace[tb + oin + 4 * col + e] = x[4 * cc + e];
                }
                if (kLnWidth && has_ln)
                    for (int i = tid; i < D; i += NT) P.trace[tb + (kind == kPhQKV ? 0 : 6 * D) + i] = xs[i];
            }
            quantize_quads<KK>(x, vq, vs, tid, P.act_row != 0, red);
            consumers_sync();
            if (!(kLnWidth && has_ln) && *slot != 0) return false;
            y = coop_q8<KK>(ring, gi, g.nrows, vq, vs, rsc, tid);
        } else {
            if (row) {
                y = sum_warp_parts(part, tid);
                if (kLnWidth && has_ln) {
                    float mean, rstd;
                    ln_stats(mean, rstd);
                    y = fmaf(rstd, fmaf(-mean, cj, y), dj);
                }
            }
        }
        // every weight read of the share is done
        if (warp == 0 && lane < g.nchunks) mbar_arrive(&empty[(gi + (uint32_t)lane) % kSlots]);
        gi += (uint32_t)g.nchunks;
        if (row) {
            if (Q8 || !(kLnWidth && has_ln)) y = __fadd_rn(y, dj);
            const unsigned tg = out_tag(tag);
            if (kind == kPhQKV) {
                st_tagged(P.qkv + j, tg, y);
                if (j >= D) P.cache[((uint64_t)p * L + l) * 2 * D + (j - D)] = y;
                if (Q8 && q8_trace_now) P.trace[(size_t)l * (8 * D + FF) + 2 * D + j] = y;
            } else if (kind == kPhFC) {
                st_tagged(P.u + j, tg, gelu_tanh(y));
            } else {
                st_tagged((kind == kPhO ? P.xb : P.xa) + j, tg, __fadd_rn(xs[j], y));
            }
        }
        gstamp(2);
        cstamp(6);
        return true;
    };

    // Attention of layer l over positions 0..p, split along the key axis.
    // Unit (head h, split sp) covers keys [k0, k1).  A warp takes KPW keys
    // per pass (LPK lanes per key, DPL dims per lane) and every lane keeps an
    // online softmax (running max, sum, weighted values).  Keys and values of
    // positions < p do not depend on this step, so a warp's first two passes
    // are loaded before waiting for q; position p's key and value come from
    // this step's tagged qkv words.  Each unit stores an unnormalised partial
    // (max, sum, o[DH]) as tagged words.
    auto attention = [&](int l, int p, int S_eff, unsigned tag) -> bool {
        constexpr int LPK = DH >= 32 ? 8 : 4;    // lanes per key
        constexpr int KPW = 32 / LPK;            // keys per warp per pass
        constexpr int DPL = DH / LPK;            // dims per lane
        constexpr int F4 = DPL / 4;              // float4 per lane per row
        constexpr int KPP = kConsumerWarps * KPW;  // keys per pass over the CTA
        static_assert(DPL % 4 == 0, "a lane holds whole float4s of a head row");
        const unsigned tin = tag - 1u, tg = out_tag(tag);
        const int ks = lane / LPK, dc = lane % LPK;
        const int n = p + 1;
        const float den = sqrtf((float)DH);
        const uint64_t kv_stride = (uint64_t)L * 2 * D;  // floats between positions in the cache
        bool first = true;
        for (int u = cta; u < P.H * S_eff; u += P.G) {
            const int h = u / S_eff, sp = u - h * S_eff;
            const int k0 = (int)(((long long)sp * n) / S_eff), k1 = (int)(((long long)(sp + 1) * n) / S_eff);
            const bool has_p = (k1 == n);  // the last split holds this position's key
            const float* kv0 = P.cache + (uint64_t)l * 2 * D + h * DH + dc * DPL;
            auto fetch = [&](int j, float4 (&kk)[F4], float4 (&vv)[F4]) {
                if (j < k1 && j < p) {
                    const float4* row = reinterpret_cast<const float4*>(kv0 + (uint64_t)j * kv_stride);
#pragma unroll
                    for (int f = 0; f < F4; ++f) {
                        kk[f] = __ldcg(row + f);
                        vv[f] = __ldcg(row + D / 4 + f);
                    }
                }
            };
            int j = k0 + warp * KPW + ks;  // this lane's key in the current pass
            float4 ka[F4], va[F4], kb[F4], vb[F4];
            fetch(j, ka, va);
            fetch(j + KPP, kb, vb);
            // q_h (threads 0..DH-1); k_p, v_p (DH..3DH-1) when this unit holds key p
            uint64_t mine = 0;
            const uint64_t* src = nullptr;
            if (tid < DH) src = P.qkv + h * DH + tid;
            else if (has_p && tid < 2 * DH) src = P.qkv + D + h * DH + (tid - DH);
            else if (has_p && tid < 3 * DH) src = P.qkv + 2 * D + h * DH + (tid - 2 * DH);
            if (src) mine = 1;
            uint64_t wq[1];
            const bool got = tagged_wait<1>(wq, mine, tin, [&](int) { return src; }, P);
            if (src) qh[tid] = val_of(wq[0]);
            if (!agree(got)) return false;
            if (first) {
                gstamp(1);
                cstamp(3);
                cstamp(4);
            }
            first = false;
            const float4* q4 = reinterpret_cast<const float4*>(qh + dc * DPL);
            float m = -INFINITY, z = 0.0f;
            float acc[DPL];
#pragma unroll
            for (int d = 0; d < DPL; ++d) acc[d] = 0.0f;
            for (int jb = k0 + warp * KPW; jb < k1; jb += KPP, j += KPP) {
                if (j == p) {
#pragma unroll
                    for (int f = 0; f < F4; ++f) {
                        ka[f] = reinterpret_cast<const float4*>(qh + DH + dc * DPL)[f];
                        va[f] = reinterpret_cast<const float4*>(qh + 2 * DH + dc * DPL)[f];
                    }
                }
                float dot = 0.0f;
#pragma unroll
                for (int f = 0; f < F4; ++f) {
                    const float4 qf = q4[f];
                    dot += qf.x * ka[f].x + qf.y * ka[f].y + qf.z * ka[f].z + qf.w * ka[f].w;
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
                        acc[4 * f + 0] = fmaf(acc[4 * f + 0], corr, e * va[f].x);
                        acc[4 * f + 1] = fmaf(acc[4 * f + 1], corr, e * va[f].y);
                        acc[4 * f + 2] = fmaf(acc[4 * f + 2], corr, e * va[f].z);
                        acc[4 * f + 3] = fmaf(acc[4 * f + 3], corr, e * va[f].w);
                    }
                    m = mn;
                }
#pragma unroll
                for (int f = 0; f < F4; ++f) {
                    ka[f] = kb[f];
                    va[f] = vb[f];
                }
                fetch(j + 2 * KPP, kb, vb);
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
#pragma unroll
                for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, stage[(w * LPK + c) * (2 + DPL)]);
                float Z = 0.0f, O = 0.0f;
#pragma unroll
                for (int w = 0; w < kConsumerWarps; ++w) {
                    const float* st = stage + (w * LPK + c) * (2 + DPL);
                    if (st[0] == -INFINITY) continue;
                    const float cw = expf(st[0] - M);
                    Z = fmaf(st[1], cw, Z);
                    O = fmaf(st[2 + d], cw, O);
                }
                uint64_t* part = P.attn_part + (size_t)u * (DH + 2);
                if (S_eff == 1) {
                    st_tagged(part + 2 + tid, tg, O / Z);  // the head's output, normalised
                } else {
                    st_tagged(part + 2 + tid, tg, O);
                    if (tid == 0) {
                        st_tagged(part, tg, M);
                        st_tagged(part + 1, tg, Z);
                    }
                }
            }
            consumers_sync();
        }
        if (first) {
            gstamp(1);
            cstamp(3);
            cstamp(4);
        }
        cstamp(5);
        return true;
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
                    const uint64_t now = globaltimer_ns();
                    if (t0 == 0) t0 = now;
                    else if (waited_long(now - t0) && ld_volatile_int(P.abort_flag)) { ok = false; break; }
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
        const bool trace_step = tracer && s == 0 && !Q8;
        q8_trace_now = Q8 && P.trace != nullptr && s == 0;
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
        const int S_eff = attn_splits_for(p + 1, S);
        for (int ph = 0; ph < nph; ++ph) {
            const int kind = ph == nph - 1 ? (int)kPhVocab : ph % 5;
            const int l = ph / 5;  // L for the vocabulary phase
            const unsigned tag = base + (unsigned)ph + 1u;  // this phase's outputs; its inputs carry tag - 1
            stp = (P.timing && s == 0 && tid == 0) ? P.timing + ((size_t)ph * P.G + cta) * kStamps : nullptr;
            gstamp(0);
            if (kind == kPhAtt) {
                if (!attention(l, p, S_eff, tag)) { alive = false; break; }
                gstamp(2);
                cstamp(6);
                continue;
            }
            const LayerParams& lp = P.lp[kind == kPhVocab ? 0 : l];
            const int mat = kind == kPhVocab ? 4 * L
                                             : 4 * l + (kind == kPhQKV ? (int)kQKV
                                                        : kind == kPhO ? (int)kO
                                                        : kind == kPhFC ? (int)kFC : (int)kP);
            const int K = kind == kPhP ? FF : D;
            const Geo g = geo_of(P, geot, mat);
            const bool spread = kind != kPhVocab && share_spread(g.nchunks, g.nrows, K, Q8);
            // spread shares take the fast phase, on gathered inputs, except
            // where the general path forms the input vector: the activation
            // trace, and the merge of split attention heads
            const bool fast = spread && !trace_step && (kind != kPhO || S_eff == 1);
            if (!fast) {
            // LayerNorm parameters (QKV: ln_1, FC: ln_2, vocabulary: ln_f) and
            // this CTA's bias rows are loaded before the wait for the inputs.
            const bool has_ln = kind == kPhQKV || kind == kPhFC || kind == kPhVocab;
            float gr[2 * PPD], br[2 * PPD];
            if (has_ln) {
                const uint64_t go = kind == kPhQKV ? lp.ln1_g : kind == kPhFC ? lp.ln2_g : P.lnf_g;
                const uint64_t bo = kind == kPhQKV ? lp.ln1_b : kind == kPhFC ? lp.ln2_b : P.lnf_b;
                load_ln_pairs<D, PPD>(P.packed + go, P.packed + bo, gr, br, tid);
            }
            const uint64_t boff = kind == kPhQKV ? lp.b_qkv : kind == kPhO ? lp.b_o : kind == kPhFC ? lp.b_fc : lp.b_p;
            const float bv = (kind != kPhVocab && g.nrows <= NT && tid < g.nrows) ? __ldg(P.packed + boff + g.r0 + tid)
                                                                                  : 0.0f;
            bool ok = true;
            // ---- inputs
            float xv[2 * PPD];  // LayerNorm phases: this thread's pairs of the residual stream
            if (kind == kPhO && S_eff == 1) {
                // single-split heads: unit h holds head h's normalised output
                float ov2[2 * PPD];
                ok = ok & gather_pairs<PPD>(
                    ov2, D / 2, tag - 1u,
                    [&](int q) {
                        const int idx = 2 * q, h = idx / DH;
                        return P.attn_part + (size_t)h * (DH + 2) + 2 + (idx - h * DH);
                    },
                    tid, P);
#pragma unroll
                for (int k = 0; k < PPD; ++k)
                    if (tid + NT * k < D / 2)
                        reinterpret_cast<float2*>(vin)[tid + NT * k] = make_float2(ov2[2 * k], ov2[2 * k + 1]);
            } else if (kind == kPhO) {
                // Every split's unnormalised outputs, as one vector of
                // S_eff * D words (word sp * D + idx, head h = idx / DH),
                // gathered in pairs into vin; the (max, sum) pair of each of
                // the H * S_eff units into stage[2u], stage[2u + 1].
                float uv[2 * PPS];
                ok = ok & gather_pairs<PPS>(
                              uv, (S_eff * D) / 2, tag - 1u,
                              [&](int q) {
                                  const int v = 2 * q, sp = v / D, idx = v - sp * D, h = idx / DH;
                                  return P.attn_part + (size_t)(h * S_eff + sp) * (DH + 2) + 2 + (idx - h * DH);
                              },
                              tid, P);
#pragma unroll
                for (int k = 0; k < PPS; ++k)
                    if (tid + NT * k < (S_eff * D) / 2)
                        reinterpret_cast<float2*>(vin)[tid + NT * k] = make_float2(uv[2 * k], uv[2 * k + 1]);
                float mz[2];
                ok = ok & gather_pairs<1>(mz, P.H * S_eff, tag - 1u,
                                          [&](int q) { return P.attn_part + (size_t)q * (DH + 2); }, tid, P);
                if (tid < P.H * S_eff) {
                    stage[2 * tid] = mz[0];
                    stage[2 * tid + 1] = mz[1];
                }
            } else if (kind == kPhQKV && l == 0) {
#pragma unroll
                for (int k = 0; k < 2 * PPD; ++k) {
                    const int i = 2 * (tid + NT * (k >> 1)) + (k & 1);
                    xv[k] = 0.0f;
                    if (i < D) {
                        const float pe = __ldg(P.packed + P.wpe_off + (uint64_t)p * D + i);
                        if constexpr (Q8) {
                            const uint8_t* row = P.vocab + (uint64_t)tok * row_bytes(D, kWQ8);
                            const float qv = (float)reinterpret_cast<const int8_t*>(row)[i];
                            const float sv = reinterpret_cast<const float*>(row + D)[i / kGroup];
                            xv[k] = __fadd_rn(__fmul_rn(qv, sv), pe);
                        } else if constexpr (WQ == kWF16) {
                            const __half* row = reinterpret_cast<const __half*>(P.vocab) + (uint64_t)tok * D;
                            xv[k] = __fadd_rn(__half2float(row[i]), pe);
                        } else {
                            xv[k] = __fadd_rn(__ldg(P.packed + P.wte_off + (uint64_t)tok * D + i), pe);
                        }
                    }
                }
            } else if (kind == kPhP) {
                float uv[2 * PPF];
                ok = ok & gather_pairs<PPF>(uv, FF / 2, tag - 1u, [&](int q) { return P.u + 2 * (size_t)q; }, tid, P);
#pragma unroll
                for (int k = 0; k < PPF; ++k)
                    if (tid + NT * k < FF / 2)
                        reinterpret_cast<float2*>(vin)[tid + NT * k] = make_float2(uv[2 * k], uv[2 * k + 1]);
            } else {
                const uint64_t* src = kind == kPhFC ? P.xb : P.xa;
                ok = ok & gather_pairs<PPD>(xv, D / 2, tag - 1u, [&](int q) { return src + 2 * (size_t)q; }, tid, P);
            }
            if (has_ln) {
                // the residual stream, kept for the epilogue's residual add (and the trace)
#pragma unroll
                for (int k = 0; k < PPD; ++k)
                    if (tid + NT * k < D / 2)
                        reinterpret_cast<float2*>(xs)[tid + NT * k] = make_float2(xv[2 * k], xv[2 * k + 1]);
            }
            if (g.nrows <= NT && tid < g.nrows) bias_s[tid] = bv;
            if (!agree(ok)) { alive = false; break; }
            gstamp(1);
            cstamp(3);
            // ---- input transform: LayerNorm, or the merge of the heads' partials
            if (has_ln) {
                layernorm_pairs<D, PPD>(xv, gr, br, vin, red, tid);
            } else if (kind == kPhO && S_eff > 1) {
                // weight of each (head, split): exp(m - M_h) / Z_h, once per CTA
                if (tid < P.H * S_eff) {
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
                // (each element's split words are read and its merged value
                // written by the same thread)
                for (int idx = tid; idx < D; idx += NT) {
                    const int h = idx / DH;
                    float O = 0.0f;
                    for (int sp = 0; sp < S_eff; ++sp) O = fmaf(ored[h * S_eff + sp], vin[sp * D + idx], O);
                    vin[idx] = O;
                }
            }
            consumers_sync();
            if constexpr (Q8) {
                // a streamed share's input (a spread share quantizes in its phase)
                if (!spread) {
                    if (kind == kPhP) quantize_vec<FF>(vin, vq, vs, warp, lane, P.act_row != 0, red);
                    else quantize_vec<D>(vin, vq, vs, warp, lane, P.act_row != 0, red);
                    consumers_sync();
                }
            }
            // ---- activation trace (step 0, CTA 0): per layer x, LN_1(x), qkv,
            // attention output, x_mid, LN_2(x_mid), GELU output; then x_final, LN_f(x_final).
            // int8 models trace here only the vocabulary phase (the layers
            // trace from the fast path).
            if (trace_step || (q8_trace_now && tracer && kind == kPhVocab)) {
                const int tb = l * trace_layer;
                if (kind == kPhO) {
                    float qv[2 * PPQ];
                    const bool okq = gather_pairs<PPQ>(qv, (3 * D) / 2, tag - 2u,
                                                       [&](int q) { return P.qkv + 2 * (size_t)q; }, tid, P);
#pragma unroll
                    for (int k = 0; k < PPQ; ++k)
                        if (tid + NT * k < (3 * D) / 2) {
                            P.trace[tb + 2 * D + 2 * (tid + NT * k)] = qv[2 * k];
                            P.trace[tb + 2 * D + 2 * (tid + NT * k) + 1] = qv[2 * k + 1];
                        }
                    if (!agree(okq)) { alive = false; break; }
                }
                const int ox = kind == kPhFC ? 6 * D : (kind == kPhQKV || kind == kPhVocab) ? 0 : -1;
                const int oy = kind == kPhQKV || kind == kPhVocab ? D : kind == kPhO ? 5 * D : kind == kPhFC ? 7 * D : 8 * D;
                for (int i = tid; i < K; i += NT) {
                    if (ox >= 0) P.trace[tb + ox + i] = xs[i];
                    P.trace[tb + oy + i] = vin[i];
                }
            }
            // ---- projection and epilogue
            if (kind == kPhVocab) best = arg_init();
            float* kv_row = P.cache + ((uint64_t)p * L + l) * 2 * D;
            float* lg = (kind == kPhVocab && P.logits) ? P.logits + (uint64_t)s * P.logits_stride : nullptr;
            int release = 0;
            cstamp(4);
            if (!spread) {
            ok = kind == kPhP ? run_gemv(KF{}, kind, g, out_tag(tag), boff, kv_row, lg, &release)
                              : run_gemv(KD{}, kind, g, out_tag(tag), boff, kv_row, lg, &release);
            if (!agree(ok)) { alive = false; break; }
            if (warp == 0 && lane < release) mbar_arrive(&empty[(gi + (uint32_t)lane) % kSlots]);
            gi += (uint32_t)release;
            gstamp(2);
            cstamp(6);
            if (kind == kPhVocab) {
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
                    const unsigned tg = out_tag(tag);
                    uint64_t* ap = P.arg_part + 2 * (size_t)cta;
                    const unsigned iw = (best.i & 0x7FFFFFFFu) | (best.nf ? 0x80000000u : 0u);
                    st_tagged(ap + 1, tg, __uint_as_float(iw));
                    // release: this CTA's KV rows and choice become visible with it
                    st_tagged_release(ap, tag_pack(tg, best.v));
                }
            }
            continue;
            }  // streamed share
            }  // general path
            // ---- spread share: gathered inputs (fast), or the vector the
            // general path formed in vin
            const bool okf = kind == kPhP ? fast_phase(KF{}, kind, l, p, tok, g, tag, !fast)
                                          : fast_phase(KD{}, kind, l, p, tok, g, tag, !fast);
            if (!okf) { alive = false; break; }
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
// kernel's own routines: the activation quantizer, then the dot products of
// one phase share (a spread share computed by the whole block, or a long
// share streamed one warp per chunk in two rounds), then the epilogue's bias
// add.  Each block copies its share of rows into a ring-shaped shared buffer.
template <int K, int WQ>
struct HookGeo {
    static constexpr bool Q8 = WQ == kWQ8;
    static constexpr int RB = row_bytes(K, WQ);
    static constexpr int RPC0 = kSlotBytes / RB;
    static constexpr int RPC = RPC0 > kMaxChunkRows ? kMaxChunkRows : RPC0;  // rows per chunk
    static constexpr int SPREADR = (kSlots / 2) * RPC < kSpreadRows ? (kSlots / 2) * RPC : kSpreadRows;
    // rows longer than the CTA are spread at most 8 to a share
    static constexpr int SPREAD0 = (!Q8 && K / 4 > kConsumerWarps * 32 && SPREADR > 8) ? 8 : SPREADR;
    static constexpr int SPREAD1 = Q8 ? kCoopTaskFloats / (K / kGroup) : SPREAD0;
    static constexpr int ROWS_SPREAD = SPREAD0 < SPREAD1 ? SPREAD0 : SPREAD1;  // the largest spread share
    static constexpr int CHUNKS_STREAM = 2 * kConsumerWarps;                    // two rounds of chunks
    static constexpr int SLOTS = CHUNKS_STREAM > kSlots / 2 ? CHUNKS_STREAM : kSlots / 2;
    static constexpr uint32_t SMEM = (uint32_t)SLOTS * kSlotBytes + align16(K * 4) + align16(K) +
                                     align16((K / kGroup) * 4) + (uint32_t)kCoopTaskFloats * 4;
    static_assert(share_spread((ROWS_SPREAD + RPC - 1) / RPC, ROWS_SPREAD, K, Q8), "hook spread share is spread");
    static_assert(!share_spread(CHUNKS_STREAM, CHUNKS_STREAM * RPC, K, Q8), "hook streamed share streams");
};

template <int K, int WQ>
__global__ void __launch_bounds__(kConsumerWarps * 32) project_kernel(const uint8_t* __restrict__ rows, int N,
                                                                      const float* __restrict__ x,
                                                                      const float* __restrict__ bias,
                                                                      float* __restrict__ y, int stream,
                                                                      int act_row) {
    using H = HookGeo<K, WQ>;
    constexpr bool Q8 = H::Q8;
    extern __shared__ __align__(128) uint8_t sm[];
    uint8_t* ring = sm;
    float* vin = reinterpret_cast<float*>(sm + H::SLOTS * kSlotBytes);
    int8_t* vq = reinterpret_cast<int8_t*>(reinterpret_cast<uint8_t*>(vin) + align16(K * 4));
    float* vs = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(vq) + align16(K));
    float* scratch = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(vs) + align16((K / kGroup) * 4));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int per_block = stream ? H::CHUNKS_STREAM * H::RPC : H::ROWS_SPREAD;
    const int w0 = blockIdx.x * per_block;
    const int wn = min(per_block, N - w0);
    // rows w0 .. w0+wn-1 into slots: row r at slot r / RPC, offset (r % RPC) * RB
    for (int i = tid; i < wn * (H::RB / 16); i += blockDim.x) {
        const int r = i / (H::RB / 16), q = i - r * (H::RB / 16);
        const int4 v = reinterpret_cast<const int4*>(rows + (size_t)(w0 + r) * H::RB)[q];
        reinterpret_cast<int4*>(ring + (size_t)(r / H::RPC) * kSlotBytes + (size_t)(r % H::RPC) * H::RB)[q] = v;
    }
    for (int i = tid; i < K; i += blockDim.x) vin[i] = x[i];
    __syncthreads();
    if constexpr (Q8) quantize_vec<K>(vin, vq, vs, warp, lane, act_row != 0, scratch);
    __syncthreads();
    auto out = [&](int j, float v) { y[j] = bias ? __fadd_rn(v, bias[j]) : v; };
    if (!stream) {
        float v;
        if constexpr (Q8) {
            v = coop_q8<K>(ring, 0u, wn, vq, vs, scratch, tid);
        } else {
            float xq[4 * Pre<K>::NC];
            load_quads<K>(vin, xq, tid);
            coop_reg<K, WQ>(ring, 0u, wn, xq, scratch, tid);
            __syncthreads();
            v = tid < wn ? sum_warp_parts(scratch, tid) : 0.0f;
        }
        if (tid < wn) out(w0 + tid, v);
        return;
    }
    const int nchunks = (wn + H::RPC - 1) / H::RPC;
    constexpr int MR = dot_rows<K, Q8>();
    for (int k = warp; k < nchunks; k += kConsumerWarps) {
        const uint8_t* w = ring + (size_t)k * kSlotBytes;
        const int n = min(H::RPC, wn - k * H::RPC);
        for (int q = 0; q < n; q += MR) {
            const int m = min(MR, n - q);
            float v;
            if constexpr (Q8) v = dot_q8<K>(w + (size_t)q * H::RB, m, vq, vs, scratch + warp * kWarpScratch, lane);
            else v = dot_f32<K, WQ>(w + (size_t)q * H::RB, m, vin, lane);
            if (lane < m) out(w0 + k * H::RPC + q + lane, v);
        }
    }
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

template <int K, int WQ>
static cudaError_t project_t(const uint8_t* rows, int N, const float* x, const float* bias, float* y, int stream,
                             int act_row, cudaStream_t st) {
    using H = HookGeo<K, WQ>;
    const int per_block = stream ? H::CHUNKS_STREAM * H::RPC : H::ROWS_SPREAD;
    cudaError_t e = cudaFuncSetAttribute(project_kernel<K, WQ>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)H::SMEM);
    if (e != cudaSuccess) return e;
    project_kernel<K, WQ><<<(N + per_block - 1) / per_block, kConsumerWarps * 32, H::SMEM, st>>>(rows, N, x, bias, y,
                                                                                               stream, act_row);
    return cudaGetLastError();
}

cudaError_t launch_project(const uint8_t* rows, int K, int N, int wq, const float* x, const float* bias, float* y,
                           int stream, int act_row, cudaStream_t st) {
#define GPT2_PROJ(KK)                                                                                        \
    if (K == KK)                                                                                             \
        return wq == kWQ8    ? project_t<KK, kWQ8>(rows, N, x, bias, y, stream, act_row, st)                 \
               : wq == kWF16 ? project_t<KK, kWF16>(rows, N, x, bias, y, stream, act_row, st)                \
                             : project_t<KK, kWF32>(rows, N, x, bias, y, stream, act_row, st);
    GPT2_PROJ(64) GPT2_PROJ(192) GPT2_PROJ(256) GPT2_PROJ(384) GPT2_PROJ(768) GPT2_PROJ(3072)
#undef GPT2_PROJ
    return cudaErrorInvalidValue;
}

cudaError_t launch_argmax(const float* v, unsigned n, uint32_t* idx, int* nonfinite, cudaStream_t st) {
    argmax_kernel<<<1, kConsumerWarps * 32, 0, st>>>(v, n, idx, nonfinite);
    return cudaGetLastError();
}

// ------------------------------------------------------------ launcher
template <int D, int FF, int DH, int WQ>
static cudaError_t launch_t(const StepPlan& P, cudaStream_t stream) {
    constexpr bool Q8 = WQ == kWQ8;
    // binary32 and binary16 fast phases read the LayerNorm folds of every layer
    if (!Q8 && P.fold == nullptr) return cudaErrorInvalidValue;
    const SmemLayout lay = smem_layout(D, FF, Q8, P.max_pos);
    auto kern = step_kernel<D, FF, DH, WQ>;
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

template <int D, int FF, int DH, int WQ>
static int max_ctas_t(int max_pos) {
    const SmemLayout lay = smem_layout(D, FF, WQ == kWQ8, max_pos);
    auto kern = step_kernel<D, FF, DH, WQ>;
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

#define GPT2_DISPATCH_WQ(FN, d, ff, dh, ...)                     \
    return wq == kWQ8 ? FN<d, ff, dh, kWQ8>(__VA_ARGS__)         \
           : wq == kWF16 ? FN<d, ff, dh, kWF16>(__VA_ARGS__)     \
                         : FN<d, ff, dh, kWF32>(__VA_ARGS__);
#define GPT2_DISPATCH(FN, ...)                                                       \
    if (D == 768 && FF == 3072 && DH == 64) GPT2_DISPATCH_WQ(FN, 768, 3072, 64, __VA_ARGS__) \
    if (D == 192 && FF == 384 && DH == 64) GPT2_DISPATCH_WQ(FN, 192, 384, 64, __VA_ARGS__)   \
    if (D == 64 && FF == 256 && DH == 16) GPT2_DISPATCH_WQ(FN, 64, 256, 16, __VA_ARGS__)

cudaError_t launch_step(const StepPlan& P, int wq, cudaStream_t stream) {
    const int D = P.D, FF = P.FF, DH = P.D / P.H;
    GPT2_DISPATCH(launch_t, P, stream)
    return cudaErrorInvalidValue;
}

int step_max_ctas(int D, int FF, int DH, int wq, int max_pos) {
    GPT2_DISPATCH(max_ctas_t, max_pos)
    return 0;
}

}  // namespace gpt2
