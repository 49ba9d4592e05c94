// cstep.cu -- the cluster step kernel: one cooperative launch of NC thread-
// block clusters of CS CTAs runs a run of cached GPT-2 steps (LeanExe GPT-2
// README, cachedStep paragraph; model paragraph for the block order).
//
// Work split (cstep.cuh has the geometry): rank r of each cluster owns the
// column slice [r*SW, (r+1)*SW) of the model width.  Every projection is
// split along its INPUT dimension by slice inside a cluster, and the slices'
// partial dot products are completed by one all-gather over distributed
// shared memory (st.async with mbarrier transaction counts).  The heads and
// FC rows are split across clusters; the out-projection and the MLP
// projection are split-K partials per head / per cluster, summed by their
// consumers in a fixed order.  Hence per layer:
//   A  [clusters with a head]  slice of x formed from the MLP partials ->
//      LN1-folded QKV partials over the slice -> all-gather (q, k, v) ->
//      attention over this CTA's keys -> all-gather (max, sum, weighted
//      values) -> merged head output -> this CTA's SW rows of the head's
//      out-projection partial -> tagged words.
//   B  [every cluster]  slice of x formed from the heads' partials ->
//      LN2-folded FC partials over the slice -> all-gather -> GELU of the
//      cluster's FC rows -> this CTA's SW rows of the MLP partial over those
//      FC rows -> tagged words.
// The vocabulary rows are split across all CTAs; the greedy choice is
// reduced at the start of the next step (one release/acquire per step, which
// also orders the KV-cache stores before the next step's attention).
//
// LayerNorm is folded into the projection that follows it,
//   y_j = rstd * (sum_i W_ji g_i (x_i - s) - (mean - s) c_j) + d_j,
// with c_j = sum_i W_ji g_i and d_j = bias_j + sum_i W_ji b_i made at load
// time.  The shift s is a mean every CTA already holds (the embedding's exact
// mean, then the previous LayerNorm's mean), so the dot products never
// carry the residual's common offset; the variance comes from each slice's
// two-pass sums of squares around its own mean, merged pairwise (Chan et
// al.'s update), so no E[x^2] - mean^2 cancellation occurs.
//
// One producer warp per CTA streams the CTA's parts of every weight matrix,
// in step order, through a shared-memory ring (cp.async.bulk, mbarriers).
// Every wait is bounded by a wall-clock limit; a CTA that gives up records
// GPT2_ERR_TIMEOUT, raises the grid's abort word and leaves its loops, and
// all CTAs of a cluster meet at a final cluster barrier so that no CTA exits
// while a peer may still write into its shared memory.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <vector>

#include "cstep.cuh"

namespace gpt2 {

namespace {

// ---------------------------------------------------------------- PTX
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t mapa(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

// 16 bytes into a peer's shared memory, completing on the peer's mbarrier.
__device__ __forceinline__ void st_async4(uint32_t raddr, float4 v, uint32_t rbar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
                     raddr),
                 "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "r"(rbar)
                 : "memory");
}

// 4 bytes into a peer's shared memory, completing on the peer's mbarrier.
__device__ __forceinline__ void st_async1(uint32_t raddr, float v, uint32_t rbar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.f32 [%0], %1, [%2];" ::"r"(raddr), "f"(v),
                 "r"(rbar)
                 : "memory");
}

// Orders this thread's earlier shared-memory writes before later bulk
// (async-proxy) copies that read them.
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Bulk copy of `bytes` (multiple of 16) from this CTA's shared memory to a
// peer's (cluster address), completing on the peer's mbarrier.
__device__ __forceinline__ void bulk_to_peer(uint32_t dst, uint32_t src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "r"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

__device__ __forceinline__ void cluster_barrier() {
    asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

// Named barrier over the consumer warps only.
__device__ __forceinline__ void csync() { asm volatile("bar.sync 1, %0;" ::"n"(kCWarps * 32) : "memory"); }

// ---------------------------------------------------------------- math
__device__ __forceinline__ float cgelu(float x) {
    const float inner = 0.7978845608f * (x + 0.044715f * x * x * x);
    return 0.5f * x * (1.0f + tanhf(inner));
}

template <int N>
__device__ __forceinline__ float transpose_sum(float (&v)[N], int lane) {
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

template <int WF>
__device__ __forceinline__ float4 w4(const uint8_t* row, int col) {
    if constexpr (WF == kWF16) {
        const uint2 h = *reinterpret_cast<const uint2*>(row + 8u * (uint32_t)col);
        const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&h.x));
        const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&h.y));
        return make_float4(a.x, a.y, b.x, b.y);
    } else {
        return *reinterpret_cast<const float4*>(row + 16u * (uint32_t)col);
    }
}

__device__ __forceinline__ float4 lds4(uint32_t a) {
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(a));
    return v;
}

// Four consecutive weights at shared address a, as binary32.
template <int WF>
__device__ __forceinline__ float4 ldsw(uint32_t a) {
    if constexpr (WF == kWF16) {
        uint32_t lo, hi;
        asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(lo), "=r"(hi) : "r"(a));
        const float2 p = __half22float2(*reinterpret_cast<const __half2*>(&lo));
        const float2 q = __half22float2(*reinterpret_cast<const __half2*>(&hi));
        return make_float4(p.x, p.y, q.x, q.y);
    } else {
        return lds4(a);
    }
}

__device__ __forceinline__ float dot4(float a, float4 w, float4 x) {
    a = fmaf(x.x, w.x, a);
    a = fmaf(x.y, w.y, a);
    a = fmaf(x.z, w.z, a);
    return fmaf(x.w, w.w, a);
}

// Bytes of one 4-weight unit of the cluster stream.
template <int WF>
__host__ __device__ constexpr uint32_t unit_bytes() { return WF == kWF16 ? 8u : 16u; }

// One ring chunk of R <= 32 rows of the cluster stream, stored interleaved
// by 4-weight units (unit c of row i at (c * R + i) * unit bytes), against x
// (W4 float4s at shared address x): lane i < R returns row i's dot product.
// A lane walks its own row, so no reduction across lanes is needed; the
// lanes of a warp read consecutive units (no bank conflicts) and the input
// unit is a broadcast.
template <int WF>
__device__ __forceinline__ float chunk_rows(uint32_t w, int R, int W4, uint32_t x, int lane) {
    constexpr uint32_t UB = unit_bytes<WF>();
    float a[8] = {0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
    if (lane < R) {
        const uint32_t step = (uint32_t)R * UB;
        uint32_t wa = w + (uint32_t)lane * UB, xa = x;
        int c = 0;
        for (; c + 8 <= W4; c += 8, wa += 8 * step, xa += 128) {
            // all sixteen loads of eight units in flight before the first multiply-add
            float4 wv[8], xv[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) wv[u] = ldsw<WF>(wa + u * step);
#pragma unroll
            for (int u = 0; u < 8; ++u) xv[u] = lds4(xa + 16u * u);
#pragma unroll
            for (int u = 0; u < 8; ++u) a[u] = dot4(a[u], wv[u], xv[u]);
        }
        for (; c < W4; ++c, wa += step, xa += 16) a[0] = dot4(a[0], ldsw<WF>(wa), lds4(xa));
    }
    return ((a[0] + a[1]) + (a[2] + a[3])) + ((a[4] + a[5]) + (a[6] + a[7]));
}

// NR consecutive K-major rows (pitch pb bytes, W4 float4 columns each) in
// shared memory against x (W4 float4s): lanes stride the columns, then one
// transpose-reduction (over NR rounded up to a power of two, the extra rows
// zero); lane i < n returns row i's total.  For the long vocabulary rows.
template <int NR, int W4, int WF>
__device__ __forceinline__ float long_rows(uint32_t w, uint32_t pb, int n, uint32_t x, int lane) {
    constexpr uint32_t UB = unit_bytes<WF>();
    constexpr int NP = NR <= 1 ? 1 : NR <= 2 ? 2 : NR <= 4 ? 4 : NR <= 8 ? 8 : NR <= 16 ? 16 : 32;
    float acc[NP];
#pragma unroll
    for (int i = 0; i < NP; ++i) acc[i] = 0.0f;
#pragma unroll
    for (int t = 0; t < (W4 + 31) / 32; ++t) {
        const int cc = lane + 32 * t;
        if ((W4 % 32) == 0 || cc < W4) {
            const float4 xv = lds4(x + 16u * (uint32_t)cc);
#pragma unroll
            for (int i = 0; i < NR; ++i)
                if (i < n) acc[i] = dot4(acc[i], ldsw<WF>(w + (uint32_t)i * pb + UB * (uint32_t)cc), xv);
        }
    }
    return transpose_sum<NP>(acc, lane);
}

__device__ __forceinline__ void crecord_error(const StepPlan& P, int code) {
    atomicCAS(P.status, 0, code);
    atomicExch(P.abort_flag, 1);
}

// Greedy choice order: larger value first, then lower index.
struct Best {
    float v;
    unsigned i;
    int nf;
};
__device__ __forceinline__ bool better(float v, unsigned i, float bv, unsigned bi) {
    return v > bv || (v == bv && i < bi);
}
__device__ __forceinline__ void best_update(Best& b, float v, unsigned j) {
    if (!isfinite(v)) b.nf = 1;
    else if (better(v, j, b.v, b.i)) { b.v = v; b.i = j; }
}
__device__ __forceinline__ void best_merge(Best& b, float v, unsigned i, int nf) {
    b.nf |= nf;
    if (better(v, i, b.v, b.i)) { b.v = v; b.i = i; }
}
__device__ __forceinline__ void best_warp(Best& b) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, b.v, o);
        const unsigned oi = __shfl_xor_sync(0xffffffffu, b.i, o);
        const int onf = __shfl_xor_sync(0xffffffffu, b.nf, o);
        best_merge(b, ov, oi, onf);
    }
}

// Cold path of a bounded wait that gave up: records the timeout and, when
// the run is profiled, which wait, CTA, step and layer (first one only).
__device__ __noinline__ void cwait_gave_up(const StepPlan& P, int kind, int cta, int step, int layer, uint64_t what,
                                          uint64_t seen) {
    if (P.timing && atomicCAS(reinterpret_cast<unsigned long long*>(P.timing), 0ull, (unsigned long long)kind) == 0ull) {
        P.timing[1] = (uint64_t)cta;
        P.timing[2] = (uint64_t)step;
        P.timing[3] = (uint64_t)layer;
        P.timing[4] = what;
        P.timing[5] = seen;
    }
    crecord_error(P, kDevTimeout);
}

// The slow part of every bounded wait, out of line (it runs once per 20 us
// of waiting): after `elapsed` ns, gives up if another CTA raised the abort
// word or the wait limit has passed, noting where in `note` (this CTA's four
// profiling words, when profiling).
__device__ __noinline__ bool cwait_expired(const StepPlan& P, uint64_t elapsed, int kind, int cta, int step, int layer,
                                           uint64_t what, uint64_t seen, uint64_t* note) {
    const bool abort = ld_volatile_int(P.abort_flag) != 0;
    if (!abort && elapsed <= P.wait_limit_ns) return false;
    if (note) {
        note[0] = (uint64_t)kind | (abort ? 0x100ull : 0ull) | ((uint64_t)threadIdx.x << 16);
        note[1] = (uint64_t)step;
        note[2] = (uint64_t)layer;
        note[3] = what;
    }
    if (!abort) cwait_gave_up(P, kind, cta, step, layer, what, seen);
    return true;
}

// Activation trace (step 0 of a traced run): copies, and a LayerNorm output
// (x - mean) * rstd * g + b of a slice; out of line, off the hot path.
__device__ __noinline__ void ctrace_copy(float* dst, const float* src, int n, int tid) {
    for (int i = tid; i < n; i += kCWarps * 32) dst[i] = src[i];
}
__device__ __noinline__ void ctrace_ln(float* dst, const float* xs, float mean, float rstd, const float* g,
                                       const float* b, int n, int tid) {
    for (int i = tid; i < n; i += kCWarps * 32) dst[i] = fmaf((xs[i] - mean) * rstd, __ldg(g + i), __ldg(b + i));
}

// A contiguous run of weight rows that one CTA streams: n rows of pb bytes,
// rpc rows per ring chunk.
struct Share {
    const uint8_t* base;
    uint32_t pb;
    int n, rpc, nch;
};
__device__ __forceinline__ Share make_share(const uint8_t* base, uint32_t pb, int n) {
    Share s;
    s.base = base;
    s.pb = pb;
    s.n = n;
    s.rpc = (int)(kCSlotBytes / pb);
    if (s.rpc > 32) s.rpc = 32;  // a chunk's rows are one warp's lanes
    if (s.rpc > n) s.rpc = n > 0 ? n : 1;
    s.nch = n > 0 ? (n + s.rpc - 1) / s.rpc : 0;
    return s;
}

// Stops checking the grid's abort word until a wait has lasted this long (a
// word polled by every thread of every CTA would be a hot L2 line).
constexpr uint64_t kCAbortCheckNs = 20000;

}  // namespace

// Phases with tagged outputs per step: per layer A (out-projection partials)
// and B (MLP partials); then the greedy partials.
__host__ __device__ inline int cphases_per_step(int L) { return 2 * L + 1; }

template <int D, int FF, int DH, int WF>
__global__ void __launch_bounds__(kCThreads, 1) cstep_kernel(const __grid_constant__ CPlan plan) {
    extern __shared__ __align__(128) uint8_t smem[];
    const CSmem lay = csmem_layout(D, DH, plan.g.CS, plan.g.SW, plan.g.nfc_max, plan.g.slots);
    {
        const uint32_t* src = reinterpret_cast<const uint32_t*>(&plan);
        uint32_t* dst = reinterpret_cast<uint32_t*>(smem + lay.plan);
        static_assert(sizeof(CPlan) % 4 == 0, "plan copies as words");
        for (int i = threadIdx.x; i < (int)(sizeof(CPlan) / 4); i += blockDim.x) dst[i] = src[i];
    }
    __syncthreads();
    const CPlan& CP = *reinterpret_cast<const CPlan*>(smem + lay.plan);
    const StepPlan& P = CP.s;
    const CGeo& GG = CP.g;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int cta = blockIdx.x;
    // the cluster size and slice width are constants of the instantiation
    // (the host builds the geometry with the same function)
    constexpr int CS = cluster_size_for(D), SW = D / CS;
    const int NSL = GG.slots;
    const int r = (int)cluster_rank();
    const int c = cta / CS;
    const int L = P.L, H = P.H;
    const int nh = cg_heads(GG, H, c);
    const int f0 = GG.fc0[c], nfc = GG.fc0[c + 1] - GG.fc0[c];
    const int nfc4 = (nfc + 3) & ~3;
    const int col0 = r * SW;
    // rank r appends rows [kv_lo, kv_hi) of a head's 3 DH q/k/v rows (its
    // keys and values) to the KV cache
    const int kv_per = (2 * DH + CS - 1) / CS;
    const int kv_lo = DH + r * kv_per, kv_hi = min(3 * DH, kv_lo + kv_per);
    constexpr int NT = kCWarps * 32;
    const uint64_t head_bytes = cg_head_bytes(GG, DH);
    const uint32_t wb = (uint32_t)GG.wb;

    uint8_t* ring = smem + lay.ring;
    const uint32_t ring_s = smem_addr(ring);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + lay.full);
    uint64_t* empty = reinterpret_cast<uint64_t*>(smem + lay.empty);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + lay.bars);  // mA[2], mT[2], mB[2], mX
    float* gA = reinterpret_cast<float*>(smem + lay.gA);
    float* gT = reinterpret_cast<float*>(smem + lay.gT);
    float* gB = reinterpret_cast<float*>(smem + lay.gB);
    float* gX = reinterpret_cast<float*>(smem + lay.gX);
    float* qkv = reinterpret_cast<float*>(smem + lay.qkv);
    float* oh = reinterpret_cast<float*>(smem + lay.oh);
    float* uu = reinterpret_cast<float*>(smem + lay.uu);
    float* xs = reinterpret_cast<float*>(smem + lay.xs);
    float* xin = reinterpret_cast<float*>(smem + lay.xin);
    float* xf = reinterpret_cast<float*>(smem + lay.xf);
    float* stage = reinterpret_cast<float*>(smem + lay.stage);
    volatile int* s_abort = reinterpret_cast<volatile int*>(smem + lay.misc);
    volatile int* s_fail = s_abort + 1;  // two slots, alternating per agreement point
    unsigned* s_tok = reinterpret_cast<unsigned*>(smem + lay.misc) + 4;
    volatile int* s_nf = s_abort + 5;
    float* s_red = reinterpret_cast<float*>(smem + lay.misc) + 8;   // [warps] block reductions
    float* s_arg = reinterpret_cast<float*>(smem + lay.misc) + 24;  // [warps][3]
    float* s_stA = reinterpret_cast<float*>(smem + lay.misc) + 48;  // stage A slice (mean, M2)
    CShareRow* shares = reinterpret_cast<CShareRow*>(smem + lay.shares);

    if (tid == 0) {
        for (int i = 0; i < NSL; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        for (int i = 0; i < 7; ++i) mbar_init(&bars[i], 1);
        // Every gather barrier is armed for its first use before any peer can
        // write into this CTA (the cluster barrier below), and re-armed for
        // its next use as soon as a use completes (gather_wait), which is
        // always before a peer can send that next use's data: a barrier is
        // never armed after data for its phase has arrived.
        {
            const int nfc_ = plan.g.fc0[blockIdx.x / plan.g.CS + 1] - plan.g.fc0[blockIdx.x / plan.g.CS];
            for (int i = 0; i < 2; ++i) {
                mbar_arrive_expect_tx(&bars[0 + i], (uint32_t)(plan.g.CS * (3 * DH + 2) * 4));
                mbar_arrive_expect_tx(&bars[2 + i], (uint32_t)(plan.g.CS * (DH + 2) * 4));
                mbar_arrive_expect_tx(&bars[4 + i], (uint32_t)(plan.g.CS * (nfc_ + 2) * 4));
            }
            mbar_arrive_expect_tx(&bars[6], (uint32_t)(D * 4));
        }
        *s_abort = ld_volatile_int(P.abort_flag);
        s_fail[0] = 0;
        s_fail[1] = 0;
        fence_mbar_init();
        // this CTA's shares of a layer: for head slot k its QKV part (2k) and
        // out-projection part (2k + 1); then FC (2 nh) and MLP (2 nh + 1)
        for (int j = 0; j < 2 * nh + 2; ++j) {
            uint64_t off;
            uint32_t pb;
            int n;
            if (j < 2 * nh) {
                const bool wo = (j & 1) != 0;
                off = (uint64_t)(j >> 1) * head_bytes + (wo ? (uint64_t)3 * DH * SW * wb : 0ull);
                pb = (uint32_t)(wo ? DH : SW) * wb;
                n = wo ? SW : 3 * DH;
            } else if (j == 2 * nh) {
                off = (uint64_t)nh * head_bytes;
                pb = (uint32_t)SW * wb;
                n = nfc;
            } else {
                off = (uint64_t)nh * head_bytes + (uint64_t)nfc * SW * wb;
                pb = (uint32_t)nfc * wb;
                n = SW;
            }
            const Share sh = make_share(nullptr, pb, n);
            shares[j] = CShareRow{(uint32_t)off, pb, n, sh.rpc, sh.nch, 0, 0, 0};
        }
    }
    __syncthreads();
    // every CTA's barriers are initialised before any peer writes into them
    cluster_barrier();

    // The share sequence of a step, identical on both sides of the ring:
    // per layer, per head slot k: QKV part, out-projection part; then the
    // FC part and the MLP part; then the vocabulary rows.
    // this CTA's part of layer 0 of the stream; layer l's is layer_bytes further
    const uint8_t* part0 = CP.cstream + GG.seg[c] + (uint64_t)r * GG.cta_bytes[c];
    // Share j of layer l, from the table the prologue built (one routine
    // for every share keeps one copy of it in the binary).
    auto share_at = [&](int l, int j) -> Share {
        const CShareRow t = shares[j];
        Share sh;
        sh.base = part0 + (uint64_t)l * GG.layer_bytes + t.off;
        sh.pb = t.pb;
        sh.n = t.n;
        sh.rpc = t.rpc;
        sh.nch = t.nch;
        return sh;
    };
    const int V = P.V;
    const int v0 = (int)(((long long)cta * V) / GG.G), v1 = (int)(((long long)(cta + 1) * V) / GG.G);
    const uint32_t rbv = (uint32_t)row_bytes(D, WF);
    // vocabulary rows per chunk: a power of two (its transpose-reduction), at most 32
    // vocabulary rows per chunk: as many as a slot holds, at most 32
    constexpr int kVocabFit = kCSlotBytes / row_bytes(D, WF);
    constexpr int kVocabRows = kVocabFit >= 32 ? 32 : kVocabFit;
    auto share_vocab = [&]() {
        Share sh = make_share(P.vocab + (uint64_t)v0 * rbv, rbv, v1 - v0);
        sh.rpc = kVocabRows < sh.n ? kVocabRows : (sh.n > 0 ? sh.n : 1);
        sh.nch = sh.n > 0 ? (sh.n + sh.rpc - 1) / sh.rpc : 0;
        return sh;
    };

    // ================================================= producer warp
    if (warp == kCWarps) {
        if (lane == 0 && !*s_abort) {
            const uint64_t pol = policy_evict_first();
            uint32_t gi = 0;                // chunks issued
            uint32_t pslot = 0, pfill = 0;  // slot of the next chunk, and how often the ring has wrapped
            bool stop = false;
            // Pacing: the block-matrix chunks are issued at least pace_ns per
            // 12 KB apart (scaled by the chunk's bytes).  Without it, the
            // slots a stage releases are refilled by every CTA at the same
            // moment, and that burst queues in front of the latency-bound
            // loads of the exchanges.  The vocabulary streams unpaced.
            uint64_t next_issue = 0;
            auto issue = [&](const Share& sh, bool paced) {
                for (int k = 0; k < sh.nch && !stop; ++k) {
                    const int slot = (int)pslot;
                    const uint32_t fill = pfill;
                    if (fill > 0) {
                        uint64_t t0 = 0;
                        uint32_t spins = 0;
                        while (!mbar_try_wait(&empty[slot], (fill - 1) & 1)) {
                            if (*s_abort) { stop = true; break; }
                            if ((++spins & 255) == 0) {
                                const uint64_t now = globaltimer_ns();
                                if (t0 == 0) t0 = now;
                                else if (now - t0 > 2 * P.wait_limit_ns) {
                                    crecord_error(P, kDevTimeout);
                                    stop = true;
                                    break;
                                }
                            }
                        }
                        if (stop) break;
                    }
                    const int r0 = k * sh.rpc;
                    const int n = min(sh.rpc, sh.n - r0);
                    const uint32_t bytes = (uint32_t)n * sh.pb;
                    if (paced && P.pace_ns != 0) {
                        uint64_t now = globaltimer_ns();
                        while (now < next_issue && !*s_abort) {
                            __nanosleep(32);
                            now = globaltimer_ns();
                        }
                        next_issue = (now > next_issue ? now : next_issue) +
                                     (uint64_t)P.pace_ns * bytes / (uint64_t)kCSlotBytes;
                    }
                    mbar_arrive_expect_tx(&full[slot], bytes);
                    bulk_load(ring + (size_t)slot * kCSlotBytes, sh.base + (uint64_t)r0 * sh.pb, bytes, &full[slot], pol);
                    ++gi;
                    if (++pslot == (uint32_t)NSL) {
                        pslot = 0;
                        ++pfill;
                    }
                }
            };
            // per step: the layers' shares in order, then the vocabulary rows
            // (layer index L), from one issue site
            for (int s = 0; s < P.n_steps && !stop; ++s) {
                for (int l = 0; l <= L && !stop; ++l) {
                    const int nj = l < L ? 2 * nh + 2 : 1;
                    for (int j = 0; j < nj && !stop; ++j) issue(l < L ? share_at(l, j) : share_vocab(), l < L);
                }
            }
            // every issued copy lands before this thread leaves
            const uint32_t nslot = gi < (uint32_t)NSL ? gi : (uint32_t)NSL;
            for (uint32_t i = 0; i < nslot; ++i) {
                const uint32_t last = gi - 1 - i;
                const int slot = (int)(last % (uint32_t)NSL);
                uint64_t t0 = 0;
                uint32_t spins = 0;
                while (!mbar_try_wait(&full[slot], (last / (uint32_t)NSL) & 1)) {
                    if ((++spins & 255) == 0) {
                        const uint64_t now = globaltimer_ns();
                        if (t0 == 0) t0 = now;
                        else if (now - t0 > 2 * P.wait_limit_ns) { crecord_error(P, kDevTimeout); break; }
                    }
                }
            }
        }
        __syncwarp();
        cluster_barrier();
        return;
    }

    // ================================================= consumer warps
    // Profiling (step 0) and the location of a wait that gave up.
    uint64_t* stamps = P.timing ? P.timing + 8 + (size_t)cta * cstamps_per_cta(L) : nullptr;
    int cur_step = 0, cur_layer = 0;
    auto stamp = [&](int k) {
        if (stamps && cur_step == 0 && tid == 0) stamps[k] = globaltimer_ns();
    };
    const unsigned per_step = (unsigned)cphases_per_step(L);
    const bool tracing = P.trace != nullptr;
    const int trace_layer = 8 * D + FF;
    const unsigned stall_tag = P.stall_phase >= 0 ? P.epoch + (unsigned)P.stall_phase : 0u;
    auto out_tag = [&](unsigned t) -> unsigned { return (cta == 0 && t == stall_tag) ? t - 1u : t; };
    int agree_no = 0;
    auto agree = [&](bool ok) -> bool {
        volatile int* slot = s_fail + (agree_no & 1);
        ++agree_no;
        if (!ok) *slot = 1;
        csync();
        return *slot == 0;
    };
    auto timed_out = [&](uint64_t& t0, int kind, uint64_t what = 0, uint64_t seen = 0) -> bool {
        const uint64_t now = globaltimer_ns();
        if (t0 == 0) { t0 = now; return false; }
        if (now - t0 <= kCAbortCheckNs) return false;
        return cwait_expired(P, now - t0, kind, cta, cur_step, cur_layer, what, seen,
                             stamps ? stamps + 16 * L + 4 : nullptr);
    };
    // Warp-uniform bounded wait for ring chunk cc.
    auto wait_chunk = [&](uint32_t slot, uint32_t par) -> bool {
        uint64_t t0 = 0;
        uint32_t spins = 0;
        while (!__all_sync(0xffffffffu, mbar_try_wait(&full[slot], par))) {
            if ((++spins & 63) == 0) {
                int give_up = lane == 0 ? (int)timed_out(t0, 1, slot | (par << 8)) : 0;
                if (__shfl_sync(0xffffffffu, give_up, 0)) return false;
            }
        }
        return true;
    };
    // The consumers' ring cursor: the slot of the next chunk to consume and
    // the parity of its fill (no division on the way).  Chunk k < slots
    // ahead of the cursor is in slot_of(k) with parity par_of(k).
    uint32_t rslot = 0, rpar = 0;
    auto ring_advance = [&](int n) {
        uint32_t t = rslot + (uint32_t)n;
        while (t >= (uint32_t)NSL) {
            t -= (uint32_t)NSL;
            rpar ^= 1u;
        }
        rslot = t;
    };
    // Bounded wait for one phase of a local mbarrier that peers complete.
    auto wait_bar = [&](uint64_t* bar, uint32_t par) -> bool {
        uint64_t t0 = 0;
        uint32_t spins = 0;
        while (!mbar_try_wait(bar, par)) {
            if ((++spins & 63) == 0 && timed_out(t0, 2, ((uint64_t)(bar - bars) << 8) | par)) return false;
        }
        return true;
    };
    // n floats (n % 4 == 0) at src into this CTA's row `dst` of a gather
    // buffer in every CTA of the cluster (same offset), completing on each
    // peer's mbarrier bar.
    // One bulk copy per peer, issued by lanes 0..CS-1 of warp 0; the writers
    // of src fenced their writes for the async proxy before the caller's
    // barrier.  The issuing lanes wait until the copies have read src, so
    // src may be rewritten after the next barrier.
    // With wait_now the issuing lanes wait until the copies have read src;
    // otherwise only until the previous call's copies have (so a caller
    // alternates between two source buffers, and a buffer is rewritten only
    // after the barrier that follows the next call).
    auto bcast = [&](const float* src, const float* dst, int n, uint64_t* bar, bool wait_now) {
        if (warp == 0 && lane < CS) {
            bulk_to_peer(mapa(smem_addr(dst), (uint32_t)lane), smem_addr(src), (uint32_t)n * 4u,
                         mapa(smem_addr(bar), (uint32_t)lane));
            asm volatile("cp.async.bulk.commit_group;" ::: "memory");
            if (wait_now) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
            else asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
        }
    };
    // One value to the same offset (local address a) of every CTA of the
    // cluster, this one included, completing 4 bytes on each one's mbarrier
    // (local address bar).  The all-gathers of partials are made of these:
    // each value leaves the thread that computed it, with no staging copy
    // and no barrier before the send.
    auto send_all = [&](uint32_t a, float v, uint32_t bar) {
#pragma unroll
        for (int q = 0; q < CS; ++q) st_async1(mapa(a, (uint32_t)q), v, mapa(bar, (uint32_t)q));
    };
    // Waits (bounded) for a gather of `bytes` on this CTA's mbarrier (armed
    // in advance), agrees on the outcome, and re-arms the barrier for its
    // next use.  Contains an agreement barrier.
    auto gather_wait = [&](uint64_t* bar, uint32_t bytes, uint32_t par, bool ok_in) -> bool {
        const bool ok = agree(ok_in && wait_bar(bar, par));
        if (ok && tid == 0) mbar_arrive_expect_tx(bar, bytes);
        return ok;
    };
    // Rows of a share against x4 (W4 float4 columns); row i's dot product to
    // out[i].  Chunk k is taken by warp k % 8.
    // The chunks are taken in rounds of one per warp with a barrier between
    // rounds.  The ring's barriers are waited on by phase parity, which is
    // only unambiguous if the previous fill of a chunk's slot has landed;
    // the rounds keep every warp within one round of the others, so the
    // previous fill of any slot this round uses (kCWarps <= slots) was
    // consumed in an earlier round.
    // With row_s != 0 each row's result is sent to offset 4 * row of row_s
    // (a gather row, local address) in every CTA of the cluster, completing
    // on bar_s; otherwise it is published as the tagged word gdst[row].
    // Either way it leaves the lane that computed it.
    auto run_share = [&](const Share& sh, const float* x, int W4, uint32_t row_s, uint32_t bar_s, uint64_t* gdst,
                         unsigned gtag) -> bool {
        bool ok = true;
        const uint32_t x_s = smem_addr(x);
        for (int k0 = 0; k0 < sh.nch; k0 += kCWarps) {
            const int k = k0 + warp;
            // this warp's chunk of the round: warp < kCWarps <= slots ahead of the cursor
            uint32_t slot = rslot + (uint32_t)warp, par = rpar;
            if (slot >= (uint32_t)NSL) {
                slot -= (uint32_t)NSL;
                par ^= 1u;
            }
            if (ok && k < sh.nch) {
                ok = wait_chunk(slot, par);
                if (ok) {
                    const uint32_t w = ring_s + slot * (uint32_t)kCSlotBytes;
                    const int n = min(sh.rpc, sh.n - k * sh.rpc);
                    const float v = chunk_rows<WF>(w, n, W4, x_s, lane);
                    if (lane < n) {
                        const int i = k * sh.rpc + lane;
                        if (row_s) send_all(row_s + 4u * (uint32_t)i, v, bar_s);
                        else st_tagged(gdst + i, gtag, v);
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&empty[slot]);
                }
            }
            ring_advance(min(kCWarps, sh.nch - k0));
            if (k0 + kCWarps < sh.nch) csync();
        }
        return ok;
    };
    // Deterministic block sum over the consumer threads (same value in all).
    auto block_sum = [&](float v) -> float {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0) s_red[warp] = v;
        csync();
        float t = 0.0f;
#pragma unroll
        for (int w = 0; w < kCWarps; ++w) t += s_red[w];
        csync();
        return t;
    };
    // Adds the nw (<= 24) partial vectors base[k * D + col0 + e] (k < nw,
    // tagged `tag`) and bias b to this slice of the residual, summed in
    // vector order: xs[e] += (sum_k v_k) + b[e].  Thread e < SW polls its
    // column's words, all loaded in one round trip per poll.  Ends with an
    // agreement barrier.
    constexpr int kMaxPollWords = 24;
    auto gather_add = [&](const uint64_t* base, int nw, unsigned tag, const float* bias) -> bool {
        bool ok = true;
        if (tid < SW) {
            uint64_t w[kMaxPollWords];
            uint32_t pending = (1u << nw) - 1u;
            const uint64_t* p0 = base + col0 + tid;
            const float bv = __ldg(bias + col0 + tid);
            uint64_t t0 = 0;
            while (pending) {
#pragma unroll
                for (int i = 0; i < kMaxPollWords; ++i)
                    if ((pending >> i) & 1u) w[i] = ld_tagged(p0 + (size_t)i * D);
#pragma unroll
                for (int i = 0; i < kMaxPollWords; ++i)
                    if (((pending >> i) & 1u) && tag_of(w[i]) == tag) pending &= ~(1u << i);
                if (pending && timed_out(t0, 3, pending)) { ok = false; break; }
            }
            if (ok) {
                float y = 0.0f;
#pragma unroll
                for (int i = 0; i < kMaxPollWords; ++i)
                    if (i < nw) y += val_of(w[i]);
                xs[tid] = __fadd_rn(xs[tid], __fadd_rn(y, bv));
            }
            fence_async_smem();
        }
        return agree(ok);
    };
    // This slice's (mean, M2) of x - s (two passes over SW values), by the
    // last consumer warp (the one without a chunk in most shares), into
    // dst[0..1].
    auto slice_stats = [&](float s, float* dst) {
        if (warp != kCWarps - 1) return;
        const float4* x4 = reinterpret_cast<const float4*>(xs);
        float a = 0.0f;
#pragma unroll 1
        for (int e = lane; e < SW / 4; e += 32) {
            const float4 v = x4[e];
            a += ((v.x - s) + (v.y - s)) + ((v.z - s) + (v.w - s));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
        const float mean = a * (1.0f / (float)SW);
        float q = 0.0f;
#pragma unroll 1
        for (int e = lane; e < SW / 4; e += 32) {
            const float4 v = x4[e];
            const float d0 = (v.x - s) - mean, d1 = (v.y - s) - mean, d2 = (v.z - s) - mean, d3 = (v.w - s) - mean;
            q = fmaf(d0, d0, fmaf(d1, d1, fmaf(d2, d2, fmaf(d3, d3, q))));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) q += __shfl_xor_sync(0xffffffffu, q, o);
        if (lane == 0) {
            dst[0] = mean;
            dst[1] = q;
        }
    };
    // Mean and inverse deviation of the whole vector from the CS slices'
    // (mean, M2) at base + r' * stride.  The slices have equal sizes, so the
    // mean is the mean of the slice means and the sum of squares is
    // sum M2_r + SW * sum (mean_r - mean)^2 (the pairwise update of Chan et
    // al. with equal counts), with no cancellation.
    auto merge_stats = [&](const float* base, int stride, float& mean, float& rstd) {
        float mu = 0.0f;
        for (int k = 0; k < CS; ++k) mu += base[k * stride];
        mu = mu * (1.0f / (float)CS);
        float m2 = 0.0f, sd = 0.0f;
        for (int k = 0; k < CS; ++k) {
            const float dl = base[k * stride] - mu;
            m2 += base[k * stride + 1];
            sd = fmaf(dl, dl, sd);
        }
        m2 = fmaf((float)SW, sd, m2);
        mean = mu;
        rstd = rsqrtf(fmaf(m2, 1.0f / (float)D, kLnEps));
    };

    // Greedy partials of the previous step (tag), reduced in every CTA; the
    // acquire pairs with each CTA's release, so the KV rows of that step are
    // visible to this step's attention.
    auto reduce_choice = [&](unsigned tag) -> bool {
        bool ok = true;
        if (tid < GG.G) {
            const uint64_t* ap = P.arg_part + 2 * (size_t)tid;
            uint64_t t0 = 0;
            uint64_t w0 = ld_tagged_acquire(ap);
            while (tag_of(w0) != tag) {
                if (timed_out(t0, 4, ((uint64_t)tid << 32) | tag, w0)) { ok = false; break; }
                w0 = ld_tagged_acquire(ap);
            }
            if (ok) {
                const uint64_t w1 = ld_tagged(ap + 1);
                if (tag_of(w1) != tag) {
                    crecord_error(P, kDevTimeout);
                    ok = false;
                }
                stage[tid] = val_of(w0);
                stage[384 + tid] = val_of(w1);
            }
        }
        if (!agree(ok)) return false;
        if (warp == 0) {
            Best b{-INFINITY, 0xFFFFFFFFu, 0};
            for (int k = lane; k < GG.G; k += 32) {
                const unsigned iw = __float_as_uint(stage[384 + k]);
                best_merge(b, stage[k], iw & 0x7FFFFFFFu, (int)(iw >> 31));
            }
            best_warp(b);
            if (lane == 0) {
                *s_tok = b.nf ? 0xFFFFFFFFu : b.i;
                *s_nf = b.nf;
            }
        }
        csync();
        return true;
    };
    auto publish_choice = [&](int s_done, unsigned choice, int nf) {
        if (tid == 0 && cta == 0) {
            if (P.tokens_out) P.tokens_out[s_done] = choice;
            *P.last_token = choice;
            if (nf) atomicCAS(P.status, 0, (int)kDevNonfinite);
        }
    };

    // Attention of head h (layer l, position p) over this CTA's keys
    // [k0, k1) of 0..p: (max, sum, unnormalised weighted values) sent to
    // words 0, 1 and 4 .. 4 + DH of gather row row_s in every CTA of the
    // cluster.  LPK lanes per key, DPL dims per lane;
    // the current position's key and value come from qkv (this step's).
    constexpr int LPK = DH >= 32 ? 8 : 4;
    constexpr int KPW = 32 / LPK;
    constexpr int DPL = DH / LPK;
    constexpr int F4 = DPL / 4;
    constexpr int KPP = kCWarps * KPW;
    static_assert(DPL % 4 == 0, "a lane holds whole float4s of a head row");
    const int ks = lane / LPK, dc = lane % LPK;
    float4 ka[F4], va[F4];
    auto fetch = [&](const float* kv0, int j, int k1, int p, float4 (&kk)[F4], float4 (&vv)[F4]) {
        if (j < k1 && j < p) {
            const float4* row = reinterpret_cast<const float4*>(kv0 + (uint64_t)j * L * 2 * D);
#pragma unroll
            for (int f = 0; f < F4; ++f) {
                kk[f] = __ldcg(row + f);
                vv[f] = __ldcg(row + D / 4 + f);
            }
        }
    };
    auto attention = [&](int l, int h, int p, int k0, int k1, uint32_t row_s, uint32_t bar_s) {
        const float* kv0 = P.cache + (uint64_t)l * 2 * D + h * DH + dc * DPL;
        const float den = sqrtf((float)DH);
        const float4* q4 = reinterpret_cast<const float4*>(qkv + dc * DPL);
        float m = -INFINITY, z = 0.0f;
        float acc[DPL];
#pragma unroll
        for (int d = 0; d < DPL; ++d) acc[d] = 0.0f;
        int j = k0 + warp * KPW + ks;
        for (int jb = k0 + warp * KPW; jb < k1; jb += KPP, j += KPP) {
            float4 kb[F4], vb[F4];
            fetch(kv0, j + KPP, k1, p, kb, vb);  // next pass
            if (j == p) {
#pragma unroll
                for (int f = 0; f < F4; ++f) {
                    ka[f] = reinterpret_cast<const float4*>(qkv + DH + dc * DPL)[f];
                    va[f] = reinterpret_cast<const float4*>(qkv + 2 * DH + dc * DPL)[f];
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
                const float corr = expf(m - mn);
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
        if (ks == 0) {
            float* st = stage + (warp * LPK + dc) * (2 + DPL);
            st[0] = m;
            st[1] = z;
#pragma unroll
            for (int d = 0; d < DPL; ++d) st[2 + d] = acc[d];
        }
        csync();
        if (tid < DH) {
            const int cq = tid / DPL, d = tid - cq * DPL;
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < kCWarps; ++w) M = fmaxf(M, stage[(w * LPK + cq) * (2 + DPL)]);
            float Z = 0.0f, O = 0.0f;
            if (M != -INFINITY) {
#pragma unroll
                for (int w = 0; w < kCWarps; ++w) {
                    const float* st = stage + (w * LPK + cq) * (2 + DPL);
                    if (st[0] == -INFINITY) continue;
                    const float cw = expf(st[0] - M);
                    Z = fmaf(st[1], cw, Z);
                    O = fmaf(st[2 + d], cw, O);
                }
            }
            send_all(row_s + 4u * (uint32_t)(4 + tid), O, bar_s);
            if (tid == 0) {
                send_all(row_s, M, bar_s);
                send_all(row_s + 4u, Z, bar_s);
            }
        }
    };

    const float* fold = P.fold;
    const uint64_t fold_words = fold_layer_words(D, FF);
    unsigned prev_choice = *P.last_token;
    bool alive = !*s_abort;
    uint32_t useA = 0, useT = 0, useB = 0;  // uses of the double-buffered gathers
    float* s_st = s_stA;                      // this slice's (mean, M2) of the LayerNorm input
    int s = 0;
    // s = n_steps only reduces the last step's greedy choice (in CTA 0, which
    // reports it), so that the reduction has one copy in the binary
    for (; s <= P.n_steps && alive; ++s) {
        const int p = P.p0 + s;
        const unsigned base = P.epoch + (unsigned)s * per_step;
        const bool tr = tracing && s == 0;
        cur_step = s;
        cur_layer = 0;
        if (s > 0) {
            if (s == P.n_steps && cta != 0) break;
            if (!reduce_choice(base)) { alive = false; break; }
            prev_choice = *s_tok;
            const int nf = *s_nf;
            publish_choice(s - 1, prev_choice, nf);
            if (nf) { alive = false; break; }
        }
        if (s == P.n_steps) break;
        // this CTA's keys [att_k0, att_k1) of positions 0..p (cached ones below att_k1c)
        const int att_k0 = (int)(((long long)r * (p + 1)) / CS), att_k1 = (int)(((long long)(r + 1) * (p + 1)) / CS);
        const int att_k1c = att_k1 < p ? att_k1 : p;
        unsigned tok = P.tokens_in ? P.tokens_in[s] : P.token0;
        if (tok == 0xFFFFFFFFu) tok = prev_choice;
        if (tok >= (unsigned)V) {
            if (tid == 0 && cta == 0) crecord_error(P, kDevToken);
            alive = false;
            break;
        }
        // ---- embedding (every CTA forms the whole vector for its exact mean)
        float esum = 0.0f;
        for (int i = tid; i < D; i += NT) {
            float te;
            if constexpr (WF == kWF16) te = __half2float(reinterpret_cast<const __half*>(P.vocab)[(uint64_t)tok * D + i]);
            else te = __ldg(P.packed + P.wte_off + (uint64_t)tok * D + i);
            const float x = __fadd_rn(te, __ldg(P.packed + P.wpe_off + (uint64_t)p * D + i));
            xf[i] = x;
            esum += x;
        }
        const float mu_emb = block_sum(esum) / (float)D;  // (block_sum ends with a barrier: xf complete)
        for (int e = tid; e < SW; e += NT) xs[e] = xf[col0 + e];
        float shift = mu_emb;  // the last LayerNorm mean every CTA of this cluster holds
        csync();

        for (int l = 0; l < L && alive; ++l) {
            cur_layer = l;
            const LayerParams& lp = P.lp[l];
            const unsigned tagA = base + 2u * (unsigned)l + 1u, tagB = tagA + 1u;
            const float* fl = fold + (uint64_t)l * fold_words;
            const float g1 = tid < SW ? __ldg(P.packed + lp.ln1_g + col0 + tid) : 0.0f;
            const float g2 = tid < SW ? __ldg(P.packed + lp.ln2_g + col0 + tid) : 0.0f;
            float ln_shift = shift;  // shift of the LayerNorm being folded
            // this layer's cached keys and values of this CTA's attention
            // positions, prefetched into L2 while the block input forms
            // (four 128-byte lines per position and head: key and value halves)
#pragma unroll 1
            for (int hs = 0; hs < nh; ++hs) {
                const float* hrow = P.cache + (uint64_t)l * 2 * D + (c + hs * GG.NC) * DH;
#pragma unroll 1
                for (int t = tid; t < (att_k1c - att_k0) * 4; t += NT) {
                    const float* row = hrow + (uint64_t)(att_k0 + (t >> 2)) * L * 2 * D + ((t >> 1) & 1) * D +
                                       (t & 1) * (DH / 2);
                    asm volatile("prefetch.global.L2 [%0];" ::"l"(row));
                }
            }
            // Micro-phases of the layer, one runtime loop so that each routine
            // (gather, dot products, all-gather, store) has one copy in the
            // binary: per head slot k of this cluster QKV (0), attention (1),
            // out-projection (2); then FC (3) and MLP projection (4).
            const int nmp = 3 * nh + 2;
            for (int mp = 0; mp < nmp; ++mp) {
                const int kind = mp < 3 * nh ? mp % 3 : 3 + (mp - 3 * nh);
                const int k = mp < 3 * nh ? mp / 3 : 0;
                const int h = c + k * GG.NC;
                // the cluster all-gather of this micro-phase (QKV partials,
                // attention partials, FC partials): use u of a double-buffered
                // gather buffer of CS rows of rowl floats, nval values per row
                const bool gat = kind == 0 || kind == 1 || kind == 3;
                uint32_t u = 0;
                int rowl = 0, nval = 0;
                float* gbuf = nullptr;
                uint64_t* bar = nullptr;
                if (kind == 0) {
                    u = useA++;
                    rowl = 3 * DH + 4;
                    nval = 3 * DH + 2;
                    gbuf = gA + (size_t)(u & 1) * CS * rowl;
                    bar = &bars[0 + (u & 1)];
                } else if (kind == 1) {
                    u = useT++;
                    rowl = DH + 4;
                    nval = DH + 2;
                    gbuf = gT + (size_t)(u & 1) * CS * rowl;
                    bar = &bars[2 + (u & 1)];
                } else if (kind == 3) {
                    u = useB++;
                    rowl = GG.nfc_max + 4;
                    nval = nfc + 2;
                    gbuf = gB + (size_t)(u & 1) * CS * rowl;
                    bar = &bars[4 + (u & 1)];
                }
                const uint32_t row_s = gat ? smem_addr(gbuf + (size_t)r * rowl) : 0u;
                const uint32_t bar_s = gat ? smem_addr(bar) : 0u;
                // ---- the residual slice a LayerNorm of this micro-phase reads
                if ((kind == 0 && k == 0) || kind == 3) {
                    // q = 0: the previous layer's MLP partials (block input);
                    // q = 1: this layer's out-projection partials (attention residual)
                    const int q0 = (l > 0 && (kind == 0 || nh == 0)) ? 0 : 1, q1 = kind == 3 ? 1 : 0;
                    for (int q = q0; q <= q1 && alive; ++q) {
                        const uint64_t* src = q == 0 ? CP.partP + (size_t)((l - 1) & 1) * GG.NC * D : CP.partO;
                        if (!gather_add(src, q == 0 ? GG.NC : H, q == 0 ? tagA - 1u : tagA,
                                        P.packed + (q == 0 ? P.lp[l - 1].b_p : lp.b_o))) {
                            alive = false;
                            break;
                        }
                        stamp(16 * l + (q == 0 ? 0 : 6));
                        if (tr && c == 0) ctrace_copy(P.trace + (size_t)l * trace_layer + (q == 0 ? 0 : 6 * D) + col0, xs, SW, tid);
                    }
                    if (!alive) break;
                    if (l == 0 && kind == 0) {
                        stamp(0);
                        if (tr && c == 0) ctrace_copy(P.trace + col0, xs, SW, tid);
                    }
                    ln_shift = shift;
                    if (tid < SW) xin[tid] = (kind == 0 ? g1 : g2) * (xs[tid] - ln_shift);
                    csync();
                    slice_stats(ln_shift, s_st);
                }
                // ---- dot products of this micro-phase's share (attention has none)
                bool ok_share = true;
                if (kind != 1) {
                    Share sh;
                    const float* xv;
                    int W4;
                    sh = share_at(l, kind == 0 ? 2 * k : kind == 2 ? 2 * k + 1 : kind == 3 ? 2 * nh : 2 * nh + 1);
                    if (kind == 0 || kind == 3) { xv = xin; W4 = SW / 4; }
                    else if (kind == 2) { xv = oh; W4 = DH / 4; }
                    else { xv = uu; W4 = nfc4 / 4; }
                    if (gat && warp == kCWarps - 1 && lane == 0) {
                        // this slice's LayerNorm statistics go with the partials
                        const uint32_t n0 = (uint32_t)(kind == 0 ? 3 * DH : nfc4);
                        send_all(row_s + 4u * n0, s_st[0], bar_s);
                        send_all(row_s + 4u * (n0 + 1u), s_st[1], bar_s);
                    }
                    // out-projection (2) or MLP (4) partials of this CTA's output
                    // rows, published as tagged words
                    uint64_t* gdst = kind == 2 ? CP.partO + (size_t)h * D + col0
                                   : kind == 4 ? CP.partP + ((size_t)(l & 1) * GG.NC + c) * D + col0 : nullptr;
                    ok_share = run_share(sh, xv, W4, row_s, bar_s, gdst, out_tag(kind == 2 ? tagA : tagB));
                    if (!gat && !agree(ok_share)) { alive = false; break; }
                    stamp(16 * l + (kind == 0 ? 1 : kind == 2 ? 5 : kind == 3 ? 7 : 9));
                } else {
                    attention(l, h, p, att_k0, att_k1, row_s, bar_s);
                    stamp(16 * l + 3);
                }
                // ---- the cluster all-gather completes, then its epilogue
                if (gat) {
                    // loaded while the gather completes: the first keys of this
                    // CTA's attention share, and this thread's fold constants
                    float cj = 0.0f, dj = 0.0f;
                    if (kind == 0)
                        fetch(P.cache + (uint64_t)l * 2 * D + h * DH + dc * DPL, att_k0 + warp * KPW + ks, att_k1, p, ka, va);
                    if ((kind == 0 && tid < 3 * DH) || (kind == 3 && tid < nfc)) {
                        const int Jt = kind == 0 ? (tid / DH) * D + h * DH + (tid % DH) : 6 * D + f0 + tid;
                        cj = __ldg(fl + Jt);
                        dj = __ldg(fl + Jt + (kind == 0 ? 3 * D : FF));
                    }
                    if (!gather_wait(bar, (uint32_t)(CS * nval * 4), (u >> 1) & 1, ok_share)) { alive = false; break; }
                    stamp(16 * l + (kind == 0 ? 2 : kind == 1 ? 4 : 8));
                    // ---- epilogues of the gathered values
                    if (kind == 1) {
                        if (tid < DH) {
                            float M = -INFINITY;
                            for (int q = 0; q < CS; ++q) M = fmaxf(M, gbuf[(size_t)q * rowl]);
                            float Z = 0.0f, O = 0.0f;
#pragma unroll
                            for (int q = 0; q < CS; ++q) {
                                const float* row = gbuf + (size_t)q * rowl;
                                if (row[0] == -INFINITY) continue;
                                const float cw = expf(row[0] - M);
                                Z = fmaf(row[1], cw, Z);
                                O = fmaf(row[4 + tid], cw, O);
                            }
                            const float o = O / Z;
                            oh[tid] = o;
                            if (tr && r == 0) P.trace[(size_t)l * trace_layer + 5 * D + h * DH + tid] = o;
                        }
                    } else {
                        // QKV (0) or FC (3): the CS slice partials summed in
                        // rank order, the LayerNorm fold, then q/k/v (and the
                        // KV append) or the GELU output
                        // (the loop's per-kind choices are selects, so that
                        // the compiler keeps one copy of its body)
                        const bool qk = kind == 0;
                        const int nrow = qk ? 3 * DH : nfc;
                        float* dstv = qk ? qkv : uu;
                        const int klo = qk ? kv_lo : 0, khi = qk ? kv_hi : 0;
                        float* kvrow = P.cache + ((uint64_t)p * L + l) * 2 * D - D;
                        float* trp = (tr && r == 0) ? P.trace + (size_t)l * trace_layer + (qk ? 2 * D : 8 * D + f0)
                                                    : nullptr;
                        const int dstride = qk ? 3 * D : FF;
                        float mean, rstd;
                        merge_stats(gbuf + (qk ? 3 * DH : nfc4), rowl, mean, rstd);
#pragma unroll 1
                        for (int j = tid; j < nrow; j += NT) {
                            float a = 0.0f;
                            float pv[16];
#pragma unroll
                            for (int q = 0; q < 16; ++q) pv[q] = q < CS ? gbuf[(size_t)q * rowl + j] : 0.0f;
#pragma unroll
                            for (int q = 0; q < 16; ++q) if (q < CS) a += pv[q];
                            const int Jr = qk ? (j / DH) * D + h * DH + (j % DH) : 6 * D + f0 + j;
                            float cc = cj, dd = dj;
                            if (j != tid) {
                                cc = __ldg(fl + Jr);
                                dd = __ldg(fl + Jr + dstride);
                            }
                            const float y0 = fmaf(rstd, fmaf(-mean, cc, a), dd);
                            const float y = qk ? y0 : cgelu(y0);
                            dstv[j] = y;
                            if (j >= klo && j < khi) kvrow[Jr] = y;
                            if (trp) trp[qk ? Jr : j] = y;
                        }
                        if (tr && c == 0 && (!qk || k == 0))
                            ctrace_ln(P.trace + (size_t)l * trace_layer + (qk ? D : 7 * D) + col0, xs, ln_shift + mean,
                                      rstd, P.packed + (qk ? lp.ln1_g : lp.ln2_g) + col0,
                                      P.packed + (qk ? lp.ln1_b : lp.ln2_b) + col0, SW, tid);
                        if (!qk || k == nh - 1) shift = ln_shift + mean;
                    }
                    csync();
                }
            }
        }
        if (!alive) break;
        // ================= final LayerNorm and the vocabulary rows
        if (!gather_add(CP.partP + (size_t)((L - 1) & 1) * GG.NC * D, GG.NC, base + 2u * (unsigned)L,
                        P.packed + P.lp[L - 1].b_p)) {
            alive = false;
            break;
        }
        stamp(16 * L + 0);
        bcast(xs, gX + col0, SW, &bars[6], true);
        {
            if (!gather_wait(&bars[6], (uint32_t)(D * 4), (uint32_t)s & 1, true)) { alive = false; break; }
        }
        stamp(16 * L + 1);
        // LN_f over the whole vector: mean, then squares around it (the oracle's two passes)
        float sx = 0.0f;
        for (int i = tid; i < D; i += NT) sx += gX[i];
        const float mean = block_sum(sx) / (float)D;
        float sq = 0.0f;
        for (int i = tid; i < D; i += NT) {
            const float d = gX[i] - mean;
            sq = fmaf(d, d, sq);
        }
        const float var = block_sum(sq) / (float)D;
        const float den = sqrtf(var + kLnEps);
        for (int i = tid; i < D; i += NT) {
            const float y = __fadd_rn(__fmul_rn(__fdiv_rn(__fsub_rn(gX[i], mean), den), __ldg(P.packed + P.lnf_g + i)),
                                      __ldg(P.packed + P.lnf_b + i));
            xf[i] = y;
        }
        if (tr && cta == 0) {
            ctrace_copy(P.trace + (size_t)L * trace_layer, gX, D, tid);
            ctrace_copy(P.trace + (size_t)L * trace_layer + D, xf, D, tid);
        }
        csync();
        stamp(16 * L + 2);
        // vocabulary rows of this CTA: logits and the running greedy choice
        {
            const Share sh = share_vocab();
            float* lg = P.logits ? P.logits + (uint64_t)s * P.logits_stride : nullptr;
            Best best{-INFINITY, 0xFFFFFFFFu, 0};
            bool ok = true;
            const uint32_t xf_s = smem_addr(xf);
            // rounds of one chunk per warp, as in run_share
            for (int k0 = 0; k0 < sh.nch; k0 += kCWarps) {
                const int kc = k0 + warp;
                uint32_t slot = rslot + (uint32_t)warp, par = rpar;
                if (slot >= (uint32_t)NSL) {
                    slot -= (uint32_t)NSL;
                    par ^= 1u;
                }
                if (ok && kc < sh.nch) {
                    ok = wait_chunk(slot, par);
                    if (ok) {
                        const uint32_t w = ring_s + slot * (uint32_t)kCSlotBytes;
                        const int n = min(sh.rpc, sh.n - kc * sh.rpc);
                        const float v = long_rows<kVocabRows, D / 4, WF>(w, sh.pb, n, xf_s, lane);
                        if (lane < n) {
                            const int j = v0 + kc * sh.rpc + lane;
                            if (lg) lg[j] = v;
                            best_update(best, v, (unsigned)j);
                        }
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&empty[slot]);
                    }
                }
                ring_advance(min(kCWarps, sh.nch - k0));
                if (k0 + kCWarps < sh.nch) csync();
            }
            best_warp(best);
            if (lane == 0) {
                s_arg[warp * 3 + 0] = best.v;
                s_arg[warp * 3 + 1] = __uint_as_float(best.i);
                s_arg[warp * 3 + 2] = (float)best.nf;
            }
            if (!agree(ok)) { alive = false; break; }
            if (tid == 0) {
                Best b = {s_arg[0], __float_as_uint(s_arg[1]), s_arg[2] != 0.0f};
                for (int w = 1; w < kCWarps; ++w)
                    best_merge(b, s_arg[w * 3 + 0], __float_as_uint(s_arg[w * 3 + 1]), s_arg[w * 3 + 2] != 0.0f);
                if (stamps && s == 0) stamps[16 * L + 3] = globaltimer_ns();
                const unsigned tg = out_tag(base + per_step);
                uint64_t* ap = P.arg_part + 2 * (size_t)cta;
                const unsigned iw = (b.i & 0x7FFFFFFFu) | (b.nf ? 0x80000000u : 0u);
                st_tagged(ap + 1, tg, __uint_as_float(iw));
                // release: this CTA's KV rows and choice become visible with it
                st_tagged_release(ap, tag_pack(tg, b.v));
            }
        }
    }
    if (tid == 0) *s_abort = 1;  // the producer stops issuing
    // this CTA's copies into its peers have landed before any CTA of the
    // cluster leaves (a run that stopped early may have some in flight)
    if (warp == 0 && lane < CS) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
    // A run that stopped early may also leave values of an all-gather in
    // flight towards a peer that will not wait for them; they land within
    // microseconds, so the CTA lingers 20 us before the cluster leaves.
    if (!alive) __nanosleep(20000);
    cluster_barrier();
}

// ------------------------------------------------------------ weight layout
// Byte offset of weight e of row i in a share of n rows of W weights (wb
// bytes each): rows are grouped into ring chunks of rpc rows (rpc =
// min(32, slot bytes / row bytes)), and inside a chunk of R rows the rows
// are interleaved by 4-weight units: unit c of row i' at (c * R + i') units.
__host__ __device__ inline uint64_t cunit_off(int i, int e, int n, int W, int wb) {
    const uint32_t pb = (uint32_t)W * (uint32_t)wb;
    int rpc = (int)(kCSlotBytes / pb);
    if (rpc > 32) rpc = 32;
    if (rpc > n) rpc = n;
    const int k = i / rpc, i2 = i - k * rpc;
    const int R = (n - k * rpc) < rpc ? (n - k * rpc) : rpc;
    const int cu = e >> 2, sub = e & 3;
    return (uint64_t)k * rpc * pb + ((uint64_t)cu * R + i2) * 4u * wb + (uint64_t)sub * wb;
}

// Copies one layer of the K-major device stream (rows [out][in], row pitch
// rbd for width-D inputs and rbf for width-FF inputs, wb bytes per weight)
// into the cluster layout: block (c*CS + r) writes CTA (c, r)'s part.
__global__ void clayout_kernel(const uint8_t* __restrict__ src, const CGeo g, int D, int H, int FF, int DH,
                               uint64_t mat_qkv, uint64_t mat_o, uint64_t mat_fc, uint64_t mat_p, uint32_t rbd,
                               uint32_t rbf, uint8_t* __restrict__ dst) {
    const int cta = blockIdx.x, c = cta / g.CS, r = cta % g.CS;
    const int wb = g.wb, SW = g.SW, col0 = r * SW;
    const int nh = cg_heads(g, H, c);
    const int f0 = g.fc0[c], nfc = g.fc0[c + 1] - f0;
    uint8_t* out = dst + g.seg[c] + (uint64_t)r * g.cta_bytes[c];
    auto copy = [&](uint8_t* d, const uint8_t* s_) {
        if (wb == 4) *reinterpret_cast<uint32_t*>(d) = *reinterpret_cast<const uint32_t*>(s_);
        else *reinterpret_cast<uint16_t*>(d) = *reinterpret_cast<const uint16_t*>(s_);
    };
    uint64_t o = 0;
    for (int k = 0; k < nh; ++k) {
        const int h = c + k * g.NC;
        for (int t = threadIdx.x; t < 3 * DH * SW; t += blockDim.x) {
            const int i = t / SW, e = t - i * SW;
            const int J = (i / DH) * D + h * DH + (i % DH);
            copy(out + o + cunit_off(i, e, 3 * DH, SW, wb),
                 src + mat_qkv + (uint64_t)J * rbd + (uint64_t)(col0 + e) * wb);
        }
        o += (uint64_t)3 * DH * SW * wb;
        for (int t = threadIdx.x; t < SW * DH; t += blockDim.x) {
            const int i = t / DH, e = t - i * DH;
            copy(out + o + cunit_off(i, e, SW, DH, wb),
                 src + mat_o + (uint64_t)(col0 + i) * rbd + (uint64_t)(h * DH + e) * wb);
        }
        o += (uint64_t)SW * DH * wb;
    }
    for (int t = threadIdx.x; t < nfc * SW; t += blockDim.x) {
        const int i = t / SW, e = t - i * SW;
        copy(out + o + cunit_off(i, e, nfc, SW, wb), src + mat_fc + (uint64_t)(f0 + i) * rbd + (uint64_t)(col0 + e) * wb);
    }
    o += (uint64_t)nfc * SW * wb;
    for (int t = threadIdx.x; t < SW * nfc; t += blockDim.x) {
        const int i = t / nfc, e = t - i * nfc;
        copy(out + o + cunit_off(i, e, SW, nfc, wb), src + mat_p + (uint64_t)(col0 + i) * rbf + (uint64_t)(f0 + e) * wb);
    }
}

// ------------------------------------------------------------ host side
namespace {

template <int D, int FF, int DH, int WF>
cudaError_t set_attrs(uint32_t smem) {
    auto kern = cstep_kernel<D, FF, DH, WF>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    return e;
}

template <int D, int FF, int DH, int WF>
cudaError_t launch_t(const CPlan& P, cudaStream_t stream) {
    const CSmem lay = csmem_layout(D, DH, P.g.CS, P.g.SW, P.g.nfc_max, P.g.slots);
    cudaError_t e = set_attrs<D, FF, DH, WF>(lay.total);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(P.g.G);
    cfg.blockDim = dim3(kCThreads);
    cfg.dynamicSmemBytes = lay.total;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)P.g.CS;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeCooperative;
    attr[1].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, cstep_kernel<D, FF, DH, WF>, P);
}

template <int D, int FF, int DH, int WF>
int max_clusters_t(int CS, uint32_t smem) {
    if (set_attrs<D, FF, DH, WF>(smem) != cudaSuccess) return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(CS);
    cfg.blockDim = dim3(kCThreads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)CS;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, (void*)cstep_kernel<D, FF, DH, WF>, &cfg) != cudaSuccess) return 0;
    return n;
}

#define CSTEP_DISPATCH_WF(FN, d, ff, dh, ...)                 \
    return wf == kWF16 ? FN<d, ff, dh, kWF16>(__VA_ARGS__) : FN<d, ff, dh, kWF32>(__VA_ARGS__);
#define CSTEP_DISPATCH(FN, ...)                                                                \
    if (D == 768 && FF == 3072 && DH == 64) { CSTEP_DISPATCH_WF(FN, 768, 3072, 64, __VA_ARGS__) } \
    if (D == 192 && FF == 384 && DH == 64) { CSTEP_DISPATCH_WF(FN, 192, 384, 64, __VA_ARGS__) }   \
    if (D == 64 && FF == 256 && DH == 16) { CSTEP_DISPATCH_WF(FN, 64, 256, 16, __VA_ARGS__) }

int max_clusters(int D, int FF, int DH, int wf, int CS, uint32_t smem) {
    CSTEP_DISPATCH(max_clusters_t, CS, smem)
    return 0;
}

// Cluster size per model width: a slice of 128 floats (one warp of float4
// columns) where the width allows.
}  // namespace

bool cstep_supported(int D, int FF, int DH, int wf) {
    if (wf != kWF32 && wf != kWF16) return false;
    return (D == 768 && FF == 3072 && DH == 64) || (D == 192 && FF == 384 && DH == 64) ||
           (D == 64 && FF == 256 && DH == 16);
}

// Chooses the cluster geometry: clusters of CS CTAs (CS = D / 128 at GPT-2
// 124M, i.e. 6), as many clusters as are co-resident (at most want_ctas / CS
// when want_ctas > 0), the FC rows split so that every CTA streams about the
// same bytes per layer (head clusters also stream QKV and out-projection
// parts), in multiples of 8 rows.
cudaError_t cgeo_make(int L, int D, int H, int FF, int wf, int want_ctas, CGeo* out) {
    (void)L;
    const int DH = D / H;
    CGeo g;
    memset(&g, 0, sizeof(g));
    const int CS = cluster_size_for(D);
    if (CS < 1 || CS > 16 || D % CS != 0 || (D / CS) % 8 != 0) return cudaErrorInvalidValue;
    g.CS = CS;
    g.SW = D / CS;
    g.wb = wf == kWF16 ? 2 : 4;
    if (g.SW > kCWarps * 32 || FF % 8 != 0 || DH % 8 != 0 || H > 24) return cudaErrorInvalidValue;
    // clusters co-resident at one CTA per SM (the kernel's ring takes what
    // shared memory the rest leaves)
    int maxc = max_clusters(D, FF, DH, wf, CS, (uint32_t)kCMaxSmem);
    if (maxc <= 0) return cudaErrorInvalidConfiguration;
    // at most 24 clusters: a CTA polls one word per cluster in one round trip
    int NC = maxc < 24 ? maxc : 24;
    if (want_ctas > 0) {
        const int w = (want_ctas + CS - 1) / CS;
        if (w < NC) NC = w;
    }
    while (NC > 1 && FF / NC < 8) --NC;
    while (NC > 1 && NC * CS > kCWarps * 32) --NC;  // one greedy partial per consumer thread
    g.NC = NC;
    g.G = NC * CS;
    g.HPC = (H + NC - 1) / NC;
    if (g.HPC > kCMaxHeadSlots) return cudaErrorInvalidValue;
    // FC rows: head clusters carry 4 * DH * SW weights of attention per head
    // and CTA; an FC row costs 2 * SW weights per CTA (FC and MLP parts), so
    // equal bytes per CTA means nfc_c = base - 2 * DH * heads(c).  frac
    // (GPT2_FC_BALANCE) scales that correction; the default 0 gives equal
    // rows, which measured faster (the stage that follows the FC rows waits
    // for the slowest cluster).
    double frac = 0.0;
    const char* env_bal = getenv("GPT2_FC_BALANCE");
    if (env_bal) frac = atof(env_bal);
    std::vector<int> nrow(NC);
    {
        double corr = 0.0;
        for (int c = 0; c < NC; ++c) corr += frac * 2.0 * DH * cg_heads(g, H, c);
        const double base = ((double)FF + corr) / NC;
        int tot = 0;
        for (int c = 0; c < NC; ++c) {
            const double w = base - frac * 2.0 * DH * cg_heads(g, H, c);
            int n = (int)(w / 8.0 + 0.5) * 8;
            if (n < 8) n = 8;
            nrow[c] = n;
            tot += n;
        }
        // bring the total to FF in steps of 8 rows, largest clusters first
        for (int it = 0; tot != FF && it < 100000; ++it) {
            int best = -1;
            for (int c = 0; c < NC; ++c) {
                if (tot > FF && nrow[c] > 8 && (best < 0 || nrow[c] > nrow[best])) best = c;
                if (tot < FF && (best < 0 || nrow[c] < nrow[best])) best = c;
            }
            if (best < 0) return cudaErrorInvalidValue;
            nrow[best] += tot > FF ? -8 : 8;
            tot += tot > FF ? -8 : 8;
        }
        if (tot != FF) return cudaErrorInvalidValue;
    }
    {
        int o = 0;
        g.nfc_max = 0;
        for (int c = 0; c < NC; ++c) {
            g.fc0[c] = o;
            o += nrow[c];
            if (nrow[c] > g.nfc_max) g.nfc_max = nrow[c];
        }
        g.fc0[NC] = o;
    }
    // stream layout
    uint64_t off = 0;
    for (int c = 0; c < NC; ++c) {
        const int nh = cg_heads(g, H, c), nfc = g.fc0[c + 1] - g.fc0[c];
        g.cta_bytes[c] = (uint64_t)nh * cg_head_bytes(g, DH) + (uint64_t)2 * nfc * g.SW * g.wb;
        g.seg[c] = off;
        off += (uint64_t)CS * g.cta_bytes[c];
    }
    g.seg[NC] = off;
    g.layer_bytes = off;
    // ring: as many slots as fit
    // at least one round of chunks (one per consumer warp) must fit the ring
    int slots = kCMaxSlots;
    while (slots > kCWarps && csmem_layout(D, DH, CS, g.SW, g.nfc_max, slots).total > (uint32_t)kCMaxSmem) --slots;
    if (csmem_layout(D, DH, CS, g.SW, g.nfc_max, slots).total > (uint32_t)kCMaxSmem) return cudaErrorInvalidValue;
    g.slots = slots;
    *out = g;
    return cudaSuccess;
}

cudaError_t cstream_build(const uint8_t* wstream, uint64_t layer_bytes, const uint64_t mat_off[4], int L, int D,
                          int H, int FF, int wf, const CGeo& g, uint8_t* dst, cudaStream_t st) {
    const uint32_t rbd = (uint32_t)row_bytes(D, wf), rbf = (uint32_t)row_bytes(FF, wf);
    for (int l = 0; l < L; ++l) {
        const uint8_t* src = wstream + (uint64_t)l * layer_bytes;
        clayout_kernel<<<g.G, 256, 0, st>>>(src, g, D, H, FF, D / H, mat_off[kQKV], mat_off[kO], mat_off[kFC],
                                            mat_off[kP], rbd, rbf, dst + (uint64_t)l * g.layer_bytes);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t launch_cstep(const CPlan& P, int wf, cudaStream_t stream) {
    const int D = P.s.D, FF = P.s.FF, DH = P.s.D / P.s.H;
    CSTEP_DISPATCH(launch_t, P, stream)
    return cudaErrorInvalidValue;
}

}  // namespace gpt2
