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

#include "gpt2_dev.cuh"

namespace gpt2 {

// ----------------------------------------------------------- smem layout
struct SmemLayout {
    uint32_t ring, full, empty, xs, vin, vq, vs, red, sc, ored, qh, rsc, misc, total;
};

__host__ __device__ inline uint32_t align16(uint32_t x) { return (x + 15u) & ~15u; }

constexpr int kRescalePerWarp = 192;  // int8 rescale scratch (rows x groups) per warp
constexpr int kMaxChunkRows = 64;

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
    s.sc = o; o = align16(o + max_pos * 4);
    s.ored = o; o = align16(o + kConsumerWarps * 32 * 4);
    s.qh = o; o = align16(o + 64 * 4);
    s.rsc = o; o = align16(o + (q8 ? kConsumerWarps * kRescalePerWarp * 4 : 0));
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

// Quantize v[0..N) per group of 64 into q/s (int8 path); one warp per group.
template <int N>
__device__ __forceinline__ void quantize_vec(const float* v, int8_t* q, float* s, int warp, int lane) {
    for (int gi = warp; gi < N / kGroup; gi += kConsumerWarps) {
        float a = v[gi * kGroup + lane], b = v[gi * kGroup + 32 + lane];
        // max of |v| starting from 0; NaN never wins a comparison, as in a plain compare loop
        float m = warp_max(fmaxf(fmaxf(fabsf(a), fabsf(b)), 0.0f));
        float sc = __fdiv_rn(m, 127.0f);
        q[gi * kGroup + lane] = (int8_t)quantize_one(a, sc);
        q[gi * kGroup + 32 + lane] = (int8_t)quantize_one(b, sc);
        if (lane == 0) s[gi] = sc;
    }
}

// --------------------------------------------------------- chunk compute
// fp32: rows of K floats in smem against x[K] in smem.  Lane 0 gets each sum.
template <int K, typename Epi>
__device__ __forceinline__ void chunk_f32(const float* w, int nrows, const float* x, int lane, int row0, Epi& epi) {
    constexpr int NV = K / 4;
    constexpr int T = (NV + 31) / 32;
    const float4* x4 = reinterpret_cast<const float4*>(x);
    const float4* w4 = reinterpret_cast<const float4*>(w);
    for (int rb = 0; rb < nrows; rb += 4) {
        const int nr = min(4, nrows - rb);
        float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
        for (int t = 0; t < T; ++t) {
            const int idx = lane + 32 * t;
            if ((NV % 32) == 0 || idx < NV) {
                const float4 xv = x4[idx];
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    if (r < nr) {
                        const float4 wv = w4[(rb + r) * NV + idx];
                        acc[r] = fmaf(xv.x, wv.x, acc[r]);
                        acc[r] = fmaf(xv.y, wv.y, acc[r]);
                        acc[r] = fmaf(xv.z, wv.z, acc[r]);
                        acc[r] = fmaf(xv.w, wv.w, acc[r]);
                    }
                }
            }
        }
#pragma unroll
        for (int r = 0; r < 4; ++r) acc[r] = warp_sum(acc[r]);
        if (lane == 0)
            for (int r = 0; r < nr; ++r) epi(row0 + rb + r, acc[r]);
    }
}

// int8: rows of [K int8][K/64 scales] against xq[K], xs[K/64].  Lane r gets
// row r of each pass.  Rescale in ascending group order, explicitly rounded.
template <int K, typename Epi>
__device__ __forceinline__ void chunk_q8(const uint8_t* w, int nrows, const int8_t* xq, const float* xs, int lane,
                                         float* scr, int row0, Epi& epi) {
    constexpr int NG = K / kGroup;
    constexpr int RB = row_bytes(K, true);
    constexpr int PR0 = kRescalePerWarp / NG;
    constexpr int PR = PR0 < 1 ? 1 : (PR0 > 32 ? 32 : PR0);
    for (int rb = 0; rb < nrows; rb += PR) {
        const int nr = min(PR, nrows - rb);
        for (int tk = lane; tk < nr * NG; tk += 32) {
            const int r = tk / NG, g = tk - r * NG;
            const uint8_t* row = w + (rb + r) * RB;
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
            scr[tk] = __fmul_rn(__fmul_rn(__int2float_rn(acc), xs[g]), sw);
        }
        __syncwarp();
        if (lane < nr) {
            float sum = 0.0f;
            for (int g = 0; g < NG; ++g) sum = __fadd_rn(sum, scr[lane * NG + g]);
            epi(row0 + rb + lane, sum);
        }
        __syncwarp();
    }
}

// -------------------------------------------------------------- kernel
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
    float* sc = reinterpret_cast<float*>(smem + lay.sc);
    float* ored = reinterpret_cast<float*>(smem + lay.ored);
    float* qh = reinterpret_cast<float*>(smem + lay.qh);
    float* rsc = reinterpret_cast<float*>(smem + lay.rsc);
    volatile int* s_abort = reinterpret_cast<volatile int*>(smem + lay.misc);
    volatile int* s_ok = s_abort + 1;
    unsigned* s_tok = reinterpret_cast<unsigned*>(smem + lay.misc) + 2;
    volatile int* s_nf = s_abort + 3;
    float* s_arg = reinterpret_cast<float*>(smem + lay.misc) + 8;  // [warps][3]

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int cta = blockIdx.x;
    const int L = P.L;
    const int phases_per_step = 4 * L + 1;

    if (tid == 0) {
        for (int i = 0; i < kSlots; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        *s_abort = ld_volatile_int(P.abort_flag);
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
        Geo pf_g = phase_geo(P, 0, cta, Q8);
        uint32_t pf_issued = 0;
        auto pf_advance = [&]() {
            // issue one prefetch at the cursor, then move it
            while (pf_s < P.n_steps && pf_k >= pf_g.nchunks) {
                pf_k = 0;
                if (++pf_ph == phases_per_step) { pf_ph = 0; ++pf_s; }
                if (pf_s < P.n_steps) pf_g = phase_geo(P, pf_ph, cta, Q8);
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
                const Geo g = phase_geo(P, ph, cta, Q8);
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
    uint32_t gi = 0;              // chunks consumed (same sequence as the producer)
    unsigned phase_no = 0;        // phases published by this run
    const int S = P.G >= P.H ? P.G / P.H : 1;  // key-axis splits per head
    const int units = P.H * S;
    const bool tracer = (P.trace != nullptr) && cta == 0;

    // Wait until every CTA has published phase `target` (warp 0 polls).
    auto grid_wait = [&](unsigned target) -> bool {
        if (warp == 0) {
            bool ok = false;
            uint64_t t0 = 0;
            while (true) {
                bool mine = true;
                for (int c = lane; c < P.G; c += 32) {
                    const unsigned f = ld_acquire_gpu(P.flags + c);
                    mine &= ((int)(f - target) >= 0);
                }
                if (__all_sync(0xffffffffu, mine)) { ok = true; break; }
                int give_up = 0;
                if (lane == 0) {
                    if (ld_volatile_int(P.abort_flag)) give_up = 1;
                    const uint64_t now = globaltimer_ns();
                    if (t0 == 0) t0 = now;
                    else if (now - t0 > P.wait_limit_ns) {
                        record_error(P, kDevTimeout);
                        give_up = 1;
                    }
                }
                if (__shfl_sync(0xffffffffu, give_up, 0)) break;
            }
            if (ok) __threadfence();
            if (lane == 0) *s_ok = ok ? 1 : 0;
        }
        consumers_sync();
        const bool ok = *s_ok != 0;
        if (!ok) *s_abort = 1;
        return ok;
    };
    auto publish = [&]() {
        ++phase_no;
        consumers_sync();
        if (tid == 0) {
            const bool skip = (cta == 0 && P.stall_phase >= 0 && (int)phase_no == P.stall_phase);
            if (!skip) {
                __threadfence();
                st_release_gpu(P.flags + cta, P.epoch + phase_no);
            }
        }
    };
    // Run this phase's chunks; false if a chunk never arrived.
    auto run_chunks = [&](int ph, auto&& body) -> bool {
        const Geo g = phase_geo(P, ph, cta, Q8);
        bool ok = true;
        for (int k = warp; k < g.nchunks; k += kConsumerWarps) {
            const uint32_t c = gi + k;
            const int slot = c % kSlots;
            uint64_t t0 = 0;
            uint32_t spins = 0;
            // every lane must observe the completed phase (acquire) before reading the slot
            while (!__all_sync(0xffffffffu, mbar_try_wait(&full[slot], (c / kSlots) & 1))) {
                if ((++spins & 255) == 0) {
                    int give_up = 0;
                    if (*s_abort || ld_volatile_int(P.abort_flag)) give_up = 1;
                    const uint64_t now = globaltimer_ns();
                    if (t0 == 0) t0 = now;
                    else if (now - t0 > P.wait_limit_ns) {
                        if (lane == 0) record_error(P, kDevTimeout);
                        give_up = 1;
                    }
                    if (__shfl_sync(0xffffffffu, give_up, 0)) { ok = false; break; }
                }
            }
            if (!ok) { *s_abort = 1; break; }
            const int row0 = g.r0 + k * g.rpc;
            const int n = min(g.rpc, g.nrows - k * g.rpc);
            body(ring + (size_t)slot * kSlotBytes, n, row0);
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);
        }
        gi += g.nchunks;
        consumers_sync();
        return ok && !*s_abort;
    };
    auto gemv = [&](int ph, int K_is_ff, auto& epi) -> bool {
        if (K_is_ff) {
            return run_chunks(ph, [&](const uint8_t* w, int n, int row0) {
                if constexpr (Q8) chunk_q8<FF>(w, n, vq, vs, lane, rsc + warp * kRescalePerWarp, row0, epi);
                else chunk_f32<FF>(reinterpret_cast<const float*>(w), n, vin, lane, row0, epi);
            });
        }
        return run_chunks(ph, [&](const uint8_t* w, int n, int row0) {
            if constexpr (Q8) chunk_q8<D>(w, n, vq, vs, lane, rsc + warp * kRescalePerWarp, row0, epi);
            else chunk_f32<D>(reinterpret_cast<const float*>(w), n, vin, lane, row0, epi);
        });
    };
    auto trace_vec = [&](int offset, const float* v, int n) {
        if (tracer)
            for (int i = tid; i < n; i += kConsumerWarps * 32) P.trace[offset + i] = v[i];
    };
    const int trace_layer = 8 * D + FF;

    unsigned prev_choice = *P.last_token;
    bool alive = true;
    for (int s = 0; s < P.n_steps && alive; ++s) {
        const int p = P.p0 + s;
        const bool trace_step = tracer && s == 0;
        // ---- token of this step
        unsigned tok = P.tokens_in ? P.tokens_in[s] : P.token0;
        if (tok == 0xFFFFFFFFu) tok = prev_choice;
        if (tok >= (unsigned)P.V) {
            if (tid == 0 && cta == 0) record_error(P, kDevToken);
            break;
        }
        for (int l = 0; l < L && alive; ++l) {
            const LayerParams& lp = P.lp[l];
            // ---------------- LN1 + QKV (+ KV append)
            if (l == 0) {
                for (int i = tid; i < D; i += kConsumerWarps * 32) {
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
                if (!grid_wait(P.epoch + phase_no)) { alive = false; break; }
                for (int i = tid; i < D; i += kConsumerWarps * 32) xs[i] = __ldcg(P.xa + i);
            }
            consumers_sync();
            layernorm<D>(xs, P.packed + lp.ln1_g, P.packed + lp.ln1_b, vin, red, tid);
            consumers_sync();
            if constexpr (Q8) {
                quantize_vec<D>(vin, vq, vs, warp, lane);
                consumers_sync();
            }
            if (trace_step) {
                trace_vec(l * trace_layer, xs, D);
                trace_vec(l * trace_layer + D, vin, D);
            }
            {
                float* kv_row = P.cache + ((uint64_t)p * L + l) * 2 * D;
                const float* bq = P.packed + lp.b_qkv;
                auto epi = [&](int j, float acc) {
                    const float y = __fadd_rn(acc, __ldg(bq + j));
                    P.qkv[j] = y;
                    if (j >= D) kv_row[j - D] = y;
                };
                if (!gemv(4 * l + kQKV, 0, epi)) { alive = false; break; }
            }
            publish();
            // ---------------- attention over positions 0..p (split along keys)
            if (!grid_wait(P.epoch + phase_no)) { alive = false; break; }
            for (int u = cta; u < units; u += P.G) {
                const int h = u / S, sp = u - h * S;
                const int n = p + 1;
                const int k0 = (int)(((long long)sp * n) / S), k1 = (int)(((long long)(sp + 1) * n) / S);
                const int nk = k1 - k0;
                if (tid < DH) qh[tid] = __ldcg(P.qkv + h * DH + tid);
                consumers_sync();
                constexpr int LPK = DH / 4;    // lanes per key
                constexpr int KPW = 32 / LPK;  // keys per warp pass
                const int sub = lane / LPK, l4 = lane % LPK;
                const float4 q4 = reinterpret_cast<const float4*>(qh)[l4];
                const float den = sqrtf((float)DH);
                for (int jb = k0 + warp * KPW; jb < k1; jb += kConsumerWarps * KPW) {
                    const int j = jb + sub;
                    float part = 0.0f;
                    if (j < k1) {
                        const float4 kv = __ldcg(reinterpret_cast<const float4*>(
                            P.cache + ((uint64_t)j * L + l) * 2 * D + h * DH + 4 * l4));
                        part = q4.x * kv.x + q4.y * kv.y + q4.z * kv.z + q4.w * kv.w;
                    }
#pragma unroll
                    for (int o = LPK / 2; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
                    if (j < k1 && l4 == 0) sc[j - k0] = part / den;
                }
                consumers_sync();
                float m = -INFINITY;
                for (int i = tid; i < nk; i += kConsumerWarps * 32) m = fmaxf(m, sc[i]);
                m = block_max(m, red, tid);
                for (int i = tid; i < nk; i += kConsumerWarps * 32) sc[i] = expf(sc[i] - m);
                consumers_sync();
                float z = 0.0f;
                for (int i = tid; i < nk; i += kConsumerWarps * 32) z += sc[i];
                z = block_sum(z, red, tid);
                constexpr int NGRP = kConsumerWarps * 32 / DH;
                const int grp = tid / DH, e = tid - grp * DH;
                float acc = 0.0f;
                for (int j = k0 + grp; j < k1; j += NGRP)
                    acc = fmaf(sc[j - k0], __ldcg(P.cache + ((uint64_t)j * L + l) * 2 * D + D + h * DH + e), acc);
                ored[grp * DH + e] = acc;
                consumers_sync();
                float* part = P.attn_part + (size_t)u * (DH + 2);
                if (tid < DH) {
                    float o = 0.0f;
                    for (int g2 = 0; g2 < NGRP; ++g2) o += ored[g2 * DH + tid];
                    part[2 + tid] = o;
                }
                if (tid == 0) {
                    part[0] = m;
                    part[1] = z;
                }
                consumers_sync();
            }
            publish();
            // ---------------- merge heads, out-projection + residual
            if (!grid_wait(P.epoch + phase_no)) { alive = false; break; }
            for (int idx = tid; idx < D; idx += kConsumerWarps * 32) {
                const int h = idx / DH, e = idx - h * DH;
                const float* hp = P.attn_part + (size_t)h * S * (DH + 2);
                float M = -INFINITY;
                for (int s2 = 0; s2 < S; ++s2) M = fmaxf(M, __ldcg(hp + s2 * (DH + 2)));
                float Z = 0.0f, O = 0.0f;
                for (int s2 = 0; s2 < S; ++s2) {
                    const float ms = __ldcg(hp + s2 * (DH + 2));
                    if (ms == -INFINITY) continue;
                    const float wgt = expf(ms - M);
                    Z = fmaf(wgt, __ldcg(hp + s2 * (DH + 2) + 1), Z);
                    O = fmaf(wgt, __ldcg(hp + s2 * (DH + 2) + 2 + e), O);
                }
                vin[idx] = O / Z;
            }
            consumers_sync();
            if constexpr (Q8) {
                quantize_vec<D>(vin, vq, vs, warp, lane);
                consumers_sync();
            }
            if (trace_step) {
                for (int i = tid; i < 3 * D; i += kConsumerWarps * 32)
                    P.trace[l * trace_layer + 2 * D + i] = __ldcg(P.qkv + i);
                trace_vec(l * trace_layer + 5 * D, vin, D);
            }
            {
                const float* bo = P.packed + lp.b_o;
                auto epi = [&](int j, float acc) { P.xb[j] = __fadd_rn(xs[j], __fadd_rn(acc, __ldg(bo + j))); };
                if (!gemv(4 * l + kO, 0, epi)) { alive = false; break; }
            }
            publish();
            // ---------------- LN2 + FC + GELU
            if (!grid_wait(P.epoch + phase_no)) { alive = false; break; }
            for (int i = tid; i < D; i += kConsumerWarps * 32) xs[i] = __ldcg(P.xb + i);
            consumers_sync();
            layernorm<D>(xs, P.packed + lp.ln2_g, P.packed + lp.ln2_b, vin, red, tid);
            consumers_sync();
            if constexpr (Q8) {
                quantize_vec<D>(vin, vq, vs, warp, lane);
                consumers_sync();
            }
            if (trace_step) {
                trace_vec(l * trace_layer + 6 * D, xs, D);
                trace_vec(l * trace_layer + 7 * D, vin, D);
            }
            {
                const float* bf = P.packed + lp.b_fc;
                auto epi = [&](int j, float acc) { P.u[j] = gelu_tanh(__fadd_rn(acc, __ldg(bf + j))); };
                if (!gemv(4 * l + kFC, 0, epi)) { alive = false; break; }
            }
            publish();
            // ---------------- MLP projection + residual
            if (!grid_wait(P.epoch + phase_no)) { alive = false; break; }
            for (int i = tid; i < FF; i += kConsumerWarps * 32) vin[i] = __ldcg(P.u + i);
            consumers_sync();
            if constexpr (Q8) {
                quantize_vec<FF>(vin, vq, vs, warp, lane);
                consumers_sync();
            }
            if (trace_step) trace_vec(l * trace_layer + 8 * D, vin, FF);
            {
                const float* bp = P.packed + lp.b_p;
                auto epi = [&](int j, float acc) { P.xa[j] = __fadd_rn(xs[j], __fadd_rn(acc, __ldg(bp + j))); };
                if (!gemv(4 * l + kP, 1, epi)) { alive = false; break; }
            }
            publish();
        }
        if (!alive) break;
        // ---------------- final LN + tied vocabulary projection + argmax
        if (!grid_wait(P.epoch + phase_no)) break;
        for (int i = tid; i < D; i += kConsumerWarps * 32) xs[i] = __ldcg(P.xa + i);
        consumers_sync();
        layernorm<D>(xs, P.packed + P.lnf_g, P.packed + P.lnf_b, vin, red, tid);
        consumers_sync();
        if constexpr (Q8) {
            quantize_vec<D>(vin, vq, vs, warp, lane);
            consumers_sync();
        }
        if (trace_step) {
            trace_vec(L * trace_layer, xs, D);
            trace_vec(L * trace_layer + D, vin, D);
        }
        ArgBest best = arg_init();
        {
            float* lg = P.logits ? P.logits + (uint64_t)s * P.logits_stride : nullptr;
            auto epi = [&](int j, float acc) {
                if (lg) lg[j] = acc;
                arg_update(best, acc, (unsigned)j);
            };
            if (!gemv(4 * L, 0, epi)) break;
        }
        // reduce the per-lane choices of this CTA
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
            float* ap = P.arg_part + (size_t)cta * 4;
            ap[0] = best.v;
            ap[1] = __uint_as_float(best.i);
            ap[2] = (float)best.nf;
        }
        publish();
        if (!grid_wait(P.epoch + phase_no)) break;
        if (tid == 0) {
            ArgBest gb = arg_init();
            for (int c = 0; c < P.G; ++c) {
                const float* ap = P.arg_part + (size_t)c * 4;
                arg_merge(gb, __ldcg(ap), __float_as_uint(__ldcg(ap + 1)), __ldcg(ap + 2) != 0.0f);
            }
            const int gnf = gb.nf;
            const unsigned choice = gnf ? 0xFFFFFFFFu : gb.i;
            *s_tok = choice;
            *s_nf = gnf;
            if (cta == 0) {
                if (P.tokens_out) P.tokens_out[s] = choice;
                *P.last_token = choice;
                if (gnf) atomicCAS(P.status, 0, (int)kDevNonfinite);
            }
        }
        consumers_sync();
        prev_choice = *s_tok;
        if (*s_nf) break;  // a non-finite logit ends the run (same decision in every CTA)
    }
    // Make the producer stop if the consumers left early.
    if (tid == 0) *s_abort = 1;
}

// ------------------------------------------------------------ test hooks
// One projection of the model on a given input vector, with the step
// kernel's own routines (activation quantizer, chunk dot products,
// epilogue bias add).  Block: 8 warps over 64 output rows.
template <int K, bool Q8>
__global__ void __launch_bounds__(kConsumerWarps * 32) project_kernel(const uint8_t* __restrict__ rows, int N,
                                                                      const float* __restrict__ x,
                                                                      const float* __restrict__ bias,
                                                                      float* __restrict__ y) {
    __shared__ __align__(16) float vin[K];
    __shared__ __align__(16) int8_t vq[K];
    __shared__ float vs[K / kGroup];
    __shared__ float scr[kConsumerWarps * kRescalePerWarp];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    for (int i = tid; i < K; i += blockDim.x) vin[i] = x[i];
    __syncthreads();
    if constexpr (Q8) quantize_vec<K>(vin, vq, vs, warp, lane);
    __syncthreads();
    auto epi = [&](int j, float acc) { y[j] = bias ? __fadd_rn(acc, bias[j]) : acc; };
    const int rb = row_bytes(K, Q8);
    const int r0 = blockIdx.x * 64 + warp * 8;
    const int n = min(8, N - r0);
    if (n <= 0) return;
    if constexpr (Q8) chunk_q8<K>(rows + (size_t)r0 * rb, n, vq, vs, lane, scr + warp * kRescalePerWarp, r0, epi);
    else chunk_f32<K>(reinterpret_cast<const float*>(rows + (size_t)r0 * rb), n, vin, lane, r0, epi);
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
    project_kernel<K, Q8><<<(N + 63) / 64, kConsumerWarps * 32, 0, st>>>(rows, N, x, bias, y);
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
    return per_sm * sms;
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
