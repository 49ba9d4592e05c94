// gpt2_dev.cuh -- device-side definitions shared by the library's kernels:
// the step plan, the device weight-stream geometry, the scratch layout and
// inline-PTX wrappers (mbarrier, bulk copies, tagged words).
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace gpt2 {

// ---------------------------------------------------------------- constants
constexpr int kGroup = 64;          // int8 group size (quantized GPT-2 abstract)
// Seven consumer warps plus the producer: at most two warps per SM
// sub-partition, so every thread may hold up to 255 registers (three warps
// on one sub-partition would cap it at 168 and spill into local memory,
// which has almost no L1 left beside the 220+ KB of shared memory).
constexpr int kConsumerWarps = 7;   // warps that compute
constexpr int kThreads = (kConsumerWarps + 1) * 32;  // + one producer warp
constexpr int kSlotBytes = 12288;   // one ring slot (one 3072-float row)
constexpr int kSlots = 16;          // ring depth: 192 KiB of weights in flight per SM
constexpr float kLnEps = 1e-5f;
// Least interval between the producer's block-weight chunk issues (ns).
// 12 KB per 300 ns per SM is about 6 TB/s over 152 SMs: enough to keep the
// ring full, while spreading the refills that a phase boundary releases.
constexpr uint32_t kDefaultPaceNs = 300;

// status words written by the device
enum DevStatus : int {
    kDevOk = 0,
    kDevToken = 2,
    kDevNonfinite = 6,
    kDevTimeout = 9,
};

// Matrix kinds in the per-layer weight stream, in stream order.
enum Mat : int { kQKV = 0, kO = 1, kFC = 2, kP = 3, kVocab = 4 };

// Packed-checkpoint word offsets of the small per-layer tensors the step
// reads directly (LayerNorm parameters and biases).
struct LayerParams {
    uint64_t ln1_g, ln1_b, b_qkv, b_o, ln2_g, ln2_b, b_fc, b_p;
};

constexpr int kMaxLayers = 16;

constexpr int kMaxSplits = 4;   // key-axis splits per attention head
constexpr int kMaxGrid = kConsumerWarps * 32;  // CTAs of the step kernel (one per SM on GB300: 152)

// Key-axis splits per head for a grid of G CTAs and H heads.
__host__ __device__ inline int attn_splits(int G, int H) {
    int s = G >= H ? G / H : 1;
    return s > kMaxSplits ? kMaxSplits : s;
}

// Splits used at a given number of keys: one per 128 keys (a unit's seven
// warps take 56 keys per pass, so a split costs at most three passes), at
// most `cap`.  Up to 128 keys a head is one unit, whose output is final: the
// out-projection then gathers it with no merge of partial softmaxes.
constexpr int kKeysPerSplit = 128;
__host__ __device__ inline int attn_splits_for(int keys, int cap) {
    const int s = (keys + kKeysPerSplit - 1) / kKeysPerSplit;
    return s < 1 ? 1 : (s > cap ? cap : s);
}

// Scratch of one step-kernel run, as byte offsets in one contiguous area.
// Every exchanged value is a 64-bit tagged word (float bits | tag << 32).
struct ScratchLayout {
    size_t words, last_token, xa, xb, qkv, u, attn, arg, total;
};

__host__ __device__ inline size_t up256(size_t x) { return (x + 255) & ~size_t(255); }

__host__ __device__ inline ScratchLayout scratch_layout(int D, int H, int FF, int G) {
    const size_t DH = (size_t)(D / H), units = (size_t)H * attn_splits(G, H);
    ScratchLayout k{};
    size_t o = 0;
    k.words = o; o = up256(o + 4 * 4);
    k.last_token = o; o = up256(o + 4 * 2);
    k.xa = o; o = up256(o + 8 * (size_t)D);
    k.xb = o; o = up256(o + 8 * (size_t)D);
    k.qkv = o; o = up256(o + 8 * 3 * (size_t)D);
    k.u = o; o = up256(o + 8 * (size_t)FF);
    k.attn = o; o = up256(o + 8 * units * (DH + 2));
    k.arg = o; o = up256(o + 8 * 2 * (size_t)G);
    k.total = o;
    return k;
}

// Everything one launch of the step kernel needs.  Passed by value.
struct StepPlan {
    // shape
    int L, D, H, FF, V, n_pos, max_pos;
    int G;  // CTAs in the grid
    // weights
    const float* packed;        // packed checkpoint on the device
    const float* fold;          // binary32: per layer the LayerNorm folds c, d of the QKV and FC rows (fold_layer_words)
    const uint8_t* wstream;     // per layer: qkv[3D] rows, o[D], fc[FF], p[D] (K-major rows)
    uint64_t layer_bytes;       // bytes of one layer in wstream
    uint64_t mat_off[4];        // byte offset of each matrix inside a layer
    const uint8_t* vocab;       // vocab rows (fp32: wte in the packed checkpoint; int8: q rows + scales)
    uint64_t wte_off, wpe_off, lnf_g, lnf_b;  // word offsets in packed
    LayerParams lp[kMaxLayers];
    // session buffers (tagged words: value bits | tag << 32)
    float* cache;               // [max_pos][L][2D]
    uint64_t* xa;               // [D] residual stream after a block
    uint64_t* xb;               // [D] residual stream after attention
    uint64_t* qkv;              // [3D]
    uint64_t* u;                // [FF]
    uint64_t* attn_part;        // [H * S][2 + DH]: max, sum, unnormalised o
    uint64_t* arg_part;         // [G][2]: best value, index | nonfinite << 31
    unsigned epoch;             // tags of this run start above this
    int* status;                // sticky device status
    int* abort_flag;            // set by any CTA that gives up
    uint32_t* last_token;       // the session's last greedy choice
    // the run
    int p0, n_steps;
    const uint32_t* tokens_in;  // [n_steps]
    uint32_t token0;            // used when tokens_in == nullptr (single host-token step)
    uint32_t* tokens_out;       // [n_steps] or null
    float* logits;              // or null
    uint64_t logits_stride;     // floats between steps' logits
    float* trace;               // or null
    uint64_t* timing;           // or null: [phase of step 0][G][3] globaltimer stamps
    // robustness
    uint64_t wait_limit_ns;     // bound of every spin-wait
    int stall_phase;            // test: CTA 0 skips publishing this phase (-1 = none)
    int prefetch_chunks;        // L2 bulk prefetch distance in chunks (0 = off)
    uint32_t pace_ns;           // least interval between block-weight chunk issues (0 = unpaced)
    int act_row;                // int8: one activation scale per projection input vector (else per 64)
};

// LayerNorm folded into the projection that follows it (binary32 models):
// with n = (x - mean) * rstd and y = W (g * n + b) + bias,
//   y_j = rstd * (sum_i W_ji g_i x_i - mean * c_j) + d_j,
//   c_j = sum_i W_ji g_i,   d_j = bias_j + sum_i W_ji b_i,
// so the dot products can start on the raw residual stream while its
// mean and variance are still being reduced.  Per layer: c_qkv[3D],
// d_qkv[3D], c_fc[FF], d_fc[FF].
__host__ __device__ constexpr uint64_t fold_layer_words(int D, int FF) { return 2ull * (3ull * D + (uint64_t)FF); }

// Weight formats of the device streams: binary32; int8 group-64 codes with
// their binary32 group scales; binary16 (weights rounded to nearest-even
// half precision, widened to binary32 before every multiply-add).
enum WeightFormat : int { kWF32 = 0, kWQ8 = 1, kWF16 = 2 };

// Bytes of one K-major weight row in the device stream.
__host__ __device__ constexpr int row_bytes(int K, int wf) {
    return wf == kWQ8 ? K + ((K / kGroup) * 4 + 15) / 16 * 16 : (wf == kWF16 ? K * 2 : K * 4);
}

// --------------------------------------------------------------- PTX helpers
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Global -> shared bulk copy completing on an mbarrier (16-byte aligned
// addresses, size a multiple of 16).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                          uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
        "%4;" ::"r"(smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void st_release_gpu(unsigned* p, unsigned v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned* p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Tagged words: one single-copy-atomic 64-bit access carries a value and
// the number of the phase that produced it.
__device__ __forceinline__ uint64_t tag_pack(unsigned tag, float v) {
    return ((uint64_t)tag << 32) | (uint64_t)__float_as_uint(v);
}
__device__ __forceinline__ unsigned tag_of(uint64_t w) { return (unsigned)(w >> 32); }
__device__ __forceinline__ float val_of(uint64_t w) { return __uint_as_float((unsigned)w); }

__device__ __forceinline__ void st_tagged(uint64_t* p, unsigned tag, float v) {
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(tag_pack(tag, v)) : "memory");
}
__device__ __forceinline__ void st_tagged_release(uint64_t* p, uint64_t w) {
    asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(w) : "memory");
}
__device__ __forceinline__ uint64_t ld_tagged(const uint64_t* p) {
    uint64_t v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
// Two consecutive tagged words in one 16-byte access (16-byte aligned);
// each word is single-copy atomic on its own.
__device__ __forceinline__ void ld_tagged_x2(const uint64_t* p, uint64_t& a, uint64_t& b) {
    asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "l"(p) : "memory");
}
__device__ __forceinline__ uint64_t ld_tagged_acquire(const uint64_t* p) {
    uint64_t v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ int ld_volatile_int(const int* p) {
    return *reinterpret_cast<const volatile int*>(p);
}

// Named barrier over the consumer warps only (the producer warp never joins).
__device__ __forceinline__ void consumers_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
}

// int8 quantization rule shared by activations and weights: nearest-even,
// saturate to [-127, 127], a zero scale or a NaN quotient gives 0.
__device__ __forceinline__ int quantize_one(float x, float s) {
    float r = 0.0f;
    if (s != 0.0f) r = rintf(__fdiv_rn(x, s));
    if (r != r) r = 0.0f;
    r = fminf(fmaxf(r, -127.0f), 127.0f);
    return static_cast<int>(r);
}

// The same code as quantize_one(x, s), given inv = 1/s rounded to nearest.
// The product y = x * inv is within 2.5 ulp of the rounded quotient x / s,
// so their nearest-even integers agree unless a half-integer lies within
// that distance; for a group's own values |x / s| <= 127, where ulp(y) <=
// 2^-17.  When y is within 8 * 2^-17 of the half-integer between its
// neighbouring integers (about one value in 8000), or out of range, or s is
// 0, the quotient itself decides.
__device__ __forceinline__ int quantize_fast(float x, float s, float inv) {
    const float y = __fmul_rn(x, inv);
    const float d = fabsf(__fsub_rn(__fsub_rn(y, floorf(y)), 0.5f));
    if (s != 0.0f && fabsf(y) < 128.0f && d > 6.103515625e-05f) {
        const float r = rintf(y);
        return static_cast<int>(fminf(fmaxf(r, -127.0f), 127.0f));
    }
    return quantize_one(x, s);
}

}  // namespace gpt2
