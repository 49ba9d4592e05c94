// cstep.cuh -- geometry of the cluster step kernel (cstep.cu), shared by the
// host code that lays out its weight stream and scratch.
//
// The kernel runs one cached GPT-2 step per iteration (LeanExe GPT-2 README,
// model and cachedStep paragraphs) on NC thread-block clusters of CS CTAs.
// Rank r of every cluster owns the column slice [r*SW, (r+1)*SW) of the
// model width (SW = D / CS).  Per layer:
//   stage A (clusters that own a head h = c, c + NC, ...): the CTA's slice of
//     the block input is formed from the previous MLP partials; each CTA
//     computes the LN1-folded QKV dot products of head h over its slice;
//     one cluster all-gather (distributed shared memory) completes q, k, v;
//     each CTA runs attention over its share of the keys; a second
//     all-gather merges the shares; each CTA projects its SW output rows of
//     the head's out-projection and publishes them (tagged words).
//   stage B (every cluster): the CTA's slice of the attention residual is
//     formed from the heads' out-projection partials; LN2-folded FC dot
//     products of the cluster's FC rows over the slice; one all-gather
//     completes the cluster's GELU outputs; each CTA projects its SW output
//     rows of the MLP projection restricted to those FC rows and publishes
//     them.
// So a layer has two grid-wide exchanges (the two sets of partials) and
// three cluster all-gathers.
#pragma once
#include <cstdint>

#include "gpt2_dev.cuh"

namespace gpt2 {

constexpr int kCMaxClusters = 32;
// Seven consumer warps plus the producer: at most two warps per SM
// sub-partition, so every thread may use 255 registers (a third warp on one
// sub-partition caps it at 168, and spills land in local memory, which has
// little L1 left beside the ring).
constexpr int kCWarps = 7;                       // consumer warps
constexpr int kCThreads = (kCWarps + 1) * 32;    // + one producer warp
constexpr int kCSlotBytes = 16384;               // one ring slot
constexpr int kCMaxSlots = 16;
constexpr int kCMaxSmem = 232448;                // opt-in shared memory per CTA on sm_103

struct CGeo {
    int CS, NC, G;      // cluster size, clusters, CTAs (NC * CS)
    int SW;             // slice width (floats of the model width per rank)
    int HPC;            // most heads one cluster owns
    int wb;             // bytes per weight in the stream (4 binary32, 2 binary16)
    int nfc_max;        // most FC rows one cluster owns
    int slots;          // ring slots
    int fc0[kCMaxClusters + 1];             // FC rows of cluster c: [fc0[c], fc0[c+1])
    uint64_t seg[kCMaxClusters + 1];        // byte offset of cluster c's part of a layer
    uint64_t cta_bytes[kCMaxClusters];      // bytes of one CTA's part of a layer (cluster c)
    uint64_t layer_bytes;                   // bytes of one layer of the stream
};

// Heads of cluster c: h = c + k * NC for k < cg_heads.
__host__ __device__ inline int cg_heads(const CGeo& g, int H, int c) { return c < H ? (H - 1 - c) / g.NC + 1 : 0; }

// Byte layout of one CTA's part of a layer, for cluster c with nh heads:
// per head slot k: QKV piece rows (3*DH rows of SW weights: the head's q,
// k, v output rows over the CTA's columns), then the out-projection piece
// (SW output rows of DH weights: the CTA's output rows over the head's
// inputs); then the FC piece (nfc rows of SW weights) and the MLP piece (SW
// output rows of nfc weights).
__host__ __device__ inline uint64_t cg_head_bytes(const CGeo& g, int DH) {
    return (uint64_t)(3 * DH * g.SW + g.SW * DH) * (uint64_t)g.wb;
}

// Everything one launch of the cluster step kernel needs.
struct CPlan {
    StepPlan s;                 // shape, weights, session buffers and run (exchange fields unused)
    CGeo g;
    const uint8_t* cstream;     // the cluster weight stream: [layer][cluster][rank] parts
    uint64_t* partO;            // [H][D] out-projection partials of each head (tagged words)
    uint64_t* partP;            // [2][NC][D] MLP-projection partials of each cluster, by layer parity (tagged words)
};

// Cluster size for width D: CS = D / 128 when that is at most 8 (GPT-2
// 124M: 6, one warp of float4 columns per CTA), else D / 32; a constant of
// the kernel's instantiation.
__host__ __device__ constexpr int cluster_size_for(int D) {
    return (D % 128 == 0 && D / 128 <= 8) ? D / 128 : (D % 32 == 0 && D / 32 <= 8) ? D / 32 : 1;
}

// Stamps per CTA in the timing buffer of the cluster kernel.
__host__ __device__ inline int cstamps_per_cta(int L) { return 16 * L + 8; }

// Scratch of one cluster-kernel run, as byte offsets in one contiguous area.
struct CScratch {
    size_t words, last_token, partO, partP, arg, total;
};

__host__ __device__ inline CScratch cscratch_layout(int D, int H, int NC, int G) {
    CScratch k{};
    size_t o = 0;
    k.words = o; o = up256(o + 4 * 4);
    k.last_token = o; o = up256(o + 4 * 2);
    k.partO = o; o = up256(o + 8 * (size_t)H * D);
    k.partP = o; o = up256(o + 8 * 2 * (size_t)NC * D);
    k.arg = o; o = up256(o + 8 * 2 * (size_t)G);
    k.total = o;
    return k;
}

// Shared-memory layout of the cluster step kernel (byte offsets).
struct CSmem {
    uint32_t ring, full, empty, bars, gA, gT, gB, gX, qkv, oh, uu, xs, xin, xf, stage, misc, shares, plan, total;
};

// Head slots per cluster at most (a layer has 2 * heads + 2 shares per CTA).
constexpr int kCMaxHeadSlots = 8;
// A CTA's share j of every layer, relative to its part of the layer.
struct CShareRow {
    uint32_t off, pb;
    int n, rpc, nch, pad0, pad1, pad2;
};

__host__ __device__ constexpr uint32_t calign16(uint32_t x) { return (x + 15u) & ~15u; }

__host__ __device__ inline CSmem csmem_layout(int D, int DH, int CS, int SW, int nfc_max, int slots) {
    CSmem s{};
    uint32_t o = 0;
    s.ring = o; o += (uint32_t)slots * kCSlotBytes;
    s.full = o; o += (uint32_t)slots * 8;
    s.empty = o; o += (uint32_t)slots * 8;
    s.bars = o; o += 8 * 8;                                        // mA[2], mT[2], mB[2], mX
    s.gA = o; o = calign16(o + 2u * CS * (3 * DH + 4) * 4);       // [2][CS][3DH + 4]
    s.gT = o; o = calign16(o + 2u * CS * (DH + 4) * 4);           // [2][CS][DH + 4]
    s.gB = o; o = calign16(o + 2u * CS * (nfc_max + 4) * 4);      // [2][CS][nfc_max + 4]
    s.gX = o; o = calign16(o + (uint32_t)D * 4);                  // all-gathered vector of the cluster
    s.qkv = o; o = calign16(o + 3u * DH * 4);
    s.oh = o; o = calign16(o + (uint32_t)DH * 4);
    s.uu = o; o = calign16(o + (uint32_t)(nfc_max + 4) * 4);
    s.xs = o; o = calign16(o + (uint32_t)SW * 4);
    s.xin = o; o = calign16(o + (uint32_t)SW * 4);
    s.xf = o; o = calign16(o + (uint32_t)D * 4);
    s.stage = o; o = calign16(o + 768u * 4);
    s.misc = o; o = calign16(o + 64u * 4);
    s.shares = o; o = calign16(o + (uint32_t)(2 * kCMaxHeadSlots + 2) * (uint32_t)sizeof(CShareRow));
    s.plan = o; o = calign16(o + (uint32_t)sizeof(CPlan));
    s.total = o;
    return s;
}

}  // namespace gpt2
