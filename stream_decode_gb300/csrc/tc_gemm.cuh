// tc_gemm.cuh -- the prefill projections on the 5th-generation tensor cores.
//
// C_part[split][m][n] = sum over this split's K range of A[m][k] * B[n][k]
// for one 128 x TN output tile per CTA (rows m of the prompt, TN = 64 or
// 128 output features n), with both operands K-major in global memory
// (activations [n_tok][K]; weights [N][K], the device layout of every block
// matrix).  The wider tile reads each activation tile for twice as many
// output features (half the activation traffic from L2) at one stage less.
//
// binary32 accuracy from TF32 tensor cores ("3xTF32"): each operand x is
// split as x = hi + lo with hi = x with its low 13 mantissa bits cleared
// (exactly a TF32 value) and lo = x - hi (exact in binary32); the tile
// accumulates hi_A*hi_B + hi_A*lo_B + lo_A*hi_B in fp32 in tensor memory.
// The dropped lo_A*lo_B term and the TF32 rounding of lo are ~2^-22
// relative, far inside the binary32 tolerance of the logits.
//
// Pipeline per CTA (128 threads): warp 0 lane 0 issues TMA tile loads (128 B
// swizzle) of A_hi, A_lo, B_hi, B_lo for each 32-wide K block into a ring of
// as many stages as the shared stage area holds (mbarriers full/empty); warp 1 lane 0 issues
// tcgen05.mma (M=128, N=TN, K=8, kind::tf32, accumulator in TMEM) and
// commits each stage back to its producer; after the last block all four
// warps read the accumulator rows (tcgen05.ld 32x32b) and store the fp32
// partial tile.  Every wait is bounded; on expiry the CTA records an error,
// drains its copies and MMAs and still frees its tensor memory.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "chain.cuh"

namespace gpt2 {
namespace tc {

constexpr int kTileM = 128;            // prompt rows per tile (the MMA's M)
constexpr int kTileN = 64;             // the narrow tile's output features (the MMA's N); a shape multiple
constexpr int kBlockK = 32;            // K per stage: one 128-byte swizzle row of fp32
constexpr int kMmaK = 8;               // K per tcgen05.mma of kind::tf32
constexpr int kTcThreads = 128;
constexpr uint32_t kABytes = kTileM * kBlockK * 4;  // 16 KB per A tile (hi or lo)
// per tile width TN (64 or 128): B tile bytes, stage bytes, stages, dynamic shared memory
__host__ __device__ constexpr uint32_t tc_bbytes(int TN) { return (uint32_t)TN * kBlockK * 4; }
// the stage area every instantiation shares: four 128 x 64 stages
constexpr uint32_t kTcArea = 4 * (2 * kABytes + 2 * 64 * kBlockK * 4);
__host__ __device__ constexpr uint32_t tc_smem(int TN) {
    return kTcArea + 1024 /* alignment slack */ + 256 /* barriers */;
}
static_assert(kABytes % 1024 == 0 && tc_bbytes(64) % 1024 == 0, "tiles stay 1024-byte aligned for the swizzle atoms");
static_assert(tc_smem(128) <= 232448, "the wide tile's stages fit in shared memory");

struct TcMaps {
    CUtensorMap a_hi, a_lo, b_hi, b_lo;  // A: dims {K, rows}; B: dims {K, N}; boxes {32, 128} / {32, 64}
};

__device__ __forceinline__ uint32_t su32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

// UMMA shared-memory descriptor of a K-major tile in the 128-byte swizzle
// layout: 8-row x 128-byte atoms stacked every 1024 bytes (stride byte
// offset), leading byte offset unused for swizzled K-major tiles (16 B),
// descriptor version 1, layout type 2 (128-byte swizzle).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);       // start address
    d |= (uint64_t)(16u >> 4) << 16;                 // leading byte offset
    d |= (uint64_t)(1024u >> 4) << 32;               // stride byte offset
    d |= (uint64_t)1 << 46;                          // version
    d |= (uint64_t)2 << 61;                          // 128-byte swizzle
    return d;
}

// Instruction descriptor: fp32 accumulator, TF32 A and B, both K-major,
// N = TN, M = kTileM.
__host__ __device__ constexpr uint32_t instr_desc(int TN) {
    return (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(TN >> 3) << 17) | ((uint32_t)(kTileM >> 4) << 24);
}

__device__ __forceinline__ void tc_mbar_init(uint64_t* b, uint32_t n) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(b)), "r"(n) : "memory");
}
__device__ __forceinline__ bool tc_try_wait(uint64_t* b, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(su32(b)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded wait: false after `limit` polls.
__device__ __forceinline__ bool tc_wait(uint64_t* b, uint32_t parity, uint32_t limit) {
    for (uint32_t i = 0; i < limit; ++i)
        if (tc_try_wait(b, parity)) return true;
    return false;
}
__device__ __forceinline__ void tc_arrive_expect(uint64_t* b, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(b)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int c0, int c1, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            su32(dst)),
        "l"(map), "r"(c0), "r"(c1), "r"(su32(bar))
        : "memory");
}
__device__ __forceinline__ void mma_tf32(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(su32(bar))
                 : "memory");
}

// One CTA: tile (blockIdx.x = n tile, blockIdx.y = split, blockIdx.z = m
// tile) over K blocks [kb0, kb1) of the split; writes part[split][row][col]
// for rows < m_rows (TMA fills rows past m_rows with zeros).  a_rows: rows
// of each A tile loaded, 128, or 64 when m_rows <= 64: accumulator row r
// depends only on A row r, so the unloaded upper half of the A tiles only
// feeds accumulator rows that are never stored.  err: set to
// err_code (if still 0) when any wait expires.
template <int TN, int AR = kTileM>
__global__ void __launch_bounds__(kTcThreads, 1)
    tf32x3_gemm_kernel(const __grid_constant__ TcMaps maps, int K, int N, int m_rows, int splits, float* part,
                       int* err, int err_code, int a_rows) {
    // AR: rows of each stored A tile (64 when the tile has at most 64 valid
    // rows: the stage is smaller and the area holds more stages; the MMA
    // still reads 128 rows of A, rows 64..127 being the bytes that follow in
    // the stage, which feed only accumulator rows that are never stored)
    constexpr uint32_t kABytes = (uint32_t)AR * kBlockK * 4;
    constexpr uint32_t kBBytes = tc_bbytes(TN), kStageBytes = 2 * kABytes + 2 * kBBytes;
    constexpr int kTcStages = (int)(kTcArea / kStageBytes) < 6 ? (int)(kTcArea / kStageBytes) : 6;
    constexpr uint32_t kTmemCols = (uint32_t)TN;  // fp32 accumulator columns
    extern __shared__ uint8_t tc_smem_raw[];
    // 1024-byte aligned stage area (swizzle atoms), barriers after it
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(tc_smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(base + kTcArea);
    uint64_t* empty = full + kTcStages;
    uint64_t* done = empty + kTcStages;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
    volatile int* s_bad = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n0 = blockIdx.x * TN;
    const int split = blockIdx.y;
    const int m0 = blockIdx.z * kTileM;
    const int nkb = K / kBlockK;
    const int kb0 = (int)(((long long)split * nkb) / splits), kb1 = (int)(((long long)(split + 1) * nkb) / splits);
    constexpr uint32_t kLimit = 1u << 22;  // polls before a wait is declared expired

    if (threadIdx.x == 0) {
        for (int i = 0; i < kTcStages; ++i) {
            tc_mbar_init(&full[i], 1);
            tc_mbar_init(&empty[i], 1);
        }
        tc_mbar_init(done, 1);
        *s_bad = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(tmem_slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = *tmem_slot;
    // everything above touched shared and tensor memory only; the A tiles
    // and the partials are the neighbouring kernels' data
    chain_enter();

    if (warp == 0 && lane == 0) {
        // ---- TMA producer
        int issued = 0;
        for (int kb = kb0; kb < kb1; ++kb) {
            const int i = kb - kb0, s = i % kTcStages;
            if (i >= kTcStages && !tc_wait(&empty[s], ((i / kTcStages) - 1) & 1, kLimit)) {
                *s_bad = 1;
                break;
            }
            uint8_t* st = base + s * kStageBytes;
            tc_arrive_expect(&full[s], 2u * (uint32_t)a_rows * kBlockK * 4u + 2u * kBBytes);
            tma_load_2d(st, &maps.a_hi, kb * kBlockK, m0, &full[s]);
            tma_load_2d(st + kABytes, &maps.a_lo, kb * kBlockK, m0, &full[s]);
            tma_load_2d(st + 2 * kABytes, &maps.b_hi, kb * kBlockK, n0, &full[s]);
            tma_load_2d(st + 2 * kABytes + kBBytes, &maps.b_lo, kb * kBlockK, n0, &full[s]);
            issued = i + 1;
        }
        // drain: the most recent fill of every stage has landed before this CTA can exit
        for (int s = 0; s < kTcStages && s < issued; ++s) {
            const int last = s + kTcStages * ((issued - 1 - s) / kTcStages);  // last fill index of stage s
            if (!tc_wait(&full[s], (last / kTcStages) & 1, kLimit)) *s_bad = 1;
        }
    } else if (warp == 1 && lane == 0) {
        // ---- MMA issuer
        const uint32_t idesc = instr_desc(TN);
        bool any = false;
        for (int kb = kb0; kb < kb1; ++kb) {
            const int i = kb - kb0, s = i % kTcStages;
            if (!tc_wait(&full[s], (i / kTcStages) & 1, kLimit)) {
                *s_bad = 1;
                break;
            }
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            const uint32_t st = su32(base + s * kStageBytes);
#pragma unroll
            for (int j = 0; j < kBlockK / kMmaK; ++j) {
                const uint32_t koff = (uint32_t)j * kMmaK * 4;  // bytes along the 128-byte row
                const uint64_t ahi = smem_desc(st + koff), alo = smem_desc(st + kABytes + koff);
                const uint64_t bhi = smem_desc(st + 2 * kABytes + koff), blo = smem_desc(st + 2 * kABytes + kBBytes + koff);
                mma_tf32(tmem, ahi, bhi, idesc, any ? 1u : 0u);
                any = true;
                mma_tf32(tmem, ahi, blo, idesc, 1u);
                mma_tf32(tmem, alo, bhi, idesc, 1u);
            }
            mma_commit(&empty[s]);
        }
        mma_commit(done);  // fires when every MMA issued above has completed
    }
    __syncwarp();
    // ---- epilogue: every warp reads its 32 accumulator lanes (tile rows)
    const bool ok = tc_wait(done, 0, kLimit);
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const int row = m0 + warp * 32 + lane;
    float* dst = part + ((size_t)split * m_rows + row) * N + n0;
#pragma unroll
    for (int c0 = 0; c0 < TN; c0 += 16) {
        uint32_t v[16];
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
            "%14, %15}, [%16];"
            : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
              "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
            : "r"(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)c0));
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
        if (ok && row < m_rows) {
#pragma unroll
            for (int q = 0; q < 16; q += 4)
                *reinterpret_cast<float4*>(dst + c0 + q) = make_float4(__uint_as_float(v[q]), __uint_as_float(v[q + 1]),
                                                                        __uint_as_float(v[q + 2]), __uint_as_float(v[q + 3]));
        }
    }
    if ((!ok || *s_bad) && threadIdx.x == 0) atomicCAS(err, 0, err_code);
    // tensor memory is freed only after every MMA has completed
    if (!ok && threadIdx.x == 0) tc_wait(done, 0, kLimit);
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == 0) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
    }
}

}  // namespace tc
}  // namespace gpt2
